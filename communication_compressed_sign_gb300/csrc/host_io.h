// host_io.h -- device side of the host-buffer step's theta download.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lc {

// Store n floats of device memory src into dst, the device address of a
// mapped page-locked host buffer, with SM threads (no copy engine).  Both
// pointers 16-byte aligned.
cudaError_t launch_store_host(const float* src, float* dst, int64_t n, cudaStream_t s);

}  // namespace lc
