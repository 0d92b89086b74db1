// guard.h -- guard bands around the library's device scratch (library-level
// bookkeeping; the step kernels do not use it).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lc {

// Status-word bit set when a guard band changed (bits 1 and 2 are the step
// kernels' own, in internal.h).
constexpr int kStatusGuard = 4;

// kGuardBytes of the byte kGuardByte sit directly before and after each
// scratch buffer the kernels write (wire, M1 partials, M1, 1/M1).
constexpr int kGuardBytes = 256;
constexpr uint32_t kGuardByte = 0xA5u;
constexpr int kMaxGuardBands = 8;

struct GuardList {
    const uint32_t* band[kMaxGuardBands];  // each kGuardBytes long, 4-byte aligned
    int n;
};

// Enqueue the check of every band in g; a changed band ORs kStatusGuard into
// *status.
cudaError_t launch_guard_check(const GuardList& g, int* status, cudaStream_t s);

}  // namespace lc
