// internal.h -- shared declarations of the lioncub CUDA library (not part of
// the public C ABI in include/lioncub.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lioncub.h"

namespace lc {

// Tiled kernels: 256 threads, 8 consecutive elements per thread, so one tile
// is 2048 elements.  Tiles never cross a tensor boundary (tensor offsets are
// multiples of 32 elements), which keeps every packed word inside one tile
// and gives each tile one tensor's M1 scale.
constexpr int kThreads = 256;
constexpr int kVec = 8;
constexpr int kTile = kThreads * kVec;
// Data-parallel exchange: each rank's chunk of the parameter vector is a
// multiple of this many elements, so a chunk's wire rows start on 16-byte
// boundaries for every code width and a packed word never spans two chunks.
constexpr int64_t kDistChunkAlign = 4096;

// One tile: elements [start, start + len); meta = tensor index, with bit 31
// set when the tensor's momentum is synchronized across workers.
struct Tile {
    int64_t start;
    int32_t len;
    uint32_t meta;
};
constexpr uint32_t kTileSync = 0x80000000u;

// Everything a step's kernels read, passed by value (about 2.2 KB).
struct StepArgs {
    const void* g[LIONCUB_MAX_WORKERS];
    float* m[LIONCUB_MAX_WORKERS];
    float* theta;
    uint32_t* wire;         // W x wire_stride words (packed signs or codes)
    int64_t wire_stride;    // words per worker, a multiple of 4
    int64_t d;
    const Tile* tiles;          // unsynchronized tensors' tiles first, then synchronized ones
    int64_t ntiles;
    int64_t nplain;             // tiles of unsynchronized tensors
    const int32_t* tile_range;  // 2K entries: tiles of tensor k are [tile_range[2k], tile_range[2k+1])
    const int64_t* numel;       // K entries
    float2* partials;           // W x ntiles compensated (hi, lo) sums of |c| (L1 mode)
    float* m1;                  // W x K (L1 mode)
    float* inv;                 // W x K: RN(qmax / M1), 0 where M1 == 0 (L1 mode)
    int* status;                // device status word: non-zero after a bounded wait gave up
    uint32_t first_wait_polls;  // fault injection: >0 caps the staged reduce's first wait at this
                                // many non-blocking polls (0: the normal bounded wait)
    // data-parallel exchange across ranks (lioncub_dist_*); all 0 otherwise
    int64_t chunk;        // sign mode: elements of each rank's chunk (a multiple of 4096); the
                          // compress pass then writes its wire words chunk-major (row c*W + i)
    int64_t chunk_words;  // words per worker and chunk in that layout
    float* sync_buf;      // new momenta of synchronized tiles, worker-major, sync_slots each:
                          // written by the compress pass, read (all ranks' workers) by the apply
    int64_t sync_slots;   // elements per worker in the sync buffers (synchronized tiles x 2048)
    int64_t qinf_step;    // the step index t (lioncub_diagnose_qinf's random counters)
    int W;
    int K;
    int nbits;
    float beta1, omega1, beta2, omega2, lr, wd, qmax;
    uint32_t zero_bit;  // the bit an exact zero is sent as: 1 on even steps, 0 on odd
    int sync_now;       // 1 when flagged tensors average their momentum this step
    int average;        // 1: u = agg / W (D-Lion Avg)
    float tie_u;        // u for agg == 0: 0, or the step's zero sign
};

// Bounds-checked builds (-DLIONCUB_BOUNDS_CHECK): every global index a kernel
// computes is validated before use; a violation sets bit 1 of the status word
// and the access is skipped (the thread keeps taking part in shuffles and
// barriers, so nothing traps or hangs).  Ordinary builds compile the checks
// away.
#ifdef LIONCUB_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif
constexpr int kStatusWaitTimeout = 1;
constexpr int kStatusOutOfBounds = 2;

#ifdef __CUDACC__
// True when an access may proceed; records a violation in checked builds.
__device__ __forceinline__ bool in_bounds(const StepArgs& a, bool ok)
{
    if constexpr (kBoundsCheck) {
        if (!ok && a.status)
            atomicOr(a.status, kStatusOutOfBounds);
        return ok;
    }
    return true;
}
#endif

// Kernel launchers (return the launch status).
cudaError_t launch_compress(const StepArgs& a, int grad_dtype, int l1_mode, cudaStream_t s);
cudaError_t launch_m1_partial(const StepArgs& a, int grad_dtype, cudaStream_t s);
cudaError_t launch_m1_finalize(const StepArgs& a, cudaStream_t s);
cudaError_t launch_reduce_apply(const StepArgs& a, int l1_mode, cudaStream_t s);
cudaError_t launch_export_agg(const StepArgs& a, int l1_mode, int32_t* agg, cudaStream_t s);
cudaError_t launch_diagnose(const StepArgs& a, int grad_dtype, int l1_mode, lioncub_diag* out, cudaStream_t s);
cudaError_t launch_diagnose_qinf(const StepArgs& a, int grad_dtype, int nbits, float* maxabs, uint64_t seed,
                                 lioncub_qinf_diag* out, cudaStream_t s);

// data-parallel exchange (dist.cu)
cudaError_t launch_compress_dist(const StepArgs& a, int grad_dtype, int l1_mode, cudaStream_t s);
cudaError_t launch_owner_reduce(const StepArgs& a, int dir_bits, void* dir, cudaStream_t s);
cudaError_t launch_code_sum_local(const StepArgs& a, int agg_bytes, void* agg, cudaStream_t s);
cudaError_t launch_apply_dir(const StepArgs& a, int dir_bits, const void* dir, cudaStream_t s);
cudaError_t launch_apply_agg(const StepArgs& a, int agg_bytes, const void* agg, cudaStream_t s);
cudaError_t launch_sync_mean(const StepArgs& a, int W_global, const float* recv, cudaStream_t s);

}  // namespace lc
