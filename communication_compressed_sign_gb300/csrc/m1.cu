// m1.cu -- per-(worker, tensor) mean absolute value M1 of the update vector
// for the L1 quantizer of Eq. (1) ("Lion Cub: Minimizing Communication
// Overhead in Distributed Lion", "What carries the argument": M1 is the mean
// absolute value).
//
// Pass 1 (k_m1_partial): one block of 128 threads per tile; for each worker
// in turn it sums |c| of the tile's 2048 elements -- 16 per thread, two
// groups of 8 at a stride of 1024 so that every load instruction is
// coalesced -- with a compensated fp32 accumulator (a hi/lo pair carrying
// ~48 significant bits; TwoSum per element), reduced over the warp with
// shuffles and over the 4 warps in a fixed order, and stores the (hi, lo)
// pair.  The pass is close to issue-bound, and the warp reduction costs as
// much per thread as the accumulation of 8 elements: with 16 elements per
// thread it measured 4.4-5.0 % faster than 256 threads of 8 (GPT-2 medium,
// the 1.3B layout), with the same M1 on every tensor.  Looping over the
// workers inside the block amortizes the block's start-up and its serial
// final merge over W tiles' worth of data; layouts with few tiles take one
// block per (tile, worker) instead, which computes the same pairs.
// GB300 runs fp64 at a small fraction of its fp32 rate, so a per-element fp64
// add would cap this pass below memory speed; the pair keeps the per-tile sum
// accurate to far below one fp32 ulp of the mean.
//
// Pass 2 (k_m1_finalize): one block per (worker, tensor).  Thread t merges
// the pairs of tiles t, t+256, ... in order into its own compensated fp32
// pair, converts it to fp64 once, and the block combines the threads in fp64
// -- a fixed xor-butterfly per warp, then the warps in order -- divides by
// numel in fp64, rounds once to fp32, and stores M1 and the scale
// inv = RN(qmax / M1) (0 when M1 == 0).  Converting and adding every tile's
// pair in fp64 instead kept the narrow fp64 pipe of the SMs holding the
// largest tensors 71 % busy and made those blocks the long pole.
//
// Both passes have fixed tilings and fixed reduction orders, so M1 is
// bit-for-bit deterministic from run to run.
#include "device_common.cuh"

namespace lc {
namespace {

// Threads of an M1 block and the element groups of 8 each thread takes.
constexpr int kM1Threads = 128;
constexpr int kM1Groups = kTile / (kM1Threads * kVec);

// Elements of group q of this thread in the tile (0..8), and its first index.
__device__ __forceinline__ int tile_group(const StepArgs& a, const Tile& tl, int q, int64_t& e0)
{
    e0 = tl.start + static_cast<int64_t>(q) * kM1Threads * kVec + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d))
        valid = 0;
    return valid;
}

// Compensated sum of |c| over worker i's part of tile `tix`: per thread in
// element order (group 0, then group 1), a fixed xor-butterfly per warp, then
// thread 0 merges the 4 warps in order (after the barrier) and stores the
// pair.  `slot` holds the warp sums; every thread of the block takes part.
template <typename GT>
__device__ __forceinline__ void tile_partial(const StepArgs& a, int i, int64_t tix, const Tile& tl, float2* slot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int q = 0; q < kM1Groups; ++q) {
        int64_t e0;
        const int valid = tile_group(a, tl, q, e0);
        if (valid > 0) {
            float g[kVec], m[kVec];
            load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                if (j < valid)
                    cacc_add(hi, lo, fabsf(update_vector(m[j], g[j], a.beta1, a.omega1)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
        const float olo = __shfl_xor_sync(0xffffffffu, lo, off);
        cacc_merge(hi, lo, ohi, olo);
    }
    if (lane == 0)
        slot[warp] = make_float2(hi, lo);
    __syncthreads();
    if (threadIdx.x == 0) {
        float h = slot[0].x, l = slot[0].y;
        for (int w = 1; w < kM1Threads / 32; ++w)
            cacc_merge(h, l, slot[w].x, slot[w].y);
        a.partials[static_cast<int64_t>(i) * a.ntiles + tix] = make_float2(h, l);
    }
}

template <typename GT>
__global__ void __launch_bounds__(kM1Threads) k_m1_partial(const StepArgs a)
{
    // Two slots alternate between consecutive workers, so one barrier per
    // worker suffices: thread 0 has read slot (i & 1) before it reaches the
    // barrier of worker i + 1, and slot (i & 1) is rewritten only at i + 2.
    __shared__ float2 red[2][kM1Threads / 32];
    const Tile tl = in_bounds(a, blockIdx.x < a.ntiles) ? a.tiles[blockIdx.x] : Tile{0, 0, 0u};
    for (int i = 0; i < a.W; ++i)
        tile_partial<GT>(a, i, blockIdx.x, tl, red[i & 1]);
}

// Small layouts (fewer tiles than a few waves of blocks): one block per
// (tile, worker) instead, so the grid still fills the SMs.  Each block runs
// exactly one iteration of the loop above, so the partials are bit-identical.
template <typename GT>
__global__ void __launch_bounds__(kM1Threads) k_m1_partial_tw(const StepArgs a)
{
    __shared__ float2 red[kM1Threads / 32];
    const Tile tl = in_bounds(a, blockIdx.x < a.ntiles) ? a.tiles[blockIdx.x] : Tile{0, 0, 0u};
    tile_partial<GT>(a, blockIdx.y, blockIdx.x, tl, red);
}

// One block per (worker, tensor): thread t merges tiles t, t + 256, ... of
// the tensor (compensated fp32), then fp64: a fixed xor-butterfly per warp
// and the 8 warp sums in order.
constexpr int kFinalThreads = 256;

__global__ void __launch_bounds__(kFinalThreads) k_m1_finalize(const StepArgs a)
{
    __shared__ double red[kFinalThreads / 32];
    const int i = blockIdx.x / a.K, k = blockIdx.x % a.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int t0 = a.tile_range[2 * k], t1 = a.tile_range[2 * k + 1];
    if (!in_bounds(a, i < a.W && 0 <= t0 && t0 <= t1 && t1 <= a.ntiles))
        t0 = t1 = 0;
    const float2* p = a.partials + static_cast<int64_t>(i) * a.ntiles;
    float hi = 0.0f, lo = 0.0f;
    for (int64_t t = t0 + static_cast<int64_t>(threadIdx.x); t < t1; t += kFinalThreads) {
        const float2 v = p[t];
        cacc_merge(hi, lo, v.x, v.y);
    }
    double s = __dadd_rn(static_cast<double>(hi), static_cast<double>(lo));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    if (lane == 0)
        red[warp] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = red[0];
        for (int w = 1; w < kFinalThreads / 32; ++w)
            tot = __dadd_rn(tot, red[w]);
        const int64_t n = a.numel[k];
        const float m1 = n > 0 ? __double2float_rn(__ddiv_rn(tot, static_cast<double>(n))) : 0.0f;
        a.m1[blockIdx.x] = m1;
        a.inv[blockIdx.x] = m1 == 0.0f ? 0.0f : __fdiv_rn(a.qmax, m1);
    }
}

}  // namespace

// Below this many tiles the worker-loop grid would be a few waves at most.
constexpr int64_t kSmallLayoutTiles = 8192;

cudaError_t launch_m1_partial(const StepArgs& a, int grad_dtype, cudaStream_t s)
{
    if (a.ntiles == 0)
        return cudaSuccess;
    const dim3 block(kM1Threads);
    if (a.ntiles < kSmallLayoutTiles) {
        const dim3 grid(static_cast<unsigned>(a.ntiles), static_cast<unsigned>(a.W));
        if (grad_dtype == LIONCUB_GRAD_BF16)
            k_m1_partial_tw<__nv_bfloat16><<<grid, block, 0, s>>>(a);
        else
            k_m1_partial_tw<float><<<grid, block, 0, s>>>(a);
        return cudaGetLastError();
    }
    const dim3 grid(static_cast<unsigned>(a.ntiles));
    if (grad_dtype == LIONCUB_GRAD_BF16)
        k_m1_partial<__nv_bfloat16><<<grid, block, 0, s>>>(a);
    else
        k_m1_partial<float><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_m1_finalize(const StepArgs& a, cudaStream_t s)
{
    const int64_t blocks = static_cast<int64_t>(a.W) * a.K;
    if (blocks == 0)
        return cudaSuccess;
    k_m1_finalize<<<static_cast<unsigned>(blocks), kFinalThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace lc
