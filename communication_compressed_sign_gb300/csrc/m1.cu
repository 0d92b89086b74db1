// m1.cu -- per-(worker, tensor) mean absolute value M1 of the update vector
// for the L1 quantizer of Eq. (1) ("Lion Cub: Minimizing Communication
// Overhead in Distributed Lion", "What carries the argument": M1 is the mean
// absolute value).
//
// One kernel, k_m1, one block per tile: for each worker in turn the block
// sums |c| of the tile's 2048 elements with a compensated fp32 accumulator (a
// hi/lo pair carrying ~48 significant bits; TwoSum per element), reduced over
// the warp with shuffles and over the 8 warps in a fixed order, and stores
// the (hi, lo) pair as the tile's partial.  GB300 runs fp64 at a small
// fraction of its fp32 rate, so a per-element fp64 add would cap this pass
// below memory speed; the pair keeps the per-tile sum accurate to far below
// one fp32 ulp of the mean.
//
// Each (worker, tensor) has a counter.  The block whose partial completes a
// tensor's count sums that tensor's tile partials in fp64 -- thread t takes
// tiles t, t+256, ... in order, then a fixed xor-butterfly per warp and the
// warps in order -- divides by numel in fp64, rounds once to fp32, stores M1
// and the scale inv = RN(qmax / M1) (0 when M1 == 0), and resets the counter.
// The combine order depends only on tile indices, never on which block
// finishes last, so M1 is bit-for-bit deterministic.
//
// The step runs this pass over a chunk of whole tensors at a time, right
// before the compress pass of the same chunk; its loads keep normal L2
// priority so that the compress pass finds the chunk's gradients and momenta
// in L2 instead of reading them from memory a second time.
#include "device_common.cuh"

namespace lc {
namespace {

// 8 gradients and 8 momenta with ordinary (L2-keeping) loads.
template <bool BF16>
__device__ __forceinline__ void load_keep(const void* g, const float* m, int64_t e0, int valid, float* gv,
                                          float* mv)
{
    if (valid == kVec) {
        if constexpr (BF16) {
            const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(g) + e0);
            gv[0] = bf16_bits_lo(v.x); gv[1] = bf16_bits_hi(v.x);
            gv[2] = bf16_bits_lo(v.y); gv[3] = bf16_bits_hi(v.y);
            gv[4] = bf16_bits_lo(v.z); gv[5] = bf16_bits_hi(v.z);
            gv[6] = bf16_bits_lo(v.w); gv[7] = bf16_bits_hi(v.w);
        } else {
            const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(g) + e0);
            const float4 a = p[0], b = p[1];
            gv[0] = a.x; gv[1] = a.y; gv[2] = a.z; gv[3] = a.w;
            gv[4] = b.x; gv[5] = b.y; gv[6] = b.z; gv[7] = b.w;
        }
        const float4* q = reinterpret_cast<const float4*>(m + e0);
        const float4 a = q[0], b = q[1];
        mv[0] = a.x; mv[1] = a.y; mv[2] = a.z; mv[3] = a.w;
        mv[4] = b.x; mv[5] = b.y; mv[6] = b.z; mv[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            if constexpr (BF16)
                gv[j] = (j < valid)
                            ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(g)[e0 + j]) << 16)
                            : 0.0f;
            else
                gv[j] = (j < valid) ? static_cast<const float*>(g)[e0 + j] : 0.0f;
            mv[j] = (j < valid) ? m[e0 + j] : 0.0f;
        }
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) k_m1(const StepArgs a, int64_t tile0)
{
    // Two slots alternate between consecutive workers, so one barrier per
    // worker suffices: thread 0 has read slot (i & 1) before it reaches the
    // next barrier, and slot (i & 1) is rewritten only two workers later.
    __shared__ float2 red[2][kThreads / 32];
    __shared__ double fred[kThreads / 32];
    __shared__ int last;
    const int64_t tile = tile0 + blockIdx.x;
    const Tile tl = a.tiles[tile];
    const int k = static_cast<int>(tl.meta & ~kTileSync);
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    const int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = a.tile_range[2 * k], t1 = a.tile_range[2 * k + 1];

    for (int i = 0; i < a.W; ++i) {
        float hi = 0.0f, lo = 0.0f;
        if (valid > 0) {
            float g[kVec], m[kVec];
            load_keep<BF16>(a.g[i], a.m[i], e0, valid, g, m);
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                if (j < valid)
                    cacc_add(hi, lo, fabsf(update_vector(m[j], g[j], a.beta1, a.omega1)));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
            const float olo = __shfl_xor_sync(0xffffffffu, lo, off);
            cacc_merge(hi, lo, ohi, olo);
        }
        float2* slot = red[i & 1];
        if (lane == 0)
            slot[warp] = make_float2(hi, lo);
        __syncthreads();
        const int64_t wk = static_cast<int64_t>(i) * a.K + k;
        if (threadIdx.x == 0) {
            float h = slot[0].x, l = slot[0].y;
            for (int w = 1; w < kThreads / 32; ++w)
                cacc_merge(h, l, slot[w].x, slot[w].y);
            a.partials[static_cast<int64_t>(i) * a.ntiles + tile] = make_float2(h, l);
            // publish the partial, then count it; the block that brings the
            // count to the tensor's tile count combines the tensor's partials
            __threadfence();
            const unsigned done = atomicAdd(&a.m1_count[wk], 1u) + 1u;
            last = (done == static_cast<unsigned>(t1 - t0)) ? 1 : 0;
        }
        __syncthreads();
        if (last) {  // block-uniform
            __threadfence();
            const float2* p = a.partials + static_cast<int64_t>(i) * a.ntiles;
            double s = 0.0;
            for (int t = t0 + threadIdx.x; t < t1; t += kThreads) {
                const float2 v = __ldcg(p + t);
                s = __dadd_rn(s, __dadd_rn(static_cast<double>(v.x), static_cast<double>(v.y)));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
            if (lane == 0)
                fred[warp] = s;
            __syncthreads();
            if (threadIdx.x == 0) {
                double tot = fred[0];
                for (int w = 1; w < kThreads / 32; ++w)
                    tot = __dadd_rn(tot, fred[w]);
                const int64_t n = a.numel[k];
                const float m1 = n > 0 ? __double2float_rn(__ddiv_rn(tot, static_cast<double>(n))) : 0.0f;
                a.m1[wk] = m1;
                a.inv[wk] = m1 == 0.0f ? 0.0f : __fdiv_rn(a.qmax, m1);
                a.m1_count[wk] = 0u;  // ready for the next step
            }
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t launch_m1(const StepArgs& a, int grad_dtype, int64_t tile0, int64_t ntiles, cudaStream_t s)
{
    if (ntiles <= 0)
        return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(ntiles)), block(kThreads);
    if (grad_dtype == LIONCUB_GRAD_BF16)
        k_m1<true><<<grid, block, 0, s>>>(a, tile0);
    else
        k_m1<false><<<grid, block, 0, s>>>(a, tile0);
    return cudaGetLastError();
}

}  // namespace lc
