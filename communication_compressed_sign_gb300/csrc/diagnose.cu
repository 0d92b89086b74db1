// diagnose.cu -- the pages' own measurements of a compressed step, computed
// from the state before the step and the step's gradients (nothing updated).
//
// "Lion Cub: Minimizing Communication Overhead in Distributed Lion":
//   Fig. 4 / Fig. 11 captions -- whether the sign of the quantized update
//   matches or flips against the full-precision update;
//   Fig. 6 caption -- the maximum, over a layer's elements, of the standard
//   deviation of the momentum between workers;
//   quoted body text -- the share of parameters whose majority vote is tied.
//
// Per element: u_q is the sign of the direction the step would apply (the
// global sign of the vote or code sum, with the tie rule); u_fp is the sign
// of s = c_0 + c_1 + ... + c_{W-1} in fp32, worker order.  Categories: match
// (u_q == u_fp), flip (u_q == -u_fp != 0), dropped (u_q == 0 != u_fp),
// spurious (u_fp == 0 != u_q); ties counts aggregates equal to 0.  The
// momentum spread is mean = (sum m_i) / W, var = (sum (m_i - mean)^2) / W,
// std = sqrt(var), all in fp32 with one rounding per operation.
//
// One block per tile; each thread takes 8 elements and loops over the
// workers, software-pipelined on full groups (a second loop re-reads the
// momenta for the variance; the first loop reads them with the default cache
// policy so that the second finds them in L2).  Per-tensor
// totals are combined with integer atomics (exact, order-free) and the
// maximum with an integer atomicMax on the non-negative float's bits.
#include "device_common.cuh"

namespace lc {
namespace {

template <int NB>
__device__ __forceinline__ int wire_value(float c, float inv, float qmax, uint32_t zero_bit)
{
    if constexpr (NB == 1) {
        const uint32_t b = c > 0.0f ? 1u : (c < 0.0f ? 0u : zero_bit);
        return b ? 1 : -1;
    } else {
        // nearest with ties to even; NaN gives 0; saturating, then clamped
        const int r = __float2int_rn(__fmul_rn(c, inv));
        const int q = static_cast<int>(qmax);
        return min(max(r, -q), q);
    }
}

__device__ __forceinline__ float sgn(float x)
{
    return x > 0.0f ? 1.0f : (x < 0.0f ? -1.0f : 0.0f);
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <typename GT, int NB>
__global__ void __launch_bounds__(kThreads) k_diagnose(const StepArgs a, lioncub_diag* out)
{
    __shared__ unsigned long long red[kThreads / 32][5];
    __shared__ float redmax[kThreads / 32];
    const Tile tl = in_bounds(a, blockIdx.x < a.ntiles) ? a.tiles[blockIdx.x] : Tile{0, 0, 0u};
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d))
        valid = 0;
    int k = static_cast<int>(tl.meta & ~kTileSync);
    if (!in_bounds(a, k < a.K))
        k = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    int agg[kVec];
    float s[kVec], ms[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        agg[j] = 0;
        s[j] = ms[j] = 0.0f;
    }
    // per worker: c, its wire value, and the running sums of c and m
    auto accumulate = [&](int i, const float* g, const float* m) {
        const float inv = (NB > 1) ? a.inv[static_cast<int64_t>(i) * a.K + k] : 0.0f;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float c = update_vector(m[j], g[j], a.beta1, a.omega1);
            agg[j] += wire_value<NB>(c, inv, a.qmax, a.zero_bit);
            s[j] = (i == 0) ? c : __fadd_rn(s[j], c);
            ms[j] = (i == 0) ? m[j] : __fadd_rn(ms[j], m[j]);
        }
    };
    if (valid == kVec) {
        // full groups: worker i+1's loads are issued before worker i is used
        // the momenta stay cached for the variance pass below
        Raw8<GT> cur, nxt;
        cur.template load<true>(a.g[0], a.m[0], e0);
        for (int i = 0; i < a.W; ++i) {
            if (i + 1 < a.W)
                nxt.template load<true>(a.g[i + 1], a.m[i + 1], e0);
            float g[kVec], m[kVec];
            cur.unpack(g, m);
            accumulate(i, g, m);
            cur = nxt;
        }
    } else if (valid > 0) {
        for (int i = 0; i < a.W; ++i) {
            float g[kVec], m[kVec];
            load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
            accumulate(i, g, m);
        }
    }
    const float fw = static_cast<float>(a.W);
    float var[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        ms[j] = __fdiv_rn(ms[j], fw);  // mean
        var[j] = 0.0f;
    }
    if (valid > 0) {
        for (int i = 0; i < a.W; ++i) {
            float m[kVec];
            load_f32(a.m[i], e0, valid, m);
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float dl = __fsub_rn(m[j], ms[j]);
                var[j] = __fadd_rn(var[j], __fmul_rn(dl, dl));
            }
        }
    }
    unsigned long long cnt[5] = {0, 0, 0, 0, 0};  // match, flip, dropped, spurious, ties
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (j < valid) {
            const float uq = agg[j] > 0 ? 1.0f : (agg[j] < 0 ? -1.0f : a.tie_u);
            const float uf = sgn(s[j]);
            if (uq == uf)
                cnt[0] += 1;
            else if (uq != 0.0f && uf != 0.0f)
                cnt[1] += 1;
            else if (uq == 0.0f)
                cnt[2] += 1;
            else
                cnt[3] += 1;
            cnt[4] += (agg[j] == 0) ? 1 : 0;
            mx = fmaxf(mx, __fsqrt_rn(__fdiv_rn(var[j], fw)));
        }
    }
#pragma unroll
    for (int c = 0; c < 5; ++c)
        cnt[c] = warp_sum(cnt[c]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) {
#pragma unroll
        for (int c = 0; c < 5; ++c)
            red[warp][c] = cnt[c];
        redmax[warp] = mx;
    }
    __syncthreads();
    if (threadIdx.x < 5) {
        unsigned long long tot = 0;
        for (int w = 0; w < kThreads / 32; ++w)
            tot += red[w][threadIdx.x];
        unsigned long long* base = reinterpret_cast<unsigned long long*>(&out[k]);
        if (tot)
            atomicAdd(base + threadIdx.x, tot);
    } else if (threadIdx.x == 5) {
        float m = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w)
            m = fmaxf(m, redmax[w]);
        atomicMax(reinterpret_cast<int*>(&out[k].max_std_m), __float_as_int(m));
    }
}

// ---- the Q_inf comparator (lioncub_diagnose_qinf) ----------------------------
//
// The max-norm quantizer with stochastic rounding that the pages compare L1
// quantization against ("Lion Cub" page, "Core claim" and the Fig. 4
// caption: on Lion's heavy-tailed update it turns most codes into zeros).
// Per (worker, tensor): M_inf = max |c|; inv = RN(qmax / M_inf) (0 when
// M_inf == 0); per element y = RN(|c| * inv), code = floor(y) + (u < y -
// floor(y)), clamped to qmax, with the sign of c.  u is the top 24 bits of
// SplitMix64 (Steele, Lea and Flood 2014) output number (t mod 2^16) * 2^48 +
// worker * 2^40 + e from the caller's seed, times 2^-24.  The codes are
// summed over the workers in order and the sign of the sum (ties by the
// handle's tie rule) is compared with the full-precision sign.

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t k)
{
    uint64_t z = seed + (k + 1ull) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// max |c| of each (worker, tensor): one block per (tile, worker), an integer
// atomicMax on the bits of the non-negative float (exact, order-free)
template <typename GT>
__global__ void __launch_bounds__(kThreads) k_qinf_maxabs(const StepArgs a, float* maxabs)
{
    __shared__ float red[kThreads / 32];
    const Tile tl = in_bounds(a, blockIdx.x < a.ntiles) ? a.tiles[blockIdx.x] : Tile{0, 0, 0u};
    const int i = blockIdx.y;
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d))
        valid = 0;
    int k = static_cast<int>(tl.meta & ~kTileSync);
    if (!in_bounds(a, k < a.K))
        k = 0;
    float mx = 0.0f;
    if (valid > 0) {
        float g[kVec], m[kVec];
        load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            if (j < valid)
                mx = fmaxf(mx, fabsf(update_vector(m[j], g[j], a.beta1, a.omega1)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w)
            b = fmaxf(b, red[w]);
        if (b > 0.0f)
            atomicMax(reinterpret_cast<int*>(maxabs + static_cast<int64_t>(i) * a.K + k), __float_as_int(b));
    }
}

template <typename GT, int NB>
__global__ void __launch_bounds__(kThreads) k_diagnose_qinf(const StepArgs a, const float* maxabs, uint64_t seed,
                                                            lioncub_qinf_diag* out)
{
    __shared__ unsigned long long red[kThreads / 32][5];
    const Tile tl = in_bounds(a, blockIdx.x < a.ntiles) ? a.tiles[blockIdx.x] : Tile{0, 0, 0u};
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d))
        valid = 0;
    int k = static_cast<int>(tl.meta & ~kTileSync);
    if (!in_bounds(a, k < a.K))
        k = 0;
    constexpr int kQmax = (1 << (NB - 1)) - 1;
    int agg[kVec];
    float s[kVec];
    uint32_t zeros = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        agg[j] = 0;
        s[j] = 0.0f;
    }
    if (valid > 0) {
        for (int i = 0; i < a.W; ++i) {
            float g[kVec], m[kVec];
            load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
            const float mi = maxabs[static_cast<int64_t>(i) * a.K + k];
            const float inv = mi > 0.0f ? __fdiv_rn(static_cast<float>(kQmax), mi) : 0.0f;
            const uint64_t kbase = (static_cast<uint64_t>(a.qinf_step & 0xffff) << 48) |
                                   (static_cast<uint64_t>(i) << 40) | static_cast<uint64_t>(e0);
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float c = update_vector(m[j], g[j], a.beta1, a.omega1);
                const float y = __fmul_rn(fabsf(c), inv);
                const float fl = floorf(y);
                const float frac = __fsub_rn(y, fl);
                const float u = static_cast<float>(static_cast<uint32_t>(splitmix64(seed, kbase + j) >> 40)) *
                                (1.0f / 16777216.0f);
                int v = static_cast<int>(fl) + (u < frac ? 1 : 0);
                v = min(v, kQmax);
                const int q = c < 0.0f ? -v : v;
                if (j < valid) {
                    agg[j] += q;
                    zeros += (q == 0) ? 1u : 0u;
                }
                s[j] = (i == 0) ? c : __fadd_rn(s[j], c);
            }
        }
    }
    uint32_t cnt[5] = {0, 0, 0, 0, zeros};  // match, flip, dropped, spurious, zero codes
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (j < valid) {
            const float uq = agg[j] > 0 ? 1.0f : (agg[j] < 0 ? -1.0f : a.tie_u);
            const float uf = sgn(s[j]);
            if (uq == uf)
                cnt[0] += 1;
            else if (uq != 0.0f && uf != 0.0f)
                cnt[1] += 1;
            else if (uq == 0.0f)
                cnt[2] += 1;
            else
                cnt[3] += 1;
        }
    }
#pragma unroll
    for (int c = 0; c < 5; ++c)
        cnt[c] = warp_sum(cnt[c]);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int c = 0; c < 5; ++c)
            red[warp][c] = cnt[c];
    }
    __syncthreads();
    if (threadIdx.x < 5) {
        unsigned long long tot = 0;
        for (int w = 0; w < kThreads / 32; ++w)
            tot += red[w][threadIdx.x];
        if (tot)
            atomicAdd(reinterpret_cast<unsigned long long*>(&out[k]) + threadIdx.x, tot);
    }
}

template <typename GT>
cudaError_t launch_typed(const StepArgs& a, int nb, lioncub_diag* out, cudaStream_t s)
{
    const unsigned grid = static_cast<unsigned>(a.ntiles);
    switch (nb) {
    case 1: k_diagnose<GT, 1><<<grid, kThreads, 0, s>>>(a, out); break;
    case 2: k_diagnose<GT, 2><<<grid, kThreads, 0, s>>>(a, out); break;
    case 4: k_diagnose<GT, 4><<<grid, kThreads, 0, s>>>(a, out); break;
    case 8: k_diagnose<GT, 8><<<grid, kThreads, 0, s>>>(a, out); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_diagnose(const StepArgs& a, int grad_dtype, int l1_mode, lioncub_diag* out, cudaStream_t s)
{
    if (a.ntiles == 0)
        return cudaSuccess;
    const int nb = l1_mode ? a.nbits : 1;
    if (grad_dtype == LIONCUB_GRAD_BF16)
        return launch_typed<__nv_bfloat16>(a, nb, out, s);
    return launch_typed<float>(a, nb, out, s);
}

}  // namespace lc

namespace lc {
namespace {

template <typename GT>
cudaError_t launch_qinf_typed(const StepArgs& a, int nbits, float* maxabs, uint64_t seed, lioncub_qinf_diag* out,
                              cudaStream_t s)
{
    k_qinf_maxabs<GT><<<dim3(static_cast<unsigned>(a.ntiles), a.W), kThreads, 0, s>>>(a, maxabs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const unsigned grid = static_cast<unsigned>(a.ntiles);
    switch (nbits) {
    case 2: k_diagnose_qinf<GT, 2><<<grid, kThreads, 0, s>>>(a, maxabs, seed, out); break;
    case 4: k_diagnose_qinf<GT, 4><<<grid, kThreads, 0, s>>>(a, maxabs, seed, out); break;
    case 8: k_diagnose_qinf<GT, 8><<<grid, kThreads, 0, s>>>(a, maxabs, seed, out); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_diagnose_qinf(const StepArgs& a, int grad_dtype, int nbits, float* maxabs, uint64_t seed,
                                 lioncub_qinf_diag* out, cudaStream_t s)
{
    if (a.ntiles == 0)
        return cudaSuccess;
    if (grad_dtype == LIONCUB_GRAD_BF16)
        return launch_qinf_typed<__nv_bfloat16>(a, nbits, maxabs, seed, out, s);
    return launch_qinf_typed<float>(a, nbits, maxabs, seed, out, s);
}

}  // namespace lc
