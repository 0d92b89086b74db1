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
// One block per tile (with sign votes: resident blocks that loop over the
// tiles); each thread takes 8 elements and loops over the workers,
// software-pipelined on full groups (a second loop re-reads the momenta for
// the variance; the first loop reads them with the default cache policy so
// that the second finds them in L2).  The pass sits near the instruction-issue
// limit, so the per-element work outside the worker loops is kept small:
// counts packed into two words and summed by warp reductions, the maximum
// taken over sums of squares before the one division and square root of a
// block.  Per-tensor totals are combined with integer atomics (exact,
// order-free) and the maximum with an integer atomicMax on the non-negative
// float's bits.
#include "device_common.cuh"

namespace lc {
namespace {

// One worker's contribution to the aggregate of one element.
//  NB == 1: 1 when the wire bit is set (c > 0, or c an exact zero -- or NaN,
//           which compares like zero -- on a step whose zero bit is ZB), else
//           0: the caller turns the count of set bits into 2 * count - W.
//  NB == 2: the code clamp(RN(c * inv), -1, 1): with ties to even it is 1
//           exactly when RN(c * inv) > 0.5 and -1 exactly when it is < -0.5
//           (NaN gives 0).
//  NB >= 4: the code, nearest with ties to even, NaN 0, clamped to qmax.
template <int NB, bool ZB>
__device__ __forceinline__ int wire_value(float c, float inv, int q)
{
    if constexpr (NB == 1) {
        return ZB ? (c < 0.0f ? 0 : 1) : (c > 0.0f ? 1 : 0);
    } else if constexpr (NB == 2) {
        const float x = __fmul_rn(c, inv);
        return (x > 0.5f ? 1 : 0) - (x < -0.5f ? 1 : 0);
    } else {
        const int r = __float2int_rn(__fmul_rn(c, inv));
        return min(max(r, -q), q);
    }
}

__device__ __forceinline__ float sgn(float x)
{
    return x > 0.0f ? 1.0f : (x < 0.0f ? -1.0f : 0.0f);
}

// Per-thread category counts packed into two words, 10 bits a field: a
// thread holds at most kVec = 8 of each and a warp 256, so the warp sums
// (one redux each) cannot carry into the next field.
struct Counts {
    uint32_t w0 = 0;  // match | flip << 10 | dropped << 20
    uint32_t w1 = 0;  // spurious | ties << 10
    __device__ __forceinline__ void add(float uq, float uf, bool tie)
    {
        if (uq == uf)
            w0 += 1u;
        else if (uq != 0.0f && uf != 0.0f)
            w0 += 1u << 10;
        else if (uq == 0.0f)
            w0 += 1u << 20;
        else
            w1 += 1u;
        w1 += tie ? (1u << 10) : 0u;
    }
    __device__ __forceinline__ uint32_t field(int c) const
    {
        return c < 3 ? (w0 >> (10 * c)) & 1023u : (w1 >> (10 * (c - 3))) & 1023u;
    }
};

// One thread's 8 elements: the running aggregate, the full-precision sum of
// c and of m over the workers (in worker order), then the sum of squared
// deviations from the mean.  The sums start at -0: -0 + x == x for every x,
// so worker 0 needs no special case.
template <int NB, bool ZB>
struct DiagAcc {
    int agg[kVec];
    float s[kVec], ms[kVec], var[kVec];

    __device__ __forceinline__ DiagAcc()
    {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            agg[j] = 0;
            s[j] = ms[j] = -0.0f;
            var[j] = 0.0f;
        }
    }
    // one worker: c, its wire value, the running sums of c and m
    __device__ __forceinline__ void add(const StepArgs& a, float inv, int q, const float* g, const float* m)
    {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float c = update_vector(m[j], g[j], a.beta1, a.omega1);
            agg[j] += wire_value<NB, ZB>(c, inv, q);
            s[j] = __fadd_rn(s[j], c);
            ms[j] = __fadd_rn(ms[j], m[j]);
        }
    }
    // after the last worker: the aggregate, and the mean RN(sum / W); for W a
    // power of two 1/W is exact and the product is the same rounding of the
    // same real number
    __device__ __forceinline__ void finish_first_pass(int W)
    {
        if constexpr (NB == 1) {
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                agg[j] = 2 * agg[j] - W;
        }
        const float fw = static_cast<float>(W);
        const bool pow2 = (W & (W - 1)) == 0;
        const float rw = __frcp_rn(fw);
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            ms[j] = pow2 ? __fmul_rn(ms[j], rw) : __fdiv_rn(ms[j], fw);
    }
    __device__ __forceinline__ void add_var(const float* m)
    {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float dl = __fsub_rn(m[j], ms[j]);
            var[j] = __fadd_rn(var[j], __fmul_rn(dl, dl));
        }
    }
};

// Block totals of the elements whose bit is set in vmask, added into tensor
// k's record.  RN(var / W) and the rounded square root are both
// non-decreasing, so the largest standard deviation is the one of the largest
// sum of squares: the maximum is taken first (fmaxf skips NaN) and the block
// divides and takes the root once.  Every thread of the block calls this.
template <int NB, bool ZB, int T>
__device__ __forceinline__ void diag_block_totals(const StepArgs& a, const DiagAcc<NB, ZB>& acc, uint32_t vmask,
                                                  int k, lioncub_diag* out, uint32_t (*red)[3])
{
    Counts cnt;
    float vmax = 0.0f;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (vmask & (1u << j)) {
            const float uq = acc.agg[j] > 0 ? 1.0f : (acc.agg[j] < 0 ? -1.0f : a.tie_u);
            cnt.add(uq, sgn(acc.s[j]), acc.agg[j] == 0);
            vmax = fmaxf(vmax, acc.var[j]);
        }
    }
    // non-negative floats order like their bit patterns
    const uint32_t w0 = __reduce_add_sync(0xffffffffu, cnt.w0);
    const uint32_t w1 = __reduce_add_sync(0xffffffffu, cnt.w1);
    const uint32_t vm = __reduce_max_sync(0xffffffffu, __float_as_uint(vmax));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        red[warp][0] = w0;
        red[warp][1] = w1;
        red[warp][2] = vm;
    }
    __syncthreads();
    if (threadIdx.x < 5) {
        unsigned long long tot = 0;
        for (int w = 0; w < T / 32; ++w) {
            Counts c;
            c.w0 = red[w][0];
            c.w1 = red[w][1];
            tot += c.field(threadIdx.x);
        }
        unsigned long long* base = reinterpret_cast<unsigned long long*>(&out[k]);
        if (tot)
            atomicAdd(base + threadIdx.x, tot);
    } else if (threadIdx.x == 5) {
        uint32_t m = 0;
        for (int w = 0; w < T / 32; ++w)
            m = max(m, red[w][2]);
        const float sd = __fsqrt_rn(__fdiv_rn(__uint_as_float(m), static_cast<float>(a.W)));
        atomicMax(reinterpret_cast<int*>(&out[k].max_std_m), __float_as_int(sd));
    }
}

// Each thread takes 8 consecutive elements of a tile and loops over the
// workers, software-pipelined on full groups; the variance loop reads the
// momenta again (the first loop leaves them in L2 with the default cache
// policy).  k_diagnose: one block per tile.  k_diagnose_persistent: a grid
// of resident blocks loops over the tiles, and at the start of its variance loop
// a block asks L2 for the gradients and momenta of the first kAheadWorkers
// workers of its next tile, so DRAM stays busy while it finishes the current
// one.  Measured with sign votes: 3.4 % faster with 8 workers (GPT-2 small)
// and 9 % with 16 (GPT-2 medium) than one block per tile; with L1 codes it
// was neutral on GPT-2 medium and 2 % slower on the 1.3B layout, so L1 mode
// keeps one block per tile.  (Asking for 1, 2, 8 or 16 workers, or at the
// start of the tile, measured slower.)  The persistent form also unrolls both
// worker loops by 4: 3.4 % (8 workers) and 2.8 % (16) faster; with L1 codes
// the unrolled loops cost registers and were slower or neutral.
constexpr int kAheadWorkers = 4;

// One tile: the block's counts and spread added into its tensor's record.
// next >= 0: the tile this block takes next, whose first kAheadWorkers
// workers are asked of L2 before the variance loop.
template <typename GT, int NB, bool ZB, int kUnroll>
__device__ __forceinline__ void diag_tile(const StepArgs& a, int64_t tix, int64_t next, lioncub_diag* out,
                                          uint32_t (*red)[3])
{
    const int q = static_cast<int>(a.qmax);
    const Tile tl = in_bounds(a, tix < a.ntiles) ? a.tiles[tix] : Tile{0, 0, 0u};
    const int64_t e0 = tl.start + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = tl.start + tl.len - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d))
        valid = 0;
    int k = static_cast<int>(tl.meta & ~kTileSync);
    if (!in_bounds(a, k < a.K))
        k = 0;

    DiagAcc<NB, ZB> acc;
    if (valid == kVec) {
        // full groups: worker i+1's loads are issued before worker i is used
        // the momenta stay cached for the variance pass below
        Raw8<GT> cur, nxt;
        cur.template load<true>(a.g[0], a.m[0], e0);
#pragma unroll kUnroll
        for (int i = 0; i < a.W; ++i) {
            if (i + 1 < a.W)
                nxt.template load<true>(a.g[i + 1], a.m[i + 1], e0);
            float g[kVec], m[kVec];
            cur.unpack(g, m);
            acc.add(a, (NB > 1) ? a.inv[static_cast<int64_t>(i) * a.K + k] : 0.0f, q, g, m);
            cur = nxt;
        }
    } else if (valid > 0) {
        for (int i = 0; i < a.W; ++i) {
            float g[kVec], m[kVec];
            load_gm<GT>(a.g[i], a.m[i], e0, valid, g, m);
            acc.add(a, (NB > 1) ? a.inv[static_cast<int64_t>(i) * a.K + k] : 0.0f, q, g, m);
        }
    }
    acc.finish_first_pass(a.W);
    if (next >= 0 && next < a.ntiles) {
        const Tile tn = a.tiles[next];
        const int64_t pe = tn.start + static_cast<int64_t>(threadIdx.x) * kVec;
        if (pe + kVec <= tn.start + tn.len) {
            for (int i = 0; i < kAheadWorkers && i < a.W; ++i) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const GT*>(a.g[i]) + pe));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.m[i] + pe));
            }
        }
    }
    if (valid > 0) {
#pragma unroll kUnroll
        for (int i = 0; i < a.W; ++i) {
            float m[kVec];
            load_f32(a.m[i], e0, valid, m);
            acc.add_var(m);
        }
    }
    diag_block_totals<NB, ZB, kThreads>(a, acc, (1u << valid) - 1u, k, out, red);
}

template <typename GT, int NB, bool ZB>
__global__ void __launch_bounds__(kThreads) k_diagnose(const StepArgs a, lioncub_diag* out)
{
    __shared__ uint32_t red[kThreads / 32][3];
    diag_tile<GT, NB, ZB, 1>(a, blockIdx.x, -1, out, red);
}

template <typename GT, int NB, bool ZB>
__global__ void __launch_bounds__(kThreads, 4) k_diagnose_persistent(const StepArgs a, lioncub_diag* out)
{
    __shared__ uint32_t red[kThreads / 32][3];
    for (int64_t tix = blockIdx.x; tix < a.ntiles; tix += gridDim.x) {
        diag_tile<GT, NB, ZB, 4>(a, tix, tix + gridDim.x, out, red);
        __syncthreads();  // red is written again for the next tile
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
        s[j] = -0.0f;  // -0 + x == x: worker 0 needs no special case
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
                s[j] = __fadd_rn(s[j], c);
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
        cnt[c] = __reduce_add_sync(0xffffffffu, cnt[c]);
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

template <typename GT, int NB, bool ZB>
cudaError_t launch_nb(const StepArgs& a, lioncub_diag* out, cudaStream_t s)
{
    // sign votes of bf16 gradients: the persistent form (fp32 gradients would
    // spill under its 64-register cap)
    if constexpr (NB == 1 && sizeof(GT) == 2) {
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_diagnose_persistent<GT, NB, ZB>, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        const int64_t resident = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
        const int64_t grid = a.ntiles < resident ? a.ntiles : resident;
        k_diagnose_persistent<GT, NB, ZB><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a, out);
    } else {
        k_diagnose<GT, NB, ZB><<<static_cast<unsigned>(a.ntiles), kThreads, 0, s>>>(a, out);
    }
    return cudaGetLastError();
}

template <typename GT>
cudaError_t launch_typed(const StepArgs& a, int nb, lioncub_diag* out, cudaStream_t s)
{
    switch (nb) {
    case 1: return a.zero_bit ? launch_nb<GT, 1, true>(a, out, s) : launch_nb<GT, 1, false>(a, out, s);
    case 2: return launch_nb<GT, 2, false>(a, out, s);
    case 4: return launch_nb<GT, 4, false>(a, out, s);
    case 8: return launch_nb<GT, 8, false>(a, out, s);
    default: return cudaErrorInvalidValue;
    }
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
