// aggregate.cuh -- the W-way aggregation of wire words and the parameter
// update, shared by the single-GPU reduce and the data-parallel exchange.
//
// "Lion Cub: Minimizing Communication Overhead in Distributed Lion", "What
// carries the argument": a quantized sum of the workers' update vectors
// followed by a global sign; "Communication Efficient Distributed Training
// with Distributed Lion", "Approach": the majority vote and the average.
// Sign mode counts set bits per element with byte-lane counters -- each
// nibble is spread to four byte lanes by one multiply (bit j of the nibble
// lands on bit 8j), so one 32-bit add counts four elements at once (exact
// for W <= 255); L1 mode sign-extends each n-bit field.
#pragma once

#include "device_common.cuh"

namespace lc {

// Per-element aggregates of 8 consecutive elements starting at e0.  For
// codes the workers are taken 8 at a time: the 8 loads are issued before any
// of them is used, so each thread keeps 8 independent requests in flight.
constexpr int kBatch = 8;

template <int NB>
struct WireChunk;  // the bits of 8 elements of one worker
template <>
struct WireChunk<1> { using T = uint8_t; };
template <>
struct WireChunk<2> { using T = uint16_t; };
template <>
struct WireChunk<4> { using T = uint32_t; };
template <>
struct WireChunk<8> { using T = uint2; };

template <int NB>
__device__ __forceinline__ void accumulate(int* agg, uint32_t& lo, uint32_t& hi, typename WireChunk<NB>::T v)
{
    if constexpr (NB == 1) {
        const uint32_t b = v;
        lo += ((b & 0xfu) * 0x204081u) & 0x01010101u;
        hi += ((b >> 4) * 0x204081u) & 0x01010101u;
    } else if constexpr (NB == 2) {
        const uint32_t h = v;
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            agg[j] += static_cast<int32_t>(h << (30 - 2 * j)) >> 30;
    } else if constexpr (NB == 4) {
        const uint32_t w = v;
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            agg[j] += static_cast<int32_t>(w << (28 - 4 * j)) >> 28;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            agg[j] += static_cast<int32_t>(v.x << (24 - 8 * j)) >> 24;
            agg[j + 4] += static_cast<int32_t>(v.y << (24 - 8 * j)) >> 24;
        }
    }
}

template <int NB>
__device__ __forceinline__ void aggregate8(const StepArgs& a, int64_t e0, int* agg)
{
    using T = typename WireChunk<NB>::T;
    // worker i's chunk for element group e0 is chunk e0/8 of its words
    const T* base = reinterpret_cast<const T*>(a.wire) + (e0 >> 3);
    const int64_t stride = a.wire_stride * 4 / static_cast<int64_t>(sizeof(T));
#pragma unroll
    for (int j = 0; j < kVec; ++j)
        agg[j] = 0;
    uint32_t lo = 0, hi = 0;  // byte-lane vote counters (sign mode)
    if constexpr (NB == 1) {
        // one byte per worker: a plain loop measured faster than batching
        for (int i = 0; i < a.W; ++i)
            accumulate<NB>(agg, lo, hi, base[static_cast<int64_t>(i) * stride]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            agg[j] = 2 * static_cast<int>((lo >> (8 * j)) & 0xffu) - a.W;
            agg[j + 4] = 2 * static_cast<int>((hi >> (8 * j)) & 0xffu) - a.W;
        }
    } else {
        for (int i0 = 0; i0 < a.W; i0 += kBatch) {
            T v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (i0 + u < a.W)
                    v[u] = base[static_cast<int64_t>(i0 + u) * stride];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (i0 + u < a.W)
                    accumulate<NB>(agg, lo, hi, v[u]);
        }
    }
}

// D-Lion average: u = RN(agg / W).  A vote sum takes only the 2W + 1 values
// -W..W, so each block tabulates the quotients once (one division per entry)
// instead of dividing per element, which made the average's reduce
// compute-bound.
constexpr int kAvgTab = 2 * LIONCUB_MAX_WORKERS + 1;

__device__ __forceinline__ void fill_avg_table(const StepArgs& a, float* tab)
{
    if (a.average)
        for (int k = threadIdx.x; k <= 2 * a.W; k += blockDim.x)
            tab[k] = __fdiv_rn(static_cast<float>(k - a.W), static_cast<float>(a.W));
}

// Update direction u from the aggregate: the global sign (a tie gives tie_u),
// or agg / W for the D-Lion average (from the block's table).
__device__ __forceinline__ float direction(const StepArgs& a, int agg, const float* avg_tab)
{
    if (a.average) {
        const int k = agg + a.W;
        return in_bounds(a, k >= 0 && k <= 2 * a.W) ? avg_tab[k] : 0.0f;
    }
    return agg > 0 ? 1.0f : (agg < 0 ? -1.0f : a.tie_u);
}

// theta' = theta - lr * (u + wd * theta)
__device__ __forceinline__ float lion_apply(float theta, float u, float lr, float wd)
{
    return __fsub_rn(theta, __fmul_rn(lr, __fadd_rn(u, __fmul_rn(wd, theta))));
}

}  // namespace lc
