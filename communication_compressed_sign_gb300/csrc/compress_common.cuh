// compress_common.cuh -- the per-worker compression of 8 elements: the wire
// field of each update vector (a 0/1 sign with the alternating-zero rule, or
// the Eq. (1) L1 code), its packing into wire words, and the new momentum.
// Shared by the single-GPU compress pass and the data-parallel exchange's.
//
// "Lion Cub: Minimizing Communication Overhead in Distributed Lion", "What
// carries the argument": the update vector c, signs sent as 0/1 with exact
// zeros sent as +1/-1 on alternating iterations, and Eq. (1).
#pragma once

#include "device_common.cuh"

namespace lc {

// Sign bit of the transmitted update: 1 = +1, 0 = -1, exact zero = zero_bit.
__device__ __forceinline__ uint32_t sign_bit(float c, uint32_t zero_bit)
{
    return c > 0.0f ? 1u : (c < 0.0f ? 0u : zero_bit);
}

// Eq. (1) code of c with the per-(worker, tensor) scale inv = RN(qmax / M1):
// y = RN(c * inv), rounded to the nearest integer with ties to even and
// clamped to [-qmax, qmax].  The conversion instruction rounds half to even,
// turns NaN into 0 and saturates out-of-range values, so clamping the integer
// equals clamping rint(y); inv == 0 (M1 == 0) gives y = 0 and code 0.
__device__ __forceinline__ int q1_code(float c, float inv, int qmax)
{
    const int r = __float2int_rn(__fmul_rn(c, inv));
    return min(max(r, -qmax), qmax);
}

// Write this thread's 8*NB wire bits (in `bits`, low bits first) of the tile
// element group starting at e0 into the worker's wire words.  Streaming
// (evict-first) stores: at these sizes the wire does not stay in L2 until the
// reduce reads it anyway, and keeping it out of L2's way measured 2.7-3.1 %
// faster for the L1 codes (0.6 % for 1-bit signs) than cache-global stores.
template <int NB>
__device__ __forceinline__ void store_wire(uint32_t* wire_i, int64_t e0, int valid, uint64_t bits)
{
    const int lane = threadIdx.x & 31;
    if constexpr (NB == 1) {
        const uint32_t b = static_cast<uint32_t>(bits);
        const uint32_t w = b | (__shfl_down_sync(0xffffffffu, b, 1) << 8) |
                           (__shfl_down_sync(0xffffffffu, b, 2) << 16) |
                           (__shfl_down_sync(0xffffffffu, b, 3) << 24);
        if ((lane & 3) == 0 && valid > 0)
            __stcs(wire_i + (e0 >> 5), w);
    } else if constexpr (NB == 2) {
        const uint32_t h = static_cast<uint32_t>(bits);
        const uint32_t w = h | (__shfl_down_sync(0xffffffffu, h, 1) << 16);
        if ((lane & 1) == 0 && valid > 0)
            __stcs(wire_i + (e0 >> 4), w);
    } else if constexpr (NB == 4) {
        if (valid > 0)
            __stcs(wire_i + (e0 >> 3), static_cast<uint32_t>(bits));
    } else {
        if (valid > 0)
            __stcs(reinterpret_cast<uint2*>(wire_i + (e0 >> 2)),
                   make_uint2(static_cast<uint32_t>(bits), static_cast<uint32_t>(bits >> 32)));
    }
}

// Per-element work of one worker on 8 elements: the wire bits of c and the
// new momentum (left in m).
template <int NB>
__device__ __forceinline__ uint64_t compress8(const StepArgs& a, const float* g, float* m, int valid, float inv)
{
    const uint64_t fmask = (NB == 8) ? 0xffull : ((1ull << NB) - 1ull);
    const int qmax_i = (1 << (NB - 1)) - 1;
    uint64_t bits = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const float c = update_vector(m[j], g[j], a.beta1, a.omega1);
        uint64_t field;
        if constexpr (NB == 1)
            field = sign_bit(c, a.zero_bit);
        else
            field = static_cast<uint64_t>(static_cast<uint32_t>(q1_code(c, inv, qmax_i))) & fmask;
        if (j < valid)
            bits |= field << (NB * j);
        m[j] = momentum(m[j], g[j], a.beta2, a.omega2);
    }
    return bits;
}

// Checked builds: the element group and its wire words lie inside the
// buffers; otherwise the group is treated as empty.
template <int NB>
__device__ __forceinline__ int checked_valid(const StepArgs& a, int64_t e0, int valid)
{
    if (valid > 0 && !in_bounds(a, e0 >= 0 && e0 + valid <= a.d &&
                                        (e0 * NB) / 32 + (kVec * NB + 31) / 32 <= a.wire_stride))
        return 0;
    return valid;
}

}  // namespace lc
