// synth.cu -- seeded, counter-based synthetic inputs for tests and the
// benchmark: gradients, initial parameters.  Holds none of the optimizer's
// arithmetic; the CUDA library and the CPU oracle both consume its output
// (the oracle gets a host copy of the same bits).
//
// Random bits: the SplitMix64 finaliser (Steele, Lea and Flood, 2014)
// applied to a key built from (seed, stream, index, draw), so any element
// can be produced independently.  Uniforms take 24 bits, offset by half a
// step so they lie strictly inside (0, 1).
//
// Distributions:
//   normal    -- Box-Muller transform.
//   student-t -- Bailey's polar method (Math. Comp. 62, 1994): draw (u, v)
//                uniform in the square [-1,1]^2 until w = u^2 + v^2 is in
//                (0, 1], then t = u * sqrt(nu * (w^(-2/nu) - 1) / w).
//                Valid for any real nu > 0.  Up to 32 draws per element.
//   outliers  -- an independent uniform per element; below `frac` the value
//                is multiplied by `mult` (before rounding to bf16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t bits64(uint64_t key, uint64_t index, uint32_t draw)
{
    return mix64(key ^ mix64(index * 64u + draw));
}

// Two uniforms in (0, 1) from one 64-bit draw.
__device__ __forceinline__ void uniform2(uint64_t x, float& a, float& b)
{
    a = (static_cast<float>(x >> 40) + 0.5f) * 5.9604644775390625e-8f;  // 2^-24
    b = (static_cast<float>((x >> 16) & 0xffffffull) + 0.5f) * 5.9604644775390625e-8f;
}

__device__ float sample(int kind, uint64_t key, uint64_t i, float p0, float p1, float p2, float p3)
{
    float a, b;
    if (kind == 0) {  // normal(0, p0)
        uniform2(bits64(key, i, 0), a, b);
        const float r = sqrtf(-2.0f * logf(a));
        return p0 * r * cospif(2.0f * b);
    }
    if (kind == 1) {  // uniform(p0, p1)
        uniform2(bits64(key, i, 0), a, b);
        return p0 + (p1 - p0) * a;
    }
    // kind 2: p1 * student_t(nu = p0), outliers with probability p2 times p3
    float t = 0.0f;
    for (uint32_t draw = 0; draw < 32; ++draw) {
        uniform2(bits64(key, i, draw), a, b);
        const float u = 2.0f * a - 1.0f, v = 2.0f * b - 1.0f;
        const float w = u * u + v * v;
        if (w > 0.0f && w <= 1.0f) {
            t = u * sqrtf(p0 * (powf(w, -2.0f / p0) - 1.0f) / w);
            break;
        }
    }
    float x = p1 * t;
    if (p2 > 0.0f) {
        uniform2(bits64(key, i, 63), a, b);
        if (a < p2)
            x *= p3;
    }
    return x;
}

__global__ void k_fill(void* out, int out_bf16, int64_t n, int kind, uint64_t key, float p0, float p1,
                       float p2, float p3)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float x = sample(kind, key, static_cast<uint64_t>(i), p0, p1, p2, p3);
        if (out_bf16)
            static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(x);
        else
            static_cast<float*>(out)[i] = x;
    }
}

}  // namespace

extern "C" {

// Fill out[0..n) (device; bf16 if out_bf16 else fp32) with samples of
// `kind` (0 normal(0,p0); 1 uniform(p0,p1); 2 p1*student_t(p0) with
// outliers p2/p3) from stream (seed, stream_id).  Returns a cudaError_t.
int synth_fill(void* out, int out_bf16, int64_t n, int kind, uint64_t seed, uint64_t stream_id,
               float p0, float p1, float p2, float p3, void* stream)
{
    if (n <= 0)
        return 0;
    uint64_t key = seed * 0xD1342543DE82EF95ull + 0x2545F4914F6CDD1Dull;
    key ^= stream_id * 0x9E3779B97F4A7C15ull;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 64)
        blocks = 152 * 64;
    k_fill<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        out, out_bf16, n, kind, key, p0, p1, p2, p3);
    return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
