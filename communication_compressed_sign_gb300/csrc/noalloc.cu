// noalloc.cu -- an allocation-free entry point for the sign-mode step.
//
// Some callers cannot call cudaMalloc when they want to run a step: a host
// application whose device memory is all reserved up front by its own
// allocator (so a side allocation can fail or fragment the pool), code that
// must not pay the implicit device synchronization cudaMalloc/cudaFree can
// cause, or a plug-in that is only allowed to allocate while it is being
// initialised.  lioncub_sign_step_noalloc serves them: it runs the same
// sign-mode step as lioncub_step (one flat tensor, majority vote, no
// momentum sync) without a handle, keeping the packed sign words in a
// fixed-size array in the library's own device memory instead of scratch
// allocated per handle.
//
// The array is a file-scope __device__ object of LIONCUB_NOALLOC_MAX_WORDS
// words (16 MiB).  Every GPU on which the library's code for this file is
// loaded holds those 16 MiB until the process exits.  Host code may not use
// the array's name as a device address (it is a host-side stand-in), so the
// first call on each device looks the address up with cudaGetSymbolAddress
// while that device is current and caches it; later calls reuse it.  With
// lazy module loading that first lookup is also what loads this file's
// module and reserves the 16 MiB, so a caller that must not allocate later
// makes one call with d == 0 (and valid pointers) on each device while it is
// initialising: that call does the set-up and launches nothing.
//
// In the bounds-checked build (a debugging aid) the kernels record an index
// outside its buffer, or a bounded wait that gave up, in a second file-scope
// word; each call first reads that word back (synchronously) and fails if a
// previous call's kernels set it.  Ordinary builds pass no status word and
// never read it.
//
// All calls share the one array.  Each call writes every word it later reads
// (the compress kernel writes all ceil(d/32) words of every worker before the
// reduce kernel reads them, padding bits included), so nothing has to be
// cleared between calls; but two calls whose kernels overlap on the GPU --
// on different streams, or from different threads -- race on the array.
#include <cstring>
#include <mutex>

#include "device_common.cuh"

namespace lc {
// Defined in lioncub.cu: the message lioncub_last_error(NULL) returns.
void set_handleless_error(const char* msg);
}  // namespace lc

namespace {

using lc::kThreads;
using lc::kTile;
using lc::kVec;

__device__ __align__(256) uint32_t g_noalloc_wire[LIONCUB_NOALLOC_MAX_WORDS];
// status bits of the bounds-checked build (LIONCUB_STATUS_*); unused otherwise
__device__ int g_noalloc_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_wire_addr[kMaxDevices] = {};
void* g_status_addr[kMaxDevices] = {};

// The sign-mode compression of one flat tensor, one block per (tile,
// worker): tile b covers elements [b*2048, min(d, (b+1)*2048)), so no tile
// table is needed.
template <typename GT>
__global__ void __launch_bounds__(kThreads) k_compress_sign_flat(const lc::StepArgs a)
{
    const int i = blockIdx.y;
    const int64_t e0 = static_cast<int64_t>(blockIdx.x) * kTile + static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t left = a.d - e0;
    int valid = left <= 0 ? 0 : (left >= kVec ? kVec : static_cast<int>(left));
    // checked builds: the group's word lies inside the worker's row
    if (valid > 0 && !lc::in_bounds(a, (e0 >> 5) < a.wire_stride && i < a.W))
        valid = 0;
    const int lane = threadIdx.x & 31;
    float g[kVec], m[kVec];
    if (valid > 0) {
        lc::load_grad<GT>(a.g[i], e0, valid, g);
        lc::load_f32(a.m[i], e0, valid, m);
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            g[j] = m[j] = 0.0f;
    }
    uint32_t bits = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const float c = lc::update_vector(m[j], g[j], a.beta1, a.omega1);
        const uint32_t b = c > 0.0f ? 1u : (c < 0.0f ? 0u : a.zero_bit);
        if (j < valid)
            bits |= b << j;
        m[j] = lc::momentum(m[j], g[j], a.beta2, a.omega2);
    }
    const uint32_t w = bits | (__shfl_down_sync(0xffffffffu, bits, 1) << 8) |
                       (__shfl_down_sync(0xffffffffu, bits, 2) << 16) |
                       (__shfl_down_sync(0xffffffffu, bits, 3) << 24);
    if ((lane & 3) == 0 && valid > 0)
        a.wire[static_cast<int64_t>(i) * a.wire_stride + (e0 >> 5)] = w;
    if (valid > 0)
        lc::store_f32(a.m[i], e0, valid, m);
}

// Device addresses of g_noalloc_wire and g_noalloc_status on the current
// device (looked up once per device, with that device current).
cudaError_t static_addresses(void** wire, int** status)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_wire_addr[dev]) {
        void* p = nullptr;
        void* q = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_wire);
        if (e == cudaSuccess)
            e = cudaGetSymbolAddress(&q, g_noalloc_status);
        if (e != cudaSuccess)
            return e;
        g_status_addr[dev] = q;
        g_wire_addr[dev] = p;
    }
    *wire = g_wire_addr[dev];
    *status = static_cast<int*>(g_status_addr[dev]);
    return cudaSuccess;
}

int fail(int code, const char* msg)
{
    lc::set_handleless_error(msg);
    return code;
}

}  // namespace

extern "C" int lioncub_sign_step_noalloc(int64_t d, int W, float beta1, float beta2, float lr, float wd,
                                         int64_t t, int grad_dtype, const void* const* grads, float* theta,
                                         float* const* m, lioncub_stream_t stream)
{
    lc::set_handleless_error("");
    if (d < 0 || W < 1 || W > LIONCUB_MAX_WORKERS || t < 0)
        return fail(LIONCUB_ERR_ARG, "noalloc step: bad sizes (d >= 0, 1 <= W <= LIONCUB_MAX_WORKERS, t >= 0)");
    if (grad_dtype != LIONCUB_GRAD_BF16 && grad_dtype != LIONCUB_GRAD_F32)
        return fail(LIONCUB_ERR_ARG, "noalloc step: unknown gradient dtype");
    const int64_t words = (d + 31) / 32;
    const int64_t stride = (words + 3) / 4 * 4;
    if (stride * W > static_cast<int64_t>(LIONCUB_NOALLOC_MAX_WORDS))
        return fail(LIONCUB_ERR_ARG,
                    "noalloc step: W * ceil(d/32) (rounded up to 4 words per worker) exceeds "
                    "LIONCUB_NOALLOC_MAX_WORDS; use lioncub_create/lioncub_step for larger problems");
    if (!grads || !theta || !m)
        return fail(LIONCUB_ERR_ARG, "noalloc step: NULL pointer argument");
    if (reinterpret_cast<uintptr_t>(theta) & 15u)
        return fail(LIONCUB_ERR_ALIGN, "noalloc step: theta is not 16-byte aligned");
    for (int i = 0; i < W; ++i) {
        if (!grads[i] || !m[i])
            return fail(LIONCUB_ERR_ARG, "noalloc step: NULL gradient or momentum pointer");
        if ((reinterpret_cast<uintptr_t>(grads[i]) | reinterpret_cast<uintptr_t>(m[i])) & 15u)
            return fail(LIONCUB_ERR_ALIGN, "noalloc step: a gradient or momentum pointer is not 16-byte aligned");
    }
    // set-up (first call on this device): look up the static arrays, which
    // also loads this file's module; a d == 0 call stops right after it
    void* wire = nullptr;
    int* status = nullptr;
    cudaError_t e = static_addresses(&wire, &status);
    if (e != cudaSuccess)
        return fail(LIONCUB_ERR_CUDA, "noalloc step: cudaGetSymbolAddress failed");
    if constexpr (lc::kBoundsCheck) {
        int bad = 0;
        e = cudaMemcpy(&bad, status, sizeof bad, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess)
            return fail(LIONCUB_ERR_CUDA, "noalloc step: reading the status word failed");
        if (bad != 0)
            return fail(LIONCUB_ERR_CUDA, "noalloc step: a previous call's kernels set the status word "
                                          "(bounds-checked build)");
    }
    if (d == 0)
        return LIONCUB_OK;

    lc::StepArgs a;
    memset(&a, 0, sizeof a);
    for (int i = 0; i < W; ++i) {
        a.g[i] = grads[i];
        a.m[i] = m[i];
    }
    a.theta = theta;
    a.status = lc::kBoundsCheck ? status : nullptr;
    a.wire = static_cast<uint32_t*>(wire);
    a.wire_stride = stride;
    a.d = d;
    a.W = W;
    a.K = 1;
    a.nbits = 1;
    a.beta1 = beta1;
    a.omega1 = 1.0f - beta1;
    a.beta2 = beta2;
    a.omega2 = 1.0f - beta2;
    a.lr = lr;
    a.wd = wd;
    a.qmax = 0.0f;
    a.zero_bit = (t % 2 == 0) ? 1u : 0u;
    a.tie_u = 0.0f;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>((d + kTile - 1) / kTile), W);
    if (grad_dtype == LIONCUB_GRAD_BF16)
        k_compress_sign_flat<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
    else
        k_compress_sign_flat<float><<<grid, kThreads, 0, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(LIONCUB_ERR_CUDA, "noalloc step: compress launch failed");
    e = lc::launch_reduce_apply(a, 0, s);
    if (e != cudaSuccess)
        return fail(LIONCUB_ERR_CUDA, "noalloc step: reduce_apply launch failed");
    return LIONCUB_OK;
}
