// lioncub.cu -- the C ABI (include/lioncub.h): handle life cycle, layout
// validation, scratch ownership, step sequencing and error reporting.
//
// A step is two launches in sign mode (compress, reduce_apply) and four in
// L1 mode (m1_partial, m1_finalize, compress, reduce_apply), all on the
// caller's stream with no host synchronization.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "guard.h"
#include "host_io.h"
#include "internal.h"

using lc::StepArgs;
using lc::Tile;

// Layouts the language bindings rely on.
static_assert(sizeof(lioncub_tensor) == 24, "lioncub_tensor must stay 24 bytes");
static_assert(sizeof(lioncub_diag) == 48, "lioncub_diag must stay 48 bytes");
static_assert(sizeof(lioncub_qinf_diag) == 40, "lioncub_qinf_diag must stay 40 bytes");
static_assert(sizeof(lioncub_dist_plan) == 104, "lioncub_dist_plan must stay 104 bytes");
static_assert(sizeof(StepArgs) <= 4096, "kernel parameters must fit the classic 4 KB limit");
static_assert(lc::kStatusWaitTimeout == LIONCUB_STATUS_WAIT_TIMEOUT &&
                  lc::kStatusOutOfBounds == LIONCUB_STATUS_OUT_OF_BOUNDS && lc::kStatusGuard == LIONCUB_STATUS_GUARD,
              "status bits are part of the ABI");

struct lioncub_s {
    int device = 0;
    int64_t d = 0;
    int W = 0;
    int K = 0;
    int mode = 0;        // LIONCUB_MODE_*
    uint32_t flags = 0;  // LIONCUB_FLAG_*
    int nbits = 1;
    int grad_dtype = 0;
    int sync_interval = 0;
    float beta1 = 0, beta2 = 0, lr = 0, wd = 0;
    int64_t t = 0;
    bool bound = false;
    float* theta = nullptr;
    float* m[LIONCUB_MAX_WORKERS] = {};

    std::vector<lioncub_tensor> layout;
    int64_t ntiles = 0;
    int64_t nplain = 0;       // tiles of unsynchronized tensors (they come first)
    int64_t wire_words = 0;   // per worker, dense
    int64_t wire_stride = 0;  // per worker, padded to 4 words

    // device scratch owned by the library: every allocation lioncub_create
    // made (allocs), and the guard bands around the buffers kernels write
    std::vector<void*> allocs;
    lc::GuardList guards{};
    uint32_t* wire = nullptr;
    Tile* tiles = nullptr;
    int32_t* tile_range = nullptr;
    int64_t* numel = nullptr;
    float2* partials = nullptr;
    float* m1 = nullptr;
    float* inv = nullptr;
    int* status = nullptr;  // set by a kernel whose bounded wait gave up
    float* maxabs = nullptr;  // W x K max |c| of lioncub_diagnose_qinf (allocated on its first call)
    // lioncub_step_host: double-buffered staging, an upload stream and the
    // events that order uploads against the steps that read them
    void* staging[2] = {nullptr, nullptr};
    int nstaging = 0;
    size_t staging_stride = 0;
    cudaStream_t up = nullptr;
    cudaEvent_t ev_up[2] = {nullptr, nullptr};
    cudaEvent_t ev_used[2] = {nullptr, nullptr};
    bool used_recorded[2] = {false, false};
    int64_t host_calls = 0;

    // fault injection (environment, read at create): the fail_alloc_at-th
    // device allocation and the fail_launch_at-th step launch of the handle
    // report an error instead of running (0 = off)
    int64_t fail_alloc_at = 0, alloc_count = 0;
    int64_t fail_launch_at = 0, launch_count = 0;
    // fault injection: the staged reduce's first wait gives up after this
    // many non-blocking polls (0 = off)
    uint32_t wait_polls = 0;

    // profiling
    int prof_steps_left = 0;   // steps still to record
    bool prof_this_call = false;
    int prof_capacity = 0;     // event-pair slots
    std::vector<cudaEvent_t> prof_events;  // pairs
    std::vector<int> prof_kernel;
    int prof_used = 0;

    // data-parallel exchange (lioncub_dist_create): this rank's share of the
    // workers (W above is the local count), the exchange plan and the
    // caller's exchange buffers
    bool dist = false;
    int nranks = 1, rank = 0, W_global = 0;
    lioncub_dist_plan plan{};
    void* xbuf[LIONCUB_DIST_BUFFERS] = {};
    bool xbound = false;
    int phase = 0;  // the next exchange call: 0 compress, 1 reduce, 2 apply

    std::string err;
};

namespace {

// Message of the last failed handle-less call on this thread (lioncub_create,
// lioncub_host_alloc, lioncub_sign_step_noalloc): no handle exists to hold
// it.  Each of those calls clears it when it succeeds.
thread_local std::string g_create_err;

int fail(lioncub_t h, int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (h)
        h->err = buf;
    else
        g_create_err = buf;
    return code;
}

int cuda_fail(lioncub_t h, cudaError_t e, const char* what)
{
    return fail(h, LIONCUB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device address of a page-locked host buffer mapped into the device's
// address space (16-byte aligned), else nullptr: pageable memory, or memory
// the device cannot address, which a copy engine then moves.
float* mapped_host_view(float* p)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();  // not a CUDA pointer: clear the non-sticky error
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer || !aligned16(attr.devicePointer))
        return nullptr;
    return static_cast<float*>(attr.devicePointer);
}

void free_scratch(lioncub_t h)
{
    for (void* p : h->allocs)
        cudaFree(p);
    h->allocs.clear();
    h->guards.n = 0;
    for (void* p : h->staging)
        if (p)
            cudaFree(p);
    h->wire = nullptr;
    h->tiles = nullptr;
    h->tile_range = nullptr;
    h->numel = nullptr;
    h->partials = nullptr;
    h->m1 = h->inv = nullptr;
    h->status = nullptr;
    h->maxabs = nullptr;
    h->staging[0] = h->staging[1] = nullptr;
    h->nstaging = 0;
    for (int b = 0; b < 2; ++b) {
        if (h->ev_up[b])
            cudaEventDestroy(h->ev_up[b]);
        if (h->ev_used[b])
            cudaEventDestroy(h->ev_used[b]);
        h->ev_up[b] = h->ev_used[b] = nullptr;
    }
    if (h->up)
        cudaStreamDestroy(h->up);
    h->up = nullptr;
}

void drop_profile(lioncub_t h)
{
    for (cudaEvent_t e : h->prof_events)
        cudaEventDestroy(e);
    h->prof_events.clear();
    h->prof_kernel.clear();
    h->prof_capacity = 0;
    h->prof_used = 0;
    h->prof_steps_left = 0;
    h->prof_this_call = false;
}

// A positive integer from the environment, else 0.
int64_t env_index(const char* name)
{
    const char* v = std::getenv(name);
    if (!v || !*v)
        return 0;
    char* end = nullptr;
    const long long x = std::strtoll(v, &end, 10);
    return (*end == '\0' && x > 0) ? static_cast<int64_t>(x) : 0;
}

// Every device allocation of a handle goes through here, so that fault
// injection can fail any one of them.
cudaError_t raw_alloc(lioncub_t h, void** p, size_t bytes)
{
    *p = nullptr;
    if (++h->alloc_count == h->fail_alloc_at)
        return cudaErrorMemoryAllocation;
    return cudaMalloc(p, bytes);
}

// count elements of T for the handle's lifetime (freed by free_scratch).
template <typename T>
cudaError_t dev_alloc(lioncub_t h, T** p, size_t count)
{
    void* base = nullptr;
    *p = nullptr;
    const cudaError_t e = raw_alloc(h, &base, (count ? count : 1) * sizeof(T));
    if (e != cudaSuccess)
        return e;
    h->allocs.push_back(base);
    *p = static_cast<T*>(base);
    return cudaSuccess;
}

// The same for a buffer that kernels write, between two guard bands of
// lc::kGuardBytes.  The buffer keeps cudaMalloc's 256-byte alignment.
template <typename T>
cudaError_t guarded_alloc(lioncub_t h, T** p, size_t count)
{
    static_assert(lc::kGuardBytes % 256 == 0 && sizeof(T) % 4 == 0, "guards keep alignment");
    const size_t inner = (count ? count : 1) * sizeof(T);
    char* base = nullptr;
    *p = nullptr;
    if (h->guards.n + 2 > lc::kMaxGuardBands)
        return cudaErrorInvalidValue;
    cudaError_t e = dev_alloc(h, &base, lc::kGuardBytes + inner + lc::kGuardBytes);
    if (e != cudaSuccess)
        return e;
    char* back = base + lc::kGuardBytes + inner;
    e = cudaMemset(base, static_cast<int>(lc::kGuardByte), lc::kGuardBytes);
    if (e == cudaSuccess)
        e = cudaMemset(back, static_cast<int>(lc::kGuardByte), lc::kGuardBytes);
    if (e != cudaSuccess)
        return e;
    h->guards.band[h->guards.n++] = reinterpret_cast<const uint32_t*>(base);
    h->guards.band[h->guards.n++] = reinterpret_cast<const uint32_t*>(back);
    *p = reinterpret_cast<T*>(base + lc::kGuardBytes);
    return cudaSuccess;
}

// Fault injection: the error the handle's next step launch reports instead
// of launching, or cudaSuccess.
cudaError_t injected_launch_fault(lioncub_t h)
{
    return (++h->launch_count == h->fail_launch_at) ? cudaErrorLaunchOutOfResources : cudaSuccess;
}

StepArgs make_args(lioncub_t h, const void* const* grads)
{
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    for (int i = 0; i < h->W; ++i) {
        a.g[i] = grads ? grads[i] : nullptr;
        a.m[i] = h->m[i];
    }
    a.theta = h->theta;
    a.wire = h->wire;
    a.wire_stride = h->wire_stride;
    a.d = h->d;
    a.tiles = h->tiles;
    a.ntiles = h->ntiles;
    a.nplain = h->nplain;
    a.tile_range = h->tile_range;
    a.numel = h->numel;
    a.partials = h->partials;
    a.m1 = h->m1;
    a.inv = h->inv;
    a.status = h->status;
    a.first_wait_polls = h->wait_polls;
    a.W = h->W;
    a.K = h->K;
    a.nbits = h->nbits;
    a.beta1 = h->beta1;
    a.omega1 = 1.0f - h->beta1;  // one fp32 rounding, on the host
    a.beta2 = h->beta2;
    a.omega2 = 1.0f - h->beta2;
    a.lr = h->lr;
    a.wd = h->wd;
    a.qmax = static_cast<float>((1 << (h->nbits - 1)) - 1);
    const bool even = (h->t % 2) == 0;
    a.zero_bit = even ? 1u : 0u;
    a.sync_now = (h->sync_interval > 0 && (h->t + 1) % h->sync_interval == 0) ? 1 : 0;
    a.average = (h->flags & LIONCUB_FLAG_AVERAGE) ? 1 : 0;
    a.tie_u = (h->flags & LIONCUB_FLAG_TIE_ALTERNATE) ? (even ? 1.0f : -1.0f) : 0.0f;
    return a;
}

// NVTX range around a call or a launch (a no-op unless a tool is attached),
// so profilers can attribute kernels to the library's steps.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Records an event before a launch when profiling is on; returns the slot.
int prof_begin(lioncub_t h, int kernel, cudaStream_t s)
{
    if (!h->prof_this_call || h->prof_used >= h->prof_capacity)
        return -1;
    const int slot = h->prof_used++;
    h->prof_kernel[slot] = kernel;
    cudaEventRecord(h->prof_events[2 * slot], s);
    return slot;
}

void prof_end(lioncub_t h, int slot, cudaStream_t s)
{
    if (slot >= 0)
        cudaEventRecord(h->prof_events[2 * slot + 1], s);
}

// One kernel launch of a step: an NVTX range named for the kernel, the
// profiling events around it, and the fault-injection check before it.
template <typename Launch>
cudaError_t step_launch(lioncub_t h, int kernel, const char* name, cudaStream_t s, Launch&& launch)
{
    NvtxRange range(name);
    const int slot = prof_begin(h, kernel, s);
    cudaError_t e = injected_launch_fault(h);
    if (e == cudaSuccess)
        e = launch();
    prof_end(h, slot, s);
    return e;
}

}  // namespace

namespace lc {
// Lets handle-less entry points (noalloc.cu) report a message through
// lioncub_last_error(NULL).
void set_handleless_error(const char* msg)
{
    g_create_err = msg;
}
}  // namespace lc

extern "C" {

const char* lioncub_strerror(int code)
{
    switch (code) {
    case LIONCUB_OK: return "LIONCUB_OK";
    case LIONCUB_ERR_ARG: return "LIONCUB_ERR_ARG";
    case LIONCUB_ERR_ALIGN: return "LIONCUB_ERR_ALIGN";
    case LIONCUB_ERR_STATE: return "LIONCUB_ERR_STATE";
    case LIONCUB_ERR_OOM: return "LIONCUB_ERR_OOM";
    case LIONCUB_ERR_CUDA: return "LIONCUB_ERR_CUDA";
    default: return "LIONCUB_ERR_UNKNOWN";
    }
}

const char* lioncub_last_error(lioncub_t h)
{
    return h ? h->err.c_str() : g_create_err.c_str();
}

int lioncub_create(lioncub_t* out, int64_t d, int W, const lioncub_tensor* layout, int K,
                   float beta1, float beta2, float lr, float wd, int mode, int nbits,
                   int grad_dtype, int sync_interval)
{
    if (!out)
        return LIONCUB_ERR_ARG;
    *out = nullptr;
    lioncub_s* h = new (std::nothrow) lioncub_s();
    if (!h)
        return LIONCUB_ERR_OOM;

    const int base_mode = mode & 0xff;
    const uint32_t flags = static_cast<uint32_t>(mode) & ~0xffu;
    int rc = LIONCUB_OK;
    if (d < 0 || W < 1 || W > LIONCUB_MAX_WORKERS || K < 0 || (K > 0 && !layout))
        rc = fail(h, LIONCUB_ERR_ARG, "bad sizes: d=%lld W=%d K=%d", (long long)d, W, K);
    else if (base_mode != LIONCUB_MODE_SIGN_MAJORITY && base_mode != LIONCUB_MODE_L1_INTSUM)
        rc = fail(h, LIONCUB_ERR_ARG, "unknown mode %d", base_mode);
    else if (flags & ~static_cast<uint32_t>(LIONCUB_FLAG_TIE_ALTERNATE | LIONCUB_FLAG_AVERAGE))
        rc = fail(h, LIONCUB_ERR_ARG, "unknown mode flags 0x%x", flags);
    else if ((flags & LIONCUB_FLAG_AVERAGE) &&
             (base_mode != LIONCUB_MODE_SIGN_MAJORITY || (flags & LIONCUB_FLAG_TIE_ALTERNATE)))
        rc = fail(h, LIONCUB_ERR_ARG, "the average rule applies to sign mode only, without tie alternation");
    else if (base_mode == LIONCUB_MODE_L1_INTSUM && nbits != 2 && nbits != 4 && nbits != 8)
        rc = fail(h, LIONCUB_ERR_ARG, "nbits must be 2, 4 or 8 in L1 mode (got %d)", nbits);
    else if (grad_dtype != LIONCUB_GRAD_BF16 && grad_dtype != LIONCUB_GRAD_F32)
        rc = fail(h, LIONCUB_ERR_ARG, "unknown gradient dtype %d", grad_dtype);
    else if (sync_interval < 0)
        rc = fail(h, LIONCUB_ERR_ARG, "sync_interval must be >= 0");
    if (rc != LIONCUB_OK) {
        g_create_err = h->err;
        delete h;
        return rc;
    }
    g_create_err.clear();

    h->d = d;
    h->W = W;
    h->mode = base_mode;
    h->flags = flags;
    h->nbits = base_mode == LIONCUB_MODE_SIGN_MAJORITY ? 1 : nbits;
    h->grad_dtype = grad_dtype;
    h->sync_interval = sync_interval;
    h->beta1 = beta1;
    h->beta2 = beta2;
    h->lr = lr;
    h->wd = wd;
    if (K == 0) {
        h->layout.push_back(lioncub_tensor{0, d, 0u});
    } else {
        h->layout.assign(layout, layout + K);
    }
    h->K = static_cast<int>(h->layout.size());

    // Validate: tensors tile [0, d) in order, 32-aligned offsets.
    int64_t next = 0;
    for (int k = 0; k < h->K; ++k) {
        const lioncub_tensor& T = h->layout[k];
        if (T.offset % 32 != 0) {
            rc = fail(h, LIONCUB_ERR_ALIGN, "tensor %d offset %lld is not a multiple of 32", k, (long long)T.offset);
            break;
        }
        if (T.offset != next || T.numel < 0) {
            rc = fail(h, LIONCUB_ERR_ARG, "tensor %d [%lld, +%lld) does not continue the layout at %lld", k,
                      (long long)T.offset, (long long)T.numel, (long long)next);
            break;
        }
        if (T.flags & ~static_cast<uint32_t>(LIONCUB_TENSOR_SYNC_M)) {
            rc = fail(h, LIONCUB_ERR_ARG, "tensor %d has unknown flags 0x%x", k, T.flags);
            break;
        }
        next += T.numel;
    }
    if (rc == LIONCUB_OK && next != d)
        rc = fail(h, LIONCUB_ERR_ARG, "layout covers %lld elements, d is %lld", (long long)next, (long long)d);
    if (rc != LIONCUB_OK) {
        g_create_err = h->err;
        delete h;
        return rc;
    }

    // Tile table: the tiles of unsynchronized tensors first, then those of
    // synchronized tensors, so that a sync step launches each group over one
    // contiguous range.  A tensor's tiles stay contiguous either way.
    std::vector<Tile> tiles;
    std::vector<int32_t> first(2 * static_cast<size_t>(h->K), 0);  // [first, end) tile range per tensor
    std::vector<int64_t> numel(h->K, 0);
    for (int pass = 0; pass < 2; ++pass) {
        for (int k = 0; k < h->K; ++k) {
            const lioncub_tensor& T = h->layout[k];
            const bool sync = (T.flags & LIONCUB_TENSOR_SYNC_M) != 0;
            if (sync != (pass == 1))
                continue;
            first[2 * k] = static_cast<int32_t>(tiles.size());
            numel[k] = T.numel;
            const uint32_t meta = static_cast<uint32_t>(k) | (sync ? lc::kTileSync : 0u);
            for (int64_t s = 0; s < T.numel; s += lc::kTile) {
                const int64_t len = (T.numel - s) < lc::kTile ? (T.numel - s) : lc::kTile;
                tiles.push_back(Tile{T.offset + s, static_cast<int32_t>(len), meta});
            }
            if (tiles.size() > 0x7fffffffu) {
                delete h;
                return fail(nullptr, LIONCUB_ERR_ARG, "too many tiles");
            }
            first[2 * k + 1] = static_cast<int32_t>(tiles.size());
        }
        if (pass == 0)
            h->nplain = static_cast<int64_t>(tiles.size());
    }
    h->ntiles = static_cast<int64_t>(tiles.size());
    h->wire_words = (d * h->nbits + 31) / 32;
    h->wire_stride = (h->wire_words + 3) / 4 * 4;

    h->fail_alloc_at = env_index("LIONCUB_FAIL_ALLOC");
    h->fail_launch_at = env_index("LIONCUB_FAIL_LAUNCH");
    const int64_t polls = env_index("LIONCUB_WAIT_POLLS");
    h->wait_polls = static_cast<uint32_t>(polls > 0xffff ? 0xffff : polls);
    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess) e = guarded_alloc(h, &h->wire, static_cast<size_t>(W) * h->wire_stride + 4);
    if (e == cudaSuccess) e = dev_alloc(h, &h->tiles, tiles.size());
    if (e == cudaSuccess) e = dev_alloc(h, &h->tile_range, first.size());
    if (e == cudaSuccess) e = dev_alloc(h, &h->numel, numel.size());
    if (e == cudaSuccess) e = dev_alloc(h, &h->status, 1);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int));
    if (e == cudaSuccess && h->mode == LIONCUB_MODE_L1_INTSUM) {
        e = guarded_alloc(h, &h->partials, static_cast<size_t>(W) * h->ntiles);
        if (e == cudaSuccess) e = guarded_alloc(h, &h->m1, static_cast<size_t>(W) * h->K);
        if (e == cudaSuccess) e = guarded_alloc(h, &h->inv, static_cast<size_t>(W) * h->K);
    }
    // Fault injection: one byte of the guard band after the wire buffer is
    // overwritten, as an overrunning kernel would.
    if (e == cudaSuccess && env_index("LIONCUB_POISON_GUARD") > 0)
        e = cudaMemset(const_cast<uint32_t*>(h->guards.band[1]), 0, 1);
    if (e == cudaSuccess && !tiles.empty())
        e = cudaMemcpy(h->tiles, tiles.data(), tiles.size() * sizeof(Tile), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(h->tile_range, first.data(), first.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !numel.empty())
        e = cudaMemcpy(h->numel, numel.data(), numel.size() * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemset(h->wire, 0, (static_cast<size_t>(W) * h->wire_stride + 4) * sizeof(uint32_t));
    // The set-up copies and fills above are ordered on the legacy default
    // stream and may still be in flight; wait for them, so that steps on any
    // stream (non-blocking ones included) see the finished tables.
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) {
        const int code = (e == cudaErrorMemoryAllocation) ? LIONCUB_ERR_OOM : LIONCUB_ERR_CUDA;
        cudaGetLastError();  // clear a non-sticky allocation error
        free_scratch(h);
        delete h;
        return fail(nullptr, code, "device set-up failed: %s", cudaGetErrorString(e));
    }
    *out = h;
    return LIONCUB_OK;
}

int lioncub_bind_state(lioncub_t h, float* theta, float* const* m)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (!theta || !m)
        return fail(h, LIONCUB_ERR_ARG, "theta and m must be non-NULL");
    if (!aligned16(theta))
        return fail(h, LIONCUB_ERR_ALIGN, "theta is not 16-byte aligned");
    for (int i = 0; i < h->W; ++i) {
        if (!m[i])
            return fail(h, LIONCUB_ERR_ARG, "m[%d] is NULL", i);
        if (!aligned16(m[i]))
            return fail(h, LIONCUB_ERR_ALIGN, "m[%d] is not 16-byte aligned", i);
    }
    h->theta = theta;
    for (int i = 0; i < h->W; ++i)
        h->m[i] = m[i];
    h->bound = true;
    h->err.clear();
    return LIONCUB_OK;
}

int lioncub_step(lioncub_t h, const void* const* grads, lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (h->dist)
        return fail(h, LIONCUB_ERR_STATE, "a data-parallel handle steps through lioncub_dist_compress/reduce/apply");
    if (!h->bound)
        return fail(h, LIONCUB_ERR_STATE, "lioncub_bind_state has not been called");
    if (!grads)
        return fail(h, LIONCUB_ERR_ARG, "grads is NULL");
    for (int i = 0; i < h->W; ++i) {
        if (!grads[i])
            return fail(h, LIONCUB_ERR_ARG, "grads[%d] is NULL", i);
        if (!aligned16(grads[i]))
            return fail(h, LIONCUB_ERR_ALIGN, "grads[%d] is not 16-byte aligned", i);
    }
    NvtxRange range("lioncub_step");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const StepArgs a = make_args(h, grads);
    const bool l1 = h->mode == LIONCUB_MODE_L1_INTSUM;
    h->prof_this_call = h->prof_steps_left > 0;
    if (h->prof_this_call)
        --h->prof_steps_left;
    cudaError_t e;
    if (l1) {
        e = step_launch(h, LIONCUB_KERNEL_M1, "m1_partial", s,
                        [&] { return lc::launch_m1_partial(a, h->grad_dtype, s); });
        if (e != cudaSuccess)
            return cuda_fail(h, e, "m1_partial launch");
        e = step_launch(h, LIONCUB_KERNEL_M1_FINAL, "m1_finalize", s, [&] { return lc::launch_m1_finalize(a, s); });
        if (e != cudaSuccess)
            return cuda_fail(h, e, "m1_finalize launch");
    }
    e = step_launch(h, LIONCUB_KERNEL_COMPRESS, "compress", s,
                    [&] { return lc::launch_compress(a, h->grad_dtype, l1 ? 1 : 0, s); });
    if (e != cudaSuccess)
        return cuda_fail(h, e, "compress launch");
    e = step_launch(h, LIONCUB_KERNEL_REDUCE_APPLY, "reduce_apply", s,
                    [&] { return lc::launch_reduce_apply(a, l1 ? 1 : 0, s); });
    if (e != cudaSuccess)
        return cuda_fail(h, e, "reduce_apply launch");
    h->t += 1;
    return LIONCUB_OK;
}

int lioncub_step_host(lioncub_t h, const void* const* grads_host, float* theta_host_out,
                      lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (h->dist)
        return fail(h, LIONCUB_ERR_STATE, "a data-parallel handle steps through lioncub_dist_compress/reduce/apply");
    if (!h->bound)
        return fail(h, LIONCUB_ERR_STATE, "lioncub_bind_state has not been called");
    if (!grads_host || !theta_host_out)
        return fail(h, LIONCUB_ERR_ARG, "grads_host and theta_host_out must be non-NULL");
    for (int i = 0; i < h->W; ++i)
        if (!grads_host[i])
            return fail(h, LIONCUB_ERR_ARG, "grads_host[%d] is NULL", i);
    const size_t gbytes = static_cast<size_t>(h->d) * (h->grad_dtype == LIONCUB_GRAD_BF16 ? 2 : 4);
    const size_t gstride = (gbytes + 255) / 256 * 256;
    if (h->nstaging == 0) {
        // First call: an upload stream that never synchronizes implicitly with
        // the legacy default stream, its events, and two staging buffers (one
        // if memory is short, which serializes uploads behind the steps).
        // (a retry after a failed first call creates only what is missing)
        cudaError_t e = cudaSuccess;
        if (!h->up)
            e = cudaStreamCreateWithFlags(&h->up, cudaStreamNonBlocking);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            if (!h->ev_up[b])
                e = cudaEventCreateWithFlags(&h->ev_up[b], cudaEventDisableTiming);
            if (e == cudaSuccess && !h->ev_used[b])
                e = cudaEventCreateWithFlags(&h->ev_used[b], cudaEventDisableTiming);
        }
        if (e != cudaSuccess)
            return cuda_fail(h, e, "host-step set-up");
        const size_t bytes = gstride * h->W + 256;
        for (int b = 0; b < 2; ++b) {
            e = raw_alloc(h, &h->staging[b], bytes);
            if (e != cudaSuccess) {
                cudaGetLastError();
                h->staging[b] = nullptr;
                break;
            }
            h->nstaging = b + 1;
        }
        if (h->nstaging == 0)
            return fail(h, e == cudaErrorMemoryAllocation ? LIONCUB_ERR_OOM : LIONCUB_ERR_CUDA,
                        "staging allocation of %zu bytes failed", bytes);
        h->staging_stride = gstride;
    }
    NvtxRange range("lioncub_step_host");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int b = static_cast<int>(h->host_calls % h->nstaging);
    cudaError_t e = cudaSuccess;
    // The upload into buffer b waits until the step that last read b is done;
    // it does not wait for the caller's stream, so it overlaps the previous
    // step's kernels and its theta download.
    if (h->used_recorded[b])
        e = cudaStreamWaitEvent(h->up, h->ev_used[b], 0);
    const void* dev[LIONCUB_MAX_WORKERS];
    for (int i = 0; i < h->W && e == cudaSuccess; ++i) {
        char* dst = static_cast<char*>(h->staging[b]) + h->staging_stride * i;
        dev[i] = dst;
        if (gbytes)
            e = cudaMemcpyAsync(dst, grads_host[i], gbytes, cudaMemcpyHostToDevice, h->up);
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(h->ev_up[b], h->up);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(s, h->ev_up[b], 0);
    if (e != cudaSuccess)
        return cuda_fail(h, e, "gradient upload");
    int rc = lioncub_step(h, dev, stream);
    if (rc != LIONCUB_OK)
        return rc;
    e = cudaEventRecord(h->ev_used[b], s);
    if (e == cudaSuccess) {
        h->used_recorded[b] = true;
        // theta download: SM stores into a mapped page-locked buffer (the
        // copy engine stays with the next upload), else a copy
        float* mapped = h->d ? mapped_host_view(theta_host_out) : nullptr;
        if (mapped)
            e = lc::launch_store_host(h->theta, mapped, h->d, s);
        else if (h->d)
            e = cudaMemcpyAsync(theta_host_out, h->theta, static_cast<size_t>(h->d) * sizeof(float),
                                cudaMemcpyDeviceToHost, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(h, e, "theta download");
    ++h->host_calls;
    return LIONCUB_OK;
}

int lioncub_dist_plan_make(int64_t d, int W, int nranks, int rank, const lioncub_tensor* layout, int K, int mode,
                           int nbits, int sync_interval, lioncub_dist_plan* out)
{
    if (!out)
        return LIONCUB_ERR_ARG;
    std::memset(out, 0, sizeof *out);
    g_create_err.clear();
    const int base_mode = mode & 0xff;
    const bool average = (mode & LIONCUB_FLAG_AVERAGE) != 0;
    if (d < 0 || W < 1 || W > LIONCUB_MAX_WORKERS || nranks < 1 || nranks > W || W % nranks != 0 || rank < 0 ||
        rank >= nranks || K < 0 || (K > 0 && !layout))
        return fail(nullptr, LIONCUB_ERR_ARG,
                    "bad exchange sizes: d=%lld W=%d nranks=%d rank=%d K=%d (need 1 <= nranks <= W, W %% nranks == 0)",
                    (long long)d, W, nranks, rank, K);
    if (base_mode != LIONCUB_MODE_SIGN_MAJORITY && base_mode != LIONCUB_MODE_L1_INTSUM)
        return fail(nullptr, LIONCUB_ERR_ARG, "unknown mode %d", base_mode);
    if (base_mode == LIONCUB_MODE_L1_INTSUM && nbits != 2 && nbits != 4 && nbits != 8)
        return fail(nullptr, LIONCUB_ERR_ARG, "nbits must be 2, 4 or 8 in L1 mode (got %d)", nbits);
    if (average && W > 127)
        return fail(nullptr, LIONCUB_ERR_ARG, "the exchanged vote sums of the average are int8: W <= 127");
    const int W_loc = W / nranks;
    out->local_workers = W_loc;
    out->first_worker = rank * W_loc;
    if (base_mode == LIONCUB_MODE_SIGN_MAJORITY) {
        const int64_t blocks = (d + lc::kDistChunkAlign - 1) / lc::kDistChunkAlign;
        const int64_t per = (blocks + nranks - 1) / nranks;
        out->chunk = (per > 0 ? per : 1) * lc::kDistChunkAlign;
        out->chunk_words = out->chunk / 32;
        out->dir_bits = average ? 8 : 2;
        out->dir_words = out->chunk * out->dir_bits / 32;
        out->bytes[LIONCUB_DIST_SEND] = static_cast<int64_t>(nranks) * W_loc * out->chunk_words * 4;
        out->bytes[LIONCUB_DIST_RECV] = static_cast<int64_t>(W) * out->chunk_words * 4;
        out->bytes[LIONCUB_DIST_DIR_CHUNK] = out->dir_words * 4;
        out->bytes[LIONCUB_DIST_DIR_ALL] = static_cast<int64_t>(nranks) * out->dir_words * 4;
    } else {
        const int qmax = (1 << (nbits - 1)) - 1;
        out->agg_bytes = (static_cast<int64_t>(W) * qmax <= 127) ? 1 : 4;
        out->bytes[LIONCUB_DIST_AGG] = (d * out->agg_bytes + 15) / 16 * 16;
    }
    if (sync_interval > 0) {
        int64_t slots = 0;
        for (int k = 0; k < K; ++k)
            if (layout[k].flags & LIONCUB_TENSOR_SYNC_M)
                slots += (layout[k].numel + lc::kTile - 1) / lc::kTile * lc::kTile;
        out->sync_slots = slots;
        out->bytes[LIONCUB_DIST_SYNC_SEND] = static_cast<int64_t>(W_loc) * slots * 4;
        out->bytes[LIONCUB_DIST_SYNC_RECV] = static_cast<int64_t>(W) * slots * 4;
    }
    return LIONCUB_OK;
}

int lioncub_dist_create(lioncub_t* out, int64_t d, int W, int nranks, int rank, const lioncub_tensor* layout, int K,
                        float beta1, float beta2, float lr, float wd, int mode, int nbits, int grad_dtype,
                        int sync_interval)
{
    if (!out)
        return LIONCUB_ERR_ARG;
    *out = nullptr;
    lioncub_dist_plan plan;
    int rc = lioncub_dist_plan_make(d, W, nranks, rank, layout, K, mode, nbits, sync_interval, &plan);
    if (rc != LIONCUB_OK)
        return rc;
    rc = lioncub_create(out, d, plan.local_workers, layout, K, beta1, beta2, lr, wd, mode, nbits, grad_dtype,
                        sync_interval);
    if (rc != LIONCUB_OK)
        return rc;
    lioncub_t h = *out;
    h->dist = true;
    h->nranks = nranks;
    h->rank = rank;
    h->W_global = W;
    h->plan = plan;
    return LIONCUB_OK;
}

int lioncub_dist_bind_buffers(lioncub_t h, void* const* bufs)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (!h->dist)
        return fail(h, LIONCUB_ERR_STATE, "not a data-parallel handle (use lioncub_dist_create)");
    if (!bufs)
        return fail(h, LIONCUB_ERR_ARG, "bufs is NULL");
    for (int b = 0; b < LIONCUB_DIST_BUFFERS; ++b) {
        if (h->plan.bytes[b] > 0 && !bufs[b])
            return fail(h, LIONCUB_ERR_ARG, "exchange buffer %d is NULL but the plan needs %lld bytes", b,
                        (long long)h->plan.bytes[b]);
        if (bufs[b] && !aligned16(bufs[b]))
            return fail(h, LIONCUB_ERR_ALIGN, "exchange buffer %d is not 16-byte aligned", b);
    }
    for (int b = 0; b < LIONCUB_DIST_BUFFERS; ++b)
        h->xbuf[b] = h->plan.bytes[b] > 0 ? bufs[b] : nullptr;
    h->xbound = true;
    h->phase = 0;
    h->err.clear();
    return LIONCUB_OK;
}

namespace {

// Checks shared by the three exchange calls.
int dist_ready(lioncub_t h, int phase, const char* what)
{
    if (!h->dist)
        return fail(h, LIONCUB_ERR_STATE, "%s: not a data-parallel handle", what);
    if (!h->bound || !h->xbound)
        return fail(h, LIONCUB_ERR_STATE, "%s: bind the state and the exchange buffers first", what);
    if (h->phase != phase)
        return fail(h, LIONCUB_ERR_STATE, "%s out of order: the next exchange call is %s", what,
                    h->phase == 0 ? "lioncub_dist_compress" : h->phase == 1 ? "lioncub_dist_reduce"
                                                                          : "lioncub_dist_apply");
    return LIONCUB_OK;
}

// StepArgs of an exchange call: the local workers, and the exchange fields.
StepArgs dist_args(lioncub_t h, const void* const* grads)
{
    StepArgs a = make_args(h, grads);
    a.sync_slots = h->plan.sync_slots;
    return a;
}

}  // namespace

int lioncub_dist_compress(lioncub_t h, const void* const* grads, lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    int rc = dist_ready(h, 0, "lioncub_dist_compress");
    if (rc != LIONCUB_OK)
        return rc;
    if (!grads)
        return fail(h, LIONCUB_ERR_ARG, "grads is NULL");
    for (int i = 0; i < h->W; ++i) {
        if (!grads[i])
            return fail(h, LIONCUB_ERR_ARG, "grads[%d] is NULL", i);
        if (!aligned16(grads[i]))
            return fail(h, LIONCUB_ERR_ALIGN, "grads[%d] is not 16-byte aligned", i);
    }
    NvtxRange range("lioncub_dist_compress");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool l1 = h->mode == LIONCUB_MODE_L1_INTSUM;
    StepArgs a = dist_args(h, grads);
    a.sync_buf = static_cast<float*>(h->xbuf[LIONCUB_DIST_SYNC_SEND]);
    if (!l1) {  // (the compress pass writes signs chunk-major: the plan's chunk is a multiple of 4096)
        a.wire = static_cast<uint32_t*>(h->xbuf[LIONCUB_DIST_SEND]);
        a.wire_stride = 0;
        a.chunk = h->plan.chunk;
        a.chunk_words = h->plan.chunk_words;
    }
    h->prof_this_call = false;
    cudaError_t e = cudaSuccess;
    if (l1) {
        e = step_launch(h, LIONCUB_KERNEL_M1, "m1_partial", s, [&] { return lc::launch_m1_partial(a, h->grad_dtype, s); });
        if (e == cudaSuccess)
            e = step_launch(h, LIONCUB_KERNEL_M1_FINAL, "m1_finalize", s, [&] { return lc::launch_m1_finalize(a, s); });
    }
    if (e == cudaSuccess)
        e = step_launch(h, LIONCUB_KERNEL_COMPRESS, "compress_dist", s,
                        [&] { return lc::launch_compress_dist(a, h->grad_dtype, l1 ? 1 : 0, s); });
    if (e != cudaSuccess)
        return cuda_fail(h, e, "exchange compress launch");
    h->phase = 1;
    return LIONCUB_OK;
}

int lioncub_dist_reduce(lioncub_t h, lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    int rc = dist_ready(h, 1, "lioncub_dist_reduce");
    if (rc != LIONCUB_OK)
        return rc;
    NvtxRange range("lioncub_dist_reduce");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    StepArgs a = dist_args(h, nullptr);
    cudaError_t e;
    if (h->mode == LIONCUB_MODE_SIGN_MAJORITY) {
        // the owner's chunk: W rows of chunk_words received words
        const int64_t c0 = static_cast<int64_t>(h->rank) * h->plan.chunk;
        const int64_t len = h->d - c0;
        a.d = len < 0 ? 0 : (len < h->plan.chunk ? len : h->plan.chunk);
        a.W = h->W_global;
        a.wire = static_cast<uint32_t*>(h->xbuf[LIONCUB_DIST_RECV]);
        a.wire_stride = h->plan.chunk_words;
        e = step_launch(h, LIONCUB_KERNEL_REDUCE_APPLY, "owner_reduce", s,
                        [&] { return lc::launch_owner_reduce(a, h->plan.dir_bits, h->xbuf[LIONCUB_DIST_DIR_CHUNK], s); });
    } else {
        e = step_launch(h, LIONCUB_KERNEL_REDUCE_APPLY, "code_sum_local", s,
                        [&] { return lc::launch_code_sum_local(a, h->plan.agg_bytes, h->xbuf[LIONCUB_DIST_AGG], s); });
    }
    if (e != cudaSuccess)
        return cuda_fail(h, e, "exchange reduce launch");
    h->phase = 2;
    return LIONCUB_OK;
}

int lioncub_dist_apply(lioncub_t h, lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    int rc = dist_ready(h, 2, "lioncub_dist_apply");
    if (rc != LIONCUB_OK)
        return rc;
    NvtxRange range("lioncub_dist_apply");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    StepArgs a = dist_args(h, nullptr);
    cudaError_t e;
    if (h->mode == LIONCUB_MODE_SIGN_MAJORITY) {
        StepArgs b = a;
        b.W = h->W_global;  // the average's table divides by every worker
        e = step_launch(h, LIONCUB_KERNEL_REDUCE_APPLY, "apply_dir", s,
                        [&] { return lc::launch_apply_dir(b, h->plan.dir_bits, h->xbuf[LIONCUB_DIST_DIR_ALL], s); });
    } else {
        e = step_launch(h, LIONCUB_KERNEL_REDUCE_APPLY, "apply_agg", s,
                        [&] { return lc::launch_apply_agg(a, h->plan.agg_bytes, h->xbuf[LIONCUB_DIST_AGG], s); });
    }
    if (e == cudaSuccess && a.sync_now && h->plan.sync_slots > 0)
        e = step_launch(h, LIONCUB_KERNEL_COMPRESS, "sync_mean", s, [&] {
            return lc::launch_sync_mean(a, h->W_global, static_cast<const float*>(h->xbuf[LIONCUB_DIST_SYNC_RECV]), s);
        });
    if (e != cudaSuccess)
        return cuda_fail(h, e, "exchange apply launch");
    h->t += 1;
    h->phase = 0;
    return LIONCUB_OK;
}

int lioncub_host_alloc(void** out, size_t bytes)
{
    if (!out)
        return LIONCUB_ERR_ARG;
    *out = nullptr;
    g_create_err.clear();
    if (bytes == 0)
        return LIONCUB_OK;
    const cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocPortable | cudaHostAllocMapped);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return fail(nullptr, e == cudaErrorMemoryAllocation ? LIONCUB_ERR_OOM : LIONCUB_ERR_CUDA,
                    "page-locked allocation of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
    }
    return LIONCUB_OK;
}

void lioncub_host_free(void* p)
{
    if (p)
        cudaFreeHost(p);
}

int lioncub_set_lr(lioncub_t h, float lr)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    h->lr = lr;
    return LIONCUB_OK;
}

int lioncub_get_step(lioncub_t h, int64_t* t)
{
    if (!h || !t)
        return LIONCUB_ERR_ARG;
    *t = h->t;
    return LIONCUB_OK;
}

int lioncub_set_step(lioncub_t h, int64_t t)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (t < 0)
        return fail(h, LIONCUB_ERR_ARG, "step must be >= 0");
    h->t = t;
    return LIONCUB_OK;
}

int64_t lioncub_wire_words(lioncub_t h)
{
    return h ? h->wire_words : -1;
}

int lioncub_debug_export(lioncub_t h, int what, void* dst_dev, lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (!dst_dev)
        return fail(h, LIONCUB_ERR_ARG, "dst_dev is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (what) {
    case LIONCUB_EXPORT_WIRE:
        if (h->wire_words)
            e = cudaMemcpy2DAsync(dst_dev, h->wire_words * sizeof(uint32_t), h->wire,
                                  h->wire_stride * sizeof(uint32_t), h->wire_words * sizeof(uint32_t), h->W,
                                  cudaMemcpyDeviceToDevice, s);
        break;
    case LIONCUB_EXPORT_M1:
        if (h->mode != LIONCUB_MODE_L1_INTSUM)
            return fail(h, LIONCUB_ERR_STATE, "M1 exists in L1 mode only");
        e = cudaMemcpyAsync(dst_dev, h->m1, static_cast<size_t>(h->W) * h->K * sizeof(float),
                            cudaMemcpyDeviceToDevice, s);
        break;
    case LIONCUB_EXPORT_STATUS:
        e = lc::launch_guard_check(h->guards, h->status, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dst_dev, h->status, sizeof(int), cudaMemcpyDeviceToDevice, s);
        break;
    case LIONCUB_EXPORT_AGG: {
        const StepArgs a = make_args(h, nullptr);
        e = lc::launch_export_agg(a, h->mode == LIONCUB_MODE_L1_INTSUM ? 1 : 0, static_cast<int32_t*>(dst_dev), s);
        break;
    }
    default:
        return fail(h, LIONCUB_ERR_ARG, "unknown export %d", what);
    }
    if (e != cudaSuccess)
        return cuda_fail(h, e, "debug export");
    return LIONCUB_OK;
}

int lioncub_diagnose(lioncub_t h, const void* const* grads, lioncub_diag* out_dev, lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (h->dist)
        return fail(h, LIONCUB_ERR_STATE, "diagnostics need every worker on one GPU (not a data-parallel handle)");
    if (!h->bound)
        return fail(h, LIONCUB_ERR_STATE, "lioncub_bind_state has not been called");
    if (!grads || !out_dev)
        return fail(h, LIONCUB_ERR_ARG, "grads and out_dev must be non-NULL");
    if (reinterpret_cast<uintptr_t>(out_dev) & 7u)
        return fail(h, LIONCUB_ERR_ALIGN, "out_dev is not 8-byte aligned");
    for (int i = 0; i < h->W; ++i) {
        if (!grads[i])
            return fail(h, LIONCUB_ERR_ARG, "grads[%d] is NULL", i);
        if (!aligned16(grads[i]))
            return fail(h, LIONCUB_ERR_ALIGN, "grads[%d] is not 16-byte aligned", i);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NvtxRange range("lioncub_diagnose");
    const StepArgs a = make_args(h, grads);
    const bool l1 = h->mode == LIONCUB_MODE_L1_INTSUM;
    cudaError_t e = cudaMemsetAsync(out_dev, 0, static_cast<size_t>(h->K) * sizeof(lioncub_diag), s);
    if (e != cudaSuccess)
        return cuda_fail(h, e, "diagnostics reset");
    if (l1) {
        e = lc::launch_m1_partial(a, h->grad_dtype, s);
        if (e == cudaSuccess)
            e = lc::launch_m1_finalize(a, s);
        if (e != cudaSuccess)
            return cuda_fail(h, e, "diagnostics M1 launch");
    }
    h->prof_this_call = h->prof_steps_left > 0;
    const int slot = prof_begin(h, LIONCUB_KERNEL_DIAGNOSE, s);
    e = lc::launch_diagnose(a, h->grad_dtype, l1 ? 1 : 0, out_dev, s);
    prof_end(h, slot, s);
    if (e != cudaSuccess)
        return cuda_fail(h, e, "diagnose launch");
    return LIONCUB_OK;
}

int lioncub_diagnose_qinf(lioncub_t h, const void* const* grads, int nbits, uint64_t seed, lioncub_qinf_diag* out_dev,
                          lioncub_stream_t stream)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (h->dist)
        return fail(h, LIONCUB_ERR_STATE, "diagnostics need every worker on one GPU (not a data-parallel handle)");
    if (!h->bound)
        return fail(h, LIONCUB_ERR_STATE, "lioncub_bind_state has not been called");
    if (!grads || !out_dev)
        return fail(h, LIONCUB_ERR_ARG, "grads and out_dev must be non-NULL");
    if (nbits != 2 && nbits != 4 && nbits != 8)
        return fail(h, LIONCUB_ERR_ARG, "nbits must be 2, 4 or 8 (got %d)", nbits);
    if (reinterpret_cast<uintptr_t>(out_dev) & 7u)
        return fail(h, LIONCUB_ERR_ALIGN, "out_dev is not 8-byte aligned");
    for (int i = 0; i < h->W; ++i) {
        if (!grads[i])
            return fail(h, LIONCUB_ERR_ARG, "grads[%d] is NULL", i);
        if (!aligned16(grads[i]))
            return fail(h, LIONCUB_ERR_ALIGN, "grads[%d] is not 16-byte aligned", i);
    }
    if (!h->maxabs) {
        const cudaError_t e = dev_alloc(h, &h->maxabs, static_cast<size_t>(h->W) * h->K);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(h, e == cudaErrorMemoryAllocation ? LIONCUB_ERR_OOM : LIONCUB_ERR_CUDA,
                        "Q_inf scratch allocation failed");
        }
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NvtxRange range("lioncub_diagnose_qinf");
    StepArgs a = make_args(h, grads);
    a.qinf_step = h->t;
    cudaError_t e = cudaMemsetAsync(out_dev, 0, static_cast<size_t>(h->K) * sizeof(lioncub_qinf_diag), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(h->maxabs, 0, static_cast<size_t>(h->W) * h->K * sizeof(float), s);
    if (e == cudaSuccess)
        e = lc::launch_diagnose_qinf(a, h->grad_dtype, nbits, h->maxabs, seed, out_dev, s);
    if (e != cudaSuccess)
        return cuda_fail(h, e, "Q_inf diagnostics");
    return LIONCUB_OK;
}

int lioncub_profile(lioncub_t h, int max_steps)
{
    if (!h)
        return LIONCUB_ERR_ARG;
    if (max_steps < 0)
        return fail(h, LIONCUB_ERR_ARG, "max_steps must be >= 0");
    drop_profile(h);
    if (max_steps == 0)
        return LIONCUB_OK;
    // one slot per kernel of a step, plus room for diagnose calls in between
    const int launches = max_steps * (LIONCUB_KERNEL_COUNT + 1);
    h->prof_events.resize(2 * static_cast<size_t>(launches));
    h->prof_kernel.assign(launches, -1);
    for (size_t i = 0; i < h->prof_events.size(); ++i) {
        cudaError_t e = cudaEventCreate(&h->prof_events[i]);
        if (e != cudaSuccess) {
            h->prof_events.resize(i);
            drop_profile(h);
            return cuda_fail(h, e, "event creation");
        }
    }
    h->prof_capacity = launches;
    h->prof_steps_left = max_steps;
    return LIONCUB_OK;
}

int lioncub_profile_read(lioncub_t h, int kernel, double* total_ms, int64_t* launches)
{
    if (!h || !total_ms || !launches)
        return LIONCUB_ERR_ARG;
    double tot = 0.0;
    int64_t n = 0;
    for (int slot = 0; slot < h->prof_used; ++slot) {
        if (h->prof_kernel[slot] != kernel)
            continue;
        cudaError_t e = cudaEventSynchronize(h->prof_events[2 * slot + 1]);
        float ms = 0.0f;
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms, h->prof_events[2 * slot], h->prof_events[2 * slot + 1]);
        if (e != cudaSuccess)
            return cuda_fail(h, e, "reading profile events");
        tot += ms;
        ++n;
    }
    *total_ms = tot;
    *launches = n;
    return LIONCUB_OK;
}

void lioncub_destroy(lioncub_t h)
{
    if (!h)
        return;
    cudaDeviceSynchronize();  // no enqueued step or upload may still use the scratch
    drop_profile(h);
    free_scratch(h);
    delete h;
}

}  // extern "C"
