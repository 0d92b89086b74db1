/*
 * lioncub.h -- C ABI of the GB300 library for the compressed Lion update step
 * of Lion Cub / Distributed Lion, with W data-parallel workers simulated as W
 * gradient and momentum buffers resident in one GPU's memory.
 *
 * Sources (page title, then the part of the page):
 *   [LC] "Lion Cub: Minimizing Communication Overhead in Distributed Lion"
 *        (machine review page): "What carries the argument" -- the update
 *        vector c_{i,t} = beta1 m_{i,t-1} + (1-beta1) grad f_i(theta_{t-1}),
 *        signs packed as 0/1 with exact zeros sent as +1/-1 on alternating
 *        iterations, the L1 quantizer of Eq. (1)
 *        Q1(x) = clamp(round((2^(n-1)-1) x / M1(x)), 2^(n-1)-1) with M1 the
 *        mean absolute value, a quantized sum followed by a global sign, and
 *        momentum synchronized only on the input-embedding and output
 *        layers; the Fig. 1 and Fig. 8 captions (1-bit and p-bit allreduce);
 *        the assumptions list (sync every 10 iterations).
 *   [DL] "Communication Efficient Distributed Training with Distributed
 *        Lion" (summary page): "Approach" -- each worker keeps its own Lion
 *        momentum and sends the sign of its local update; the aggregate is
 *        the majority vote (MaVo) or the average (Avg).
 *   The theta and momentum rules are textbook Lion (Chen et al. 2023), which
 *   both pages cite.
 *
 * One step, with t the 0-based step index:
 *   c_i   = RN(RN(beta1*m_i) + RN(omega1*g_i)),  omega1 = RN(1 - beta1)
 *   sign mode:  bit_i = 1 if c_i > 0, 0 if c_i < 0, (t even ? 1 : 0) if c_i == 0
 *               agg = sum_i (2*bit_i - 1)                      in [-W, W]
 *   L1 mode:    M1_{i,k} = mean over tensor k of |c_i| (fp64 sum, one
 *               rounding to fp32); inv = RN(qmax / M1);
 *               q_i = clamp(rint(RN(c_i*inv)), -qmax, qmax), qmax = 2^(n-1)-1
 *               (q = 0 where M1 == 0); agg = sum_i q_i
 *   u     = sign(agg) in {-1, 0, +1}  (ties give 0); with
 *           LIONCUB_FLAG_TIE_ALTERNATE a tie gives t even ? +1 : -1; with
 *           LIONCUB_FLAG_AVERAGE (sign mode only) u = RN(agg / W)
 *   theta = RN(theta - RN(lr * RN(u + RN(wd*theta))))
 *   m_i   = RN(RN(beta2*m_i) + RN(omega2*g_i)),  omega2 = RN(1 - beta2)
 *   sync: on tensors flagged LIONCUB_TENSOR_SYNC_M, when sync_interval > 0
 *         and (t+1) % sync_interval == 0: s = m_0; s = RN(s + m_j) for
 *         j = 1..W-1; every m_i = RN(s / W)
 *   t     = t + 1
 * RN is one IEEE fp32 rounding to nearest-even; no multiply-add is fused.
 *
 * Wire format (what a real worker would send): sign mode packs element e of
 * worker i into bit e%32 of word e/32 (LSB first, 1 = +1); L1 mode packs
 * two's-complement n-bit codes, 32/n per word, element e in field e%(32/n)
 * of word e*n/32.  Bits past d are 0.
 *
 * A handle is not thread-safe: calls on one handle must not overlap.  Calls
 * on different handles may run concurrently.
 *
 * Return codes: LIONCUB_OK (0) or a negative LIONCUB_ERR_*.  After an error,
 * lioncub_last_error(h) describes it.  Kernel faults are asynchronous: they
 * surface as LIONCUB_ERR_CUDA at a later call or at the caller's stream
 * synchronization.  No call synchronizes the device except the ones marked
 * "synchronizes".
 *
 * Fault injection for tests (environment variables, read by lioncub_create
 * for the handle it creates; unset, they cost nothing):
 *   LIONCUB_FAIL_ALLOC=k   the handle's k-th device allocation (lioncub_create's
 *                          first, then lioncub_step_host's staging) fails as
 *                          out of memory;
 *   LIONCUB_FAIL_LAUNCH=k  the handle's k-th step kernel launch reports
 *                          cudaErrorLaunchOutOfResources without launching;
 *   LIONCUB_POISON_GUARD=1 one byte of the guard band after the wire buffer is
 *                          overwritten at creation, so the next status export
 *                          reports LIONCUB_STATUS_GUARD;
 *   LIONCUB_WAIT_POLLS=k   the first wait of the staged reduce (for the bulk
 *                          copies of its wire bytes) gives up after k
 *                          non-blocking polls (k <= 65535) instead of its
 *                          normal bound, as a wait that runs out would: the
 *                          block sets LIONCUB_STATUS_WAIT_TIMEOUT, still waits
 *                          (with the normal bound) for its own copies to land,
 *                          and returns without updating its part of theta.
 */
#ifndef LIONCUB_H
#define LIONCUB_H

#include <stddef.h>
#include <stdint.h>

/* Exported entry points keep default visibility even when the library is
 * built with hidden visibility. */
#if defined(__GNUC__)
#define LIONCUB_API __attribute__((visibility("default")))
#else
#define LIONCUB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lioncub_s* lioncub_t;
/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* lioncub_stream_t;

/* One tensor of the flat parameter vector: elements [offset, offset+numel).
 * The tensors of a layout tile [0, d) in order, and every offset is a
 * multiple of 32 elements (so a packed word never spans two tensors). */
typedef struct {
    int64_t offset;
    int64_t numel;
    uint32_t flags; /* LIONCUB_TENSOR_SYNC_M or 0 */
} lioncub_tensor;

enum {
    LIONCUB_TENSOR_SYNC_M = 1 /* average this tensor's momentum across workers */
};

enum {
    LIONCUB_MODE_SIGN_MAJORITY = 0, /* 1-bit signs, majority vote          */
    LIONCUB_MODE_L1_INTSUM = 1,     /* n-bit Eq. (1) codes, integer sum    */
    LIONCUB_FLAG_TIE_ALTERNATE = 0x100, /* OR into mode: tie -> step's zero sign */
    LIONCUB_FLAG_AVERAGE = 0x200        /* OR into mode: D-Lion Avg, u = agg/W  */
};

enum { LIONCUB_GRAD_BF16 = 0, LIONCUB_GRAD_F32 = 1 };

enum {
    LIONCUB_OK = 0,
    LIONCUB_ERR_ARG = -1,   /* invalid argument                                 */
    LIONCUB_ERR_ALIGN = -2, /* offset not a multiple of 32 / pointer not 16-byte */
    LIONCUB_ERR_STATE = -3, /* state not bound, or call out of order            */
    LIONCUB_ERR_OOM = -4,   /* device or host allocation failed                 */
    LIONCUB_ERR_CUDA = -5   /* a CUDA call or launch failed                     */
};

enum { LIONCUB_MAX_WORKERS = 128 };

/* What lioncub_debug_export copies. */
enum {
    LIONCUB_EXPORT_WIRE = 0, /* W x lioncub_wire_words() uint32: last step's packed words/codes */
    LIONCUB_EXPORT_M1 = 1,   /* W x K float: last step's M1 (L1 mode)               */
    LIONCUB_EXPORT_AGG = 2,  /* d int32: the aggregate of the last step's wire words */
    LIONCUB_EXPORT_STATUS = 3 /* 1 int32 of LIONCUB_STATUS_* bits, 0 when all is well */
};

/* Bits of the device status word (sticky until lioncub_destroy). */
enum {
    LIONCUB_STATUS_WAIT_TIMEOUT = 1,  /* a kernel's bounded wait for its own bulk copies gave
                                         up; that step's theta is invalid                */
    LIONCUB_STATUS_OUT_OF_BOUNDS = 2, /* bounds-checked builds only: a kernel computed an
                                         index outside its buffer and skipped the access  */
    LIONCUB_STATUS_GUARD = 4          /* a guard band around the library's scratch buffers
                                         was overwritten (checked at each status export) */
};

/* Per-tensor diagnostics of a step (lioncub_diagnose), 48 bytes. */
typedef struct {
    int64_t match;    /* elements whose applied sign equals the full-precision sign */
    int64_t flip;     /* applied sign is the opposite, both non-zero                */
    int64_t dropped;  /* applied sign 0, full-precision sign non-zero               */
    int64_t spurious; /* applied sign non-zero, full-precision sign 0               */
    int64_t ties;     /* elements whose aggregate is exactly 0                      */
    float max_std_m;  /* max over the tensor of the inter-worker std of m           */
    uint32_t reserved;
} lioncub_diag;

/* Kernels whose launches lioncub_profile_read reports. */
enum {
    LIONCUB_KERNEL_COMPRESS = 0,     /* c, sign bits or Q1 codes, momentum, sync */
    LIONCUB_KERNEL_M1 = 1,           /* per-tile compensated sums of |c| (L1)   */
    LIONCUB_KERNEL_M1_FINAL = 2,     /* per-tensor M1 and 1/M1 scale (L1 mode)   */
    LIONCUB_KERNEL_REDUCE_APPLY = 3, /* W-way vote / integer sum, sign, theta    */
    LIONCUB_KERNEL_DIAGNOSE = 4,     /* lioncub_diagnose's counting pass          */
    LIONCUB_KERNEL_COUNT = 5
};

/*
 * Source: [DL] "Approach" (W workers, each with its own Lion state) and [LC]
 * "What carries the argument" (the compression choices and the layers whose
 * momentum is synchronized).
 * Create a handle for d parameters, W workers (1..LIONCUB_MAX_WORKERS) and a
 * layout of K tensors (layout may be NULL with K == 0: one tensor [0, d)).
 * mode: LIONCUB_MODE_* optionally OR'ed with LIONCUB_FLAG_*.  nbits: 2, 4 or
 * 8 in L1 mode (ignored in sign mode).  grad_dtype: LIONCUB_GRAD_*.
 * sync_interval: 0 = never sync, else sync flagged tensors every
 * sync_interval steps.  The library allocates its own device scratch (wire
 * words or codes, M1 partials, tile table) here and frees it in
 * lioncub_destroy; the caller's layout array is copied.  Errors: ERR_ARG,
 * ERR_ALIGN, ERR_OOM, ERR_CUDA (*out is set to NULL).  Uses the current
 * CUDA device, which must stay current for every later call on the handle.
 * Synchronizes the legacy default stream once, at the end, so the tables it
 * uploaded are in place before a step on any stream reads them.
 */
LIONCUB_API int lioncub_create(lioncub_t* out, int64_t d, int W, const lioncub_tensor* layout, int K,
                   float beta1, float beta2, float lr, float wd, int mode, int nbits,
                   int grad_dtype, int sync_interval);

/*
 * Source: [DL] "Approach" (each worker keeps its own Lion momentum; the
 * parameters are shared) and [LC] "What carries the argument" (m_{i,t-1} in
 * the update vector of worker i).
 * Bind the optimizer state: theta (d fp32, device) and m[0..W-1] (W device
 * pointers to d fp32 each; the host array is read during the call only).
 * The caller owns the memory and keeps it alive while the handle uses it.
 * Every pointer must be 16-byte aligned (ERR_ALIGN), non-NULL (ERR_ARG).
 */
LIONCUB_API int lioncub_bind_state(lioncub_t h, float* theta, float* const* m);

/*
 * Source: the whole step at the top of this header -- [LC] "What carries the
 * argument" (c, 0/1 signs with alternating zeros, Eq. (1), the quantized sum
 * and its global sign, selective momentum sync) with textbook Lion for theta
 * and m; [DL] "Approach" for the majority vote and the average.
 * Enqueue one step on `stream`: grads[0..W-1] are W device pointers to d
 * gradients of the handle's dtype, 16-byte aligned; the host array is read
 * during the call only, the device buffers must stay unchanged until the
 * step has run.  theta and m are updated in place; the step counter advances
 * only if every launch was enqueued.  Launch order: (L1 mode: M1 pass, M1
 * combine,) compress (writes the wire and m), reduce_apply (writes theta).
 * If the compress launch or one before it fails, theta and m are unchanged
 * and the step can be retried; if reduce_apply fails, m has already moved,
 * so restore the state from a checkpoint.  Errors: ERR_STATE (unbound),
 * ERR_ARG, ERR_ALIGN, ERR_CUDA.  Does not synchronize.
 */
LIONCUB_API int lioncub_step(lioncub_t h, const void* const* grads, lioncub_stream_t stream);
/* lioncub_step only enqueues kernels (no allocation, no synchronization), so
 * it can be captured into a CUDA graph.  The step counter advances when the
 * step is enqueued and its parity is baked into the captured kernels (the
 * sign of exact zeros, and the sync steps), so a loop with fixed gradient
 * buffers captures an even and an odd step and replays them alternately. */

/*
 * The same step fed from host memory: copies grads_host[0..W-1] (W host
 * buffers of d gradients; page-locked memory gives full copy speed) into
 * library-owned device staging, runs the step on `stream`, and copies the
 * updated theta into theta_host_out (d floats, host) on `stream`.  When
 * `stream` has completed the call's work, theta_host_out holds the result
 * and grads_host may be reused; the host buffers must stay valid until then.
 * The uploads run on an internal non-blocking stream into one of two staging
 * buffers (allocated on the first call, kept until destroy; one if memory is
 * short), so the next call's upload overlaps this call's kernels and theta
 * download; `stream` waits for the upload before the step's kernels.  When
 * theta_host_out is page-locked memory mapped into the device's address
 * space (e.g. from cudaHostAlloc) and 16-byte aligned, SM threads store theta
 * into it, leaving the copy engine to the uploads; otherwise it is copied.
 * Errors as lioncub_step, plus ERR_OOM for the staging.
 */
LIONCUB_API int lioncub_step_host(lioncub_t h, const void* const* grads_host, float* theta_host_out,
                      lioncub_stream_t stream);

/*
 * Page-locked host memory for lioncub_step_host's buffers: `bytes` bytes,
 * mapped into every device's address space, allocated directly by the CUDA
 * runtime (no caching allocator in between), so that uploads from it and
 * theta stores into it run at the host link's full rate.  *out is set to
 * NULL when bytes == 0.  The memory stays valid until lioncub_host_free.
 * Errors: ERR_ARG (out NULL), ERR_OOM, ERR_CUDA (messages via
 * lioncub_last_error(NULL)).
 * lioncub_host_free releases it (NULL is a no-op); it synchronizes the device.
 */
LIONCUB_API int lioncub_host_alloc(void** out, size_t bytes);
LIONCUB_API void lioncub_host_free(void* p);

/* Learning rate of later steps (textbook Lion's lr). */
LIONCUB_API int lioncub_set_lr(lioncub_t h, float lr);
/* Step counter t (the parity of t decides the sign of an exact zero: [LC]
 * "What carries the argument", alternating iterations).  Saving theta, the
 * W momenta and t, then restoring them into a new handle resumes the run
 * bit for bit. */
LIONCUB_API int lioncub_get_step(lioncub_t h, int64_t* t);
LIONCUB_API int lioncub_set_step(lioncub_t h, int64_t t);

/* Source: [LC] "What carries the argument" (signs packed as 0/1) and the
 * Fig. 1 / Fig. 8 captions (1-bit and p-bit containers): the size of what one
 * worker would send.
 * Words per worker of the wire buffer: ceil(d/32) in sign mode, ceil(d*n/32)
 * in L1 mode; -1 for a NULL handle. */
LIONCUB_API int64_t lioncub_wire_words(lioncub_t h);

/*
 * Source: the wire format of [LC] "What carries the argument" and Fig. 1 /
 * Fig. 8 captions (packed 0/1 signs, p-bit integer containers); M1 of Eq. (1).
 * Copy diagnostic data of the last step into dst_dev (device memory the
 * caller owns; sizes in the LIONCUB_EXPORT_* comments) on `stream`.  For
 * LIONCUB_EXPORT_AGG a kernel recomputes the aggregate from the wire words;
 * for LIONCUB_EXPORT_STATUS a kernel first checks the guard bands (256
 * bytes before and after each of the wire, M1-partial, M1 and 1/M1
 * buffers).  For tests; never part of a timed step.
 */
LIONCUB_API int lioncub_debug_export(lioncub_t h, int what, void* dst_dev, lioncub_stream_t stream);

/*
 * The pages' own measurements for the step that `grads` would drive, from
 * the current state; nothing is updated and the step counter does not move.
 * "Lion Cub" Fig. 4 / Fig. 11 (whether quantized update signs match or flip
 * against the full-precision update), Fig. 6 (maximum inter-worker standard
 * deviation of the momentum per layer) and the share of tied majority votes.
 * Per element, the applied sign is the sign of the direction the step would
 * use (global sign of the vote or code sum, with the tie rule); the
 * full-precision sign is that of s = c_0 + ... + c_{W-1} (fp32, worker
 * order).  The momentum spread uses mean = (sum m_i)/W and var =
 * (sum (m_i - mean)^2)/W in fp32, std = sqrt(var).  out_dev: K lioncub_diag
 * in device memory the caller owns, zeroed and filled on `stream`.  In L1
 * mode the M1 pass runs first and replaces the M1 that LIONCUB_EXPORT_M1
 * returns.  Errors: ERR_STATE (unbound), ERR_ARG, ERR_ALIGN, ERR_CUDA.
 */
LIONCUB_API int lioncub_diagnose(lioncub_t h, const void* const* grads, lioncub_diag* out_dev,
                                 lioncub_stream_t stream);

/*
 * The max-norm quantizer the pages compare Eq. (1) against, as a comparator
 * of the same kind: [LC] "Core claim" (the standard max-norm quantizer Q_inf
 * turns most entries of Lion's heavy-tailed update into zeros), the Fig. 4
 * caption (its stochastic codes are mostly zero, so few signs match or
 * flip) and the referee report (Q_inf rounds
 * stochastically).  The pages do not print Q_inf; this library reads it as:
 * per (worker, tensor) M_inf = max |c|, inv = RN(qmax / M_inf) (0 when
 * M_inf == 0), y = RN(|c| * inv), code = floor(y) + (u < y - floor(y) ? 1 :
 * 0), clamped to qmax = 2^(nbits-1) - 1, with the sign of c; u is the top 24
 * bits of SplitMix64 (Steele, Lea and Flood 2014) output number
 * (t mod 2^16) * 2^48 + i * 2^40 + e of the generator started from `seed`,
 * times 2^-24 (t the handle's step counter, i the worker, e the element's
 * flat index).  The codes of the W workers are summed in order, and the
 * sign of the sum (ties by the handle's tie rule; never the average) is
 * compared, per element, with the sign of the full-precision sum of c as in
 * lioncub_diagnose.  Nothing is updated.  out_dev: K records in device memory
 * the caller owns, 8-byte aligned, zeroed and filled on `stream`.  nbits: 2,
 * 4 or 8, whatever the handle's mode.  Errors: ERR_STATE (unbound, or a
 * data-parallel handle), ERR_ARG, ERR_ALIGN, ERR_OOM (its W x K scratch is
 * allocated on the first call), ERR_CUDA.
 */
typedef struct {
    int64_t match, flip, dropped, spurious;
    int64_t zero_codes; /* (worker, element) codes equal to 0 */
} lioncub_qinf_diag;
LIONCUB_API int lioncub_diagnose_qinf(lioncub_t h, const void* const* grads, int nbits, uint64_t seed,
                                      lioncub_qinf_diag* out_dev, lioncub_stream_t stream);

/*
 * Per-kernel timing with CUDA events on the step's stream.  lioncub_profile
 * (h, n) records an event pair around every kernel launch of the next n
 * lioncub_step calls (and of lioncub_diagnose calls made while steps remain
 * to be recorded); n == 0 turns recording off and drops the records.  lioncub_profile_read
 * (synchronizes on the recorded events) gives, for one LIONCUB_KERNEL_*, the
 * summed milliseconds and the number of launches recorded.
 */
LIONCUB_API int lioncub_profile(lioncub_t h, int max_steps);
LIONCUB_API int lioncub_profile_read(lioncub_t h, int kernel, double* total_ms, int64_t* launches);

/* Source: none on the pages (they define no interface); error reporting
 * follows the ownership rule above -- the caller owns its buffers and the
 * stream, the library owns its scratch and its messages.
 * Message for the last error on h (never NULL; "" when none).  The string
 * belongs to the library and stays valid until the next call on h.  With
 * h == NULL: the message of the last failed handle-less call on this thread
 * (lioncub_create, lioncub_host_alloc, lioncub_sign_step_noalloc); each of
 * those clears it when it succeeds, so read it right after a non-OK return. */
LIONCUB_API const char* lioncub_last_error(lioncub_t h);
/* Static name of a LIONCUB_* return code. */
LIONCUB_API const char* lioncub_strerror(int code);

/*
 * ---- Data-parallel exchange: the W workers spread over several ranks ----
 *
 * Source: [LC] the quoted body text on the implementation (1-bit Lion Cub
 * exchanges its packed signs with an AlltoAll; the 4-bit and wider variants
 * sum their codes with an AllReduce), "What carries the argument" (an
 * allreduce of 1-bit words built for the majority vote: each worker's packed
 * signs are split into chunks, the owner of a chunk takes its vote, the
 * result is gathered back; momentum averaged on the input-embedding and
 * output layers) and the Fig. 1 / Fig. 8 captions.
 *
 * N ranks (one GPU each) hold W/N workers each -- rank r the global workers
 * r*W/N .. (r+1)*W/N - 1 -- and each a copy of theta.  The library does
 * every arithmetic step in its kernels; the caller's collective library
 * (NCCL, for example through torch.distributed) moves the exchange buffers
 * between the three calls of a step, on the same stream:
 *
 *   sign mode:  lioncub_dist_compress      (wire words -> SEND, chunk-major)
 *               all-to-all SEND -> RECV    (equal segments of bytes[SEND]/N:
 *                                           segment r goes to rank r, and the
 *                                           segment from rank s lands at
 *                                           segment s of RECV)
 *               lioncub_dist_reduce        (vote of this rank's chunk ->
 *                                           DIR_CHUNK)
 *               allgather DIR_CHUNK -> DIR_ALL (rank order)
 *               [sync step: allgather SYNC_SEND -> SYNC_RECV (rank order)]
 *               lioncub_dist_apply         (theta, synchronized momenta)
 *   L1 mode:    lioncub_dist_compress      (M1, codes of the local workers)
 *               lioncub_dist_reduce        (their code sum -> AGG, int8 or
 *                                           int32 per element, see agg_bytes)
 *               allreduce (sum) of AGG in place
 *               [sync step: allgather SYNC_SEND -> SYNC_RECV]
 *               lioncub_dist_apply
 *
 * A sync step is one with sync_interval > 0 and (t+1) % sync_interval == 0
 * for the handle's step counter t before lioncub_dist_apply.  Every rank ends
 * the step with the same theta, and each rank's momenta equal those of the
 * same workers in a single-GPU lioncub_step over all W workers, bit for bit:
 * integer sums do not depend on their order, and the momentum average sums
 * the gathered momenta in worker order on every rank.
 *
 * Sign mode: rank r owns elements [r*chunk, min(d, (r+1)*chunk)); SEND holds
 * N*(W/N) rows of chunk_words words, row (c*(W/N) + i) carrying local worker
 * i's packed signs of chunk c (LSB first, as the single-GPU wire); RECV holds
 * W rows (global worker order) of this rank's chunk.  DIR_CHUNK packs one
 * field per element of the chunk: dir_bits = 2, the two's-complement
 * direction -1, 0 or +1 after the tie rule; dir_bits = 8 (with
 * LIONCUB_FLAG_AVERAGE), the vote sum itself.  DIR_ALL is N such chunks.
 * L1 mode: AGG holds d sums of agg_bytes (1 when W*qmax <= 127, else 4).
 * SYNC_SEND holds, per local worker, the new momenta of the synchronized
 * tensors in layout order, each padded to a multiple of 2048 elements
 * (sync_slots per worker); SYNC_RECV holds W such rows in worker order.
 */
enum {
    LIONCUB_DIST_SEND = 0,
    LIONCUB_DIST_RECV = 1,
    LIONCUB_DIST_DIR_CHUNK = 2,
    LIONCUB_DIST_DIR_ALL = 3,
    LIONCUB_DIST_AGG = 4,
    LIONCUB_DIST_SYNC_SEND = 5,
    LIONCUB_DIST_SYNC_RECV = 6,
    LIONCUB_DIST_BUFFERS = 7
};

typedef struct {
    int64_t chunk;          /* sign mode: elements per rank's chunk (a multiple of 4096) */
    int64_t chunk_words;    /* sign mode: words per worker and chunk (chunk / 32)        */
    int64_t dir_words;      /* sign mode: words of one chunk's directions               */
    int64_t sync_slots;     /* elements per worker in the sync buffers                  */
    int32_t local_workers;  /* W / nranks                                               */
    int32_t first_worker;   /* rank * W / nranks                                        */
    int32_t dir_bits;       /* sign mode: 2, or 8 with the average                      */
    int32_t agg_bytes;      /* L1 mode: 1 (int8) or 4 (int32)                            */
    int64_t bytes[LIONCUB_DIST_BUFFERS]; /* size of each exchange buffer; 0 = unused     */
} lioncub_dist_plan;

/*
 * The exchange plan of rank `rank` of `nranks` for a step of W workers on d
 * parameters (arguments as lioncub_create; W % nranks == 0).  Host
 * arithmetic only: no CUDA call, no device needed.  Errors: ERR_ARG.
 */
LIONCUB_API int lioncub_dist_plan_make(int64_t d, int W, int nranks, int rank, const lioncub_tensor* layout,
                                       int K, int mode, int nbits, int sync_interval, lioncub_dist_plan* out);

/*
 * A handle for rank `rank` of `nranks`, holding the W/nranks local workers
 * (arguments otherwise as lioncub_create).  lioncub_bind_state then takes
 * W/nranks momenta.  The single-GPU lioncub_step, lioncub_step_host,
 * lioncub_diagnose and lioncub_diagnose_qinf refuse such a handle
 * (ERR_STATE).
 */
LIONCUB_API int lioncub_dist_create(lioncub_t* out, int64_t d, int W, int nranks, int rank,
                                    const lioncub_tensor* layout, int K, float beta1, float beta2, float lr,
                                    float wd, int mode, int nbits, int grad_dtype, int sync_interval);

/*
 * Bind the exchange buffers: bufs[LIONCUB_DIST_BUFFERS] device pointers,
 * each at least the plan's bytes[b] (NULL where that is 0), 16-byte aligned,
 * owned by the caller (so that its collective library can register them).
 * Errors: ERR_STATE (not a data-parallel handle), ERR_ARG, ERR_ALIGN.
 */
LIONCUB_API int lioncub_dist_bind_buffers(lioncub_t h, void* const* bufs);

/*
 * The three launches of a step, in this order (ERR_STATE otherwise), with
 * the caller's collectives between them as described above.  compress
 * reads the local gradients (grads: W/nranks device pointers, like
 * lioncub_step); apply advances the step counter.  None synchronizes.
 */
LIONCUB_API int lioncub_dist_compress(lioncub_t h, const void* const* grads, lioncub_stream_t stream);
LIONCUB_API int lioncub_dist_reduce(lioncub_t h, lioncub_stream_t stream);
LIONCUB_API int lioncub_dist_apply(lioncub_t h, lioncub_stream_t stream);

/*
 * Allocation-free sign-mode step.  It has no counterpart on the pages: it is
 * for callers that cannot allocate device memory at the time they run a step
 * -- for example an application whose allocator has reserved all device
 * memory up front, code that must avoid the device synchronization that
 * cudaMalloc/cudaFree can cause, or a plug-in that may only allocate while it
 * is initialised.  It computes the same step as lioncub_step in sign mode
 * (one flat tensor of d elements, majority vote, ties give 0, no momentum
 * sync) at step index t, without a handle: grads[0..W-1], theta and
 * m[0..W-1] are the caller's device buffers (16-byte aligned), as in
 * lioncub_bind_state / lioncub_step; the caller keeps the step counter.
 *
 * The packed sign words live in one array of LIONCUB_NOALLOC_MAX_WORDS
 * uint32 (16 MiB) of the library's static device memory, which every GPU
 * that uses this call keeps until the process exits.  Limit:
 * W * (ceil(d/32) rounded up to a multiple of 4) <= LIONCUB_NOALLOC_MAX_WORDS
 * (for example W = 8 and d up to 16,777,216); larger sizes return
 * LIONCUB_ERR_ARG with a message in lioncub_last_error(NULL).  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Its first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Under CUDA's lazy module loading that first
 * lookup is also what loads the array, i.e. when its 16 MiB are taken from
 * the device: a caller that must not allocate later makes one call with
 * d == 0 (and valid, aligned pointers) on each device while it initialises;
 * that call does the set-up, launches nothing and returns LIONCUB_OK, and
 * later calls allocate nothing.  All calls share the array: each call
 * rewrites every word it reads, so nothing needs clearing, but calls whose
 * kernels overlap on the GPU (other streams, other threads) race on it.
 * Errors: ERR_ARG, ERR_ALIGN, ERR_CUDA (messages via
 * lioncub_last_error(NULL), which the call clears when it starts).  In the
 * bounds-checked build (a debugging aid) each call first reads back, with a
 * synchronous copy, a status word that the previous calls' kernels set on an
 * out-of-range index, and returns ERR_CUDA if it is set.
 */
enum { LIONCUB_NOALLOC_MAX_WORDS = 4194304 };
LIONCUB_API int lioncub_sign_step_noalloc(int64_t d, int W, float beta1, float beta2, float lr, float wd,
                                          int64_t t, int grad_dtype, const void* const* grads, float* theta,
                                          float* const* m, lioncub_stream_t stream);

/* Source: [DL] "Approach" (the per-worker state is the caller's: theta and
 * m stay with the caller, only the library's own scratch is released).
 * Free the handle's scratch and events.  Synchronizes the device first, so
 * no enqueued step still uses the scratch.  NULL is a no-op. */
LIONCUB_API void lioncub_destroy(lioncub_t h);

#ifdef __cplusplus
}
#endif
#endif /* LIONCUB_H */
