/*
 * lioncub_oracle.h -- CPU oracle for the compressed Lion update step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of the method, used by the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark to check the CUDA library.  The
 * product path never links, loads or calls it, and it shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources (page title, then the part of the page):
 *   [LC]  "Lion Cub: Minimizing Communication Overhead in Distributed Lion"
 *         (machine review page): "What carries the argument" (update vector
 *         c, 0/1 sign packing, alternating zeros, Eq. (1) L1 quantizer,
 *         global sign, selective momentum sync), "Core claim", the
 *         assumptions list (alternating-sign rule, Fig. 10; sync interval of
 *         10 iterations, Figs. 5 and 8), the Fig. 1 and Fig. 8 captions
 *         (1-bit and p-bit allreduce) and the quoted body text on tied
 *         majority votes.
 *   [DL]  "Communication Efficient Distributed Training with Distributed
 *         Lion" (summary page): "Approach" (per-worker Lion state, sign of
 *         the local update, Avg or MaVo aggregation).
 *   Textbook Lion (Chen et al. 2023, cited by both pages) for the theta and
 *   momentum rules, which the pages do not print.
 *
 * Arithmetic: every float operation is one IEEE fp32 operation rounded to
 * nearest-even; the file is compiled with -ffp-contract=off so no multiply
 * and add are fused.  M1 is accumulated in fp64.
 *
 * Parity unpinned: the last bits of M1 where the fp64 sum order matters
 * (the oracle sums in index order; nothing on the pages fixes an order),
 * and L1 codes at near-ties that follow from those bits.
 */
#ifndef LIONCUB_ORACLE_H
#define LIONCUB_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One tensor of the flat parameter vector: elements [offset, offset+numel). */
typedef struct {
    int64_t offset;
    int64_t numel;
    uint32_t flags; /* bit 0: this tensor's momentum is averaged across workers */
} lco_tensor;

#define LCO_TENSOR_SYNC_M 1u

#define LCO_MODE_SIGN 0  /* 1-bit sign, majority vote                       */
#define LCO_MODE_L1 1    /* n-bit L1 quantization, integer sum               */

#define LCO_GRAD_BF16 0
#define LCO_GRAD_F32 1

#define LCO_FLAG_TIE_ALTERNATE 0x100u /* a tied vote takes the step's zero sign */
#define LCO_FLAG_AVERAGE 0x200u       /* D-Lion Avg: update = vote sum / W     */

/* omega = 1 - beta in fp32 (one rounding). */
float lco_omega(float beta);

/* c = beta1*m + omega1*g, each product and the sum rounded to fp32. */
float lco_update_vector(float m, float g, float beta1, float omega1);

/* m' = beta2*m + omega2*g, each product and the sum rounded to fp32. */
float lco_momentum(float m, float g, float beta2, float omega2);

/* The transmitted bit of c at step t: 1 for +1, 0 for -1; an exact zero is
 * +1 on even t and -1 on odd t. */
int lco_sign_bit(float c, int64_t t);

/* Pack the sign bits of c[0..n) LSB-first, 32 per word; words[] gets
 * ceil(n/32) entries and unused high bits of the last word are 0. */
void lco_pack_signs(const float* c, int64_t n, int64_t t, uint32_t* words);

/* Mean absolute value of c[0..n): fp64 sum in index order, fp64 division by
 * n, one rounding to fp32.  n == 0 gives 0. */
float lco_m1(const float* c, int64_t n);

/* Eq. (1): q = clamp(round(qmax * c / M1), -qmax, qmax), qmax = 2^(n-1)-1,
 * with the scale taken once as inv = qmax / M1 (fp32) and round() ties to
 * even.  M1 == 0 gives all-zero codes. */
void lco_q1(const float* c, int64_t n, int nbits, float m1, int8_t* q);

/* Pack n-bit two's-complement codes, 32/nbits per word, LSB-first;
 * words[] gets ceil(n*nbits/32) entries and unused high bits are 0. */
void lco_pack_codes(const int8_t* q, int64_t n, int nbits, uint32_t* words);

/* The sign-mode aggregate of element e: sum over workers of +1 (bit set) or
 * -1 (bit clear). */
int32_t lco_vote(const uint32_t* const* words, int W, int64_t e);

/* The L1-mode aggregate of element e: sum over workers of the decoded code. */
int32_t lco_code_sum(const uint32_t* const* words, int W, int nbits, int64_t e);

/* The update direction u from an aggregate: sign(agg) in {-1,0,+1}; with
 * LCO_FLAG_TIE_ALTERNATE a zero becomes +1 on even t and -1 on odd t; with
 * LCO_FLAG_AVERAGE it is agg / W (sign mode only). */
float lco_direction(int32_t agg, int W, uint32_t flags, int64_t t);

/* theta' = theta - lr*(u + wd*theta), one fp32 rounding per operation. */
float lco_apply(float theta, float u, float lr, float wd);

/* Average m_0..m_{W-1} over [lo, hi): s = m_0; s += m_j (j = 1..W-1) in
 * fp32; every m_i[e] = s / W. */
void lco_sync_average(float* const* m, int W, int64_t lo, int64_t hi);

/*
 * One full step at 0-based step index t, in the order: update vectors and
 * compression for every worker and tensor; aggregation; theta; momentum;
 * momentum sync on flagged tensors when sync_interval > 0 and
 * (t + 1) % sync_interval == 0.
 *
 * grads[i] points at d bf16 (as uint16 bit patterns) or fp32 values.
 * theta (d) and m[i] (d each) are updated in place.
 * Optional outputs (NULL to skip):
 *   wire_out[i]: worker i's packed words (ceil(d/32) in sign mode,
 *                ceil(d*nbits/32) in L1 mode);
 *   m1_out:      W*K floats, [i*K + k] (L1 mode only);
 *   agg_out:     d int32 aggregates.
 * layout may be NULL with K == 0, meaning one tensor covering [0, d).
 * Returns 0, or -1 for invalid arguments, -2 for an allocation failure.
 */
int lco_step(int64_t d, int W, const lco_tensor* layout, int K,
             float beta1, float beta2, float lr, float wd,
             int mode, int nbits, uint32_t flags, int sync_interval, int64_t t,
             int grad_dtype, const void* const* grads,
             float* theta, float* const* m,
             uint32_t* const* wire_out, float* m1_out, int32_t* agg_out);

/*
 * Diagnostics of one step (the pages' own measurements), computed from the
 * state before the step and the step's gradients; nothing is updated.
 * Per element: u_q = sign of the update direction the step would apply
 * (lco_direction of the method's aggregate); u_fp = sign of the full-
 * precision sum s = c_0 + c_1 + ... + c_{W-1} (fp32, in worker order).
 *   match:    u_q == u_fp
 *   flip:     u_q == -u_fp != 0
 *   dropped:  u_q == 0 != u_fp
 *   spurious: u_fp == 0 != u_q
 *   ties:     elements whose aggregate is exactly 0
 * max_std_m: the largest, over the tensor's elements, inter-worker standard
 * deviation of the momentum: mean = (sum_i m_i) / W, var = (sum_i
 * (m_i - mean)^2) / W, both sums in worker order in fp32, std = sqrt(var).
 * [LC] Fig. 4 / Fig. 11 captions (sign match and flip rates of quantized
 * updates), Fig. 6 caption (maximum inter-worker standard deviation per
 * layer), the quoted body text on tied votes.
 */
typedef struct {
    int64_t match, flip, dropped, spurious, ties;
    float max_std_m;
    uint32_t pad;
} lco_diag;

/* Inter-worker standard deviation of values x_0..x_{W-1} (as above). */
float lco_worker_std(const float* x, int W);

/* Classify one element: returns 0 match, 1 flip, 2 dropped, 3 spurious. */
int lco_classify(float u_q, float u_fp);

/* Diagnostics for every tensor (out[k], K entries; layout NULL/K = 0 means
 * one tensor).  Arguments as in lco_step.  Returns 0, -1 or -2 as lco_step. */
int lco_diagnose(int64_t d, int W, const lco_tensor* layout, int K,
                 float beta1, int mode, int nbits, uint32_t flags, int64_t t,
                 int grad_dtype, const void* const* grads, const float* const* m,
                 lco_diag* out);

/*
 * The max-norm quantizer with stochastic rounding that the pages compare L1
 * quantization against ([LC] "Core claim": the standard max-norm quantizer
 * Q_inf turns most entries of Lion's heavy-tailed update into zeros; the
 * Fig. 4 caption: its stochastic codes are mostly zero, so few signs match or
 * flip; the referee report: Q_inf uses stochastic
 * rounding).  The pages do not print it; the reading here:
 *   M_inf = max |c| over the tensor (per worker), inv = qmax / M_inf in fp32
 *   (0 when M_inf == 0), y = |c| * inv in fp32, q = floor(y) + (u < y -
 *   floor(y) ? 1 : 0), clamped to qmax, with the sign of c; qmax = 2^(n-1)-1.
 * u is uniform in [0, 1): the top 24 bits of one SplitMix64 output times
 * 2^-24 (lco_qinf_uniform).
 */

/* SplitMix64 (Steele, Lea and Flood 2014): output number k (k = 0, 1, ...)
 * of the generator whose state starts at `seed` (state += 0x9e3779b97f4a7c15
 * before each output, which is the state passed through the mixing
 * function). */
uint64_t lco_splitmix64(uint64_t seed, uint64_t k);

/* The uniform of element e (index in the flat parameter vector, < 2^40) of
 * worker `worker` (< 256) at step t: SplitMix64 output number
 * (t mod 2^16) * 2^48 + worker * 2^40 + e from `seed`, top 24 bits * 2^-24. */
float lco_qinf_uniform(uint64_t seed, int64_t t, int worker, int64_t e);

/* max |c[e]| over [0, n); 0 for n == 0. */
float lco_maxabs(const float* c, int64_t n);

/* Q_inf codes of c[0..n) for worker `worker` at step t; c[e] is element
 * e_first + e of the flat vector. */
void lco_qinf(const float* c, int64_t n, int nbits, float maxabs, uint64_t seed, int64_t t, int worker,
              int64_t e_first, int8_t* q);

/* Per-tensor comparison of the Q_inf aggregate with the full-precision
 * update: every worker's Q_inf codes (nbits, its own M_inf per tensor) are
 * summed in worker order; u_q = sign of lco_direction(sum, W, flags without
 * the average, t); u_fp and the categories as in lco_diagnose; zero_codes
 * counts the (worker, element) codes equal to 0.  e_base is the flat index
 * of element 0 of the vector passed (tensors start at e_base + offset). */
typedef struct {
    int64_t match, flip, dropped, spurious, zero_codes;
} lco_qinf_diag;

int lco_diagnose_qinf(int64_t d, int W, const lco_tensor* layout, int K, float beta1, int nbits, uint32_t flags,
                      int64_t t, uint64_t seed, int64_t e_base, int grad_dtype, const void* const* grads,
                      const float* const* m, lco_qinf_diag* out);

#ifdef __cplusplus
}
#endif
#endif
