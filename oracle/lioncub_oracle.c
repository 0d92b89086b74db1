/*
 * lioncub_oracle.c -- CPU oracle for the compressed Lion update step.
 *
 * TEST INFRASTRUCTURE ONLY: see lioncub_oracle.h.  Plain loops, one
 * element at a time, in the order the method states; compile with
 * -O2 -ffp-contract=off so that every float operation rounds once.
 */
#include "lioncub_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* A bf16 value is the high half of an fp32 bit pattern, so widening is a
 * shift (exact). */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float lco_omega(float beta)
{
    return 1.0f - beta;
}

/* [LC] "What carries the argument": c_{i,t} = beta1 m_{i,t-1} +
 * (1 - beta1) grad f_i(theta_{t-1}). */
float lco_update_vector(float m, float g, float beta1, float omega1)
{
    float a = beta1 * m;
    float b = omega1 * g;
    return a + b;
}

/* Textbook Lion momentum, kept per worker ([DL] "Approach": each worker
 * keeps its own Lion momentum state). */
float lco_momentum(float m, float g, float beta2, float omega2)
{
    float a = beta2 * m;
    float b = omega2 * g;
    return a + b;
}

/* [LC] "What carries the argument": signs packed as 0/1, exact zeros forced
 * to +1 or -1 on alternating iterations; the assumptions list (Fig. 10)
 * names the parities.  Reading: +1 on even t. */
int lco_sign_bit(float c, int64_t t)
{
    if (c > 0.0f)
        return 1;
    if (c < 0.0f)
        return 0;
    return (t % 2 == 0) ? 1 : 0;
}

void lco_pack_signs(const float* c, int64_t n, int64_t t, uint32_t* words)
{
    int64_t nw = (n + 31) / 32;
    for (int64_t w = 0; w < nw; ++w)
        words[w] = 0u;
    for (int64_t e = 0; e < n; ++e) {
        uint32_t bit = (uint32_t)lco_sign_bit(c[e], t);
        words[e / 32] |= bit << (e % 32);
    }
}

/* [LC] Eq. (1): M1 is the mean absolute value. */
float lco_m1(const float* c, int64_t n)
{
    if (n <= 0)
        return 0.0f;
    double s = 0.0;
    for (int64_t e = 0; e < n; ++e)
        s += fabs((double)c[e]);
    return (float)(s / (double)n);
}

/* [LC] Eq. (1): Q1(x) = clamp(round((2^(n-1)-1) x / M1(x)), 2^(n-1)-1). */
void lco_q1(const float* c, int64_t n, int nbits, float m1, int8_t* q)
{
    int qmax_i = (1 << (nbits - 1)) - 1;
    float qmax = (float)qmax_i;
    if (m1 == 0.0f) {
        for (int64_t e = 0; e < n; ++e)
            q[e] = 0;
        return;
    }
    float inv = qmax / m1;
    for (int64_t e = 0; e < n; ++e) {
        float y = c[e] * inv;
        float r = rintf(y); /* default rounding mode: nearest, ties to even */
        if (r != r)
            r = 0.0f;
        if (r > qmax)
            r = qmax;
        if (r < -qmax)
            r = -qmax;
        q[e] = (int8_t)r;
    }
}

/* [LC] Fig. 1 / Fig. 8 captions: the p-bit container carries small integers
 * that are summed. Two's-complement fields, LSB-first. */
void lco_pack_codes(const int8_t* q, int64_t n, int nbits, uint32_t* words)
{
    int64_t per = 32 / nbits;
    int64_t nw = (n * nbits + 31) / 32;
    uint32_t mask = (nbits == 32) ? 0xffffffffu : ((1u << nbits) - 1u);
    for (int64_t w = 0; w < nw; ++w)
        words[w] = 0u;
    for (int64_t e = 0; e < n; ++e) {
        uint32_t field = (uint32_t)(int32_t)q[e] & mask;
        words[e / per] |= field << (nbits * (e % per));
    }
}

/* [LC] "What carries the argument" (a sum of the workers' vectors) and
 * [DL] "Approach" (majority vote): the sum of +1/-1 over workers. */
int32_t lco_vote(const uint32_t* const* words, int W, int64_t e)
{
    int32_t s = 0;
    for (int i = 0; i < W; ++i) {
        uint32_t bit = (words[i][e / 32] >> (e % 32)) & 1u;
        s += bit ? 1 : -1;
    }
    return s;
}

int32_t lco_code_sum(const uint32_t* const* words, int W, int nbits, int64_t e)
{
    int64_t per = 32 / nbits;
    uint32_t mask = (1u << nbits) - 1u;
    int32_t half = 1 << (nbits - 1);
    int32_t s = 0;
    for (int i = 0; i < W; ++i) {
        int32_t f = (int32_t)((words[i][e / per] >> (nbits * (e % per))) & mask);
        if (f >= half)
            f -= 2 * half;
        s += f;
    }
    return s;
}

/* [LC] "What carries the argument": a global sign of the summed vector.
 * A tie is 0 (no update) unless the alternating encoding is asked for.
 * [DL] "Approach": Avg aggregation uses the mean of the worker signs. */
float lco_direction(int32_t agg, int W, uint32_t flags, int64_t t)
{
    if (flags & LCO_FLAG_AVERAGE)
        return (float)agg / (float)W;
    if (agg > 0)
        return 1.0f;
    if (agg < 0)
        return -1.0f;
    if (flags & LCO_FLAG_TIE_ALTERNATE)
        return (t % 2 == 0) ? 1.0f : -1.0f;
    return 0.0f;
}

/* Textbook Lion parameter update with decoupled weight decay. */
float lco_apply(float theta, float u, float lr, float wd)
{
    float a = wd * theta;
    float b = u + a;
    float c = lr * b;
    return theta - c;
}

/* [LC] "What carries the argument" / "Core claim": momentum synchronized
 * only on the input-embedding and output layers; synchronizing means the
 * workers' momenta are replaced by their mean. */
void lco_sync_average(float* const* m, int W, int64_t lo, int64_t hi)
{
    for (int64_t e = lo; e < hi; ++e) {
        float s = m[0][e];
        for (int j = 1; j < W; ++j)
            s = s + m[j][e];
        float avg = s / (float)W;
        for (int i = 0; i < W; ++i)
            m[i][e] = avg;
    }
}

static float load_grad(const void* g, int grad_dtype, int64_t e)
{
    if (grad_dtype == LCO_GRAD_BF16)
        return bf16_bits_to_float(((const uint16_t*)g)[e]);
    return ((const float*)g)[e];
}

int lco_step(int64_t d, int W, const lco_tensor* layout, int K,
             float beta1, float beta2, float lr, float wd,
             int mode, int nbits, uint32_t flags, int sync_interval, int64_t t,
             int grad_dtype, const void* const* grads,
             float* theta, float* const* m,
             uint32_t* const* wire_out, float* m1_out, int32_t* agg_out)
{
    if (d < 0 || W < 1 || !grads || !theta || !m)
        return -1;
    if (mode != LCO_MODE_SIGN && mode != LCO_MODE_L1)
        return -1;
    if (mode == LCO_MODE_L1 && nbits != 2 && nbits != 4 && nbits != 8)
        return -1;
    if (grad_dtype != LCO_GRAD_BF16 && grad_dtype != LCO_GRAD_F32)
        return -1;
    if ((flags & LCO_FLAG_AVERAGE) && (mode != LCO_MODE_SIGN || (flags & LCO_FLAG_TIE_ALTERNATE)))
        return -1;

    lco_tensor whole;
    whole.offset = 0;
    whole.numel = d;
    whole.flags = 0;
    if (!layout || K == 0) {
        layout = &whole;
        K = 1;
    }
    /* The tensors tile [0, d) in order, each starting on a 32-element
     * boundary so that packed words never straddle two tensors. */
    {
        int64_t next = 0;
        for (int k = 0; k < K; ++k) {
            if (layout[k].offset != next || layout[k].numel < 0 || layout[k].offset % 32 != 0)
                return -1;
            next += layout[k].numel;
        }
        if (next != d)
            return -1;
    }

    int bits = (mode == LCO_MODE_SIGN) ? 1 : nbits;
    int64_t nwords = (d * bits + 31) / 32;
    int64_t maxn = 0;
    for (int k = 0; k < K; ++k)
        if (layout[k].numel > maxn)
            maxn = layout[k].numel;

    int rc = 0;
    uint32_t** wire = (uint32_t**)calloc((size_t)W, sizeof(uint32_t*));
    float* c = (float*)malloc((size_t)(maxn > 0 ? maxn : 1) * sizeof(float));
    int8_t* q = (int8_t*)malloc((size_t)(maxn > 0 ? maxn : 1));
    uint32_t* tmpw = (uint32_t*)malloc((size_t)((maxn * bits + 31) / 32 + 1) * sizeof(uint32_t));
    if (!wire || !c || !q || !tmpw) {
        rc = -2;
        goto done;
    }
    for (int i = 0; i < W; ++i) {
        wire[i] = (uint32_t*)calloc((size_t)(nwords > 0 ? nwords : 1), sizeof(uint32_t));
        if (!wire[i]) {
            rc = -2;
            goto done;
        }
    }

    /* 1-2. Update vector and compression, worker by worker, tensor by
     * tensor.  Tensor offsets are multiples of 32 elements, so a tensor's
     * packed words start on a word boundary. */
    for (int i = 0; i < W; ++i) {
        for (int k = 0; k < K; ++k) {
            int64_t off = layout[k].offset, n = layout[k].numel;
            for (int64_t e = 0; e < n; ++e) {
                float g = load_grad(grads[i], grad_dtype, off + e);
                c[e] = lco_update_vector(m[i][off + e], g, beta1, lco_omega(beta1));
            }
            int64_t w0 = off * bits / 32;
            int64_t nw = (n * bits + 31) / 32;
            if (mode == LCO_MODE_SIGN) {
                lco_pack_signs(c, n, t, tmpw);
            } else {
                float m1 = lco_m1(c, n);
                if (m1_out)
                    m1_out[(int64_t)i * K + k] = m1;
                lco_q1(c, n, nbits, m1, q);
                lco_pack_codes(q, n, nbits, tmpw);
            }
            for (int64_t w = 0; w < nw; ++w)
                wire[i][w0 + w] |= tmpw[w];
        }
    }

    /* 3-4. Aggregate over workers, global direction, theta. */
    for (int64_t e = 0; e < d; ++e) {
        int32_t agg = (mode == LCO_MODE_SIGN)
                          ? lco_vote((const uint32_t* const*)wire, W, e)
                          : lco_code_sum((const uint32_t* const*)wire, W, nbits, e);
        if (agg_out)
            agg_out[e] = agg;
        float u = lco_direction(agg, W, flags, t);
        theta[e] = lco_apply(theta[e], u, lr, wd);
    }

    /* 5. Momentum of every worker from its old value and its own gradient. */
    for (int i = 0; i < W; ++i)
        for (int64_t e = 0; e < d; ++e)
            m[i][e] = lco_momentum(m[i][e], load_grad(grads[i], grad_dtype, e),
                                   beta2, lco_omega(beta2));

    /* 6. Selective momentum sync on flagged tensors. */
    if (sync_interval > 0 && (t + 1) % sync_interval == 0)
        for (int k = 0; k < K; ++k)
            if (layout[k].flags & LCO_TENSOR_SYNC_M)
                lco_sync_average(m, W, layout[k].offset, layout[k].offset + layout[k].numel);

    if (wire_out)
        for (int i = 0; i < W; ++i)
            if (wire_out[i])
                memcpy(wire_out[i], wire[i], (size_t)nwords * sizeof(uint32_t));

done:
    if (wire) {
        for (int i = 0; i < W; ++i)
            free(wire[i]);
        free(wire);
    }
    free(c);
    free(q);
    free(tmpw);
    return rc;
}

/* ---- diagnostics ---------------------------------------------------------
 * [LC] Fig. 4 / Fig. 11 captions: whether the signs of the quantized updates
 * match or flip against the full-precision update; Fig. 6 caption: the
 * maximum standard deviation between workers, per layer, over its elements;
 * quoted body text: the share of tied majority votes. */

float lco_worker_std(const float* x, int W)
{
    float s = x[0];
    for (int i = 1; i < W; ++i)
        s = s + x[i];
    float mean = s / (float)W;
    float v = 0.0f;
    for (int i = 0; i < W; ++i) {
        float dlt = x[i] - mean;
        float sq = dlt * dlt;
        v = v + sq;
    }
    return sqrtf(v / (float)W);
}

int lco_classify(float u_q, float u_fp)
{
    if (u_q == u_fp)
        return 0;
    if (u_q != 0.0f && u_fp != 0.0f)
        return 1;
    if (u_q == 0.0f)
        return 2;
    return 3;
}

static float sign_of(float x)
{
    return x > 0.0f ? 1.0f : (x < 0.0f ? -1.0f : 0.0f);
}

int lco_diagnose(int64_t d, int W, const lco_tensor* layout, int K,
                 float beta1, int mode, int nbits, uint32_t flags, int64_t t,
                 int grad_dtype, const void* const* grads, const float* const* m,
                 lco_diag* out)
{
    if (d < 0 || W < 1 || !grads || !m || !out)
        return -1;
    if (mode != LCO_MODE_SIGN && mode != LCO_MODE_L1)
        return -1;
    if (mode == LCO_MODE_L1 && nbits != 2 && nbits != 4 && nbits != 8)
        return -1;
    lco_tensor whole;
    whole.offset = 0;
    whole.numel = d;
    whole.flags = 0;
    if (!layout || K == 0) {
        layout = &whole;
        K = 1;
    }
    int64_t maxn = 0;
    for (int k = 0; k < K; ++k)
        if (layout[k].numel > maxn)
            maxn = layout[k].numel;
    int rc = 0;
    float* c = (float*)malloc((size_t)(maxn > 0 ? maxn : 1) * (size_t)W * sizeof(float));
    int8_t* q = (int8_t*)malloc((size_t)(maxn > 0 ? maxn : 1) * (size_t)W);
    float* col = (float*)malloc((size_t)W * sizeof(float));
    if (!c || !q || !col) {
        rc = -2;
        goto done;
    }
    for (int k = 0; k < K; ++k) {
        int64_t off = layout[k].offset, n = layout[k].numel;
        lco_diag r;
        memset(&r, 0, sizeof r);
        /* update vectors of every worker, and their codes in L1 mode */
        for (int i = 0; i < W; ++i) {
            float* ci = c + (int64_t)i * n;
            for (int64_t e = 0; e < n; ++e)
                ci[e] = lco_update_vector(m[i][off + e], load_grad(grads[i], grad_dtype, off + e), beta1,
                                          lco_omega(beta1));
            if (mode == LCO_MODE_L1)
                lco_q1(ci, n, nbits, lco_m1(ci, n), q + (int64_t)i * n);
        }
        for (int64_t e = 0; e < n; ++e) {
            int32_t agg = 0;
            float s = 0.0f;
            for (int i = 0; i < W; ++i) {
                float ci = c[(int64_t)i * n + e];
                if (mode == LCO_MODE_SIGN)
                    agg += lco_sign_bit(ci, t) ? 1 : -1;
                else
                    agg += q[(int64_t)i * n + e];
                s = (i == 0) ? ci : s + ci;
            }
            if (agg == 0)
                r.ties += 1;
            float u_q = sign_of(lco_direction(agg, W, flags, t));
            switch (lco_classify(u_q, sign_of(s))) {
            case 0: r.match += 1; break;
            case 1: r.flip += 1; break;
            case 2: r.dropped += 1; break;
            default: r.spurious += 1; break;
            }
            for (int i = 0; i < W; ++i)
                col[i] = m[i][off + e];
            float sd = lco_worker_std(col, W);
            if (sd > r.max_std_m)
                r.max_std_m = sd;
        }
        out[k] = r;
    }
done:
    free(c);
    free(q);
    free(col);
    return rc;
}

/* ---- Q_inf: max-norm scaling with stochastic rounding (see the header) ---- */

uint64_t lco_splitmix64(uint64_t seed, uint64_t k)
{
    uint64_t z = seed + (k + 1u) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

float lco_qinf_uniform(uint64_t seed, int64_t t, int worker, int64_t e)
{
    uint64_t k = (((uint64_t)t & 0xffffu) << 48) | ((uint64_t)(unsigned)worker << 40) | (uint64_t)e;
    uint64_t bits = lco_splitmix64(seed, k) >> 40; /* 24 bits */
    return (float)bits * (1.0f / 16777216.0f);
}

float lco_maxabs(const float* c, int64_t n)
{
    float mx = 0.0f;
    for (int64_t e = 0; e < n; ++e)
        if (fabsf(c[e]) > mx)
            mx = fabsf(c[e]);
    return mx;
}

void lco_qinf(const float* c, int64_t n, int nbits, float maxabs, uint64_t seed, int64_t t, int worker,
              int64_t e_first, int8_t* q)
{
    int qmax = (1 << (nbits - 1)) - 1;
    float inv = maxabs > 0.0f ? (float)qmax / maxabs : 0.0f;
    for (int64_t e = 0; e < n; ++e) {
        float y = fabsf(c[e]) * inv;
        float fl = floorf(y);
        float frac = y - fl;
        float u = lco_qinf_uniform(seed, t, worker, e_first + e);
        int v = (int)fl + (u < frac ? 1 : 0);
        if (v > qmax)
            v = qmax;
        q[e] = (int8_t)(c[e] < 0.0f ? -v : v);
    }
}

int lco_diagnose_qinf(int64_t d, int W, const lco_tensor* layout, int K, float beta1, int nbits, uint32_t flags,
                      int64_t t, uint64_t seed, int64_t e_base, int grad_dtype, const void* const* grads,
                      const float* const* m, lco_qinf_diag* out)
{
    if (d < 0 || W < 1 || W > 255 || !grads || !m || !out)
        return -1;
    if (nbits != 2 && nbits != 4 && nbits != 8)
        return -1;
    lco_tensor whole;
    whole.offset = 0;
    whole.numel = d;
    whole.flags = 0;
    if (!layout || K == 0) {
        layout = &whole;
        K = 1;
    }
    int64_t maxn = 0;
    for (int k = 0; k < K; ++k)
        if (layout[k].numel > maxn)
            maxn = layout[k].numel;
    int rc = 0;
    float* c = (float*)malloc((size_t)(maxn > 0 ? maxn : 1) * sizeof(float));
    int8_t* q = (int8_t*)malloc((size_t)(maxn > 0 ? maxn : 1) * (size_t)W);
    float* s = (float*)malloc((size_t)(maxn > 0 ? maxn : 1) * sizeof(float));
    if (!c || !q || !s) {
        rc = -2;
        goto done;
    }
    uint32_t dir_flags = flags & ~LCO_FLAG_AVERAGE;
    for (int k = 0; k < K; ++k) {
        int64_t off = layout[k].offset, n = layout[k].numel;
        lco_qinf_diag r;
        memset(&r, 0, sizeof r);
        /* each worker: update vector, its max-norm, its Q_inf codes; the
         * full-precision sum in worker order */
        for (int i = 0; i < W; ++i) {
            for (int64_t e = 0; e < n; ++e) {
                c[e] = lco_update_vector(m[i][off + e], load_grad(grads[i], grad_dtype, off + e), beta1,
                                         lco_omega(beta1));
                s[e] = (i == 0) ? c[e] : s[e] + c[e];
            }
            lco_qinf(c, n, nbits, lco_maxabs(c, n), seed, t, i, e_base + off, q + (int64_t)i * n);
        }
        for (int64_t e = 0; e < n; ++e) {
            int32_t agg = 0;
            for (int i = 0; i < W; ++i) {
                int8_t qi = q[(int64_t)i * n + e];
                agg += qi;
                if (qi == 0)
                    r.zero_codes += 1;
            }
            float u_q = sign_of(lco_direction(agg, W, dir_flags, t));
            switch (lco_classify(u_q, sign_of(s[e]))) {
            case 0: r.match += 1; break;
            case 1: r.flip += 1; break;
            case 2: r.dropped += 1; break;
            default: r.spurious += 1; break;
            }
        }
        out[k] = r;
    }
done:
    free(c);
    free(q);
    free(s);
    return rc;
}
