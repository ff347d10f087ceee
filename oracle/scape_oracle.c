/*
 * scape_oracle.c -- plain, slow CPU oracle of the SCAPE sharded optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant with the CUDA
 * library; it is written from the method's description alone.
 *
 * Sources (cited by page title and section):
 *   [P1] "SCAPE: Accurate and Efficient LLM Training with Extremely Sparse
 *        Communication" (arXiv 2607.01678, Chinese translation page):
 *        abstract, Sec. I, Sec. II-A (sharded data parallel, Eq. 1),
 *        Sec. II-B (top-k with error feedback), Sec. II-C (AdamS, Eq. 2).
 *   [P2] "Sintesi Tecnica: SCAPE" (gist.science technical summary):
 *        Sec. 2 "Metodologia" -- partitioned mask synchronisation, lagged mask
 *        use (one-step lag), single-buffer second-moment reconstruction,
 *        memory optimisation (single-bit compacted formats).
 *
 * Precision: the pages fix the optimizer states and the error-feedback buffer
 * at FP32 ([P1] Sec. II-A and II-B), so every floating-point value here is a
 * C `float` and every operation is written out one IEEE-754 binary32 operation
 * at a time (compile with -ffp-contract=off, never -ffast-math).  sqrtf and
 * '/' are the correctly rounded IEEE operations.
 *
 * Readings of points the pages leave open (each is listed in the design notes):
 *   shard partition      contiguous, boundary s = floor(s*P/W)            ([P1] II-A "evenly partitioned")
 *   k per shard          k_s = ceil(n_s * (1e6 - ppm) / 1e6), ppm = sparsity in parts per million
 *   top-k key            IEEE bits of m with the sign bit cleared, compared as uint32;
 *                        equal keys are ordered by ascending global index
 *   off-mask coordinates w and m are left unchanged (only masked coordinates update)
 *   step 1               dense (mask of all ones); the lag starts from the mask built after step 1
 *   synchronised buffer  mean of the masked error-fed gradients, summed in worker order 0..W-1
 *                        and divided by W
 *   bias correction      bc_i = (float)(1 - beta_i^t), computed in double from the float beta
 *   weight decay         decoupled, inside the lr product, on w_{t-1}
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

/* gradient element types */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/* ------------------------------------------------------------------------- */
/* Shard layout: [P1] Sec. II-A -- the distributed optimizer partitions the   */
/* optimizer state and the parameters evenly over the W data-parallel         */
/* workers; [P2] Sec. 2 -- mask generation is aligned with that sharding.     */
/* ------------------------------------------------------------------------- */
int oracle_layout(int64_t P, int W, int64_t sparsity_ppm, int64_t *shard_start,
                  int64_t *shard_k)
{
    if (P < 0 || W < 1 || sparsity_ppm < 0 || sparsity_ppm >= 1000000)
        return ORACLE_EINVAL;
    for (int s = 0; s <= W; ++s)
        shard_start[s] = ((int64_t)s * P) / W;
    for (int s = 0; s < W; ++s) {
        int64_t n = shard_start[s + 1] - shard_start[s];
        /* keep a (1 - sparsity) fraction of the shard, rounded up */
        shard_k[s] = (n * (1000000 - sparsity_ppm) + 999999) / 1000000;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Mask refresh: [P2] Sec. 2 "partitioned mask synchronisation" -- each       */
/* worker takes the top-k of its own optimizer shard only, and the shard      */
/* masks are gathered (concatenated) into the global mask; [P1] Sec. I and    */
/* [P2] Sec. 2 "lagged mask use" -- the mask comes from first-moment          */
/* statistics, not from the raw gradient.  Top-k per [P1] Sec. II-B: keep the */
/* k entries of largest magnitude.  The global mask is kept as one bit per    */
/* parameter ([P2] Sec. 2, single-bit compacted formats), bit i%32 of word    */
/* i/32.                                                                      */
/* ------------------------------------------------------------------------- */
typedef struct {
    uint32_t key;
    int64_t index;
} oracle_entry;

static uint32_t magnitude_key(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u & 0x7FFFFFFFu; /* |x| as an ordered integer; -0 and +0 coincide */
}

/* larger magnitude first; among equal magnitudes, smaller index first */
static int entry_order(const void *pa, const void *pb)
{
    const oracle_entry *a = (const oracle_entry *)pa;
    const oracle_entry *b = (const oracle_entry *)pb;
    if (a->key != b->key)
        return a->key > b->key ? -1 : 1;
    if (a->index != b->index)
        return a->index < b->index ? -1 : 1;
    return 0;
}

int oracle_topk_mask(const float *m, int64_t P, int S, const int64_t *shard_start,
                     const int64_t *shard_k, uint32_t *bits, uint32_t *idx,
                     int64_t *k_total)
{
    int64_t nwords = (P + 31) / 32;
    memset(bits, 0, (size_t)nwords * sizeof(uint32_t));
    for (int s = 0; s < S; ++s) {
        int64_t lo = shard_start[s], hi = shard_start[s + 1], n = hi - lo;
        if (n <= 0)
            continue;
        if (shard_k[s] > n)
            return ORACLE_EINVAL;
        oracle_entry *ent = (oracle_entry *)malloc((size_t)n * sizeof(oracle_entry));
        if (!ent)
            return ORACLE_EINVAL;
        for (int64_t i = lo; i < hi; ++i) {
            ent[i - lo].key = magnitude_key(m[i]);
            ent[i - lo].index = i;
        }
        qsort(ent, (size_t)n, sizeof(oracle_entry), entry_order);
        for (int64_t r = 0; r < shard_k[s]; ++r) {
            int64_t i = ent[r].index;
            bits[i / 32] |= 1u << (i % 32);
        }
        free(ent);
    }
    /* packed index list: the set positions of the global mask, ascending */
    int64_t k = 0;
    for (int64_t i = 0; i < P; ++i)
        if ((bits[i / 32] >> (i % 32)) & 1u)
            idx[k++] = (uint32_t)i;
    *k_total = k;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* One optimizer step t (1-based) under a given mask.                         */
/*                                                                            */
/* Error feedback, [P1] Sec. II-B: the sent gradient is TopK(g_t + e_t), here */
/* the part of g_t + e_t selected by the mask, and the residual becomes       */
/* e_{t+1} = g_t + e_t - (sent part).                                         */
/* Compaction: each worker's selected values are packed, in ascending index   */
/* order, into a k-long buffer ([P1] Sec. II-B "compressed buffer").          */
/* Synchronisation: the W packed buffers are averaged ([P1] Sec. II-B,        */
/* averaging the sparsified gradients; [P2] Sec. 2 single synchronised        */
/* buffer) -- on one device this is an ordered sum and a division by W.       */
/* Update, [P1] Sec. II-C Eq. 2 with its bias corrections:                    */
/*     m_t = b1 m_{t-1} + (1 - b1) g                                          */
/*     v_t = b2 m_{t-1}^2 + (1 - b2) g^2      (v is not stored)               */
/*     w_t = w_{t-1} - lr (m_hat / (sqrt(v_hat) + eps) + wd w_{t-1})          */
/* with m_hat = m_t / (1 - b1^t), v_hat = v_t / (1 - b2^t), applied at the    */
/* masked coordinates, m_t and v_t both drawn from the one synchronised       */
/* buffer ([P2] Sec. 2, single-buffer second-moment reconstruction).          */
/* ------------------------------------------------------------------------- */
static float widen_grad(const void *g, int dtype, int64_t i)
{
    if (dtype == ORACLE_F32)
        return ((const float *)g)[i];
    uint16_t h = ((const uint16_t *)g)[i];
    uint32_t u = (uint32_t)h << 16; /* bfloat16 is the top half of a binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int oracle_step(int64_t t, int64_t P, int W, int grad_dtype, const void *const *grads,
                float *const *e, float *w, float *m, const uint32_t *bits,
                const uint32_t *idx, int64_t k, float beta1, float beta2, float lr,
                float eps, float wd, float *pack, float *gbar)
{
    if (t < 1 || P < 0 || W < 1 || k < 0 || k > P)
        return ORACLE_EINVAL;
    if (grad_dtype != ORACLE_F32 && grad_dtype != ORACLE_BF16)
        return ORACLE_EINVAL;

    /* error feedback add, compaction of the sent part, residual update */
    for (int wk = 0; wk < W; ++wk) {
        int64_t r = 0;
        for (int64_t i = 0; i < P; ++i) {
            float a = widen_grad(grads[wk], grad_dtype, i) + e[wk][i];
            int selected = (bits[i / 32] >> (i % 32)) & 1u;
            float sent = selected ? a : 0.0f;
            if (selected) {
                if (r >= k)
                    return ORACLE_EINVAL;
                pack[(int64_t)wk * k + r] = a;
                r = r + 1;
            }
            e[wk][i] = a - sent;
        }
        if (r != k)
            return ORACLE_EINVAL;
    }

    /* average of the W packed buffers, summed in worker order */
    for (int64_t j = 0; j < k; ++j) {
        float sum = pack[j];
        for (int wk = 1; wk < W; ++wk)
            sum = sum + pack[(int64_t)wk * k + j];
        gbar[j] = sum / (float)W;
    }

    /* AdamS at the masked coordinates */
    float one_minus_b1 = 1.0f - beta1;
    float one_minus_b2 = 1.0f - beta2;
    float bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    float bc2 = (float)(1.0 - pow((double)beta2, (double)t));
    for (int64_t j = 0; j < k; ++j) {
        int64_t i = idx[j];
        float g = gbar[j];
        float m_prev = m[i];
        float w_prev = w[i];

        float m_new = beta1 * m_prev + one_minus_b1 * g;
        float v = beta2 * (m_prev * m_prev) + one_minus_b2 * (g * g);
        float m_hat = m_new / bc1;
        float v_hat = v / bc2;
        float step = m_hat / (sqrtf(v_hat) + eps) + wd * w_prev;
        w[i] = w_prev - lr * step;
        m[i] = m_new;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Variant readings of the pages, selected by flags (one step, given mask).  */
/*                                                                            */
/* ORACLE_VARIANT_DENSE_OFFMASK: the other reading of what happens off the    */
/*   mask -- every unselected coordinate also takes the AdamS update of       */
/*   [P1] Sec. II-C with a zero synchronised gradient (m decays, v = b2 m^2). */
/* ORACLE_VARIANT_MOMENT_SYNC: the single synchronised buffer holds the       */
/*   first moment ([P2] Sec. 2, "deriving the global mean gradient ... from   */
/*   the synchronised first-moment buffer"): each worker sends                */
/*   b = b1 m_{t-1} + (1 - b1) a at its selected coordinates, the buffer is   */
/*   the mean of the b, m_t is that mean, and the gradient the second moment  */
/*   needs is recovered as g = (b_mean - b1 m_{t-1}) / (1 - b1).              */
/* The residual is the unsent part of g + e in both ([P1] Sec. II-B).        */
/* ------------------------------------------------------------------------- */
#define ORACLE_VARIANT_DENSE_OFFMASK 1
#define ORACLE_VARIANT_MOMENT_SYNC 2

static void adams_one(float g, float *wi, float *mi, float beta1, float beta2, float bc1,
                      float bc2, float lr, float eps, float wd)
{
    float m_prev = *mi, w_prev = *wi;
    float m_new = beta1 * m_prev + (1.0f - beta1) * g;
    float v = beta2 * (m_prev * m_prev) + (1.0f - beta2) * (g * g);
    float m_hat = m_new / bc1;
    float v_hat = v / bc2;
    *wi = w_prev - lr * (m_hat / (sqrtf(v_hat) + eps) + wd * w_prev);
    *mi = m_new;
}

int oracle_step_variant(int64_t t, int64_t P, int W, int grad_dtype, const void *const *grads,
                        float *const *e, float *w, float *m, const uint32_t *bits,
                        const uint32_t *idx, int64_t k, float beta1, float beta2, float lr,
                        float eps, float wd, int variant, float *pack, float *gbar)
{
    if (t < 1 || P < 0 || W < 1 || k < 0 || k > P)
        return ORACLE_EINVAL;
    if (grad_dtype != ORACLE_F32 && grad_dtype != ORACLE_BF16)
        return ORACLE_EINVAL;
    int msync = (variant & ORACLE_VARIANT_MOMENT_SYNC) != 0;
    float one_minus_b1 = 1.0f - beta1;
    float one_minus_b2 = 1.0f - beta2;
    float bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    float bc2 = (float)(1.0 - pow((double)beta2, (double)t));

    for (int wk = 0; wk < W; ++wk) {
        int64_t r = 0;
        for (int64_t i = 0; i < P; ++i) {
            float a = widen_grad(grads[wk], grad_dtype, i) + e[wk][i];
            int selected = (bits[i / 32] >> (i % 32)) & 1u;
            float sent = selected ? a : 0.0f;
            if (selected) {
                if (r >= k)
                    return ORACLE_EINVAL;
                pack[(int64_t)wk * k + r] = msync ? beta1 * m[i] + one_minus_b1 * a : a;
                r = r + 1;
            }
            e[wk][i] = a - sent;
        }
        if (r != k)
            return ORACLE_EINVAL;
    }
    for (int64_t j = 0; j < k; ++j) {
        float sum = pack[j];
        for (int wk = 1; wk < W; ++wk)
            sum = sum + pack[(int64_t)wk * k + j];
        gbar[j] = sum / (float)W;
    }
    for (int64_t j = 0; j < k; ++j) {
        int64_t i = idx[j];
        if (!msync) {
            adams_one(gbar[j], &w[i], &m[i], beta1, beta2, bc1, bc2, lr, eps, wd);
        } else {
            float m_prev = m[i], w_prev = w[i];
            float m_new = gbar[j];
            float g = (m_new - beta1 * m_prev) / one_minus_b1;
            float v = beta2 * (m_prev * m_prev) + one_minus_b2 * (g * g);
            float m_hat = m_new / bc1;
            float v_hat = v / bc2;
            w[i] = w_prev - lr * (m_hat / (sqrtf(v_hat) + eps) + wd * w_prev);
            m[i] = m_new;
        }
    }
    if (variant & ORACLE_VARIANT_DENSE_OFFMASK) {
        for (int64_t i = 0; i < P; ++i)
            if (!((bits[i / 32] >> (i % 32)) & 1u))
                adams_one(0.0f, &w[i], &m[i], beta1, beta2, bc1, bc2, lr, eps, wd);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Dense baselines the pages compare SCAPE against (abstract, Sec. I): dense */
/* AdamS ([P1] Sec. II-C, Eq. 2) and dense AdamW, both on the plain mean of   */
/* the W workers' gradients (no error feedback, no mask).  AdamW keeps the   */
/* second moment as an EMA of g^2: v_t = b2 v_{t-1} + (1 - b2) g^2, with the */
/* same bias corrections and decoupled weight decay.                         */
/* ------------------------------------------------------------------------- */
static float mean_grad(const void *const *grads, int W, int grad_dtype, int64_t i)
{
    float sum = widen_grad(grads[0], grad_dtype, i);
    for (int wk = 1; wk < W; ++wk)
        sum = sum + widen_grad(grads[wk], grad_dtype, i);
    return sum / (float)W;
}

int oracle_dense_adams_step(int64_t t, int64_t P, int W, int grad_dtype,
                            const void *const *grads, float *w, float *m, float beta1,
                            float beta2, float lr, float eps, float wd)
{
    if (t < 1 || P < 0 || W < 1 || (grad_dtype != ORACLE_F32 && grad_dtype != ORACLE_BF16))
        return ORACLE_EINVAL;
    float bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    float bc2 = (float)(1.0 - pow((double)beta2, (double)t));
    for (int64_t i = 0; i < P; ++i)
        adams_one(mean_grad(grads, W, grad_dtype, i), &w[i], &m[i], beta1, beta2, bc1, bc2, lr,
                  eps, wd);
    return ORACLE_OK;
}

int oracle_adamw_step(int64_t t, int64_t P, int W, int grad_dtype, const void *const *grads,
                      float *w, float *m, float *v, float beta1, float beta2, float lr,
                      float eps, float wd)
{
    if (t < 1 || P < 0 || W < 1 || (grad_dtype != ORACLE_F32 && grad_dtype != ORACLE_BF16))
        return ORACLE_EINVAL;
    float bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    float bc2 = (float)(1.0 - pow((double)beta2, (double)t));
    for (int64_t i = 0; i < P; ++i) {
        float g = mean_grad(grads, W, grad_dtype, i);
        float w_prev = w[i];
        float m_new = beta1 * m[i] + (1.0f - beta1) * g;
        float v_new = beta2 * v[i] + (1.0f - beta2) * (g * g);
        float m_hat = m_new / bc1;
        float v_hat = v_new / bc2;
        w[i] = w_prev - lr * (m_hat / (sqrtf(v_hat) + eps) + wd * w_prev);
        m[i] = m_new;
        v[i] = v_new;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Gradient top-k with error feedback and a union mask: the second           */
/* synchronisation scheme of [P1] Sec. II-B, the baseline SCAPE's partitioned */
/* mask is designed against.  Each worker selects the k_worker largest |a^w|, */
/* a^w = g^w + e^w, over the whole vector (larger magnitude first, lower      */
/* index on ties); the masks are gathered into their union; every worker     */
/* sends its a^w at every union position (the all-reduce over the global     */
/* mask), so its residual becomes a - a there and stays a elsewhere; the     */
/* mean over the workers drives AdamS ([P1] Sec. II-C) at the union          */
/* positions, the others are left unchanged.  As W grows the union fills in. */
/* ------------------------------------------------------------------------- */
int oracle_union_topk_step(int64_t t, int64_t P, int W, int grad_dtype,
                           const void *const *grads, float *const *e, float *w, float *m,
                           int64_t k_worker, float beta1, float beta2, float lr, float eps,
                           float wd, uint32_t *union_bits, uint32_t *idx, int64_t *k_union,
                           float *pack, float *gbar)
{
    if (t < 1 || P < 1 || W < 1 || k_worker < 0 || k_worker > P)
        return ORACLE_EINVAL;
    if (grad_dtype != ORACLE_F32 && grad_dtype != ORACLE_BF16)
        return ORACLE_EINVAL;
    int64_t nwords = (P + 31) / 32;
    memset(union_bits, 0, (size_t)nwords * sizeof(uint32_t));
    oracle_entry *ent = (oracle_entry *)malloc((size_t)P * sizeof(oracle_entry));
    if (!ent)
        return ORACLE_EINVAL;
    for (int wk = 0; wk < W; ++wk) {
        for (int64_t i = 0; i < P; ++i) {
            e[wk][i] = widen_grad(grads[wk], grad_dtype, i) + e[wk][i]; /* a^w */
            ent[i].key = magnitude_key(e[wk][i]);
            ent[i].index = i;
        }
        qsort(ent, (size_t)P, sizeof(oracle_entry), entry_order);
        for (int64_t r = 0; r < k_worker; ++r) {
            int64_t i = ent[r].index;
            union_bits[i / 32] |= 1u << (i % 32);
        }
    }
    free(ent);
    int64_t k = 0;
    for (int64_t i = 0; i < P; ++i)
        if ((union_bits[i / 32] >> (i % 32)) & 1u)
            idx[k++] = (uint32_t)i;
    *k_union = k;
    for (int wk = 0; wk < W; ++wk) {
        for (int64_t j = 0; j < k; ++j) {
            int64_t i = idx[j];
            float a = e[wk][i];
            pack[(int64_t)wk * k + j] = a;
            e[wk][i] = a - a;
        }
    }
    float bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    float bc2 = (float)(1.0 - pow((double)beta2, (double)t));
    for (int64_t j = 0; j < k; ++j) {
        float sum = pack[j];
        for (int wk = 1; wk < W; ++wk)
            sum = sum + pack[(int64_t)wk * k + j];
        gbar[j] = sum / (float)W;
        adams_one(gbar[j], &w[idx[j]], &m[idx[j]], beta1, beta2, bc1, bc2, lr, eps, wd);
    }
    return ORACLE_OK;
}
