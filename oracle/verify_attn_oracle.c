/*
 * CPU oracle for tree-verify attention over a paged MLA latent KV pool.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's cpu_baseline / reference arm load this file's library.  The
 * product path (the CUDA library and its Python binding) never does, and it
 * shares no code, header or table with this file.
 *
 * What it computes (plain definition, written out; the GPU's split-KV +
 * log-sum-exp combine is an exact rearrangement of the same result):
 *
 *   For request b: T_b = qo_indptr[b+1]-qo_indptr[b] draft tokens,
 *   L_b = kv_indptr[b+1]-kv_indptr[b] prefix keys ("The Capture-Safe Kernel",
 *   Decision 2: the prefix length is derived from kv_indptr), N_b = L_b+T_b.
 *   Key j < L_b lives in pool slot kv_indices[kv_indptr[b]+j]; key j >= L_b
 *   is draft token j-L_b, whose own slot is out_cache_loc[qo_indptr[b]+j-L_b]
 *   ("The Capture-Safe Kernel", Decision 1: native kv_indices /
 *   out_cache_loc buffers read directly; the old host-side concatenation of
 *   the two is what was removed, section The Core Problem).
 *   Draft token i of b sees key j iff bit mask_indptr[b] + i*N_b + j of the
 *   packed custom_mask is set ("The Capture-Safe Kernel", Decision 5: index
 *   the raw custom_mask through mask_indptr), LSB-first within each byte.
 *   For global token t = qo_indptr[b]+i and head h (output row t*H+h):
 *     s_j   = sm_scale * <q[t,h,0:576], pool[slot_j, 0:576]>   (visible j)
 *     m     = max_j s_j,  Z = sum_j exp(s_j - m)
 *     out   = sum_j exp(s_j - m) * pool[slot_j, 0:512] / Z
 *     lse   = m + ln Z   (natural log)
 *   A row that sees no key gets out = 0 and lse = -inf.
 *   ("The Integration Chasm", section Decision: MLA attention after q
 *   projection and absorption, so attention runs in the 576-wide latent
 *   space; V is the first 512 latent dims.)
 *
 * Precision: bf16 inputs are widened exactly to double; every product, sum,
 * exp and division is done in double.  Two passes per row (scores, then max,
 * then weighted sum) -- no online rescaling, no blocking.
 *
 * Split mode (num_splits > 0) is the pages' flash-decode partial-plus-reduce
 * ("The Capture-Safe Kernel", Decision 3 and Input Knowledge item 3): keys
 * [0,N_b) are cut into chunks of c_b = ceil(N_b/num_splits); each chunk
 * yields a normalised partial output and its lse (empty chunk: lse = -inf);
 * the partials are merged with weights exp(lse_s - max_s lse_s).  It exists
 * only so tests can check that the result does not depend on the split
 * count.
 *
 * Parity status: every part is pinned by tests/test_oracle_pins.py (library
 * SDPA on dense inputs, causal and full-attention special cases, closed
 * forms, single-key exactness, permutation / packing invariances and a
 * hand-derived packed-mask fixture).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_D 576
#define ORACLE_DV 512

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_ARG = -1,
    ORACLE_ERR_SLOT = -2,      /* a slot id outside [0, pool_size) */
    ORACLE_ERR_MASK = -3,      /* mask_indptr does not give T_b*N_b bits */
    ORACLE_ERR_ROW = -4,       /* requested row outside [0, total_q*H) */
    ORACLE_ERR_NOMEM = -5,
};

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int mask_bit(const uint8_t *mask, int64_t bit)
{
    return (mask[bit >> 3] >> (bit & 7)) & 1;
}

/* Request that owns global draft token t (qo_indptr is non-decreasing). */
static int find_request(const int32_t *qo_indptr, int batch, int64_t t)
{
    for (int b = 0; b < batch; ++b)
        if (t >= qo_indptr[b] && t < qo_indptr[b + 1])
            return b;
    return -1;
}

typedef struct {
    const uint16_t *q;
    int64_t q_stride_tok, q_stride_head;
    const uint16_t *kv_pool;
    int64_t pool_size;
    const int32_t *qo_indptr, *kv_indptr, *kv_indices;
    const int64_t *out_cache_loc;
    const uint8_t *custom_mask;
    const int64_t *mask_indptr;
    double sm_scale;
    int batch, num_heads;
} oracle_args;

/* Slot of key j of request b. */
static int64_t key_slot(const oracle_args *a, int b, int64_t j)
{
    int64_t L = a->kv_indptr[b + 1] - a->kv_indptr[b];
    if (j < L)
        return a->kv_indices[a->kv_indptr[b] + j];
    return a->out_cache_loc[a->qo_indptr[b] + (j - L)];
}

/*
 * Attention of one output row over keys [k0, k1) of its request.
 * Writes the normalised output (ORACLE_DV doubles) and returns its lse
 * through *lse_out; a range with no visible key gives zeros and -inf.
 */
static int attend_range(const oracle_args *a, int b, int64_t i, int h, int64_t k0, int64_t k1,
                        double *scores, double *out, double *lse_out)
{
    int64_t L = a->kv_indptr[b + 1] - a->kv_indptr[b];
    int64_t T = a->qo_indptr[b + 1] - a->qo_indptr[b];
    int64_t N = L + T;
    int64_t t = a->qo_indptr[b] + i;
    const uint16_t *qrow = a->q + t * a->q_stride_tok + (int64_t)h * a->q_stride_head;

    /* pass 1: scores of visible keys, and their maximum */
    double m = -INFINITY;
    int any = 0;
    for (int64_t j = k0; j < k1; ++j) {
        if (!mask_bit(a->custom_mask, a->mask_indptr[b] + i * N + j)) {
            scores[j - k0] = -INFINITY;
            continue;
        }
        int64_t slot = key_slot(a, b, j);
        if (slot < 0 || slot >= a->pool_size)
            return ORACLE_ERR_SLOT;
        const uint16_t *krow = a->kv_pool + slot * ORACLE_D;
        double dot = 0.0;
        for (int d = 0; d < ORACLE_D; ++d)
            dot += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
        double s = a->sm_scale * dot;
        scores[j - k0] = s;
        if (s > m)
            m = s;
        any = 1;
    }
    for (int d = 0; d < ORACLE_DV; ++d)
        out[d] = 0.0;
    if (!any) {
        *lse_out = -INFINITY;
        return ORACLE_OK;
    }
    /* pass 2: softmax weights and the weighted sum of V = first 512 dims */
    double z = 0.0;
    for (int64_t j = k0; j < k1; ++j) {
        if (scores[j - k0] == -INFINITY)
            continue;
        double w = exp(scores[j - k0] - m);
        z += w;
        const uint16_t *vrow = a->kv_pool + key_slot(a, b, j) * ORACLE_D;
        for (int d = 0; d < ORACLE_DV; ++d)
            out[d] += w * bf16_to_double(vrow[d]);
    }
    for (int d = 0; d < ORACLE_DV; ++d)
        out[d] /= z;
    *lse_out = m + log(z);
    return ORACLE_OK;
}

/* One output row: direct definition (num_splits == 0) or split + combine. */
static int oracle_row(const oracle_args *a, int64_t row, int num_splits, double *out, double *lse)
{
    int64_t total_q = a->qo_indptr[a->batch];
    if (row < 0 || row >= total_q * a->num_heads)
        return ORACLE_ERR_ROW;
    int64_t t = row / a->num_heads;
    int h = (int)(row % a->num_heads);
    int b = find_request(a->qo_indptr, a->batch, t);
    if (b < 0)
        return ORACLE_ERR_ROW;
    int64_t i = t - a->qo_indptr[b];
    int64_t L = a->kv_indptr[b + 1] - a->kv_indptr[b];
    int64_t N = L + (a->qo_indptr[b + 1] - a->qo_indptr[b]);

    double *scores = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!scores)
        return ORACLE_ERR_NOMEM;
    int rc;
    if (num_splits <= 0) {
        rc = attend_range(a, b, i, h, 0, N, scores, out, lse);
    } else {
        int64_t chunk = (N + num_splits - 1) / num_splits;
        double *part = (double *)malloc(sizeof(double) * (size_t)num_splits * ORACLE_DV);
        double *plse = (double *)malloc(sizeof(double) * (size_t)num_splits);
        if (!part || !plse) {
            free(part); free(plse); free(scores);
            return ORACLE_ERR_NOMEM;
        }
        rc = ORACLE_OK;
        for (int s = 0; s < num_splits && rc == ORACLE_OK; ++s) {
            int64_t k0 = (int64_t)s * chunk, k1 = k0 + chunk;
            if (k0 > N) k0 = N;
            if (k1 > N) k1 = N;
            rc = attend_range(a, b, i, h, k0, k1, scores, part + (size_t)s * ORACLE_DV, plse + s);
        }
        if (rc == ORACLE_OK) {
            double mx = -INFINITY;
            for (int s = 0; s < num_splits; ++s)
                if (plse[s] > mx) mx = plse[s];
            for (int d = 0; d < ORACLE_DV; ++d)
                out[d] = 0.0;
            if (mx == -INFINITY) {
                *lse = -INFINITY;
            } else {
                double wsum = 0.0;
                for (int s = 0; s < num_splits; ++s) {
                    if (plse[s] == -INFINITY) continue;
                    double w = exp(plse[s] - mx);
                    wsum += w;
                    for (int d = 0; d < ORACLE_DV; ++d)
                        out[d] += w * part[(size_t)s * ORACLE_DV + d];
                }
                for (int d = 0; d < ORACLE_DV; ++d)
                    out[d] /= wsum;
                *lse = mx + log(wsum);
            }
        }
        free(part);
        free(plse);
    }
    free(scores);
    return rc;
}

static int check_layout(const oracle_args *a)
{
    if (!a->q || !a->kv_pool || !a->qo_indptr || !a->kv_indptr || !a->custom_mask ||
        !a->mask_indptr || a->batch < 0 || a->num_heads <= 0 || a->pool_size <= 0)
        return ORACLE_ERR_ARG;
    for (int b = 0; b < a->batch; ++b) {
        int64_t T = a->qo_indptr[b + 1] - a->qo_indptr[b];
        int64_t L = a->kv_indptr[b + 1] - a->kv_indptr[b];
        if (T < 0 || L < 0)
            return ORACLE_ERR_ARG;
        if (a->mask_indptr[b + 1] - a->mask_indptr[b] != T * (L + T))
            return ORACLE_ERR_MASK;
    }
    return ORACLE_OK;
}

/*
 * Compute output rows.  rows == NULL means every row 0 .. total_q*H-1, in
 * which case out is [total_q*H, 512] and lse [total_q*H]; otherwise out and
 * lse hold the n_rows requested rows in the order given.
 * num_splits == 0: direct definition; > 0: split + combine (tests only).
 * Returns 0 or a negative ORACLE_ERR_*.
 */
int oracle_verify_attn(const uint16_t *q, int64_t q_stride_tok, int64_t q_stride_head,
                       const uint16_t *kv_pool, int64_t pool_size,
                       const int32_t *qo_indptr, const int32_t *kv_indptr,
                       const int32_t *kv_indices, const int64_t *out_cache_loc,
                       const uint8_t *custom_mask, const int64_t *mask_indptr,
                       double sm_scale, int batch, int num_heads,
                       const int64_t *rows, int64_t n_rows, int num_splits,
                       double *out, double *lse)
{
    oracle_args a = {q, q_stride_tok, q_stride_head, kv_pool, pool_size, qo_indptr, kv_indptr,
                     kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, batch,
                     num_heads};
    int rc = check_layout(&a);
    if (rc != ORACLE_OK)
        return rc;
    int64_t count = rows ? n_rows : (int64_t)qo_indptr[batch] * num_heads;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t k = 0; k < count; ++k) {
        int64_t row = rows ? rows[k] : k;
        int r = oracle_row(&a, row, num_splits, out + k * ORACLE_DV, lse + k);
        if (r != ORACLE_OK) {
#pragma omp critical
            err = r;
        }
    }
    return err;
}

/* Threads for later calls (timing only; results do not depend on it). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Number of OpenMP threads the oracle runs with (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
