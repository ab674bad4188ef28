/*
 * CPU oracle for the dense prefill indexer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The product path never calls it and never falls
 * back to it.  It shares no code, header, table or constant with the CUDA
 * library: the number formats are decoded here from their definitions.
 *
 * What it computes (all per query row, rows are independent):
 *
 *   logit[t,j] = sum_h w[t,h] * ReLU( s_q[t,h] * s_k[j] * <q[t,h,:], k[j,:]> )
 *
 * for the keys j < compress_len(t) of the row's request, in fp64, then
 *   - top-k: the k eligible keys with the largest logit, ties to the lower
 *     key index, padded with -1;
 *   - candidate blocks: the maximum logit of every 8-key block (blocks
 *     aligned at key 0, only eligible keys pooled), the top blocks by that
 *     pooled score (ties to the lower block index), as a 0/1 byte per block;
 *   - masked top-k: the top-k over keys that are eligible AND whose block is
 *     a candidate.
 *
 * Sources, by page and section:
 *   - "chunked-prefill-memory.md" section 1: the chunk's T query rows are
 *     scored against the whole compressed prefix, output [T, max_seqlen_k];
 *     section 2.3: per-block top-k, top-k of the union is exact, candidate
 *     source pools 8-key blocks and keeps the top-2048 blocks, consumers
 *     mask non-candidates before the top-k.
 *   - SGLang PR #39187 "Bound the dense prefill indexer transient",
 *     Modifications and Accuracy: row chunks change nothing, selected
 *     indices are raw key indices, residual differences are tie order.
 *   - The score formula is the DeepSeek-V4 / NSA indexer's own (the pages
 *     name its fp8 MQA logits kernels but never print it); the lower-index
 *     tie-break and fp64 accumulation are the readings used throughout.
 *
 * Number formats (decoded from their definitions, no library):
 *   e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals at
 *         exponent 0, code 0x7F/0xFF is NaN, largest finite 448.
 *         Every finite e4m3 value is an integer multiple of 2^-9.
 *   e2m1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, subnormal at
 *         exponent 0: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Every value
 *         is an integer multiple of 2^-1.
 *   ue8m0: 2^(e-127), e = 255 is NaN.
 *
 * Exactness: a dot product of integer multiples is formed from the integer
 * multiples (|m| <= 229376 for e4m3), so every partial sum is an integer
 * below 2^53 and is exact in a double.  The only roundings are the final
 * products by the scales and the sum over heads, all in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NAN (-2)
#define ORACLE_ERR_NOMEM (-3)

/* ---------------------------------------------------------------- formats */

/* e4m3 byte -> value / 2^-9 (an integer), *nan set for the NaN codes. */
static double e4m3_multiple(uint8_t b, int *nan)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) {
        *nan = 1;
        return 0.0;
    }
    if (e == 0)
        mag = (double)m;                       /* m/8 * 2^-6 = m * 2^-9 */
    else
        mag = ldexp((double)(8 + m), e - 1);   /* (1+m/8) 2^(e-7) = (8+m) 2^(e-1) * 2^-9 */
    return sign ? -mag : mag;
}

/* e2m1 nibble -> value / 2^-1 (an integer). */
static double e2m1_multiple(uint8_t nib)
{
    int sign = (nib >> 3) & 1;
    int e = (nib >> 1) & 0x3;
    int m = nib & 0x1;
    double mag;
    if (e == 0)
        mag = (double)m;                       /* m/2 = m * 2^-1 */
    else
        mag = ldexp((double)(2 + m), e - 1);   /* (1+m/2) 2^(e-1) = (2+m) 2^(e-1) * 2^-1 */
    return sign ? -mag : mag;
}

double oracle_e4m3_value(uint8_t b)
{
    int nan = 0;
    double v = ldexp(e4m3_multiple(b, &nan), -9);
    return nan ? NAN : v;
}

double oracle_e2m1_value(uint8_t nib) { return ldexp(e2m1_multiple(nib & 0xF), -1); }

double oracle_ue8m0_value(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

/* ---------------------------------------------------------------- scores */

/*
 * Logits of nrows query rows of ONE request against the request's L keys.
 *   kdtype 0: k is e4m3 [L, D] bytes, k_scale is float s_k[L]
 *   kdtype 1: k is e2m1 [L, D/2] packed (element 2i in the low nibble),
 *             k_scale is uint8 ue8m0 [L, D/32]; s_k is 1
 * out[r, j] for j < L: the logit if j < compress_len[r], -inf otherwise.
 */
int oracle_logits(int H, int D, int kdtype, int64_t nrows, const uint8_t *q,
                  const float *s_q, const float *w, int64_t L, const uint8_t *k,
                  const void *k_scale, const int32_t *compress_len, double *out,
                  int nthreads)
{
    if (H <= 0 || D <= 0 || nrows < 0 || L < 0 || (kdtype != 0 && kdtype != 1))
        return ORACLE_ERR_ARG;
    /* fp4 keys: one ue8m0 scale per 32 elements, at most 8 blocks (D <= 256) */
    if (kdtype == 1 && ((D % 32) != 0 || D > 256))
        return ORACLE_ERR_ARG;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        double *qm = (double *)malloc(sizeof(double) * (size_t)H * (size_t)D);
        double *km = (double *)malloc(sizeof(double) * (size_t)D);
        if (!qm || !km) {
            free(qm);
            free(km);
            bad |= 4;
            continue;
        }
        int nan = 0;
        for (int64_t i = 0; i < (int64_t)H * D; ++i)
            qm[i] = e4m3_multiple(q[r * (int64_t)H * D + i], &nan);
        int64_t clen = compress_len[r];
        double *orow = out + r * L;
        for (int64_t j = 0; j < L; ++j) {
            if (j >= clen) {
                orow[j] = -INFINITY;
                continue;
            }
            /* decode key j into integer multiples */
            double kscale_pow2[8];
            int nblk = 0;
            if (kdtype == 0) {
                for (int d = 0; d < D; ++d)
                    km[d] = e4m3_multiple(k[j * (int64_t)D + d], &nan);
            } else {
                const uint8_t *kp = k + j * (int64_t)(D / 2);
                for (int d = 0; d < D; ++d) {
                    uint8_t byte = kp[d / 2];
                    km[d] = e2m1_multiple((d & 1) ? (byte >> 4) : (byte & 0xF));
                }
                nblk = D / 32;
                const uint8_t *ue = (const uint8_t *)k_scale + j * (int64_t)nblk;
                for (int b = 0; b < nblk; ++b) {
                    if (ue[b] == 255)
                        nan = 1;
                    kscale_pow2[b] = ldexp(1.0, (int)ue[b] - 127);
                }
            }
            double acc = 0.0;
            for (int h = 0; h < H; ++h) {
                const double *qh = qm + (int64_t)h * D;
                double dot;
                if (kdtype == 0) {
                    double s = 0.0; /* integer-valued, exact */
                    for (int d = 0; d < D; ++d)
                        s += qh[d] * km[d];
                    dot = ldexp(s, -18) * (double)((const float *)k_scale)[j];
                } else {
                    dot = 0.0;
                    for (int b = 0; b < nblk; ++b) {
                        double s = 0.0; /* integer-valued, exact */
                        for (int d = 32 * b; d < 32 * b + 32; ++d)
                            s += qh[d] * km[d];
                        dot += ldexp(s, -10) * kscale_pow2[b];
                    }
                }
                double x = (double)s_q[r * H + h] * dot;
                double relu = x > 0.0 ? x : 0.0;
                acc += (double)w[r * H + h] * relu;
            }
            orow[j] = acc;
        }
        if (nan)
            bad |= 2;
        free(qm);
        free(km);
    }
    if (bad & 4)
        return ORACLE_ERR_NOMEM;
    if (bad & 2)
        return ORACLE_ERR_NAN;
    return ORACLE_OK;
}

/* ------------------------------------------------------------- selection */

typedef struct {
    double v;
    int64_t j;
} scored;

/* larger value first, then lower index first */
static int by_score_then_index(const void *a, const void *b)
{
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

/*
 * Top-k of explicit (value, index) pairs, ties to the lower index.
 * Writes min(k, n) indices (and values) in rank order, pads with -1 / -inf.
 */
int oracle_select_pairs(int64_t n, const double *vals, const int64_t *idx, int k,
                        int64_t *out_idx, double *out_val)
{
    if (n < 0 || k < 0)
        return ORACLE_ERR_ARG;
    scored *s = (scored *)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    if (!s)
        return ORACLE_ERR_NOMEM;
    for (int64_t i = 0; i < n; ++i) {
        s[i].v = vals[i];
        s[i].j = idx[i];
    }
    qsort(s, (size_t)n, sizeof(scored), by_score_then_index);
    for (int i = 0; i < k; ++i) {
        out_idx[i] = i < n ? s[i].j : -1;
        if (out_val)
            out_val[i] = i < n ? s[i].v : -INFINITY;
    }
    free(s);
    return ORACLE_OK;
}

/*
 * Per-row top-k over dense rows vals[r, 0..ld).  Key j of row r is eligible
 * when j < compress_len[r] and, if a mask is given, mask[r, j / mask_block]
 * is non-zero.  out_idx[r, 0..k): eligible keys in rank order, then -1.
 */
int oracle_topk(int64_t nrows, const double *vals, int64_t ld, const int32_t *compress_len,
                const uint8_t *mask, int64_t ld_mask, int mask_block, int k,
                int32_t *out_idx, double *out_val, int nthreads)
{
    if (nrows < 0 || k < 0 || ld < 0 || (mask && mask_block <= 0))
        return ORACLE_ERR_ARG;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t clen = compress_len[r];
        if (clen > ld)
            clen = ld;
        if (clen < 0)
            clen = 0;
        scored *s = (scored *)malloc(sizeof(scored) * (size_t)(clen > 0 ? clen : 1));
        if (!s) {
            bad |= 1;
            continue;
        }
        int64_t n = 0;
        for (int64_t j = 0; j < clen; ++j) {
            if (mask && !mask[r * ld_mask + j / mask_block])
                continue;
            s[n].v = vals[r * ld + j];
            s[n].j = j;
            ++n;
        }
        qsort(s, (size_t)n, sizeof(scored), by_score_then_index);
        for (int i = 0; i < k; ++i) {
            out_idx[r * k + i] = i < n ? (int32_t)s[i].j : -1;
            if (out_val)
                out_val[r * k + i] = i < n ? s[i].v : -INFINITY;
        }
        free(s);
    }
    return bad ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * Candidate blocks: pooled[b] = max of vals[r, j] over eligible keys j in
 * [block*b, block*b + block); block b exists when block*b < compress_len[r].
 * The cand_topk existing blocks with the largest pooled score (ties to the
 * lower block index) get mask byte 1; every other byte of the row's
 * ld_mask bytes gets 0.  If pooled_out is given it receives the pooled
 * scores (-inf for blocks that do not exist), ld_mask per row.
 */
int oracle_candidates(int64_t nrows, const double *vals, int64_t ld,
                      const int32_t *compress_len, int block, int cand_topk,
                      uint8_t *mask_out, int64_t ld_mask, double *pooled_out, int nthreads)
{
    if (nrows < 0 || block <= 0 || cand_topk < 0 || ld_mask < 0)
        return ORACLE_ERR_ARG;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t clen = compress_len[r];
        if (clen > ld)
            clen = ld;
        if (clen < 0)
            clen = 0;
        int64_t nb = (clen + block - 1) / block;
        if (nb > ld_mask) {
            bad |= 2;
            continue;
        }
        scored *s = (scored *)malloc(sizeof(scored) * (size_t)(nb > 0 ? nb : 1));
        if (!s) {
            bad |= 1;
            continue;
        }
        for (int64_t b = 0; b < nb; ++b) {
            double m = -INFINITY;
            for (int64_t j = b * block; j < (b + 1) * block && j < clen; ++j)
                if (vals[r * ld + j] > m)
                    m = vals[r * ld + j];
            s[b].v = m;
            s[b].j = b;
        }
        if (pooled_out) {
            for (int64_t b = 0; b < ld_mask; ++b)
                pooled_out[r * ld_mask + b] = b < nb ? s[b].v : -INFINITY;
        }
        qsort(s, (size_t)nb, sizeof(scored), by_score_then_index);
        memset(mask_out + r * ld_mask, 0, (size_t)ld_mask);
        for (int64_t i = 0; i < nb && i < cand_topk; ++i)
            mask_out[r * ld_mask + s[i].j] = 1;
        free(s);
    }
    if (bad & 2)
        return ORACLE_ERR_ARG;
    return bad ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
