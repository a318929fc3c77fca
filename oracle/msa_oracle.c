/*
 * msa_oracle.c -- plain, slow, obviously-correct CPU oracle of MSA (MiniMax
 * Sparse Attention) block-sparse GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path calls, links or loads
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Source of every formula: the page «MiniMax-M3：MSA 技术报告速读» (MSA tech-report
 * digest), section 核心机制：两个分支，先选后算 (two branches, select then compute):
 *   - 索引分支 (Index Branch): token score S^{idx,(r)}_{i,j} = Q^idx(r)_i . K^idx_j / sqrt(d_idx)
 *     and block score M^{idx,(r)}_{i,b} = max over j in block b with j <= i (eq. S^idx / M^idx);
 *     selection I^{(r)}_i = TopK_b(M^{idx,(r)}_{i,.}, k) (eq. I^(r)_i), done per GQA group,
 *     with the query's own (local) block always included (two key details, second item).
 *   - 主分支 (Main Branch): O^{(h)}_i = softmax(Q^(h)_i K^(r)[I]^T / sqrt(d_h)) V^(r)[I] over
 *     the visible tokens of the selected blocks; all query heads of group r share I^(r)_i
 *     (eq. O^(h)_i).
 *   - section Kernel: the forward also emits the per-row log-sum-exp (LSE).
 * and the section 训练：top-k 不可导怎么办 (training), eq. P^idx / P / L_KL: the KL alignment
 *   loss of a row and group over its selected token set, the main branch's group-averaged
 *   attention (teacher) against the index branch's softmax (student); and its gradient with
 *   respect to the index branch's inputs with the teacher held fixed (gradient detach).
 *
 * Readings where the page is silent (each is listed with its reason in the design notes):
 *   - k counts the forced local block: I = {l} U top-(k-1) of the blocks b < l.
 *   - ties in the block score go to the lower block index.
 *   - only tokens j <= i are visible, inside the local block too; blocks entirely in the
 *     future have block score -inf and are never selected.
 *   - fewer than k visible blocks: all of them are selected, the rest is -1.
 *   - head h belongs to group r = h / (H_q / H_kv); index head r pairs with KV head r.
 *   - LSE is the natural log of the sum of exp of the scaled scores.
 *   - I is stored ascending, padded with -1.
 *   - the selection compares block scores rounded once to fp32 (the precision the
 *     CUDA path decides in); everything else is fp64 from exactly-widened bf16 inputs.
 *   - decode: the query is the last cache row i = L-1 of its sequence.
 *   - KL loss: the selected token set is the main branch's T (visible tokens of the selected
 *     blocks); both softmaxes normalise over T; the teacher's scores are the main branch's
 *     scaled scores; the result is one value per (row, group), no reduction over rows.
 *
 * Layouts (row-major, bf16 passed as uint16 bit patterns):
 *   Q [N,H_q,d_h], K,V [N,H_kv,d_h], Q_idx [N,H_kv,d_idx], K_idx [N,d_idx],
 *   M [H_kv, q_count, nblk], I [H_kv, N, k], O [rows,H_q,d_h], LSE [rows,H_q].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- numbers -- */

/* Exact widening of a bf16 bit pattern (the top half of an IEEE binary32). */
static double bf16_to_f64(uint16_t u)
{
    uint32_t bits = (uint32_t)u << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round an fp64 value to bf16 (8 significant bits, 8-bit exponent like binary32),
 * round-to-nearest-even, straight from the definition: scale the value so that its
 * last kept bit is the unit, round to an integer with ties to even, scale back. */
static uint16_t f64_to_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    int e;
    (void)frexp(fabs(x), &e);            /* |x| = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                       /* weight of the 8th significant bit */
    if (q < -133) q = -133;              /* bf16 subnormal step 2^-133 */
    double r = nearbyint(ldexp(fabs(x), -q));   /* default mode: nearest, ties even */
    double y = ldexp(r, q);
    float f = (float)y;                  /* exact (<= 8 significant bits) or inf */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t h = (uint16_t)(bits >> 16);
    if (x < 0) h |= 0x8000;
    return h;
}

static int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

/* ------------------------------------------------------ index branch (L1) -- */

/* Block scores of one (query i, group r) row:
 *   S_j = (sum_d Q_idx[i,r,d] * K_idx[j,d]) / sqrt(d_idx)   for j = 0..i
 *   M_b = max_{j in block b, j <= i} S_j                     for b = 0..floor(i/B)
 * qrow points at Q_idx[i, r, 0]; kidx at K_idx[0, 0] of the sequence. */
static void row_block_scores(const uint16_t *qrow, const uint16_t *kidx, int64_t i,
                             int d_idx, int B, double *Mrow)
{
    const double scale = 1.0 / sqrt((double)d_idx);
    const int64_t l = i / B;
    for (int64_t b = 0; b <= l; ++b) Mrow[b] = -INFINITY;
    for (int64_t j = 0; j <= i; ++j) {
        const uint16_t *krow = kidx + j * (int64_t)d_idx;
        double dot = 0.0;
        for (int d = 0; d < d_idx; ++d) dot += bf16_to_f64(qrow[d]) * bf16_to_f64(krow[d]);
        const double s = dot * scale;
        const int64_t b = j / B;
        if (s > Mrow[b]) Mrow[b] = s;
    }
}

/* ------------------------------------------------ selection (TopK + local) -- */

typedef struct { float m; int32_t b; } cand_t;

/* Higher block score first; equal scores: lower block index first. */
static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *c = (const cand_t *)pb;
    if (a->m > c->m) return -1;
    if (a->m < c->m) return 1;
    return (a->b > c->b) - (a->b < c->b);
}

static int int_cmp(const void *pa, const void *pb)
{
    const int32_t a = *(const int32_t *)pa, c = *(const int32_t *)pb;
    return (a > c) - (a < c);
}

/* I = {l} U (the k-1 best blocks b < l by (M desc, b asc)); all visible blocks when
 * l + 1 <= k.  Output ascending, padded with -1. */
static void row_select(const float *Mrow, int64_t l, int k, int32_t *out)
{
    int n = 0;
    if (l + 1 <= k) {
        for (int64_t b = 0; b <= l; ++b) out[n++] = (int32_t)b;
    } else {
        cand_t *c = (cand_t *)malloc((size_t)l * sizeof(cand_t));
        for (int64_t b = 0; b < l; ++b) { c[b].m = Mrow[b]; c[b].b = (int32_t)b; }
        qsort(c, (size_t)l, sizeof(cand_t), cand_cmp);
        for (int t = 0; t < k - 1; ++t) out[n++] = c[t].b;
        free(c);
        qsort(out, (size_t)n, sizeof(int32_t), int_cmp);
        out[n++] = (int32_t)l;                  /* every other pick is < l */
    }
    for (; n < k; ++n) out[n] = -1;
}

/* ----------------------------------------------------- main branch (L3) ---- */

/* For every query head h of row i (group r = h / G), over the visible tokens T of the
 * blocks listed in sel[r*kk .. r*kk+kk-1] (entries < 0 are skipped):
 *   s_j = Q[i,h] . K[j,r] / sqrt(d_h),  LSE = ln sum_j exp(s_j),  O = sum_j exp(s_j - LSE) V[j,r]
 * q_i points at Q[i,0,0]; K, V at token 0 of the sequence. */
static void row_attend(const uint16_t *q_i, const uint16_t *K, const uint16_t *V, int64_t i,
                       int H_q, int H_kv, int d_h, int B, const int32_t *sel, int kk,
                       double *O, double *lse, double *s_buf, int64_t *j_buf)
{
    const int G = H_q / H_kv;
    const double scale = 1.0 / sqrt((double)d_h);
    for (int h = 0; h < H_q; ++h) {
        const int r = h / G;
        const uint16_t *qh = q_i + (int64_t)h * d_h;
        int64_t nt = 0;
        for (int t = 0; t < kk; ++t) {
            const int64_t b = sel[r * kk + t];
            if (b < 0) continue;
            const int64_t j1 = imin64(b * B + B - 1, i);
            for (int64_t j = b * B; j <= j1; ++j) {
                const uint16_t *kj = K + (j * H_kv + r) * (int64_t)d_h;
                double dot = 0.0;
                for (int d = 0; d < d_h; ++d) dot += bf16_to_f64(qh[d]) * bf16_to_f64(kj[d]);
                s_buf[nt] = dot * scale;
                j_buf[nt] = j;
                ++nt;
            }
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < nt; ++t) if (s_buf[t] > m) m = s_buf[t];
        double sum = 0.0;
        for (int64_t t = 0; t < nt; ++t) sum += exp(s_buf[t] - m);
        const double L = m + log(sum);
        lse[h] = L;
        double *oh = O + (int64_t)h * d_h;
        for (int d = 0; d < d_h; ++d) oh[d] = 0.0;
        for (int64_t t = 0; t < nt; ++t) {
            const double p = exp(s_buf[t] - L);
            const uint16_t *vj = V + (j_buf[t] * H_kv + r) * (int64_t)d_h;
            for (int d = 0; d < d_h; ++d) oh[d] += p * bf16_to_f64(vj[d]);
        }
    }
}

/* ------------------------------------------------ KL alignment loss (L4) -- */

/* KL alignment loss of row i, group r over the selected token set T (the visible tokens of
 * the blocks sel[0..kk), entries < 0 skipped):
 *   student  P^idx_j = exp(S^idx_j) / sum_{u in T} exp(S^idx_u),
 *            S^idx_j = Q_idx[i,r] . K_idx[j] / sqrt(d_idx)
 *   teacher  P_j = (1/G) sum over the G heads h of group r of exp(s^h_j) / sum_{u in T} exp(s^h_u),
 *            s^h_j = Q[i,h] . K[j,r] / sqrt(d_h)
 *   KL = sum_{j in T} P_j (ln P_j - ln P^idx_j)      (a term with P_j = 0 contributes 0)
 * q_i points at Q[i,0,0], qidx_ir at Q_idx[i,r,0]; K, K_idx at token 0 of the sequence. */
static double row_kl(const uint16_t *q_i, const uint16_t *qidx_ir, const uint16_t *K,
                     const uint16_t *K_idx, int64_t i, int r, int H_q, int H_kv, int d_h,
                     int d_idx, int B, const int32_t *sel, int kk, double *s_buf, double *p_buf,
                     int64_t *j_buf)
{
    const int G = H_q / H_kv;
    int64_t nt = 0;
    for (int t = 0; t < kk; ++t) {
        const int64_t b = sel[t];
        if (b < 0) continue;
        const int64_t j1 = imin64(b * B + B - 1, i);
        for (int64_t j = b * B; j <= j1; ++j) j_buf[nt++] = j;
    }
    /* teacher: the mean over the group's heads of each head's softmax over T */
    const double scale_h = 1.0 / sqrt((double)d_h);
    for (int64_t t = 0; t < nt; ++t) p_buf[t] = 0.0;
    for (int h = r * G; h < (r + 1) * G; ++h) {
        const uint16_t *qh = q_i + (int64_t)h * d_h;
        double m = -INFINITY;
        for (int64_t t = 0; t < nt; ++t) {
            const uint16_t *kj = K + (j_buf[t] * H_kv + r) * (int64_t)d_h;
            double dot = 0.0;
            for (int d = 0; d < d_h; ++d) dot += bf16_to_f64(qh[d]) * bf16_to_f64(kj[d]);
            s_buf[t] = dot * scale_h;
            if (s_buf[t] > m) m = s_buf[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < nt; ++t) z += exp(s_buf[t] - m);
        for (int64_t t = 0; t < nt; ++t) p_buf[t] += exp(s_buf[t] - m) / z / G;
    }
    /* student: the index branch's softmax over T, kept as log-probabilities */
    const double scale_idx = 1.0 / sqrt((double)d_idx);
    double m = -INFINITY;
    for (int64_t t = 0; t < nt; ++t) {
        const uint16_t *kj = K_idx + j_buf[t] * (int64_t)d_idx;
        double dot = 0.0;
        for (int d = 0; d < d_idx; ++d) dot += bf16_to_f64(qidx_ir[d]) * bf16_to_f64(kj[d]);
        s_buf[t] = dot * scale_idx;
        if (s_buf[t] > m) m = s_buf[t];
    }
    double z = 0.0;
    for (int64_t t = 0; t < nt; ++t) z += exp(s_buf[t] - m);
    const double lse_idx = m + log(z);
    double kl = 0.0;
    for (int64_t t = 0; t < nt; ++t)
        if (p_buf[t] > 0.0) kl += p_buf[t] * (log(p_buf[t]) - (s_buf[t] - lse_idx));
    return kl;
}

/* Gradient of L = sum over rows of g[r,i] * KL[r,i] with respect to the index branch's inputs
 * for one (row i, group r), the teacher held fixed (the gradient detach of section 训练):
 *   dKL/dS^idx_j = (sum_u P_u) P^idx_j - P_j      (the KL as defined above, differentiated)
 *   dQ_idx[i,r] += g sum_j dS_j K_idx[j] / sqrt(d_idx),  dK_idx[j] += g dS_j Q_idx[i,r] / sqrt(d_idx)
 * dq: [d_idx] for this row; dk: [N, d_idx] accumulated.  Also returns the student's LSE over T
 * and the teacher's total mass sum_j P_j in *lse_idx_out, *psum_out. */
static void row_kl_grad(const uint16_t *q_i, const uint16_t *qidx_ir, const uint16_t *K,
                        const uint16_t *K_idx, int64_t i, int r, int H_q, int H_kv, int d_h,
                        int d_idx, int B, const int32_t *sel, int kk, double g, double *dq,
                        double *dk, double *lse_idx_out, double *psum_out, double *s_buf,
                        double *p_buf, int64_t *j_buf)
{
    const int G = H_q / H_kv;
    int64_t nt = 0;
    for (int t = 0; t < kk; ++t) {
        const int64_t b = sel[t];
        if (b < 0) continue;
        const int64_t j1 = imin64(b * B + B - 1, i);
        for (int64_t j = b * B; j <= j1; ++j) j_buf[nt++] = j;
    }
    const double scale_h = 1.0 / sqrt((double)d_h);
    for (int64_t t = 0; t < nt; ++t) p_buf[t] = 0.0;
    for (int h = r * G; h < (r + 1) * G; ++h) {
        const uint16_t *qh = q_i + (int64_t)h * d_h;
        double m = -INFINITY;
        for (int64_t t = 0; t < nt; ++t) {
            const uint16_t *kj = K + (j_buf[t] * H_kv + r) * (int64_t)d_h;
            double dot = 0.0;
            for (int d = 0; d < d_h; ++d) dot += bf16_to_f64(qh[d]) * bf16_to_f64(kj[d]);
            s_buf[t] = dot * scale_h;
            if (s_buf[t] > m) m = s_buf[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < nt; ++t) z += exp(s_buf[t] - m);
        for (int64_t t = 0; t < nt; ++t) p_buf[t] += exp(s_buf[t] - m) / z / G;
    }
    const double scale_idx = 1.0 / sqrt((double)d_idx);
    double m = -INFINITY;
    for (int64_t t = 0; t < nt; ++t) {
        const uint16_t *kj = K_idx + j_buf[t] * (int64_t)d_idx;
        double dot = 0.0;
        for (int d = 0; d < d_idx; ++d) dot += bf16_to_f64(qidx_ir[d]) * bf16_to_f64(kj[d]);
        s_buf[t] = dot * scale_idx;
        if (s_buf[t] > m) m = s_buf[t];
    }
    double z = 0.0, psum = 0.0;
    for (int64_t t = 0; t < nt; ++t) {
        z += exp(s_buf[t] - m);
        psum += p_buf[t];
    }
    const double lse_idx = m + log(z);
    *lse_idx_out = lse_idx;
    *psum_out = psum;
    for (int d = 0; d < d_idx; ++d) dq[d] = 0.0;
    for (int64_t t = 0; t < nt; ++t) {
        const double ds = g * (psum * exp(s_buf[t] - lse_idx) - p_buf[t]) * scale_idx;
        const uint16_t *kj = K_idx + j_buf[t] * (int64_t)d_idx;
        double *dkj = dk + j_buf[t] * (int64_t)d_idx;
        for (int d = 0; d < d_idx; ++d) {
            dq[d] += ds * bf16_to_f64(kj[d]);
            dkj[d] += ds * bf16_to_f64(qidx_ir[d]);
        }
    }
}

/* ------------------------------------------- main branch backward (L3) ---- */

/* Gradient of the main branch for row i given dO [H_q, d_h] (bf16 bits) of that row, for every
 * head h (group r = h / G), over the same T as row_attend:
 *   p_j = exp(s_j - LSE),  dP_j = dO[i,h] . V[j,r],  D = sum_j p_j dP_j,  dS_j = p_j (dP_j - D)
 *   dQ[i,h] = sum_j dS_j K[j,r] / sqrt(d_h),  dK[j,r] += dS_j Q[i,h] / sqrt(d_h),
 *   dV[j,r] += p_j dO[i,h]
 * (the softmax attention of eq. O^(h)_i differentiated).  dq: [H_q, d_h] for this row; dk, dv:
 * [N, H_kv, d_h] accumulated. */
static void row_attend_grad(const uint16_t *q_i, const uint16_t *do_i, const uint16_t *K,
                            const uint16_t *V, int64_t i, int H_q, int H_kv, int d_h, int B,
                            const int32_t *sel, int kk, int h_begin, int h_end, double *dq,
                            double *dk, double *dv, double *s_buf, double *p_buf, int64_t *j_buf)
{
    const int G = H_q / H_kv;
    const double scale = 1.0 / sqrt((double)d_h);
    for (int h = h_begin; h < h_end; ++h) {
        const int r = h / G;
        const uint16_t *qh = q_i + (int64_t)h * d_h, *doh = do_i + (int64_t)h * d_h;
        int64_t nt = 0;
        for (int t = 0; t < kk; ++t) {
            const int64_t b = sel[r * kk + t];
            if (b < 0) continue;
            const int64_t j1 = imin64(b * B + B - 1, i);
            for (int64_t j = b * B; j <= j1; ++j) {
                const uint16_t *kj = K + (j * H_kv + r) * (int64_t)d_h;
                double dot = 0.0;
                for (int d = 0; d < d_h; ++d) dot += bf16_to_f64(qh[d]) * bf16_to_f64(kj[d]);
                s_buf[nt] = dot * scale;
                j_buf[nt] = j;
                ++nt;
            }
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < nt; ++t) if (s_buf[t] > m) m = s_buf[t];
        double z = 0.0;
        for (int64_t t = 0; t < nt; ++t) z += exp(s_buf[t] - m);
        const double L = m + log(z);
        double D = 0.0;
        for (int64_t t = 0; t < nt; ++t) {
            const uint16_t *vj = V + (j_buf[t] * H_kv + r) * (int64_t)d_h;
            double dp = 0.0;
            for (int d = 0; d < d_h; ++d) dp += bf16_to_f64(doh[d]) * bf16_to_f64(vj[d]);
            p_buf[t] = exp(s_buf[t] - L);
            s_buf[t] = dp;                                    /* dP_j from here on */
            D += p_buf[t] * dp;
        }
        double *dqh = dq + (int64_t)h * d_h;
        for (int d = 0; d < d_h; ++d) dqh[d] = 0.0;
        for (int64_t t = 0; t < nt; ++t) {
            const double ds = p_buf[t] * (s_buf[t] - D) * scale;
            const int64_t row = (j_buf[t] * H_kv + r) * (int64_t)d_h;
            for (int d = 0; d < d_h; ++d) {
                dqh[d] += ds * bf16_to_f64(K[row + d]);
                dk[row + d] += ds * bf16_to_f64(qh[d]);
                dv[row + d] += p_buf[t] * bf16_to_f64(doh[d]);
            }
        }
    }
}

/* ------------------------------------------------------------- exports ----- */

void msa_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int msa_oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Index-branch block scores for query rows [q_start, q_start+q_count).
 * M64 (nullable): fp64 [H_kv, q_count, nblk]; M32 (nullable): the same rounded once to
 * fp32.  Entries of blocks after the query's own block are -inf. */
void msa_oracle_block_scores(const uint16_t *q_idx, const uint16_t *k_idx, int64_t N, int H_kv,
                             int d_idx, int B, int64_t q_start, int64_t q_count, double *M64,
                             float *M32)
{
    const int64_t nblk = (N + B - 1) / B;
#pragma omp parallel
    {
        double *row = (double *)malloc((size_t)nblk * sizeof(double));
#pragma omp for schedule(dynamic, 4) collapse(2)
        for (int r = 0; r < H_kv; ++r)
            for (int64_t t = 0; t < q_count; ++t) {
                const int64_t i = q_start + t;
                const int64_t l = i / B;
                row_block_scores(q_idx + (i * H_kv + r) * (int64_t)d_idx, k_idx, i, d_idx, B, row);
                const int64_t o = ((int64_t)r * q_count + t) * nblk;
                for (int64_t b = 0; b < nblk; ++b) {
                    const double v = b <= l ? row[b] : -INFINITY;
                    if (M64) M64[o + b] = v;
                    if (M32) M32[o + b] = (float)v;
                }
            }
        free(row);
    }
}

/* Per-group block selection for rows [q_start, q_start+q_count) from fp32 block scores
 * M [H_kv, q_count, nblk]; writes I [H_kv, N, k] rows q_start.. */
void msa_oracle_select_blocks(const float *M, int64_t N, int H_kv, int B, int k,
                              int64_t q_start, int64_t q_count, int32_t *I)
{
    const int64_t nblk = (N + B - 1) / B;
#pragma omp parallel for schedule(dynamic, 16) collapse(2)
    for (int r = 0; r < H_kv; ++r)
        for (int64_t t = 0; t < q_count; ++t) {
            const int64_t i = q_start + t;
            row_select(M + ((int64_t)r * q_count + t) * nblk, i / B, k,
                       I + ((int64_t)r * N + i) * k);
        }
}

/* Main branch for the given rows (rows == NULL: all N rows) with a given selection
 * I [H_kv, N, kk].  O64 [n_rows,H_q,d_h], O16 (nullable, bf16 RNE of O64),
 * LSE [n_rows,H_q]. */
void msa_oracle_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int32_t *I, int64_t N, int H_q, int H_kv, int d_h, int B,
                            int kk, const int64_t *rows, int64_t n_rows, double *O64,
                            uint16_t *O16, double *LSE)
{
    if (!rows) n_rows = N;
#pragma omp parallel
    {
        double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
        int32_t *sel = (int32_t *)malloc((size_t)H_kv * kk * sizeof(int32_t));
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < n_rows; ++t) {
            const int64_t i = rows ? rows[t] : t;
            for (int r = 0; r < H_kv; ++r)
                for (int u = 0; u < kk; ++u) sel[r * kk + u] = I[((int64_t)r * N + i) * kk + u];
            double *o = O64 + t * H_q * (int64_t)d_h;
            row_attend(q + i * H_q * (int64_t)d_h, k, v, i, H_q, H_kv, d_h, B, sel, kk, o,
                       LSE + t * H_q, s_buf, j_buf);
            if (O16)
                for (int64_t e = 0; e < (int64_t)H_q * d_h; ++e)
                    O16[t * H_q * (int64_t)d_h + e] = f64_to_bf16(o[e]);
        }
        free(s_buf);
        free(j_buf);
        free(sel);
    }
}

/* Main branch for the listed rows only, with their projections and selections given compactly:
 * row t is query position rows[t]; q_rows [n_rows,H_q,d_h] and I_rows [n_rows,H_kv,kk] hold that
 * row's queries and selection; K, V are the full sequence.  Outputs as msa_oracle_sparse_attn. */
void msa_oracle_sparse_attn_rows(const uint16_t *q_rows, const uint16_t *k, const uint16_t *v,
                                 const int32_t *I_rows, int H_q, int H_kv, int d_h, int B, int kk,
                                 const int64_t *rows, int64_t n_rows, double *O64, uint16_t *O16,
                                 double *LSE)
{
#pragma omp parallel
    {
        double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < n_rows; ++t) {
            double *o = O64 + t * H_q * (int64_t)d_h;
            row_attend(q_rows + t * H_q * (int64_t)d_h, k, v, rows[t], H_q, H_kv, d_h, B,
                       I_rows + t * H_kv * (int64_t)kk, kk, o, LSE + t * H_q, s_buf, j_buf);
            if (O16)
                for (int64_t e = 0; e < (int64_t)H_q * d_h; ++e)
                    O16[t * H_q * (int64_t)d_h + e] = f64_to_bf16(o[e]);
        }
        free(s_buf);
        free(j_buf);
    }
}

/* The whole prefill path (scores -> selection -> main branch) for the given rows only.
 * q_rows [n_rows,H_q,d_h] and q_idx_rows [n_rows,H_kv,d_idx] hold the projections of the
 * listed rows only (row t is query position rows[t]); K, V, K_idx are the full sequence.
 * I_out [n_rows,H_kv,kk]; M32_out (nullable) [n_rows,H_kv,nblk]; O64/O16/LSE as above. */
void msa_oracle_prefill_rows(const uint16_t *q_rows, const uint16_t *k, const uint16_t *v,
                             const uint16_t *q_idx_rows, const uint16_t *k_idx, int64_t N, int H_q,
                             int H_kv, int d_h, int d_idx, int B, int kk, const int64_t *rows,
                             int64_t n_rows, int32_t *I_out, float *M32_out, double *O64,
                             uint16_t *O16, double *LSE)
{
    const int64_t nblk = (N + B - 1) / B;
#pragma omp parallel
    {
        double *m64 = (double *)malloc((size_t)nblk * sizeof(double));
        float *m32 = (float *)malloc((size_t)nblk * sizeof(float));
        double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
        int32_t *sel = (int32_t *)malloc((size_t)H_kv * kk * sizeof(int32_t));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n_rows; ++t) {
            const int64_t i = rows[t];
            const int64_t l = i / B;
            for (int r = 0; r < H_kv; ++r) {
                row_block_scores(q_idx_rows + (t * H_kv + r) * (int64_t)d_idx, k_idx, i, d_idx, B,
                                 m64);
                for (int64_t b = 0; b < nblk; ++b) m32[b] = b <= l ? (float)m64[b] : -INFINITY;
                if (M32_out) memcpy(M32_out + (t * H_kv + r) * nblk, m32, (size_t)nblk * sizeof(float));
                row_select(m32, l, kk, sel + r * kk);
            }
            memcpy(I_out + t * H_kv * (int64_t)kk, sel, (size_t)H_kv * kk * sizeof(int32_t));
            double *o = O64 + t * H_q * (int64_t)d_h;
            row_attend(q_rows + t * H_q * (int64_t)d_h, k, v, i, H_q, H_kv, d_h, B, sel, kk, o,
                       LSE + t * H_q, s_buf, j_buf);
            if (O16)
                for (int64_t e = 0; e < (int64_t)H_q * d_h; ++e)
                    O16[t * H_q * (int64_t)d_h + e] = f64_to_bf16(o[e]);
        }
        free(m64);
        free(m32);
        free(s_buf);
        free(j_buf);
        free(sel);
    }
}

/* Decode: for each listed sequence s (seqs == NULL: all S), the query is the new token,
 * cache row i = L_s - 1 of the packed cache (rows cu_seqlens[s] .. cu_seqlens[s+1]-1),
 * with q [S,H_q,d_h] and q_idx [S,H_kv,d_idx] holding the new token's projections.
 * Runs scores -> selection -> main branch on that one row.
 * I_out [n,H_kv,kk]; M32_out (nullable) [n,H_kv,m32_stride]; O64/O16 [n,H_q,d_h]; LSE [n,H_q]. */
void msa_oracle_decode(const uint16_t *q, const uint16_t *q_idx, const uint16_t *k_cache,
                       const uint16_t *v_cache, const uint16_t *k_idx_cache,
                       const int64_t *cu_seqlens, int S, int H_q, int H_kv, int d_h, int d_idx,
                       int B, int kk, const int32_t *seqs, int n_seqs, int32_t *I_out,
                       float *M32_out, int64_t m32_stride, double *O64, uint16_t *O16,
                       double *LSE)
{
    if (!seqs) n_seqs = S;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < n_seqs; ++t) {
        const int s = seqs ? seqs[t] : t;
        const int64_t base = cu_seqlens[s];
        const int64_t L = cu_seqlens[s + 1] - base;
        const int64_t i = L - 1;
        const int64_t l = i / B;
        double *m64 = (double *)malloc((size_t)(l + 1) * sizeof(double));
        float *m32 = (float *)malloc((size_t)(l + 1) * sizeof(float));
        double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
        int32_t *sel = I_out + (int64_t)t * H_kv * kk;
        for (int r = 0; r < H_kv; ++r) {
            row_block_scores(q_idx + ((int64_t)s * H_kv + r) * d_idx, k_idx_cache + base * d_idx,
                             i, d_idx, B, m64);
            for (int64_t b = 0; b <= l; ++b) m32[b] = (float)m64[b];
            if (M32_out) {
                float *dst = M32_out + ((int64_t)t * H_kv + r) * m32_stride;
                for (int64_t b = 0; b < m32_stride; ++b) dst[b] = b <= l ? m32[b] : -INFINITY;
            }
            row_select(m32, l, kk, sel + r * kk);
        }
        double *o = O64 + (int64_t)t * H_q * d_h;
        row_attend(q + (int64_t)s * H_q * d_h, k_cache + base * H_kv * (int64_t)d_h,
                   v_cache + base * H_kv * (int64_t)d_h, i, H_q, H_kv, d_h, B, sel, kk, o,
                   LSE + (int64_t)t * H_q, s_buf, j_buf);
        if (O16)
            for (int64_t e = 0; e < (int64_t)H_q * d_h; ++e)
                O16[(int64_t)t * H_q * d_h + e] = f64_to_bf16(o[e]);
        free(m64);
        free(m32);
        free(s_buf);
        free(j_buf);
    }
}

/* KL alignment loss for the listed rows: row t is query position rows[t]; q_rows [n,H_q,d_h],
 * q_idx_rows [n,H_kv,d_idx] and I_rows [n,H_kv,kk] hold that row's projections and selection;
 * K, K_idx are the full sequence.  KL [n, H_kv], fp64. */
void msa_oracle_kl_loss(const uint16_t *q_rows, const uint16_t *k, const uint16_t *q_idx_rows,
                        const uint16_t *k_idx, const int32_t *I_rows, int H_q, int H_kv, int d_h,
                        int d_idx, int B, int kk, const int64_t *rows, int64_t n_rows, double *KL)
{
#pragma omp parallel
    {
        double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        double *p_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < n_rows; ++t)
            for (int r = 0; r < H_kv; ++r)
                KL[t * H_kv + r] = row_kl(q_rows + t * H_q * (int64_t)d_h,
                                          q_idx_rows + (t * H_kv + r) * (int64_t)d_idx, k, k_idx,
                                          rows[t], r, H_q, H_kv, d_h, d_idx, B,
                                          I_rows + (t * H_kv + r) * (int64_t)kk, kk, s_buf, p_buf,
                                          j_buf);
        free(s_buf);
        free(p_buf);
        free(j_buf);
    }
}

/* Index-branch gradient of L = sum_{r,i} G_KL[r,i] KL[r,i] over all N rows, teacher fixed.
 * G_KL [H_kv, N] fp64; outputs dQ_idx [N, H_kv, d_idx], dK_idx [N, d_idx] (fp64, overwritten),
 * LSE_idx [H_kv, N] (the student's LSE over T) and PSUM [H_kv, N] (the teacher's mass over T).
 * Single-threaded over rows for dK_idx (a plain sum in row order). */
void msa_oracle_kl_loss_grad(const uint16_t *q, const uint16_t *k, const uint16_t *q_idx,
                             const uint16_t *k_idx, const int32_t *I, const double *G_KL,
                             int64_t N, int H_q, int H_kv, int d_h, int d_idx, int B, int kk,
                             double *dQ_idx, double *dK_idx, double *LSE_idx, double *PSUM)
{
    double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
    double *p_buf = (double *)malloc((size_t)kk * B * sizeof(double));
    int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
    for (int64_t e = 0; e < N * (int64_t)d_idx; ++e) dK_idx[e] = 0.0;
    for (int64_t i = 0; i < N; ++i)
        for (int r = 0; r < H_kv; ++r)
            row_kl_grad(q + i * H_q * (int64_t)d_h, q_idx + (i * H_kv + r) * (int64_t)d_idx, k,
                        k_idx, i, r, H_q, H_kv, d_h, d_idx, B, I + ((int64_t)r * N + i) * kk, kk,
                        G_KL[(int64_t)r * N + i], dQ_idx + (i * H_kv + r) * (int64_t)d_idx, dK_idx,
                        LSE_idx + (int64_t)r * N + i, PSUM + (int64_t)r * N + i, s_buf, p_buf,
                        j_buf);
    free(s_buf);
    free(p_buf);
    free(j_buf);
}

/* Main-branch gradient over all N rows with a given selection I [H_kv, N, kk] and upstream dO
 * [N, H_q, d_h] (bf16 bits): dQ [N, H_q, d_h], dK, dV [N, H_kv, d_h] (fp64, overwritten).
 * One thread per KV group r (only the heads of group r touch dK[:, r] and dV[:, r]); within a
 * group, dK and dV are plain sums in row order, then head order. */
void msa_oracle_sparse_attn_grad(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const uint16_t *dO, const int32_t *I, int64_t N, int H_q,
                                 int H_kv, int d_h, int B, int kk, double *dQ, double *dK,
                                 double *dV)
{
    const int G = H_q / H_kv;
    for (int64_t e = 0; e < N * (int64_t)H_kv * d_h; ++e) dK[e] = dV[e] = 0.0;
#pragma omp parallel for schedule(static, 1)
    for (int r = 0; r < H_kv; ++r) {
        double *s_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        double *p_buf = (double *)malloc((size_t)kk * B * sizeof(double));
        int64_t *j_buf = (int64_t *)malloc((size_t)kk * B * sizeof(int64_t));
        int32_t *sel = (int32_t *)malloc((size_t)H_kv * kk * sizeof(int32_t));
        for (int64_t i = 0; i < N; ++i) {
            for (int u = 0; u < kk; ++u) sel[r * kk + u] = I[((int64_t)r * N + i) * kk + u];
            row_attend_grad(q + i * H_q * (int64_t)d_h, dO + i * H_q * (int64_t)d_h, k, v, i,
                            H_q, H_kv, d_h, B, sel, kk, r * G, (r + 1) * G,
                            dQ + i * H_q * (int64_t)d_h, dK, dV, s_buf, p_buf, j_buf);
        }
        free(s_buf);
        free(p_buf);
        free(j_buf);
        free(sel);
    }
}

/* Exposed for the pins on the rounding step. */
uint16_t msa_oracle_f64_to_bf16(double x) { return f64_to_bf16(x); }
double msa_oracle_bf16_to_f64(uint16_t u) { return bf16_to_f64(u); }
