/*
 * oracle.c -- plain, slow, fp64 CPU reference for block-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file; only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * with the CUDA path.
 *
 * What it computes (the plain definition, no blocking, no fusion):
 *   for every requested query row (b, hq, i), with kv head hk = hq / (Hq/Hkv):
 *     1. s_j   = scale * sum_d q[b,hq,i,d] * k[b,hk,j,d]   for all j < kv_len
 *        (one full row of the T x T score matrix, inputs upcast to double;
 *        FlexAttention Guide, "The Core Design Principles of FlexAttention",
 *        item 1: S_ij = q_i^T k_j / sqrt(d))
 *     2. s'_j  = score_mod(s_j, b, hq, i, j)           (same section, item 1)
 *     3. s'_j  = -inf where mask_mod(b, hq, i, j) is false   (item 2)
 *     4. safe softmax: M = max_j s'_j; if M = -inf the row attends to nothing
 *        and O = 0, lse = -inf; else p_j = exp(s'_j - M), L = sum p_j,
 *        O = sum_j p_j v[b,hk,j] / L, lse = M + ln L.
 *
 * The built-in score_mods and mask_mods follow the FlexAttention Guide:
 *   soft-cap    C * tanh(s / C), s already scaled by 1/sqrt(d)
 *               ("The Problem: The Custom Attention Fragility Wall", the
 *               soft-capping formula S_ij = C tanh(q^T k / (C sqrt d)))
 *   ALiBi       s - slope[hq] * |i - j|   ("Implementation" script, the
 *               composite score_mod's bias term)
 *   ALiBi then soft-cap   C * tanh((s - slope[hq] |i - j|) / C)
 *               ("Implementation" script, composite_score_mod: bias added
 *               first, the sum capped)
 *   rel. bias   s + table[hq][clamp(i - j, -R, R) + R]   (named in "The Core
 *               Design Principles", item 1, "position-dependent biases"; the
 *               table form is this library's reading)
 *   causal      i >= j                    ("Implementation" script)
 *   window      i >= j and i - j <= W     ("Implementation" script: the
 *               sliding-window mask is causal and (q_idx - kv_idx) <= 512)
 *   document    seg[i] == seg[j]          ("Production Engineering", item 1)
 *   prefix-LM   j < P or i >= j           ("Production Engineering", item 2)
 *   table       table[b][i][j] != 0       ("Production Engineering", item 3:
 *               tree attention's parent-child relation as a direct index
 *               lookup in mask_mod)
 *
 * The brute-force tile scan (oracle_block_mask) evaluates the same predicate
 * on every in-range pair of every 128 x 128 tile ("Systems Mechanics", item 1:
 * full / empty / partial blocks) and writes the index lists.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_MASK_FULL = 0, OR_MASK_CAUSAL = 1, OR_MASK_SLIDING_WINDOW = 2,
       OR_MASK_DOCUMENT = 3, OR_MASK_PREFIX_LM = 4, OR_MASK_TABLE = 5 };
enum { OR_SCORE_NONE = 0, OR_SCORE_SOFTCAP = 1, OR_SCORE_ALIBI = 2,
       OR_SCORE_REL_BIAS = 3, OR_SCORE_ALIBI_SOFTCAP = 4 };

typedef struct {
    int kind;
    int window;             /* sliding window: i - j <= window          */
    int prefix_len;         /* prefix-LM: j < prefix_len attends always */
    const int32_t *seg;     /* document: [seg_batch, seg_len]           */
    int seg_batch;
    int seg_len;
    const uint8_t *table;   /* table: [table_batch, table_q, table_kv], 1 = attend */
    int table_batch;
    int table_q;
    int table_kv;
} or_mask;

typedef struct {
    int kind;
    double softcap;
    const float *slopes;    /* [Hq]                  */
    const float *rel_bias;  /* [Hq, 2 * rel_max + 1] */
    int rel_max;
} or_score;

/* mask_mod(b, h, q_idx, kv_idx): the attend predicate. */
static int or_mask_mod(const or_mask *m, int b, int i, int j)
{
    switch (m->kind) {
    case OR_MASK_FULL:
        return 1;
    case OR_MASK_CAUSAL:
        return i >= j;
    case OR_MASK_SLIDING_WINDOW:
        return i >= j && (i - j) <= m->window;
    case OR_MASK_DOCUMENT: {
        const int32_t *row = m->seg + (size_t)(m->seg_batch == 1 ? 0 : b) * m->seg_len;
        return row[i] == row[j];
    }
    case OR_MASK_PREFIX_LM:
        return j < m->prefix_len || i >= j;
    case OR_MASK_TABLE: {
        /* a mask_mod that is a direct index lookup (tree attention's
           ancestor table) */
        const uint8_t *t = m->table + (size_t)(m->table_batch == 1 ? 0 : b) * m->table_q * m->table_kv;
        return t[(size_t)i * m->table_kv + j] != 0;
    }
    }
    return 0;
}

/* score_mod(score, b, h, q_idx, kv_idx) on an already scaled score. */
static double or_score_mod(const or_score *sc, double s, int h, int i, int j)
{
    switch (sc->kind) {
    case OR_SCORE_NONE:
        return s;
    case OR_SCORE_SOFTCAP:
        return sc->softcap * tanh(s / sc->softcap);
    case OR_SCORE_ALIBI:
        return s - (double)sc->slopes[h] * fabs((double)(i - j));
    case OR_SCORE_ALIBI_SOFTCAP: {
        /* the "Implementation" script's composite_score_mod: the ALiBi bias
           first, then the soft-cap of the biased score */
        const double u = s - (double)sc->slopes[h] * fabs((double)(i - j));
        return sc->softcap * tanh(u / sc->softcap);
    }
    case OR_SCORE_REL_BIAS: {
        int r = i - j;
        if (r < -sc->rel_max) r = -sc->rel_max;
        if (r > sc->rel_max) r = sc->rel_max;
        return s + (double)sc->rel_bias[(size_t)h * (2 * sc->rel_max + 1) + (r + sc->rel_max)];
    }
    }
    return s;
}

/* d score_mod / d s at the scaled score s (the biases do not depend on s). */
static double or_score_mod_ds(const or_score *sc, double s, int h, int i, int j)
{
    switch (sc->kind) {
    case OR_SCORE_SOFTCAP: {
        const double t = tanh(s / sc->softcap);
        return 1.0 - t * t;
    }
    case OR_SCORE_ALIBI_SOFTCAP: {
        const double u = s - (double)sc->slopes[h] * fabs((double)(i - j));
        const double t = tanh(u / sc->softcap);
        return 1.0 - t * t;
    }
    }
    return 1.0;
}

/*
 * Attention rows.  q: [B, Hq, Tq, D], k, v: [B, Hkv, Tkv, D] (fp32 values,
 * exact copies of bf16 inputs where the inputs are bf16).  rows[r] is the
 * flat index (b * Hq + hq) * Tq + i of the r-th requested row; out_o is
 * [nrows, D], out_lse is [nrows].  Returns 0, or -1 on bad arguments.
 */
int oracle_fwd_rows(const float *q, const float *k, const float *v,
                    int B, int Hq, int Hkv, int Tq, int Tkv, int D, double scale,
                    const or_mask *mask, const or_score *score,
                    const int64_t *rows, int64_t nrows,
                    double *out_o, double *out_lse, int nthreads)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Tq <= 0 || Tkv <= 0 || D <= 0)
        return -1;
    const int group = Hq / Hkv;
    int bad = 0;

#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1) reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Tkv);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !acc) {
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t flat = rows[r];
                const int i = (int)(flat % Tq);
                const int hq = (int)((flat / Tq) % Hq);
                const int b = (int)(flat / ((int64_t)Tq * Hq));
                if (flat < 0 || b >= B) { bad = 1; continue; }
                const int hk = hq / group;
                const float *qi = q + (((size_t)b * Hq + hq) * Tq + i) * D;
                const float *kb = k + ((size_t)b * Hkv + hk) * (size_t)Tkv * D;
                const float *vb = v + ((size_t)b * Hkv + hk) * (size_t)Tkv * D;

                /* steps 1-3: one full row of the score matrix */
                double M = -INFINITY;
                for (int j = 0; j < Tkv; ++j) {
                    const float *kj = kb + (size_t)j * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += (double)qi[d] * (double)kj[d];
                    double sj = or_score_mod(score, scale * dot, hq, i, j);
                    if (!or_mask_mod(mask, b, i, j))
                        sj = -INFINITY;
                    s[j] = sj;
                    if (sj > M) M = sj;
                }

                /* step 4: safe softmax and the weighted sum of V */
                double *o = out_o + (size_t)r * D;
                if (M == -INFINITY) {
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    out_lse[r] = -INFINITY;
                    continue;
                }
                double L = 0.0;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int j = 0; j < Tkv; ++j) {
                    if (s[j] == -INFINITY) continue;
                    const double p = exp(s[j] - M);
                    L += p;
                    const float *vj = vb + (size_t)j * D;
                    for (int d = 0; d < D; ++d)
                        acc[d] += p * (double)vj[d];
                }
                for (int d = 0; d < D; ++d) o[d] = acc[d] / L;
                out_lse[r] = M + log(L);
            }
        }
        free(s);
        free(acc);
    }
    return bad ? -1 : 0;
}

/*
 * Brute-force BlockMask.  For every (b < Bm, h < Hm, q-block, kv-block) tile
 * of block x block elements, counts the in-range pairs (i < Tq, j < Tkv) for
 * which mask_mod is true.  A tile is
 *   empty   when the count is 0,
 *   full    when the tile is complete (block x block pairs in range) and
 *           every pair is true,
 *   partial otherwise.
 * kv_num_blocks / full_kv_num_blocks: [Bm, Hm, nq]; kv_indices /
 * full_kv_indices: [Bm, Hm, nq, nkv], ascending kv-block index, unused
 * entries -1.  Partial tiles go to kv_*, full tiles to full_kv_*.
 */
int oracle_block_mask(const or_mask *mask, int Bm, int Hm, int Tq, int Tkv, int block,
                      int32_t *kv_num_blocks, int32_t *kv_indices,
                      int32_t *full_kv_num_blocks, int32_t *full_kv_indices, int nthreads)
{
    if (Bm <= 0 || Hm <= 0 || Tq <= 0 || Tkv <= 0 || block <= 0)
        return -1;
    const int nq = (Tq + block - 1) / block;
    const int nkv = (Tkv + block - 1) / block;

#pragma omp parallel for collapse(2) num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
    for (int bh = 0; bh < Bm * Hm; ++bh) {
        for (int qb = 0; qb < nq; ++qb) {
            const int b = bh / Hm;
            const size_t row = (size_t)bh * nq + qb;
            int npart = 0, nfull = 0;
            for (int kb = 0; kb < nkv; ++kb) {
                int64_t count = 0, inrange = 0;
                for (int i = qb * block; i < (qb + 1) * block; ++i) {
                    for (int j = kb * block; j < (kb + 1) * block; ++j) {
                        if (i >= Tq || j >= Tkv) continue;
                        ++inrange;
                        count += or_mask_mod(mask, b, i, j);
                    }
                }
                const int complete = inrange == (int64_t)block * block;
                if (count == 0) continue;
                if (complete && count == inrange)
                    full_kv_indices[row * nkv + nfull++] = kb;
                else
                    kv_indices[row * nkv + npart++] = kb;
            }
            for (int t = npart; t < nkv; ++t) kv_indices[row * nkv + t] = -1;
            for (int t = nfull; t < nkv; ++t) full_kv_indices[row * nkv + t] = -1;
            kv_num_blocks[row] = npart;
            full_kv_num_blocks[row] = nfull;
        }
    }
    return 0;
}


/*
 * Gradients of the forward with respect to q, k and v for an upstream dO
 * (the backward pass the FlexAttention Guide's "Implementation" script takes
 * through autograd): for every query row (b, hq, i), with P_j the row's
 * softmax weights as in the forward,
 *     dP_j    = dO_i . v_j
 *     Delta_i = sum_j P_j dP_j
 *     dS_j    = P_j (dP_j - Delta_i) * d score_mod / d s (s_j)
 *     dq_i    = scale sum_j dS_j k_j
 *     dk_j   += scale dS_j q_i,   dv_j += P_j dO_i
 * (masked pairs have P_j = 0; a row that attends to nothing contributes
 * nothing).  dq: [B, Hq, Tq, D], dk, dv: [B, Hkv, Tkv, D], all written.
 * Each kv head (b, hk) is one task, so dk and dv need no reduction across
 * threads.  Returns 0, or -1 on bad arguments.
 */
int oracle_bwd(const float *q, const float *k, const float *v, const float *dout,
               int B, int Hq, int Hkv, int Tq, int Tkv, int D, double scale,
               const or_mask *mask, const or_score *score,
               double *dq, double *dk, double *dv, int nthreads)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Tq <= 0 || Tkv <= 0 || D <= 0)
        return -1;
    const int group = Hq / Hkv;
    int bad = 0;

#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1) reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Tkv);
        double *sraw = (double *)malloc(sizeof(double) * (size_t)Tkv);
        double *p = (double *)malloc(sizeof(double) * (size_t)Tkv);
        double *dp = (double *)malloc(sizeof(double) * (size_t)Tkv);
        if (!s || !sraw || !p || !dp) {
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int task = 0; task < B * Hkv; ++task) {
                const int b = task / Hkv, hk = task % Hkv;
                const float *kb = k + ((size_t)b * Hkv + hk) * (size_t)Tkv * D;
                const float *vb = v + ((size_t)b * Hkv + hk) * (size_t)Tkv * D;
                double *dkb = dk + ((size_t)b * Hkv + hk) * (size_t)Tkv * D;
                double *dvb = dv + ((size_t)b * Hkv + hk) * (size_t)Tkv * D;
                for (size_t x = 0; x < (size_t)Tkv * D; ++x) dkb[x] = dvb[x] = 0.0;
                for (int hq = hk * group; hq < (hk + 1) * group; ++hq) {
                    for (int i = 0; i < Tq; ++i) {
                        const size_t row = ((size_t)b * Hq + hq) * Tq + i;
                        const float *qi = q + row * D;
                        const float *gi = dout + row * D;
                        double *dqi = dq + row * D;
                        for (int d = 0; d < D; ++d) dqi[d] = 0.0;
                        /* the forward's row: scores, mask, softmax weights */
                        double M = -INFINITY;
                        for (int j = 0; j < Tkv; ++j) {
                            const float *kj = kb + (size_t)j * D;
                            double dot = 0.0;
                            for (int d = 0; d < D; ++d)
                                dot += (double)qi[d] * (double)kj[d];
                            sraw[j] = scale * dot;
                            double sj = or_score_mod(score, sraw[j], hq, i, j);
                            if (!or_mask_mod(mask, b, i, j))
                                sj = -INFINITY;
                            s[j] = sj;
                            if (sj > M) M = sj;
                        }
                        if (M == -INFINITY) continue;
                        double L = 0.0;
                        for (int j = 0; j < Tkv; ++j) {
                            p[j] = s[j] == -INFINITY ? 0.0 : exp(s[j] - M);
                            L += p[j];
                        }
                        double delta = 0.0;
                        for (int j = 0; j < Tkv; ++j) {
                            p[j] /= L;
                            const float *vj = vb + (size_t)j * D;
                            double t = 0.0;
                            for (int d = 0; d < D; ++d)
                                t += (double)gi[d] * (double)vj[d];
                            dp[j] = t;
                            delta += p[j] * t;
                        }
                        for (int j = 0; j < Tkv; ++j) {
                            if (p[j] == 0.0) continue;
                            const double ds = p[j] * (dp[j] - delta) * or_score_mod_ds(score, sraw[j], hq, i, j);
                            const float *kj = kb + (size_t)j * D;
                            double *dkj = dkb + (size_t)j * D;
                            double *dvj = dvb + (size_t)j * D;
                            for (int d = 0; d < D; ++d) {
                                dqi[d] += scale * ds * (double)kj[d];
                                dkj[d] += scale * ds * (double)qi[d];
                                dvj[d] += p[j] * (double)gi[d];
                            }
                        }
                    }
                }
            }
        }
        free(s);
        free(sraw);
        free(p);
        free(dp);
    }
    return bad ? -1 : 0;
}
