/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A slow, plain, double-precision CPU statement of exact softmax attention,
 * used to check the GPU library.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the GPU path never links or calls
 * it, and it includes no header, helper or constant from the GPU path.
 *
 * What it computes (per batch b, head h; query row i in [0,Sq), key row j in
 * [0,Sk); q,k,v already rounded to the 16-bit input type and widened to
 * double):
 *
 *   S_ij  = scale * sum_c q_ic k_jc          where key j is visible to row i
 *         = -inf                             otherwise
 *   m_i   = max_j S_ij
 *   P_ij  = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)
 *   O_i   = sum_j P_ij v_j
 *   lse_i = m_i + ln sum_j exp(S_ij - m_i)   (natural log of the scaled
 *                                             row's sum of exponentials)
 *
 * Sources: the attention definition softmax(Q K^T / sqrt(d)) V and the naive
 * three-pass evaluation that writes S, then P, then O ("FlashAttention: Why
 * Tiling Attention Makes Transformers Fast...", section "The problem is
 * memory, not arithmetic"; "Flash attention and memory-efficient attention
 * variants", section "Two kinds of memory live on every GPU"); the safe
 * softmax with the row maximum subtracted ("FlashAttention: Why Tiling...",
 * section "Why softmax seems to block tiling"); the per-row logsumexp output
 * ("FlashAttention: IO-aware attention kernels", table "What goes in, what
 * comes out").
 *
 * Visibility (readings where the pages are silent):
 *   mask_kind 0  none:     every key j < Sk.
 *   mask_kind 1  causal:   j <= i (top-left aligned, as torch's is_causal).
 *   mask_kind 2  window W: i - W < j <= i (W keys including the diagonal).
 * A row that sees no key (possible only with a window when Sq > Sk) gets
 * O_i = 0 and lse_i = -inf: the pages ask that a fully masked row be guarded
 * instead of producing NaN ("FlashAttention: IO-aware attention kernels",
 * "Failure modes").
 *
 * oracle_attn_naive materialises the rows of S and P it works on, one block of
 * query rows at a time (never the whole S x S matrix: 18000^2 doubles would be
 * 2.6 GB), which is the "write S, read S / write P, read P" evaluation.
 * oracle_attn_blocked is the second, independent form: the tiled online
 * softmax with a running max m, running sum l and unnormalised accumulator,
 * rescaled by exp(m_old - m_new) and divided by l once at the end, taken in
 * the order the pages give ("FlashAttention: Why Tiling...", sections "The
 * tiled forward pass" and "Online softmax: correct as you go"; "Flash
 * attention and memory-efficient attention variants", section "Tiling and the
 * running (online) softmax").  oracle_online_trace records the running
 * statistics after every key block for one query row, so the hand-traced
 * worked example ("Flash attention and memory-efficient attention variants",
 * section "Worked example: tracing the running statistics by hand") can be
 * checked step by step.
 *
 * Grouped-query attention (a variant the first page names: "FlashAttention:
 * Why Tiling...", section "Using it in practice"): K and V carry Hkv heads,
 * Hkv dividing H, and query head h reads K/V head h / (H / Hkv), i.e. each run
 * of H/Hkv consecutive query heads shares one K/V head (the reading of the
 * page, which names the variant without defining it; it is the grouping
 * PyTorch's enable_gqa uses).  Hkv == H is ordinary multi-head attention,
 * Hkv == 1 multi-query attention.
 *
 * All arrays are C-contiguous (q: [B, H, Sq, d]; k and v: [B, Hkv, Sk, d]),
 * o is [rows, d], lse is [rows].  Functions return 0 on success, -1 on bad
 * arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MASK_NONE 0
#define ORC_MASK_CAUSAL 1
#define ORC_MASK_WINDOW 2

/* Rows of S and P held at once by one worker in the naive form. */
#define ORC_ROW_BLOCK 64

static int orc_visible(int mask_kind, int window, int64_t i, int64_t j)
{
    if (mask_kind == ORC_MASK_NONE)
        return 1;
    if (j > i)
        return 0;
    if (mask_kind == ORC_MASK_WINDOW && j <= i - (int64_t)window)
        return 0;
    return 1;
}

static int orc_check(int B, int H, int Hkv, int Sq, int Sk, int d, int mask_kind, int window)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sq < 0 || Sk < 1 || d < 1)
        return -1;
    if (mask_kind < 0 || mask_kind > 2)
        return -1;
    if (mask_kind == ORC_MASK_WINDOW && window < 1)
        return -1;
    return 0;
}

/* Offset of the K/V head that query head (b, h) reads, in elements. */
static int64_t orc_kv_offset(int64_t bh, int H, int Hkv, int Sk, int d)
{
    const int64_t b = bh / H, h = bh % H;
    const int64_t kvh = h / (H / Hkv);
    return (b * Hkv + kvh) * (int64_t)Sk * d;
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Naive attention for a list of query rows.  rows[r] is a flat row index
 * (b*H + h)*Sq + i; rows == NULL means every row in order.  Each worker takes
 * up to ORC_ROW_BLOCK consecutive list entries, writes their score rows S,
 * turns them into probability rows P in place, then forms O = P V.
 */
int oracle_attn_naive(const double *q, const double *k, const double *v,
                      int B, int H, int Hkv, int Sq, int Sk, int d, double scale,
                      int mask_kind, int window,
                      const int64_t *rows, int64_t nrows,
                      double *o, double *lse)
{
    if (orc_check(B, H, Hkv, Sq, Sk, d, mask_kind, window) != 0)
        return -1;
    const int64_t total_rows = (int64_t)B * H * Sq;
    if (rows == NULL)
        nrows = total_rows;
    if (nrows < 0)
        return -1;
    if (rows != NULL) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total_rows)
                return -1;
    }
    const int64_t nblocks = (nrows + ORC_ROW_BLOCK - 1) / ORC_ROW_BLOCK;
    int failed = 0;

#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)ORC_ROW_BLOCK * (size_t)Sk);
        double *mrow = (double *)malloc(sizeof(double) * ORC_ROW_BLOCK);
        double *lrow = (double *)malloc(sizeof(double) * ORC_ROW_BLOCK);
        if (S == NULL || mrow == NULL || lrow == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t blk = 0; blk < nblocks; ++blk) {
            if (S == NULL || mrow == NULL || lrow == NULL)
                continue;
            const int64_t r0 = blk * ORC_ROW_BLOCK;
            const int64_t r1 = (r0 + ORC_ROW_BLOCK < nrows) ? r0 + ORC_ROW_BLOCK : nrows;
            /* Pass 1: score rows S_ij = scale * q_i . k_j (or -inf). */
            for (int64_t r = r0; r < r1; ++r) {
                const int64_t flat = rows ? rows[r] : r;
                const int64_t bh = flat / Sq, i = flat % Sq;
                const double *qi = q + flat * (int64_t)d;
                const double *kh = k + orc_kv_offset(bh, H, Hkv, Sk, d);
                double *Si = S + (r - r0) * (int64_t)Sk;
                for (int64_t j = 0; j < Sk; ++j) {
                    if (!orc_visible(mask_kind, window, i, j)) {
                        Si[j] = -INFINITY;
                        continue;
                    }
                    const double *kj = kh + j * (int64_t)d;
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c)
                        dot += qi[c] * kj[c];
                    Si[j] = scale * dot;
                }
            }
            /* Pass 2: row softmax with the row maximum subtracted; P replaces S. */
            for (int64_t r = r0; r < r1; ++r) {
                double *Si = S + (r - r0) * (int64_t)Sk;
                double m = -INFINITY;
                for (int64_t j = 0; j < Sk; ++j)
                    if (Si[j] > m)
                        m = Si[j];
                mrow[r - r0] = m;
                if (m == -INFINITY) { /* no visible key: guarded row */
                    for (int64_t j = 0; j < Sk; ++j)
                        Si[j] = 0.0;
                    lrow[r - r0] = 0.0;
                    continue;
                }
                double l = 0.0;
                for (int64_t j = 0; j < Sk; ++j) {
                    const double e = (Si[j] == -INFINITY) ? 0.0 : exp(Si[j] - m);
                    Si[j] = e;
                    l += e;
                }
                for (int64_t j = 0; j < Sk; ++j)
                    Si[j] /= l;
                lrow[r - r0] = l;
            }
            /* Pass 3: O_i = sum_j P_ij v_j, and the row logsumexp. */
            for (int64_t r = r0; r < r1; ++r) {
                const int64_t flat = rows ? rows[r] : r;
                const int64_t bh = flat / Sq;
                const double *vh = v + orc_kv_offset(bh, H, Hkv, Sk, d);
                const double *Pi = S + (r - r0) * (int64_t)Sk;
                double *oi = o + r * (int64_t)d;
                for (int c = 0; c < d; ++c)
                    oi[c] = 0.0;
                for (int64_t j = 0; j < Sk; ++j) {
                    const double p = Pi[j];
                    if (p == 0.0)
                        continue;
                    const double *vj = vh + j * (int64_t)d;
                    for (int c = 0; c < d; ++c)
                        oi[c] += p * vj[c];
                }
                lse[r] = (lrow[r - r0] > 0.0) ? mrow[r - r0] + log(lrow[r - r0]) : -INFINITY;
            }
        }
        free(S);
        free(mrow);
        free(lrow);
    }
    return failed ? -1 : 0;
}

/*
 * Online-softmax evaluation of one query row over key blocks of block_size.
 * trace_m / trace_l / trace_o (may be NULL) receive, after each key block, the
 * running max, running sum and unnormalised accumulator.  Returns the number
 * of key blocks.
 */
static int64_t orc_online_row(const double *qi, const double *kh, const double *vh,
                              int Sk, int d, double scale, int mask_kind, int window,
                              int64_t i, int block_size, double *sblk, double *acc,
                              double *out_o, double *out_lse,
                              double *trace_m, double *trace_l, double *trace_o)
{
    double m = -INFINITY; /* running row maximum */
    double l = 0.0;       /* running sum of exponentials against m */
    for (int c = 0; c < d; ++c)
        acc[c] = 0.0;     /* running unnormalised output against m */
    int64_t nblk = 0;
    for (int64_t start = 0; start < Sk; start += block_size, ++nblk) {
        const int64_t end = (start + block_size < Sk) ? start + block_size : Sk;
        /* This block's scores and its maximum. */
        double bmax = -INFINITY;
        for (int64_t j = start; j < end; ++j) {
            double s = -INFINITY;
            if (orc_visible(mask_kind, window, i, j)) {
                const double *kj = kh + j * (int64_t)d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += qi[c] * kj[c];
                s = scale * dot;
            }
            sblk[j - start] = s;
            if (s > bmax)
                bmax = s;
        }
        const double m_new = (bmax > m) ? bmax : m;
        if (m_new != -INFINITY) {
            /* Correction for what was accumulated against the old maximum;
             * nothing was accumulated while m was still -inf. */
            const double corr = (m == -INFINITY) ? 0.0 : exp(m - m_new);
            double psum = 0.0;
            for (int c = 0; c < d; ++c)
                acc[c] *= corr;
            for (int64_t j = start; j < end; ++j) {
                const double p = (sblk[j - start] == -INFINITY) ? 0.0 : exp(sblk[j - start] - m_new);
                psum += p;
                if (p != 0.0) {
                    const double *vj = vh + j * (int64_t)d;
                    for (int c = 0; c < d; ++c)
                        acc[c] += p * vj[c];
                }
            }
            l = corr * l + psum;
            m = m_new;
        }
        if (trace_m)
            trace_m[nblk] = m;
        if (trace_l)
            trace_l[nblk] = l;
        if (trace_o)
            for (int c = 0; c < d; ++c)
                trace_o[nblk * (int64_t)d + c] = acc[c];
    }
    /* Divide by the final sum once; a row that saw no key stays at zero. */
    if (l > 0.0) {
        for (int c = 0; c < d; ++c)
            out_o[c] = acc[c] / l;
        *out_lse = m + log(l);
    } else {
        for (int c = 0; c < d; ++c)
            out_o[c] = 0.0;
        *out_lse = -INFINITY;
    }
    return nblk;
}

int oracle_attn_blocked(const double *q, const double *k, const double *v,
                        int B, int H, int Hkv, int Sq, int Sk, int d, double scale,
                        int mask_kind, int window, int block_size,
                        double *o, double *lse)
{
    if (orc_check(B, H, Hkv, Sq, Sk, d, mask_kind, window) != 0 || block_size < 1)
        return -1;
    const int64_t total_rows = (int64_t)B * H * Sq;
    int failed = 0;
#pragma omp parallel
    {
        double *sblk = (double *)malloc(sizeof(double) * (size_t)block_size);
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        if (sblk == NULL || acc == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t flat = 0; flat < total_rows; ++flat) {
            if (sblk == NULL || acc == NULL)
                continue;
            const int64_t bh = flat / Sq, i = flat % Sq;
            orc_online_row(q + flat * (int64_t)d, k + orc_kv_offset(bh, H, Hkv, Sk, d),
                           v + orc_kv_offset(bh, H, Hkv, Sk, d), Sk, d, scale, mask_kind, window, i,
                           block_size, sblk, acc, o + flat * (int64_t)d, lse + flat,
                           NULL, NULL, NULL);
        }
        free(sblk);
        free(acc);
    }
    return failed ? -1 : 0;
}

/*
 * One query row qi against one head's K, V (Sk x d), unmasked, with the
 * running statistics recorded after each of the ceil(Sk/block_size) blocks.
 */
int oracle_online_trace(const double *qi, const double *kh, const double *vh,
                        int Sk, int d, double scale, int block_size,
                        double *trace_m, double *trace_l, double *trace_o,
                        double *o, double *lse)
{
    if (Sk < 1 || d < 1 || block_size < 1)
        return -1;
    double *sblk = (double *)malloc(sizeof(double) * (size_t)block_size);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    if (sblk == NULL || acc == NULL) {
        free(sblk);
        free(acc);
        return -1;
    }
    orc_online_row(qi, kh, vh, Sk, d, scale, ORC_MASK_NONE, 0, 0, block_size, sblk, acc,
                   o, lse, trace_m, trace_l, trace_o);
    free(sblk);
    free(acc);
    return 0;
}

/*
 * The normalised probability matrix P (Sq x Sk) of one head, as the naive
 * evaluation forms it.  Rows with no visible key are all zero.
 */
int oracle_probs(const double *qh, const double *kh, int Sq, int Sk, int d, double scale,
                 int mask_kind, int window, double *P)
{
    if (orc_check(1, 1, 1, Sq, Sk, d, mask_kind, window) != 0)
        return -1;
    for (int64_t i = 0; i < Sq; ++i) {
        double *Pi = P + i * (int64_t)Sk;
        double m = -INFINITY;
        for (int64_t j = 0; j < Sk; ++j) {
            double s = -INFINITY;
            if (orc_visible(mask_kind, window, i, j)) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += qh[i * (int64_t)d + c] * kh[j * (int64_t)d + c];
                s = scale * dot;
            }
            Pi[j] = s;
            if (s > m)
                m = s;
        }
        if (m == -INFINITY) {
            for (int64_t j = 0; j < Sk; ++j)
                Pi[j] = 0.0;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < Sk; ++j) {
            Pi[j] = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m);
            l += Pi[j];
        }
        for (int64_t j = 0; j < Sk; ++j)
            Pi[j] /= l;
    }
    return 0;
}

/*
 * Gradients of the attention output, by the chain the first page gives for the
 * backward pass ("FlashAttention: Why Tiling...", section "The backward pass:
 * recompute instead of storing"), written out for whole rows instead of tiles:
 * with dO the gradient of the loss with respect to O,
 *
 *   P_ij  = softmax row i of the scaled, masked scores (as in the forward)
 *   dV_j  = sum_i P_ij dO_i                      (dV = P^T dO)
 *   dP_ij = dO_i . v_j                           (dP = dO V^T)
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (softmax Jacobian on row i)
 *   dQ_i  = scale * sum_j dS_ij k_j              (S = scale Q K^T)
 *   dK_j  = scale * sum_i dS_ij q_i
 *
 * Hidden pairs have P_ij = 0 and so dS_ij = 0; a row with no visible key
 * contributes nothing.  With grouped K/V heads, dK and dV of a K/V head sum
 * over the query heads that read it.  q, dout, dq: [B, H, Sq, d]; k, v, dk,
 * dv: [B, Hkv, Sk, d].
 *
 * Two passes so that both can run in parallel without shared accumulators:
 * the first goes over query rows (P_i, dP_i, the Jacobian's row term, dQ_i,
 * and the row's max and sum of exponentials); the second goes over key rows
 * and forms each P_ij again from that row's max and sum, then dS_ij, and
 * accumulates dK_j and dV_j.
 */
static double orc_dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c)
        s += a[c] * b[c];
    return s;
}

int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int B, int H, int Hkv, int Sq, int Sk, int d, double scale,
                    int mask_kind, int window, double *dq, double *dk, double *dv)
{
    if (orc_check(B, H, Hkv, Sq, Sk, d, mask_kind, window) != 0)
        return -1;
    const int group = H / Hkv;
    const int64_t n_rows = (int64_t)B * H * Sq;
    /* per query row: max m_i, sum of exponentials l_i, row term sum_k P_ik dP_ik */
    double *rm = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    double *rl = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    double *rt = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    if (rm == NULL || rl == NULL || rt == NULL) {
        free(rm);
        free(rl);
        free(rt);
        return -1;
    }
    int failed = 0;

    /* Pass 1: query rows. */
#pragma omp parallel
    {
        double *P = (double *)malloc(sizeof(double) * (size_t)Sk);
        double *dP = (double *)malloc(sizeof(double) * (size_t)Sk);
        if (P == NULL || dP == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (P == NULL || dP == NULL)
                continue;
            const int64_t bh = r / Sq, i = r % Sq;
            const double *kh = k + orc_kv_offset(bh, H, Hkv, Sk, d);
            const double *vh = v + orc_kv_offset(bh, H, Hkv, Sk, d);
            const double *qi = q + r * (int64_t)d;
            const double *doi = dout + r * (int64_t)d;
            double *dqi = dq + r * (int64_t)d;
            for (int c = 0; c < d; ++c)
                dqi[c] = 0.0;
            double m = -INFINITY;
            for (int64_t j = 0; j < Sk; ++j) {
                P[j] = orc_visible(mask_kind, window, i, j)
                           ? scale * orc_dot(qi, kh + j * (int64_t)d, d) : -INFINITY;
                if (P[j] > m)
                    m = P[j];
            }
            rm[r] = m;
            rl[r] = 0.0;
            rt[r] = 0.0;
            if (m == -INFINITY)
                continue; /* no visible key: no gradient flows through row i */
            double l = 0.0;
            for (int64_t j = 0; j < Sk; ++j) {
                P[j] = (P[j] == -INFINITY) ? 0.0 : exp(P[j] - m);
                l += P[j];
            }
            for (int64_t j = 0; j < Sk; ++j)
                P[j] /= l;
            double rowdot = 0.0;
            for (int64_t j = 0; j < Sk; ++j) {
                dP[j] = orc_dot(doi, vh + j * (int64_t)d, d);
                rowdot += P[j] * dP[j];
            }
            for (int64_t j = 0; j < Sk; ++j) {
                if (P[j] == 0.0)
                    continue;
                const double ds = P[j] * (dP[j] - rowdot);
                const double *kj = kh + j * (int64_t)d;
                for (int c = 0; c < d; ++c)
                    dqi[c] += scale * ds * kj[c];
            }
            rl[r] = l;
            rt[r] = rowdot;
        }
        free(P);
        free(dP);
    }

    /* Pass 2: key rows of every K/V head, over the query heads that read it. */
    const int64_t n_keys = (int64_t)B * Hkv * Sk;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t kr = 0; kr < n_keys; ++kr) {
        const int64_t bk = kr / Sk, j = kr % Sk;
        const int64_t b = bk / Hkv, kvh = bk % Hkv;
        const double *kj = k + kr * (int64_t)d;
        const double *vj = v + kr * (int64_t)d;
        double *dkj = dk + kr * (int64_t)d;
        double *dvj = dv + kr * (int64_t)d;
        for (int c = 0; c < d; ++c) {
            dkj[c] = 0.0;
            dvj[c] = 0.0;
        }
        for (int64_t h = kvh * group; h < (kvh + 1) * group; ++h) {
            for (int64_t i = 0; i < Sq; ++i) {
                const int64_t r = (b * H + h) * Sq + i;
                if (rl[r] == 0.0 || !orc_visible(mask_kind, window, i, j))
                    continue;
                const double *qi = q + r * (int64_t)d;
                const double *doi = dout + r * (int64_t)d;
                const double Pij = exp(scale * orc_dot(qi, kj, d) - rm[r]) / rl[r];
                const double ds = Pij * (orc_dot(doi, vj, d) - rt[r]);
                for (int c = 0; c < d; ++c) {
                    dkj[c] += scale * ds * qi[c];
                    dvj[c] += Pij * doi[c];
                }
            }
        }
    }
    free(rm);
    free(rl);
    free(rt);
    return failed ? -1 : 0;
}

/*
 * Attention of new query rows over a paged key/value cache
 * ("Flash attention and memory-efficient attention variants", sections
 * "A different bottleneck: the KV cache during inference" and "PagedAttention:
 * memory management borrowed from an operating system"): the cache is split
 * into fixed-size physical blocks of block_size tokens, and each request's
 * block table maps its logical block n (tokens n*block_size ..) to a physical
 * block anywhere in the pool; the attention walks the table and gathers.
 *
 * Request b holds seq_lens[b] cached tokens, the last Sq of which belong to
 * its Sq new query rows (Sq = 1 is one decoding step).  Query row i sits at
 * position seq_lens[b] - Sq + i.  Visibility (the reading for decoding, where
 * the newest token is the last position):
 *   mask_kind 0  none:    every cached token j < seq_lens[b];
 *   mask_kind 1  causal:  tokens j <= seq_lens[b] - Sq + i.
 *
 * q: [B, H, Sq, d]; k_cache, v_cache: [num_blocks, Hkv, block_size, d];
 * block_table: [B, max_blocks] (entries past the request's last block are not
 * read); seq_lens: [B], each in [Sq, max_blocks * block_size]; o: [B, H, Sq,
 * d]; lse: [B, H, Sq].  Query head h reads K/V head h / (H / Hkv).
 */
int oracle_attn_paged(const double *q, const double *k_cache, const double *v_cache,
                      const int32_t *block_table, const int32_t *seq_lens, int B, int H, int Hkv,
                      int Sq, int d, int block_size, int max_blocks, int num_blocks,
                      double scale, int mask_kind, double *o, double *lse)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sq < 1 || d < 1 || block_size < 1 ||
        max_blocks < 1 || num_blocks < 1 || (mask_kind != ORC_MASK_NONE && mask_kind != ORC_MASK_CAUSAL))
        return -1;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        if (L < Sq || L > max_blocks * block_size)
            return -1;
        for (int n = 0; n < (L + block_size - 1) / block_size; ++n)
            if (block_table[(int64_t)b * max_blocks + n] < 0 ||
                block_table[(int64_t)b * max_blocks + n] >= num_blocks)
                return -1;
    }
    const int group = H / Hkv;
    const int64_t n_rows = (int64_t)B * H * Sq;
    int failed = 0;
#pragma omp parallel
    {
        int max_len = 0;
        for (int b = 0; b < B; ++b)
            if (seq_lens[b] > max_len)
                max_len = seq_lens[b];
        double *S = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (S == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (S == NULL)
                continue;
            const int64_t b = r / ((int64_t)H * Sq), h = (r / Sq) % H, i = r % Sq;
            const int64_t kvh = h / group;
            const int L = seq_lens[b];
            const int64_t last = (mask_kind == ORC_MASK_CAUSAL) ? L - Sq + i : L - 1;
            const double *qi = q + r * (int64_t)d;
            double m = -INFINITY;
            for (int64_t j = 0; j <= last; ++j) {
                const int64_t blk = block_table[b * max_blocks + j / block_size];
                const double *kj = k_cache + ((blk * Hkv + kvh) * block_size + j % block_size) * (int64_t)d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += qi[c] * kj[c];
                S[j] = scale * dot;
                if (S[j] > m)
                    m = S[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j <= last; ++j) {
                S[j] = exp(S[j] - m);
                l += S[j];
            }
            double *oi = o + r * (int64_t)d;
            for (int c = 0; c < d; ++c)
                oi[c] = 0.0;
            for (int64_t j = 0; j <= last; ++j) {
                const int64_t blk = block_table[b * max_blocks + j / block_size];
                const double *vj = v_cache + ((blk * Hkv + kvh) * block_size + j % block_size) * (int64_t)d;
                for (int c = 0; c < d; ++c)
                    oi[c] += (S[j] / l) * vj[c];
            }
            lse[r] = m + log(l);
        }
        free(S);
    }
    return failed ? -1 : 0;
}
