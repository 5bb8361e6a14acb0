/*
 * CPU oracle for the exact attention forward pass  O = softmax(Q K^T * scale) V.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the
 * bench's CPU-baseline leg call it; the CUDA product path never does, and
 * this file shares no code, header or constant with it.
 *
 * Plain, slow and meant to be checked by eye.  Everything is computed in
 * double precision from float32 inputs (which hold the exact bf16 or fp32
 * values the GPU sees).  For one query row it follows the three loops of
 * "Safe Softmax and the Three Passes" in "The Details of Flash Attention"
 * (ggluo.github.io), with the scores x_j of the section "The Attention
 * Computation":
 *
 *   x_j  = scale * sum_t Q[i,t] K[j,t]              for every key j in range
 *   pass 1: m   = max_j x_j
 *   pass 2: d_T = sum_j exp(x_j - m)
 *   pass 3: O[i,:] = sum_j exp(x_j - m) / d_T * V[j,:]
 *
 * and the per-row log-sum-exp  LSE_i = m + ln d_T, the natural log of
 * sum_j exp(x_j).  Keys in range are all N keys, or j <= i under the causal
 * mask (keys after the query are set to -inf before the softmax, as the
 * masked_fill in "PyTorch Implementation" of the rohit.vision post
 * "Transformer Attention: A Mathematical Deep Dive" does).  The scores of
 * one row are kept in a work buffer of N doubles between the passes; no
 * N x N matrix is ever formed.
 *
 * Layout: contiguous row-major float32, Q [B, H, Nq, dk], K [B, H, Nk, dk],
 * V [B, H, Nk, dv].  A "row id" is bh * Nq + i with bh = b * H + h.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* Returns 0 on success, 1 on a bad argument, 2 when a row has no key in
 * range (cannot happen for Nk >= 1: the causal row i always sees key 0).
 *
 * Q is [B, H, Nq, dk], K is [B, H, Nk, dk], V is [B, H, Nk, dv] (the shapes
 * (n, d_k), (m, d_k), (m, d_v) per head of "The Attention Formula" in
 * "Transformer Attention: A Mathematical Deep Dive"); a row id is
 * bh * Nq + i; O rows are dv wide.  Under the causal mask query i sees keys
 * j <= i. */
int oracle_attention_rows_qkv(const float *q, const float *k, const float *v,
                              int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                              int64_t dk, int64_t dv, double scale, int causal,
                              const int64_t *rows, int64_t nrows,
                              double *o, double *lse, double *work)
{
    if (!q || !k || !v || !rows || !o || !work) return 1;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || dk < 1 || dv < 1 || nrows < 0) return 1;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t id = rows[r];
        if (id < 0 || id >= B * H * Nq) return 1;
        int64_t bh = id / Nq;
        int64_t i = id % Nq;
        const float *qi = q + (bh * Nq + i) * dk;
        const float *kh = k + bh * Nk * dk;
        const float *vh = v + bh * Nk * dv;
        int64_t nkeys = causal ? (i + 1 < Nk ? i + 1 : Nk) : Nk;
        if (nkeys < 1) return 2;

        /* scores x_j */
        for (int64_t j = 0; j < nkeys; ++j) {
            double dot = 0.0;
            for (int64_t t = 0; t < dk; ++t)
                dot += (double)qi[t] * (double)kh[j * dk + t];
            work[j] = scale * dot;
        }
        /* pass 1: the row maximum m */
        double m = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j)
            if (work[j] > m) m = work[j];
        /* pass 2: the denominator d_T */
        double dT = 0.0;
        for (int64_t j = 0; j < nkeys; ++j)
            dT += exp(work[j] - m);
        /* pass 3: the weighted sum of the value rows */
        double *oi = o + r * dv;
        for (int64_t t = 0; t < dv; ++t) oi[t] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            double w = exp(work[j] - m) / dT;
            for (int64_t t = 0; t < dv; ++t)
                oi[t] += w * (double)vh[j * dv + t];
        }
        if (lse) lse[r] = m + log(dT);
    }
    return 0;
}

/* The self-attention case: Nq = Nk = N, dk = dv = d. */
int oracle_attention_rows(const float *q, const float *k, const float *v,
                          int64_t B, int64_t H, int64_t N, int64_t d,
                          double scale, int causal,
                          const int64_t *rows, int64_t nrows,
                          double *o, double *lse, double *work)
{
    return oracle_attention_rows_qkv(q, k, v, B, H, N, N, d, d, scale, causal,
                                     rows, nrows, o, lse, work);
}

/*
 * Gradients of the forward pass for one head (bh), fp64, from the plain
 * definition: with L = sum_i dO_i . O_i, P the softmax weights above and
 * S_ij = scale * q_i . k_j (masked entries have P_ij = 0),
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij (dP_ij - delta_i),   delta_i = sum_j P_ij dP_ij
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 *
 * This is what "FlashAttention" (ai360xpert.com, "Recomputation in the
 * backward pass") recomputes tile by tile from the stored row statistics.
 * Layout: Q, K, V, dO contiguous [B, H, N, d]; dq, dk, dv receive this
 * head's [N, d] blocks; work holds N * N doubles (P).  Returns 0 on success.
 */
int oracle_attention_backward_head(const float *q, const float *k, const float *v, const float *dout,
                                   int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                                   int64_t bh, double *dq, double *dk, double *dv, double *work)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !work) return 1;
    if (B < 1 || H < 1 || N < 1 || d < 1 || bh < 0 || bh >= B * H) return 1;
    const float *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d, *gh = dout + bh * N * d;
    double *P = work;
    /* the softmax weights, row by row, by the three passes */
    for (int64_t i = 0; i < N; ++i) {
        int64_t nkeys = causal ? i + 1 : N;
        double *pr = P + i * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            if (j >= nkeys) { pr[j] = 0.0; continue; }
            double dot = 0.0;
            for (int64_t t = 0; t < d; ++t) dot += (double)qh[i * d + t] * (double)kh[j * d + t];
            pr[j] = scale * dot;
            if (pr[j] > m) m = pr[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) den += exp(pr[j] - m);
        for (int64_t j = 0; j < nkeys; ++j) pr[j] = exp(pr[j] - m) / den;
    }
    for (int64_t x = 0; x < N * d; ++x) { dq[x] = 0.0; dk[x] = 0.0; dv[x] = 0.0; }
    for (int64_t i = 0; i < N; ++i) {
        const double *pr = P + i * N;
        /* delta_i = sum_j P_ij (dO_i . v_j) */
        double delta = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (pr[j] == 0.0) continue;
            double dp = 0.0;
            for (int64_t t = 0; t < d; ++t) dp += (double)gh[i * d + t] * (double)vh[j * d + t];
            delta += pr[j] * dp;
        }
        for (int64_t j = 0; j < N; ++j) {
            if (pr[j] == 0.0) continue;
            double dp = 0.0;
            for (int64_t t = 0; t < d; ++t) dp += (double)gh[i * d + t] * (double)vh[j * d + t];
            const double ds = pr[j] * (dp - delta);
            for (int64_t t = 0; t < d; ++t) {
                dv[j * d + t] += pr[j] * (double)gh[i * d + t];
                dq[i * d + t] += scale * ds * (double)kh[j * d + t];
                dk[j * d + t] += scale * ds * (double)qh[i * d + t];
            }
        }
    }
    return 0;
}
