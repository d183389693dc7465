/*
 * fp64 CPU oracle for the exact scaled-dot-product attention forward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path never does.
 * It shares no source, header or helper with the CUDA path.
 *
 * What it computes is the plain definition of the method, written out once per
 * query row (no tiling, no online rescaling, no reordering):
 *
 *   visible set   V_i = { j : 0 <= j < N  and, under the causal mask, j <= i }
 *   scores        s_j = scale * sum_t q[i,t] * k[j,t]            (j in V_i)
 *   stable soft-  m   = max_j s_j,  e_j = exp(s_j - m),  l = sum_j e_j
 *   max
 *   output        O[i,:] = sum_j e_j * v[j,:] / l
 *   logsumexp     LSE[i] = m + ln(l)          (natural log of the scaled scores)
 *
 * Passages followed:
 *  - "Programming an attention kernel in Triton", Kernel 3 (fused softmax):
 *    subtract the row max, exponentiate, sum, divide.
 *  - same page, Kernel 4 (a self-attention kernel): scores = scale * Q K^T over
 *    the keys inside the sequence, softmax along the key axis, weights times V.
 *  - "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel" (profile-driven
 *    FlashAttention-2 page), Round 4 / Causal tile-skipping: a key is kept iff
 *    k_pos < N_KEYS and, when causal, k_pos <= q_pos (top-left aligned).
 *  - same page, Round 4 / exp2: L is reported in natural-log units and must
 *    equal torch.logsumexp of the scaled scores.
 *
 * Inputs are fp64 arrays, row-major [B*H][N][d]; callers upcast the 16-bit
 * tensors exactly before the call. Every row has at least one visible key
 * (key 0, and key i itself under the causal mask), so m and l are finite.
 *
 * oracle_attn_fwd_qk generalises to Nq query rows against Nk keys (the query
 * rows of "Programming an attention kernel in Triton", Kernel 4, may be fewer
 * or more than the keys). Under the causal mask the query rows are taken to be
 * the LAST Nq positions of the Nk-long sequence (a KV-cache decode step, the
 * extension named at the end of "Getting the kernel correct, then benchmarking
 * it honestly"): row i sees keys j <= i + Nk - Nq. With Nq = Nk this is the
 * top-left mask above. causal = 2 keeps the top-left alignment for any Nq, Nk
 * (row i sees keys j <= i, the k_pos <= q_pos test of the profile-driven
 * FlashAttention-2 page, "Round 4 / Causal tile-skipping", whose kernel takes
 * N_QUERIES and N_KEYS separately). A row that sees no key (only when causal and
 * Nq > Nk, bottom-right) gets O = 0 and LSE = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row i of one head. K and V point at that head's [N][d] block.
 * s is scratch of at least N doubles. */
static void oracle_row(const double* qi, const double* K, const double* V,
                       int64_t N, int64_t d, int64_t i, int causal, double scale,
                       double* s, double* oi, double* lse_i)
{
    const int64_t n_vis = causal ? (i + 1 < N ? i + 1 : N) : N;
    double m = -INFINITY;
    for (int64_t j = 0; j < n_vis; ++j) {
        const double* kj = K + j * d;
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += qi[t] * kj[t];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        const double e = s[j];
        const double* vj = V + j * d;
        for (int64_t t = 0; t < d; ++t) oi[t] += e * vj[t];
    }
    for (int64_t t = 0; t < d; ++t) oi[t] /= l;
    *lse_i = m + log(l);
}

static int bad_args(const void* q, const void* k, const void* v, const void* o,
                    const void* lse, int64_t BH, int64_t N, int64_t d, double scale)
{
    if (!q || !k || !v || !o || !lse) return 1;
    if (BH < 1 || N < 1 || d < 1) return 1;
    if (!(scale > 0.0) || !isfinite(scale)) return 1;
    return 0;
}

/* Full forward: o[BH][N][d], lse[BH][N]. Returns 0, or -1 on bad arguments,
 * or -2 when scratch memory cannot be had. */
int oracle_attn_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse, int64_t B, int64_t H, int64_t N,
                    int64_t d, int causal, double scale)
{
    const int64_t BH = B * H;
    if (B < 1 || H < 1 || bad_args(q, k, v, o, lse, BH, N, d, scale)) return -1;
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* s = (double*)malloc((size_t)N * sizeof(double));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16) collapse(2)
            for (int64_t bh = 0; bh < BH; ++bh) {
                for (int64_t i = 0; i < N; ++i) {
                    const double* base_q = q + (bh * N + i) * d;
                    oracle_row(base_q, k + bh * N * d, v + bh * N * d, N, d, i, causal, scale,
                               s, o + (bh * N + i) * d, lse + bh * N + i);
                }
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* Selected rows only: rows[r] is the flat index bh*N + i. Outputs are packed:
 * o[r][d], lse[r]. Used to check sampled outputs of workloads too large to
 * recompute whole. */
int oracle_attn_rows(const double* q, const double* k, const double* v,
                     int64_t BH, int64_t N, int64_t d, int causal, double scale,
                     const int64_t* rows, int64_t nrows, double* o, double* lse)
{
    if (!rows || nrows < 0 || bad_args(q, k, v, o, lse, BH, N, d, scale)) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= BH * N) return -1;
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* s = (double*)malloc((size_t)N * sizeof(double));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t bh = rows[r] / N, i = rows[r] % N;
                oracle_row(q + rows[r] * d, k + bh * N * d, v + bh * N * d, N, d, i, causal,
                           scale, s, o + r * d, lse + r);
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* Query row i of one head against keys [0, n_vis) (n_vis may be 0). */
static void oracle_row_n(const double* qi, const double* K, const double* V, int64_t d,
                         int64_t n_vis, double scale, double* s, double* oi, double* lse_i)
{
    if (n_vis <= 0) {
        for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
        *lse_i = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n_vis; ++j) {
        const double* kj = K + j * d;
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += qi[t] * kj[t];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
    for (int64_t j = 0; j < n_vis; ++j) {
        const double e = s[j];
        const double* vj = V + j * d;
        for (int64_t t = 0; t < d; ++t) oi[t] += e * vj[t];
    }
    for (int64_t t = 0; t < d; ++t) oi[t] /= l;
    *lse_i = m + log(l);
}

/* Nq query rows against Nk keys: q, o [BH][Nq][d]; k, v [BH][Nk][d]; lse [BH][Nq].
 * causal = 0: every key; 1: row i sees keys j <= i + Nk - Nq; 2: keys j <= i. */
int oracle_attn_fwd_qk(const double* q, const double* k, const double* v, double* o,
                       double* lse, int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int causal,
                       double scale)
{
    if (!q || !k || !v || !o || !lse || BH < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    if (!(scale > 0.0) || !isfinite(scale)) return -1;
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* s = (double*)malloc((size_t)Nk * sizeof(double));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4) collapse(2)
            for (int64_t bh = 0; bh < BH; ++bh) {
                for (int64_t i = 0; i < Nq; ++i) {
                    int64_t n_vis = Nk;
                    if (causal) {
                        /* last visible key: bottom-right (1) or top-left (2) alignment */
                        const int64_t last = causal == 2 ? i : i + Nk - Nq;
                        n_vis = last < 0 ? 0 : (last + 1 < Nk ? last + 1 : Nk);
                    }
                    oracle_row_n(q + (bh * Nq + i) * d, k + bh * Nk * d, v + bh * Nk * d, d, n_vis,
                                 scale, s, o + (bh * Nq + i) * d, lse + bh * Nq + i);
                }
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* Sliding windows and key padding, for Nq query rows against Nk keys. The
 * profile-driven FlashAttention-2 page ("Future articles") names padding masks and
 * sliding windows as the kernels in which a row can be fully masked; it defines
 * neither, so the plainest readings are taken:
 *  - key padding: batch element b has kv_lens[b] valid keys (0 <= kv_lens[b] <= Nk;
 *    NULL = all Nk), the right-padded layout of a batch of different lengths;
 *  - the diagonal of row i is key i + off_b, with off_b = 0 (top-left, align = 0)
 *    or off_b = n_b - Nq (bottom-right, align = 1: the query rows are the last Nq
 *    positions of each sequence), n_b the valid key count of its batch element;
 *  - a sliding window keeps keys i + off_b - left <= j <= i + off_b + right
 *    (left or right < 0: unbounded on that side; right = 0 is the causal mask).
 * Row i of batch element b sees keys j with 0 <= j < n_b inside the window. A row
 * that sees none gets O = 0 and LSE = -inf. */
int oracle_attn_fwd_window(const double* q, const double* k, const double* v, double* o,
                           double* lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                           int64_t left, int64_t right, const int64_t* kv_lens, int align,
                           double scale)
{
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    if (!(scale > 0.0) || !isfinite(scale)) return -1;
    if (kv_lens)
        for (int64_t b = 0; b < B; ++b)
            if (kv_lens[b] < 0 || kv_lens[b] > Nk) return -1;
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* s = (double*)malloc((size_t)Nk * sizeof(double));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4) collapse(2)
            for (int64_t bh = 0; bh < B * H; ++bh) {
                for (int64_t i = 0; i < Nq; ++i) {
                    const int64_t n_b = kv_lens ? kv_lens[bh / H] : Nk;
                    const int64_t diag = i + (align ? n_b - Nq : 0);
                    int64_t lo = left < 0 ? 0 : diag - left;
                    int64_t hi = right < 0 ? n_b - 1 : diag + right;
                    if (lo < 0) lo = 0;
                    if (hi > n_b - 1) hi = n_b - 1;
                    const double* qi = q + (bh * Nq + i) * d;
                    double* oi = o + (bh * Nq + i) * d;
                    double* li = lse + bh * Nq + i;
                    if (hi < lo) {
                        for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
                        *li = -INFINITY;
                        continue;
                    }
                    /* keys lo..hi of this head: the row routine over a shifted block */
                    oracle_row_n(qi, k + (bh * Nk + lo) * d, v + (bh * Nk + lo) * d, d, hi - lo + 1,
                                 scale, s, oi, li);
                }
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* Backward of the forward above: the vector-Jacobian product of O = attn(Q, K, V)
 * with an upstream gradient dO, i.e. the gradients of sum(dO * O) with respect to
 * Q, K and V. "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel", "Future
 * articles", names it as the FA2 backward that consumes the saved L; the forward
 * there is a torch.autograd.Function, so its backward is the chain rule through the
 * definition, written out per query row i over its visible keys j:
 *
 *   P_ij  = exp(s_ij - LSE_i)             softmax weights (LSE of the row itself)
 *   dV_j += P_ij dO_i                     O_i = sum_j P_ij v_j
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij              (equals dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)            Jacobian of the row softmax
 *   dQ_i  = scale sum_j dS_ij k_j         s_ij = scale q_i . k_j
 *   dK_j += scale dS_ij q_i
 *
 * q, k, v, dout, dq, dk, dv: [BH][N][d]. One head per OpenMP task, rows in order,
 * so the result does not depend on the thread count. */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, int64_t BH, int64_t N, int64_t d,
                    int causal, double scale)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || BH < 1 || N < 1 || d < 1) return -1;
    if (!(scale > 0.0) || !isfinite(scale)) return -1;
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* p = (double*)malloc((size_t)N * sizeof(double));
        double* dp = (double*)malloc((size_t)N * sizeof(double));
        if (!p || !dp) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < BH; ++bh) {
                const double* Q = q + bh * N * d;
                const double* K = k + bh * N * d;
                const double* V = v + bh * N * d;
                const double* DO = dout + bh * N * d;
                double* DQ = dq + bh * N * d;
                double* DK = dk + bh * N * d;
                double* DV = dv + bh * N * d;
                memset(DK, 0, (size_t)(N * d) * sizeof(double));
                memset(DV, 0, (size_t)(N * d) * sizeof(double));
                for (int64_t i = 0; i < N; ++i) {
                    const int64_t n_vis = causal ? i + 1 : N;
                    const double* qi = Q + i * d;
                    const double* doi = DO + i * d;
                    double m = -INFINITY;
                    for (int64_t j = 0; j < n_vis; ++j) {
                        double dot = 0.0;
                        for (int64_t t = 0; t < d; ++t) dot += qi[t] * K[j * d + t];
                        p[j] = scale * dot;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (int64_t j = 0; j < n_vis; ++j) l += exp(p[j] - m);
                    const double lse = m + log(l);
                    double Di = 0.0;
                    for (int64_t j = 0; j < n_vis; ++j) {
                        p[j] = exp(p[j] - lse);
                        double dot = 0.0;
                        for (int64_t t = 0; t < d; ++t) dot += doi[t] * V[j * d + t];
                        dp[j] = dot;
                        Di += p[j] * dot;
                    }
                    for (int64_t t = 0; t < d; ++t) DQ[i * d + t] = 0.0;
                    for (int64_t j = 0; j < n_vis; ++j) {
                        const double ds = p[j] * (dp[j] - Di);
                        for (int64_t t = 0; t < d; ++t) {
                            DV[j * d + t] += p[j] * doi[t];
                            DQ[i * d + t] += scale * ds * K[j * d + t];
                            DK[j * d + t] += scale * ds * qi[t];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return failed ? -2 : 0;
}

/* Backward of oracle_attn_fwd_window: the gradients of sum(dO * O) for Nq query rows
 * against Nk keys with key padding and a sliding window, each row over exactly the
 * keys the forward lets it see (same readings as oracle_attn_fwd_window), with the
 * chain rule of oracle_attn_bwd. q, dout, dq: [BH][Nq][d]; k, v, dk, dv: [BH][Nk][d].
 * Rows that see no key have dQ = 0 and add nothing to dK, dV; padded keys get
 * dK = dV = 0. One head per OpenMP task, rows in order. */
int oracle_attn_bwd_window(const double* q, const double* k, const double* v, const double* dout,
                           double* dq, double* dk, double* dv, int64_t B, int64_t H, int64_t Nq,
                           int64_t Nk, int64_t d, int64_t left, int64_t right,
                           const int64_t* kv_lens, int align, double scale)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1)
        return -1;
    if (!(scale > 0.0) || !isfinite(scale)) return -1;
    if (kv_lens)
        for (int64_t b = 0; b < B; ++b)
            if (kv_lens[b] < 0 || kv_lens[b] > Nk) return -1;
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* p = (double*)malloc((size_t)Nk * sizeof(double));
        double* dp = (double*)malloc((size_t)Nk * sizeof(double));
        if (!p || !dp) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < B * H; ++bh) {
                const double* Q = q + bh * Nq * d;
                const double* K = k + bh * Nk * d;
                const double* V = v + bh * Nk * d;
                const double* DO = dout + bh * Nq * d;
                double* DQ = dq + bh * Nq * d;
                double* DK = dk + bh * Nk * d;
                double* DV = dv + bh * Nk * d;
                memset(DK, 0, (size_t)(Nk * d) * sizeof(double));
                memset(DV, 0, (size_t)(Nk * d) * sizeof(double));
                const int64_t n_b = kv_lens ? kv_lens[bh / H] : Nk;
                for (int64_t i = 0; i < Nq; ++i) {
                    const int64_t diag = i + (align ? n_b - Nq : 0);
                    int64_t lo = left < 0 ? 0 : diag - left;
                    int64_t hi = right < 0 ? n_b - 1 : diag + right;
                    if (lo < 0) lo = 0;
                    if (hi > n_b - 1) hi = n_b - 1;
                    const double* qi = Q + i * d;
                    const double* doi = DO + i * d;
                    for (int64_t t = 0; t < d; ++t) DQ[i * d + t] = 0.0;
                    if (hi < lo) continue;
                    double m = -INFINITY;
                    for (int64_t j = lo; j <= hi; ++j) {
                        double dot = 0.0;
                        for (int64_t t = 0; t < d; ++t) dot += qi[t] * K[j * d + t];
                        p[j] = scale * dot;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (int64_t j = lo; j <= hi; ++j) l += exp(p[j] - m);
                    const double lse = m + log(l);
                    double Di = 0.0;
                    for (int64_t j = lo; j <= hi; ++j) {
                        p[j] = exp(p[j] - lse);
                        double dot = 0.0;
                        for (int64_t t = 0; t < d; ++t) dot += doi[t] * V[j * d + t];
                        dp[j] = dot;
                        Di += p[j] * dot;
                    }
                    for (int64_t j = lo; j <= hi; ++j) {
                        const double ds = p[j] * (dp[j] - Di);
                        for (int64_t t = 0; t < d; ++t) {
                            DV[j * d + t] += p[j] * doi[t];
                            DQ[i * d + t] += scale * ds * K[j * d + t];
                            DK[j * d + t] += scale * ds * qi[t];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return failed ? -2 : 0;
}

/* Threads an OpenMP parallel region of this library uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
