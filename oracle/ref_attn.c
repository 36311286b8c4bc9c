/*
 * Plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header or table with the CUDA
 * path.
 *
 * What it computes is the plain definition of attention that the pages say
 * the tiled method reproduces exactly ("exata, identica matematicamente a
 * versao padrao"):
 *
 *   S = tau * Q K^T                      (scaled scores, one row per query)
 *   P = softmax_row(S)  over the visible keys J(i)
 *   O = P V
 *   LSE_i = m_i + ln l_i,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
 *
 * Sources (page title, section):
 *   - tonho.wtf "flash attention" encyclopedia entry, section "como funciona":
 *     the scores tau*Q_i K_j^T, the per-row running max m and sum l, and that
 *     the output and the statistics (m, l) are what is stored.
 *   - same page, section "como funciona", backward paragraph: the backward
 *     keeps only O and (m, l), rebuilds S and P, and uses D_i = P_i . dP_i,
 *     which equals dO_i . O_i.
 *   - "Atencao eficiente - FlashAttention, sparse e hibrida", section
 *     "Insight 2 - Online softmax": the blocked softmax is identical to the
 *     softmax over the whole row.
 *
 * Readings where the pages are silent:
 *   - causal: key j is visible from query i iff j <= i (equal query and key
 *     lengths, so top-left and bottom-right alignment coincide);
 *   - sliding window of w keys ("Atencao eficiente - FlashAttention, sparse e
 *     hibrida", section "Atencao hibrida: local + global intercalados": local
 *     layers attend within a window of the most recent tokens): key j is
 *     visible from query i iff i - w < j <= i, so w counts the query's own key;
 *     w >= N is plain causal attention;
 *   - block-sparse attention ("FlashAttention e o gargalo real de
 *     inferencia", section "o que isso custou": the block-sparse variant is an
 *     approximation that skips blocks; "Atencao eficiente - FlashAttention,
 *     sparse e hibrida", section "Sparse e hibrida": each token attends to a
 *     subset, a local window plus global anchor tokens): a mask of blk x blk
 *     blocks; key j is visible from query i only if mask[i / blk][j / blk] is
 *     nonzero (and j <= i when causal).  A row that sees no key is an empty
 *     sum: O_i = 0, LSE_i = -inf, and it contributes nothing to any gradient;
 *   - decode ("Atencao eficiente - FlashAttention, sparse e hibrida", box
 *     "FlashAttention nao acelera o decode token a token": each decode step
 *     brings one new query row that reads the whole KV cache): Nq query rows
 *     against Nk >= Nq cached keys, the queries being the last Nq positions of
 *     the sequence, so with causal query i sees keys j <= i + (Nk - Nq);
 *   - LSE is in natural-log units of the tau-scaled scores;
 *   - the backward is the analytic gradient of O with respect to Q, K, V for
 *     an upstream gradient dO, with the softmax Jacobian written out as
 *     dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik).
 *
 * Layout: every tensor is a contiguous array [BH][N][d] of doubles (row-major,
 * d fastest); LSE and D are [BH][N].  BH is batch * heads.
 *
 * No blocking, fusion or reordering: each query row is done on its own, in
 * the order of the definition above.  OpenMP only splits independent rows
 * or heads across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Which keys each query sees. */
typedef struct {
    int causal;            /* only keys j <= i + offset */
    int64_t offset;        /* causal offset: Nk - Nq for decode, 0 when square */
    int64_t window;        /* > 0: only the `window` most recent keys, i - window < j */
    const uint8_t* blocks; /* NULL, or block masks [heads][nqb][nkb] (nonzero = visible) */
    int64_t blk;           /* edge of a mask block, in rows and in keys */
    int64_t nkb;           /* key blocks per mask row */
    int64_t head_stride;   /* bytes from one head's mask to the next (0: shared mask) */
} Visibility;

/* Key j is visible from query i of head bh. */
static int visible(const Visibility* vs, int64_t bh, int64_t i, int64_t j)
{
    if (vs->causal && j > i + vs->offset) return 0;
    if (vs->window > 0 && j <= i - vs->window) return 0;
    if (vs->blocks && !vs->blocks[bh * vs->head_stride + (i / vs->blk) * vs->nkb + j / vs->blk])
        return 0;
    return 1;
}

static double dot(const double* a, const double* b, int64_t d)
{
    double s = 0.0;
    for (int64_t k = 0; k < d; ++k) s += a[k] * b[k];
    return s;
}

/*
 * One query row of the forward pass.
 *   q     : the query row (d values)
 *   K, V  : the keys and values of this head ([N][d])
 *   vs,bh,i: which keys query i of head bh sees
 *   p     : scratch of N doubles; on return p[j] = P_ij (0 for hidden keys)
 *   o     : d outputs, O_i = sum_j P_ij V_j
 *   lse   : m + ln l
 * A query that sees no key gets p = 0, o = 0 and lse = -inf (the empty sum).
 */
static void row_forward(const double* q, const double* K, const double* V,
                        const Visibility* vs, int64_t bh, int64_t i, int64_t N, int64_t d,
                        double tau, double* p, double* o, double* lse)
{
    double m = -INFINITY;
    int64_t seen = 0;
    for (int64_t j = 0; j < N; ++j) {
        if (visible(vs, bh, i, j)) {
            p[j] = tau * dot(q, K + j * d, d);
            if (p[j] > m) m = p[j];
            ++seen;
        }
    }
    if (seen == 0) {
        for (int64_t j = 0; j < N; ++j) p[j] = 0.0;
        for (int64_t k = 0; k < d; ++k) o[k] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (visible(vs, bh, i, j)) {
            p[j] = exp(p[j] - m);
            l += p[j];
        } else {
            p[j] = 0.0;
        }
    }
    for (int64_t j = 0; j < N; ++j) p[j] /= l;
    for (int64_t k = 0; k < d; ++k) o[k] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (p[j] == 0.0) continue;
        const double* v = V + j * d;
        for (int64_t k = 0; k < d; ++k) o[k] += p[j] * v[k];
    }
    *lse = m + log(l);
}

/* Number of threads a parallel region of this library uses. */
int ora_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ora_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * The attention probabilities P [BH][N][N] (row i is the softmax of the
 * visible scaled scores of query i; hidden keys get 0).  For small checks.
 */
static void attn_probs(const double* Q, const double* K, const double* V,
                       int64_t BH, int64_t N, int64_t d, double tau, const Visibility* vs,
                       double* P)
{
    int64_t rows = BH * N;
#pragma omp parallel
    {
        double* o = (double*)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t bh = r / N, i = r % N;
            double lse;
            row_forward(Q + r * d, K + bh * N * d, V + bh * N * d, vs, bh, i, N, d, tau,
                        P + r * N, o, &lse);
        }
        free(o);
    }
}

/* Forward pass over every row: O [BH][N][d], LSE [BH][N]. */
static void attn_fwd(const double* Q, const double* K, const double* V,
                     int64_t BH, int64_t N, int64_t d, double tau, const Visibility* vs,
                     double* O, double* LSE)
{
    int64_t rows = BH * N;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t bh = r / N, i = r % N;
            row_forward(Q + r * d, K + bh * N * d, V + bh * N * d, vs, bh, i, N, d, tau,
                        p, O + r * d, LSE + r);
        }
        free(p);
    }
}

/*
 * Forward pass on a chosen set of rows.  rows[k] = bh * N + i names query i of
 * head bh; outputs O_rows [nrows][d] and LSE_rows [nrows] in the same order.
 */
static void attn_fwd_rows(const double* Q, const double* K, const double* V,
                          int64_t BH, int64_t N, int64_t d, double tau, const Visibility* vs,
                          const int64_t* rows, int64_t nrows,
                          double* O_rows, double* LSE_rows)
{
    (void)BH;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t k = 0; k < nrows; ++k) {
            int64_t r = rows[k];
            int64_t bh = r / N, i = r % N;
            row_forward(Q + r * d, K + bh * N * d, V + bh * N * d, vs, bh, i, N, d, tau,
                        p, O_rows + k * d, LSE_rows + k);
        }
        free(p);
    }
}

/*
 * Backward pass: the gradients of O = softmax(tau Q K^T) V with respect to
 * Q, K and V for an upstream gradient dO, per head:
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = sum_j P_ij dP_ij          (softmax Jacobian term)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = tau sum_j dS_ij K_j
 *   dK_j  = tau sum_i dS_ij Q_i
 *
 * P is recomputed here from Q and K (the oracle's own fp64 forward).  O_out,
 * LSE_out and D_out are optional extra outputs (pass NULL to skip); D_out is
 * the softmax-Jacobian row sum above, so a test can hold it against dO_i . O_i.
 */
static void attn_bwd(const double* Q, const double* K, const double* V,
                     const double* dO,
                     int64_t BH, int64_t N, int64_t d, double tau, const Visibility* vs,
                     double* dQ, double* dK, double* dV,
                     double* O_out, double* LSE_out, double* D_out)
{
#pragma omp parallel
    {
        double* P = (double*)malloc(sizeof(double) * (size_t)(N * N));
        double* dS = (double*)malloc(sizeof(double) * (size_t)(N * N));
        double* o = (double*)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < BH; ++bh) {
            const double* Qh = Q + bh * N * d;
            const double* Kh = K + bh * N * d;
            const double* Vh = V + bh * N * d;
            const double* dOh = dO + bh * N * d;
            double* dQh = dQ + bh * N * d;
            double* dKh = dK + bh * N * d;
            double* dVh = dV + bh * N * d;

            /* forward: P and (optionally) O, LSE */
            for (int64_t i = 0; i < N; ++i) {
                double lse;
                row_forward(Qh + i * d, Kh, Vh, vs, bh, i, N, d, tau, P + i * N, o, &lse);
                if (O_out) memcpy(O_out + (bh * N + i) * d, o, sizeof(double) * (size_t)d);
                if (LSE_out) LSE_out[bh * N + i] = lse;
            }
            /* dP, D and dS, row by row */
            for (int64_t i = 0; i < N; ++i) {
                double* dSi = dS + i * N;
                const double* Pi = P + i * N;
                double Di = 0.0;
                for (int64_t j = 0; j < N; ++j) {
                    dSi[j] = visible(vs, bh, i, j) ? dot(dOh + i * d, Vh + j * d, d) : 0.0;
                    Di += Pi[j] * dSi[j];
                }
                for (int64_t j = 0; j < N; ++j) dSi[j] = Pi[j] * (dSi[j] - Di);
                if (D_out) D_out[bh * N + i] = Di;
            }
            /* dQ_i = tau sum_j dS_ij K_j */
            for (int64_t i = 0; i < N; ++i) {
                double* g = dQh + i * d;
                for (int64_t k = 0; k < d; ++k) g[k] = 0.0;
                for (int64_t j = 0; j < N; ++j) {
                    double w = dS[i * N + j];
                    if (w == 0.0) continue;
                    for (int64_t k = 0; k < d; ++k) g[k] += w * Kh[j * d + k];
                }
                for (int64_t k = 0; k < d; ++k) g[k] *= tau;
            }
            /* dK_j = tau sum_i dS_ij Q_i ;  dV_j = sum_i P_ij dO_i */
            for (int64_t j = 0; j < N; ++j) {
                double* gk = dKh + j * d;
                double* gv = dVh + j * d;
                for (int64_t k = 0; k < d; ++k) { gk[k] = 0.0; gv[k] = 0.0; }
                for (int64_t i = 0; i < N; ++i) {
                    double ws = dS[i * N + j], wp = P[i * N + j];
                    if (ws != 0.0)
                        for (int64_t k = 0; k < d; ++k) gk[k] += ws * Qh[i * d + k];
                    if (wp != 0.0)
                        for (int64_t k = 0; k < d; ++k) gv[k] += wp * dOh[i * d + k];
                }
                for (int64_t k = 0; k < d; ++k) gk[k] *= tau;
            }
        }
        free(P);
        free(dS);
        free(o);
    }
}

/* ---------------------------------------------------------------- exports --
 * Plain entry points (no window), sliding-window entry points (causal, key j
 * visible from query i iff i - window < j <= i, window >= 1) and block-mask
 * entry points (blocks: [mask_heads][nqb][nkb] bytes with nqb = nkb =
 * ceil(N / blk), mask_heads 1 = one mask for every head, else BH). */
static Visibility plain_vis(int causal, int64_t window)
{
    Visibility vs = {causal, 0, window, NULL, 1, 0, 0};
    return vs;
}

static Visibility block_vis(int causal, const uint8_t* blocks, int64_t blk, int64_t mask_heads,
                            int64_t N)
{
    int64_t nb = (N + blk - 1) / blk;
    Visibility vs = {causal, 0, 0, blocks, blk, nb, mask_heads == 1 ? 0 : nb * nb};
    return vs;
}

void ora_attn_probs(const double* Q, const double* K, const double* V, int64_t BH, int64_t N,
                    int64_t d, double tau, int causal, double* P)
{
    Visibility vs = plain_vis(causal, 0);
    attn_probs(Q, K, V, BH, N, d, tau, &vs, P);
}

void ora_attn_fwd(const double* Q, const double* K, const double* V, int64_t BH, int64_t N,
                  int64_t d, double tau, int causal, double* O, double* LSE)
{
    Visibility vs = plain_vis(causal, 0);
    attn_fwd(Q, K, V, BH, N, d, tau, &vs, O, LSE);
}

void ora_attn_fwd_rows(const double* Q, const double* K, const double* V, int64_t BH, int64_t N,
                       int64_t d, double tau, int causal, const int64_t* rows, int64_t nrows,
                       double* O_rows, double* LSE_rows)
{
    Visibility vs = plain_vis(causal, 0);
    attn_fwd_rows(Q, K, V, BH, N, d, tau, &vs, rows, nrows, O_rows, LSE_rows);
}

void ora_attn_bwd(const double* Q, const double* K, const double* V, const double* dO,
                  int64_t BH, int64_t N, int64_t d, double tau, int causal,
                  double* dQ, double* dK, double* dV, double* O_out, double* LSE_out, double* D_out)
{
    Visibility vs = plain_vis(causal, 0);
    attn_bwd(Q, K, V, dO, BH, N, d, tau, &vs, dQ, dK, dV, O_out, LSE_out, D_out);
}

void ora_attn_probs_window(const double* Q, const double* K, const double* V, int64_t BH,
                           int64_t N, int64_t d, double tau, int64_t window, double* P)
{
    Visibility vs = plain_vis(1, window);
    attn_probs(Q, K, V, BH, N, d, tau, &vs, P);
}

void ora_attn_fwd_window(const double* Q, const double* K, const double* V, int64_t BH, int64_t N,
                         int64_t d, double tau, int64_t window, double* O, double* LSE)
{
    Visibility vs = plain_vis(1, window);
    attn_fwd(Q, K, V, BH, N, d, tau, &vs, O, LSE);
}

void ora_attn_fwd_rows_window(const double* Q, const double* K, const double* V, int64_t BH,
                              int64_t N, int64_t d, double tau, int64_t window,
                              const int64_t* rows, int64_t nrows, double* O_rows, double* LSE_rows)
{
    Visibility vs = plain_vis(1, window);
    attn_fwd_rows(Q, K, V, BH, N, d, tau, &vs, rows, nrows, O_rows, LSE_rows);
}

void ora_attn_bwd_window(const double* Q, const double* K, const double* V, const double* dO,
                         int64_t BH, int64_t N, int64_t d, double tau, int64_t window,
                         double* dQ, double* dK, double* dV, double* O_out, double* LSE_out,
                         double* D_out)
{
    Visibility vs = plain_vis(1, window);
    attn_bwd(Q, K, V, dO, BH, N, d, tau, &vs, dQ, dK, dV, O_out, LSE_out, D_out);
}

void ora_attn_probs_blocks(const double* Q, const double* K, const double* V, int64_t BH,
                           int64_t N, int64_t d, double tau, int causal, const uint8_t* blocks,
                           int64_t blk, int64_t mask_heads, double* P)
{
    Visibility vs = block_vis(causal, blocks, blk, mask_heads, N);
    attn_probs(Q, K, V, BH, N, d, tau, &vs, P);
}

void ora_attn_fwd_blocks(const double* Q, const double* K, const double* V, int64_t BH, int64_t N,
                         int64_t d, double tau, int causal, const uint8_t* blocks, int64_t blk,
                         int64_t mask_heads, double* O, double* LSE)
{
    Visibility vs = block_vis(causal, blocks, blk, mask_heads, N);
    attn_fwd(Q, K, V, BH, N, d, tau, &vs, O, LSE);
}

void ora_attn_fwd_rows_blocks(const double* Q, const double* K, const double* V, int64_t BH,
                              int64_t N, int64_t d, double tau, int causal, const uint8_t* blocks,
                              int64_t blk, int64_t mask_heads, const int64_t* rows, int64_t nrows,
                              double* O_rows, double* LSE_rows)
{
    Visibility vs = block_vis(causal, blocks, blk, mask_heads, N);
    attn_fwd_rows(Q, K, V, BH, N, d, tau, &vs, rows, nrows, O_rows, LSE_rows);
}

void ora_attn_bwd_blocks(const double* Q, const double* K, const double* V, const double* dO,
                         int64_t BH, int64_t N, int64_t d, double tau, int causal,
                         const uint8_t* blocks, int64_t blk, int64_t mask_heads,
                         double* dQ, double* dK, double* dV, double* O_out, double* LSE_out,
                         double* D_out)
{
    Visibility vs = block_vis(causal, blocks, blk, mask_heads, N);
    attn_bwd(Q, K, V, dO, BH, N, d, tau, &vs, dQ, dK, dV, O_out, LSE_out, D_out);
}

/*
 * Decode forward: Nq query rows per head ([BH][Nq][d]) against Nk cached keys
 * and values ([BH][Nk][d]); with causal, query i is at position Nk - Nq + i
 * and sees keys j <= i + (Nk - Nq).  Outputs O [BH][Nq][d], LSE [BH][Nq].
 */
void ora_attn_fwd_decode(const double* Q, const double* K, const double* V, int64_t BH,
                         int64_t Nq, int64_t Nk, int64_t d, double tau, int causal,
                         double* O, double* LSE)
{
    Visibility vs = {causal, Nk - Nq, 0, NULL, 1, 0, 0};
    int64_t rows = BH * Nq;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t bh = r / Nq, i = r % Nq;
            row_forward(Q + r * d, K + bh * Nk * d, V + bh * Nk * d, &vs, bh, i, Nk, d, tau,
                        p, O + r * d, LSE + r);
        }
        free(p);
    }
}

/*
 * FP8 inputs.  The FP8 forward of the pages' FlashAttention-3 note ("Atencao
 * eficiente - FlashAttention, sparse e hibrida", the FlashAttention-4 box)
 * takes e4m3 tensors with one scale each; the attention it approximates is
 * the plain definition above on the decoded values x * scale, so the oracle
 * only adds the decoding.  OCP FP8 E4M3: bit 7 sign, bits 3-6 exponent e
 * (bias 7), bits 0-2 mantissa m; e = 0 is subnormal, (m / 8) 2^-6; otherwise
 * (1 + m / 8) 2^(e - 7); e = 15 with m = 7 is NaN; there are no infinities.
 */
void ora_e4m3_decode(const uint8_t* x, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) {
        const int s = x[i] >> 7, e = (x[i] >> 3) & 15, m = x[i] & 7;
        double v;
        if (e == 15 && m == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m / 8.0, -6);
        else
            v = ldexp(1.0 + (double)m / 8.0, e - 7);
        out[i] = s ? -v : v;
    }
}
