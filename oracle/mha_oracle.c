/*
 * mha_oracle.c -- fp64 CPU oracle for the multi-head attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker that the GPU path is
 * compared against. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it. It shares no code, header, table or
 * helper with the CUDA library, and it includes nothing from it.
 *
 * What it computes is the plain definition of the sublayer, in the order the
 * pages give it, with no blocking, fusion or reordering:
 *
 *   "The Annotated Transformer" (Chinese rendering), section "Attention",
 *   function attention():  scores = Q K^T / sqrt(d_k);
 *                          scores = scores.masked_fill(mask == 0, -1e9);
 *                          p_attn = softmax(scores, dim=-1);  out = p_attn V
 *   "003-Transformer" tutorial, section "Multi-head attention"
 *   (MultiHeadedAttention.forward):  four nn.Linear(d_model, d_model) layers,
 *     the first three applied to query/key/value and viewed as
 *     (B, L, h, d_k) -> (B, h, L, d_k); attention() per head with the mask
 *     broadcast over heads (mask.unsqueeze(1)); heads transposed back and
 *     concatenated to (B, L, h*d_k); the fourth Linear applied last.
 *   nn.Linear convention: y = x W^T + b with W stored [out, in].
 *
 * Mask (1 = may attend, 0 = masked); the three parts are AND-ed:
 *   causal:  key j allowed for query i iff j <= i ("The Annotated Transformer",
 *            subsequent_mask(): triu(ones, diagonal=1) == 0, diagonal allowed;
 *            the 5x5 matrix printed in the "003-Transformer" tutorial, section
 *            "Masks").
 *   key valid length (d2l MultiHeadAttention valid_lens, d2l Transformer
 *            chapter summary): key j allowed iff j < valid_lens[b].
 *   dense:   a byte mask [B, mq, L_k] with mq in {1, L_q}; mq == 1 broadcasts
 *            over queries (labml mha: "query dimension 1 is broadcast").
 *
 * Dropout is the identity (forward / evaluation).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* nn.Linear: y[r, o] = sum_i x[r, i] * W[o, i] + b[o]; b may be NULL (no bias). */
void oracle_linear(const double* x, const double* W, const double* b,
                   long rows, int din, int dout, double* y)
{
    long r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        const double* xr = x + r * (long)din;
        double* yr = y + r * (long)dout;
        for (int o = 0; o < dout; ++o) {
            const double* wo = W + (long)o * din;
            double acc = 0.0;
            for (int i = 0; i < din; ++i) acc += xr[i] * wo[i];
            yr[o] = acc + (b ? b[o] : 0.0);
        }
    }
}

/* mask(b, i, j) of the pages: 1 = query i of batch b may attend to key j. */
static int oracle_allowed(int b, int i, int j, int Lq, int Lk, int causal,
                          const int* valid_lens, const unsigned char* dense,
                          int dense_mq)
{
    if (causal && j > i) return 0;
    if (valid_lens && j >= valid_lens[b]) return 0;
    if (dense) {
        long qi = (dense_mq == 1) ? 0 : i;
        long mq = (dense_mq == 1) ? 1 : Lq;
        if (dense[((long)b * mq + qi) * Lk + j] == 0) return 0;
    }
    return 1;
}

/*
 * oracle_mha_forward -- the whole sublayer in fp64.
 *
 * query [B, Lq, d], key [B, Lk, d], value [B, Lk, d]   (row-major)
 * w_* [d, d] (out, in), b_* [d] or NULL
 * rows: NULL for every query position, else nrows query positions (each in
 *       [0, Lq)) whose outputs are wanted; out is then [B, nrows, d] and
 *       p_attn [B, h, nrows, Lk].
 * out:  [B, nrows or Lq, d];  p_attn: NULL or [B, h, nrows or Lq, Lk].
 *
 * Returns 0 on success, 1 if d is not a multiple of h or a size is not
 * positive (the pages assert embedding_dim % head == 0), 2 on allocation
 * failure, 3 if a requested row is out of range.
 */
int oracle_mha_forward(const double* query, const double* key, const double* value,
                       const double* w_q, const double* b_q,
                       const double* w_k, const double* b_k,
                       const double* w_v, const double* b_v,
                       const double* w_o, const double* b_o,
                       int B, int Lq, int Lk, int d, int h,
                       int causal, const int* valid_lens,
                       const unsigned char* dense, int dense_mq,
                       const int* rows, int nrows,
                       double* out, double* p_attn)
{
    if (B <= 0 || Lq <= 0 || Lk <= 0 || d <= 0 || h <= 0 || d % h != 0) return 1;
    const int dk = d / h;
    const int nr = rows ? nrows : Lq;
    if (nr <= 0) return 1;
    if (rows)
        for (int r = 0; r < nr; ++r)
            if (rows[r] < 0 || rows[r] >= Lq) return 3;
    const double sqrt_dk = sqrt((double)dk);

    double* Kp = (double*)malloc(sizeof(double) * (size_t)Lk * d);
    double* Vp = (double*)malloc(sizeof(double) * (size_t)Lk * d);
    double* Xq = (double*)malloc(sizeof(double) * (size_t)nr * d);
    double* Qp = (double*)malloc(sizeof(double) * (size_t)nr * d);
    double* ctx = (double*)malloc(sizeof(double) * (size_t)nr * d);
    if (!Kp || !Vp || !Xq || !Qp || !ctx) {
        free(Kp); free(Vp); free(Xq); free(Qp); free(ctx);
        return 2;
    }

    for (int b = 0; b < B; ++b) {
        /* Step 1: the three input projections (K and V for every key). */
        oracle_linear(key + (long)b * Lk * d, w_k, b_k, Lk, d, d, Kp);
        oracle_linear(value + (long)b * Lk * d, w_v, b_v, Lk, d, d, Vp);
        for (int r = 0; r < nr; ++r) {
            int i = rows ? rows[r] : r;
            memcpy(Xq + (long)r * d, query + ((long)b * Lq + i) * d, sizeof(double) * d);
        }
        oracle_linear(Xq, w_q, b_q, nr, d, d, Qp);

        /* Steps 2-6: per query row and head, scores, fill, softmax, P.V, concat. */
        int r;
#pragma omp parallel for schedule(dynamic, 1)
        for (r = 0; r < nr; ++r) {
            const int i = rows ? rows[r] : r;
            double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
            for (int hh = 0; hh < h; ++hh) {
                const double* q = Qp + (long)r * d + (long)hh * dk;
                /* scores = q . k_j / sqrt(d_k), then masked_fill(mask == 0, -1e9) */
                for (int j = 0; j < Lk; ++j) {
                    const double* kj = Kp + (long)j * d + (long)hh * dk;
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) acc += q[c] * kj[c];
                    s[j] = acc / sqrt_dk;
                    if (!oracle_allowed(b, i, j, Lq, Lk, causal, valid_lens, dense, dense_mq))
                        s[j] = -1e9;
                }
                /* softmax over keys: exp(s - max) / sum */
                double m = s[0];
                for (int j = 1; j < Lk; ++j) if (s[j] > m) m = s[j];
                double z = 0.0;
                for (int j = 0; j < Lk; ++j) { s[j] = exp(s[j] - m); z += s[j]; }
                for (int j = 0; j < Lk; ++j) s[j] /= z;
                if (p_attn) {
                    double* pr = p_attn + (((long)b * h + hh) * nr + r) * Lk;
                    for (int j = 0; j < Lk; ++j) pr[j] = s[j];
                }
                /* head output p . V, written at the head's place in the concat */
                double* o = ctx + (long)r * d + (long)hh * dk;
                for (int c = 0; c < dk; ++c) o[c] = 0.0;
                for (int j = 0; j < Lk; ++j) {
                    const double* vj = Vp + (long)j * d + (long)hh * dk;
                    const double pj = s[j];
                    for (int c = 0; c < dk; ++c) o[c] += pj * vj[c];
                }
            }
            free(s);
        }
        /* Step 7: output projection W_o. */
        oracle_linear(ctx, w_o, b_o, nr, d, d, out + (long)b * nr * d);
    }
    free(Kp); free(Vp); free(Xq); free(Qp); free(ctx);
    return 0;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * oracle_ffn_forward -- position-wise feed-forward network in fp64
 * ("003-Transformer" tutorial, section on the feed-forward layer, and "From RNN
 * to Attention", part 3, FFN: FFN(x) = max(0, x W_1 + b_1) W_2 + b_2, as
 * PositionwiseFeedForward: w_1 = nn.Linear(d_model, d_ff), w_2 = nn.Linear(d_ff,
 * d_model), relu between them; dropout is the identity).
 * x [rows, d_model]; w_1 [d_ff, d_model]; w_2 [d_model, d_ff]; b_* or NULL.
 * Returns 0, or 1 on non-positive sizes, 2 on allocation failure.
 */
int oracle_ffn_forward(const double* x, const double* w_1, const double* b_1,
                       const double* w_2, const double* b_2,
                       long rows, int d_model, int d_ff, double* out)
{
    if (rows <= 0 || d_model <= 0 || d_ff <= 0) return 1;
    double* hid = (double*)malloc(sizeof(double) * (size_t)rows * d_ff);
    if (!hid) return 2;
    oracle_linear(x, w_1, b_1, rows, d_model, d_ff, hid);
    for (long i = 0; i < rows * (long)d_ff; ++i) if (hid[i] < 0.0) hid[i] = 0.0;   /* relu */
    oracle_linear(hid, w_2, b_2, rows, d_ff, d_model, out);
    free(hid);
    return 0;
}

/*
 * oracle_layernorm -- per row of x [rows, d] in fp64.
 * kind 0 ("The Annotated Transformer", LayerNorm):
 *     a * (x - mean) / (std + eps) + b,  std = sqrt(sum (x - mean)^2 / (d - 1))  (unbiased)
 * kind 1 (nn.LayerNorm, "003-Transformer" SublayerConnection):
 *     a * (x - mean) / sqrt(var + eps) + b,  var = sum (x - mean)^2 / d  (biased)
 * a, b [d] or NULL (= ones / zeros). Returns 0, or 1 on bad sizes / kind.
 */
int oracle_layernorm(const double* x, const double* a, const double* b, long rows, int d, double eps,
                     int kind, double* y)
{
    if (rows <= 0 || d <= 0 || (kind != 0 && kind != 1) || (kind == 0 && d < 2)) return 1;
    long r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        const double* xr = x + r * (long)d;
        double* yr = y + r * (long)d;
        double mean = 0.0;
        for (int i = 0; i < d; ++i) mean += xr[i];
        mean /= d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += (xr[i] - mean) * (xr[i] - mean);
        const double denom = (kind == 0) ? sqrt(ss / (d - 1)) + eps : sqrt(ss / d + eps);
        for (int i = 0; i < d; ++i)
            yr[i] = (a ? a[i] : 1.0) * (xr[i] - mean) / denom + (b ? b[i] : 0.0);
    }
    return 0;
}
