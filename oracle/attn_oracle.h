/*
 * attn_oracle.h -- plain, slow, fp64 CPU oracle for scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call
 * this library; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition, per batch b, head h and query row i):
 *   Eq. (1)  Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V
 *     -- "Attention Is All You Need" (rockcohen.cc), section 5.1 "scaled
 *        dot-product attention"; vlmlib.cn paper summary, "scaled dot-product
 *        attention"; attention-paper-guide, section 03.2.
 *   Illegal connections get -inf at the softmax INPUT, so their weight is an
 *   exact 0 -- rockcohen.cc sections 5.3 and 6.3.
 *   Causal (decoder self-attention): key j is illegal for query i when j > i.
 *   Key padding (encoder, cross-attention): key j is illegal when j >= key_lens[b]
 *   (right padding; the reading of the csdn blog's padding mask).
 *   Decode (autoregressive generation, one step of n_q new queries against a key
 *   cache of key_lens[b] entries): query i sits at position key_lens[b] - n_q + i
 *   and key j is illegal when j > key_lens[b] - n_q + i. This is the causal mask
 *   of decoder self-attention applied to the newest n_q positions (attention-paper-
 *   guide section 05 and rockcohen.cc section 6.3: generation proceeds one position
 *   at a time and each position sees only positions up to itself).
 *   Local window (restricted self-attention, the pages' long-sequence proposal:
 *   attend only to positions within a neighbourhood r, cost O(r n d); csdn blog
 *   section 4.3, vlmlib.cn "limitations"): key j is illegal when |i - j| > window.
 *
 * Conventions chosen where the pages are silent:
 *   - a row with no legal key returns o = 0 and lse = -inf;
 *   - lse_i = ln sum_{j legal} exp(scale * q_i . k_j)  (natural log);
 *   - scale is used exactly as given (callers pass 1/sqrt(d_k)).
 *
 * Layouts: Q [B,H,n_q,d_k], K [B,H,n_k,d_k], V [B,H,n_k,d_v], O [B,H,n_q,d_v],
 * all contiguous row-major, the per-head layout of the csdn blog's split_heads.
 */
#ifndef ATTN_ORACLE_H
#define ATTN_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* element type of the Q/K/V input arrays */
enum { ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_BF16 = 2 /* raw bf16 bit patterns, uint16 */ };
/* mask bits */
enum { ORACLE_MASK_CAUSAL = 1, ORACLE_MASK_KEY_PADDING = 2, ORACLE_MASK_DECODE = 4, ORACLE_MASK_WINDOW = 8 };

/* Full output. out: B*H*n_q*d_v doubles; lse: B*H*n_q doubles or NULL.
 * key_lens: B ints, required iff mask bit 2 or 4 is set. Bits 1 and 4 are exclusive.
 * window: radius of mask bit 8 (>= 0), ignored otherwise; bits 4 and 8 are exclusive.
 * n_threads <= 0 means 1.
 * Returns 0, or -1 on an invalid argument. */
int oracle_attn(const void* q, const void* k, const void* v, int dtype,
                int B, int H, int n_q, int n_k, int d_k, int d_v, double scale,
                int mask_mode, const int* key_lens, int window,
                double* out, double* lse, int n_threads);

/* A subset of query rows. row_ids[r] = (b*H + h)*n_q + i. out_rows: n_rows*d_v,
 * lse_rows: n_rows (or NULL). Same semantics as oracle_attn for those rows. */
int oracle_attn_rows(const void* q, const void* k, const void* v, int dtype,
                     int B, int H, int n_q, int n_k, int d_k, int d_v, double scale,
                     int mask_mode, const int* key_lens, int window,
                     long long n_rows, const long long* row_ids,
                     double* out_rows, double* lse_rows, int n_threads);

/* The softmax weight matrix A = softmax(scale * Q K^T + mask): B*H*n_q*n_k doubles.
 * Illegal entries are exactly 0.0; a row with no legal key is all zeros. */
int oracle_attn_weights(const void* q, const void* k, int dtype,
                        int B, int H, int n_q, int n_k, int d_k, double scale,
                        int mask_mode, const int* key_lens, int window, double* weights);

/* Gradients of L = sum(dout * O) with respect to Q, K and V (training needs them:
 * attention-paper-guide section 05, vlmlib.cn "training"), for the same mask
 * semantics. dout has O's shape and the inputs' dtype. Per row i:
 *   P_i  = softmax row of the forward (illegal entries exactly 0)
 *   dP_ij = dout_i . v_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)       (the softmax Jacobian)
 *   dq_i  = scale sum_j dS_ij k_j,  dk_j += scale dS_ij q_i,  dv_j += P_ij dout_i
 * dq: B*H*n_q*d_k, dk: B*H*n_k*d_k, dv: B*H*n_k*d_v doubles. Threads split the heads. */
int oracle_attn_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
                    int B, int H, int n_q, int n_k, int d_k, int d_v, double scale,
                    int mask_mode, const int* key_lens, int window,
                    double* dq, double* dk, double* dv, int n_threads);

/* Multi-head attention (vlmlib.cn "multi-head attention": MultiHead(Q,K,V) =
 * Concat(head_1..head_h) W^O with head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V); the
 * csdn blog's MultiHeadAttention: linear projections with biases, split_heads,
 * attention, transpose back and concatenate, output projection):
 *   x_q [B, n_q, d_model] (the queries' source), x_kv [B, n_k, d_model] (keys' and
 *   values' source; the same array for self-attention);
 *   w_q, w_k [d_model, H*d_k], w_v [d_model, H*d_v], w_o [H*d_v, d_model], row-major
 *   as in x W (the paper's orientation); W_i^Q is columns i*d_k .. i*d_k + d_k - 1;
 *   b_q, b_k [H*d_k], b_v [H*d_v], b_o [d_model], each may be NULL (no bias);
 *   every input has the same dtype; mask_mode/key_lens as oracle_attn (causal and key
 *   padding only); y [B, n_q, d_model] doubles. Everything is accumulated in fp64
 *   with no intermediate rounding. Returns 0, or -1 on an invalid argument. */
int oracle_mha(const void* x_q, const void* x_kv, int dtype, const void* w_q, const void* b_q,
               const void* w_k, const void* b_k, const void* w_v, const void* b_v,
               const void* w_o, const void* b_o, int B, int n_q, int n_k, int d_model, int H,
               int d_k, int d_v, double scale, int mask_mode, const int* key_lens, double* y,
               int n_threads);

/* One linear projection of the multi-head layer (vlmlib.cn "multi-head attention":
 * the per-head matrices W_i side by side, x W; the csdn blog's nn.Linear with its
 * bias): y[m, n] = bias[n] + sum_k x[m, k] w[k, n], x [M, K] and w [K, N] row-major
 * in the paper's x W orientation, bias [N] or NULL, every input of one dtype, y
 * [M, N] doubles accumulated in fp64 with no intermediate rounding. Returns 0, or -1
 * on an invalid argument. */
int oracle_linear(const void* x, const void* w, const void* bias, int dtype, int M, int N, int K, double* y);

#ifdef __cplusplus
}
#endif
#endif
