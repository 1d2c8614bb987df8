/*
 * attn_gb300.h -- C ABI of the GB300 (sm_103a) scaled dot-product attention
 * forward library, libattn_gb300.so.
 *
 * The operation (per batch b, head h, query row i):
 *
 *   O[b,h,i,:] = sum_j softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] + mask(b,i,j) ) V[b,h,j,:]
 *
 * i.e. Eq. (1), Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, of "Attention
 * Is All You Need" (rockcohen.cc/paper/t1-transformer, section 5.1; vlmlib.cn
 * paper summary, "scaled dot-product attention"), applied independently to
 * every head of multi-head attention (vlmlib.cn, "multi-head attention";
 * rockcohen.cc section 5.2). mask(b,i,j) is 0 for a legal connection and -inf for
 * an illegal one, added at the softmax input, so illegal keys get an exact zero
 * weight (rockcohen.cc sections 5.3 and 6.3). The three uses of attention
 * (rockcohen.cc section 5.3) are expressed through mask_mode and the shapes:
 *   encoder self-attention      ATTN_MASK_KEY_PADDING, n_q == n_k
 *   decoder masked self-attn.   ATTN_MASK_CAUSAL (optionally | KEY_PADDING), n_q == n_k
 *   encoder-decoder attention   ATTN_MASK_KEY_PADDING or NONE, n_q != n_k allowed
 *
 * Conventions shared by the entry points below:
 *   - Layouts are contiguous row-major [B, h, n, d] (the per-head layout that a
 *     split_heads reshape produces, csdn blog reimplementation):
 *       q   [B, h, n_q, d_k]    k [B, h, n_k, d_k]    v [B, h, n_k, d_v]
 *       out [B, h, n_q, d_v]    lse [B, h, n_q] (float32, optional)
 *   - Every pointer is a DEVICE pointer owned by the caller (the *_host entry points
 *     excepted). The library allocates no device memory; it neither keeps nor frees
 *     the pointers.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*, NULL
 *     for the legacy default stream) and return before the GPU work finishes.
 *   - scale is used exactly as given; callers normally pass 1/sqrt(d_k) computed
 *     in double and rounded to float.
 *   - key_lens (int32 [B], device memory) gives each batch's number of valid keys
 *     (right padding); key j of batch b is illegal when j >= key_lens[b]. It is
 *     read only when mask_mode has ATTN_MASK_KEY_PADDING and may be NULL otherwise.
 *     Values are clamped to [0, n_k].
 *   - With ATTN_MASK_CAUSAL, key j is illegal for query i when j > i; it requires
 *     n_q == n_k.
 *   - lse[b,h,i] = ln sum_{j legal} exp(scale * q_i . k_j). A query row with no
 *     legal key (key length 0) gets out = 0 and lse = -inf. lse may be NULL.
 *   - Errors are returned as a status; nothing is printed and the process never
 *     exits. A status other than ATTN_OK means nothing was launched.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = -1,     /* null pointer, non-positive size, non-finite scale, bad mask,
                                causal with n_q != n_k, misaligned pointer, size overflow */
  ATTN_ERR_UNSUPPORTED = -2, /* shape this path does not implement (see each entry point) */
  ATTN_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed (no GPU, launch error, ...) */
  ATTN_ERR_TIMEOUT = -4      /* a kernel gave up waiting on an internal barrier (reported by
                                attn_fault_status) */
} attn_status;

enum { ATTN_MASK_NONE = 0, ATTN_MASK_CAUSAL = 1, ATTN_MASK_KEY_PADDING = 2 };

/* attn_bwd flags */
enum { ATTN_BWD_DETERMINISTIC = 1 };

/*
 * attn_fwd -- bf16 inputs and output, fp32 accumulation (sm_103a tensor cores).
 *   q, k, v, out: bf16 (raw 16-bit) arrays, 16-byte aligned.
 *   lse: float32 or NULL.
 *   Supported: d_k == d_v in {64, 128}; any B, h, n_q, n_k >= 1 whose element
 *   counts fit in int32 per head-row index and whose byte strides fit TMA limits.
 *   Otherwise ATTN_ERR_UNSUPPORTED.
 * Numerics: QK^T and PV accumulate in fp32 on the tensor cores; the softmax is the
 * online (running max / running sum) form in fp32 with exp2 and the scale folded
 * in; the probabilities are rounded to bf16 before the PV product; the output is
 * divided by the row sum in fp32 and rounded to bf16 (nearest-even).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
             int B, int h, int n_q, int n_k, int d_k, int d_v, float scale,
             int mask_mode, const int32_t* key_lens, void* stream);

/*
 * attn_weights -- the softmax weights of Eq. (1) themselves (rockcohen.cc "Attention Is
 * All You Need" section 5.1), the second value the pages' scaled_dot_product_attention
 * returns beside the output (csdn blog reimplementation, scaled_dot_product_attention):
 *   w[b, h, i, j] = exp(scale * q_i . k_j - lse_i) for every legal key j of row i
 *   (the mask of attn_fwd), and exactly 0 for the others and for every key of a row
 *   with no legal key (lse_i = -inf).
 * With lse the log-sum-exp that attn_fwd returned for the same q, k, scale, mask_mode
 * and key_lens, each row of legal weights sums to 1 up to that lse's rounding.
 *   q [B, h, n_q, d], k [B, h, n_k, d]: bf16 device arrays, 16-byte aligned.
 *   lse [B, h, n_q]: float32 device array (required).
 *   w [B, h, n_q, n_k]: float32 device array, 16-byte aligned, written in full;
 *           B*h*n_q*n_k floats, owned by the caller.
 *   mask_mode, key_lens, scale and stream as in attn_fwd.
 * Supported: d in {64, 128}; otherwise ATTN_ERR_UNSUPPORTED. The score q_i . k_j
 * accumulates in fp32 on the tensor cores; the exponential is exp2 of the scaled score
 * in log2 units. The matrix is B*h*n_q*n_k floats: this is for inspecting attention
 * (the forward never forms it), and its cost is that write.
 */
int attn_weights(const void* q, const void* k, const float* lse, float* w, int B, int h, int n_q, int n_k, int d,
                 float scale, int mask_mode, const int32_t* key_lens, void* stream);

/*
 * attn_fwd_host_workspace_size -- bytes of device workspace attn_fwd_host needs for
 * this shape and mask (four chunk slots of Q, K, V, out, lse plus the key lengths;
 * the mask enters through the chunk plan). Returns 0 for an invalid shape or mask
 * (d must be 64 or 128). Depends only on the arguments.
 */
size_t attn_fwd_host_workspace_size(int B, int h, int n_q, int n_k, int d, int mask_mode);

/*
 * attn_fwd_host -- attn_fwd for operands that live in HOST memory, the call an
 * application makes when its Q, K, V are not yet on the GPU. Same operation, masks,
 * numerics and results as attn_fwd (bit for bit: the same kernel runs on each chunk).
 *   q, k, v, key_lens: host memory, read by the call;   out, lse: host memory, written.
 *   Page-locked (pinned) host memory is strongly recommended: with pageable memory the
 *   copies are staged by the driver and do not overlap the kernels.
 *   workspace: device scratch of at least attn_fwd_host_workspace_size(B, h, n_q,
 *   n_k, d_k, mask_mode) bytes, 256-byte aligned, owned by the caller.
 * The flattened (b, h) head range is cut into chunks. Chunk c's host-to-device copy,
 * its attention kernel and its device-to-host copy run on the library's own streams
 * (one for each direction, one per slot for the kernels) through a four-slot ring in
 * the workspace, so transfers overlap computation and consecutive kernels overlap
 * each other. Every stream waits for what `stream` had queued before the call, and
 * `stream` waits for all of them. The call is asynchronous: the host buffers must
 * stay valid and unmodified (q, k, v, key_lens) or unread (out, lse) until `stream`
 * reaches this call's end, which includes every copy back; calls made
 * from several host threads are serialised per device. Errors as attn_fwd; a failure
 * after some chunks were queued returns ATTN_ERR_CUDA with those chunks in flight.
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse,
                  int B, int h, int n_q, int n_k, int d_k, int d_v, float scale,
                  int mask_mode, const int32_t* key_lens, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * attn_fwd_local -- restricted (local-window) self-attention, bf16, on the same
 * tensor-core kernel as attn_fwd. The pages propose, for very long sequences,
 * letting each position attend only to positions within a neighbourhood r, which
 * lowers the cost from O(n^2 d) to O(r n d) (csdn blog section 4.3 and "future
 * work"; vlmlib.cn "limitations"). Here r = `window` is a radius: key j is legal
 * for query i only if |i - j| <= window, in addition to whatever mask_mode imposes
 * (ATTN_MASK_CAUSAL makes the window one-sided, i - window <= j <= i;
 * ATTN_MASK_KEY_PADDING as in attn_fwd). Self-attention only: q, k, v, out are
 * [B, h, n, d]. K/V tiles outside every row's window are never loaded.
 * window >= 0 (ATTN_ERR_INVALID otherwise); a window of n or more restricts nothing
 * (|i - j| < n always). Other rules as attn_fwd.
 */
int attn_fwd_local(const void* q, const void* k, const void* v, void* out, float* lse,
                   int B, int h, int n, int d_k, int d_v, float scale, int window,
                   int mask_mode, const int32_t* key_lens, void* stream);

/*
 * attn_fwd_f32 -- float32 inputs and output, float32 arithmetic throughout
 * (CUDA cores). Same semantics and conventions as attn_fwd; pointers 4-byte
 * aligned; 1 <= d_k, d_v <= 256, otherwise ATTN_ERR_UNSUPPORTED.
 */
int attn_fwd_f32(const float* q, const float* k, const float* v, float* out, float* lse,
                 int B, int h, int n_q, int n_k, int d_k, int d_v, float scale,
                 int mask_mode, const int32_t* key_lens, void* stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode needs for
 * this shape (the split-K partial results: fp32 partial outputs, running maxima
 * and sums). Returns 0 for an invalid shape. Depends only on the arguments.
 */
size_t attn_decode_workspace_size(int B, int h, int n_q, int n_max, int d);

/*
 * attn_decode -- one autoregressive decoding step against a key/value cache:
 * n_q new queries per (b, h) attend to the cached keys up to their own position.
 * Generation proceeds one position at a time under the causal mask of decoder
 * self-attention (attention-paper-guide section 05; rockcohen.cc sections 5.3,
 * 6.3); query i of batch b sits at position cache_lens[b] - n_q + i and key j is
 * legal iff j <= cache_lens[b] - n_q + i. The result equals the last n_q rows of
 * causal self-attention over the first cache_lens[b] positions.
 *   q       bf16 [B, h, n_q, d]         k_cache, v_cache  bf16 [B, h, n_max, d]
 *   out     bf16 [B, h, n_q, d]         lse  float [B, h, n_q] or NULL
 *   cache_lens  int32 [B], device, each in [0, n_max] (a value outside is clamped to
 *           that range before the query positions are placed). A query whose
 *           position is negative (cache_lens[b] < n_q) has no legal key: out = 0,
 *           lse = -inf.
 *   workspace   device scratch of at least attn_decode_workspace_size(...) bytes,
 *           16-byte aligned, owned by the caller; its contents on entry do not
 *           matter and on return are undefined. Two calls that run at the same time
 *           must not share a workspace.
 * Supported: 1 <= n_q <= 16, d in {64, 128}, B*h <= 65535. Pointers 16-byte
 * aligned. fp32 arithmetic throughout (scores, exp2, sums, P.V); the output is
 * rounded to bf16 once. Asynchronous on `stream`; two kernels are launched (one
 * warp per cache chunk for n_q = 1, one block per cache range for n_q > 1; then the
 * merge).
 */
int attn_decode(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                int B, int h, int n_q, int n_max, int d, float scale,
                const int32_t* cache_lens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device memory.
 * (An addition of this library; the paper has no counterpart.)
 * Some callers have no way to obtain device scratch: plug-ins whose host framework
 * owns every device buffer and hands a kernel only its inputs and outputs,
 * latency-critical serving loops that must not enter the allocator (cudaMalloc and
 * cudaFree can synchronise the whole device), and programs that fix their device
 * memory at start-up. This entry point takes the same arguments as attn_decode minus
 * the workspace and allocates nothing: no cudaMalloc, cudaFree or allocating
 * library call. Its scratch is a static buffer of ATTN_DECODE_NOALLOC_MAX_BYTES
 * inside the library's device image, present on every GPU that loads the library
 * until the process exits.
 *   - The first call on a device looks up the buffer's device address (with that
 *     device current) and keeps it; make that first call before any stream capture.
 *     A cudaDeviceReset after that first call is not supported: the kept address
 *     belongs to the context the reset destroyed.
 *   - Every call on a device shares the one buffer, which keeps the last call's
 *     contents (the kernels write every slot before reading it, an abandoned range
 *     included, so nothing needs clearing). Calls whose GPU work overlaps -- on
 *     different streams, or from several host threads -- race on it: order them,
 *     e.g. on one stream.
 *   - A shape whose workspace (attn_decode_workspace_size) exceeds
 *     ATTN_DECODE_NOALLOC_MAX_BYTES returns ATTN_ERR_UNSUPPORTED and launches
 *     nothing; use attn_decode with a caller workspace for it.
 * Results are those of attn_decode on the same inputs.
 */
#define ATTN_DECODE_NOALLOC_MAX_BYTES (4u << 20)
int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                        int B, int h, int n_q, int n_max, int d, float scale,
                        const int32_t* cache_lens, void* stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs for this shape,
 * head size d and flags: two fp32 per query row (-lse_i log2(e) and -D_i below),
 * padded to whole 128-row tiles, plus, for the fused schedule (d = 64 without
 * ATTN_BWD_DETERMINISTIC), an fp32 dQ accumulator of B*h*n_q*64 floats. Returns 0 for
 * an invalid shape, head size or flag.
 */
size_t attn_bwd_workspace_size(int B, int h, int n_q, int d, int flags);

/*
 * attn_bwd -- gradients of attn_fwd with respect to q, k and v, given the gradient
 * dout of the output. Training the model by gradient descent needs them
 * (attention-paper-guide section 05; vlmlib.cn "training"). With P the softmax
 * weights of Eq. (1) (rockcohen.cc section 5.1) recomputed from lse,
 * P[i,j] = exp(scale * q_i . k_j - lse_i) on legal pairs and 0 on illegal ones:
 *   dv_j = sum_i P[i,j] dout_i
 *   dP[i,j] = dout_i . v_j,  D_i = dout_i . out_i,  dS[i,j] = P[i,j] (dP[i,j] - D_i)
 *   dq_i = scale sum_j dS[i,j] k_j,      dk_j = scale sum_i dS[i,j] q_i
 *   q, k, v, out, dout: bf16 as in attn_fwd (out and lse are those attn_fwd returned
 *           for the same q, k, v, scale, mask_mode and key_lens; lse is required)
 *   dq [B, h, n_q, d], dk, dv [B, h, n_k, d]: bf16, written in full (a key that no
 *           query may see gets dk = dv = 0; a query with no legal key gets dq = 0)
 *   flags: 0, or ATTN_BWD_DETERMINISTIC (any other bit: ATTN_ERR_INVALID).
 *   workspace: device scratch of at least attn_bwd_workspace_size(B, h, n_q, d_k,
 *           flags) bytes, 16-byte aligned, owned by the caller, contents undefined on
 *           return; concurrent calls must not share it.
 * mask_mode and key_lens as in attn_fwd. Supported: d_k == d_v in {64, 128}.
 * Numerics: S and dP accumulate in fp32 on the tensor cores; P and dS are rounded to
 * bf16 before the three products that consume them, which accumulate in fp32; D_i
 * is accumulated in fp32 from the bf16 out and dout; results are rounded to bf16
 * once. Schedules:
 *   - fused (d = 64, flags = 0): each of the five products is computed once; the
 *     partial dQ of every 128-key tile is added into the fp32 workspace accumulator
 *     with TMA reduce-adds, whose order varies, so the last bits of dq can differ
 *     from run to run (dk and dv are deterministic). A memset and three kernels.
 *   - deterministic (d = 128, or ATTN_BWD_DETERMINISTIC): a dK/dV kernel and a dQ
 *     kernel that recomputes S and dP (seven products), no atomics: bit-identical
 *     results on every run. Three kernels.
 * All launches are on `stream`.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int h, int n_q, int n_k, int d_k, int d_v, float scale,
             int mask_mode, const int32_t* key_lens, int flags, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * attn_bwd_local -- gradients of attn_fwd_local (restricted self-attention: key j is
 * legal for query i only if |i - j| <= window, together with mask_mode; vlmlib.cn
 * "restricted self-attention"), exactly as attn_bwd computes them for
 * attn_fwd: the same definitions, numerics, schedules, flags and workspace
 * (attn_bwd_workspace_size(B, h, n, d_k, flags)), with n_q = n_k = n and the window
 * entering P's mask. out and lse are those attn_fwd_local returned for the same
 * q, k, v, scale, window, mask_mode and key_lens. window < 0: ATTN_ERR_INVALID; a
 * window of n or more is the unrestricted mask (as in attn_fwd_local).
 * Key tiles no query of a query tile may see, and query tiles outside a key tile's
 * window, are skipped; every dq, dk, dv element is still written.
 */
int attn_bwd_local(const void* q, const void* k, const void* v, const void* out, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int h, int n, int d_k, int d_v,
                   float scale, int window, int mask_mode, const int32_t* key_lens, int flags, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * attn_bwd_host_workspace_size -- bytes of device workspace attn_bwd_host needs for
 * this shape, head size, mask and flags (four chunk slots of the nine per-head tensors
 * and their gradient workspace, plus the key lengths). Returns 0 for an invalid shape,
 * head size, mask or flag. Depends only on the arguments.
 */
size_t attn_bwd_host_workspace_size(int B, int h, int n_q, int n_k, int d, int mask_mode, int flags);

/*
 * attn_bwd_host -- attn_bwd for operands that live in HOST memory (a training step
 * whose tensors are on the host). Same gradients, schedules, flags and numerics as
 * attn_bwd: the same kernels run on each chunk of heads (dk and dv bit-identical to
 * attn_bwd on the same data; dq as well with ATTN_BWD_DETERMINISTIC).
 *   q, k, v, out, dout, lse, key_lens: host memory, read;   dq, dk, dv: host memory,
 *   written. Page-locked (pinned) host memory is strongly recommended.
 *   workspace: device scratch of at least attn_bwd_host_workspace_size(B, h, n_q, n_k,
 *   d_k, mask_mode, flags) bytes, 256-byte aligned, owned by the caller.
 * The flattened (b, h) head range is cut into chunks whose host-to-device copies,
 * gradient kernels and device-to-host copies run on the library's own streams through
 * a four-slot ring in the workspace, as in attn_fwd_host. The call is asynchronous on
 * `stream` and ordered with it at both ends; the host buffers must stay valid (and the
 * inputs unmodified) until `stream` reaches the end of the call. Errors as attn_bwd.
 */
int attn_bwd_host(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, int B, int h, int n_q, int n_k, int d_k, int d_v, float scale,
                  int mask_mode, const int32_t* key_lens, int flags, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * attn_linear -- one linear projection of the multi-head layer, bf16 in and out:
 *   y[M, N] = x[M, K] w[K, N] + bias[N]
 * The layer projects queries, keys and values with per-head matrices W_i^Q, W_i^K,
 * W_i^V and the concatenated heads with W^O (vlmlib.cn paper summary, "multi-head
 * attention"; the csdn blog's MultiHeadAttention uses nn.Linear layers with biases);
 * placing the h per-head matrices side by side makes each projection this product.
 *   x  [M, K], w [K, N] (the paper's x W orientation; an nn.Linear weight is the
 *      transpose), y [M, N]: row-major bf16, 16-byte aligned, caller-owned device memory
 *   bias [N] bf16, 16-byte aligned, or NULL for none.
 * Supported: N and K multiples of 8 (16-byte rows); otherwise ATTN_ERR_UNSUPPORTED.
 * Numerics: the products accumulate in fp32 on the sm_103a tensor cores (tcgen05,
 * operands staged by TMA); the bias is added in fp32 and the sum rounded to bf16
 * (nearest-even) once. One launch on `stream`; x and y must not overlap.
 */
int attn_linear(const void* x, const void* w, const void* bias, void* y, int M, int N, int K, void* stream);

/*
 * attn_mha_workspace_size -- bytes of device workspace attn_mha_fwd needs: the
 * projected Q', K', V' and the concatenated heads (bf16, each padded to 256 bytes).
 * Returns 0 for an invalid or unsupported shape.
 */
size_t attn_mha_workspace_size(int B, int n_q, int n_k, int d_model, int h, int d);

/*
 * attn_mha_fwd -- the multi-head attention layer (vlmlib.cn "multi-head attention":
 * MultiHead(Q,K,V) = Concat(head_1..head_h) W^O, head_i = Attention(Q W_i^Q, K W_i^K,
 * V W_i^V); the csdn blog's MultiHeadAttention with its linear projections, split_heads
 * and concatenation), bf16 in and out:
 *   Q' = x_q W^Q + b_Q, K' = x_kv W^K + b_K, V' = x_kv W^V + b_V     [B, n, h*d]
 *   A  = attn_fwd(Q', K', V') per head, heads concatenated          [B, n_q, h*d]
 *   out = A W^O + b_O                                                [B, n_q, d_model]
 *   x_q  [B, n_q, d_model], x_kv [B, n_k, d_model] (pass x_q twice for self-attention)
 *   w_q, w_k, w_v [d_model, h*d], w_o [h*d, d_model]: row-major, the paper's x W
 *           orientation (an nn.Linear weight is the transpose); head i uses columns
 *           i*d .. i*d + d - 1 of W^Q, W^K, W^V and rows i*d .. of W^O
 *   b_q, b_k, b_v [h*d], b_o [d_model]: bf16 or NULL for no bias
 *   out  [B, n_q, d_model] bf16
 *   mask_mode, key_lens, scale: as attn_fwd (scale is normally 1/sqrt(d)).
 *   workspace: device scratch of at least attn_mha_workspace_size(...) bytes, 16-byte
 *           aligned, owned by the caller, contents undefined on return; concurrent
 *           calls must not share it.
 * Supported: d_k == d_v in {64, 128}, d_model a multiple of 8; every pointer 16-byte
 * aligned. The four projections have the numerics of attn_linear (fp32 accumulation
 * on the tensor cores, bias added in fp32, one rounding to bf16); the three input
 * projections run as one launch of the projection kernel. The attention is the
 * attn_fwd kernel reading Q', K', V' and writing A in their [B, n, h*d] layout, so
 * splitting and concatenating the heads moves no data. Three launches on `stream`.
 */
int attn_mha_fwd(const void* x_q, const void* x_kv, const void* w_q, const void* b_q, const void* w_k,
                 const void* b_k, const void* w_v, const void* b_v, const void* w_o, const void* b_o, void* out,
                 int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v, float scale, int mask_mode,
                 const int32_t* key_lens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fault_status -- synchronises `stream`, then reports whether any kernel of
 * this library on the current device gave up waiting on one of its internal
 * barriers since the last clear (each such wait is bounded in time; a kernel that
 * gives up writes no further output and returns). Returns ATTN_OK,
 * ATTN_ERR_TIMEOUT, or ATTN_ERR_CUDA. If `clear` is non-zero the record is reset.
 * `fault_code` (may be NULL) receives the raw record: bit 0 producer, bit 1 MMA
 * issuer, bit 2 softmax, bit 3 epilogue (attn_fwd), bit 4 decode copy (attn_decode),
 * bit 5 gradient kernels (attn_bwd), bit 6 attn_fwd found its shared memory not
 * 1024-byte aligned (it then writes nothing), bit 7 projection kernel (attn_linear,
 * attn_mha_fwd), bit 8 attn_weights.
 */
int attn_fault_status(void* stream, int clear, uint32_t* fault_code);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_GB300_H */
