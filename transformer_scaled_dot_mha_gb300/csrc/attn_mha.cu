// attn_mha.cu -- the multi-head attention layer around the attention kernel:
//   Q' = x_q W^Q + b_Q,  K' = x_kv W^K + b_K,  V' = x_kv W^V + b_V      [B, n, h*d]
//   A  = Attention(Q', K', V') per head, written concatenated          [B, n_q, h*d]
//   Y  = A W^O + b_O                                                    [B, n_q, d_model]
// (vlmlib.cn "multi-head attention": MultiHead = Concat(head_1..head_h) W^O with
// head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V); the csdn blog's MultiHeadAttention.)
//
// Three launches on the caller's stream: the three input projections as one launch
// of the projection kernel (attn_linear.cu; for self-attention its tile order lets
// the three projections share the x rows they read through L2), the attention
// kernel, and the output projection. split_heads and the concatenation cost no
// copies: the attention kernel reads Q', K', V' and writes A in their [B, n, h*d]
// layout through its heads-interleaved tensor maps (head i = columns i*d .. i*d+d-1).
// All three allow programmatic dependent launch, so each one's set-up (barriers, TMEM,
// tensor maps) overlaps the end of the one before it.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

}  // namespace

size_t mha_workspace_bytes(int B, int n_q, int n_k, int H, int d) {
  const size_t hd = (size_t)H * d * 2;
  return align_up((size_t)B * n_q * hd) * 2 + align_up((size_t)B * n_k * hd) * 2;
}

int launch_attn_mha(const MhaArgs& a, PFN_encodeTiled enc, void* workspace) {
  const size_t hd = (size_t)a.H * a.d * 2;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* qp = base;
  uint8_t* kp = qp + align_up((size_t)a.B * a.n_q * hd);
  uint8_t* vp = kp + align_up((size_t)a.B * a.n_k * hd);
  uint8_t* ao = vp + align_up((size_t)a.B * a.n_k * hd);
  const int Mq = a.B * a.n_q, Mk = a.B * a.n_k, HD = a.H * a.d;
  const LinearJob in[3] = {{a.x_q, a.w_q, a.b_q, qp, Mq, HD, a.d_model},
                           {a.x_kv, a.w_k, a.b_k, kp, Mk, HD, a.d_model},
                           {a.x_kv, a.w_v, a.b_v, vp, Mk, HD, a.d_model}};
  int st;
  if ((st = launch_linear(in, 3, enc, a.stream)) != ATTN_OK) return st;
  TcArgs t{qp, kp, vp, ao, nullptr, a.B, a.H, a.n_q, a.n_k, a.d, a.scale, a.mask_mode, a.key_lens, a.stream, -1};
  t.heads_interleaved = 1;
  if ((st = launch_attn_tc(t, enc)) != ATTN_OK) return st;
  const LinearJob outj = {ao, a.w_o, a.b_o, a.out, Mq, a.d_model, HD};
  return launch_linear(&outj, 1, enc, a.stream);
}

}  // namespace attn
