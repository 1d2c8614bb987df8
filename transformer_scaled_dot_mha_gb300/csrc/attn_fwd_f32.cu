// attn_fwd_f32.cu -- float32 scaled dot-product attention forward on the CUDA
// cores, for inputs that stay in float32 (any 1 <= d_k, d_v <= 256).
//
// Eq. (1), softmax(Q K^T / sqrt(d_k)) V ("Attention Is All You Need",
// rockcohen.cc section 5.1), with -inf at illegal connections (sections 5.3,
// 6.3). One warp owns one query row: lane x scores key j0 + x of each 32-key
// block, the block maximum and sum come from warp shuffles, and the running
// output (lane x holds dimensions x, x+32, ...) is rescaled whenever the running
// maximum moves (online softmax). All arithmetic is float32 with accurate expf /
// logf and IEEE division.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int WARPS = 4;
constexpr int MAXD = 256;

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;
  const int32_t* key_lens;
  int H, n_q, n_k, d_k, d_v, mask_mode;
  long long rows;  // B * H * n_q
  float scale;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(WARPS * 32) attn_fwd_f32_kernel(const F32Params p) {
  __shared__ float q_s[WARPS][MAXD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * WARPS + warp;
  if (row >= p.rows) return;  // uniform per warp
  const long long bh = row / p.n_q;
  const int i = (int)(row % p.n_q);
  const int b = (int)(bh / p.H);
  int lim = p.n_k;  // keys [0, lim) are legal for this row
  if (p.mask_mode & 2) lim = min(lim, max(p.key_lens[b], 0));
  if (p.mask_mode & 1) lim = min(lim, i + 1);

  const float* qrow = p.q + row * p.d_k;
  for (int t = lane; t < p.d_k; t += 32) q_s[warp][t] = qrow[t];
  __syncwarp();
  const float* kb = p.k + bh * (long long)p.n_k * p.d_k;
  const float* vb = p.v + bh * (long long)p.n_k * p.d_v;

  float acc[MAXD / 32];
#pragma unroll
  for (int u = 0; u < MAXD / 32; ++u) acc[u] = 0.0f;
  float m = -INFINITY, l = 0.0f;

  for (int j0 = 0; j0 < lim; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < lim) {
      const float* krow = kb + (long long)j * p.d_k;
      float dot = 0.0f;
      for (int t = 0; t < p.d_k; ++t) dot = fmaf(q_s[warp][t], krow[t], dot);
      s = dot * p.scale;
    }
    const float m_new = fmaxf(m, warp_max(s));  // finite: key j0 is legal
    const float alpha = expf(m - m_new);        // 0 on the first block
    const float pj = (j < lim) ? expf(s - m_new) : 0.0f;
    l = l * alpha + warp_sum(pj);
#pragma unroll
    for (int u = 0; u < MAXD / 32; ++u) acc[u] *= alpha;
    const int cnt = min(32, lim - j0);
    for (int jj = 0; jj < cnt; ++jj) {
      const float w = __shfl_sync(0xffffffffu, pj, jj);
      const float* vrow = vb + (long long)(j0 + jj) * p.d_v;
#pragma unroll
      for (int u = 0; u < MAXD / 32; ++u) {
        const int t = lane + 32 * u;
        if (t < p.d_v) acc[u] = fmaf(w, vrow[t], acc[u]);
      }
    }
    m = m_new;
  }

  float* orow = p.out + row * p.d_v;
#pragma unroll
  for (int u = 0; u < MAXD / 32; ++u) {
    const int t = lane + 32 * u;
    if (t < p.d_v) orow[t] = (l > 0.0f) ? acc[u] / l : 0.0f;
  }
  if (lane == 0 && p.lse) p.lse[row] = (l > 0.0f) ? m + logf(l) : -INFINITY;
}

}  // namespace

int launch_attn_f32(const F32Args& a) {
  F32Params p;
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.out = a.out;
  p.lse = a.lse;
  p.key_lens = a.key_lens;
  p.H = a.H;
  p.n_q = a.n_q;
  p.n_k = a.n_k;
  p.d_k = a.d_k;
  p.d_v = a.d_v;
  p.mask_mode = a.mask_mode;
  p.rows = (long long)a.B * a.H * a.n_q;
  p.scale = a.scale;
  if (a.d_k > MAXD || a.d_v > MAXD) return ATTN_ERR_UNSUPPORTED;
  const long long blocks = (p.rows + WARPS - 1) / WARPS;
  if (blocks > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  attn_fwd_f32_kernel<<<(unsigned)blocks, WARPS * 32, 0, a.stream>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
