// attn_bwd_host.cu -- attn_bwd for operands in host memory: the gradient step of a
// training loop whose tensors live on the host. Heads are independent in the
// gradients as in the forward, so the flattened (b, h) range is cut into chunks that
// move through a four-slot device ring on three kinds of stream, as attn_fwd_host's:
//
//   h2d stream:        Q, K, V, O, dO, lse of chunk c -> slot s = c % kSlots (event in_c)
//   slot s's stream:   wait in_c; attn_bwd on the slot                         (event done_c)
//   d2h stream:        wait done_c; dQ, dK, dV of chunk c -> host              (event out_c)
//
// The chunk plan is plan_chunks' with the gradient's copy bytes and kernel time. A
// chunk's attn_bwd calls cover its heads in at most three rectangles (head_rect), each
// with its own part of the slot's gradient workspace (that workspace is linear in the
// number of heads), so each call is exactly attn_bwd on those heads.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 4;
constexpr size_t kAlign = 256;
constexpr double kBwdFlopsPerUs = 0.65e9;  // the gradient kernels' rate, only to choose the plan

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct BwdHostState {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[kSlots] = {};
  cudaEvent_t start = nullptr, in[kSlots], done[kSlots], out[kSlots];
};

BwdHostState g_bwd_host[kMaxDevices];

int ensure_streams(BwdHostState& st) {
  if (st.ready) return ATTN_OK;
  if (cudaStreamCreateWithFlags(&st.h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&st.d2h, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&st.start, cudaEventDisableTiming) != cudaSuccess)
    return ATTN_ERR_CUDA;
  for (int s = 0; s < kSlots; ++s)
    if (cudaStreamCreateWithFlags(&st.comp[s], cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.in[s], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.done[s], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.out[s], cudaEventDisableTiming) != cudaSuccess)
      return ATTN_ERR_CUDA;
  st.ready = true;
  return ATTN_OK;
}

// Per-head bytes: q-shaped tensors (Q, O, dO, dQ), k-shaped ones (K, V, dK, dV), lse,
// and the gradient workspace of one head.
struct BwdHeadBytes {
  size_t q, kv, l, ws;
};

BwdHeadBytes bwd_head_bytes(int n_q, int n_k, int d, int flags) {
  return {(size_t)n_q * d * 2, (size_t)n_k * d * 2, (size_t)n_q * 4, bwd_workspace_bytes(1, 1, n_q, d, flags)};
}

// Slot layout for `heads` heads: Q, O, dO, K, V, lse, dQ, dK, dV, workspace.
struct SlotPtrs {
  uint8_t *q, *o, *dout, *k, *v, *lse, *dq, *dk, *dv, *ws;
};

size_t slot_bytes(long long heads, const BwdHeadBytes& hb) {
  return 4 * align_up(heads * hb.q) + 4 * align_up(heads * hb.kv) + align_up(heads * hb.l) + align_up(heads * hb.ws);
}

SlotPtrs slot_ptrs(uint8_t* base, long long heads, const BwdHeadBytes& hb) {
  SlotPtrs p;
  const size_t q = align_up(heads * hb.q), kv = align_up(heads * hb.kv);
  p.q = base;
  p.o = p.q + q;
  p.dout = p.o + q;
  p.k = p.dout + q;
  p.v = p.k + kv;
  p.lse = p.v + kv;
  p.dq = p.lse + align_up(heads * hb.l);
  p.dk = p.dq + q;
  p.dv = p.dk + kv;
  p.ws = p.dv + kv;
  return p;
}

int bwd_chunk_plan(int B, int H, int n_q, int n_k, int d, int mask_mode, const BwdHeadBytes& hb, long long* sizes) {
  const bool causal = (mask_mode & ATTN_MASK_CAUSAL) != 0;
  const double pairs = causal ? 0.5 * n_q * (n_q + 1.0) : (double)n_q * n_k;
  const size_t in_bytes = 3 * hb.q + 2 * hb.kv + hb.l, out_bytes = hb.q + 2 * hb.kv;
  return plan_chunks((long long)B * H, in_bytes, out_bytes, 10.0 * d * pairs / kBwdFlopsPerUs, sizes);
}

void slot_caps(const long long* sizes, int n, long long caps[kSlots]) {
  for (int s = 0; s < kSlots; ++s) caps[s] = 0;
  for (int c = 0; c < n; ++c)
    if (sizes[c] > caps[c % kSlots]) caps[c % kSlots] = sizes[c];
}

}  // namespace

size_t bwd_host_workspace_bytes(int B, int H, int n_q, int n_k, int d, int mask_mode, int flags) {
  const BwdHeadBytes hb = bwd_head_bytes(n_q, n_k, d, flags);
  long long sizes[kMaxHostChunks], caps[kSlots];
  slot_caps(sizes, bwd_chunk_plan(B, H, n_q, n_k, d, mask_mode, hb, sizes), caps);
  size_t total = align_up((size_t)B * 4);  // key lengths
  for (int s = 0; s < kSlots; ++s) total += slot_bytes(caps[s], hb);
  return total;
}

int launch_attn_bwd_host(const BwdArgs& a, PFN_encodeTiled enc, void* workspace) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  BwdHostState& st = g_bwd_host[dev];
  std::lock_guard<std::mutex> lock(st.mu);
  int rc = ensure_streams(st);
  if (rc != ATTN_OK) return rc;
  const BwdHeadBytes hb = bwd_head_bytes(a.n_q, a.n_k, a.d, a.flags);
  long long sizes[kMaxHostChunks], caps[kSlots];
  const int n_chunks = bwd_chunk_plan(a.B, a.H, a.n_q, a.n_k, a.d, a.mask_mode, hb, sizes);
  slot_caps(sizes, n_chunks, caps);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int32_t* d_lens = reinterpret_cast<int32_t*>(base);
  SlotPtrs slot[kSlots];
  size_t off = align_up((size_t)a.B * 4);
  for (int s = 0; s < kSlots; ++s) {
    slot[s] = slot_ptrs(base + off, caps[s], hb);
    off += slot_bytes(caps[s], hb);
  }
  const bool padding = (a.mask_mode & ATTN_MASK_KEY_PADDING) != 0;
  cudaStream_t cs = a.stream;
  // the previous call's last copies back must be done before slots are reused
  for (int s = 0; s < kSlots; ++s)
    if (cudaStreamWaitEvent(st.h2d, st.out[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
  // anything the caller queued before this call comes first
  if (cudaEventRecord(st.start, cs) != cudaSuccess || cudaStreamWaitEvent(st.h2d, st.start, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (padding && cudaMemcpyAsync(d_lens, a.key_lens, (size_t)a.B * 4, cudaMemcpyHostToDevice, st.h2d) != cudaSuccess)
    return ATTN_ERR_CUDA;
  auto h2d = [&](void* dst, const void* src, long long f0, size_t per, long long nh) {
    return cudaMemcpyAsync(dst, static_cast<const uint8_t*>(src) + f0 * per, nh * per, cudaMemcpyHostToDevice,
                           st.h2d) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, long long f0, size_t per, long long nh) {
    return cudaMemcpyAsync(static_cast<uint8_t*>(dst) + f0 * per, src, nh * per, cudaMemcpyDeviceToHost,
                           st.d2h) == cudaSuccess;
  };
  long long f0 = 0;  // first flattened head of the chunk
  for (int c = 0; c < n_chunks; ++c) {
    const long long nh = sizes[c], f1 = f0 + nh;
    const int s = c % kSlots;
    const SlotPtrs& sp = slot[s];
    if (c >= kSlots && cudaStreamWaitEvent(st.h2d, st.out[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
    if (!h2d(sp.q, a.q, f0, hb.q, nh) || !h2d(sp.k, a.k, f0, hb.kv, nh) || !h2d(sp.v, a.v, f0, hb.kv, nh) ||
        !h2d(sp.o, a.out, f0, hb.q, nh) || !h2d(sp.dout, a.dout, f0, hb.q, nh) || !h2d(sp.lse, a.lse, f0, hb.l, nh) ||
        cudaEventRecord(st.in[s], st.h2d) != cudaSuccess ||
        cudaStreamWaitEvent(st.comp[s], st.in[s], 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    for (long long f = f0; f < f1;) {
      int b, pb, ph;
      head_rect(f, f1, a.H, b, pb, ph);
      const long long r = f - f0;  // heads into the slot
      BwdArgs t{sp.q + r * hb.q, sp.k + r * hb.kv, sp.v + r * hb.kv, sp.o + r * hb.q, sp.dout + r * hb.q,
                reinterpret_cast<const float*>(sp.lse + r * hb.l), sp.dq + r * hb.q, sp.dk + r * hb.kv,
                sp.dv + r * hb.kv, pb, ph, a.n_q, a.n_k, a.d, a.scale, a.mask_mode,
                padding ? d_lens + b : nullptr, st.comp[s], a.flags};
      if ((rc = launch_attn_bwd(t, enc, sp.ws + r * hb.ws)) != ATTN_OK) return rc;
      f += (long long)pb * ph;
    }
    if (cudaEventRecord(st.done[s], st.comp[s]) != cudaSuccess ||
        cudaStreamWaitEvent(st.d2h, st.done[s], 0) != cudaSuccess || !d2h(a.dq, sp.dq, f0, hb.q, nh) ||
        !d2h(a.dk, sp.dk, f0, hb.kv, nh) || !d2h(a.dv, sp.dv, f0, hb.kv, nh) ||
        cudaEventRecord(st.out[s], st.d2h) != cudaSuccess)
      return ATTN_ERR_CUDA;
    f0 = f1;
  }
  // the caller's stream is complete only when every gradient is back on the host
  for (int s = 0; s < kSlots && s < n_chunks; ++s)
    if (cudaStreamWaitEvent(cs, st.out[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn
