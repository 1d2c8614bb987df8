// attn_host.cu -- attn_fwd for operands in host memory. The flattened (b, h) range
// of heads is cut into chunks whose host-to-device copies, attention kernels and
// device-to-host copies run on their own streams, so that the transfers, which bound
// this call, overlap the computation instead of adding to it.
//
//   h2d stream:        Q, K, V of chunk c  -> ring slot s = c % kSlots   (event in_c)
//   slot s's stream:   wait in_c; attn_fwd on the slot                    (event done_c)
//   d2h stream:        wait done_c; O (and lse) of chunk c -> host       (event out_c)
//
// When the copies bound the call, chunk sizes ramp up from a minimum and then fall by
// halves: no kernel can start before the first chunk has arrived, and the last
// chunk's kernel and copy back overlap no transfer, so both ends are small. When the
// kernels take about as long as the copies, the chunks are equal and small enough
// that consecutive kernels, each on its slot's own stream, interleave and keep the
// SMs busy. The h2d stream waits out_{c - kSlots}
// before it refills a slot; at the end the caller's stream waits every copy back, so
// the call is ordered on `stream` like any other entry point.
//
// A chunk is a contiguous range of the [B, h] head index, so each tensor moves in one
// copy; its kernel launches cover the range in at most three rectangles (the rest of
// one batch, whole batches, the start of one batch), each with its batches' key
// lengths. The kernel variant is chosen for the whole problem, so the results equal
// attn_fwd's on the same data bit for bit.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 4;
constexpr int kMaxChunks = kMaxHostChunks;
constexpr size_t kAlign = 256;
constexpr size_t kMinChunkBytes = size_t(8) << 20;  // host-to-device bytes of the smallest chunk
// Rates used only to choose the chunk plan (results do not depend on it): the
// attention kernel's throughput on long sequences and the host link's copy rate.
constexpr double kKernelFlopsPerUs = 1.0e9;  // about 1 PFLOP/s
constexpr double kLinkBytesPerUs = 2.0e5;    // about 200 GB/s

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct HostState {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[kSlots] = {};
  cudaEvent_t start = nullptr, in[kSlots], done[kSlots], out[kSlots];
};

HostState g_host[kMaxDevices];

int ensure_streams(HostState& st) {
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

// Per-head byte counts of one slot's buffers.
struct HeadBytes {
  size_t q, kv, o, l;
};

HeadBytes head_bytes(int n_q, int n_k, int d) {
  return {(size_t)n_q * d * 2, (size_t)n_k * d * 2, (size_t)n_q * d * 2, (size_t)n_q * 4};
}

// The forward's chunk plan (see plan_chunks).
int chunk_plan(long long bh, const HeadBytes& hb, int n_q, int n_k, int d, bool causal,
               long long sizes[kMaxChunks]) {
  const double pairs = causal ? 0.5 * n_q * (n_q + 1.0) : (double)n_q * n_k;
  return plan_chunks(bh, hb.q + 2 * hb.kv, hb.o, 4.0 * d * pairs / kKernelFlopsPerUs, sizes);
}

// Bytes of a slot holding `heads` heads: q, k, v, out, lse, each 256-byte aligned.
size_t slot_bytes(long long heads, const HeadBytes& hb) {
  return align_up(heads * hb.q) + 2 * align_up(heads * hb.kv) + align_up(heads * hb.o) + align_up(heads * hb.l);
}

// Heads each slot must hold: the largest chunk that uses it (chunk c uses c % kSlots).
void slot_caps(const long long* sizes, int n, long long caps[kSlots]) {
  for (int s = 0; s < kSlots; ++s) caps[s] = 0;
  for (int c = 0; c < n; ++c)
    if (sizes[c] > caps[c % kSlots]) caps[c % kSlots] = sizes[c];
}

}  // namespace

// Chunk sizes (in heads) for bh heads of in_bytes copied in and out_bytes copied back
// each, whose kernel takes about kernel_us: every chunk at least kMinChunkBytes of
// input, the remainder merged into the last chunk when it would fall below that.
//  - Transfer-bound (a head's kernel time well under its copy time, e.g. causal or
//    short sequences): a ramp that starts at the minimum and doubles but never takes
//    more than half of what is left, so the sizes rise and then fall by halves. Only
//    the first copy and the last kernel + copy back overlap nothing, so both are small.
//  - Otherwise: eight equal chunks, each a fraction of a wave of CTAs, whose kernels
//    interleave on the slot streams and keep every SM busy.
int plan_chunks(long long bh, size_t in_bytes, size_t out_bytes, double kernel_us, long long* sizes) {
  long long min_heads = (long long)((kMinChunkBytes + in_bytes - 1) / in_bytes);
  if (min_heads < 1) min_heads = 1;
  const double copy_us = (double)(in_bytes + out_bytes) / kLinkBytesPerUs;
  const bool ramped = kernel_us < 0.6 * copy_us;
  int n = 0;
  long long left = bh, ramp = min_heads;
  while (left > 0) {
    long long c = ramped ? (left + 1) / 2 : (bh + 7) / 8;
    if (ramped && c > ramp) c = ramp;
    if (c < min_heads) c = min_heads;
    if (left - c < min_heads || n == kMaxHostChunks - 1) c = left;
    sizes[n++] = c;
    left -= c;
    if (ramp < bh) ramp *= 2;
  }
  return n;
}

size_t host_workspace_bytes(int B, int H, int n_q, int n_k, int d, int mask_mode) {
  const HeadBytes hb = head_bytes(n_q, n_k, d);
  long long sizes[kMaxChunks];
  long long caps[kSlots];
  slot_caps(sizes, chunk_plan((long long)B * H, hb, n_q, n_k, d, (mask_mode & ATTN_MASK_CAUSAL) != 0, sizes), caps);
  size_t total = align_up((size_t)B * 4);  // key lengths
  for (int s = 0; s < kSlots; ++s) total += slot_bytes(caps[s], hb);
  return total;
}

int launch_attn_host(const TcArgs& a, PFN_encodeTiled enc, void* workspace) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  HostState& st = g_host[dev];
  std::lock_guard<std::mutex> lock(st.mu);
  int rc = ensure_streams(st);
  if (rc != ATTN_OK) return rc;
  const HeadBytes hb = head_bytes(a.n_q, a.n_k, a.d);
  long long sizes[kMaxChunks];
  const int n_chunks =
      chunk_plan((long long)a.B * a.H, hb, a.n_q, a.n_k, a.d, (a.mask_mode & ATTN_MASK_CAUSAL) != 0, sizes);
  long long caps[kSlots];
  slot_caps(sizes, n_chunks, caps);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int32_t* d_lens = reinterpret_cast<int32_t*>(base);
  uint8_t* slot_base[kSlots] = {};
  size_t off = align_up((size_t)a.B * 4);
  for (int s = 0; s < kSlots; ++s) {
    slot_base[s] = base + off;
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
  const uint8_t* hq = static_cast<const uint8_t*>(a.q);
  const uint8_t* hk = static_cast<const uint8_t*>(a.k);
  const uint8_t* hv = static_cast<const uint8_t*>(a.v);
  uint8_t* ho = static_cast<uint8_t*>(a.out);
  long long f0 = 0;  // first flattened head of the chunk
  for (int c = 0; c < n_chunks; ++c) {
    const long long nh = sizes[c], f1 = f0 + nh;
    const int s = c % kSlots;
    uint8_t* sq = slot_base[s];
    uint8_t* sk = sq + align_up(caps[s] * hb.q);
    uint8_t* sv = sk + align_up(caps[s] * hb.kv);
    uint8_t* so = sv + align_up(caps[s] * hb.kv);
    uint8_t* sl = so + align_up(caps[s] * hb.o);
    if (c >= kSlots && cudaStreamWaitEvent(st.h2d, st.out[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpyAsync(sq, hq + f0 * hb.q, nh * hb.q, cudaMemcpyHostToDevice, st.h2d) != cudaSuccess ||
        cudaMemcpyAsync(sk, hk + f0 * hb.kv, nh * hb.kv, cudaMemcpyHostToDevice, st.h2d) != cudaSuccess ||
        cudaMemcpyAsync(sv, hv + f0 * hb.kv, nh * hb.kv, cudaMemcpyHostToDevice, st.h2d) != cudaSuccess ||
        cudaEventRecord(st.in[s], st.h2d) != cudaSuccess ||
        cudaStreamWaitEvent(st.comp[s], st.in[s], 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    // cover heads [f0, f1) with rectangles of (batches x heads)
    for (long long f = f0; f < f1;) {
      int b, pb, ph;  // first batch, batches and heads per batch of this rectangle
      head_rect(f, f1, a.H, b, pb, ph);
      const long long r = f - f0;  // heads into the slot
      TcArgs t{sq + r * hb.q, sk + r * hb.kv, sv + r * hb.kv, so + r * hb.o,
               a.lse ? reinterpret_cast<float*>(sl + r * hb.l) : nullptr, pb, ph, a.n_q, a.n_k, a.d, a.scale,
               a.mask_mode, padding ? d_lens + b : nullptr, st.comp[s], -1};
      if ((rc = launch_attn_tc(t, enc)) != ATTN_OK) return rc;
      f += (long long)pb * ph;
    }
    if (cudaEventRecord(st.done[s], st.comp[s]) != cudaSuccess ||
        cudaStreamWaitEvent(st.d2h, st.done[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(ho + f0 * hb.o, so, nh * hb.o, cudaMemcpyDeviceToHost, st.d2h) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (a.lse && cudaMemcpyAsync(a.lse + f0 * a.n_q, sl, nh * hb.l, cudaMemcpyDeviceToHost, st.d2h) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (cudaEventRecord(st.out[s], st.d2h) != cudaSuccess) return ATTN_ERR_CUDA;
    f0 = f1;
  }
  // the caller's stream is complete only when every result is back on the host
  for (int s = 0; s < kSlots && s < n_chunks; ++s)
    if (cudaStreamWaitEvent(cs, st.out[s], 0) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn
