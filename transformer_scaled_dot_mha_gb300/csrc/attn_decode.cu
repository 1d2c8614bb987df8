// attn_decode.cu -- one autoregressive decoding step: n_q (1..16) new queries per
// (batch, head) against a key/value cache, bf16 in and out, fp32 arithmetic.
//
// Query i of batch b sits at position cache_len[b] - n_q + i and attends to cache
// keys 0..position: the causal mask of decoder self-attention applied to the newest
// positions (generation proceeds one position at a time; attention-paper-guide
// section 05, rockcohen.cc sections 5.3 and 6.3), with Eq. (1) softmax(QK^T/sqrt(d_k))V
// per head (rockcohen.cc section 5.1).
//
// The work per query is tiny (a dot product and an axpy per cached key) while the
// cache is large, so the step is bound by reading K and V from HBM once. One query
// per (b, h) (the usual generation step) runs attn_decode_warp_kernel: the cache is
// cut into chunks, one independent warp per chunk (see there). Two to sixteen
// queries run the block kernel:
//   * split-K: the cache of each (b, h) is cut into `splits` ranges of whole
//     128-key tiles, one CTA per (range, b*h), enough CTAs to fill every SM;
//   * each CTA streams its 128-key K and V tiles with bulk asynchronous copies
//     (cp.async.bulk, completion counted on an mbarrier) through a 3-stage ring,
//     and runs the online softmax over its range in fp32: scores (thread = key),
//     per-query max / exp2 / sum (warp per query), P.V (thread = value column
//     pair x key part), with the running output rescaled when the maximum moves;
//   * it writes its unnormalised partial output o, running maximum m and sum l to
//     the workspace; a second kernel merges the ranges (or chunks) of each (b, h):
//     o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, M = max_s m_s.
// Waits on the copy barriers are bounded in time; a wait that runs out records a
// fault bit (attn_fault_status) and the CTA stops after its copies have landed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace attn {

__device__ unsigned int g_decode_fault_word;  // fault record of the decode kernels

// Scratch of attn_decode_noalloc: a fixed buffer in the library's own device
// memory, one per device that loads the library, kept until the process exits.
// Host code must not use the symbol itself as an address; it looks the device
// address up once per device (decode_noalloc_scratch below).
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_NOALLOC_MAX_BYTES];

namespace {

constexpr int TK = 128;       // keys per tile
constexpr int NTHREADS = 128;  // 4 warps
constexpr int STAGES = 3;
constexpr int MAX_NQ = 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr uint32_t FAULT_DECODE = 16;

template <int D>
struct DCfg {
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_BYTES = TK * ROW_BYTES;  // one K or V tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + STAGES * TILE_BYTES;    // float q_s[MAX_NQ][D]
  static constexpr int OFF_S = OFF_Q + MAX_NQ * D * 4;         // float s_s[MAX_NQ][TK]
  static constexpr int OFF_A = OFF_S + MAX_NQ * TK * 4;        // float alpha_s[MAX_NQ]
  static constexpr int OFF_BAR = OFF_A + MAX_NQ * 4;           // uint64 full[STAGES]
  static constexpr int SMEM_BYTES = OFF_BAR + STAGES * 8 + 16;
  static constexpr int PARTS = NTHREADS / (D / 2);             // key parts in the P.V phase
  static_assert(OFF_BAR % 8 == 0, "barrier alignment");
};

struct DecodeParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* out;
  float* lse;
  const int32_t* cache_lens;
  float* ws_o;   // [BH][splits][n_q][D]
  float* ws_ml;  // [BH][splits][n_q][2]
  int H, n_q, n_max, splits;
  int BH;          // B * H
  int chunk_keys;  // one query: keys per chunk (one warp each)
  float scale_log2;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

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

// Tiles [t0, t1) of the cache range of this split.
__device__ __forceinline__ void split_tiles(int len, int splits, int s, int& t0, int& t1) {
  const int tiles = (len + TK - 1) / TK;
  const int per = (tiles + splits - 1) / splits;
  t0 = min(s * per, tiles);
  t1 = min(t0 + per, tiles);
}

// ---------------------------------------------------------------- one query
// One query per (b, h), the usual generation step: every warp is independent. The
// cache of each (b, h) is cut into chunks of `chunk_keys` keys, one warp each; the
// warp streams its chunk's 32-key K and V tiles through a private ring of bulk copies
// (its own mbarriers, no block-wide barrier anywhere) and keeps the online softmax in
// registers. Within a tile, a K or V row of D bf16 is read by D / 8 lanes, 16 bytes
// each (lane group = key, lane within the group = 8 value columns): a score is the
// lane's 8-term dot product summed over its group with shuffles; the lane's 8 output
// columns accumulate p * v over the keys of its slot, and the slots are summed once at
// the end. The partial (o, m, l) of each chunk goes to the workspace as a split of the
// merge kernel below.
// One warp per CTA, so that a warp whose chunk is short or empty hands its SM slot
// back at once; a two-tile ring keeps a CTA at 16 KB (d = 64), thirteen of them per SM.
// (Same-box sweeps over 1-8 warps per CTA, 1-4 stages, 16-64-key tiles and 1-4 tasks
// per resident warp: this setting was fastest on both decode workloads.)
template <int D>
struct WCfg {
  static constexpr int TKW = 32;                       // keys per tile
  static constexpr int STAGES = 2;                     // tiles in flight per warp
  static constexpr int WARPS = 1;                      // warps per CTA
  static constexpr int LPR = D / 8;                    // lanes per K/V row (16 bytes each)
  static constexpr int KPL = 32 / LPR;                 // keys per warp-wide load
  static constexpr int NL = TKW / KPL;                 // loads per lane per tile
  static constexpr int TILE_BYTES = TKW * D * 2;
  static constexpr int WARP_BYTES = STAGES * 2 * TILE_BYTES;  // K ring, then V ring
  static constexpr int OFF_BAR = WARPS * WARP_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + WARPS * STAGES * 8;
  static constexpr int MIN_CHUNK = 4 * TKW;            // at least four tiles per warp
  static constexpr int CTAS_PER_SM = (228 * 1024) / (SMEM_BYTES + 1024);  // 1 KB reserved per CTA
  static constexpr int TASKS_PER_WARP = 2;              // chunks per resident warp
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  // ordered after the mbarrier wait that made the tile visible (memory clobber)
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr)
               : "memory");
  return r;
}

// Streams one chunk of the cache of (b, h) = bh and writes its partial (o, m, l) to
// workspace row ws_row; false if a copy never completed (recorded as a fault).
template <int D>
__device__ __forceinline__ bool stream_chunk(const DecodeParams& p, int bh, int k0, int nk, size_t ws_row, int warp,
                                             int lane) {
  using C = WCfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t s_w = ptx::smem_u32(smem) + warp * C::WARP_BYTES;
  const uint32_t bar0 = ptx::smem_u32(smem) + C::OFF_BAR + warp * C::STAGES * 8;
  const int n_tiles = (nk + C::TKW - 1) / C::TKW;
  const size_t row0 = (size_t)bh * p.n_max + k0;  // first cache row of the chunk
  if (lane == 0) {
    for (int st = 0; st < C::STAGES; ++st) ptx::mbar_init(bar0 + 8 * st, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int it) {  // tile it of the chunk into stage it % STAGES
    const int rows = min(C::TKW, nk - it * C::TKW);
    const uint32_t bytes = (uint32_t)rows * D * 2;
    const int st = it % C::STAGES;
    const size_t off = (row0 + (size_t)it * C::TKW) * D;
    ptx::mbar_arrive_expect_tx(bar0 + 8 * st, 2 * bytes);
    bulk_load(s_w + st * C::TILE_BYTES, p.k + off, bytes, bar0 + 8 * st);
    bulk_load(s_w + (C::STAGES + st) * C::TILE_BYTES, p.v + off, bytes, bar0 + 8 * st);
  };
  if (lane == 0)
    for (int it = 0; it < min(C::STAGES, n_tiles); ++it) issue(it);

  // this lane's 8 query columns, widened and pre-multiplied by scale * log2(e)
  const int cg = lane % C::LPR, ks = lane / C::LPR;
  float qf[8];
  {
    const uint4 qw = *reinterpret_cast<const uint4*>(p.q + (size_t)bh * D + 8 * cg);
    const uint32_t w4[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[2 * e] = __uint_as_float(w4[e] << 16) * p.scale_log2;
      qf[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u) * p.scale_log2;
    }
  }
  float o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;

  bool ok = true;
  int it_fail = 0;
  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % C::STAGES;
    if (!__all_sync(0xffffffffu, wait_full(bar0 + 8 * st, (it / C::STAGES) & 1))) {
      ok = false;
      it_fail = it;
      break;
    }
    const int rows = min(C::TKW, nk - it * C::TKW);
    const uint32_t k_t = s_w + st * C::TILE_BYTES + cg * 16;
    const uint32_t v_t = s_w + (C::STAGES + st) * C::TILE_BYTES + cg * 16;
    // scores of the keys ks + KPL * i of this tile (log2 units)
    float sc[C::NL];
#pragma unroll
    for (int i = 0; i < C::NL; ++i) {
      const uint4 kw = lds128(k_t + (ks + C::KPL * i) * (D * 2));
      const uint32_t w4[4] = {kw.x, kw.y, kw.z, kw.w};
      float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        d0 = fmaf(qf[2 * e], __uint_as_float(w4[e] << 16), d0);
        d1 = fmaf(qf[2 * e + 1], __uint_as_float(w4[e] & 0xffff0000u), d1);
      }
      sc[i] = d0 + d1;
    }
#pragma unroll
    for (int x = 1; x < C::LPR; x <<= 1)
#pragma unroll
      for (int i = 0; i < C::NL; ++i) sc[i] += __shfl_xor_sync(0xffffffffu, sc[i], x);
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < C::NL; ++i) {
      if (ks + C::KPL * i >= rows) sc[i] = -INFINITY;  // past the end of the cache
      mt = fmaxf(mt, sc[i]);
    }
#pragma unroll
    for (int x = C::LPR; x < 32; x <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, x));
    const float m_new = fmaxf(m_run, mt);
    const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
    const float alpha = ptx::ex2(m_run - m_use);  // 0 while nothing was legal
    float pr[C::NL], ps = 0.0f;
#pragma unroll
    for (int i = 0; i < C::NL; ++i) {
      pr[i] = ptx::ex2(sc[i] - m_use);
      ps += pr[i];
    }
#pragma unroll
    for (int x = C::LPR; x < 32; x <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, x);
    l_run = l_run * alpha + ps;
    m_run = m_new;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] *= alpha;
#pragma unroll
    for (int i = 0; i < C::NL; ++i) {
      if (ks + C::KPL * i < rows) {  // rows past the end hold stale bytes
        const uint4 vw = lds128(v_t + (ks + C::KPL * i) * (D * 2));
        const uint32_t w4[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[2 * e] = fmaf(pr[i], __uint_as_float(w4[e] << 16), o[2 * e]);
          o[2 * e + 1] = fmaf(pr[i], __uint_as_float(w4[e] & 0xffff0000u), o[2 * e + 1]);
        }
      }
    }
    __syncwarp();  // every lane has read stage st
    if (lane == 0 && it + C::STAGES < n_tiles) issue(it + C::STAGES);
  }

  if (!ok) {
    // a copy never completed: record it, let this warp's copies in flight land, stop
    if (lane == 0) {
      atomicOr(&g_decode_fault_word, FAULT_DECODE);
      for (int it = it_fail; it < min(it_fail + C::STAGES, n_tiles); ++it) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar0 + 8 * (it % C::STAGES), (it / C::STAGES) & 1))
          if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) break;
      }
    }
    __syncwarp();
    return false;
  }
  // sum the key slots; the lanes of slot 0 write the chunk's 8-column pieces
#pragma unroll
  for (int x = C::LPR; x < 32; x <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] += __shfl_xor_sync(0xffffffffu, o[e], x);
  if (ks == 0) {
    float4* dst = reinterpret_cast<float4*>(p.ws_o + ws_row * D + 8 * cg);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
  }
  if (lane == 0) {
    p.ws_ml[ws_row * 2 + 0] = m_run;
    p.ws_ml[ws_row * 2 + 1] = l_run;
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(WCfg<D>::WARPS * 32) attn_decode_warp_kernel(const DecodeParams p) {
  using C = WCfg<D>;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long task = (long long)blockIdx.x * C::WARPS + warp;  // (b*h, chunk)
  if (task >= (long long)p.BH * p.splits) return;
  const int bh = (int)(task / p.splits), chunk = (int)(task % p.splits);
  const int b = bh / p.H;
  const int len = min(max(p.cache_lens[b], 0), p.n_max);
  const int k0 = chunk * p.chunk_keys;
  const int nk = max(0, min(len - k0, p.chunk_keys));
  const size_t ws_row = (size_t)bh * p.splits + chunk;
  if (nk > 0) {
    if (!stream_chunk<D>(p, bh, k0, nk, ws_row, warp, lane)) {
      if (lane == 0) p.ws_ml[ws_row * 2 + 1] = 0.0f;  // a failed chunk contributes nothing
    }
  } else if (lane == 0) {  // nothing of this (b, h) in the chunk: an empty split
    p.ws_ml[ws_row * 2 + 0] = -INFINITY;
    p.ws_ml[ws_row * 2 + 1] = 0.0f;
  }
}

// NQ: compile-time bucket of the query count (n_q <= NQ), so that the per-query
// loops are as long as needed and no longer.
template <int D, int NQ>
__global__ void __launch_bounds__(NTHREADS) attn_decode_split_kernel(const DecodeParams p) {
  using C = DCfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t s_base = ptx::smem_u32(smem);
  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* s_s = reinterpret_cast<float*>(smem + C::OFF_S);
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_A);
  auto full = [&](int st) -> uint32_t { return s_base + C::OFF_BAR + 8u * st; };

  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bh = blockIdx.y, b = bh / p.H;
  const int n_q = p.n_q;
  const int len = min(max(p.cache_lens[b], 0), p.n_max);
  int t_begin, t_end;
  split_tiles(len, p.splits, split, t_begin, t_end);
  const int n_tiles = t_end - t_begin;
  const size_t cache_row0 = (size_t)bh * p.n_max;

  if (tid == 0) {
    for (int st = 0; st < STAGES; ++st) ptx::mbar_init(full(st), 1);
    ptx::fence_mbar_init();
  }
  // queries, widened to fp32 (raw bf16 bits -> float)
  for (int x = tid; x < n_q * D; x += NTHREADS) {
    const uint32_t bits = (uint32_t)p.q[((size_t)bh * n_q) * D + x] << 16;
    q_s[x] = __uint_as_float(bits);
  }
  __syncthreads();

  auto issue = [&](int it) {  // copy tile t_begin + it into stage it % STAGES
    const int tile = t_begin + it;
    const int rows = min(TK, len - tile * TK);
    const uint32_t bytes = (uint32_t)rows * C::ROW_BYTES;
    const int st = it % STAGES;
    ptx::mbar_arrive_expect_tx(full(st), 2 * bytes);
    const size_t off = (cache_row0 + (size_t)tile * TK) * D;
    bulk_load(s_base + C::OFF_K + st * C::TILE_BYTES, p.k + off, bytes, full(st));
    bulk_load(s_base + C::OFF_V + st * C::TILE_BYTES, p.v + off, bytes, full(st));
  };
  if (tid == 0)
    for (int it = 0; it < min(STAGES, n_tiles); ++it) issue(it);

  // per-query running state, replicated over the lanes of the warp that owns the query
  constexpr int QPW = (NQ + 3) / 4;  // queries per warp in the softmax phase
  float m_run[QPW], l_run[QPW];
#pragma unroll
  for (int x = 0; x < QPW; ++x) {
    m_run[x] = -INFINITY;
    l_run[x] = 0.0f;
  }
  // P.V accumulators: this thread's value column pair, all queries, its key part
  const int dp = tid % (D / 2), part = tid / (D / 2);
  float2 acc[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) acc[q] = make_float2(0.0f, 0.0f);

  bool ok = true;
  int it_fail = 0;
  for (int it = 0; it < n_tiles && ok; ++it) {
    const int st = it % STAGES;
    const int tile = t_begin + it;
    const int rows = min(TK, len - tile * TK);
    ok = __syncthreads_and(wait_full(full(st), (it / STAGES) & 1));
    if (!ok) {
      it_fail = it;
      break;
    }
    const uint32_t* k_t = reinterpret_cast<const uint32_t*>(smem + C::OFF_K + st * C::TILE_BYTES);
    const uint32_t* v_t = reinterpret_cast<const uint32_t*>(smem + C::OFF_V + st * C::TILE_BYTES);

    // ---- scores: thread = key; word order rotated by the key to spread banks; two
    // accumulator chains per query (even and odd value column)
    {
      const int kk = tid;
      float dot0[NQ], dot1[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) dot0[q] = dot1[q] = 0.0f;
      if (kk < rows) {
#pragma unroll 4
        for (int x = 0; x < D / 2; ++x) {
          const int w = (x + kk) & (D / 2 - 1);
          const uint32_t kw = k_t[kk * (D / 2) + w];
          const float k0 = __uint_as_float(kw << 16), k1 = __uint_as_float(kw & 0xffff0000u);
#pragma unroll
          for (int q = 0; q < NQ; ++q)
            if (q < n_q) {
              const float2 qv = *reinterpret_cast<const float2*>(&q_s[q * D + 2 * w]);
              dot0[q] = fmaf(qv.x, k0, dot0[q]);
              dot1[q] = fmaf(qv.y, k1, dot1[q]);
            }
        }
      }
      const int j = tile * TK + kk;  // cache position of this key
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q < n_q)
          s_s[q * TK + kk] = (kk < rows && j <= len - n_q + q) ? (dot0[q] + dot1[q]) * p.scale_log2 : -INFINITY;
    }
    __syncthreads();

    // ---- online softmax: warp w owns queries w, w+4, w+8, w+12
#pragma unroll
    for (int x = 0; x < QPW; ++x) {
      const int q = warp + 4 * x;
      if (q < n_q) {
        float sv[TK / 32];
        float mt = -INFINITY;
#pragma unroll
        for (int y = 0; y < TK / 32; ++y) {
          sv[y] = s_s[q * TK + lane + 32 * y];
          mt = fmaxf(mt, sv[y]);
        }
        mt = warp_max(mt);
        const float m_new = fmaxf(m_run[x], mt);
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = ptx::ex2(m_run[x] - m_use);  // 0 while nothing was legal
        float ps = 0.0f;
#pragma unroll
        for (int y = 0; y < TK / 32; ++y) {
          const float pv = ptx::ex2(sv[y] - m_use);
          s_s[q * TK + lane + 32 * y] = pv;
          ps += pv;
        }
        ps = warp_sum(ps);
        l_run[x] = l_run[x] * alpha + ps;
        m_run[x] = m_new;
        if (lane == 0) alpha_s[q] = alpha;
      }
    }
    __syncthreads();

    // ---- P.V: thread = (value column pair dp, key part); keys of the part in order
    {
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q < n_q) {
          const float a = alpha_s[q];
          acc[q].x *= a;
          acc[q].y *= a;
        }
      constexpr int KPP = TK / C::PARTS;  // keys per part
      const int k_lo = part * KPP, k_hi = min(k_lo + KPP, rows);
      for (int kk = k_lo; kk < k_hi; ++kk) {
        const uint32_t vw = v_t[kk * (D / 2) + dp];
        const float v0 = __uint_as_float(vw << 16), v1 = __uint_as_float(vw & 0xffff0000u);
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (q < n_q) {
            const float pv = s_s[q * TK + kk];
            acc[q].x = fmaf(pv, v0, acc[q].x);
            acc[q].y = fmaf(pv, v1, acc[q].y);
          }
      }
    }
    __syncthreads();  // stage `st` and s_s are free again
    if (tid == 0 && it + STAGES < n_tiles) issue(it + STAGES);
  }

  if (!ok) {
    // a copy never completed: record it, let the copies still in flight (tiles
    // it_fail .. it_fail + STAGES - 1) land, then stop
    if (tid == 0) {
      atomicOr(&g_decode_fault_word, FAULT_DECODE);
      for (int it = it_fail; it < min(it_fail + STAGES, n_tiles); ++it) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(full(it % STAGES), (it / STAGES) & 1))
          if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) break;
      }
    }
    // publish an empty partial (l = 0) for every query of this range, so that the
    // merge skips it instead of reading whatever the workspace held before
    const size_t ws_row_f = ((size_t)bh * p.splits + split) * n_q;
    for (int q = tid; q < n_q; q += NTHREADS) {
      p.ws_ml[(ws_row_f + q) * 2 + 0] = -INFINITY;
      p.ws_ml[(ws_row_f + q) * 2 + 1] = 0.0f;
    }
    __syncthreads();
    return;
  }

  // ---- reduce the key parts through shared memory (the K ring is free), write partials
  float* red = reinterpret_cast<float*>(smem + C::OFF_K);  // [PARTS][n_q][D]
#pragma unroll
  for (int q = 0; q < NQ; ++q)
    if (q < n_q) *reinterpret_cast<float2*>(&red[(part * n_q + q) * D + 2 * dp]) = acc[q];
  __syncthreads();
  const size_t ws_row = ((size_t)bh * p.splits + split) * n_q;
  for (int x = tid; x < n_q * D; x += NTHREADS) {
    float o = 0.0f;
#pragma unroll
    for (int pp = 0; pp < C::PARTS; ++pp) o += red[pp * n_q * D + x];
    p.ws_o[ws_row * D + x] = o;
  }
#pragma unroll
  for (int x = 0; x < QPW; ++x) {
    const int q = warp + 4 * x;
    if (q < n_q && lane == 0) {
      p.ws_ml[(ws_row + q) * 2 + 0] = m_run[x];
      p.ws_ml[(ws_row + q) * 2 + 1] = l_run[x];
    }
  }
}

// Merge the split ranges of one (b, h): thread x handles output element x of n_q x D.
template <int D>
__global__ void __launch_bounds__(NTHREADS) attn_decode_combine_kernel(const DecodeParams p) {
  ptx::grid_dep_wait();  // the partials of the split kernel
  ptx::grid_dep_launch();
  const int bh = blockIdx.x;
  const int n_q = p.n_q;
  for (int x = threadIdx.x; x < n_q * D; x += NTHREADS) {
    const int q = x / D;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) {
      const size_t r = ((size_t)bh * p.splits + s) * n_q + q;
      if (p.ws_ml[r * 2 + 1] > 0.0f) M = fmaxf(M, p.ws_ml[r * 2]);
    }
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
      for (int s = 0; s < p.splits; ++s) {
        const size_t r = ((size_t)bh * p.splits + s) * n_q + q;
        const float l_s = p.ws_ml[r * 2 + 1];
        if (l_s > 0.0f) {
          const float w = ptx::ex2(p.ws_ml[r * 2] - M);
          L = fmaf(w, l_s, L);
          o = fmaf(w, p.ws_o[r * D + (x % D)], o);
        }
      }
    }
    const float res = (L > 0.0f) ? o / L : 0.0f;
    p.out[((size_t)bh * n_q) * D + x] = __bfloat16_as_ushort(__float2bfloat16_rn(res));
    if (p.lse && (x % D) == 0)
      p.lse[(size_t)bh * n_q + q] = (L > 0.0f) ? (M + __log2f(L)) * 0.69314718055994530942f : -INFINITY;
  }
}

// Launches `kernel` on `stream` with programmatic dependent launch allowed: the kernel's
// CTAs may start while the previous grid on the stream finishes, and wait in
// grid_dep_wait before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D>
int launch_decode(const DecodeArgs& a, float* ws) {
  using C = DCfg<D>;
  DecodeParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.k = static_cast<const uint16_t*>(a.k);
  p.v = static_cast<const uint16_t*>(a.v);
  p.out = static_cast<uint16_t*>(a.out);
  p.lse = a.lse;
  p.cache_lens = a.cache_lens;
  p.H = a.H;
  p.n_q = a.n_q;
  p.n_max = a.n_max;
  p.splits = decode_splits(a.B, a.H, a.n_q, a.n_max, D);
  p.chunk_keys = decode_chunk_keys(a.B, a.H, a.n_max, D);
  p.scale_log2 = (float)((double)a.scale * 1.4426950408889634074);
  const long long bh = (long long)a.B * a.H;
  if (bh > 65535) return ATTN_ERR_UNSUPPORTED;  // one grid row per (b, h)
  p.BH = (int)bh;
  p.ws_o = ws;
  p.ws_ml = ws + (size_t)bh * p.splits * a.n_q * D;
  if (a.n_q == 1) {
    using W = WCfg<D>;
    if (cudaFuncSetAttribute(attn_decode_warp_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             W::SMEM_BYTES) != cudaSuccess)
      return ATTN_ERR_CUDA;
    // one warp per (b*h, chunk) task, consecutive chunks of a (b, h) in one CTA
    const unsigned blocks = (unsigned)((bh * p.splits + W::WARPS - 1) / W::WARPS);
    if (launch_pdl(attn_decode_warp_kernel<D>, dim3(blocks), dim3(W::WARPS * 32), W::SMEM_BYTES, a.stream, p) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
  } else {
    void (*split_kernel)(const DecodeParams) = a.n_q <= 2   ? attn_decode_split_kernel<D, 2>
                                               : a.n_q <= 4 ? attn_decode_split_kernel<D, 4>
                                               : a.n_q <= 8 ? attn_decode_split_kernel<D, 8>
                                                            : attn_decode_split_kernel<D, 16>;
    if (cudaFuncSetAttribute(split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    if (launch_pdl(split_kernel, dim3(p.splits, (unsigned)bh), dim3(NTHREADS), C::SMEM_BYTES, a.stream, p) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (cudaPeekAtLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  if (launch_pdl(attn_decode_combine_kernel<D>, dim3((unsigned)bh), dim3(NTHREADS), 0, a.stream, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

// One query: keys per warp task. About TASKS_PER_WARP tasks per resident warp over the
// whole cache extent, at least MIN_CHUNK keys each, a whole number of 32-key tiles.
template <int D>
static long long decode_tasks_target() {
  using W = WCfg<D>;
  return (long long)W::TASKS_PER_WARP * 152 * W::CTAS_PER_SM * W::WARPS;
}

int decode_chunk_keys(int B, int H, int n_max, int d) {
  const long long bh = (long long)B * H;
  const long long target = d == 64 ? decode_tasks_target<64>() : decode_tasks_target<128>();
  const int min_chunk = d == 64 ? WCfg<64>::MIN_CHUNK : WCfg<128>::MIN_CHUNK;
  long long per = (target + bh - 1) / bh;  // chunks per (b, h)
  const long long most = (n_max + min_chunk - 1) / min_chunk;
  if (per > most) per = most;
  if (per < 1) per = 1;
  const long long chunk = ((n_max + per - 1) / per + 31) / 32 * 32;
  return (int)chunk;
}

int decode_splits(int B, int H, int n_q, int n_max, int d) {
  const long long bh = (long long)B * H;
  if (n_q == 1) {
    const int chunk = decode_chunk_keys(B, H, n_max, d);
    return (n_max + chunk - 1) / chunk;
  }
  const long long target = 4LL * 152;  // CTAs to cover every SM a few times
  long long s = (target + bh - 1) / bh;
  const long long tiles = (n_max + TK - 1) / TK;
  if (s > tiles) s = tiles;
  if (s > 64) s = 64;
  return (int)(s < 1 ? 1 : s);
}

size_t decode_workspace_bytes(int B, int H, int n_q, int n_max, int d) {
  const size_t rows = (size_t)B * H * decode_splits(B, H, n_q, n_max, d) * n_q;
  return rows * ((size_t)d + 2) * sizeof(float);
}

int read_decode_fault_word(int clear, uint32_t* out) {
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_decode_fault_word, sizeof w) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_decode_fault_word, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  *out = w;
  return ATTN_OK;
}

namespace {
std::mutex g_scratch_mutex;
void* g_scratch_ptr[64];  // device address of g_decode_scratch, per device, once looked up
}  // namespace

// Device address of the static scratch on the current device; the first call on a
// device looks it up (cudaGetSymbolAddress) with that device current.
static int decode_noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

int launch_attn_decode_noalloc(const DecodeArgs& a) {
  if (decode_workspace_bytes(a.B, a.H, a.n_q, a.n_max, a.d) > sizeof(g_decode_scratch)) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int st = decode_noalloc_scratch(&scratch);
  if (st != ATTN_OK) return st;
  // every slot the kernels read is written first in the same call: nothing to clear
  return launch_attn_decode(a, scratch);
}

int launch_attn_decode(const DecodeArgs& a, void* workspace) {
  float* ws = static_cast<float*>(workspace);
  if (a.d == 64) return launch_decode<64>(a, ws);
  if (a.d == 128) return launch_decode<128>(a, ws);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
