// attn_bwd.cu -- gradients of scaled dot-product attention (dQ, dK, dV) on the
// sm_103a tensor cores, bf16 in and out, fp32 accumulation.
//
// For L = sum(dO * O) with O = softmax(scale Q K^T + mask) V (Eq. (1) of "Attention
// Is All You Need", rockcohen.cc section 5.1; masks of sections 5.3, 6.3), with
// P the softmax weights recomputed from the forward's log-sum-exp:
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),   D_i = sum_j P_ij dP_ij = dO_i . O_i
//   dQ = scale dS K,   dK = scale dS^T Q
// (training the model needs them: attention-paper-guide section 05; vlmlib.cn
// "training").
//
// Two schedules. The deterministic one (any d, or on request) has three kernels and
// no atomics:
//   attn_bwd_dot_kernel   D_i = dO_i . O_i (fp32), d / 8 lanes per row, written with
//                         -lse_i log2(e) into a per-tile table the other two kernels
//                         read (the dK/dV kernel with one bulk copy per query tile);
//   attn_bwd_dkdv_kernel  one CTA per 128-key tile of one (b, h); it streams the
//                         query tiles that can see its keys (Q_i, dO_i by TMA;
//                         lse_i, D_i by the producer warp), computes
//                         S^T = K Q_i^T and dP^T = V dO_i^T into TMEM, turns them
//                         into P^T and dS^T (bf16, written back into TMEM over
//                         the consumed columns; thread = key = TMEM lane), and
//                         accumulates dV += P^T dO_i and dK += dS^T Q_i in TMEM;
//   attn_bwd_dq_kernel    one CTA per 128-query tile; it streams the key tiles,
//                         computes S = Q K_j^T and dP = dO V_j^T, forms dS (thread =
//                         query) and accumulates dQ += dS K_j.
// The fused one (d = 64) computes each product once: the dK/dV kernel also writes
// dS^T to shared memory and forms the partial dQ_i = dS_i K (one more MMA per
// streamed tile, into one of two TMEM buffers, issued by a second MMA warp so that
// one thread does not issue every MMA of the tile); four drain warps move each partial
// through shared memory into an fp32 accumulator in global memory with TMA
// reduce-adds, and attn_bwd_dq_convert_kernel scales and rounds it to bf16. Five
// products instead of seven; the order of the reduce-adds, and so the last bits of
// dQ, varies from run to run.
// Every operand layout is one the forward kernel already uses: a [rows][d] tile
// loaded with 128-byte swizzling is a K-major operand along d and an MN-major
// operand along d. Waits are bounded as in the forward kernel; a wait that runs
// out records a fault bit (attn_fault_status), every role stops and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace attn {

__device__ unsigned int g_bwd_fault_word;  // fault record of the gradient kernels

namespace {

constexpr int T = 128;          // rows per tile (queries or keys)
// warps 0-7 elementwise (two warpgroups, one per half of every streamed tile: its
// rows 0-63 and 64-127), warp 8 TMA producer, warps 9 and 10 MMA issuers (one per
// half for the dQ kernel at d = 128; elsewhere warp 9 serves both halves, and in the
// fused kernel warp 10 issues the dQ partials)
constexpr int EW_THREADS = 256;
constexpr int WARP_LOAD = 8, WARP_MMA = 9;
constexpr int WARP_DRAIN = 12;  // fused: warps 12-15 drain the dQ partials (warp 11 idles)
constexpr int kMaxDevices = 64;
constexpr int kHeadGroup = 4;  // heads whose CTAs run together (L2 holds their streams and dQ sums)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr uint32_t FAULT_BWD = 32;

template <int D, bool FUSED = false>
struct BCfg {
  static_assert(!FUSED || D == 64, "the fused schedule is for d = 64");
  static constexpr int THREADS = FUSED ? 512 : EW_THREADS + 96;
  // fused: setmaxnreg split of the 512 x 128 launch registers
  static constexpr int REGS_EW = 176, REGS_CTRL = 80;
  static_assert(!FUSED || EW_THREADS * REGS_EW + (THREADS - EW_THREADS) * REGS_CTRL == THREADS * (65536 / THREADS),
                "register split");
  // ring depth; with d = 64 the deeper ring also keeps a second CTA (which would
  // block on the 512-column TMEM allocation) off the SM; the fused schedule gives
  // one stage to the dS and dQ staging tiles
  static constexpr int STAGES = FUSED ? 3 : D == 64 ? 4 : 2;
  static constexpr int CHUNKS = D / 64;
  static constexpr int CHUNK_BYTES = T * 128;
  static constexpr int TILE_BYTES = T * D * 2;
  // resident tiles (A operands) and a ring of streamed tile pairs
  static constexpr int OFF_A0 = 0;                          // K (dkdv) or Q (dq)
  static constexpr int OFF_A1 = OFF_A0 + TILE_BYTES;        // V (dkdv) or dO (dq)
  static constexpr int OFF_R0 = OFF_A1 + TILE_BYTES;        // ring: Q_i (dkdv) or K_j (dq)
  static constexpr int OFF_R1 = OFF_R0 + STAGES * TILE_BYTES;  // ring: dO_i (dkdv) or V_j (dq)
  static constexpr int OFF_VEC = OFF_R1 + STAGES * TILE_BYTES;  // float [STAGES][-lse*log2e[T], -D[T]]
  // fused: dS^T of the streamed tile, [2 query halves][T keys][128 B] (128-byte
  // swizzle; the MN-major A operand of dQ_i = dS_i K), then the fp32 dQ staging tiles,
  // [4 row quarters][2 column halves][32 rows][128 B] (128-byte swizzle, the reduce's box)
  static constexpr int OFF_DS = (OFF_VEC + 2 * STAGES * T * 4 + 1023) & ~1023;
  static constexpr int OFF_DQS = OFF_DS + (FUSED ? 2 * CHUNK_BYTES : 0);
  static constexpr int OFF_BAR = OFF_DQS + (FUSED ? 2 * CHUNK_BYTES : 0);
  // barriers: a_full, full[S], empty[S], mm_full[2 halves], p_full[2 halves], acc_done, drain[2 issuers],
  // fused: dq_full[2 buffers] (partial computed), dq_free[2 buffers] (partial read out of TMEM)
  static constexpr int B_AFULL = 0, B_FULL = 1, B_EMPTY = B_FULL + STAGES, B_MMFULL = B_EMPTY + STAGES;
  static constexpr int B_PFULL = B_MMFULL + 2, B_ACC = B_PFULL + 2, B_DRAIN = B_ACC + 1;
  static constexpr int B_DQFULL = B_DRAIN + 2, B_DQFREE = B_DQFULL + 2, NUM_BARS = B_DQFREE + 2;
  static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_SLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;
  // TMEM: per half h of the streamed tile, X_h = 128h + [0,64) holds S^T or S and
  // Y_h = 128h + [64,128) dP^T or dP (64 streamed rows each); the accumulators follow
  // from column 256 (acc_col). The bf16 pairs written back (P^T / dS^T, or dS) take the
  // first 32 columns of X_h / Y_h, which their warpgroup has already read.
  __host__ __device__ static constexpr uint32_t tm_x(int h) { return 128u * h; }
  __host__ __device__ static constexpr uint32_t tm_y(int h) { return 128u * h + 64u; }
  static constexpr uint32_t IDESC_NN = ptx::idesc_bf16_f32(T, T / 2, false);  // both operands K-major
  static constexpr uint32_t IDESC_ACC = ptx::idesc_bf16_f32(T, D, true);  // B MN-major
  static constexpr uint32_t IDESC_DQ = ptx::idesc_bf16_f32(T, D, true, true);  // A and B MN-major
  // fused: the two dQ partial buffers follow the dK and dV accumulators
  static constexpr uint32_t TMEM_DQ = 256u + 2u * D;
  static_assert(!FUSED || TMEM_DQ + 2 * D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct BwdParams {
  const float* stats;  // [BH][q_tiles][2][T]: -lse_i log2(e), then -D_i; rows past n_q hold -inf, 0
  uint16_t* g0;        // dkdv: dK [BH][n_k][D];  dq: dQ [BH][n_q][D]
  uint16_t* g1;        // dkdv: dV [BH][n_k][D]
  const int32_t* key_lens;
  int H, n_q, n_k, mask_mode, BH, tiles, q_tiles;
  int group;   // heads per group of the CTA order (see the kernel)
  int window;  // local window: key j legal for query i only if |i - j| <= window; -1: none
  float scale, scale_log2;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_bwd_fault_word, FAULT_BWD);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) return;
}

// Contiguous global -> shared copy (both 16-byte aligned, bytes a multiple of 16),
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}


// ------------------------------------------------------------------ D_i = dO_i . O_i
// Row r of the padded table (bh, tile, i): -lse_i log2(e) and -D_i, D_i = dO_i . O_i;
// rows past n_q get -inf (so P = 0) and 0. A row of O or dO (D bf16) is read by D / 8
// lanes, 16 bytes each, so a warp reads whole rows with coalesced 16-byte loads; each
// warp takes DOT_STEPS groups of rows and issues all their loads before the arithmetic,
// which keeps enough bytes in flight to stream O and dO at HBM speed.
constexpr int DOT_STEPS = 4;
template <int D>
__host__ __device__ constexpr int dot_rows_per_warp() {
  return (32 / (D / 8)) * DOT_STEPS;
}

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_dot_kernel(const uint16_t* out, const uint16_t* dout, const float* lse,
                                                           float* stats, int n_q, int q_tiles, long long rows) {
  constexpr int LPR = D / 8;      // lanes per row
  constexpr int RPS = 32 / LPR;   // rows per warp per step
  const int lane = threadIdx.x & 31, cg = lane % LPR;
  const long long first = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * dot_rows_per_warp<D>() + lane / LPR;
  const long long per_bh = (long long)q_tiles * T;
  uint4 o4[DOT_STEPS], g4[DOT_STEPS];
  long long src[DOT_STEPS];  // row of out / dout / lse, or -1 for a padding row or none
#pragma unroll
  for (int u = 0; u < DOT_STEPS; ++u) {
    const long long row = first + (long long)u * RPS;  // bh * q_tiles * T + i
    const long long bh = row / per_bh;
    const int i = (int)(row - bh * per_bh);
    src[u] = (row < rows && i < n_q) ? bh * n_q + i : -1;
    o4[u] = make_uint4(0, 0, 0, 0);
    g4[u] = make_uint4(0, 0, 0, 0);
    if (src[u] >= 0) {
      o4[u] = __ldg(reinterpret_cast<const uint4*>(out + src[u] * D) + cg);
      g4[u] = __ldg(reinterpret_cast<const uint4*>(dout + src[u] * D) + cg);
    }
  }
#pragma unroll
  for (int u = 0; u < DOT_STEPS; ++u) {
    const uint32_t a[4] = {o4[u].x, o4[u].y, o4[u].z, o4[u].w}, b[4] = {g4[u].x, g4[u].y, g4[u].z, g4[u].w};
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(a[e] << 16), __uint_as_float(b[e] << 16), acc);
      acc = fmaf(__uint_as_float(a[e] & 0xffff0000u), __uint_as_float(b[e] & 0xffff0000u), acc);
    }
#pragma unroll
    for (int off = 1; off < LPR; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const long long row = first + (long long)u * RPS;
    if (cg == 0 && row < rows) {
      const long long bh = row / per_bh;
      const int i = (int)(row - bh * per_bh);
      float* dst = stats + (bh * q_tiles + i / T) * 2 * T + (i % T);
      dst[0] = src[u] >= 0 ? -lse[src[u]] * 1.4426950408889634f : -INFINITY;
      dst[T] = src[u] >= 0 ? -acc : 0.0f;
    }
  }
}

// Legal key range of query row i of batch b: keys [0, lim).
__device__ __forceinline__ int key_limit(int i, int kv_len, bool causal) { return causal ? min(kv_len, i + 1) : kv_len; }

// ------------------------------------------------------------------ dK, dV
// KV tile kt of head bh; query tiles it = q_begin .. tiles-1 (causal: those at or
// after the key tile). MODE selects the operand roles (see the file comment). LOCAL:
// the local-window instantiation; the others see a constant window of -1, so their
// tile ranges and column bounds fold to the full-attention forms.
template <int D, bool DKDV, bool FUSED = false, bool LOCAL = false>
__global__ void __launch_bounds__(BCfg<D, FUSED>::THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                       const __grid_constant__ CUtensorMap tm_r0, const __grid_constant__ CUtensorMap tm_r1,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BCfg<D, FUSED>;
  static_assert(!FUSED || DKDV, "the fused schedule extends the dK/dV kernel");
  constexpr int STAGES = C::STAGES;
  // One issuer per half, each with its own accumulators (summed in the epilogue): for
  // the dQ kernel at D = 128, where the two halves' MMAs outrun one issuing thread
  // (same-box A/B: +3 %; at D = 64, and for dK/dV, one issuer measured as fast or
  // faster, and two dK/dV issuers would not fit TMEM at D = 128).
  constexpr bool SPLIT = !DKDV && D == 128;
  // TMEM column of accumulator `which` (DKDV: 0 = dK, 1 = dV; dQ: 0) of half h
  auto acc_col = [](int which, int h) -> uint32_t {
    if (!DKDV) return 256u + (SPLIT ? h : 0) * D;
    return SPLIT ? 256u + h * 128u + which * 64u : 256u + which * D;
  };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = ptx::smem_u32(smem);
  auto bar = [&](int x) -> uint32_t { return s_base + C::OFF_BAR + 8u * x; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SLOT);
  float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC);  // [S][-lse log2(e)[T], -D[T]]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // CTA order: groups of p.group heads, one after the other; within a group the own
  // tiles busiest first -- keys (DKDV: the low causal tiles) or queries (dQ: the high
  // ones) -- with the group's heads interleaved. The CTAs resident at one time then
  // work on a few heads, whose streamed tiles and fp32 dQ accumulators stay in L2.
  const int per_group = p.group * p.tiles;
  const int grp = (int)(blockIdx.x / per_group);
  const int gsize = min(p.group, p.BH - grp * p.group);
  const int within = (int)(blockIdx.x - (unsigned)grp * per_group);
  const int bh = grp * p.group + within % gsize;
  const int own = DKDV ? within / gsize : p.tiles - 1 - within / gsize;
  const int b = bh / p.H;
  const bool causal = (p.mask_mode & 1) != 0;
  int kv_len = p.n_k;
  if (p.mask_mode & 2) kv_len = min(max(p.key_lens[b], 0), p.n_k);
  const int own0 = own * T;
  const int window = LOCAL ? p.window : -1;
  // streamed tiles [s_begin, s_end): the tiles holding a row some own row may pair with
  int s_begin, s_end;
  if constexpr (!LOCAL) {
    if (DKDV) {  // query tiles that see any key of [own0, own0 + T)
      s_begin = (causal ? own0 : 0) / T;
      s_end = (own0 < kv_len) ? (p.n_q + T - 1) / T : s_begin;
    } else {     // key tiles any query of [own0, own0 + T) sees
      s_begin = 0;
      const int hi = causal ? min(kv_len, own0 + T) : kv_len;
      s_end = (own0 < p.n_q) ? (hi + T - 1) / T : 0;
    }
  } else if (DKDV) {  // queries [lo, hi) that see a key of [own0, own0 + T)
    const int lo = causal ? own0 : max(0, own0 - window);
    const int hi = min(p.n_q, own0 + T + window);
    s_begin = min(lo, p.n_q) / T;
    s_end = (own0 < kv_len && lo < hi) ? (hi + T - 1) / T : s_begin;
  } else {            // keys [lo, hi) that a query of [own0, own0 + T) sees
    const int lo = max(0, own0 - window);
    const int hi = min(causal ? min(kv_len, own0 + T) : kv_len, own0 + T + window);
    s_begin = min(lo, kv_len) / T;
    s_end = (own0 < p.n_q && lo < hi) ? (hi + T - 1) / T : s_begin;
  }
  const int n_s = max(0, s_end - s_begin);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(C::B_AFULL), 1);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(C::B_FULL + s), 1);  // TMA bytes
      ptx::mbar_init(bar(C::B_EMPTY + s), SPLIT ? 2 : 1);  // one commit per issuer
    }
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(bar(C::B_MMFULL + h), 1);
      ptx::mbar_init(bar(C::B_PFULL + h), EW_THREADS / 2);
    }
    ptx::mbar_init(bar(C::B_ACC), SPLIT ? 2 : 1);
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    ptx::mbar_init(bar(C::B_DRAIN + 1), 1);
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bar(C::B_DQFULL + x), 1);  // MMA commit
      ptx::mbar_init(bar(C::B_DQFREE + x), 4);  // one arrival per drain warp
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Fused: warpgroups 0-1 (elementwise) take registers from warpgroups 2-3 (producer,
  // issuer, idle warp, drain warps); the sum equals the launch allocation.
  if (warp >= 8) {
  if constexpr (FUSED) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CTRL));
  if (warp == WARP_LOAD) {
    // ================================================================ producer (whole warp)
    bool ok = true;
    int issued = 0;
    if (n_s > 0) {
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(C::B_AFULL), 2 * C::TILE_BYTES);
        for (int c = 0; c < C::CHUNKS; ++c) {
          ptx::tma_load_3d(s_base + C::OFF_A0 + c * C::CHUNK_BYTES, &tm_a0, bar(C::B_AFULL), c * 64, own0, bh, 0);
          ptx::tma_load_3d(s_base + C::OFF_A1 + c * C::CHUNK_BYTES, &tm_a1, bar(C::B_AFULL), c * 64, own0, bh, 0);
        }
      }
      for (int u = 0; u < n_s && ok; ++u) {
        const int st = u % STAGES;
        ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_EMPTY + st), ((u / STAGES) & 1) ^ 1, abort_flag));
        if (!ok) break;
        const int r0 = (s_begin + u) * T;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar(C::B_FULL + st), 2 * C::TILE_BYTES + (DKDV ? 2 * T * 4 : 0));
          if (DKDV)  // -lse log2(e) and -D of the 128 queries of this tile
            bulk_copy(s_base + C::OFF_VEC + st * 2 * T * 4, p.stats + ((size_t)bh * p.q_tiles + s_begin + u) * 2 * T,
                      2 * T * 4, bar(C::B_FULL + st));
          for (int c = 0; c < C::CHUNKS; ++c) {
            ptx::tma_load_3d(s_base + C::OFF_R0 + st * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_r0, bar(C::B_FULL + st),
                             c * 64, r0, bh, 0);
            ptx::tma_load_3d(s_base + C::OFF_R1 + st * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_r1, bar(C::B_FULL + st),
                             c * 64, r0, bh, 0);
          }
        }
        issued = u + 1;
      }
    }
    if (!ok && lane == 0) {
      drain_wait(bar(C::B_AFULL), 0);
      for (int u = max(0, issued - STAGES); u < issued; ++u) drain_wait(bar(C::B_FULL + u % STAGES), (u / STAGES) & 1);
    }
    __syncwarp();
  } else if (warp == WARP_MMA || warp == WARP_MMA + 1) {
    // ================================================================ MMA issuers
    // Half h of streamed tile u: S_h(u) and dP_h(u) (64 streamed rows), then, once its
    // warpgroup has stored P / dS, the accumulations. SPLIT: warp WARP_MMA + h serves
    // half h. Otherwise warp WARP_MMA serves both, in the order acc_h(u-1), S/dP_h(u)
    // for h = 0, 1; FUSED: warp WARP_MMA + 1 issues dQ_u = dS_u K once both halves of
    // tile u have stored dS (its own TMEM buffers: the other accumulators keep the
    // order and bits of the single-issuer schedule), else it idles.
    if (lane == 0 && n_s > 0 && (SPLIT || FUSED || warp == WARP_MMA)) {
      // Shared-memory descriptors are built once and advanced by adding (offset >> 4)
      // to the start-address field (addresses stay below 2^18, so the 14-bit field never
      // carries): this thread issues every MMA of the CTA and is kept lean.
      const uint64_t d_a0 = ptx::sdesc_sw128(s_base + C::OFF_A0, 16, 1024);
      const uint64_t d_a1 = ptx::sdesc_sw128(s_base + C::OFF_A1, 16, 1024);
      const uint64_t d_r0k = ptx::sdesc_sw128(s_base + C::OFF_R0, 16, 1024);              // K-major view
      const uint64_t d_r1k = ptx::sdesc_sw128(s_base + C::OFF_R1, 16, 1024);
      const uint64_t d_r0m = ptx::sdesc_sw128(s_base + C::OFF_R0, C::CHUNK_BYTES, 1024);  // MN-major view
      const uint64_t d_r1m = ptx::sdesc_sw128(s_base + C::OFF_R1, C::CHUNK_BYTES, 1024);
      auto koff16 = [](int kk) { return (uint64_t)(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4); };
      // fused: dQ_w = dS_w K into TMEM buffer w & 1; A = dS^T tile read MN-major (query
      // halves 16 KB apart), B = the resident K tile read MN-major, 16 keys per MMA
      const uint64_t d_ds = ptx::sdesc_sw128(s_base + C::OFF_DS, C::CHUNK_BYTES, 1024);
      const uint64_t d_a0m = ptx::sdesc_sw128(s_base + C::OFF_A0, C::CHUNK_BYTES, 1024);
      auto issue_dq = [&](int w) {
        const uint32_t d_col = tmem + C::TMEM_DQ + (uint32_t)(w & 1) * D;
#pragma unroll
        for (int kk = 0; kk < T / 16; ++kk) {
          const uint64_t ko = (uint64_t)((kk * 2048) >> 4);
          ptx::mma_ss(d_col, d_ds + ko, d_a0m + ko, C::IDESC_DQ, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar(C::B_DQFULL + (w & 1)));
      };
      // X_h = A0 R0_h^T, Y_h = A1 R1_h^T (both operands K-major along d); rows 64h.. of
      // a streamed slab start 64h * 128 bytes in
      auto issue_sdp = [&](int u, int h) {
        const uint64_t so = (uint64_t)(((u % STAGES) * C::TILE_BYTES + h * (T / 2) * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss(tmem + C::tm_x(h), d_a0 + koff16(kk), d_r0k + so + koff16(kk), C::IDESC_NN, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ss(tmem + C::tm_y(h), d_a1 + koff16(kk), d_r1k + so + koff16(kk), C::IDESC_NN, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(C::B_MMFULL + h));
      };
      // DKDV: dV += P_h^T dO_h, dK += dS_h^T Q_h; dQ: dQ += dS_h K_h. The bf16 pairs of
      // streamed rows 64h + 16kk .. + 15 sit at X_h / Y_h + 8kk; B rows are MN-major.
      auto issue_acc = [&](int u, int h) {
        const uint64_t so = (uint64_t)(((u % STAGES) * C::TILE_BYTES) >> 4);
        const uint32_t first = (u > 0 || (!SPLIT && h > 0)) ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t brow = (uint64_t)(((h * 4 + kk) * 2048) >> 4);
          const uint32_t accum = kk > 0 ? 1u : first;
          if (DKDV) {
            ptx::mma_ts(tmem + acc_col(1, h), tmem + C::tm_x(h) + kk * 8, d_r1m + so + brow, C::IDESC_ACC, accum);
            ptx::mma_ts(tmem + acc_col(0, h), tmem + C::tm_y(h) + kk * 8, d_r0m + so + brow, C::IDESC_ACC, accum);
          } else {
            ptx::mma_ts(tmem + acc_col(0, h), tmem + C::tm_x(h) + kk * 8, d_r0m + so + brow, C::IDESC_ACC, accum);
          }
        }
      };
      bool ok = wait_bar(bar(C::B_AFULL), 0, abort_flag) && wait_bar(bar(C::B_FULL), 0, abort_flag);
      if (FUSED && warp == WARP_MMA + 1) {
        for (int w = 0; w < n_s && ok; ++w) {
          // dS_w complete in shared memory (both halves); the buffer's previous partial
          // (tile w - 2) read out of TMEM
          ok = wait_bar(bar(C::B_PFULL), w & 1, abort_flag) && wait_bar(bar(C::B_PFULL + 1), w & 1, abort_flag);
          if (ok && w >= 2) ok = wait_bar(bar(C::B_DQFREE + (w & 1)), ((w >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_dq(w);
        }
      } else if (SPLIT) {
        // this warp serves half hs only: acc_hs(u-1), then S/dP_hs(u)
        const int hs = warp - WARP_MMA;
        if (ok) {
          ptx::tc_fence_after();
          issue_sdp(0, hs);
        }
        for (int u = 1; u <= n_s && ok; ++u) {
          if (u < n_s) {
            ok = wait_bar(bar(C::B_FULL + u % STAGES), (u / STAGES) & 1, abort_flag);
            if (!ok) break;
          }
          ok = wait_bar(bar(C::B_PFULL + hs), (u - 1) & 1, abort_flag);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_acc(u - 1, hs);
          ptx::mma_commit(bar(C::B_EMPTY + (u - 1) % STAGES));  // this half of tile u-1 is consumed
          if (u < n_s) issue_sdp(u, hs);
        }
      } else {
      if (ok) {
        ptx::tc_fence_after();
        issue_sdp(0, 0);
        issue_sdp(0, 1);
      }
      for (int u = 1; u <= n_s && ok; ++u) {
        if (u < n_s) {
          ok = wait_bar(bar(C::B_FULL + u % STAGES), (u / STAGES) & 1, abort_flag);
          if (!ok) break;
        }
        for (int h = 0; h < 2 && ok; ++h) {
          ok = wait_bar(bar(C::B_PFULL + h), (u - 1) & 1, abort_flag);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_acc(u - 1, h);
          if (h == 1) ptx::mma_commit(bar(C::B_EMPTY + (u - 1) % STAGES));  // tile u-1's stage is consumed
          if (u < n_s) issue_sdp(u, h);
        }
      }
      }
      if (ok && !(FUSED && warp == WARP_MMA + 1)) ptx::mma_commit(bar(C::B_ACC));
      if (!ok) {
        ptx::mma_commit(bar(C::B_DRAIN + (warp - WARP_MMA)));
        drain_wait(bar(C::B_DRAIN + (warp - WARP_MMA)), 0);
      }
    }
    __syncwarp();
  } else if (FUSED && warp >= WARP_DRAIN) {
    // ================================================================ dQ drain (fused; warps 12-15)
    // Thread = query row of the streamed tile = TMEM lane; warp w owns rows
    // 32 (w % 4) .. + 31 and needs no other warp. Each partial goes TMEM -> registers ->
    // the warp's swizzled fp32 staging tiles -> two TMA reduce-adds (columns 0-31 and
    // 32-63, 32 rows each) into the fp32 accumulator; rows past n_q fall outside the
    // tensor and are skipped. Lane 0 issues the reduces and, before the staging tiles
    // are refilled, waits until the previous ones have read them.
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage = s_base + C::OFF_DQS + quarter * 2 * 4096;  // [2 column halves][32 rows][128 B]
    bool ok = true;
    for (int u = 0; u < n_s && ok; ++u) {
      const int buf = u & 1;
      ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_DQFULL + buf), (u >> 1) & 1, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      if (lane == 0) ptx::bulk_wait_read0();
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16 columns at a time: column half c / 2, units 4 (c & 1) ..
        uint32_t v[16];
        ptx::tmem_ld16(tmem + lane_off + C::TMEM_DQ + (uint32_t)buf * D + c * 16, v);
        ptx::tmem_wait_ld();
        const uint32_t row = stage + (c >> 1) * 4096 + lane * 128;
#pragma unroll
        for (int x = 0; x < 4; ++x)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (uint32_t)((((c & 1) * 4 + x) ^ (lane & 7)) << 4)),
                       "r"(v[4 * x]), "r"(v[4 * x + 1]), "r"(v[4 * x + 2]), "r"(v[4 * x + 3])
                       : "memory");
      }
      ptx::tc_fence_before();
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(bar(C::B_DQFREE + buf));
        const int y = (s_begin + u) * T + quarter * 32;
        ptx::tma_reduce_add_3d(&tm_dq, stage, 0, y, bh);
        ptx::tma_reduce_add_3d(&tm_dq, stage + 4096, 32, y, bh);
        ptx::bulk_commit();
      }
    }
    if (lane == 0) ptx::bulk_wait0();
    __syncwarp();
  }
  } else {
    if constexpr (FUSED) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_EW));
    // ================================================================ elementwise warpgroups (warps 0-7)
    // Thread = own row (key for DKDV, query for dQ) = TMEM lane; warpgroup g takes half
    // g of every streamed tile (its rows 64g .. 64g + 63 = the columns of X_g, Y_g). No
    // element needs another: P and dS of one (key, query) pair use only that pair's S,
    // dP and the query's lse and D.
    const int g = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_x = tmem + lane_off + C::tm_x(g), t_y = tmem + lane_off + C::tm_y(g);
    const int own_row = own0 + r;
    const uint64_t c2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    // dQ: this thread's query statistics
    uint64_t nl2 = 0ull, nd2 = 0ull;  // (-lse*log2e, -lse*log2e), (-D, -D)
    // the rows this thread's row pairs with: [my_lo, my_hi) (keys for dQ, queries for dK/dV)
    int my_lo = 0, my_hi = 0;
    if (!DKDV && own_row < p.n_q) {
      const float* srow = p.stats + ((size_t)bh * p.q_tiles + own) * 2 * T + r;
      const float nl = srow[0];
      const float nd = srow[T];
      nl2 = ptx::f2_pack(nl, nl);
      nd2 = ptx::f2_pack(nd, nd);
      my_hi = key_limit(own_row, kv_len, causal);
      if (LOCAL) {
        my_lo = max(0, own_row - window);
        my_hi = min(my_hi, own_row + window + 1);
      }
    }
    if (LOCAL && DKDV && own_row < kv_len) {  // query >= key (causal), |query - key| <= window
      my_lo = causal ? own_row : max(0, own_row - window);
      my_hi = own_row + window + 1;  // rows past n_q carry P = 0
    }
    const bool row_dead = LOCAL ? my_lo >= my_hi : (DKDV ? own_row >= kv_len : my_hi == 0);
    bool ok = true;
    for (int u = 0; u < n_s && ok; ++u) {
      const int st = u % STAGES;
      ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_MMFULL + g), u & 1, abort_flag));
      // the stage's lse / D vectors (DKDV): already complete, waited on for ordering
      if (DKDV && ok) ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_FULL + st), (u / STAGES) & 1, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      const int s0 = (s_begin + u) * T + g * 64;  // streamed row of this thread's first column
      // columns [lo, hi) are legal for this thread; the rest get P = 0
      int lo = 0, hi = 64;
      if constexpr (LOCAL) {  // my_hi - s0 stays in range: the window is at most n
        if (row_dead) {
          hi = 0;
        } else {
          lo = max(0, my_lo - s0);
          hi = max(0, min(64, my_hi - s0));
        }
      } else if (DKDV) {
        if (row_dead) hi = 0;
        else if (causal) lo = max(0, own_row - s0);  // query >= key
      } else {
        hi = max(0, min(64, my_hi - s0));
      }
      const bool full = (lo == 0 && hi == 64);
      const float* vnl = vec + st * 2 * T + g * 64;      // -lse*log2e of the columns (DKDV)
      const float* vnd = vec + st * 2 * T + T + g * 64;  // -D of the columns (DKDV)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t xs[32], ys[32];
        ptx::tmem_ld32(t_x + ch * 32, xs);
        ptx::tmem_ld32(t_y + ch * 32, ys);
        ptx::tmem_wait_ld();
        uint32_t pw[16], dw[16];
        float4 nl4, nd4;  // DKDV: -lse*log2e and -D of four columns, one 16-byte broadcast load each
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const int cc = ch * 32 + x;  // column within this warpgroup's half
          uint64_t nl, nd;
          if (DKDV) {
            if ((x & 2) == 0) {
              nl4 = *reinterpret_cast<const float4*>(vnl + cc);
              nd4 = *reinterpret_cast<const float4*>(vnd + cc);
            }
            nl = (x & 2) ? ptx::f2_pack(nl4.z, nl4.w) : ptx::f2_pack(nl4.x, nl4.y);
            nd = (x & 2) ? ptx::f2_pack(nd4.z, nd4.w) : ptx::f2_pack(nd4.x, nd4.y);
          } else {
            nl = nl2;
            nd = nd2;
          }
          float a0, a1;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(xs[x]), __uint_as_float(xs[x + 1])), c2, nl), a0, a1);
          float p0 = ptx::ex2(a0), p1 = ptx::ex2(a1);
          if (!full) {
            p0 = (cc >= lo && cc < hi) ? p0 : 0.0f;
            p1 = (cc + 1 >= lo && cc + 1 < hi) ? p1 : 0.0f;
          }
          const uint64_t pp = ptx::f2_pack(p0, p1);
          const uint64_t dp = ptx::f2_add(ptx::f2_pack(__uint_as_float(ys[x]), __uint_as_float(ys[x + 1])), nd);
          float d0, d1;
          ptx::f2_unpack(ptx::f2_mul(pp, dp), d0, d1);
          if (DKDV) pw[x >> 1] = ptx::pack_bf16x2(p0, p1);
          dw[x >> 1] = ptx::pack_bf16x2(d0, d1);
        }
        // P^T over X_g and dS^T over Y_g (DKDV), or dS over X_g (dQ), at columns 16 ch:
        // already read (chunk ch covers columns 32 ch .. 32 ch + 31)
        if (FUSED) {
          // dS^T row of this key into the A tile of dQ_u = dS_u K: query half g, 16-byte
          // unit c at (c ^ (key & 7)); the tile is free once dQ_{u-1} has been computed
          if (ch == 0 && u > 0)
            ok = __all_sync(0xffffffffu,
                            wait_bar(bar(C::B_DQFULL + ((u - 1) & 1)), ((u - 1) >> 1) & 1, abort_flag));
          if (ok) {
            const uint32_t row = s_base + C::OFF_DS + g * C::CHUNK_BYTES + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (uint32_t)(((ch * 4 + j) ^ (r & 7)) << 4)),
                           "r"(dw[4 * j]), "r"(dw[4 * j + 1]), "r"(dw[4 * j + 2]), "r"(dw[4 * j + 3])
                           : "memory");
          }
        }
        if (DKDV) {
          asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                       ::"r"(t_x + ch * 16), "r"(pw[0]), "r"(pw[1]), "r"(pw[2]), "r"(pw[3]), "r"(pw[4]),
                       "r"(pw[5]), "r"(pw[6]), "r"(pw[7]), "r"(pw[8]), "r"(pw[9]), "r"(pw[10]), "r"(pw[11]), "r"(pw[12]),
                       "r"(pw[13]), "r"(pw[14]), "r"(pw[15]) : "memory");
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                     ::"r"((DKDV ? t_y : t_x) + ch * 16), "r"(dw[0]), "r"(dw[1]), "r"(dw[2]), "r"(dw[3]), "r"(dw[4]),
                     "r"(dw[5]), "r"(dw[6]), "r"(dw[7]), "r"(dw[8]), "r"(dw[9]), "r"(dw[10]), "r"(dw[11]), "r"(dw[12]),
                     "r"(dw[13]), "r"(dw[14]), "r"(dw[15]) : "memory");
      }
      ptx::tmem_wait_st();
      if (!ok) break;
      if (FUSED) ptx::fence_proxy_async_smem();  // dS^T stores before the dQ MMA reads them
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_PFULL + g));
    }

    // ---------------------------------------------------------------- epilogue
    // DKDV: warpgroup 0 writes dK = scale * (its accumulators), warpgroup 1 dV.
    // dQ: warpgroup g writes columns [g D/2, g D/2 + D/2) of dQ = scale * accumulator.
    // With one issuer per half (SPLIT) each result is the sum of the halves' accumulators.
    // A tile with nothing to stream (all keys padding, or rows past the end) writes zeros.
    const int n_rows = DKDV ? p.n_k : p.n_q;
    const bool row_valid = own_row < n_rows;
    if (ok && n_s > 0) {
      ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_ACC), 0, abort_flag));
      if (ok) ptx::tc_fence_after();
    }
    if (ok) {
      uint16_t* gout = (DKDV && g == 1) ? p.g1 : p.g0;
      const float mul = (DKDV && g == 1) ? 1.0f : p.scale;
      const uint32_t col0 = DKDV ? acc_col(g, 0) : acc_col(0, 0) + g * (D / 2);
      const uint32_t col1 = DKDV ? acc_col(g, 1) : acc_col(0, 1) + g * (D / 2);  // the other half's (SPLIT)
      constexpr int NCH = DKDV ? D / 32 : D / 64;  // 32-column chunks this thread writes
      uint16_t* grow = gout + ((size_t)bh * n_rows + (size_t)(row_valid ? own_row : 0)) * D + (DKDV ? 0 : g * (D / 2));
#pragma unroll
      for (int q4 = 0; q4 < NCH; ++q4) {
        uint32_t o[32];
        if (n_s > 0) {
          ptx::tmem_ld32(tmem + lane_off + col0 + q4 * 32, o);
          if (SPLIT) {
            uint32_t o1[32];
            ptx::tmem_ld32(tmem + lane_off + col1 + q4 * 32, o1);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) + __uint_as_float(o1[x]));
          } else {
            ptx::tmem_wait_ld();
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = ptx::pack_bf16x2(__uint_as_float(o[2 * x]) * mul, __uint_as_float(o[2 * x + 1]) * mul);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(grow + q4 * 32);
#pragma unroll
          for (int x = 0; x < 4; ++x) dst[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// dQ = scale * (the fp32 sum of the per-key-tile partials), rounded to bf16 once;
// four elements per thread.
__global__ void __launch_bounds__(256) attn_bwd_dq_convert_kernel(const float4* acc, uint2* dq, float scale,
                                                                  long long n4) {
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n4; i += (long long)gridDim.x * 256) {
    const float4 a = acc[i];
    dq[i] = make_uint2(ptx::pack_bf16x2(a.x * scale, a.y * scale), ptx::pack_bf16x2(a.z * scale, a.w * scale));
  }
}

// The fp32 dQ accumulator [bh][n][64] as the reduce target: boxes of 32 columns
// (128 bytes) x 32 rows, 128-byte swizzle.
CUresult encode_acc(PFN_encodeTiled enc, CUtensorMap* map, const float* base, int n, int bh) {
  cuuint64_t dims[3] = {64, (cuuint64_t)n, (cuuint64_t)bh};
  cuuint64_t strides[2] = {64 * 4, (cuuint64_t)64 * 4 * (cuuint64_t)n};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode(PFN_encodeTiled enc, CUtensorMap* map, const void* base, int d, int n, int bh) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)n};
  cuuint32_t box[3] = {64, (cuuint32_t)T, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int D, bool DKDV, bool FUSED, bool LOCAL>
int set_smem_attr() {
  static std::atomic<bool> done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  if (!done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(attn_bwd_tc_kernel<D, DKDV, FUSED, LOCAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BCfg<D, FUSED>::SMEM_BYTES) != cudaSuccess)
      return ATTN_ERR_CUDA;
    done[dev].store(true, std::memory_order_release);
  }
  return ATTN_OK;
}

// dq_acc: the fp32 dQ accumulator of the fused schedule, or null for the
// deterministic one.
template <int D, bool LOCAL>
int launch_bwd(const BwdArgs& a, PFN_encodeTiled enc, float* stats, float* dq_acc) {
  const int BH = a.B * a.H;
  const bool fused = dq_acc != nullptr;
  CUtensorMap mq, mk, mv, mdo, macc;
  if (encode(enc, &mq, a.q, D, a.n_q, BH) != CUDA_SUCCESS || encode(enc, &mk, a.k, D, a.n_k, BH) != CUDA_SUCCESS ||
      encode(enc, &mv, a.v, D, a.n_k, BH) != CUDA_SUCCESS || encode(enc, &mdo, a.dout, D, a.n_q, BH) != CUDA_SUCCESS)
    return ATTN_ERR_UNSUPPORTED;
  if (fused && encode_acc(enc, &macc, dq_acc, a.n_q, BH) != CUDA_SUCCESS) return ATTN_ERR_UNSUPPORTED;
  if (!fused) macc = mq;  // not read by the deterministic kernels
  if (fused) {
    if constexpr (D == 64) {
      if (set_smem_attr<D, true, true, LOCAL>() != ATTN_OK) return ATTN_ERR_CUDA;
    } else {
      return ATTN_ERR_UNSUPPORTED;
    }
  } else if (set_smem_attr<D, true, false, LOCAL>() != ATTN_OK || set_smem_attr<D, false, false, LOCAL>() != ATTN_OK) {
    return ATTN_ERR_CUDA;
  }
  if (fused && cudaMemsetAsync(dq_acc, 0, (size_t)BH * a.n_q * D * sizeof(float), a.stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int q_tiles = (a.n_q + T - 1) / T;
  const long long rows = (long long)BH * q_tiles * T;
  const long long rows_per_block = 8LL * dot_rows_per_warp<D>();
  if ((rows + rows_per_block - 1) / rows_per_block > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  attn_bwd_dot_kernel<D><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, a.stream>>>(
      static_cast<const uint16_t*>(a.out), static_cast<const uint16_t*>(a.dout), a.lse, stats, a.n_q, q_tiles, rows);
  if (cudaPeekAtLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  BwdParams p;
  p.stats = stats;
  p.q_tiles = q_tiles;
  p.key_lens = a.key_lens;
  p.H = a.H;
  p.n_q = a.n_q;
  p.n_k = a.n_k;
  p.mask_mode = a.mask_mode;
  p.BH = BH;
  p.group = BH < kHeadGroup ? (int)BH : kHeadGroup;
  p.window = a.window;
  p.scale = a.scale;
  p.scale_log2 = (float)((double)a.scale * 1.4426950408889634074);
  // dK, dV: own = key tiles; A0 = K, A1 = V; streamed R0 = Q, R1 = dO
  p.g0 = static_cast<uint16_t*>(a.dk);
  p.g1 = static_cast<uint16_t*>(a.dv);
  p.tiles = (a.n_k + T - 1) / T;
  long long grid = (long long)BH * p.tiles;
  if (grid > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (fused) {
    if constexpr (D == 64) {
      using CF = BCfg<D, true>;
      attn_bwd_tc_kernel<D, true, true, LOCAL><<<(unsigned)grid, CF::THREADS, CF::SMEM_BYTES, a.stream>>>(
          mk, mv, mq, mdo, macc, p);
      if (cudaPeekAtLastError() != cudaSuccess) return ATTN_ERR_CUDA;
      const long long n4 = (long long)BH * a.n_q * D / 4;
      const long long blocks = std::min<long long>((n4 + 255) / 256, 152LL * 8);
      attn_bwd_dq_convert_kernel<<<(unsigned)blocks, 256, 0, a.stream>>>(
          reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(a.dq), a.scale, n4);
      return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
  }
  attn_bwd_tc_kernel<D, true, false, LOCAL><<<(unsigned)grid, BCfg<D>::THREADS, BCfg<D>::SMEM_BYTES, a.stream>>>(
      mk, mv, mq, mdo, macc, p);
  if (cudaPeekAtLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  // dQ: own = query tiles; A0 = Q, A1 = dO; streamed R0 = K, R1 = V
  p.g0 = static_cast<uint16_t*>(a.dq);
  p.g1 = nullptr;
  p.tiles = (a.n_q + T - 1) / T;
  grid = (long long)BH * p.tiles;
  if (grid > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  attn_bwd_tc_kernel<D, false, false, LOCAL><<<(unsigned)grid, BCfg<D>::THREADS, BCfg<D>::SMEM_BYTES, a.stream>>>(
      mq, mdo, mk, mv, macc, p);
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

bool bwd_fused(int d, int flags) { return d == 64 && !(flags & ATTN_BWD_DETERMINISTIC); }

// per (b, h) and 128-row query tile: -lse log2(e) and -D of its rows, 2 x 128 floats;
// then, for the fused schedule, the fp32 dQ accumulator [B h][n_q][64]
size_t bwd_workspace_bytes(int B, int H, int n_q, int d, int flags) {
  const size_t stats = (size_t)B * H * ((n_q + T - 1) / T) * 2 * T * sizeof(float);
  return stats + (bwd_fused(d, flags) ? (size_t)B * H * n_q * 64 * sizeof(float) : 0);
}

int launch_attn_bwd(const BwdArgs& a, PFN_encodeTiled enc, void* workspace) {
  float* stats = static_cast<float*>(workspace);
  float* dq_acc = bwd_fused(a.d, a.flags) ? stats + (size_t)a.B * a.H * ((a.n_q + T - 1) / T) * 2 * T : nullptr;
  const bool local = a.window >= 0;
  if (a.d == 64)
    return local ? launch_bwd<64, true>(a, enc, stats, dq_acc) : launch_bwd<64, false>(a, enc, stats, dq_acc);
  if (a.d == 128)
    return local ? launch_bwd<128, true>(a, enc, stats, nullptr) : launch_bwd<128, false>(a, enc, stats, nullptr);
  return ATTN_ERR_UNSUPPORTED;
}

int read_bwd_fault_word(int clear, uint32_t* out) {
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_bwd_fault_word, sizeof w) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_bwd_fault_word, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  *out = w;
  return ATTN_OK;
}

}  // namespace attn
