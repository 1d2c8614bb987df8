// attn_weights.cu -- the softmax weights of scaled dot-product attention themselves,
// P[i, j] = softmax_j(scale * q_i . k_j) over the legal keys of row i and 0 on the
// others: the second value the pages' scaled_dot_product_attention returns beside the
// output (csdn blog reimplementation, scaled_dot_product_attention; rockcohen.cc
// "Attention Is All You Need" section 5.1, Eq. (1)). The forward never forms this
// matrix; here it is computed from q, k and the log-sum-exp lse that attn_fwd returned
// for the same inputs: P[i, j] = exp(scale * q_i . k_j - lse_i).
//
// One CTA per (b, h, 128-row Q tile), 192 threads: warps 0-3 turn S tiles into weights
// (thread = query row = TMEM lane), warp 4 is the TMA producer (Q once, K tiles through a
// two-stage ring), warp 5 owns TMEM and issues S = Q K_j^T into one of two 128-column
// buffers. Key tiles that no row of the Q tile may see (past the causal diagonal or the
// key length) are not computed: their weights are written as zeros.
#include <atomic>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace attn {

__device__ unsigned int g_weights_fault_word;  // fault record read by attn_fault_status

namespace {

constexpr int WBM = 128;  // query rows per CTA
constexpr int WBN = 128;  // keys per tile
constexpr uint64_t kWLimitNs = 2000000000ull;    // 2 s per wait, then give up
constexpr uint64_t kWDrainLimitNs = 200000000ull;
constexpr uint32_t FAULT_WEIGHTS = 256;          // bit 8 of the fault record
constexpr int kMaxDevicesW = 64;

template <int D>
struct WCfg {
  static constexpr int CHUNKS = D / 64;          // 128-byte swizzle atoms per row
  static constexpr int CHUNK_BYTES = WBM * 128;  // one 128-row x 64-column slab
  static constexpr int TILE_BYTES = WBM * D * 2;
  static constexpr int STAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = TILE_BYTES;
  static constexpr int OFF_BAR = OFF_K + STAGES * TILE_BYTES;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;                 // [STAGES]
  static constexpr int B_KEMPTY = B_KFULL + STAGES;  // [STAGES]
  static constexpr int B_SFULL = B_KEMPTY + STAGES;  // [2] S buffer computed
  static constexpr int B_SFREE = B_SFULL + 2;        // [2] S buffer loaded by every row thread
  static constexpr int B_DRAIN = B_SFREE + 2;        // MMA drain after an abort
  static constexpr int NUM_BARS = B_DRAIN + 1;
  // per row warp, a 32 x 32 fp32 staging block (rows 128 bytes, 16-byte chunks swizzled by
  // the row's low three bits) that turns one-row-per-thread results into row-contiguous
  // global stores
  static constexpr int OFF_STG = (OFF_BAR + NUM_BARS * 8 + 127) & ~127;
  static constexpr int STG_BYTES = 32 * 32 * 4;
  static constexpr int OFF_SLOT = OFF_STG + 4 * STG_BYTES;
  static constexpr int OFF_ABORT = OFF_SLOT + 4;
  static constexpr int SMEM_USED = OFF_ABORT + 4;
  // at least 80 KB, so that no more than two CTAs (2 x 256 TMEM columns) share an SM
  static constexpr int SMEM_BYTES = SMEM_USED > 80 * 1024 ? SMEM_USED : 80 * 1024;
  static constexpr uint32_t TMEM_COLS = 2 * WBN;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(WBM, WBN, false);  // Q, K both K-major
  static constexpr int THREADS = 192;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct WParams {
  float* w;
  const float* lse;
  const int32_t* key_lens;
  int H, n_q, n_k, mask_mode, num_qblocks;
  float c;  // scale * log2(e)
};

__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_weights_fault_word, FAULT_WEIGHTS);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void wdrain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > kWDrainLimitNs) return;
}

template <int D>
__global__ void __launch_bounds__(WCfg<D>::THREADS, 2)
    attn_weights_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const WParams p) {
  using C = WCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((ptx::smem_u32(smem) & 1023u) != 0) {  // every thread of the CTA takes this branch alike
    if (threadIdx.x == 0) atomicOr(&g_weights_fault_word, FAULT_WEIGHTS);
    return;
  }
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t s_q = s_base + C::OFF_Q, s_k = s_base + C::OFF_K;
  auto bar = [&](int i) -> uint32_t { return s_base + C::OFF_BAR + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SLOT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(bar(C::B_KFULL + s), 1);
      ptx::mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bar(C::B_SFULL + x), 1);
      ptx::mbar_init(bar(C::B_SFREE + x), WBM);  // every row thread arrives
    }
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int qb = (int)(blockIdx.x % (unsigned)p.num_qblocks);
  const int bh = (int)(blockIdx.x / (unsigned)p.num_qblocks);
  const int b = bh / p.H;
  const int row0 = qb * WBM;
  const bool causal = (p.mask_mode & ATTN_MASK_CAUSAL) != 0;
  int kv_len = p.n_k;
  if (p.mask_mode & ATTN_MASK_KEY_PADDING) kv_len = min(max(p.key_lens[b], 0), p.n_k);
  // key tiles holding a key that some row of this Q tile may see
  int n_s = (kv_len + WBN - 1) / WBN;
  if (causal) n_s = min(n_s, (row0 + WBM - 1) / WBN + 1);

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && n_s > 0) {
      ptx::mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE_BYTES);
      for (int c = 0; c < C::CHUNKS; ++c)
        ptx::tma_load_3d(s_q + c * C::CHUNK_BYTES, &tm_q, bar(C::B_QFULL), c * 64, row0, bh,
                         ptx::policy_evict_first());
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_s; ++j) {
        const int s = j % C::STAGES;
        ok = wwait(bar(C::B_KEMPTY + s), ((j / C::STAGES) & 1) ^ 1, abort_flag);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
        for (int c = 0; c < C::CHUNKS; ++c)
          ptx::tma_load_3d(s_k + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, bar(C::B_KFULL + s), c * 64,
                           j * WBN, bh, ptx::policy_evict_last());
        issued = j + 1;
      }
      if (!ok) {  // copies still in flight must land before the shared memory goes away
        wdrain(bar(C::B_QFULL), 0);
        for (int j = max(0, issued - C::STAGES); j < issued; ++j)
          wdrain(bar(C::B_KFULL + j % C::STAGES), (j / C::STAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_s > 0) {
      bool ok = wwait(bar(C::B_QFULL), 0, abort_flag);
      for (int j = 0; j < n_s && ok; ++j) {
        const int s = j % C::STAGES, x = j & 1;
        ok = wwait(bar(C::B_KFULL + s), (j / C::STAGES) & 1, abort_flag) &&
             (j < 2 || wwait(bar(C::B_SFREE + x), ((j - 2) >> 1) & 1, abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t k_stage = s_k + s * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          ptx::mma_ss(tmem + x * WBN, ptx::sdesc_sw128(s_q + koff, 16, 1024),
                      ptx::sdesc_sw128(k_stage + koff, 16, 1024), C::IDESC, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar(C::B_SFULL + x));
        ptx::mma_commit(bar(C::B_KEMPTY + s));
      }
      if (!ok) {  // every MMA already issued finishes before TMEM is released
        ptx::mma_commit(bar(C::B_DRAIN));
        wdrain(bar(C::B_DRAIN), 0);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- weights
    const int r = warp * 32 + lane;  // row within the tile = TMEM lane
    const int i = row0 + r;
    const bool row_valid = i < p.n_q;
    const float lse_i = row_valid ? p.lse[(size_t)bh * p.n_q + i] : -INFINITY;
    const bool any_legal = lse_i > -INFINITY;  // -inf: the row has no legal key
    const float l2 = lse_i * 1.4426950408889634f;
    const int lim = causal ? min(kv_len, i + 1) : kv_len;  // legal keys of row i: [0, lim)
    const bool vec = (p.n_k & 3) == 0;  // rows start on 16-byte boundaries
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // this warp's 32 rows: the store of row rr (0..31) goes to w + (first + rr) * n_k
    const int warp_row0 = row0 + warp * 32;
    const int rows_here = max(0, min(32, p.n_q - warp_row0));
    float* wbase = p.w + ((size_t)bh * p.n_q + (size_t)min(warp_row0, p.n_q - 1)) * p.n_k;
    uint8_t* stg = smem + C::OFF_STG + warp * C::STG_BYTES;
    // 32 columns [c0, c0 + cols) of this warp's rows from the staging block, row-contiguous
    auto flush_block = [&](int c0, int cols) {
      __syncwarp();
      if (vec && cols == 32) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int rr = 4 * t + (lane >> 3), v = lane & 7;
          const float4 val = *reinterpret_cast<const float4*>(stg + rr * 128 + ((v ^ (rr & 7)) << 4));
          if (rr < rows_here) *reinterpret_cast<float4*>(wbase + (size_t)rr * p.n_k + c0 + 4 * v) = val;
        }
      } else {
        for (int rr = 0; rr < rows_here; ++rr) {
          const float val = *reinterpret_cast<const float*>(stg + rr * 128 + (((lane >> 2) ^ (rr & 7)) << 4) +
                                                             (lane & 3) * 4);
          if (lane < cols) wbase[(size_t)rr * p.n_k + c0 + lane] = val;
        }
      }
      __syncwarp();
    };
    bool ok = true;
    for (int j = 0; j < n_s; ++j) {
      const int x = j & 1;
      ok = __all_sync(0xffffffffu, wwait(bar(C::B_SFULL + x), (j >> 1) & 1, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) ptx::tmem_ld32(tmem + lane_off + x * WBN + q4 * 32, sr[q4]);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_SFREE + x));  // the buffer may take S(j+2)
      if (rows_here == 0) continue;  // warp-uniform
      const int j0 = j * WBN;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int c0 = j0 + q4 * 32;
        if (c0 >= p.n_k) break;
        float pv[32];
#pragma unroll
        for (int x2 = 0; x2 < 32; ++x2) {
          const int key = c0 + x2;
          pv[x2] = (any_legal && key < lim) ? ptx::ex2(__uint_as_float(sr[q4][x2]) * p.c - l2) : 0.0f;
        }
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<float4*>(stg + lane * 128 + ((v ^ (lane & 7)) << 4)) =
              make_float4(pv[4 * v], pv[4 * v + 1], pv[4 * v + 2], pv[4 * v + 3]);
        flush_block(c0, min(32, p.n_k - c0));
      }
    }
    // keys of tiles no row may see: weight 0, row-contiguous
    if (ok && rows_here > 0) {
      const int z0 = n_s * WBN;
      if (vec) {
        for (int rr = 0; rr < rows_here; ++rr)
          for (int c4 = z0 + 4 * lane; c4 < p.n_k; c4 += 128)
            *reinterpret_cast<float4*>(wbase + (size_t)rr * p.n_k + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        for (int rr = 0; rr < rows_here; ++rr)
          for (int c1 = z0 + lane; c1 < p.n_k; c1 += 32) wbase[(size_t)rr * p.n_k + c1] = 0.0f;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// [B*h, n, d] bf16: the map spans (d, n, B*h); boxes of 64 columns x 128 rows, 128-byte swizzle.
CUresult encode_w(PFN_encodeTiled enc, CUtensorMap* map, const void* base, int d, int n, int bh) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)n};
  cuuint32_t box[3] = {64, (cuuint32_t)WBM, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int D>
int launch_w(const WeightsArgs& a, PFN_encodeTiled enc) {
  using C = WCfg<D>;
  CUtensorMap mq, mk;
  if (encode_w(enc, &mq, a.q, D, a.n_q, a.B * a.H) != CUDA_SUCCESS ||
      encode_w(enc, &mk, a.k, D, a.n_k, a.B * a.H) != CUDA_SUCCESS)
    return ATTN_ERR_UNSUPPORTED;
  static std::atomic<bool> attr_done[kMaxDevicesW];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesW) return ATTN_ERR_CUDA;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(attn_weights_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  WParams p;
  p.w = a.w;
  p.lse = a.lse;
  p.key_lens = a.key_lens;
  p.H = a.H;
  p.n_q = a.n_q;
  p.n_k = a.n_k;
  p.mask_mode = a.mask_mode;
  p.num_qblocks = (a.n_q + WBM - 1) / WBM;
  p.c = (float)((double)a.scale * 1.4426950408889634074);
  const long long grid = (long long)a.B * a.H * p.num_qblocks;
  if (grid > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  attn_weights_kernel<D><<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(mq, mk, p);
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int launch_attn_weights(const WeightsArgs& a, PFN_encodeTiled enc) {
  if (a.d == 64) return launch_w<64>(a, enc);
  if (a.d == 128) return launch_w<128>(a, enc);
  return ATTN_ERR_UNSUPPORTED;
}

int read_weights_fault_word(int clear, uint32_t* out) {
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_weights_fault_word, sizeof w) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_weights_fault_word, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  *out = w;
  return ATTN_OK;
}

}  // namespace attn
