// attn_linear.cu -- the linear projections of the multi-head attention layer on the
// sm_103a tensor cores (TMA + tcgen05 + TMEM):
//
//   Y[M, N] = X[M, K] W[K, N] (+ b[N])     bf16 in and out, fp32 accumulation
//
// The multi-head layer projects its inputs with per-head matrices and its
// concatenated heads with W^O: MultiHead(Q,K,V) = Concat(head_1..head_h) W^O with
// head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V) (vlmlib.cn paper summary, "multi-head
// attention"); the csdn blog's MultiHeadAttention does the same with nn.Linear layers
// (biases on). Stacking the h per-head matrices side by side makes each projection
// one GEMM whose column block i*d .. i*d + d - 1 is head i.
//
// Work decomposition. One launch computes up to three independent problems (the
// Q', K', V' projections share a launch). The output is cut into 128 x 256 tiles;
// a persistent grid of one CTA per SM walks the tile list in strides of the grid.
// When every problem has the same shape (self-attention: the three projections read
// the same rows of x) the list interleaves them -- (row block, problem, column
// block) -- so that the CTAs working at the same time read the same x rows, which
// then come from L2. Per CTA, 192 threads:
//   warp 0      TMA producer: per 64-wide K step one 128 x 64 tile of X (K-major)
//               and four 64 x 64 boxes of W (MN-major), 128-byte swizzled, into a
//               four-stage ring (48 KB per stage);
//   warp 1      allocates the 512 TMEM columns; one thread issues the MMAs: four
//               M128 N256 K16 tcgen05.mma per K step into one of two 256-column
//               fp32 accumulators, and releases each ring stage with a commit;
//   warps 2-5   epilogue (thread = output row = TMEM lane): load the accumulator
//               64 columns at a time, add the bias in fp32, round to bf16 (nearest
//               even), write the warp's 32 x 64 slab into one of its two 128-byte-
//               swizzled staging buffers and store it with one TMA tensor store
//               (coalesced, tails clipped by the tensor map); then hand the
//               accumulator back, so that it drains while the MMAs fill the other.
// Every mbarrier wait is bounded in time; a wait that runs out records a fault bit
// (attn_fault_status), raises the CTA's abort flag, and every role stops: the
// producer lets its copies in flight land, the issuer waits for its MMAs, TMEM is
// freed and the CTA returns. Nothing traps.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace attn {

__device__ unsigned int g_linear_fault_word;  // fault record of the projection kernel

namespace {

constexpr int BM = 128;                            // output rows per tile (= TMEM lanes)
constexpr int BN = 256;                            // output columns per tile
constexpr int BK = 64;                             // K per ring stage (one 128-byte swizzle row)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;               // 16 KB
constexpr int B_BOX_BYTES = BK * 64 * 2;           // 8 KB: 64 K rows x 64 columns
constexpr int B_BYTES = (BN / 64) * B_BOX_BYTES;   // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int STG_BYTES = 32 * 64 * 2;             // one 32-row x 64-column bf16 slab
constexpr int OFF_STG = OFF_B + STAGES * B_BYTES;  // two slabs per epilogue warp
constexpr int OFF_BAR = OFF_STG + 4 * 2 * STG_BYTES;
constexpr int B_FULL = 0, B_EMPTY = STAGES, B_ACC_FULL = 2 * STAGES, B_ACC_EMPTY = 2 * STAGES + 2,
              B_DRAIN = 2 * STAGES + 4;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN, true);  // X K-major, W MN-major
constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr uint32_t FAULT_LINEAR = 128;
// Launches of at least this many 128 x 256 tiles run as 2-CTA clusters sharing each W
// tile (same-box A/B: +5-6 % on 16384 x 2048 x 2048 and on the three Q/K/V projections
// at 16384 x 1024; -2 % on a single 16384 x 1024 x 1024 projection of 512 tiles).
constexpr long long kClusterMinTiles = 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct LinProblem {
  uint16_t* y;
  const uint16_t* bias;  // nullptr: no bias
  int M, N, K;
  int n_blocks;    // column blocks of 256
  int tile_begin;  // first tile of this problem in the list (z-major order)
};

struct LinParams {
  LinProblem pr[3];
  int n_prob;
  int total_tiles;  // units of CL row blocks x one column block
  int interleave;  // all problems share M and N: list order (row unit, problem, column block)
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
        atomicOr(&g_linear_fault_word, FAULT_LINEAR);
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

// Tile t of the list -> problem z, row unit mu (CL row blocks), column block nb.
__device__ __forceinline__ void tile_of(const LinParams& p, int t, int& z, int& mb, int& nb) {
  if (p.interleave) {
    const int nbk = p.pr[0].n_blocks;
    const int per_m = p.n_prob * nbk;
    mb = t / per_m;
    const int r = t - mb * per_m;
    z = r / nbk;
    nb = r - z * nbk;
  } else {
    z = (p.n_prob > 2 && t >= p.pr[2].tile_begin) ? 2 : (p.n_prob > 1 && t >= p.pr[1].tile_begin) ? 1 : 0;
    const int r = t - p.pr[z].tile_begin;
    mb = r / p.pr[z].n_blocks;
    nb = r - mb * p.pr[z].n_blocks;
  }
}

// CL: CTAs per cluster. With CL = 2 the two CTAs of a cluster take row blocks 2u and
// 2u + 1 of the same column block: each loads its own X rows and half of the W tile,
// multicast into both CTAs, so each CTA's L2 traffic per K step drops from 48 to 32 KB.
// A ring stage is then free only once both CTAs' MMAs have read it (the issuers commit
// to the stage's barrier in both CTAs), and cluster barriers bracket the CTAs' lives.
template <int CL>
__global__ void __launch_bounds__(THREADS, 1)
    attn_linear_kernel(const __grid_constant__ CUtensorMap tm_x0, const __grid_constant__ CUtensorMap tm_w0,
                       const __grid_constant__ CUtensorMap tm_y0, const __grid_constant__ CUtensorMap tm_x1,
                       const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_y1,
                       const __grid_constant__ CUtensorMap tm_x2, const __grid_constant__ CUtensorMap tm_w2,
                       const __grid_constant__ CUtensorMap tm_y2, const __grid_constant__ LinParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((ptx::smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(&g_linear_fault_word, FAULT_LINEAR);
    return;
  }
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t s_a = s_base + OFF_A, s_b = s_base + OFF_B;
  auto bar = [&](int i) -> uint32_t { return s_base + OFF_BAR + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM_SLOT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(B_FULL + s), 1);
      ptx::mbar_init(bar(B_EMPTY + s), CL);  // one commit from the MMA issuer of each CTA of the cluster
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(B_ACC_FULL + b), 1);
      ptx::mbar_init(bar(B_ACC_EMPTY + b), 4 * 32);  // every epilogue thread arrives
    }
    ptx::mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_x0);
    ptx::prefetch_tmap(&tm_w0);
    ptx::prefetch_tmap(&tm_y0);
    if (p.n_prob > 1) {
      ptx::prefetch_tmap(&tm_x1);
      ptx::prefetch_tmap(&tm_w1);
      ptx::prefetch_tmap(&tm_y1);
    }
    if (p.n_prob > 2) {
      ptx::prefetch_tmap(&tm_x2);
      ptx::prefetch_tmap(&tm_w2);
      ptx::prefetch_tmap(&tm_y2);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) ptx::cluster_sync();  // the peer's barriers exist before any multicast
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::grid_dep_wait();  // X may be the previous grid's output
  ptx::grid_dep_launch();
  const int rank = CL > 1 ? (int)ptx::cluster_ctarank() : 0;
  const int unit0 = (int)(blockIdx.x / CL), units_step = (int)(gridDim.x / CL);
  constexpr uint16_t kPeers = (uint16_t)((1u << CL) - 1);

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_last();  // X rows and W are each read by several CTAs
      uint32_t it = 0;
      bool ok = true;
      for (int t = unit0; t < p.total_tiles && ok; t += units_step) {
        int z, mu, nb;
        tile_of(p, t, z, mu, nb);
        const int mb = mu * CL + rank;
        const CUtensorMap* tx = z == 0 ? &tm_x0 : z == 1 ? &tm_x1 : &tm_x2;
        const CUtensorMap* tw = z == 0 ? &tm_w0 : z == 1 ? &tm_w1 : &tm_w2;
        const int k_steps = (p.pr[z].K + BK - 1) / BK;
        for (int kb = 0; kb < k_steps; ++kb, ++it) {
          const int s = it % STAGES;
          if (!wait_bar(bar(B_EMPTY + s), ((it / STAGES) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(bar(B_FULL + s), A_BYTES + B_BYTES);
          ptx::tma_load_2d(s_a + s * A_BYTES, tx, bar(B_FULL + s), kb * BK, mb * BM, pol);
          if constexpr (CL == 1) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              ptx::tma_load_2d(s_b + s * B_BYTES + c * B_BOX_BYTES, tw, bar(B_FULL + s), nb * BN + c * 64, kb * BK,
                               pol);
          } else {  // this CTA's share of the W boxes, into every CTA of the cluster
#pragma unroll
            for (int c = rank * (BN / 64 / CL); c < (rank + 1) * (BN / 64 / CL); ++c)
              ptx::tma_load_2d_mc(s_b + s * B_BYTES + c * B_BOX_BYTES, tw, bar(B_FULL + s), nb * BN + c * 64,
                                  kb * BK, kPeers, pol);
          }
        }
      }
      if (!ok) {
        // copies still in flight must land before this CTA's shared memory goes away
        for (uint32_t x = it > STAGES ? it - STAGES : 0; x < it; ++x)
          drain_wait(bar(B_FULL + x % STAGES), (x / STAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      int lt = 0;
      bool ok = true;
      for (int t = unit0; t < p.total_tiles && ok; t += units_step, ++lt) {
        int z, mu, nb;
        tile_of(p, t, z, mu, nb);
        const int buf = lt & 1;
        ok = wait_bar(bar(B_ACC_EMPTY + buf), ((lt >> 1) & 1) ^ 1, abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        const int k_steps = (p.pr[z].K + BK - 1) / BK;
        for (int kb = 0; kb < k_steps; ++kb, ++it) {
          const int s = it % STAGES;
          ok = wait_bar(bar(B_FULL + s), (it / STAGES) & 1, abort_flag);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t a_st = s_a + s * A_BYTES, b_st = s_b + s * B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // 16 K = 32 bytes of an X row = 16 rows of W
            ptx::mma_ss(d, ptx::sdesc_sw128(a_st + kk * 32, 16, 1024),
                        ptx::sdesc_sw128(b_st + kk * 2048, B_BOX_BYTES, 1024), IDESC, (kb | kk) ? 1u : 0u);
          if constexpr (CL == 1)
            ptx::mma_commit(bar(B_EMPTY + s));
          else
            ptx::mma_commit_mc(bar(B_EMPTY + s), kPeers);
        }
        if (!ok) break;
        ptx::mma_commit(bar(B_ACC_FULL + buf));
      }
      if (!ok) {
        // let every MMA already issued finish before TMEM is released
        ptx::mma_commit(bar(B_DRAIN));
        drain_wait(bar(B_DRAIN), 0);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may read
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t stg = s_base + OFF_STG + (warp - 2) * 2 * STG_BYTES;
    int sb = 0;  // staging slab to fill next
    int lt = 0;
    for (int t = unit0; t < p.total_tiles; t += units_step, ++lt) {
      int z, mu, nb;
      tile_of(p, t, z, mu, nb);
      const int mb = mu * CL + rank;
      const int buf = lt & 1;
      if (!__all_sync(0xffffffffu, wait_bar(bar(B_ACC_FULL + buf), (lt >> 1) & 1, abort_flag))) break;
      ptx::tc_fence_after();
      const LinProblem& P = p.pr[z];
      const CUtensorMap* ty = z == 0 ? &tm_y0 : z == 1 ? &tm_y1 : &tm_y2;
      // rows of this warp's slabs inside Y (the second CTA of a pair can lie wholly past M)
      const bool row_ok = mb * BM + quarter * 32 < P.M;
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t v[64];
        ptx::tmem_ld32(tmem + lane_off + buf * BN + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        ptx::tmem_ld32(tmem + lane_off + buf * BN + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        ptx::tmem_wait_ld();
        const int col0 = nb * BN + c * 64;
        if (col0 < P.N && row_ok) {
          uint32_t w[32];
#pragma unroll
          for (int x = 0; x < 8; ++x) {  // eight columns (one 16-byte bias piece) at a time
            uint4 bw = make_uint4(0, 0, 0, 0);
            if (P.bias && col0 + 8 * x < P.N) bw = __ldg(reinterpret_cast<const uint4*>(P.bias + col0) + x);
            const uint32_t b4[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[4 * x + e] = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 2 * e]) + __uint_as_float(b4[e] << 16),
                                              __uint_as_float(v[8 * x + 2 * e + 1]) +
                                                  __uint_as_float(b4[e] & 0xffff0000u));
          }
          // the slab is free once the store issued from it two rounds ago has read it
          if (lane == 0) ptx::bulk_wait_read1();
          __syncwarp();
          const uint32_t slab = stg + sb * STG_BYTES;
#pragma unroll
          for (int x = 0; x < 8; ++x)  // 128-byte swizzle: 16-byte piece x of row r goes to x ^ (r & 7)
            ptx::st_shared_v4(slab + lane * 128 + ((x ^ (lane & 7)) << 4), w[4 * x], w[4 * x + 1], w[4 * x + 2],
                              w[4 * x + 3]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(ty, slab, col0, mb * BM + quarter * 32);
            ptx::bulk_commit();
          }
          sb ^= 1;
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(B_ACC_EMPTY + buf));
    }
    if (lane == 0) ptx::bulk_wait0();  // every store has landed before the CTA exits
    __syncwarp();
  }

  // ---- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) ptx::cluster_sync();  // no CTA leaves while its peer may still write to it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// X [M, K] row-major: the map spans (K, M), box 64 x 128.
CUresult encode_x(PFN_encodeTiled enc, CUtensorMap* map, const void* base, int M, int K) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {BK, BM};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Y [M, N] row-major, stored by the epilogue: the map spans (N, M), box 64 x 32.
CUresult encode_y(PFN_encodeTiled enc, CUtensorMap* map, const void* base, int M, int N) {
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// W [K, N] row-major: the map spans (N, K), box 64 x 64.
CUresult encode_w(PFN_encodeTiled enc, CUtensorMap* map, const void* base, int K, int N) {
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {64, BK};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Persistent grid of CL-CTA clusters: as many as can be resident at once.
template <int CL>
int resident_clusters(int dev) {
  static std::atomic<int> cached[kMaxDevices];
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (CL == 1) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * 64);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, attn_linear_kernel<CL>, &cfg) != cudaSuccess) return 0;
  }
  if (n <= 0) return 0;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int CL>
int launch_linear_cl(const LinearJob* jobs, int n_jobs, PFN_encodeTiled enc, cudaStream_t stream, int dev) {
  static std::atomic<bool> attr_done[kMaxDevices];
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(attn_linear_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int clusters = resident_clusters<CL>(dev);
  if (clusters <= 0) return ATTN_ERR_CUDA;
  CUtensorMap mx[3], mw[3], my[3];
  LinParams p{};
  p.n_prob = n_jobs;
  long long tiles = 0;
  bool same = true;
  for (int z = 0; z < n_jobs; ++z) {
    const LinearJob& j = jobs[z];
    if (encode_x(enc, &mx[z], j.x, j.M, j.K) != CUDA_SUCCESS || encode_w(enc, &mw[z], j.w, j.K, j.N) != CUDA_SUCCESS ||
        encode_y(enc, &my[z], j.y, j.M, j.N) != CUDA_SUCCESS)
      return ATTN_ERR_UNSUPPORTED;
    LinProblem& P = p.pr[z];
    P.y = static_cast<uint16_t*>(j.y);
    P.bias = static_cast<const uint16_t*>(j.bias);
    P.M = j.M;
    P.N = j.N;
    P.K = j.K;
    P.n_blocks = (j.N + BN - 1) / BN;
    P.tile_begin = (int)tiles;
    const long long m_units = ((long long)(j.M + BM - 1) / BM + CL - 1) / CL;
    tiles += m_units * P.n_blocks;
    if (tiles > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    same = same && j.M == jobs[0].M && j.N == jobs[0].N;
  }
  for (int z = n_jobs; z < 3; ++z) {  // unused slots repeat the first problem's maps
    mx[z] = mx[0];
    mw[z] = mw[0];
    my[z] = my[0];
    p.pr[z] = p.pr[0];
  }
  p.total_tiles = (int)tiles;
  p.interleave = (n_jobs > 1 && same) ? 1 : 0;
  const int grid = CL * (int)(tiles < clusters ? tiles : clusters);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, attn_linear_kernel<CL>, mx[0], mw[0], my[0], mx[1], mw[1], my[1], mx[2], mw[2], my[2],
                         p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int launch_linear(const LinearJob* jobs, int n_jobs, PFN_encodeTiled enc, cudaStream_t stream) {
  if (n_jobs < 1 || n_jobs > 3) return ATTN_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  long long tiles = 0;
  for (int z = 0; z < n_jobs; ++z)
    tiles += (long long)((jobs[z].M + BM - 1) / BM) * ((jobs[z].N + BN - 1) / BN);
  if (tiles >= kClusterMinTiles) return launch_linear_cl<2>(jobs, n_jobs, enc, stream, dev);
  return launch_linear_cl<1>(jobs, n_jobs, enc, stream, dev);
}

int read_linear_fault_word(int clear, uint32_t* out) {
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_linear_fault_word, sizeof w) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_linear_fault_word, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  *out = w;
  return ATTN_OK;
}

}  // namespace attn
