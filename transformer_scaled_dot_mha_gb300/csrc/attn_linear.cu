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
// then come from L2. Launches of many tiles pair the SMs: two CTAs of a cluster
// compute a 256 x 256 tile with the 2-SM MMA (tcgen05.mma.cta_group::2), each holding
// half of the operands. Per CTA, 192 threads:
//   warp 0      TMA producer: per 64-wide K step one 128 x 64 tile of X (K-major)
//               and four 64 x 64 boxes of W (MN-major; the pair: this CTA's two),
//               128-byte swizzled, into a ring of 48 KB stages (four; the pair: six
//               of 32 KB);
//   warp 1      allocates the 512 TMEM columns; one thread issues the MMAs: four
//               M128 N256 K16 tcgen05.mma per K step (the pair: M256 N256 from CTA 0)
//               into one of two 256-column fp32 accumulators, and releases each ring
//               stage with a commit;
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

constexpr int BM = 128;                            // output rows per CTA tile (= TMEM lanes)
constexpr int BN = 256;                            // output columns per tile
constexpr int BK = 64;                             // K per ring stage (one 128-byte swizzle row)
constexpr int A_BYTES = BM * BK * 2;               // 16 KB
constexpr int B_BOX_BYTES = BK * 64 * 2;           // 8 KB: 64 K rows x 64 columns
constexpr int STG_BYTES = 32 * 64 * 2;             // one 32-row x 64-column bf16 slab
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;

// Shared-memory plan. PAIR: the two CTAs of a cluster run one M256 N256 MMA on the
// tensor cores of both SMs (tcgen05.mma.cta_group::2): each CTA holds its 128 rows of X
// and its 128 columns of W, so a ring stage is 32 KB instead of 48 and there are six.
template <bool PAIR>
struct LCfg {
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int B_BYTES = (PAIR ? BN / 2 / 64 : BN / 64) * B_BOX_BYTES;  // 16 or 32 KB
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_STG = OFF_B + STAGES * B_BYTES;  // two slabs per epilogue warp
  static constexpr int OFF_BAR = OFF_STG + 4 * 2 * STG_BYTES;
  static constexpr int B_FULL = 0, B_EMPTY = STAGES, B_ACC_FULL = 2 * STAGES, B_ACC_EMPTY = 2 * STAGES + 2,
                       B_DRAIN = 2 * STAGES + 4;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4;
  // X K-major, W MN-major; the pair's MMA spans both CTAs' 128 rows
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, true);
  static constexpr uint32_t IDESC_HALF = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN / 2, true);  // a half tile
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};
constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr uint32_t FAULT_LINEAR = 128;
// Launches of at least this many 128 x 256 tiles run the 2-SM MMA (PAIR).
constexpr long long kPairMinTiles = 512;

// ---- the pair's instructions (cta_group::2). TMEM is allocated collectively: one warp
// of each CTA of the pair runs the same alloc / relinquish / dealloc, and both receive
// the same column address. The MMA is issued from the even CTA; operand A (128 rows per
// CTA) and B (128 columns per CTA) are read at the same shared-memory offsets in both
// CTAs, and the accumulator's rows 128 r .. 128 r + 127 land in CTA r's TMEM lanes.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem_slot), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// Arrives once on the barrier at offset `bar` of every CTA in cta_mask when the pair
// MMAs this thread issued before it have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
// A box into this CTA's shared memory, counted on a barrier of either CTA of the pair
// (`bar` a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, uint32_t bar, int x, int y,
                                                 uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "l"(cache_hint)
      : "memory");
}
// The shared::cluster address of offset `addr` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrival on a barrier of another CTA of the cluster, ordered after this thread's
// earlier memory operations at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

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
  int total_tiles;  // a row block (a pair: two) x one column block each
  int split_from;   // the walk's items from here on are half tiles, two per tile
  int total_items;
  int interleave;  // all problems share M and N: list order (row unit, problem, column block)
};

// Item `it` of the walk -> its tile; half = -1 for the whole 256-column tile, else 0 or
// 1 for its columns [0, 128) or [128, 256). The tiles of a last, partly filled round of
// the grid are split in two, so that round takes half as long on twice as many SMs.
__device__ __forceinline__ int item_tile(const LinParams& p, int it, int& half) {
  if (it < p.split_from) {
    half = -1;
    return it;
  }
  const int h = it - p.split_from;
  half = h & 1;
  return p.split_from + (h >> 1);
}

// cluster: acquire at cluster scope (arrivals that come from the other CTA of a pair)
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         bool cluster = false) {
  auto probe = [&]() { return cluster ? mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (probe()) return true;
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

// Tile t of the list -> problem z, row unit mu (one row block; a pair: two), column block nb.
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

// PAIR: clusters of two CTAs; the pair computes the 256 x 256 tile of row blocks 2u and
// 2u + 1 with one MMA stream issued by CTA 0 on both SMs. Each CTA loads its own X rows
// and its half of the W columns, so per 64-deep K step an SM receives 32 KB and its
// tensor core reads 32 KB (one CTA alone: 48 and 48 for the same MMA work). Every load
// is counted on CTA 0's full barrier, which expects both CTAs' bytes; CTA 0's commits
// release the ring stage in both CTAs and hand each CTA its accumulator rows; both
// CTAs' epilogues return an accumulator to CTA 0's empty barrier; cluster barriers
// bracket the CTAs' lives.
template <bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    attn_linear_kernel(const __grid_constant__ CUtensorMap tm_x0, const __grid_constant__ CUtensorMap tm_w0,
                       const __grid_constant__ CUtensorMap tm_y0, const __grid_constant__ CUtensorMap tm_x1,
                       const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_y1,
                       const __grid_constant__ CUtensorMap tm_x2, const __grid_constant__ CUtensorMap tm_w2,
                       const __grid_constant__ CUtensorMap tm_y2, const __grid_constant__ LinParams p) {
  constexpr int CL = PAIR ? 2 : 1;  // CTAs per cluster
  using C = LCfg<PAIR>;
  constexpr int STAGES = C::STAGES, B_BYTES = C::B_BYTES;
  constexpr int B_FULL = C::B_FULL, B_EMPTY = C::B_EMPTY, B_ACC_FULL = C::B_ACC_FULL, B_ACC_EMPTY = C::B_ACC_EMPTY,
                B_DRAIN = C::B_DRAIN;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((ptx::smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(&g_linear_fault_word, FAULT_LINEAR);
    return;
  }
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t s_a = s_base + C::OFF_A, s_b = s_base + C::OFF_B;
  auto bar = [&](int i) -> uint32_t { return s_base + C::OFF_BAR + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(B_FULL + s), 1);
      // one commit from the MMA issuer (PAIR: CTA 0's, multicast to both CTAs)
      ptx::mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(B_ACC_FULL + b), 1);
      // every epilogue thread arrives (PAIR: those of both CTAs, on CTA 0's barrier)
      ptx::mbar_init(bar(B_ACC_EMPTY + b), (PAIR ? 2 : 1) * 4 * 32);
    }
    ptx::mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
      ptx::tmem_relinquish();
    }
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
  if constexpr (PAIR) ptx::cluster_sync();  // the peer's barriers exist before any remote arrival
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::grid_dep_wait();  // X may be the previous grid's output
  ptx::grid_dep_launch();
  const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
  const int unit0 = (int)(blockIdx.x / CL), units_step = (int)(gridDim.x / CL);
  constexpr uint16_t kPeers = (uint16_t)((1u << CL) - 1);

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_last();  // X rows and W are each read by several CTAs
      uint32_t it = 0;
      bool ok = true;
      for (int i = unit0; i < p.total_items && ok; i += units_step) {
        int z, mu, nb, half;
        tile_of(p, item_tile(p, i, half), z, mu, nb);
        const int mb = mu * CL + rank;
        const int col_base = nb * BN + (half > 0 ? BN / 2 : 0);
        const int boxes = (half >= 0 ? BN / 2 : BN) / CL / 64;  // W boxes this CTA loads per K step
        const CUtensorMap* tx = z == 0 ? &tm_x0 : z == 1 ? &tm_x1 : &tm_x2;
        const CUtensorMap* tw = z == 0 ? &tm_w0 : z == 1 ? &tm_w1 : &tm_w2;
        const int k_steps = (p.pr[z].K + BK - 1) / BK;
        for (int kb = 0; kb < k_steps; ++kb, ++it) {
          const int s = it % STAGES;
          if (!wait_bar(bar(B_EMPTY + s), ((it / STAGES) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (PAIR) {  // both CTAs' boxes counted on CTA 0's barrier
            const uint32_t full0 = cluster_addr(bar(B_FULL + s), 0);
            if (rank == 0) ptx::mbar_arrive_expect_tx(bar(B_FULL + s), 2 * (A_BYTES + boxes * B_BOX_BYTES));
            tma_load_2d_pair(s_a + s * A_BYTES, tx, full0, kb * BK, mb * BM, pol);
            for (int c = 0; c < boxes; ++c)
              tma_load_2d_pair(s_b + s * B_BYTES + c * B_BOX_BYTES, tw, full0, col_base + (rank * boxes + c) * 64,
                               kb * BK, pol);
            continue;
          }
          ptx::mbar_arrive_expect_tx(bar(B_FULL + s), A_BYTES + boxes * B_BOX_BYTES);
          ptx::tma_load_2d(s_a + s * A_BYTES, tx, bar(B_FULL + s), kb * BK, mb * BM, pol);
          for (int c = 0; c < boxes; ++c)
            ptx::tma_load_2d(s_b + s * B_BYTES + c * B_BOX_BYTES, tw, bar(B_FULL + s), col_base + c * 64, kb * BK, pol);
        }
      }
      if (!ok && (!PAIR || rank == 0)) {
        // copies still in flight must land before this CTA's shared memory goes away
        // (PAIR: CTA 0's barriers count the copies of both CTAs)
        for (uint32_t x = it > STAGES ? it - STAGES : 0; x < it; ++x)
          drain_wait(bar(B_FULL + x % STAGES), (x / STAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {
      uint32_t it = 0;
      int lt = 0;
      bool ok = true;
      for (int i = unit0; i < p.total_items && ok; i += units_step, ++lt) {
        int z, mu, nb, half;
        tile_of(p, item_tile(p, i, half), z, mu, nb);
        const uint32_t idesc = half >= 0 ? C::IDESC_HALF : C::IDESC;
        const int buf = lt & 1;
        ok = wait_bar(bar(B_ACC_EMPTY + buf), ((lt >> 1) & 1) ^ 1, abort_flag, PAIR);
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
          for (int kk = 0; kk < BK / 16; ++kk) {  // 16 K = 32 bytes of an X row = 16 rows of W
            const uint64_t ad = ptx::sdesc_sw128(a_st + kk * 32, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(b_st + kk * 2048, B_BOX_BYTES, 1024);
            if constexpr (PAIR)
              mma_ss_pair(d, ad, bd, idesc, (kb | kk) ? 1u : 0u);
            else
              ptx::mma_ss(d, ad, bd, idesc, (kb | kk) ? 1u : 0u);
          }
          if constexpr (PAIR)
            mma_commit_pair(bar(B_EMPTY + s), kPeers);
          else
            ptx::mma_commit(bar(B_EMPTY + s));
        }
        if (!ok) break;
        if constexpr (PAIR)
          mma_commit_pair(bar(B_ACC_FULL + buf), kPeers);
        else
          ptx::mma_commit(bar(B_ACC_FULL + buf));
      }
      if (!ok) {
        // let every MMA already issued finish before TMEM is released
        if constexpr (PAIR)
          mma_commit_pair(bar(B_DRAIN), 1);
        else
          ptx::mma_commit(bar(B_DRAIN));
        drain_wait(bar(B_DRAIN), 0);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may read
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t stg = s_base + C::OFF_STG + (warp - 2) * 2 * STG_BYTES;
    int sb = 0;  // staging slab to fill next
    int lt = 0;
    for (int i = unit0; i < p.total_items; i += units_step, ++lt) {
      int z, mu, nb, half;
      tile_of(p, item_tile(p, i, half), z, mu, nb);
      const int mb = mu * CL + rank;
      const int col_base = nb * BN + (half > 0 ? BN / 2 : 0);
      const int buf = lt & 1;
      if (!__all_sync(0xffffffffu, wait_bar(bar(B_ACC_FULL + buf), (lt >> 1) & 1, abort_flag))) break;
      ptx::tc_fence_after();
      const LinProblem& P = p.pr[z];
      const CUtensorMap* ty = z == 0 ? &tm_y0 : z == 1 ? &tm_y1 : &tm_y2;
      // rows of this warp's slabs inside Y (the second CTA of a pair can lie wholly past M)
      const bool row_ok = mb * BM + quarter * 32 < P.M;
#pragma unroll 1
      for (int c = 0; c < (half >= 0 ? BN / 2 : BN) / 64; ++c) {
        uint32_t v[64];
        ptx::tmem_ld32(tmem + lane_off + buf * BN + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        ptx::tmem_ld32(tmem + lane_off + buf * BN + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        ptx::tmem_wait_ld();
        const int col0 = col_base + c * 64;
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
      if (PAIR && rank != 0)
        mbar_arrive_remote(cluster_addr(bar(B_ACC_EMPTY + buf), 0));
      else
        ptx::mbar_arrive(bar(B_ACC_EMPTY + buf));
    }
    if (lane == 0) ptx::bulk_wait0();  // every store has landed before the CTA exits
    __syncwarp();
  }

  // ---- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();  // no CTA leaves while its peer may still write to it
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, TMEM_COLS);
    else
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

// Persistent grid of clusters (PAIR: two CTAs, else one): as many as can be resident.
template <bool PAIR>
int resident_clusters(int dev) {
  constexpr int CL = PAIR ? 2 : 1;
  static std::atomic<int> cached[kMaxDevices];
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (CL == 1) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * 64);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = LCfg<PAIR>::SMEM_BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, attn_linear_kernel<PAIR>, &cfg) != cudaSuccess) return 0;
  }
  if (n <= 0) return 0;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <bool PAIR>
int launch_linear_cl(const LinearJob* jobs, int n_jobs, PFN_encodeTiled enc, cudaStream_t stream, int dev) {
  constexpr int CL = PAIR ? 2 : 1;
  constexpr int SMEM_BYTES = LCfg<PAIR>::SMEM_BYTES;
  static std::atomic<bool> attr_done[kMaxDevices];
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(attn_linear_kernel<PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int clusters = resident_clusters<PAIR>(dev);
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
    if (tiles > 0x7fff0000LL) return ATTN_ERR_UNSUPPORTED;  // room for the split items
    same = same && j.M == jobs[0].M && j.N == jobs[0].N;
  }
  for (int z = n_jobs; z < 3; ++z) {  // unused slots repeat the first problem's maps
    mx[z] = mx[0];
    mw[z] = mw[0];
    my[z] = my[0];
    p.pr[z] = p.pr[0];
  }
  p.total_tiles = (int)tiles;
  // a last round of the grid that is partly filled: split its tiles when their halves
  // fit in one round
  const long long rem = tiles % clusters;
  p.split_from = (int)((rem > 0 && 2 * rem <= clusters) ? tiles - rem : tiles);
  p.total_items = p.split_from + 2 * (p.total_tiles - p.split_from);
  p.interleave = (n_jobs > 1 && same) ? 1 : 0;
  const int grid = CL * (p.total_items < clusters ? p.total_items : clusters);
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
  if (cudaLaunchKernelEx(&cfg, attn_linear_kernel<PAIR>, mx[0], mw[0], my[0], mx[1], mw[1], my[1], mx[2], mw[2],
                         my[2], p) != cudaSuccess)
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
  if (tiles >= kPairMinTiles) return launch_linear_cl<true>(jobs, n_jobs, enc, stream, dev);
  return launch_linear_cl<false>(jobs, n_jobs, enc, stream, dev);
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
