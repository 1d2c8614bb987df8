// attn_mha.cu -- the multi-head attention layer around the attention kernel:
//   Q' = x_q W^Q + b_Q,  K' = x_kv W^K + b_K,  V' = x_kv W^V + b_V      [B, n, h*d]
//   A  = Attention(Q', K', V') per head, written concatenated          [B, n_q, h*d]
//   Y  = A W^O + b_O                                                    [B, n_q, d_model]
// (vlmlib.cn "multi-head attention": MultiHead = Concat(head_1..head_h) W^O with
// head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V); the csdn blog's MultiHeadAttention.)
//
// The four projections are plain bf16 GEMMs with fp32 accumulation on cuBLASLt, the
// bias added in the GEMM epilogue. split_heads and the concatenation cost no copies:
// the attention kernel reads Q', K', V' and writes A in their [B, n, h*d] layout
// through its heads-interleaved tensor maps (head i = columns i*d .. i*d + d - 1).
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kLtWorkspaceBytes = 32u << 20;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// One GEMM shape: Y[M, N] = X[M, K] W[K, N] (+ bias[N]), all row-major bf16.
// cuBLASLt is column-major, so it computes Y^T (N x M) = W^T (N x K) X^T (K x M):
// the row-major arrays are exactly those column-major transposes, no op flags.
struct Plan {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t lw = nullptr, lx = nullptr, ly = nullptr;
  cublasLtMatmulAlgo_t algo{};
  bool ok = false;
};

struct DeviceState {
  std::mutex mu;
  cublasLtHandle_t handle = nullptr;
  std::map<std::tuple<long long, long long, long long, bool>, Plan> plans;
};

DeviceState g_state[kMaxDevices];

bool make_plan(cublasLtHandle_t handle, long long M, long long N, long long K, bool bias, Plan& pl) {
  if (cublasLtMatmulDescCreate(&pl.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return false;
  const cublasOperation_t no = CUBLAS_OP_N;
  cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_TRANSA, &no, sizeof no);
  cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_TRANSB, &no, sizeof no);
  if (bias) {
    const cublasLtEpilogue_t epi = CUBLASLT_EPILOGUE_BIAS;
    const int32_t bt = CUDA_R_16BF;
    // the heuristic reads only the pointer's alignment: promise 16 bytes, the
    // alignment the entry point requires of a bias
    const void* probe = reinterpret_cast<const void*>(uintptr_t(16));
    if (cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_EPILOGUE, &epi, sizeof epi) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_BIAS_DATA_TYPE, &bt, sizeof bt) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &probe, sizeof probe) !=
            CUBLAS_STATUS_SUCCESS)
      return false;
  }
  if (cublasLtMatrixLayoutCreate(&pl.lw, CUDA_R_16BF, N, K, N) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&pl.lx, CUDA_R_16BF, K, M, K) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&pl.ly, CUDA_R_16BF, N, M, N) != CUBLAS_STATUS_SUCCESS)
    return false;
  cublasLtMatmulPreference_t pref = nullptr;
  if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) return false;
  const size_t ws = kLtWorkspaceBytes;
  const uint32_t align16 = 16;
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws, sizeof ws);
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, &align16, sizeof align16);
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES, &align16, sizeof align16);
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, &align16, sizeof align16);
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES, &align16, sizeof align16);
  cublasLtMatmulHeuristicResult_t res{};
  int n_res = 0;
  const cublasStatus_t st =
      cublasLtMatmulAlgoGetHeuristic(handle, pl.op, pl.lw, pl.lx, pl.ly, pl.ly, pref, 1, &res, &n_res);
  cublasLtMatmulPreferenceDestroy(pref);
  if (st != CUBLAS_STATUS_SUCCESS || n_res < 1 || res.workspaceSize > kLtWorkspaceBytes) return false;
  pl.algo = res.algo;
  pl.ok = true;
  return true;
}

// Enqueues one projection on `stream`. Holds the device's lock while the bias
// pointer is set and the GEMM is enqueued (the plan is shared by host threads).
int gemm(DeviceState& ds, const void* x, const void* w, const void* bias, void* y, long long M, long long N,
         long long K, void* lt_ws, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(ds.mu);
  if (!ds.handle && cublasLtCreate(&ds.handle) != CUBLAS_STATUS_SUCCESS) {
    ds.handle = nullptr;
    return ATTN_ERR_CUDA;
  }
  const auto key = std::make_tuple(M, N, K, bias != nullptr);
  auto it = ds.plans.find(key);
  if (it == ds.plans.end()) {
    Plan pl;
    make_plan(ds.handle, M, N, K, bias != nullptr, pl);
    it = ds.plans.emplace(key, pl).first;
  }
  Plan& pl = it->second;
  if (!pl.ok) return ATTN_ERR_UNSUPPORTED;
  if (bias &&
      cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof bias) !=
          CUBLAS_STATUS_SUCCESS)
    return ATTN_ERR_CUDA;
  const float one = 1.0f, zero = 0.0f;
  const cublasStatus_t st = cublasLtMatmul(ds.handle, pl.op, &one, w, pl.lw, x, pl.lx, &zero, y, pl.ly, y, pl.ly,
                                           &pl.algo, lt_ws, kLtWorkspaceBytes, stream);
  return st == CUBLAS_STATUS_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

size_t mha_workspace_bytes(int B, int n_q, int n_k, int H, int d) {
  const size_t hd = (size_t)H * d * 2;
  return align_up((size_t)B * n_q * hd) * 2 + align_up((size_t)B * n_k * hd) * 2 + kLtWorkspaceBytes;
}

int launch_attn_mha(const MhaArgs& a, PFN_encodeTiled enc, void* workspace) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  DeviceState& ds = g_state[dev];
  const size_t hd = (size_t)a.H * a.d * 2;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* qp = base;
  uint8_t* kp = qp + align_up((size_t)a.B * a.n_q * hd);
  uint8_t* vp = kp + align_up((size_t)a.B * a.n_k * hd);
  uint8_t* ao = vp + align_up((size_t)a.B * a.n_k * hd);
  uint8_t* lt = ao + align_up((size_t)a.B * a.n_q * hd);
  const long long Mq = (long long)a.B * a.n_q, Mk = (long long)a.B * a.n_k, HD = (long long)a.H * a.d;
  int st;
  if ((st = gemm(ds, a.x_q, a.w_q, a.b_q, qp, Mq, HD, a.d_model, lt, a.stream)) != ATTN_OK) return st;
  if ((st = gemm(ds, a.x_kv, a.w_k, a.b_k, kp, Mk, HD, a.d_model, lt, a.stream)) != ATTN_OK) return st;
  if ((st = gemm(ds, a.x_kv, a.w_v, a.b_v, vp, Mk, HD, a.d_model, lt, a.stream)) != ATTN_OK) return st;
  TcArgs t{qp, kp, vp, ao, nullptr, a.B, a.H, a.n_q, a.n_k, a.d, a.scale, a.mask_mode, a.key_lens, a.stream, -1};
  t.heads_interleaved = 1;
  if ((st = launch_attn_tc(t, enc)) != ATTN_OK) return st;
  return gemm(ds, ao, a.w_o, a.b_o, a.out, Mq, a.d_model, HD, lt, a.stream);
}

}  // namespace attn
