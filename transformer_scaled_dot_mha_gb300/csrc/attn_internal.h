// attn_internal.h -- declarations shared by the host API and the kernels of
// libattn_gb300.so (not part of the public C ABI; see include/attn_gb300.h).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_gb300.h"

namespace attn {

// cuTensorMapEncodeTiled, fetched from the driver at run time (no -lcuda link).
typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Validated arguments of one bf16 call.
struct TcArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int B, H, n_q, n_k, d;
  float scale;
  int mask_mode;
  const int32_t* key_lens;
  cudaStream_t stream;
  int window;  // local-window radius (>= 0), or -1 for none
  int heads_interleaved = 0;  // 1: q, k, v, out are [B, n, H*d] instead of [B, H, n, d]
};

// Validated arguments of one attn_weights call.
struct WeightsArgs {
  const void* q;
  const void* k;
  const float* lse;
  float* w;
  int B, H, n_q, n_k, d;
  float scale;
  int mask_mode;
  const int32_t* key_lens;
  cudaStream_t stream;
};

// Validated arguments of one fp32 call.
struct F32Args {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;
  int B, H, n_q, n_k, d_k, d_v;
  float scale;
  int mask_mode;
  const int32_t* key_lens;
  cudaStream_t stream;
};

// Validated arguments of one decode step.
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int B, H, n_q, n_max, d;
  float scale;
  const int32_t* cache_lens;
  cudaStream_t stream;
};

// Validated arguments of one gradient call (d_k == d_v == d).
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* out;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int B, H, n_q, n_k, d;
  float scale;
  int mask_mode;
  const int32_t* key_lens;
  cudaStream_t stream;
  int flags = 0;    // ATTN_BWD_DETERMINISTIC
  int window = -1;  // local-window radius (>= 0), or -1 for none
};

// Validated arguments of one multi-head layer call (d_k == d_v == d).
struct MhaArgs {
  const void* x_q;
  const void* x_kv;
  const void* w_q;
  const void* b_q;
  const void* w_k;
  const void* b_k;
  const void* w_v;
  const void* b_v;
  const void* w_o;
  const void* b_o;
  void* out;
  int B, n_q, n_k, d_model, H, d;
  float scale;
  int mask_mode;
  const int32_t* key_lens;
  cudaStream_t stream;
};

// One projection Y[M, N] = X[M, K] W[K, N] (+ bias[N]), bf16, row-major, validated.
struct LinearJob {
  const void* x;
  const void* w;
  const void* bias;  // nullptr: no bias
  void* y;
  int M, N, K;
};

int launch_attn_tc(const TcArgs& a, PFN_encodeTiled enc);   // attn_fwd_tc.cu
int launch_attn_f32(const F32Args& a);                       // attn_fwd_f32.cu
int read_fault_word(cudaStream_t stream, int clear, uint32_t* out);  // attn_fwd_tc.cu
void arm_wait_timeout_injection(uint64_t wait_ns, int skip_v_tile);  // attn_fwd_tc.cu (tests only)
int decode_splits(int B, int H, int n_q, int n_max, int d);               // attn_decode.cu
int decode_chunk_keys(int B, int H, int n_max, int d);                    // attn_decode.cu
size_t decode_workspace_bytes(int B, int H, int n_q, int n_max, int d);  // attn_decode.cu
int launch_attn_decode(const DecodeArgs& a, void* workspace);            // attn_decode.cu
int launch_attn_decode_noalloc(const DecodeArgs& a);                     // attn_decode.cu
int read_decode_fault_word(int clear, uint32_t* out);                   // attn_decode.cu
size_t bwd_workspace_bytes(int B, int H, int n_q, int d, int flags);     // attn_bwd.cu
int launch_attn_bwd(const BwdArgs& a, PFN_encodeTiled enc, void* workspace);  // attn_bwd.cu
bool bwd_fused(int d, int flags);                                        // attn_bwd.cu
size_t bwd_host_workspace_bytes(int B, int H, int n_q, int n_k, int d, int mask_mode, int flags);  // attn_bwd_host.cu
int launch_attn_bwd_host(const BwdArgs& a, PFN_encodeTiled enc, void* workspace);                 // attn_bwd_host.cu
int read_bwd_fault_word(int clear, uint32_t* out);                       // attn_bwd.cu
int launch_linear(const LinearJob* jobs, int n_jobs, PFN_encodeTiled enc, cudaStream_t stream);  // attn_linear.cu
int read_linear_fault_word(int clear, uint32_t* out);                    // attn_linear.cu
int launch_attn_weights(const WeightsArgs& a, PFN_encodeTiled enc);     // attn_weights.cu
int read_weights_fault_word(int clear, uint32_t* out);                   // attn_weights.cu
size_t mha_workspace_bytes(int B, int n_q, int n_k, int H, int d);         // attn_mha.cu
int launch_attn_mha(const MhaArgs& a, PFN_encodeTiled enc, void* workspace);  // attn_mha.cu
// Host-operand pipelines (attn_host.cu, attn_bwd_host.cu): chunks of the flattened
// [B, h] head range, each covered by at most three (batches x heads) rectangles.
constexpr int kMaxHostChunks = 64;
int plan_chunks(long long bh, size_t in_bytes, size_t out_bytes, double kernel_us, long long* sizes);  // attn_host.cu
// The rectangle that starts at flattened head f of [f, f1): batch b, pb whole batches of
// H heads, or (pb = 1) ph heads of batch b up to the end of the batch or of the range.
inline void head_rect(long long f, long long f1, int H, int& b, int& pb, int& ph) {
  b = (int)(f / H);
  const int h = (int)(f % H);
  if (h != 0 || f1 - f < H) {
    pb = 1;
    ph = (int)((f1 - f < H - h) ? f1 - f : H - h);
  } else {
    pb = (int)((f1 - f) / H);
    ph = H;
  }
}
size_t host_workspace_bytes(int B, int H, int n_q, int n_k, int d, int mask_mode);  // attn_host.cu
int launch_attn_host(const TcArgs& a, PFN_encodeTiled enc, void* workspace);  // attn_host.cu

}  // namespace attn
