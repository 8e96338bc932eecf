// Internal declarations shared by the translation units of libkda (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr float kL2Eps = 1e-6f;  // L2-norm epsilon: x / sqrt(sum(x^2) + eps)

// Arguments of the chunked forward (fixed-length when cu_seqlens == nullptr).
struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta_logits;
  const float* a_log;
  const float* dt_bias;
  const float* initial_state;  // nullable
  void* out;
  float* final_state;          // nullable
  const int32_t* cu_seqlens;   // nullable (fixed length)
  float scale;
  float lower_bound;
  int B;        // sequences (B for fixed length, N for varlen)
  int T;        // tokens per sequence (fixed length) -- unused for varlen
  int total_T;  // tokens in the packed token axis (varlen); B*T for fixed length
  int H;
  int dk;
  int dv;
  int chunk;
  // Variants of the kernel_delta_attention call (all zero: the kda_tkg-style gate and beta,
  // L2-normalised q / k, decay before the delta write).
  const float* decay;  // gate_head: per-head log-decay [rows, H], NULL = no decay
  int gate_head;       // 1: gamma = decay[t, h] on every channel (g, a_log, dt_bias unused)
  int beta_prob;       // 1: beta_logits hold the rate itself (no sigmoid)
  int no_l2norm;       // 1: q, k used as given (scale still multiplies q)
  int literal;         // 1: the error term reads the memory before its decay
};

// Gated linear recurrent attention (kda_recurrent_attention_fwd).
struct GlaArgs {
  const void* q;               // [B, T, Hq, D]
  const void* k;               // [B, T, Hkv, D]
  const void* v;               // [B, T, Hkv, D]
  const float* g;              // [B, T, Hq, D] or NULL
  const float* g_gamma;        // [B, Hq] or NULL
  const float* gk;             // [B, T, Hq, D] or NULL
  const float* gv;             // [B, T, Hq, D] or NULL
  const float* initial_state;  // [nseq, Hq, D, D] or NULL
  void* out;                   // [B, T, Hq, D]
  float* final_state;          // [nseq, Hq, D, D] or NULL
  const int32_t* cu_seqlens;   // [nseq + 1] or NULL (then nseq = B)
  float scale;
  int T;                       // tokens per sequence, or the packed token count
  int nseq, Hq, Hkv, D;
  int reverse;
};

struct DecodeArgs {
  const float* q;
  const float* k;
  const float* v;
  const float* g;
  const float* beta_logits;
  const float* a_log;
  const float* dt_bias;
  float* out;
  float* S;
  float scale;
  float lower_bound;
  int B, H, dk, dv;
};

// Launchers (return cudaGetLastError() of their launch).
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
unsigned int decode_read_error(bool reset);
cudaError_t launch_chunk_simt(const ChunkArgs& a, bool bf16, cudaStream_t stream);
// Backward of the chunked forward (fixed-length, decay first, kda_tkg gate): checkpointed
// forward scan, reverse scan, elementwise chain rules.
size_t backward_workspace(int B, int T, int H, int dk, int dv);
cudaError_t launch_backward(const ChunkArgs& f, const void* d_out, const float* d_final,
                            void* dq, void* dk, void* dv, float* dg, float* dbeta_logits,
                            float* da_log, float* ddt_bias, float* d_initial, void* workspace,
                            bool bf16, cudaStream_t stream);
// Chunked tensor-core backward (bf16, dk = dv = 128, 64-token chunks, fixed length, default
// variant): forward records and states, reverse chunk scan, per-chunk products.
bool chunk_bwd_supported(const ChunkArgs& a, bool bf16);
size_t chunk_bwd_workspace(const ChunkArgs& a);
// The training forward: the output and final state, plus the records and per-chunk states
// the backward reads, left in its workspace (same configurations and size).
cudaError_t launch_chunk_fwd_train(const ChunkArgs& a, void* workspace, cudaStream_t stream);
// saved: the workspace already holds what launch_chunk_fwd_train left for these inputs.
cudaError_t launch_chunk_bwd(const ChunkArgs& a, const void* d_out, const float* d_final,
                             void* dq, void* dk, void* dv, float* dg, float* dbeta_logits,
                             float* da_log, float* ddt_bias, float* d_initial, void* workspace,
                             bool saved, cudaStream_t stream);
unsigned int chunk_bwd_read_error(bool reset);
cudaError_t launch_gla(const GlaArgs& a, bool bf16, cudaStream_t stream);
// Chunked tensor-core form of the same recurrence (key-axis gates only, bf16, D = 128,
// forward order): per-chunk prep over all chunks, then the state pass, through a workspace.
bool gla_chunk_supported(const GlaArgs& a, bool bf16);
size_t gla_chunk_workspace(const GlaArgs& a);
bool gla_chunk_index_ok(const GlaArgs& a);
cudaError_t launch_gla_chunk(const GlaArgs& a, void* workspace, cudaStream_t stream);
unsigned int gla_chunk_read_error(bool reset);
// One bounded wait on a barrier nothing arrives on (the give-up path of every kernel wait).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);
unsigned int selftest_read_error(bool reset);
// Sequential (token by token) scan: any supported shape, dtype and variant.
cudaError_t launch_recurrent(const ChunkArgs& a, bool bf16, cudaStream_t stream);
// Tensor-core chunk kernel: bf16 q/k/v, dk = dv = 128, 64-token chunks, default variant.
bool chunk_tc_supported(const ChunkArgs& a, bool bf16);
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream);
unsigned int chunk_tc_read_error(bool reset);
// Two-launch tensor-core path (same configurations as chunk_tc_supported): per-chunk
// prep over all chunks at once, then the sequential state pass, through a workspace.
size_t chunk_split_workspace(const ChunkArgs& a);
bool chunk_split_index_ok(const ChunkArgs& a);
cudaError_t launch_chunk_split(const ChunkArgs& a, void* workspace, cudaStream_t stream);
unsigned int chunk_split_read_error(bool reset);

// Device helpers ------------------------------------------------------------------

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Activated per-channel log-decay: lower_bound * sigmoid(exp(a_log) * (g + dt_bias)),
// with exp(a_log) passed in pre-computed.
__device__ __forceinline__ float gate_gamma(float g, float dt_bias, float exp_a_log,
                                            float lower_bound) {
  return lower_bound * sigmoidf_(exp_a_log * (g + dt_bias));
}

__device__ __forceinline__ float load_as_float(const float* p) { return *p; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
__device__ __forceinline__ void store_from_float(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_from_float(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Token range of sequence `seq` (clamped into [0, total_T] for packed inputs).
__device__ __forceinline__ void seq_range(const ChunkArgs& a, int seq, long long& bos,
                                          int& len) {
  if (a.cu_seqlens != nullptr) {
    int lo = a.cu_seqlens[seq], hi = a.cu_seqlens[seq + 1];
    lo = min(max(lo, 0), a.total_T);
    hi = min(max(hi, lo), a.total_T);
    bos = lo;
    len = hi - lo;
  } else {
    bos = (long long)seq * a.T;
    len = a.T;
  }
}

}  // namespace kda
