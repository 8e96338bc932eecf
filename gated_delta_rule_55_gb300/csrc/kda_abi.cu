// The C ABI of libkda (declared in include/kda.h): host-side argument validation,
// kernel selection and launch on the caller's stream.  Nothing here allocates memory.
#include <math.h>

#include "kda_internal.cuh"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

// The library is built for compute capability 10.3 only; check the current device once
// per device ordinal.
int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return KDA_ERR_DEVICE;
  }
  static int dev_state[64] = {0};  // per device: 0 unchecked, 1 usable, -1 not
  if (dev < 64 && dev_state[dev] != 0) return dev_state[dev] > 0 ? KDA_OK : KDA_ERR_DEVICE;
  int major = 0, minor = 0;
  const bool ok =
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
      major == 10 && minor == 3;
  cudaGetLastError();
  if (dev < 64) dev_state[dev] = ok ? 1 : -1;
  return ok ? KDA_OK : KDA_ERR_DEVICE;
}

// Head dimensions and the query scale (scale <= 0 selects dk^-0.5).
int check_dims_scale(float* scale, int dk, int dv) {
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDA_ERR_HEAD_DIM;
  if (!isfinite(*scale)) return KDA_ERR_SCALE;
  if (*scale <= 0.0f) *scale = 1.0f / sqrtf((float)dk);
  return KDA_OK;
}

int check_common(float* scale, float lower_bound, int dk, int dv) {
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDA_ERR_HEAD_DIM;
  if (!(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_LOWER_BOUND;
  return check_dims_scale(scale, dk, dv);
}

// The kernel_delta_attention call takes the two-launch tensor-core path for bf16 q/k/v with
// dk = dv = 128 in the chunked mode with 64-token chunks.
bool attn_split(int dk, int dv, int chunk, int flags, int dtype) {
  return dtype == KDA_BF16 && dk == 128 && dv == 128 && chunk == 64 &&
         !(flags & KDA_ATTN_RECURRENT);
}

// kda_attention_fwd (use_ws false) and kda_attention_fwd_ws (true).
int attention_common(const void* query, const void* key, const void* value, const float* beta,
                     const float* decay, const float* initial_state, void* out,
                     float* final_state, float softmax_scale, int B, int T, int H, int dk, int dv,
                     int chunk, int flags, int dtype, void* workspace, size_t workspace_bytes,
                     bool use_ws, kda_stream_t stream) {
  if (!query || !key || !value || !beta || !out) return KDA_ERR_NULL_POINTER;
  if (B < 0 || T < 0 || H <= 0) return KDA_ERR_BAD_SHAPE;
  if (flags & ~(KDA_ATTN_NO_QK_L2NORM | KDA_ATTN_RECURRENT | KDA_ATTN_ORDER_LITERAL))
    return KDA_ERR_FLAGS;
  int s = check_dims_scale(&softmax_scale, dk, dv);
  if (s != KDA_OK) return s;
  if ((long long)B * T > 0x7fffffffLL) return KDA_ERR_TOO_LARGE;
  kda::ChunkArgs a{};
  a.q = query; a.k = key; a.v = value; a.beta_logits = beta; a.decay = decay;
  a.initial_state = initial_state; a.out = out; a.final_state = final_state;
  a.scale = softmax_scale; a.lower_bound = 0.f;
  a.B = B; a.T = T; a.total_T = B * T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
  a.gate_head = 1; a.beta_prob = 1;
  a.no_l2norm = (flags & KDA_ATTN_NO_QK_L2NORM) ? 1 : 0;
  a.literal = (flags & KDA_ATTN_ORDER_LITERAL) ? 1 : 0;
  if (a.chunk != 16 && a.chunk != 64) return KDA_ERR_CHUNK;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  const void* ptrs[] = {query, key, value, beta, decay, initial_state, out, final_state};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  const double elems = (double)a.total_T * H * (dk > dv ? dk : dv);
  if (elems >= 1099511627776.0 || (double)B * H * dk * dv >= 1099511627776.0 || B > 65535 ||
      H > 65535)
    return KDA_ERR_TOO_LARGE;
  // the workspace entry takes the two-launch tensor-core path where it applies (a
  // configuration with no tokens needs no workspace: the SIMT path passes the state through)
  const bool split = use_ws && attn_split(dk, dv, chunk, flags, dtype) &&
                     kda::chunk_split_workspace(a) > 0;
  if (split) {
    if (!kda::chunk_split_index_ok(a)) return KDA_ERR_TOO_LARGE;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < kda::chunk_split_workspace(a))
      return KDA_ERR_WORKSPACE;
  }
  s = check_device();
  if (s != KDA_OK) return s;
  if (B == 0) return KDA_OK;
  const bool bf16 = dtype == KDA_BF16;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (split)
    e = kda::launch_chunk_split(a, workspace, st);
  else
    e = (flags & KDA_ATTN_RECURRENT) ? kda::launch_recurrent(a, bf16, st)
                                     : kda::launch_chunk_simt(a, bf16, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// kda_recurrent_attention_fwd (use_ws false) and its workspace variant (true).
int recurrent_common(const void* query, const void* key, const void* value, const float* g,
                     const float* g_gamma, const float* gk, const float* gv,
                     float softmax_scale, const float* initial_state, void* out,
                     float* final_state, const int32_t* cu_seqlens, int N, int B, int T, int Hq,
                     int Hkv, int D, int reverse, int dtype, void* workspace,
                     size_t workspace_bytes, bool use_ws, kda_stream_t stream) {
  if (!query || !key || !value || !out) return KDA_ERR_NULL_POINTER;
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return KDA_ERR_BAD_SHAPE;
  if (cu_seqlens && (B != 1 || N < 0)) return KDA_ERR_BAD_SHAPE;
  if (!head_dim_ok(D)) return KDA_ERR_HEAD_DIM;
  if (!isfinite(softmax_scale)) return KDA_ERR_SCALE;
  if (softmax_scale <= 0.f) softmax_scale = 1.0f / sqrtf((float)D);
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  const void* ptrs[] = {query, key, value, g, g_gamma, gk, gv, initial_state, out,
                        final_state, cu_seqlens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  const long long nseq = cu_seqlens ? N : B;
  if ((double)B * T * Hq * D >= 1099511627776.0 || (double)nseq * Hq * D * D >= 1099511627776.0 ||
      (long long)B * T > 0x7fffffffLL || nseq > 65535 || Hq > 65535)
    return KDA_ERR_TOO_LARGE;
  kda::GlaArgs a{};
  a.q = query; a.k = key; a.v = value; a.g = g; a.g_gamma = g_gamma; a.gk = gk; a.gv = gv;
  a.initial_state = initial_state; a.out = out; a.final_state = final_state;
  a.cu_seqlens = cu_seqlens; a.scale = softmax_scale; a.T = T; a.nseq = (int)nseq;
  a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.reverse = reverse ? 1 : 0;
  // the workspace entry takes the chunked tensor-core path where it applies (no tokens:
  // none needed, the token-serial kernel passes the state through)
  const bool chunked = use_ws && kda::gla_chunk_supported(a, dtype == KDA_BF16) &&
                       nseq > 0 && T > 0;
  if (chunked) {
    if (!kda::gla_chunk_index_ok(a)) return KDA_ERR_TOO_LARGE;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < kda::gla_chunk_workspace(a))
      return KDA_ERR_WORKSPACE;
  }
  int s = check_device();
  if (s != KDA_OK) return s;
  if (nseq == 0) return KDA_OK;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = chunked ? kda::launch_gla_chunk(a, workspace, st)
                                : kda::launch_gla(a, dtype == KDA_BF16, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// workspace == nullptr: the single-pass kernels; otherwise (a non-zero workspace size was
// required and checked) the two-launch path.
int chunk_common(const kda::ChunkArgs& a, int dtype, cudaStream_t st,
                 void* workspace = nullptr, size_t workspace_bytes = 0, bool use_ws = false) {
  if (a.chunk != 16 && a.chunk != 64) return KDA_ERR_CHUNK;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  const void* ptrs[] = {a.q, a.k, a.v, a.g, a.beta_logits, a.a_log, a.dt_bias,
                        a.initial_state, a.out, a.final_state, a.cu_seqlens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  // Element offsets are 64-bit in the kernels; keep every tensor under 2^40 elements and
  // the sequence count within one grid dimension.
  const double elems = (double)a.total_T * a.H * (a.dk > a.dv ? a.dk : a.dv);
  const double state_elems = (double)a.B * a.H * a.dk * a.dv;
  if (elems >= 1099511627776.0 || state_elems >= 1099511627776.0 || a.B > 65535 ||
      a.H > 65535)
    return KDA_ERR_TOO_LARGE;
  const bool bf16 = dtype == KDA_BF16;
  // (a configuration whose workspace size is 0 -- no tokens -- takes the single pass)
  const bool split = use_ws && kda::chunk_tc_supported(a, bf16) &&
                     kda::chunk_split_workspace(a) > 0;
  if (split) {
    if (!kda::chunk_split_index_ok(a)) return KDA_ERR_TOO_LARGE;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < kda::chunk_split_workspace(a))
      return KDA_ERR_WORKSPACE;
  }
  int s = check_device();
  if (s != KDA_OK) return s;
  if (a.B == 0) return KDA_OK;
  cudaError_t e;
  if (split)
    e = kda::launch_chunk_split(a, workspace, st);
  else
    e = kda::chunk_tc_supported(a, bf16) ? kda::launch_chunk_tc(a, st)
                                         : kda::launch_chunk_simt(a, bf16, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// Argument structures of the fixed-length and packed entry points (validated sizes).
int fill_fixed(kda::ChunkArgs& a, const void* q, const void* k, const void* v, const float* g,
               const float* beta_logits, const float* a_log, const float* dt_bias, float scale,
               float lower_bound, const float* initial_state, void* out, float* final_state,
               int B, int T, int H, int dk, int dv, int chunk) {
  if (!q || !k || !v || !g || !beta_logits || !a_log || !dt_bias || !out)
    return KDA_ERR_NULL_POINTER;
  if (B < 0 || T < 0 || H <= 0) return KDA_ERR_BAD_SHAPE;
  int s = check_common(&scale, lower_bound, dk, dv);
  if (s != KDA_OK) return s;
  if ((long long)B * T > 0x7fffffffLL) return KDA_ERR_TOO_LARGE;
  a = kda::ChunkArgs{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta_logits = beta_logits; a.a_log = a_log;
  a.dt_bias = dt_bias; a.initial_state = initial_state; a.out = out;
  a.final_state = final_state; a.cu_seqlens = nullptr; a.scale = scale;
  a.lower_bound = lower_bound; a.B = B; a.T = T; a.total_T = B * T;
  a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
  return KDA_OK;
}

int fill_varlen(kda::ChunkArgs& a, const void* q, const void* k, const void* v,
                const float* g, const float* beta_logits, const float* a_log,
                const float* dt_bias, float scale, float lower_bound, const int32_t* cu_seqlens,
                int N, int total_T, const float* initial_state, void* out, float* final_state,
                int H, int dk, int dv, int chunk) {
  if (!q || !k || !v || !g || !beta_logits || !a_log || !dt_bias || !out || !cu_seqlens)
    return KDA_ERR_NULL_POINTER;
  if (N < 0 || total_T < 0 || H <= 0) return KDA_ERR_BAD_SHAPE;
  int s = check_common(&scale, lower_bound, dk, dv);
  if (s != KDA_OK) return s;
  a = kda::ChunkArgs{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta_logits = beta_logits; a.a_log = a_log;
  a.dt_bias = dt_bias; a.initial_state = initial_state; a.out = out;
  a.final_state = final_state; a.cu_seqlens = cu_seqlens; a.scale = scale;
  a.lower_bound = lower_bound; a.B = N; a.T = 0; a.total_T = total_T;
  a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
  return KDA_OK;
}

// Workspace bytes of the two-launch path (0 when the configuration does not use it or the
// arguments are invalid).
size_t ws_size(const kda::ChunkArgs& a, int dtype) {
  if (a.chunk != 16 && a.chunk != 64) return 0;
  if (dtype != KDA_BF16 || !kda::chunk_tc_supported(a, true)) return 0;
  return kda::chunk_split_workspace(a);
}

}  // namespace

extern "C" {

int kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta_logits, const float* a_log, const float* dt_bias,
                  float scale, float lower_bound, const float* initial_state, void* out,
                  float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                  int dtype, kda_stream_t stream) {
  kda::ChunkArgs a;
  const int s = fill_fixed(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                           initial_state, out, final_state, B, T, H, dk, dv, chunk);
  if (s != KDA_OK) return s;
  return chunk_common(a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

int kda_chunk_fwd_varlen(const void* q, const void* k, const void* v, const float* g,
                         const float* beta_logits, const float* a_log, const float* dt_bias,
                         float scale, float lower_bound, const int32_t* cu_seqlens, int N,
                         int total_T, const float* initial_state, void* out,
                         float* final_state, int H, int dk, int dv, int chunk, int dtype,
                         kda_stream_t stream) {
  kda::ChunkArgs a;
  const int s = fill_varlen(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                            cu_seqlens, N, total_T, initial_state, out, final_state, H, dk, dv,
                            chunk);
  if (s != KDA_OK) return s;
  return chunk_common(a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

int kda_recurrent_attention_fwd(const void* query, const void* key, const void* value,
                                const float* g, const float* g_gamma, const float* gk,
                                const float* gv, float softmax_scale, const float* initial_state,
                                void* out, float* final_state, const int32_t* cu_seqlens, int N,
                                int B, int T, int Hq, int Hkv, int D, int reverse, int dtype,
                                kda_stream_t stream) {
  return recurrent_common(query, key, value, g, g_gamma, gk, gv, softmax_scale, initial_state,
                          out, final_state, cu_seqlens, N, B, T, Hq, Hkv, D, reverse, dtype,
                          nullptr, 0, false, stream);
}

size_t kda_recurrent_attention_fwd_workspace_size(int N, int B, int T, int Hq, int Hkv, int D,
                                                  int flags, int dtype) {
  if (flags & ~(KDA_REC_PACKED | KDA_REC_VALUE_GATE | KDA_REC_REVERSE)) return 0;
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || N < 0) return 0;
  if ((long long)B * T > 0x7fffffffLL) return 0;
  static const int32_t marker = 0;  // only the presence of cu_seqlens matters here
  kda::GlaArgs a{};
  a.cu_seqlens = (flags & KDA_REC_PACKED) ? &marker : nullptr;
  a.gv = (flags & KDA_REC_VALUE_GATE) ? reinterpret_cast<const float*>(&marker) : nullptr;
  a.reverse = (flags & KDA_REC_REVERSE) ? 1 : 0;
  a.T = T;  // tokens per sequence, or the packed token count
  a.nseq = (flags & KDA_REC_PACKED) ? N : B;
  a.Hq = Hq; a.Hkv = Hkv; a.D = D;
  if (!kda::gla_chunk_supported(a, dtype == KDA_BF16) || a.nseq == 0 || T == 0) return 0;
  return kda::gla_chunk_workspace(a);
}

int kda_recurrent_attention_fwd_ws(const void* query, const void* key, const void* value,
                                   const float* g, const float* g_gamma, const float* gk,
                                   const float* gv, float softmax_scale,
                                   const float* initial_state, void* out, float* final_state,
                                   const int32_t* cu_seqlens, int N, int B, int T, int Hq,
                                   int Hkv, int D, int reverse, int dtype, void* workspace,
                                   size_t workspace_bytes, kda_stream_t stream) {
  return recurrent_common(query, key, value, g, g_gamma, gk, gv, softmax_scale, initial_state,
                          out, final_state, cu_seqlens, N, B, T, Hq, Hkv, D, reverse, dtype,
                          workspace, workspace_bytes, true, stream);
}

int kda_attention_fwd(const void* query, const void* key, const void* value, const float* beta,
                      const float* decay, const float* initial_state, void* out,
                      float* final_state, float softmax_scale, int B, int T, int H, int dk,
                      int dv, int chunk, int flags, int dtype, kda_stream_t stream) {
  return attention_common(query, key, value, beta, decay, initial_state, out, final_state,
                          softmax_scale, B, T, H, dk, dv, chunk, flags, dtype, nullptr, 0, false,
                          stream);
}

size_t kda_attention_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                        int flags, int dtype) {
  if (B < 0 || T < 0 || H <= 0 || (long long)B * T > 0x7fffffffLL) return 0;
  if (!attn_split(dk, dv, chunk, flags, dtype)) return 0;
  kda::ChunkArgs a{};
  a.B = B; a.T = T; a.total_T = B * T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
  return kda::chunk_split_workspace(a);
}

int kda_attention_fwd_ws(const void* query, const void* key, const void* value,
                         const float* beta, const float* decay, const float* initial_state,
                         void* out, float* final_state, float softmax_scale, int B, int T, int H,
                         int dk, int dv, int chunk, int flags, int dtype, void* workspace,
                         size_t workspace_bytes, kda_stream_t stream) {
  return attention_common(query, key, value, beta, decay, initial_state, out, final_state,
                          softmax_scale, B, T, H, dk, dv, chunk, flags, dtype, workspace,
                          workspace_bytes, true, stream);
}


}  // extern "C"

namespace {

// Backward arguments for sizing only (no pointers are read).
kda::ChunkArgs bwd_shape(int B, int T, int H, int dk, int dv) {
  kda::ChunkArgs a{};
  a.B = B; a.T = T; a.total_T = B * T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = 64;
  return a;
}

int bwd_common(const void* q, const void* k, const void* v, const float* g,
               const float* beta_logits, const float* a_log, const float* dt_bias, float scale,
               float lower_bound, const float* initial_state, const void* d_out,
               const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
               float* dbeta_logits, float* da_log, float* ddt_bias, float* d_initial_state,
               int B, int T, int H, int dim_k, int dim_v, int dtype, void* workspace,
               size_t workspace_bytes, kda_stream_t stream, bool saved) {
  kda::ChunkArgs a;
  int s = fill_fixed(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                     initial_state, dq, nullptr, B, T, H, dim_k, dim_v, 64);
  if (s != KDA_OK) return s;
  if (!d_out || !dq || !dk || !dv || !dg || !dbeta_logits || !da_log || !ddt_bias)
    return KDA_ERR_NULL_POINTER;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  const void* ptrs[] = {q, k, v, g, beta_logits, a_log, dt_bias, initial_state, d_out,
                        d_final_state, dq, dk, dv, dg, dbeta_logits, da_log, ddt_bias,
                        d_initial_state};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  const double elems = (double)a.total_T * H * (dim_k > dim_v ? dim_k : dim_v);
  if (elems >= 1099511627776.0 ||
      (double)B * H * dim_k * dim_v * ((T + 63) / 64 + 64) >= 1099511627776.0 || B > 65535 ||
      H > 65535)
    return KDA_ERR_TOO_LARGE;
  const bool chunked = B > 0 && kda::chunk_bwd_supported(a, dtype == KDA_BF16);
  // the saved-records entry serves exactly the tensor-core configurations (no tokens: the
  // plain path, which has nothing to read back)
  if (saved && !chunked && (long long)B * T > 0)
    return dtype != KDA_BF16 ? KDA_ERR_DTYPE : KDA_ERR_HEAD_DIM;
  const size_t need =
      chunked ? kda::chunk_bwd_workspace(a) : kda::backward_workspace(B, T, H, dim_k, dim_v);
  if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                   workspace_bytes < need))
    return KDA_ERR_WORKSPACE;
  s = check_device();
  if (s != KDA_OK) return s;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (B == 0) {
    e = cudaMemsetAsync(da_log, 0, sizeof(float) * H, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * dim_k * H, st);
  } else if (chunked) {
    e = kda::launch_chunk_bwd(a, d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log,
                              ddt_bias, d_initial_state, workspace, saved, st);
  } else {
    e = kda::launch_backward(a, d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log,
                             ddt_bias, d_initial_state, workspace, dtype == KDA_BF16, st);
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

size_t kda_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, int dtype) {
  if (B < 0 || T < 0 || H <= 0 || !head_dim_ok(dk) || !head_dim_ok(dv) ||
      (long long)B * T > 0x7fffffffLL || (dtype != KDA_F32 && dtype != KDA_BF16))
    return 0;
  const kda::ChunkArgs a = bwd_shape(B, T, H, dk, dv);
  if (B > 0 && kda::chunk_bwd_supported(a, dtype == KDA_BF16)) return kda::chunk_bwd_workspace(a);
  return kda::backward_workspace(B, T, H, dk, dv);
}

int kda_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta_logits, const float* a_log, const float* dt_bias,
                  float scale, float lower_bound, const float* initial_state, const void* d_out,
                  const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                  float* dbeta_logits, float* da_log, float* ddt_bias, float* d_initial_state,
                  int B, int T, int H, int dim_k, int dim_v, int dtype, void* workspace,
                  size_t workspace_bytes, kda_stream_t stream) {
  return bwd_common(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound, initial_state,
                    d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log, ddt_bias,
                    d_initial_state, B, T, H, dim_k, dim_v, dtype, workspace, workspace_bytes,
                    stream, false);
}

int kda_chunk_bwd_saved(const void* q, const void* k, const void* v, const float* g,
                        const float* beta_logits, const float* a_log, const float* dt_bias,
                        float scale, float lower_bound, const float* initial_state,
                        const void* d_out, const float* d_final_state, void* dq, void* dk,
                        void* dv, float* dg, float* dbeta_logits, float* da_log, float* ddt_bias,
                        float* d_initial_state, int B, int T, int H, int dim_k, int dim_v,
                        int dtype, void* workspace, size_t workspace_bytes,
                        kda_stream_t stream) {
  return bwd_common(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound, initial_state,
                    d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log, ddt_bias,
                    d_initial_state, B, T, H, dim_k, dim_v, dtype, workspace, workspace_bytes,
                    stream, true);
}

size_t kda_chunk_bwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dv,
                                          int dtype) {
  if (N < 0 || total_T < 0 || H <= 0 || !head_dim_ok(dk) || !head_dim_ok(dv)) return 0;
  static const int32_t marker = 0;  // only the presence of cu_seqlens matters here
  kda::ChunkArgs a = bwd_shape(N, 0, H, dk, dv);
  a.cu_seqlens = &marker;
  a.total_T = total_T;
  if (!kda::chunk_bwd_supported(a, dtype == KDA_BF16)) return 0;
  return kda::chunk_bwd_workspace(a);
}

}  // extern "C"

namespace {

int bwd_varlen_common(const void* q, const void* k, const void* v, const float* g,
                      const float* beta_logits, const float* a_log, const float* dt_bias,
                      float scale, float lower_bound, const int32_t* cu_seqlens, int N,
                      int total_T, const float* initial_state, const void* d_out,
                      const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                      float* dbeta_logits, float* da_log, float* ddt_bias, float* d_initial_state,
                      int H, int dim_k, int dim_v, int dtype, void* workspace,
                      size_t workspace_bytes, kda_stream_t stream, bool saved) {
  kda::ChunkArgs a;
  int s = fill_varlen(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                      cu_seqlens, N, total_T, initial_state, dq, nullptr, H, dim_k, dim_v, 64);
  if (s != KDA_OK) return s;
  if (!d_out || !dq || !dk || !dv || !dg || !dbeta_logits || !da_log || !ddt_bias)
    return KDA_ERR_NULL_POINTER;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  // packed sequences are served on the tensor-core path only
  if (!kda::chunk_bwd_supported(a, dtype == KDA_BF16))
    return dtype != KDA_BF16 ? KDA_ERR_DTYPE
                             : (dim_k != 128 || dim_v != 128) ? KDA_ERR_HEAD_DIM
                                                              : KDA_ERR_TOO_LARGE;
  const void* ptrs[] = {q, k, v, g, beta_logits, a_log, dt_bias, cu_seqlens, initial_state,
                        d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log, ddt_bias,
                        d_initial_state};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  if ((double)total_T * H * 128 >= 1099511627776.0 || N > 65535 || H > 65535)
    return KDA_ERR_TOO_LARGE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < kda::chunk_bwd_workspace(a))
    return KDA_ERR_WORKSPACE;
  s = check_device();
  if (s != KDA_OK) return s;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (N == 0) {
    e = cudaMemsetAsync(da_log, 0, sizeof(float) * H, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * dim_k * H, st);
  } else {
    e = kda::launch_chunk_bwd(a, d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log,
                              ddt_bias, d_initial_state, workspace, saved, st);
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int kda_chunk_bwd_varlen(const void* q, const void* k, const void* v, const float* g,
                         const float* beta_logits, const float* a_log, const float* dt_bias,
                         float scale, float lower_bound, const int32_t* cu_seqlens, int N,
                         int total_T, const float* initial_state, const void* d_out,
                         const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                         float* dbeta_logits, float* da_log, float* ddt_bias,
                         float* d_initial_state, int H, int dim_k, int dim_v, int dtype,
                         void* workspace, size_t workspace_bytes, kda_stream_t stream) {
  return bwd_varlen_common(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                           cu_seqlens, N, total_T, initial_state, d_out, d_final_state, dq, dk,
                           dv, dg, dbeta_logits, da_log, ddt_bias, d_initial_state, H, dim_k,
                           dim_v, dtype, workspace, workspace_bytes, stream, false);
}

int kda_chunk_bwd_saved_varlen(const void* q, const void* k, const void* v, const float* g,
                               const float* beta_logits, const float* a_log,
                               const float* dt_bias, float scale, float lower_bound,
                               const int32_t* cu_seqlens, int N, int total_T,
                               const float* initial_state, const void* d_out,
                               const float* d_final_state, void* dq, void* dk, void* dv,
                               float* dg, float* dbeta_logits, float* da_log, float* ddt_bias,
                               float* d_initial_state, int H, int dim_k, int dim_v, int dtype,
                               void* workspace, size_t workspace_bytes, kda_stream_t stream) {
  return bwd_varlen_common(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                           cu_seqlens, N, total_T, initial_state, d_out, d_final_state, dq, dk,
                           dv, dg, dbeta_logits, da_log, ddt_bias, d_initial_state, H, dim_k,
                           dim_v, dtype, workspace, workspace_bytes, stream, true);
}

int kda_chunk_fwd_train_varlen(const void* q, const void* k, const void* v, const float* g,
                               const float* beta_logits, const float* a_log,
                               const float* dt_bias, float scale, float lower_bound,
                               const int32_t* cu_seqlens, int N, int total_T,
                               const float* initial_state, void* out, float* final_state, int H,
                               int dk, int dv, int chunk, int dtype, void* workspace,
                               size_t workspace_bytes, kda_stream_t stream) {
  kda::ChunkArgs a;
  const int s = fill_varlen(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                            cu_seqlens, N, total_T, initial_state, out, final_state, H, dk, dv,
                            chunk);
  if (s != KDA_OK) return s;
  if (N == 0 || total_T == 0)  // no tokens: the plain forward (state copy), nothing to keep
    return chunk_common(a, dtype, reinterpret_cast<cudaStream_t>(stream));
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
  if (chunk != 16 && chunk != 64) return KDA_ERR_CHUNK;
  if (!kda::chunk_bwd_supported(a, dtype == KDA_BF16))
    return dtype != KDA_BF16 ? KDA_ERR_DTYPE
           : chunk != 64     ? KDA_ERR_CHUNK
           : (dk != 128 || dv != 128) ? KDA_ERR_HEAD_DIM : KDA_ERR_TOO_LARGE;
  const void* ptrs[] = {q, k, v, g, beta_logits, a_log, dt_bias, cu_seqlens, initial_state,
                        out, final_state};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  if ((double)total_T * H * 128 >= 1099511627776.0 || N > 65535 || H > 65535)
    return KDA_ERR_TOO_LARGE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < kda::chunk_bwd_workspace(a))
    return KDA_ERR_WORKSPACE;
  const int d = check_device();
  if (d != KDA_OK) return d;
  const cudaError_t e =
      kda::launch_chunk_fwd_train(a, workspace, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

int kda_chunk_fwd_train(const void* q, const void* k, const void* v, const float* g,
                        const float* beta_logits, const float* a_log, const float* dt_bias,
                        float scale, float lower_bound, const float* initial_state, void* out,
                        float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                        int dtype, void* workspace, size_t workspace_bytes,
                        kda_stream_t stream) {
  kda::ChunkArgs a;
  const int s = fill_fixed(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                           initial_state, out, final_state, B, T, H, dk, dv, chunk);
  if (s != KDA_OK) return s;
  if ((long long)B * T == 0)  // no tokens: the plain forward (state copy), nothing to keep
    return chunk_common(a, dtype, reinterpret_cast<cudaStream_t>(stream));
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
  if (chunk != 16 && chunk != 64) return KDA_ERR_CHUNK;
  if (!kda::chunk_bwd_supported(a, dtype == KDA_BF16))
    return dtype != KDA_BF16 ? KDA_ERR_DTYPE : chunk != 64 ? KDA_ERR_CHUNK : KDA_ERR_HEAD_DIM;
  const void* ptrs[] = {q, k, v, g, beta_logits, a_log, dt_bias, initial_state, out,
                        final_state};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  if ((double)a.total_T * H * 128 >= 1099511627776.0 || B > 65535 || H > 65535)
    return KDA_ERR_TOO_LARGE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < kda::chunk_bwd_workspace(a))
    return KDA_ERR_WORKSPACE;
  const int d = check_device();
  if (d != KDA_OK) return d;
  const cudaError_t e =
      kda::launch_chunk_fwd_train(a, workspace, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                    int dtype) {
  if (B < 0 || T < 0 || H <= 0 || (long long)B * T > 0x7fffffffLL) return 0;
  kda::ChunkArgs a{};
  a.B = B; a.T = T; a.total_T = B * T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
  return ws_size(a, dtype);
}

size_t kda_chunk_fwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dv,
                                           int chunk, int dtype) {
  if (N < 0 || total_T < 0 || H <= 0) return 0;
  static const int32_t marker = 0;  // only the presence of cu_seqlens matters here
  kda::ChunkArgs a{};
  a.cu_seqlens = &marker;
  a.B = N; a.total_T = total_T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
  return ws_size(a, dtype);
}

int kda_chunk_fwd_ws(const void* q, const void* k, const void* v, const float* g,
                     const float* beta_logits, const float* a_log, const float* dt_bias,
                     float scale, float lower_bound, const float* initial_state, void* out,
                     float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                     int dtype, void* workspace, size_t workspace_bytes, kda_stream_t stream) {
  kda::ChunkArgs a;
  const int s = fill_fixed(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                           initial_state, out, final_state, B, T, H, dk, dv, chunk);
  if (s != KDA_OK) return s;
  return chunk_common(a, dtype, reinterpret_cast<cudaStream_t>(stream), workspace,
                      workspace_bytes, true);
}

int kda_chunk_fwd_varlen_ws(const void* q, const void* k, const void* v, const float* g,
                            const float* beta_logits, const float* a_log,
                            const float* dt_bias, float scale, float lower_bound,
                            const int32_t* cu_seqlens, int N, int total_T,
                            const float* initial_state, void* out, float* final_state, int H,
                            int dk, int dv, int chunk, int dtype, void* workspace,
                            size_t workspace_bytes, kda_stream_t stream) {
  kda::ChunkArgs a;
  const int s = fill_varlen(a, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                            cu_seqlens, N, total_T, initial_state, out, final_state, H, dk, dv,
                            chunk);
  if (s != KDA_OK) return s;
  return chunk_common(a, dtype, reinterpret_cast<cudaStream_t>(stream), workspace,
                      workspace_bytes, true);
}

int kda_decode_step(const float* q, const float* k, const float* v, const float* g,
                    const float* beta_logits, const float* a_log, const float* dt_bias,
                    float scale, float lower_bound, float* out, float* S, int B, int H,
                    int dk, int dv, kda_stream_t stream) {
  if (!q || !k || !v || !g || !beta_logits || !a_log || !dt_bias || !out || !S)
    return KDA_ERR_NULL_POINTER;
  if (B < 0 || H <= 0) return KDA_ERR_BAD_SHAPE;
  int s = check_common(&scale, lower_bound, dk, dv);
  if (s != KDA_OK) return s;
  const void* ptrs[] = {q, k, v, g, beta_logits, a_log, dt_bias, out, S};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KDA_ERR_MISALIGNED;
  if ((double)B * H * dk * dv >= 1099511627776.0 || (long long)B * H > 0x7fffffffLL)
    return KDA_ERR_TOO_LARGE;
  s = check_device();
  if (s != KDA_OK) return s;
  if (B == 0) return KDA_OK;
  kda::DecodeArgs a{q, k, v, g, beta_logits, a_log, dt_bias, out, S, scale, lower_bound,
                    B, H, dk, dv};
  const cudaError_t e = kda::launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case KDA_ERR_BAD_SHAPE: return "invalid size (negative, or zero heads)";
    case KDA_ERR_HEAD_DIM: return "dk and dv must each be 32, 64 or 128";
    case KDA_ERR_CHUNK: return "chunk must be 16 or 64";
    case KDA_ERR_LOWER_BOUND: return "lower_bound must be finite and in [-5, 0]";
    case KDA_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
    case KDA_ERR_DTYPE: return "dtype must be KDA_F32 or KDA_BF16";
    case KDA_ERR_LAUNCH: return "CUDA launch failed";
    case KDA_ERR_DEVICE: return "no usable CUDA device of compute capability 10.3";
    case KDA_ERR_SCALE: return "scale must be finite";
    case KDA_ERR_TOO_LARGE: return "problem too large for the kernels' index limits";
    case KDA_ERR_WORKSPACE: return "workspace NULL, smaller than required or not 256-byte aligned";
    case KDA_ERR_FLAGS: return "unknown bits in the flags argument";
    default: return "unknown kda status";
  }
}

int kda_version(void) { return 100; }

int kda_device_error(int reset) {
  int s = check_device();
  if (s != KDA_OK) return s;
  return (int)(kda::chunk_tc_read_error(reset != 0) | kda::chunk_split_read_error(reset != 0) |
               kda::chunk_bwd_read_error(reset != 0) | kda::decode_read_error(reset != 0) |
               kda::selftest_read_error(reset != 0) | kda::gla_chunk_read_error(reset != 0));
}

int kda_selftest_bounded_wait(unsigned long long limit_ns, kda_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return KDA_ERR_BAD_SHAPE;
  const int s = check_device();
  if (s != KDA_OK) return s;
  return kda::launch_wait_selftest(limit_ns, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KDA_OK
             : KDA_ERR_LAUNCH;
}

}  // extern "C"
