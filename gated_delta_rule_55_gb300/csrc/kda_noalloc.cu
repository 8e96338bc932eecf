// kda_chunk_fwd_noalloc: the workspace variant of the chunked forward with its scratch in a
// file-scope device array instead of a caller buffer (an interface convenience with no
// counterpart on the source pages).  The array lives in this translation unit's own module,
// so its device memory is taken only when the entry point is first used.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;  // ~3590 (chunk, head) records
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of the scratch array, looked up once per device ordinal.
void* scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                     const float* g, const float* beta_logits,
                                     const float* a_log, const float* dt_bias, float scale,
                                     float lower_bound, const float* initial_state, void* out,
                                     float* final_state, int B, int T, int H, int dk, int dv,
                                     int chunk, int dtype, kda_stream_t stream) {
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype);
  if (need > kScratchBytes) return KDA_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0 && !(ws = scratch_address())) return KDA_ERR_DEVICE;
  return kda_chunk_fwd_ws(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                          initial_state, out, final_state, B, T, H, dk, dv, chunk, dtype, ws,
                          need, stream);
}
