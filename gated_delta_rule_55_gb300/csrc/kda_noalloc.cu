// kda_chunk_fwd_noalloc: the workspace variant of the chunked forward with its scratch in a
// file-scope device array instead of a caller buffer (an interface convenience with no
// counterpart on the source pages), for callers that cannot allocate device memory.  The
// array lives in this translation unit's own module: under lazy module loading (the CUDA
// default) its device memory is reserved when that module is first loaded on a device,
// which this entry point's first call does; with CUDA_MODULE_LOADING=EAGER every context
// that loads the library reserves it at start-up.
#include <cuda.h>

#include <mutex>
#include <unordered_map>

#include "kda_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;  // ~3590 (chunk, head) records
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's id of the calling thread's current context (unique for the life of the
// process, so a context created after a cudaDeviceReset never reuses an old id), or 0 when
// there is none yet or the driver does not say.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current context.  The set-up (the symbol
// lookup, which loads the module) runs once per context, on the first call made with that
// context current; later calls find the address in the table.  A device address belongs to
// its context, so a context that replaced an earlier one (after cudaDeviceReset) gets a
// lookup of its own instead of the old, unmapped address.
void* scratch_address() {
  static std::mutex mu;
  static std::unordered_map<unsigned long long, void*> by_context;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_context_id();
  if (id != 0) {
    const auto it = by_context.find(id);
    if (it != by_context.end()) return it->second;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  const unsigned long long now = current_context_id();  // the lookup made one current
  if (now != 0) by_context[now] = p;
  return p;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                     const float* g, const float* beta_logits,
                                     const float* a_log, const float* dt_bias, float scale,
                                     float lower_bound, const float* initial_state, void* out,
                                     float* final_state, int B, int T, int H, int dk, int dv,
                                     int chunk, int dtype, kda_stream_t stream) {
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype);
  if (need > kScratchBytes) {
    // Argument errors come first, in kda_chunk_fwd's order: without a workspace the entry
    // validates everything and, when all is valid, stops at its workspace check before any
    // device work is enqueued.
    const int s = kda_chunk_fwd_ws(q, k, v, g, beta_logits, a_log, dt_bias, scale,
                                   lower_bound, initial_state, out, final_state, B, T, H, dk,
                                   dv, chunk, dtype, nullptr, 0, stream);
    return s != KDA_OK ? s : KDA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  if (need > 0 && !(ws = scratch_address())) return KDA_ERR_DEVICE;
  return kda_chunk_fwd_ws(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                          initial_state, out, final_state, B, T, H, dk, dv, chunk, dtype, ws,
                          need, stream);
}
