// Gated linear recurrent attention (ejkernel "recurrent" page, recurrent_attention): per
// (sequence, query head) a state h in R^{D x D} advanced token by token,
//
//   a_t = g_t + gk_t + g_gamma   (log-decay along the key axis; each term when given)
//   h_t = diag(e^{a_t}) h_{t-1} diag(e^{gv_t}) + k_t v_t^T,        o_t = h_t^T (scale q_t)
//
// (the page names the gates but prints no formula: this is the reading stated with the
// oracle).  Query head h reads key / value head h / (Hq / Hkv); `reverse` walks each
// sequence from its last token to its first.
//
// One CTA of 128 threads per (sequence, query head, 32-wide slice of the value axis): thread
// (r, c) = (tid / 8, tid % 8) owns columns 4 c .. 4 c + 3 on rows r, r + 16, ...; the state
// slice stays in registers, and every staged key-channel vector feeds four columns.  The
// state update needs no other thread's data, and no token needs an earlier token's output,
// so tokens go in blocks of kTB: the block's inputs are staged in shared memory (gate
// exponentials applied), every thread advances its state through the whole block keeping one
// partial output per token, and the outputs are reduced over the key axis once per block.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kDVS = 32;
constexpr int kTB = 16;  // tokens per staged block

template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) gla_kernel(GlaArgs a) {
  constexpr int RPT = D / 16;          // rows per thread
  __shared__ float4 s_kaq[kTB][D];     // (k, e^{a}, scale q, -) per token and key channel
  __shared__ __align__(16) float2 s_vb[kTB][kDVS];   // (v, e^{gv}) per token and column
  __shared__ __align__(16) float s_o[kTB][4][kDVS];  // per-warp partial outputs

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int r16 = tid >> 3, c4 = tid & 7;
  const int j0 = blockIdx.x * kDVS, h = blockIdx.y, seq = blockIdx.z;
  const int Hq = a.Hq, Hkv = a.Hkv, hk = h / (Hq / Hkv);
  long long bos;
  int len;
  if (a.cu_seqlens) {
    int lo = a.cu_seqlens[seq], hi = a.cu_seqlens[seq + 1];
    lo = min(max(lo, 0), a.T);
    hi = min(max(hi, lo), a.T);
    bos = lo;
    len = hi - lo;
  } else {
    bos = (long long)seq * a.T;
    len = a.T;
  }
  const int bidx = a.cu_seqlens ? 0 : seq;  // batch row of g_gamma
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  Tin* out = static_cast<Tin*>(a.out);
  const long long st_off = ((long long)seq * Hq + h) * D * D;
  const float gamma = a.g_gamma ? a.g_gamma[bidx * Hq + h] : 0.f;

  float S[RPT][4];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      S[i][jj] = a.initial_state
                     ? a.initial_state[st_off + (r16 + 16 * i) * D + j0 + 4 * c4 + jj]
                     : 0.f;

  // token slot u of a block starting at position p0 is position p0 + u (forward) or
  // p0 - u (reverse)
  const int dir = a.reverse ? -1 : 1;
  for (int b0 = 0; b0 < len; b0 += kTB) {
    const int nb = min(kTB, len - b0);
    const int p0 = a.reverse ? len - 1 - b0 : b0;
    // stage the block (rows past nb are never read)
    for (int e = tid; e < nb * D; e += kThreads) {
      const int u = e / D, c = e % D;
      const long long tok = bos + p0 + dir * u;
      const long long rq = tok * Hq + h;
      float x = gamma;
      if (a.g) x += a.g[rq * D + c];
      if (a.gk) x += a.gk[rq * D + c];
      s_kaq[u][c] = make_float4(load_as_float(k + (tok * Hkv + hk) * D + c), expf(x),
                                a.scale * load_as_float(q + rq * D + c), 0.f);
    }
    for (int e = tid; e < nb * kDVS; e += kThreads) {
      const int u = e / kDVS, jj = e % kDVS;
      const long long tok = bos + p0 + dir * u;
      s_vb[u][jj] = make_float2(load_as_float(v + (tok * Hkv + hk) * D + j0 + jj),
                                a.gv ? expf(a.gv[(tok * Hq + h) * D + j0 + jj]) : 1.f);
    }
    __syncthreads();
    for (int u = 0; u < nb; ++u) {
      const float4 vb01 = *reinterpret_cast<const float4*>(&s_vb[u][4 * c4]);
      const float4 vb23 = *reinterpret_cast<const float4*>(&s_vb[u][4 * c4 + 2]);
      const float vv[4] = {vb01.x, vb01.z, vb23.x, vb23.z};
      const float bb[4] = {vb01.y, vb01.w, vb23.y, vb23.w};
      float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float4 kaq = s_kaq[u][r16 + 16 * i];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          S[i][jj] = kaq.y * bb[jj] * S[i][jj] + kaq.x * vv[jj];
          o[jj] += S[i][jj] * kaq.z;
        }
      }
      // the warp's four row groups (lanes c4, c4 + 8, c4 + 16, c4 + 24) share columns
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        o[jj] += __shfl_xor_sync(0xffffffffu, o[jj], 8);
        o[jj] += __shfl_xor_sync(0xffffffffu, o[jj], 16);
      }
      if (lane < 8)
        *reinterpret_cast<float4*>(&s_o[u][w][4 * c4]) = make_float4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();
    for (int e = tid; e < nb * kDVS; e += kThreads) {
      const int u = e / kDVS, jj = e % kDVS;
      const float tot = s_o[u][0][jj] + s_o[u][1][jj] + s_o[u][2][jj] + s_o[u][3][jj];
      store_from_float(out + ((bos + p0 + dir * u) * Hq + h) * D + j0 + jj, tot);
    }
    __syncthreads();  // the staged block and the partials are rewritten next
  }
  if (a.final_state) {
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        a.final_state[st_off + (r16 + 16 * i) * D + j0 + 4 * c4 + jj] = S[i][jj];
  }
}

template <typename Tin, int D>
cudaError_t launch_t(const GlaArgs& a, cudaStream_t st) {
  const dim3 grid(D / kDVS, a.Hq, a.nseq);
  gla_kernel<Tin, D><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dtype(const GlaArgs& a, cudaStream_t st) {
  switch (a.D) {
    case 32: return launch_t<Tin, 32>(a, st);
    case 64: return launch_t<Tin, 64>(a, st);
    default: return launch_t<Tin, 128>(a, st);
  }
}

}  // namespace

cudaError_t launch_gla(const GlaArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? launch_dtype<__nv_bfloat16>(a, st) : launch_dtype<float>(a, st);
}

}  // namespace kda
