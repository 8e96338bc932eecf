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
// (rg, j) owns column j on rows rg, rg + 4, ...; the state slice stays in registers.  Each
// token needs one reduction over the key axis (the output); the next token's inputs are
// loaded into registers while the current one is processed.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kDVS = 32;

template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) gla_kernel(GlaArgs a) {
  constexpr int RPT = D / 4;
  __shared__ float s_q[D], s_k[D], s_a[D];
  __shared__ float s_v[kDVS], s_b[kDVS];
  __shared__ float s_red[4][kDVS];

  const int tid = threadIdx.x, lane = tid & 31, rg = tid >> 5;
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
  const float gamma = (a.g_gamma && tid < D) ? a.g_gamma[bidx * Hq + h] : 0.f;

  float S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    S[i] = a.initial_state ? a.initial_state[st_off + (rg + 4 * i) * D + j0 + lane] : 0.f;

  // inputs of token t (position within the sequence): channel tid of q, k and the key-axis
  // log-decay (tid < D); column j0 + tid of v and of the value-axis log-decay (tid < 32)
  struct In { float q, k, a, v, b; };
  auto load = [&](int t) {
    In r{0.f, 0.f, 0.f, 0.f, 0.f};
    const long long tok = bos + t;
    const long long rq = tok * Hq + h, rk = tok * Hkv + hk;
    if (tid < D) {
      r.q = load_as_float(q + rq * D + tid);
      r.k = load_as_float(k + rk * D + tid);
      float x = gamma;
      if (a.g) x += a.g[rq * D + tid];
      if (a.gk) x += a.gk[rq * D + tid];
      r.a = x;
    }
    if (tid < kDVS) {
      r.v = load_as_float(v + rk * D + j0 + tid);
      r.b = a.gv ? a.gv[rq * D + j0 + tid] : 0.f;
    }
    return r;
  };
  const int step = a.reverse ? -1 : 1;
  int t = a.reverse ? len - 1 : 0;
  In nx = len > 0 ? load(t) : In{0.f, 0.f, 0.f, 0.f, 0.f};
  for (int it = 0; it < len; ++it, t += step) {
    const In cur = nx;
    if (it + 1 < len) nx = load(t + step);
    if (tid < D) {
      s_q[tid] = a.scale * cur.q;
      s_k[tid] = cur.k;
      s_a[tid] = expf(cur.a);
    }
    if (tid < kDVS) {
      s_v[tid] = cur.v;
      s_b[tid] = expf(cur.b);
    }
    __syncthreads();
    const float bj = s_b[lane], vj = s_v[lane];
    float o = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int c = rg + 4 * i;
      S[i] = s_a[c] * bj * S[i] + s_k[c] * vj;
      o += S[i] * s_q[c];
    }
    s_red[rg][lane] = o;
    __syncthreads();
    if (tid < kDVS) {
      const float tot = s_red[0][tid] + s_red[1][tid] + s_red[2][tid] + s_red[3][tid];
      store_from_float(out + ((bos + t) * Hq + h) * D + j0 + tid, tot);
    }
    __syncthreads();  // shared vectors are rewritten by the next token
  }
  if (a.final_state) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) a.final_state[st_off + (rg + 4 * i) * D + j0 + lane] = S[i];
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
