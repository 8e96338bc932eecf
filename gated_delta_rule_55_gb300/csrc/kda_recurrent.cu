// Sequential KDA forward: the recurrence advanced one token at a time
// (kernel_delta_attention page, "Algorithm modes: Recurrent: pure sequential scan",
// use_chunked=False).  It keeps no chunk buffers: the only memory per (sequence, head) is
// the state slice, in registers.
//
// One CTA of 128 threads per (sequence, head, 32-wide slice of dv).  Thread (rg, j)
// (rg = warp, j = lane) owns column j of the slice on rows rg, rg + 4, ...  Per token, with
// d = e^{gamma} (per channel, or one per-head value broadcast to every channel):
//   p_k = S^T (d k^)  (decay first)  or  S^T k^  (literal order: the error term reads the
//         memory before its decay)
//   p_q = S^T (d q^)
//   u   = beta (v - p_k),   o = p_q + u (k^ . q^),   S <- diag(d) S + k^ u^T
// which is o = S_t^T q^ after the update in both orders.  The next token's inputs are
// loaded into registers while the current one is processed.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kDVS = 32;

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(ChunkArgs a) {
  constexpr int RPT = DK / 4;  // state rows per thread
  __shared__ float s_kd[DK], s_qd[DK], s_k[DK], s_d[DK];
  __shared__ float s_pk[4][kDVS], s_pq[4][kDVS];
  __shared__ float s_part[3][4];
  __shared__ float s_u[kDVS];
  __shared__ float s_beta;

  const int tid = threadIdx.x, lane = tid & 31, rg = tid >> 5;
  const int j0 = blockIdx.x * kDVS;
  const int h = blockIdx.y, seq = blockIdx.z;
  const int H = a.H, DV = a.dv;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  Tin* out = static_cast<Tin*>(a.out);
  const long long state_off = ((long long)seq * H + h) * DK * DV;

  float S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int c = rg + 4 * i;
    S[i] = a.initial_state ? a.initial_state[state_off + (long long)c * DV + j0 + lane] : 0.f;
  }
  // per-channel gate constants (thread tid < DK owns channel tid)
  const float exp_a = (a.gate_head || tid >= DK) ? 0.f : expf(a.a_log[h]);
  const float db = (a.gate_head || tid >= DK) ? 0.f : a.dt_bias[tid * H + h];

  // inputs of token t: channel tid of q, k, g (tid < DK); column j0 + lane of v (warp 0);
  // beta and the per-head decay (thread 0)
  auto load = [&](int t, float& xq, float& xk, float& xg, float& xv, float& xb) {
    xq = xk = xg = xv = xb = 0.f;
    if (t >= len) return;
    const long long row = (bos + t) * H + h;
    if (tid < DK) {
      xq = load_as_float(q + row * DK + tid);
      xk = load_as_float(k + row * DK + tid);
      if (!a.gate_head) xg = a.g[row * DK + tid];
    }
    if (tid < kDVS) xv = load_as_float(v + row * DV + j0 + tid);
    if (tid == 0) {
      xb = a.beta_logits[row];
      if (a.gate_head && a.decay) xg = a.decay[row];
    }
  };
  float nq, nk, ng, nv, nb;
  load(0, nq, nk, ng, nv, nb);

  for (int t = 0; t < len; ++t) {
    const float xq = nq, xk = nk, xg = ng, xv = nv, xb = nb;
    load(t + 1, nq, nk, ng, nv, nb);  // in flight while this token is processed

    // norms and k . q over the channels (warps hold 32 channels each)
    if (tid < DK) {
      const float kk = warp_sum(xk * xk), qq = warp_sum(xq * xq), kq = warp_sum(xk * xq);
      if (lane == 0) {
        s_part[0][rg] = kk;
        s_part[1][rg] = qq;
        s_part[2][rg] = kq;
      }
    }
    if (tid == 0) {
      s_beta = a.beta_prob ? xb : sigmoidf_(xb);
      if (a.gate_head) s_d[0] = xg;  // the per-head log-decay, broadcast below
    }
    __syncthreads();
    float kk = 0.f, qq = 0.f, kq = 0.f;
#pragma unroll
    for (int w = 0; w < DK / 32; ++w) {
      kk += s_part[0][w];
      qq += s_part[1][w];
      kq += s_part[2][w];
    }
    const float rk = a.no_l2norm ? 1.f : rsqrtf(kk + kL2Eps);
    const float rq = a.no_l2norm ? a.scale : a.scale * rsqrtf(qq + kL2Eps);
    const float khq = kq * rk * rq;  // k^ . q^
    const float dhead = a.gate_head ? expf(s_d[0]) : 0.f;
    __syncthreads();  // s_d[0] read by everyone before it is overwritten
    if (tid < DK) {
      const float d = a.gate_head ? dhead : expf(gate_gamma(xg, db, exp_a, a.lower_bound));
      const float kh = xk * rk, qh = xq * rq;
      s_d[tid] = d;
      s_k[tid] = kh;
      s_kd[tid] = a.literal ? kh : d * kh;
      s_qd[tid] = d * qh;
    }
    if (tid < kDVS) s_u[tid] = xv;  // v, replaced by u below
    __syncthreads();

    // partial products over this thread's rows
    float pk = 0.f, pq = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int c = rg + 4 * i;
      pk += S[i] * s_kd[c];
      pq += S[i] * s_qd[c];
    }
    s_pk[rg][lane] = pk;
    s_pq[rg][lane] = pq;
    __syncthreads();
    if (tid < kDVS) {
      const float tk = s_pk[0][lane] + s_pk[1][lane] + s_pk[2][lane] + s_pk[3][lane];
      const float tq = s_pq[0][lane] + s_pq[1][lane] + s_pq[2][lane] + s_pq[3][lane];
      const float u = s_beta * (s_u[lane] - tk);
      store_from_float(out + ((bos + t) * H + h) * DV + j0 + lane, tq + u * khq);
      s_u[lane] = u;
    }
    __syncthreads();
    const float u = s_u[lane];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int c = rg + 4 * i;
      S[i] = s_d[c] * S[i] + s_k[c] * u;
    }
    __syncthreads();  // shared vectors are rewritten by the next token
  }

  if (a.final_state) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int c = rg + 4 * i;
      a.final_state[state_off + (long long)c * DV + j0 + lane] = S[i];
    }
  }
}

template <typename Tin, int DK>
cudaError_t launch_t(const ChunkArgs& a, cudaStream_t st) {
  const dim3 grid(a.dv / kDVS, a.H, a.B);
  recurrent_kernel<Tin, DK><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dtype(const ChunkArgs& a, cudaStream_t st) {
  switch (a.dk) {
    case 32: return launch_t<Tin, 32>(a, st);
    case 64: return launch_t<Tin, 64>(a, st);
    default: return launch_t<Tin, 128>(a, st);
  }
}

}  // namespace

cudaError_t launch_recurrent(const ChunkArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? launch_dtype<__nv_bfloat16>(a, st) : launch_dtype<float>(a, st);
}

}  // namespace kda
