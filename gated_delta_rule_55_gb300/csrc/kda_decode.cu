// Single-token KDA decode step (NKI "KDA TKG Kernel API Reference", kda_tkg): for every
// (request b, head h) the fp32 memory S[b, h] ([dk, dv]) is streamed from HBM exactly
// once, decayed, given the delta-rule write and written back in place, while the output
// o = S_new^T q^ is formed from the same registers.
//
// Per (b, h), with S' = diag(exp(gamma)) S:
//   p_k = S'^T k^,  p_q = S'^T q^            (reductions over the dk rows)
//   u   = beta (v - p_k)
//   S   = S' + k^ u^T
//   o   = S^T q^ = p_q + u (k^ . q^)
// Every value column is independent (the reductions run over dk only), so one pass
// over S suffices.  The kernel is bound by HBM: 2 * dk * dv * 4 bytes of state traffic
// against ~6 flops per state element.
//
// Layout of the work: one CTA of 128 threads per (b, h, 64-column slice); thread
// (rg, cg) owns columns 4cg..4cg+3 of the rows rg, rg + NRG, ... so that a warp reads
// 256-byte row segments as 16-byte vectors (coalesced, one pass, no shared-memory
// staging).  Small CTAs keep several slices in flight per SM.
#include "kda_internal.cuh"

namespace kda {
namespace {

// Column-slice blocks: every (b, h) state tile is cut into DV / DVB independent slices
// of DVB value columns (the reductions run over dk only, so slices never interact); the
// small per-(b, h) prologue is recomputed by each slice.
template <int DK, int DV, int DVB, int NT>
__global__ void __launch_bounds__(NT) decode_kernel(DecodeArgs a) {
  constexpr int NCG = DVB / 4;                 // 16-byte column groups per row slice
  constexpr int NRG = NT / NCG;                // row groups
  constexpr int RPT = DK / NRG;                // rows per thread
  constexpr int NSL = DV / DVB;                // slices per (b, h)
  static_assert(DK % NRG == 0 && RPT >= 1 && NT >= DK && NT >= DVB, "tile shape");

  __shared__ float s_k[DK], s_q[DK], s_dec[DK];
  __shared__ float s_v[DVB], s_u[DVB];
  __shared__ __align__(16) float s_red_k[NRG][DVB + 4];
  __shared__ __align__(16) float s_red_q[NRG][DVB + 4];
  __shared__ float s_norm[3][4];
  __shared__ float s_beta;

  const int tid = threadIdx.x;
  const int cg = tid % NCG;
  const int rg = tid / NCG;
  const long long blk = blockIdx.x;
  const long long bh = blk / NSL;
  const int j0 = (int)(blk % NSL) * DVB;
  const int b = (int)(bh / a.H);
  const int h = (int)(bh % a.H);

  // 1. Put this slice of the state in flight first (streaming: touched once per step).
  float4* Sp = reinterpret_cast<float4*>(a.S + bh * (long long)(DK * DV) + j0);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = __ldcs(Sp + (i * NRG + rg) * (DV / 4) + cg);

  // 2. Prologue while the state loads are in flight: gate, norms, beta.
  float kq = 0.f;
  if (tid < DK) {
    const int c = tid;
    const long long off = ((long long)b * DK + c) * a.H + h;  // [B, dk, H]
    const float kc = a.k[off], qc = a.q[off], gc = a.g[off];
    const float gamma = gate_gamma(gc, a.dt_bias[c * a.H + h], expf(a.a_log[h]),
                                   a.lower_bound);
    s_dec[c] = expf(gamma);
    s_k[c] = kc;
    s_q[c] = qc;
    const float kk = warp_sum(kc * kc), qq = warp_sum(qc * qc), kqs = warp_sum(kc * qc);
    if ((tid & 31) == 0) {
      s_norm[0][tid >> 5] = kk;
      s_norm[1][tid >> 5] = qq;
      s_norm[2][tid >> 5] = kqs;
    }
  }
  if (tid < DVB) s_v[tid] = a.v[bh * DV + j0 + tid];  // [B, H, dv]
  if (tid == 0) s_beta = sigmoidf_(a.beta_logits[bh]);  // [B, 1, H]
  __syncthreads();
  {
    float k2 = 0.f, q2 = 0.f, kq2 = 0.f;
#pragma unroll
    for (int w = 0; w < DK / 32; ++w) {
      k2 += s_norm[0][w];
      q2 += s_norm[1][w];
      kq2 += s_norm[2][w];
    }
    const float rk = 1.0f / sqrtf(k2 + kL2Eps);
    const float rq = a.scale / sqrtf(q2 + kL2Eps);
    kq = kq2 * rk * rq;  // k^ . q^ (scale included)
    __syncthreads();     // everyone has read s_norm / raw s_k, s_q
    if (tid < DK) {
      s_k[tid] *= rk;
      s_q[tid] *= rq;
    }
  }
  __syncthreads();

  // 3. Decay and the two partial reductions over this thread's rows.
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = i * NRG + rg;
    const float d = s_dec[row], kr = s_k[row], qr = s_q[row];
    s[i].x *= d; s[i].y *= d; s[i].z *= d; s[i].w *= d;
    pk.x += s[i].x * kr; pk.y += s[i].y * kr; pk.z += s[i].z * kr; pk.w += s[i].w * kr;
    pq.x += s[i].x * qr; pq.y += s[i].y * qr; pq.z += s[i].z * qr; pq.w += s[i].w * qr;
  }
  *reinterpret_cast<float4*>(&s_red_k[rg][4 * cg]) = pk;
  *reinterpret_cast<float4*>(&s_red_q[rg][4 * cg]) = pq;
  __syncthreads();

  // 4. Column totals, the delta u and the output.
  if (tid < DVB) {
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int r = 0; r < NRG; ++r) {
      sk += s_red_k[r][tid];
      sq += s_red_q[r][tid];
    }
    const float u = s_beta * (s_v[tid] - sk);
    s_u[tid] = u;
    a.out[bh * DV + j0 + tid] = sq + u * kq;  // [B, H, dv]
  }
  __syncthreads();

  // 5. Rank-1 delta write and the in-place store.
  const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * cg]);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const float kr = s_k[i * NRG + rg];
    s[i].x += kr * u4.x; s[i].y += kr * u4.y; s[i].z += kr * u4.z; s[i].w += kr * u4.w;
    __stcs(Sp + (i * NRG + rg) * (DV / 4) + cg, s[i]);
  }
}

template <int DK, int DV>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
  // 64-column slices of 128 threads (16 rows x 4 columns per thread) for the wide tiles;
  // whole tiles for the narrow ones.
  constexpr int DVB = DV > 64 ? 64 : DV;
  constexpr int NT = DK > DVB ? DK : DVB;
  const dim3 grid((unsigned)((long long)a.B * a.H * (DV / DVB)));
  decode_kernel<DK, DV, DVB, (NT < 128 ? 128 : NT)><<<grid, (NT < 128 ? 128 : NT), 0, st>>>(a);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const DecodeArgs& a, cudaStream_t st) {
  switch (a.dv) {
    case 32: return launch_t<DK, 32>(a, st);
    case 64: return launch_t<DK, 64>(a, st);
    default: return launch_t<DK, 128>(a, st);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  switch (a.dk) {
    case 32: return launch_dk<32>(a, st);
    case 64: return launch_dk<64>(a, st);
    default: return launch_dk<128>(a, st);
  }
}

}  // namespace kda

namespace kda {
// The decode kernel has no bounded waits (it synchronises only with __syncthreads), so it
// records no device-side errors.
unsigned int decode_read_error(bool) { return 0; }
}  // namespace kda
