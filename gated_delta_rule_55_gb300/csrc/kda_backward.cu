// Backward of the KDA forward (decay-first recurrence, kda_tkg-style gate and beta logits):
// gradients of L = <d_out, out> + <d_final_state, final_state> with respect to q, k, v, the
// raw gate g, the beta logits, a_log, dt_bias and the initial state.  The pages give no
// backward; this is reverse-mode differentiation of each token step,
//
//   S' = D S,  p = S'^T k^,  u = beta (v - p),  S_new = S' + k^ u^T,  o = S_new^T q^
//
// taken in reverse token order with the adjoint dS of S_new:
//
//   dS += q^ do^T;  dq^ = S_new do;  du = dS^T k^;  dv = beta du;  dbeta = du . (v - p)
//   dp = -beta du;  dk^ = dS u + S' dp;  dS' = dS + k^ dp^T
//   dgamma = e^{gamma} * rowsum(dS' * S);  dS <- D dS'
//
// Three launches:
//   bwd_forward_kernel  the forward scan once, keeping the state at every 64-token chunk
//                       boundary (checkpoints);
//   bwd_scan_kernel     chunks in reverse: the chunk's pre-token states are recomputed from
//                       its checkpoint into scratch, then its tokens are walked backwards;
//                       writes dv, d_initial_state and the per-token dq^, dk^, dgamma, dbeta;
//   bwd_post_kernel     elementwise: the L2-norm, sigmoid and gate chain rules, and the
//                       a_log / dt_bias sums (one atomic add per channel and token block).
//
// The value columns of the state are independent in the forward, so every scan runs on
// 32-column slices: one CTA of 128 threads per (sequence, head, slice); thread (rg, j) owns
// column j of the slice on rows rg, rg + 4, ...; the state and its adjoint stay in
// registers.  Sums over all value columns (dq^, dk^, dgamma, dbeta) are written per slice
// and added up by the elementwise pass.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kCK = 64;   // tokens per checkpoint interval
constexpr int kDVS = 32;  // value columns per CTA
constexpr int kBT = 4 * kDVS;  // threads per scan CTA

struct BwdArgs {
  ChunkArgs f;              // forward arguments (q, k, v, g, beta_logits, a_log, dt_bias, ...)
  const void* d_out;        // [B, T, H, dv] dtype
  const float* d_final;     // [B, H, dk, dv] or NULL
  void* dq;                 // [B, T, H, dk] dtype
  void* dk;
  void* dv;                 // [B, T, H, dv] dtype
  float* dg;                // [B, T, H, dk]
  float* dbeta_logits;      // [B, T, H]
  float* da_log;            // [H] (accumulated)
  float* ddt_bias;          // [dk, H] (accumulated)
  float* d_initial;         // [B, H, dk, dv] or NULL
  float* ckpt;              // [B, H, nck, dk, dv]
  float* chunk_states;      // [B, H, kCK, dk, dv]
  float* dqh;               // [ns][B, T, H, dk] per-slice gradient w.r.t. q^ (scale in q^)
  float* dkh;               // [ns][B, T, H, dk]
  float* dgam;              // [ns][B, T, H, dk] gradient w.r.t. gamma
  float* dbeta;             // [ns][B, T, H] gradient w.r.t. beta
  long long rows;           // B * T * H
  int nck;
  int ns;                   // value-column slices (dv / 32)
};

// Per-token quantities shared by the CTA: normalised k and q, decay, v, beta.
template <int DK>
struct TokenSmem {
  float k[DK], q[DK], d[DK];
  float v[kDVS], dout[kDVS];
  float part[3][4];
  float beta;
};

// A token's raw inputs in registers (loaded one step ahead): channel tid of k, q and g
// (tid < DK), column j0 + tid of v and d_out (tid < 32), the beta logit (thread 0).
struct TokenRegs {
  float k, q, g, v, dout, blog;
};

template <typename Tin, int DK>
__device__ __forceinline__ TokenRegs fetch_token(const BwdArgs& b, long long row, int tid, int j0,
                                                 bool want_q) {
  const ChunkArgs& a = b.f;
  const int DV = a.dv;
  TokenRegs r{0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (tid < DK) {
    r.k = load_as_float(static_cast<const Tin*>(a.k) + row * DK + tid);
    if (want_q) r.q = load_as_float(static_cast<const Tin*>(a.q) + row * DK + tid);
    r.g = a.g[row * DK + tid];
  }
  if (tid < kDVS) {
    r.v = load_as_float(static_cast<const Tin*>(a.v) + row * DV + j0 + tid);
    if (want_q) r.dout = load_as_float(static_cast<const Tin*>(b.d_out) + row * DV + j0 + tid);
  }
  if (tid == 0) r.blog = a.beta_logits[row];
  return r;
}

// Stages a fetched token in shared memory: k^, q^ (scale folded), e^{gamma}, this slice's
// v and d_out, beta.  Threads tid < DK own channel tid.  Ends with a barrier.
template <int DK>
__device__ void stage_token(const ChunkArgs& a, const TokenRegs& r, TokenSmem<DK>& s, int tid,
                            float exp_a, float db) {
  const int lane = tid & 31, w = tid >> 5;
  if (tid < DK) {
    s.d[tid] = expf(gate_gamma(r.g, db, exp_a, a.lower_bound));
    const float kk = warp_sum(r.k * r.k), qq = warp_sum(r.q * r.q);
    if (lane == 0) {
      s.part[0][w] = kk;
      s.part[1][w] = qq;
    }
  }
  if (tid < kDVS) {
    s.v[tid] = r.v;
    s.dout[tid] = r.dout;
  }
  if (tid == 0) s.beta = sigmoidf_(r.blog);
  __syncthreads();
  if (tid < DK) {
    float kk = 0.f, qq = 0.f;
#pragma unroll
    for (int i = 0; i < DK / 32; ++i) {
      kk += s.part[0][i];
      qq += s.part[1][i];
    }
    s.k[tid] = r.k * rsqrtf(kk + kL2Eps);
    s.q[tid] = r.q * a.scale * rsqrtf(qq + kL2Eps);
  }
  __syncthreads();
}

// One forward token step on the register state S (rows rg + 4 i of slice column j):
// S <- D S + k^ u^T with u = beta (v - (D S)^T k^).  Uses red[4][kDVS].
template <int DK>
__device__ void forward_step(float (&S)[DK / 4], const TokenSmem<DK>& s, float (*red)[kDVS],
                             int rg, int j) {
  constexpr int RPT = DK / 4;
  float p = 0.f;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int c = rg + 4 * i;
    S[i] *= s.d[c];
    p += S[i] * s.k[c];
  }
  red[rg][j] = p;
  __syncthreads();
  const float u = s.beta * (s.v[j] - (red[0][j] + red[1][j] + red[2][j] + red[3][j]));
#pragma unroll
  for (int i = 0; i < RPT; ++i) S[i] += s.k[rg + 4 * i] * u;
  __syncthreads();  // red[] is rewritten by the next step
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kBT) bwd_forward_kernel(BwdArgs b) {
  constexpr int RPT = DK / 4;
  __shared__ TokenSmem<DK> s;
  __shared__ float red[4][kDVS];
  const ChunkArgs& a = b.f;
  const int tid = threadIdx.x, rg = tid / kDVS, j = tid % kDVS;
  const int j0 = blockIdx.x * kDVS, h = blockIdx.y, seq = blockIdx.z, H = a.H, DV = a.dv;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  const long long sh = (long long)seq * H + h;
  const float exp_a = tid < DK ? expf(a.a_log[h]) : 0.f;
  const float db = tid < DK ? a.dt_bias[tid * H + h] : 0.f;
  float S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    S[i] = a.initial_state ? a.initial_state[sh * DK * DV + (rg + 4 * i) * DV + j0 + j] : 0.f;
  TokenRegs nx = len > 0 ? fetch_token<Tin, DK>(b, bos * H + h, tid, j0, false) : TokenRegs{};
  for (int t = 0; t < len; ++t) {
    if (t % kCK == 0) {
      float* cp = b.ckpt + (sh * b.nck + t / kCK) * DK * DV + j0 + j;
#pragma unroll
      for (int i = 0; i < RPT; ++i) cp[(rg + 4 * i) * DV] = S[i];
    }
    const TokenRegs cur = nx;
    if (t + 1 < len) nx = fetch_token<Tin, DK>(b, (bos + t + 1) * H + h, tid, j0, false);
    stage_token<DK>(a, cur, s, tid, exp_a, db);
    forward_step<DK>(S, s, red, rg, j);
  }
}

// Reduce-scatter of RPT values across the 32 lanes of a warp: afterwards lane l holds, in
// x[0], the warp sum of row index row_of_lane(l) (lanes that share a row hold equal sums).
template <int RPT>
__device__ __forceinline__ void warp_reduce_scatter(float (&x)[RPT], int lane) {
  int bit = 16;
#pragma unroll
  for (int half = RPT / 2; half >= 1; half >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? x[i] : x[i + half];
      const float keep = up ? x[i + half] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
  for (; bit >= 1; bit >>= 1) x[0] += __shfl_xor_sync(0xffffffffu, x[0], bit);
}
template <int RPT>
__device__ __forceinline__ int row_of_lane(int lane) {
  int r = 0, bit = 16;
  for (int half = RPT / 2; half >= 1; half >>= 1, bit >>= 1)
    if (lane & bit) r += half;
  return r;
}
// lanes holding a distinct row after the reduce-scatter (one writer per row): the low
// log2(32 / RPT) lane bits were summed over
template <int RPT>
__device__ __forceinline__ bool row_writer(int lane) {
  return (lane & (32 / RPT - 1)) == 0;
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kBT) bwd_scan_kernel(BwdArgs b) {
  constexpr int RPT = DK / 4;
  __shared__ TokenSmem<DK> s;
  __shared__ float red[4][kDVS];
  __shared__ float bred[4];
  const ChunkArgs& a = b.f;
  const int tid = threadIdx.x, lane = tid & 31, rg = tid / kDVS, j = tid % kDVS;
  const int slice = blockIdx.x, j0 = slice * kDVS, h = blockIdx.y, seq = blockIdx.z;
  const int H = a.H, DV = a.dv;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  const long long sh = (long long)seq * H + h;
  const float exp_a = tid < DK ? expf(a.a_log[h]) : 0.f;
  const float db = tid < DK ? a.dt_bias[tid * H + h] : 0.f;
  // this CTA's chunk scratch: [kCK][DK][kDVS]
  float* const cs = b.chunk_states + (sh * b.ns + slice) * kCK * DK * kDVS;
  const long long pofs = (long long)slice * b.rows;  // offset of this slice's partials

  float dS[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    dS[i] = b.d_final ? b.d_final[sh * DK * DV + (rg + 4 * i) * DV + j0 + j] : 0.f;

  const int nck = (len + kCK - 1) / kCK;
  for (int ck = nck - 1; ck >= 0; --ck) {
    const int t0 = ck * kCK, t1 = min(len, t0 + kCK);
    // recompute the chunk's pre-token states from its checkpoint
    {
      float S[RPT];
      const float* cp = b.ckpt + (sh * b.nck + ck) * DK * DV + j0 + j;
#pragma unroll
      for (int i = 0; i < RPT; ++i) S[i] = cp[(rg + 4 * i) * DV];
      TokenRegs nx = fetch_token<Tin, DK>(b, (bos + t0) * H + h, tid, j0, false);
      for (int t = t0; t < t1; ++t) {
        float* dst = cs + (t - t0) * DK * kDVS + j;
#pragma unroll
        for (int i = 0; i < RPT; ++i) dst[(rg + 4 * i) * kDVS] = S[i];
        if (t + 1 < t1) {  // the last token's own update is not needed
          const TokenRegs cur = nx;
          if (t + 2 < t1) nx = fetch_token<Tin, DK>(b, (bos + t + 1) * H + h, tid, j0, false);
          stage_token<DK>(a, cur, s, tid, exp_a, db);
          forward_step<DK>(S, s, red, rg, j);
        }
      }
    }
    __syncthreads();
    // walk the chunk backwards; the next (earlier) token's inputs and pre-token state are
    // loaded into registers while the current one is processed
    TokenRegs nx = fetch_token<Tin, DK>(b, (bos + t1 - 1) * H + h, tid, j0, true);
    float Sn[RPT];
    {
      const float* src = cs + (t1 - 1 - t0) * DK * kDVS + j;
#pragma unroll
      for (int i = 0; i < RPT; ++i) Sn[i] = src[(rg + 4 * i) * kDVS];
    }
    for (int t = t1 - 1; t >= t0; --t) {
      const long long row = (bos + t) * H + h;
      const TokenRegs cur = nx;
      float Sp[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) Sp[i] = Sn[i];
      if (t > t0) {
        nx = fetch_token<Tin, DK>(b, row - H, tid, j0, true);
        const float* src = cs + (t - 1 - t0) * DK * kDVS + j;
#pragma unroll
        for (int i = 0; i < RPT; ++i) Sn[i] = src[(rg + 4 * i) * kDVS];
      }
      stage_token<DK>(a, cur, s, tid, exp_a, db);
      float p = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int c = rg + 4 * i;
        p += s.d[c] * Sp[i] * s.k[c];
      }
      red[rg][j] = p;
      __syncthreads();
      const float pj = red[0][j] + red[1][j] + red[2][j] + red[3][j];
      const float vmp = s.v[j] - pj;
      const float u = s.beta * vmp;
      const float doj = s.dout[j];
      // dS += q^ do^T, then du = dS^T k^
      float du_part = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int c = rg + 4 * i;
        dS[i] += s.q[c] * doj;
        du_part += dS[i] * s.k[c];
      }
      __syncthreads();  // red[] (p) read by everyone
      red[rg][j] = du_part;
      __syncthreads();
      const float du = red[0][j] + red[1][j] + red[2][j] + red[3][j];
      const float dp = -s.beta * du;
      // per-row partial products over this slice's columns, reduced across the warp's 32
      // lanes (= the slice's columns):
      //   dq^_c = sum_j S_new[c][j] do_j,  dk^_c = sum_j (dS u + S' dp),
      //   dgamma_c / d_c = sum_j dS'[c][j] S[c][j]   (then dS <- D dS')
      float x[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int c = rg + 4 * i;
        x[i] = (s.d[c] * Sp[i] + s.k[c] * u) * doj;
      }
      warp_reduce_scatter<RPT>(x, lane);
      if (row_writer<RPT>(lane))
        b.dqh[(pofs + row) * DK + rg + 4 * row_of_lane<RPT>(lane)] = x[0];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int c = rg + 4 * i;
        x[i] = dS[i] * u + s.d[c] * Sp[i] * dp;
      }
      warp_reduce_scatter<RPT>(x, lane);
      if (row_writer<RPT>(lane))
        b.dkh[(pofs + row) * DK + rg + 4 * row_of_lane<RPT>(lane)] = x[0];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int c = rg + 4 * i;
        const float dSd = dS[i] + s.k[c] * dp;  // dS'
        x[i] = dSd * Sp[i];
        dS[i] = s.d[c] * dSd;                   // adjoint of the previous state
      }
      warp_reduce_scatter<RPT>(x, lane);
      if (row_writer<RPT>(lane)) {
        const int c = rg + 4 * row_of_lane<RPT>(lane);
        b.dgam[(pofs + row) * DK + c] = x[0] * s.d[c];
      }
      // dv and the dbeta partial (row group 0 holds one copy of every slice column)
      if (rg == 0) {
        store_from_float(static_cast<Tin*>(b.dv) + row * DV + j0 + j, s.beta * du);
        const float dbp = warp_sum(du * vmp);
        if (lane == 0) b.dbeta[pofs + row] = dbp;
      }
      __syncthreads();  // shared token data and red[] are rewritten by the next token
    }
  }
  if (b.d_initial) {
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      b.d_initial[sh * DK * DV + (rg + 4 * i) * DV + j0 + j] = dS[i];
  }
}

// Elementwise chain rules per token row, one warp per (token, head) row; each CTA takes
// kPostTok tokens of one (sequence, head) and accumulates dt_bias / a_log partials.
constexpr int kPostTok = 32;

template <typename Tin, int DK>
__global__ void __launch_bounds__(128) bwd_post_kernel(BwdArgs b) {
  constexpr int CPL = DK / 32;  // channels per lane
  const ChunkArgs& a = b.f;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int h = blockIdx.x, seq = blockIdx.z, H = a.H;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  const int tb = blockIdx.y * kPostTok;
  const float ea = expf(a.a_log[h]);
  float db[CPL], acc_b[CPL];
#pragma unroll
  for (int m = 0; m < CPL; ++m) {
    db[m] = a.dt_bias[(lane + 32 * m) * H + h];
    acc_b[m] = 0.f;
  }
  float acc_a = 0.f;
  for (int tt = w; tt < kPostTok; tt += 4) {
    const int t = tb + tt;
    if (t >= len) break;
    const long long row = (bos + t) * H + h;
    float qv[CPL], kv[CPL], dq[CPL], dk[CPL];
    float qq = 0.f, kk = 0.f, qd = 0.f, kd = 0.f;
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
      const int c = lane + 32 * m;
      qv[m] = load_as_float(static_cast<const Tin*>(a.q) + row * DK + c);
      kv[m] = load_as_float(static_cast<const Tin*>(a.k) + row * DK + c);
      float sq = 0.f, sk = 0.f;
      for (int sl = 0; sl < b.ns; ++sl) {
        sq += b.dqh[(sl * b.rows + row) * DK + c];
        sk += b.dkh[(sl * b.rows + row) * DK + c];
      }
      dq[m] = a.scale * sq;
      dk[m] = sk;
      qq += qv[m] * qv[m];
      kk += kv[m] * kv[m];
      qd += qv[m] * dq[m];
      kd += kv[m] * dk[m];
    }
    qq = warp_sum(qq); kk = warp_sum(kk); qd = warp_sum(qd); kd = warp_sum(kd);
    const float rq = rsqrtf(qq + kL2Eps), rk = rsqrtf(kk + kL2Eps);
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
      const int c = lane + 32 * m;
      store_from_float(static_cast<Tin*>(b.dq) + row * DK + c,
                       dq[m] * rq - qv[m] * qd * rq * rq * rq);
      store_from_float(static_cast<Tin*>(b.dk) + row * DK + c,
                       dk[m] * rk - kv[m] * kd * rk * rk * rk);
      // gamma = lb sigmoid(z), z = e^{a_log} (g + dt_bias)
      const float z = ea * (a.g[row * DK + c] + db[m]);
      const float sz = sigmoidf_(z);
      float dgm = 0.f;
      for (int sl = 0; sl < b.ns; ++sl) dgm += b.dgam[(sl * b.rows + row) * DK + c];
      const float dz = dgm * a.lower_bound * sz * (1.f - sz);
      b.dg[row * DK + c] = dz * ea;
      acc_b[m] += dz * ea;
      acc_a += dz * z;
    }
    if (lane == 0) {
      const float beta = sigmoidf_(a.beta_logits[row]);
      float dbt = 0.f;
      for (int sl = 0; sl < b.ns; ++sl) dbt += b.dbeta[sl * b.rows + row];
      b.dbeta_logits[row] = dbt * beta * (1.f - beta);
    }
  }
#pragma unroll
  for (int m = 0; m < CPL; ++m) atomicAdd(&b.ddt_bias[(lane + 32 * m) * H + h], acc_b[m]);
  acc_a = warp_sum(acc_a);
  if (lane == 0) atomicAdd(&b.da_log[h], acc_a);
}

template <typename Tin, int DK>
cudaError_t launch_t(const BwdArgs& b, cudaStream_t st) {
  const ChunkArgs& a = b.f;
  const dim3 grid(b.ns, a.H, a.B);
  bwd_forward_kernel<Tin, DK><<<grid, kBT, 0, st>>>(b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_scan_kernel<Tin, DK><<<grid, kBT, 0, st>>>(b);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 pgrid(a.H, (a.T + kPostTok - 1) / kPostTok, a.B);
  if (a.T > 0) bwd_post_kernel<Tin, DK><<<pgrid, 128, 0, st>>>(b);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dtype(const BwdArgs& b, cudaStream_t st) {
  switch (b.f.dk) {
    case 32: return launch_t<Tin, 32>(b, st);
    case 64: return launch_t<Tin, 64>(b, st);
    default: return launch_t<Tin, 128>(b, st);
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t backward_workspace(int B, int T, int H, int dk, int dv) {
  const size_t nck = (size_t)(T + kCK - 1) / kCK;
  const size_t st = (size_t)dk * dv * 4;
  const size_t rows = (size_t)B * T * H, ns = (size_t)dv / kDVS;
  return align256((size_t)B * H * nck * st) + align256((size_t)B * H * kCK * st) +
         3 * align256(ns * rows * dk * 4) + align256(ns * rows * 4);
}

cudaError_t launch_backward(const ChunkArgs& f, const void* d_out, const float* d_final,
                            void* dq, void* dk, void* dv, float* dg, float* dbeta_logits,
                            float* da_log, float* ddt_bias, float* d_initial, void* workspace,
                            bool bf16, cudaStream_t st) {
  BwdArgs b{};
  b.f = f;
  b.d_out = d_out; b.d_final = d_final;
  b.dq = dq; b.dk = dk; b.dv = dv; b.dg = dg; b.dbeta_logits = dbeta_logits;
  b.da_log = da_log; b.ddt_bias = ddt_bias; b.d_initial = d_initial;
  b.nck = (f.T + kCK - 1) / kCK;
  b.ns = f.dv / kDVS;
  const size_t st_bytes = (size_t)f.dk * f.dv * 4;
  const size_t rows = (size_t)f.B * f.T * f.H;
  b.rows = (long long)rows;
  uint8_t* p = static_cast<uint8_t*>(workspace);
  b.ckpt = reinterpret_cast<float*>(p);
  p += align256((size_t)f.B * f.H * b.nck * st_bytes);
  b.chunk_states = reinterpret_cast<float*>(p);
  p += align256((size_t)f.B * f.H * kCK * st_bytes);
  b.dqh = reinterpret_cast<float*>(p);
  p += align256(b.ns * rows * f.dk * 4);
  b.dkh = reinterpret_cast<float*>(p);
  p += align256(b.ns * rows * f.dk * 4);
  b.dgam = reinterpret_cast<float*>(p);
  p += align256(b.ns * rows * f.dk * 4);
  b.dbeta = reinterpret_cast<float*>(p);
  cudaError_t e = cudaMemsetAsync(da_log, 0, sizeof(float) * f.H, st);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * f.dk * f.H, st)) != cudaSuccess) return e;
  return bf16 ? launch_dtype<__nv_bfloat16>(b, st) : launch_dtype<float>(b, st);
}

}  // namespace kda
