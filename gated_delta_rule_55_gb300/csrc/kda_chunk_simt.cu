// Chunked KDA forward on the fp32 SIMT pipes: the accurate path (fp32 inputs to 1e-4)
// and the general fallback for shapes the tensor-core kernel does not take.
//
// One CTA per (sequence, head, 32-wide slice of dv) walks its sequence in chunks of 16
// tokens (one sub-chunk of the chunked algorithm; the result does not depend on the
// chunk size beyond rounding).  Per chunk, with G_r the in-chunk cumulative log-decay
// (kernel_delta_attention page, "Algorithm modes: chunked"; decay-first recurrence):
//   Xk_r = k^_r e^{G_r}, Xq_r = q^_r e^{G_r}, Kd_s = k^_s e^{-G_s}      (|G| <= 16*5)
//   (literal order, the error term reading the memory before the token's decay:
//    Xk_r = k^_r e^{G_{r-1}}; everything else is unchanged)
//   A_rs = Xk_r . Kd_s (s < r),  M_rs = Xq_r . Kd_s (s <= r)             (gate-scaled K K^T, Q K^T)
//   T    = (I + diag(beta) A)^{-1} diag(beta)                            (UT / WY transform)
//   W    = T Xk,  U~ = T V
//   U    = U~ - W S,  O = Xq S + M U,  S <- diag(e^{G_C}) S + (Kd e^{G_C})^T U
// The dv slice only changes the value columns, so slices are independent.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kC = 16;      // tokens per chunk
constexpr int kDVS = 32;    // value columns per CTA
constexpr int kThreads = 128;

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreads) chunk_simt_kernel(ChunkArgs a) {
  constexpr int LD = DK + 1;  // padded row pitch for row-dot-row products
  extern __shared__ float smem[];
  float* sQ = smem;                 // [kC][LD]  q^ then Xq
  float* sK = sQ + kC * LD;         // [kC][LD]  k^ then Xk
  float* sKd = sK + kC * LD;        // [kC][LD]  k^ e^{-G}
  float* sKh = sKd + kC * LD;       // [kC][LD]  k^ e^{G_C - G}
  float* sW = sKh + kC * LD;        // [kC][LD]  W = T Xk
  float* sG = sW + kC * LD;         // [kC][DK]  raw g, then G
  float* sS = sG + kC * DK;         // [DK][kDVS] state slice (fp32 master)
  float* sV = sS + DK * kDVS;       // [kC][kDVS]
  float* sU = sV + kC * kDVS;       // [kC][kDVS] U~ then U
  float* sA = sU + kC * kDVS;       // [kC][kC+1]
  float* sM = sA + kC * (kC + 1);   // [kC][kC+1]
  float* sT = sM + kC * (kC + 1);   // [kC][kC+1]
  float* sDec = sT + kC * (kC + 1); // [DK] e^{G_C}
  float* sBeta = sDec + DK;         // [kC]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int j0 = blockIdx.x * kDVS;
  const int h = blockIdx.y;
  const int seq = blockIdx.z;
  const int H = a.H, DV = a.dv;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);

  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  Tin* out = static_cast<Tin*>(a.out);
  const long long state_off = ((long long)seq * H + h) * DK * DV;
  const float exp_a = a.gate_head ? 0.f : expf(a.a_log[h]);

  // State slice: initial_state or zeros.
  for (int i = tid; i < DK * kDVS; i += kThreads) {
    const int c = i / kDVS, j = i % kDVS;
    sS[i] = a.initial_state ? a.initial_state[state_off + (long long)c * DV + j0 + j] : 0.f;
  }

  for (int t0 = 0; t0 < len; t0 += kC) {
    const int n = min(kC, len - t0);
    __syncthreads();  // previous chunk fully consumed

    // -- load the chunk (rows >= n are zero)
    for (int i = tid; i < kC * DK; i += kThreads) {
      const int r = i / DK, c = i % DK;
      float xq = 0.f, xk = 0.f, xg = 0.f;
      if (r < n) {
        const long long off = ((bos + t0 + r) * H + h) * DK + c;
        xq = load_as_float(q + off);
        xk = load_as_float(k + off);
        if (!a.gate_head)
          xg = a.g[off];
        else if (a.decay)
          xg = a.decay[(bos + t0 + r) * H + h];  // one log-decay for every channel
      }
      sQ[r * LD + c] = xq;
      sK[r * LD + c] = xk;
      sG[r * DK + c] = xg;
    }
    for (int i = tid; i < kC * kDVS; i += kThreads) {
      const int r = i / kDVS, j = i % kDVS;
      sV[i] = r < n ? load_as_float(v + ((bos + t0 + r) * H + h) * DV + j0 + j) : 0.f;
    }
    if (tid < kC) {
      float b = 0.f;
      if (tid < n) {
        b = a.beta_logits[(bos + t0 + tid) * H + h];
        if (!a.beta_prob) b = sigmoidf_(b);
      }
      sBeta[tid] = b;
    }
    __syncthreads();

    // -- prologue: L2 norms (warp per row) and the cumulative gate (thread per channel)
    for (int r = warp; r < kC; r += kThreads / 32) {
      float sq = 0.f, sk = 0.f;
      for (int c = lane; c < DK; c += 32) {
        sq += sQ[r * LD + c] * sQ[r * LD + c];
        sk += sK[r * LD + c] * sK[r * LD + c];
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      const float rq = a.no_l2norm ? a.scale : a.scale / sqrtf(sq + kL2Eps);
      const float rk = a.no_l2norm ? 1.0f : 1.0f / sqrtf(sk + kL2Eps);
      for (int c = lane; c < DK; c += 32) {
        sQ[r * LD + c] *= rq;
        sK[r * LD + c] *= rk;
      }
    }
    for (int c = tid; c < DK; c += kThreads) {
      const float db = a.gate_head ? 0.f : a.dt_bias[c * H + h];
      float G = 0.f;
      for (int r = 0; r < n; ++r) {
        G += a.gate_head ? sG[r * DK + c] : gate_gamma(sG[r * DK + c], db, exp_a, a.lower_bound);
        sG[r * DK + c] = G;
      }
    }
    __syncthreads();

    // -- gate factors
    for (int c = tid; c < DK; c += kThreads) {
      const float Gc = sG[(n - 1) * DK + c];
      const float decC = expf(Gc);
      sDec[c] = decC;
      for (int r = 0; r < kC; ++r) {
        float xk = 0.f, xq = 0.f, kd = 0.f, kh = 0.f;
        if (r < n) {
          const float G = sG[r * DK + c];
          const float e = expf(G);
          const float khat = sK[r * LD + c];
          xk = khat * (a.literal ? (r > 0 ? expf(sG[(r - 1) * DK + c]) : 1.f) : e);
          xq = sQ[r * LD + c] * e;
          kd = khat / e;
          kh = khat * expf(Gc - G);
        }
        sK[r * LD + c] = xk;
        sQ[r * LD + c] = xq;
        sKd[r * LD + c] = kd;
        sKh[r * LD + c] = kh;
      }
    }
    __syncthreads();

    // -- intra-chunk products A (strictly lower) and M (lower incl. diagonal)
    for (int i = tid; i < 2 * kC * kC; i += kThreads) {
      const int which = i / (kC * kC), rem = i % (kC * kC);
      const int r = rem / kC, s = rem % kC;
      const float* X = which ? sQ : sK;
      float acc = 0.f;
      if (r < n && (which ? s <= r : s < r)) {
#pragma unroll 8
        for (int c = 0; c < DK; ++c) acc += X[r * LD + c] * sKd[s * LD + c];
      }
      (which ? sM : sA)[r * (kC + 1) + s] = acc;
    }
    __syncthreads();

    // -- T = (I + diag(beta) A)^{-1} diag(beta), one column per thread
    if (tid < kC) {
      const int s = tid;
      float x[kC];
#pragma unroll
      for (int r = 0; r < kC; ++r) {
        float acc = (r == s) ? 1.f : 0.f;
        if (r > s) {
          float dot = 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m) dot += sA[r * (kC + 1) + m] * x[m];
          acc = -sBeta[r] * dot;
        }
        x[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < kC; ++r) sT[r * (kC + 1) + s] = x[r] * sBeta[s];
    }
    __syncthreads();

    // -- W = T Xk, U~ = T V
    for (int c = tid; c < DK; c += kThreads) {
      for (int r = 0; r < kC; ++r) {
        float acc = 0.f;
        for (int s = 0; s <= r; ++s) acc += sT[r * (kC + 1) + s] * sK[s * LD + c];
        sW[r * LD + c] = acc;
      }
    }
    for (int i = tid; i < kC * kDVS; i += kThreads) {
      const int r = i / kDVS, j = i % kDVS;
      float acc = 0.f;
      for (int s = 0; s <= r; ++s) acc += sT[r * (kC + 1) + s] * sV[s * kDVS + j];
      sU[i] = acc;
    }
    __syncthreads();

    // -- U = U~ - W S
    for (int i = tid; i < kC * kDVS; i += kThreads) {
      const int r = i / kDVS, j = i % kDVS;
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < DK; ++c) acc += sW[r * LD + c] * sS[c * kDVS + j];
      sU[i] -= acc;
    }
    __syncthreads();

    // -- O = Xq S + M U  (reads the chunk-start state)
    for (int i = tid; i < kC * kDVS; i += kThreads) {
      const int r = i / kDVS, j = i % kDVS;
      if (r < n) {
        float acc = 0.f;
#pragma unroll 8
        for (int c = 0; c < DK; ++c) acc += sQ[r * LD + c] * sS[c * kDVS + j];
        for (int s = 0; s <= r; ++s) acc += sM[r * (kC + 1) + s] * sU[s * kDVS + j];
        store_from_float(out + ((bos + t0 + r) * H + h) * DV + j0 + j, acc);
      }
    }
    __syncthreads();

    // -- S <- diag(e^{G_C}) S + Kh^T U
    for (int i = tid; i < DK * kDVS; i += kThreads) {
      const int c = i / kDVS, j = i % kDVS;
      float acc = sDec[c] * sS[i];
      for (int s = 0; s < n; ++s) acc += sKh[s * LD + c] * sU[s * kDVS + j];
      sS[i] = acc;
    }
  }
  __syncthreads();
  if (a.final_state) {
    for (int i = tid; i < DK * kDVS; i += kThreads) {
      const int c = i / kDVS, j = i % kDVS;
      a.final_state[state_off + (long long)c * DV + j0 + j] = sS[i];
    }
  }
}

template <int DK>
constexpr size_t simt_smem_bytes() {
  return sizeof(float) * (5 * kC * (DK + 1) + kC * DK + DK * kDVS + 2 * kC * kDVS +
                          3 * kC * (kC + 1) + DK + kC);
}

template <typename Tin, int DK>
cudaError_t launch_t(const ChunkArgs& a, cudaStream_t st) {
  const size_t smem = simt_smem_bytes<DK>();
  cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<Tin, DK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.dv / kDVS, a.H, a.B);
  chunk_simt_kernel<Tin, DK><<<grid, kThreads, smem, st>>>(a);
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

cudaError_t launch_chunk_simt(const ChunkArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? launch_dtype<__nv_bfloat16>(a, st) : launch_dtype<float>(a, st);
}

}  // namespace kda
