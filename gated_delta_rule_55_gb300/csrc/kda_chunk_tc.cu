// Chunked KDA forward on the 5th-generation tensor cores (tcgen05) for bf16 q/k/v with
// dk = dv = 128 and 64-token chunks.
//
// One CTA of 512 threads (4 warpgroups) walks one (sequence, head) pair chunk by chunk.
// Per chunk (kernel_delta_attention page, "Algorithm modes: chunked"; decay-first
// recurrence), with G the in-chunk cumulative log-decay and the chunk cut into four
// 16-token sub-chunks R whose reference point P_R is G just before the sub-chunk:
//
//  prologue (SIMT, fused): L2 norms of q and k, gate activation and its cumulative sum,
//    beta, and the gate-scaled operands
//      Xl = [k^_r e^{G_r - P_R}; q^_r e^{G_r - P_R}]                 (128 x dk, smem)
//      Kb = [k^_s e^{P_S - G_s} (diagonal sub-chunks);                (160 x dk, smem)
//            the same times e^{P_R - P_S} for every later sub-chunk R]
//      Q~ = q^ e^{G}, K^^T = (k^ e^{G_C - G})^T, K~^T = (k^ e^{G})^T, V^T
//  MMA1  [A; M] = Xl Kb^T                              gate-scaled K K^T and Q K^T
//  solve T = (I + diag(beta) tril(A, -1))^{-1} diag(beta)     (fp32, blocked by 16)
//  MMA2  W^T = K~^T T^T,  U~^T = V^T T^T                         (UT / WY transform)
//  MMA3  U^T = U~^T - S^T W^T,  O^T = S^T Q~^T
//  MMA4  O^T += U^T M^T (M = tril(QK^T-part)),  dS^T = U^T K^
//  state S^T <- S^T diag(e^{G_C}) + dS^T   (fp32 master in registers, bf16 copy in TMEM)
//
// The sequential dependence is only through S; everything is oriented so that the value
// index j is the TMEM lane (M = dv = 128) for the state-dependent products, and the
// state-independent operands are built by the same threads that hold the gate sums.
// Every exponential factor is <= e^{80} or >= e^{-80} (lower_bound >= -5), so nothing
// leaves the fp32 / bf16 exponent range.
#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "tc_prims.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kKbRows = 160;  // 64 diagonal + 16 + 32 + 48 off-diagonal key rows

// Dynamic shared memory (byte offsets from a 1024-aligned base).
constexpr int OFF_Q = 0;                    // raw q tile, two SW128 boxes [64 tok x 64 ch]
constexpr int OFF_K = OFF_Q + 16384;        // raw k tile
constexpr int OFF_V = OFF_K + 16384;        // raw v tile
constexpr int OFF_XL = OFF_V + 16384;       // Xl [128 x 128] bf16, K-major SW128
constexpr int OFF_KB = OFF_XL + 32768;      // Kb [160 x 128]
constexpr int OFF_QT = OFF_KB + 40960;      // Q~ [64 x 128]
constexpr int OFF_KHT = OFF_QT + 16384;     // K^^T [128 x 64]
constexpr int OFF_M = OFF_KHT + 16384;      // M [64 x 64]
constexpr int OFF_END = OFF_M + 8192;
// Re-used inside the Xl/Kb region once MMA1 has completed.
constexpr int LDL = 65;
constexpr int OFF_L = OFF_XL;               // fp32 [64][65] beta-scaled strict lower A
constexpr int OFF_X = OFF_L + 16896;        // fp32 [64][65] (I + L)^{-1}
constexpr int OFF_T = OFF_XL + 34816;       // T [64 x 64] bf16 SW128 (1024-aligned)
constexpr int OFF_W = OFF_T + 8192;         // -W [64 x 128] bf16 SW128
constexpr int OFF_Y = OFF_W + 16384;        // fp32 [3][16][16] solve temporaries
static_assert(OFF_Y + 3072 <= OFF_QT, "solve scratch must fit in the Xl/Kb region");
constexpr size_t kSmemBytes = OFF_END + 1024;

// Tensor Memory columns (512 allocated).
constexpr uint32_t TM_D1 = 0;     // [A; M] accumulator, 160 columns
constexpr uint32_t TM_DW = 0;     // W^T accumulator (after D1 is consumed), 64
constexpr uint32_t TM_KT = 64;    // K~^T A operand (bf16 pairs), 32
constexpr uint32_t TM_UA = 128;   // U^T A operand, 32
constexpr uint32_t TM_DU = 160;   // U~^T then U^T accumulator, 64
constexpr uint32_t TM_DO = 224;   // O^T accumulator, 64
constexpr uint32_t TM_DS = 288;   // dS^T accumulator, 128
constexpr uint32_t TM_SA = 416;   // S^T A operand, 64
constexpr uint32_t TM_VA = 480;   // V^T A operand, 32
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kTxBytes = 3 * 16384;  // q, k, v tiles per chunk

__device__ unsigned int g_tc_error;  // bit 0: an mbarrier wait timed out

struct TcParams {
  ChunkArgs a;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__device__ __forceinline__ void st_bf16(uint8_t* base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float ld_bf16(const uint8_t* base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

// tcgen05.st of 8 columns (shape 32x32b, x8), waited for.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ float s_rk[kC], s_rq[kC], s_beta[kC], s_dec[kD];
  __shared__ float s_gtot[4][kD];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7;            // warpgroup: token quarter / channel quarter
  const int ln = tid & 127;           // TMEM lane of this thread = channel c or value j
  const int lane_base = 32 * (warp & 3);
  const int h = blockIdx.x, seq = blockIdx.y;
  const int H = a.H;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  const long long state_off = ((long long)seq * H + h) * kD * kD;

  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(lane_base) << 16);  // this warp's lane window

  // Initial state: thread (j = ln, quarter wg) owns S^T[j][32 wg .. 32 wg + 31] in fp32.
  float S[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int c = 32 * wg + i;
    S[i] = a.initial_state ? a.initial_state[state_off + (long long)c * kD + ln] : 0.f;
  }
  {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
    tmem_st16(tl + TM_SA + 16 * wg, w);
  }

  const float exp_a = expf(a.a_log[h]);
  const float db = a.dt_bias[ln * H + h];
  const int nchunks = (len + kC - 1) / kC;
  const uint32_t idesc_m160 = make_idesc(1, 128, 160);
  const uint32_t idesc_m64 = make_idesc(1, 128, 64);
  const uint32_t idesc_m128 = make_idesc(1, 128, 128);
  uint32_t mma_phase = 0;
  bool ok = true;
  bool tma_pending = false;   // a TMA batch was issued and not yet waited for
  uint32_t tma_parity = 0;    // parity of that batch

  if (tid == 0 && nchunks > 0) {
    mbar_arrive_expect_tx(&bar_tma, kTxBytes);
    for (int half = 0; half < 2; ++half) {
      const int row = (int)bos;
      tma_load_3d(sm + OFF_Q + half * 8192, &map_q, &bar_tma, 64 * half, h, row);
      tma_load_3d(sm + OFF_K + half * 8192, &map_k, &bar_tma, 64 * half, h, row);
      tma_load_3d(sm + OFF_V + half * 8192, &map_v, &bar_tma, 64 * half, h, row);
    }
  }
  tma_pending = nchunks > 0;
  tma_parity = 0;

  // Raw gates of this thread's channel and token quarter, loaded one chunk ahead.
  float graw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int t = 16 * wg + i;
    graw[i] = (t < len) ? a.g[((bos + t) * H + h) * kD + ln] : 0.f;
  }

  auto mma_wait = [&]() -> bool {
    const bool w = mbar_wait(&bar_mma, mma_phase & 1);
    ++mma_phase;
    return w;
  };

  for (int ch = 0; ch < nchunks; ++ch) {
    const int t0 = ch * kC;
    const int n = min(kC, len - t0);
    const long long tok0 = bos + t0;

    // ---------------- prologue: beta, norms, gates
    if (tid < kC) {
      s_beta[tid] = tid < n ? sigmoidf_(a.beta_logits[(tok0 + tid) * H + h]) : 0.f;
    }
    bool w = mbar_wait(&bar_tma, ch & 1);
    if (!__syncthreads_and(w)) { ok = false; break; }
    tma_pending = false;
    {
      // warp w reduces tokens 4w .. 4w + 3 of q and k; lane holds channels 4l .. 4l + 3
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = 4 * warp + u;
        const uint32_t off = sw128_offset<2>(64, t, 4 * lane);
        const uint2 qv = *reinterpret_cast<const uint2*>(sm + OFF_Q + off);
        const uint2 kv = *reinterpret_cast<const uint2*>(sm + OFF_K + off);
        float sq = 0.f, sk = 0.f;
        const uint32_t qw[2] = {qv.x, qv.y}, kw[2] = {kv.x, kv.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float q0 = __uint_as_float(qw[e] << 16), q1 = __uint_as_float(qw[e] & 0xffff0000u);
          const float k0 = __uint_as_float(kw[e] << 16), k1 = __uint_as_float(kw[e] & 0xffff0000u);
          sq += q0 * q0 + q1 * q1;
          sk += k0 * k0 + k1 * k1;
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (lane == 0) {
          s_rq[t] = t < n ? a.scale / sqrtf(sq + kL2Eps) : 0.f;
          s_rk[t] = t < n ? 1.0f / sqrtf(sk + kL2Eps) : 0.f;
        }
      }
    }
    // gate: per channel ln, tokens 16 wg .. 16 wg + 15, local inclusive prefix
    float gl[16];
    {
      float run = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = 16 * wg + i;
        const float gam = (t < n) ? gate_gamma(graw[i], db, exp_a, a.lower_bound) : 0.f;
        run += gam;
        gl[i] = run;
      }
      s_gtot[wg][ln] = run;
    }
    __syncthreads();
    // prefetch the next chunk's raw gates (consumed at the next prologue)
    if (ch + 1 < nchunks) {
      const int tn = t0 + kC;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = tn + 16 * wg + i;
        graw[i] = (t < len) ? a.g[((bos + t) * H + h) * kD + ln] : 0.f;
      }
    }
    // per-channel reference points: P_R = sum of the totals of quarters < R
    float P[4];
    P[0] = 0.f;
    P[1] = s_gtot[0][ln];
    P[2] = P[1] + s_gtot[1][ln];
    P[3] = P[2] + s_gtot[2][ln];
    const float Gc = P[3] + s_gtot[3][ln];
    const float Pme = P[wg];
    const float eP = expf(Pme);            // e^{P_R}
    const float eCP = expf(Gc - Pme);      // e^{G_C - P_R}
    float cR[4];                           // e^{P_R' - P_R} for later sub-chunks R'
#pragma unroll
    for (int r = 0; r < 4; ++r) cR[r] = (r > wg) ? expf(P[r] - Pme) : 0.f;
    if (wg == 0) s_dec[ln] = expf(Gc);

    // ---------------- gate-scaled operands for this thread's (channel, 16 tokens)
    uint32_t kt_pack[8], vt_pack[8];
    {
      const int c = ln;
      float kh_prev = 0.f, kt_prev = 0.f, v_prev = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = 16 * wg + i;
        const uint32_t roff = sw128_offset<2>(64, t, c);
        const float kr = ld_bf16(sm + OFF_K, roff) * s_rk[t];
        const float qr = ld_bf16(sm + OFF_Q, roff) * s_rq[t];
        const float vr = (t < n) ? ld_bf16(sm + OFF_V, roff) : 0.f;
        const float e = expf(gl[i]);       // e^{G_t - P_R} in [e^{-80}, 1]
        const float kd = kr / e;           // k^ e^{P_R - G_t}, at most e^{80}
        const float xk = kr * e, xq = qr * e;
        st_bf16(sm + OFF_XL, sw128_offset<2>(128, t, c), xk);
        st_bf16(sm + OFF_XL, sw128_offset<2>(128, 64 + t, c), xq);
        st_bf16(sm + OFF_KB, sw128_offset<2>(kKbRows, t, c), kd);
        if (wg < 1) st_bf16(sm + OFF_KB, sw128_offset<2>(kKbRows, 64 + t, c), kd * cR[1]);
        if (wg < 2) st_bf16(sm + OFF_KB, sw128_offset<2>(kKbRows, 80 + t, c), kd * cR[2]);
        if (wg < 3) st_bf16(sm + OFF_KB, sw128_offset<2>(kKbRows, 112 + t, c), kd * cR[3]);
        st_bf16(sm + OFF_QT, sw128_offset<2>(64, t, c), xq * eP);  // q^ e^{G_t}
        const float kh = kd * eCP;         // k^ e^{G_C - G_t}
        const float ktil = xk * eP;        // k^ e^{G_t}
        if (i & 1) {
          // K^^T row c holds tokens contiguously: store the pair (t - 1, t)
          *reinterpret_cast<uint32_t*>(sm + OFF_KHT + sw128_offset<2>(128, c, t - 1)) =
              pack_bf16(kh_prev, kh);
          kt_pack[i >> 1] = pack_bf16(kt_prev, ktil);
          vt_pack[i >> 1] = pack_bf16(v_prev, vr);
        }
        kh_prev = kh;
        kt_prev = ktil;
        v_prev = vr;
      }
    }
    tmem_st8(tl + TM_VA + 8 * wg, vt_pack);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // raw tiles are consumed: start the next chunk's loads now
    if (tid == 0 && ch + 1 < nchunks) {
      const int row = (int)(tok0 + kC);
      mbar_arrive_expect_tx(&bar_tma, kTxBytes);
      for (int half = 0; half < 2; ++half) {
        tma_load_3d(sm + OFF_Q + half * 8192, &map_q, &bar_tma, 64 * half, h, row);
        tma_load_3d(sm + OFF_K + half * 8192, &map_k, &bar_tma, 64 * half, h, row);
        tma_load_3d(sm + OFF_V + half * 8192, &map_v, &bar_tma, 64 * half, h, row);
      }
    }
    tma_pending = (ch + 1 < nchunks);
    tma_parity = (ch + 1) & 1;

    // ---------------- MMA1: [A; M] = Xl Kb^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t xa = smem_u32(sm + OFF_XL), kb = smem_u32(sm + OFF_KB);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ss(tm + TM_D1, sw128_kdesc<2>(xa, 128, s), sw128_kdesc<2>(kb, kKbRows, s),
               idesc_m160, s > 0);
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!__syncthreads_and(w)) { ok = false; break; }
    tc_fence_after();

    // ---------------- read A (lanes 0..63) and M (lanes 64..127)
    if (wg == 0) {
      const int r = ln & 63;
      const int R = r >> 4;
      float* L = reinterpret_cast<float*>(sm + OFF_L);
      const bool is_a = ln < 64;
      const float br = s_beta[r];
      float rowv[64];
#pragma unroll
      for (int m = 0; m < 64; ++m) rowv[m] = 0.f;
      // Every warp loads the same columns (tcgen05.ld is warp-collective); each lane keeps
      // the blocks of its own sub-chunk R.  Diagonal block: columns 16q .. 16q + 15.
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v16[16];
        tmem_ld16(tl + TM_D1 + 16 * q, v16);
#pragma unroll
        for (int m = 0; m < 16; ++m) rowv[16 * q + m] = (q == R) ? v16[m] : rowv[16 * q + m];
      }
      // Earlier sub-chunks q < R' for row block R': columns off(R') + 16q, off = 64, 80, 112.
#pragma unroll
      for (int Rp = 1; Rp < 4; ++Rp) {
        const int offR = (Rp == 1) ? 64 : (Rp == 2) ? 80 : 112;
#pragma unroll
        for (int q = 0; q < Rp; ++q) {
          float v16[16];
          tmem_ld16(tl + TM_D1 + offR + 16 * q, v16);
#pragma unroll
          for (int m = 0; m < 16; ++m)
            rowv[16 * q + m] = (Rp == R) ? v16[m] : rowv[16 * q + m];
        }
      }
      if (is_a) {
#pragma unroll
        for (int s = 0; s < 64; ++s) L[r * LDL + s] = (s < r) ? br * rowv[s] : 0.f;
      } else {
        // M row r: columns s <= r, bf16, K-major SW128 [64 x 64]
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          uint32_t wv[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int s0 = 8 * s8 + 2 * p;
            const float m0 = (s0 <= r) ? rowv[s0] : 0.f;
            const float m1 = (s0 + 1 <= r) ? rowv[s0 + 1] : 0.f;
            wv[p] = pack_bf16(m0, m1);
          }
          *reinterpret_cast<uint4*>(sm + OFF_M + sw128_offset<2>(64, r, 8 * s8)) =
              make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
    __syncthreads();

    // ---------------- T = (I + L)^{-1} diag(beta), blocked by 16
    {
      const float* L = reinterpret_cast<const float*>(sm + OFF_L);
      float* X = reinterpret_cast<float*>(sm + OFF_X);
      float* Y = reinterpret_cast<float*>(sm + OFF_Y);
      if (tid < 64) {
        const int blk = tid >> 4, s = tid & 15, b0 = 16 * blk;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            if (m < r) acc += L[(b0 + r) * LDL + b0 + m] * x[m];
          x[r] = (r == s) ? 1.f : ((r > s) ? -acc : 0.f);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) X[(b0 + r) * LDL + b0 + s] = x[r];
      }
      __syncthreads();
      for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        for (int e = tid; e < nb * 256; e += kThreads) {
          const int bi = e >> 8, ii = d + bi, jj = ii - d;
          const int ra = (e >> 4) & 15, cb = e & 15;
          float acc = 0.f;
          for (int kk = jj; kk < ii; ++kk)
#pragma unroll
            for (int m = 0; m < 16; ++m)
              acc += L[(16 * ii + ra) * LDL + 16 * kk + m] * X[(16 * kk + m) * LDL + 16 * jj + cb];
          Y[bi * 256 + ra * 16 + cb] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nb * 256; e += kThreads) {
          const int bi = e >> 8, ii = d + bi, jj = ii - d;
          const int ra = (e >> 4) & 15, cb = e & 15;
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            acc += X[(16 * ii + ra) * LDL + 16 * ii + m] * Y[bi * 256 + m * 16 + cb];
          X[(16 * ii + ra) * LDL + 16 * jj + cb] = -acc;
        }
        __syncthreads();
      }
      // T[r][s] = X[r][s] beta_s (s <= r), bf16 K-major SW128 [64 x 64]
      for (int e = tid; e < 64 * 8; e += kThreads) {
        const int r = e >> 3, s8 = e & 7;
        uint32_t wv[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int s0 = 8 * s8 + 2 * p;
          const float t0v = (s0 <= r) ? X[r * LDL + s0] * s_beta[s0] : 0.f;
          const float t1v = (s0 + 1 <= r) ? X[r * LDL + s0 + 1] * s_beta[s0 + 1] : 0.f;
          wv[p] = pack_bf16(t0v, t1v);
        }
        *reinterpret_cast<uint4*>(sm + OFF_T + sw128_offset<2>(64, r, 8 * s8)) =
            make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
    // K~^T operand into TMEM (D1 columns are free now)
    tmem_st8(tl + TM_KT + 8 * wg, kt_pack);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------- MMA2: W^T = K~^T T^T, U~^T = V^T T^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ts = smem_u32(sm + OFF_T);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t bd = sw128_kdesc<2>(ts, 64, s);
        mma_ts(tm + TM_DW, tm + TM_KT + 8 * s, bd, idesc_m64, s > 0);
        mma_ts(tm + TM_DU, tm + TM_VA + 8 * s, bd, idesc_m64, s > 0);
      }
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!__syncthreads_and(w)) { ok = false; break; }
    tc_fence_after();
    // -W into smem: thread (c = ln, rows 16 wg .. 16 wg + 15)
    {
      float v16[16];
      tmem_ld16(tl + TM_DW + 16 * wg, v16);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        st_bf16(sm + OFF_W, sw128_offset<2>(64, 16 * wg + i, ln), -v16[i]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------- MMA3: U^T += S^T (-W)^T, O^T = S^T Q~^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ws = smem_u32(sm + OFF_W), qs = smem_u32(sm + OFF_QT);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        mma_ts(tm + TM_DU, tm + TM_SA + 8 * s, sw128_kdesc<2>(ws, 64, s), idesc_m64, 1);
        mma_ts(tm + TM_DO, tm + TM_SA + 8 * s, sw128_kdesc<2>(qs, 64, s), idesc_m64, s > 0);
      }
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!__syncthreads_and(w)) { ok = false; break; }
    tc_fence_after();
    // U^T -> bf16 A operand: thread (j = ln, tokens 16 wg .. 16 wg + 15)
    {
      float v16[16];
      tmem_ld16(tl + TM_DU + 16 * wg, v16);
      uint32_t up[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) up[i] = pack_bf16(v16[2 * i], v16[2 * i + 1]);
      tmem_st8(tl + TM_UA + 8 * wg, up);
    }
    tc_fence_before();
    __syncthreads();

    // ---------------- MMA4: O^T += U^T M^T, dS^T = U^T K^
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ms = smem_u32(sm + OFF_M), ks = smem_u32(sm + OFF_KHT);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        mma_ts(tm + TM_DO, tm + TM_UA + 8 * s, sw128_kdesc<2>(ms, 64, s), idesc_m64, 1);
        mma_ts(tm + TM_DS, tm + TM_UA + 8 * s, sw128_kdesc<2>(ks, 128, s), idesc_m128, s > 0);
      }
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!__syncthreads_and(w)) { ok = false; break; }
    tc_fence_after();
    // state update (channels 32 wg .. 32 wg + 31 of row j = ln) and the output
    {
      float inc[32];
      tmem_ld32(tl + TM_DS + 32 * wg, inc);
      uint32_t sp[16];
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] = s_dec[32 * wg + i] * S[i] + inc[i];
#pragma unroll
      for (int i = 0; i < 16; ++i) sp[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
      tmem_st16(tl + TM_SA + 16 * wg, sp);
      float o16[16];
      tmem_ld16(tl + TM_DO + 16 * wg, o16);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 16 * wg + i;
        if (r < n) out[((tok0 + r) * H + h) * kD + ln] = __float2bfloat16_rn(o16[i]);
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (!ok) {
    if (tid == 0) atomicOr(&g_tc_error, 1u);
    // let any copy still in flight land before the shared memory is released
    if (tma_pending) mbar_wait(&bar_tma, tma_parity, 1000000000ull);
    // and the last tensor-core batch, if its completion was what timed out
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  } else if (a.final_state) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      a.final_state[state_off + (long long)c * kD + ln] = S[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows, H, 128] bf16, box {64 ch, 1 head, 64 tokens}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs& a, bool bf16) {
  return bf16 && a.dk == kD && a.dv == kD && a.chunk == 64;
}

cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t st) {
  const long long rows = a.cu_seqlens ? a.total_T : (long long)a.B * a.T;
  if (rows <= 0) {
    // nothing to load: still run the kernel so the state passes through
  }
  CUtensorMap mq, mk, mv;
  const long long map_rows = rows > 0 ? rows : 1;
  if (!make_map(&mq, a.q, map_rows, a.H) || !make_map(&mk, a.k, map_rows, a.H) ||
      !make_map(&mv, a.v, map_rows, a.H))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.H, a.B);
  chunk_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

unsigned int chunk_tc_read_error(bool reset) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v));
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_tc_error, &z, sizeof(z));
  }
  return v;
}

}  // namespace kda
