// Chunked KDA forward on the 5th-generation tensor cores (tcgen05) for bf16 q/k/v with
// dk = dv = 128 and 64-token chunks.
//
// One CTA of 512 threads (4 warpgroups) walks one (sequence, head) pair chunk by chunk.
// Per chunk (kernel_delta_attention page, "Algorithm modes: chunked"; decay-first
// recurrence), with G the in-chunk cumulative log-decay and the chunk cut into four
// 16-token sub-chunks R whose reference point P_R is G just before the sub-chunk:
//
//  prologue (SIMT, fused): L2 norms of q and k, gate activation and its cumulative sum,
//    beta, and the gate-scaled bf16 operands (K-major, 128-byte swizzle, shared memory)
//      Xl  = [k^_r e^{G_r - P_R}; q^_r e^{G_r - P_R}]                (128 x dk)
//      Kb  = [k^_s e^{P_S - G_s} (diagonal sub-chunks);               (160 x dk)
//             the same times e^{P_R - P_S} for every later sub-chunk R]
//      Q~  = q^ e^{G},  K^^T = (k^ e^{G_C - G})^T,  K~^T = (k^ e^{G})^T,  V^T
//  MMA1  [A; M] = Xl Kb^T                              gate-scaled K K^T and Q K^T
//  solve T = (I + diag(beta) tril(A, -1))^{-1} diag(beta)     (fp32, blocked by 16)
//  MMA2  W^T = K~^T T^T,  U~^T = V^T T^T                         (UT / WY transform)
//  MMA3  U^T = U~^T - S^T W^T,  O^T = S^T Q~^T                   (S^T: bf16 copy in TMEM)
//  MMA4  O^T += U^T M^T (M = tril(Q K^T part)),  S^T <- S^T diag(e^{G_C}) + U^T K^
//        (the fp32 master state lives in Tensor Memory; it is decayed in place before
//         MMA4 accumulates the chunk's update onto it)
//
// The sequential dependence is only through S.  The state-dependent products are
// oriented so that the value index j is the TMEM lane (M = dv = 128).  Every
// exponential factor lies in [e^{-80}, e^{80}] (lower_bound >= -5), inside the fp32 and
// bf16 exponent range.  Transcendentals use the fast hardware approximations (this path
// rounds every operand to bf16 anyway).
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
constexpr int OFF_KTT = OFF_KHT + 16384;    // K~^T [128 x 64]
constexpr int OFF_VT = OFF_KTT + 16384;     // V^T [128 x 64]
constexpr int OFF_M = OFF_VT + 16384;       // M [64 x 64]
constexpr int OFF_W = OFF_M + 8192;         // -W [64 x 128]
constexpr int OFF_END = OFF_W + 16384;
// Re-used inside the Xl/Kb region once MMA1 has completed.
constexpr int LDL = 68;                     // fp32 row pitch (16-byte aligned rows)
constexpr int OFF_L = OFF_XL;               // fp32 [64][68] beta-scaled strict lower A
constexpr int OFF_X = OFF_L + 64 * LDL * 4; // fp32 [64][68] (I + L)^{-1}
constexpr int OFF_Y = OFF_X + 64 * LDL * 4; // fp32 [3][16][17] solve temporaries
constexpr int OFF_T = OFF_XL + 40960;       // T [64 x 64] bf16 SW128 (1024-aligned)
static_assert(OFF_Y + 3 * 16 * 17 * 4 <= OFF_T, "solve scratch overlaps T");
static_assert(OFF_T + 8192 <= OFF_QT, "T must stay inside the Xl/Kb region");
constexpr size_t kSmemBytes = OFF_END + 1024;

// Tensor Memory columns (512 allocated).
constexpr uint32_t TM_D1 = 0;     // [A; M] accumulator, 160 columns
constexpr uint32_t TM_DW = 0;     // W^T accumulator (after D1 is consumed), 64
constexpr uint32_t TM_UA = 128;   // U^T A operand (bf16 pairs), 32
constexpr uint32_t TM_DU = 160;   // U~^T then U^T accumulator, 64
constexpr uint32_t TM_DO = 224;   // O^T accumulator, 64
constexpr uint32_t TM_S = 288;    // fp32 master state S^T, 128
constexpr uint32_t TM_SA = 416;   // bf16 copy of S^T (A operand), 64
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kTxBytes = 3 * 16384;  // q, k, v tiles per chunk

__device__ unsigned int g_tc_error;  // bit 0: an mbarrier wait timed out

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float fast_exp(float x) { return __expf(x); }
__device__ __forceinline__ float fast_rcp(float x) { return __fdividef(1.0f, x); }

// tcgen05.st of 8 columns (shape 32x32b, x8), waited for.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// tcgen05.st of 32 columns, waited for.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Byte offset of the 16-byte chunk holding tokens 8 tg .. 8 tg + 7 of row c of a
// transposed [128 x 64] tile (rows = channels, tokens contiguous, one 128-byte block).
__device__ __forceinline__ uint32_t trow_off(int c, int tg) {
  return uint32_t((c >> 3) * 1024 + (c & 7) * 128 + ((tg ^ (c & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ __align__(16) float s_rk[kC];
  __shared__ __align__(16) float s_rq[kC];
  __shared__ __align__(16) float s_beta[kC];
  __shared__ __align__(16) float s_dec[kD];
  __shared__ __align__(16) float s_gtot[8][kD];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[2];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7;            // warpgroup
  const int ln = tid & 127;           // TMEM lane of this thread (value index j)
  const int lane_base = 32 * (warp & 3);
  // prologue mapping: channel pair c0, c0 + 1 and tokens 8 tg .. 8 tg + 7 (quarter R)
  const int cp = tid & 63, tg = tid >> 6, Rq = tg >> 1;
  const int c0 = 2 * cp;
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

  // Initial state: thread (j = ln, warpgroup wg) owns S^T[j][32 wg .. 32 wg + 31].
  {
    float S[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      S[i] = a.initial_state ? a.initial_state[state_off + (long long)c * kD + ln] : 0.f;
    }
    tmem_st32(tl + TM_S + 32 * wg, S);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
    tmem_st16(tl + TM_SA + 16 * wg, w);
  }

  const float exp_a = __expf(a.a_log[h]);
  const float db0 = a.dt_bias[c0 * H + h], db1 = a.dt_bias[(c0 + 1) * H + h];
  const int nchunks = (len + kC - 1) / kC;
  const uint32_t idesc_n160 = make_idesc(1, 128, 160);
  const uint32_t idesc_n64 = make_idesc(1, 128, 64);
  const uint32_t idesc_n128 = make_idesc(1, 128, 128);
  // swizzle of this thread's channel pair inside a 128-byte row: kb block, chunk, byte
  const uint32_t c_kb = uint32_t(c0 >> 6);
  const uint32_t c_chunk = uint32_t(((c0 & 63) * 2) >> 4);
  const uint32_t c_byte = uint32_t(((c0 & 63) * 2) & 15);
  auto row_off = [&](int rows, int r) -> uint32_t {  // element (r, c0) of a K-major tile
    return c_kb * uint32_t(rows * 128) + uint32_t((r >> 3) * 1024 + (r & 7) * 128) +
           (((c_chunk ^ uint32_t(r & 7)) << 4) | c_byte);
  };

  uint32_t mma_phase = 0;
  bool ok = true;
  bool tma_pending = false;  // a TMA batch was issued and not yet waited for
  uint32_t tma_parity = 0;   // parity of that batch

  if (tid == 0 && nchunks > 0) {
    mbar_arrive_expect_tx(&bar_tma, kTxBytes);
    for (int half = 0; half < 2; ++half) {
      tma_load_3d(sm + OFF_Q + half * 8192, &map_q, &bar_tma, 64 * half, h, (int)bos);
      tma_load_3d(sm + OFF_K + half * 8192, &map_k, &bar_tma, 64 * half, h, (int)bos);
      tma_load_3d(sm + OFF_V + half * 8192, &map_v, &bar_tma, 64 * half, h, (int)bos);
    }
  }
  tma_pending = nchunks > 0;

  // Raw gates of this thread's channel pair and 8 tokens, loaded one chunk ahead.
  float2 graw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = 8 * tg + i;
    graw[i] = (t < len) ? *reinterpret_cast<const float2*>(a.g + ((bos + t) * H + h) * kD + c0)
                        : make_float2(0.f, 0.f);
  }

  // beta logits of the next chunk, loaded one chunk ahead by threads < 64
  float blog = (tid < kC && tid < len) ? a.beta_logits[(bos + tid) * H + h] : 0.f;

  // One thread polls the barrier; the block learns the outcome through shared memory
  // (alternating slots: consecutive calls are always separated by this __syncthreads).
  uint32_t wait_calls = 0;
  auto block_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t slot = wait_calls++ & 1;
    if (tid == 0) s_wait_ok[slot] = mbar_wait(bar, parity) ? 1 : 0;
    __syncthreads();
    return s_wait_ok[slot] != 0;
  };
  auto mma_wait = [&]() -> bool {
    const bool w = block_wait(&bar_mma, mma_phase & 1);
    ++mma_phase;
    return w;
  };

  for (int ch = 0; ch < nchunks; ++ch) {
    const int t0 = ch * kC;
    const int n = min(kC, len - t0);
    const long long tok0 = bos + t0;

    // ---- beta, then wait for this chunk's q/k/v tiles
    if (tid < kC) {
      s_beta[tid] = tid < n ? sigmoidf_(blog) : 0.f;
      const int tn = t0 + kC + tid;
      blog = (tn < len) ? a.beta_logits[(bos + tn) * H + h] : 0.f;
    }
    bool w = block_wait(&bar_tma, ch & 1);
    if (!w) { ok = false; break; }
    tma_pending = false;

    // ---- norms (warp w: tokens 4w .. 4w + 3) and the gate prefix (thread: 2 channels)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = 4 * warp + u;
      const uint32_t off = sw128_offset<2>(64, t, 4 * lane);
      const uint2 qv = *reinterpret_cast<const uint2*>(sm + OFF_Q + off);
      const uint2 kv = *reinterpret_cast<const uint2*>(sm + OFF_K + off);
      float sq = bf16_lo(qv.x) * bf16_lo(qv.x) + bf16_hi(qv.x) * bf16_hi(qv.x) +
                 bf16_lo(qv.y) * bf16_lo(qv.y) + bf16_hi(qv.y) * bf16_hi(qv.y);
      float sk = bf16_lo(kv.x) * bf16_lo(kv.x) + bf16_hi(kv.x) * bf16_hi(kv.x) +
                 bf16_lo(kv.y) * bf16_lo(kv.y) + bf16_hi(kv.y) * bf16_hi(kv.y);
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      if (lane == 0) {
        s_rq[t] = t < n ? a.scale * rsqrtf(sq + kL2Eps) : 0.f;
        s_rk[t] = t < n ? rsqrtf(sk + kL2Eps) : 0.f;
      }
    }
    float loc0[8], loc1[8];  // G_t - (G before this 8-token group), channels c0, c0 + 1
    {
      float r0 = 0.f, r1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = 8 * tg + i;
        float g0 = 0.f, g1 = 0.f;
        if (t < n) {
          g0 = a.lower_bound * fast_rcp(1.f + fast_exp(-exp_a * (graw[i].x + db0)));
          g1 = a.lower_bound * fast_rcp(1.f + fast_exp(-exp_a * (graw[i].y + db1)));
        }
        r0 += g0;
        r1 += g1;
        loc0[i] = r0;
        loc1[i] = r1;
      }
      *reinterpret_cast<float2*>(&s_gtot[tg][c0]) = make_float2(r0, r1);
    }
    __syncthreads();
    // prefetch the next chunk's raw gates (consumed at the next gate prefix)
    if (ch + 1 < nchunks) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = t0 + kC + 8 * tg + i;
        graw[i] = (t < len)
                      ? *reinterpret_cast<const float2*>(a.g + ((bos + t) * H + h) * kD + c0)
                      : make_float2(0.f, 0.f);
      }
    }

    // ---- gate-scaled operands for (channels c0, c0 + 1) x (tokens 8 tg .. 8 tg + 7)
    {
      float2 tot[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) tot[g] = *reinterpret_cast<const float2*>(&s_gtot[g][c0]);
      float P0[4], P1[4];  // P_R: G just before quarter R
      P0[0] = 0.f;
      P1[0] = 0.f;
#pragma unroll
      for (int r = 1; r < 4; ++r) {
        P0[r] = P0[r - 1] + tot[2 * r - 2].x + tot[2 * r - 1].x;
        P1[r] = P1[r - 1] + tot[2 * r - 2].y + tot[2 * r - 1].y;
      }
      const float Gc0 = P0[3] + tot[6].x + tot[7].x, Gc1 = P1[3] + tot[6].y + tot[7].y;
      float Pm0 = P0[0], Pm1 = P1[0];
#pragma unroll
      for (int r = 1; r < 4; ++r)
        if (Rq == r) { Pm0 = P0[r]; Pm1 = P1[r]; }
      // offset of this group inside its quarter (odd groups follow an even one)
      const float o0 = (tg & 1) ? tot[tg - 1].x : 0.f, o1 = (tg & 1) ? tot[tg - 1].y : 0.f;
      const float eP0 = fast_exp(Pm0), eP1 = fast_exp(Pm1);            // e^{P_R}
      const float eCP0 = fast_exp(Gc0 - Pm0), eCP1 = fast_exp(Gc1 - Pm1);  // e^{G_C - P_R}
      float cR0[4], cR1[4];  // e^{P_R' - P_R}, later sub-chunks R'
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        cR0[r] = (r > Rq) ? fast_exp(P0[r] - Pm0) : 0.f;
        cR1[r] = (r > Rq) ? fast_exp(P1[r] - Pm1) : 0.f;
      }
      if (tg == 0) *reinterpret_cast<float2*>(&s_dec[c0]) = make_float2(fast_exp(Gc0), fast_exp(Gc1));

      uint32_t kh0[4], kh1[4], kt0[4], kt1[4], vt0[4], vt1[4];  // transposed packs
      float pkh0 = 0.f, pkh1 = 0.f, pkt0 = 0.f, pkt1 = 0.f, pv0 = 0.f, pv1 = 0.f;
      const float4 rk4a = *reinterpret_cast<const float4*>(&s_rk[8 * tg]);
      const float4 rk4b = *reinterpret_cast<const float4*>(&s_rk[8 * tg + 4]);
      const float4 rq4a = *reinterpret_cast<const float4*>(&s_rq[8 * tg]);
      const float4 rq4b = *reinterpret_cast<const float4*>(&s_rq[8 * tg + 4]);
      const float rkv[8] = {rk4a.x, rk4a.y, rk4a.z, rk4a.w, rk4b.x, rk4b.y, rk4b.z, rk4b.w};
      const float rqv[8] = {rq4a.x, rq4a.y, rq4a.z, rq4a.w, rq4b.x, rq4b.y, rq4b.z, rq4b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = 8 * tg + i;
        const uint32_t roff = row_off(64, t);
        const uint32_t kw = *reinterpret_cast<const uint32_t*>(sm + OFF_K + roff);
        const uint32_t qw = *reinterpret_cast<const uint32_t*>(sm + OFF_Q + roff);
        const uint32_t vw = *reinterpret_cast<const uint32_t*>(sm + OFF_V + roff);
        const float k0 = bf16_lo(kw) * rkv[i], k1 = bf16_hi(kw) * rkv[i];
        const float q0 = bf16_lo(qw) * rqv[i], q1 = bf16_hi(qw) * rqv[i];
        const float v0 = (t < n) ? bf16_lo(vw) : 0.f, v1 = (t < n) ? bf16_hi(vw) : 0.f;
        const float e0 = fast_exp(loc0[i] + o0), e1 = fast_exp(loc1[i] + o1);  // e^{G_t - P_R}
        const float i0 = fast_rcp(e0), i1 = fast_rcp(e1);
        const float xk0 = k0 * e0, xk1 = k1 * e1, xq0 = q0 * e0, xq1 = q1 * e1;
        const float kd0 = k0 * i0, kd1 = k1 * i1;  // k^ e^{P_R - G_t}
        *reinterpret_cast<uint32_t*>(sm + OFF_XL + row_off(128, t)) = pack_bf16(xk0, xk1);
        *reinterpret_cast<uint32_t*>(sm + OFF_XL + row_off(128, 64 + t)) = pack_bf16(xq0, xq1);
        *reinterpret_cast<uint32_t*>(sm + OFF_KB + row_off(kKbRows, t)) = pack_bf16(kd0, kd1);
        if (Rq < 1)
          *reinterpret_cast<uint32_t*>(sm + OFF_KB + row_off(kKbRows, 64 + t)) =
              pack_bf16(kd0 * cR0[1], kd1 * cR1[1]);
        if (Rq < 2)
          *reinterpret_cast<uint32_t*>(sm + OFF_KB + row_off(kKbRows, 80 + t)) =
              pack_bf16(kd0 * cR0[2], kd1 * cR1[2]);
        if (Rq < 3)
          *reinterpret_cast<uint32_t*>(sm + OFF_KB + row_off(kKbRows, 112 + t)) =
              pack_bf16(kd0 * cR0[3], kd1 * cR1[3]);
        *reinterpret_cast<uint32_t*>(sm + OFF_QT + row_off(64, t)) =
            pack_bf16(xq0 * eP0, xq1 * eP1);  // q^ e^{G_t}
        const float kh0v = kd0 * eCP0, kh1v = kd1 * eCP1;  // k^ e^{G_C - G_t}
        const float kt0v = xk0 * eP0, kt1v = xk1 * eP1;    // k^ e^{G_t}
        if (i & 1) {
          kh0[i >> 1] = pack_bf16(pkh0, kh0v);
          kh1[i >> 1] = pack_bf16(pkh1, kh1v);
          kt0[i >> 1] = pack_bf16(pkt0, kt0v);
          kt1[i >> 1] = pack_bf16(pkt1, kt1v);
          vt0[i >> 1] = pack_bf16(pv0, v0);
          vt1[i >> 1] = pack_bf16(pv1, v1);
        }
        pkh0 = kh0v; pkh1 = kh1v; pkt0 = kt0v; pkt1 = kt1v; pv0 = v0; pv1 = v1;
      }
      const uint32_t ta = trow_off(c0, tg), tb = trow_off(c0 + 1, tg);
      *reinterpret_cast<uint4*>(sm + OFF_KHT + ta) = make_uint4(kh0[0], kh0[1], kh0[2], kh0[3]);
      *reinterpret_cast<uint4*>(sm + OFF_KHT + tb) = make_uint4(kh1[0], kh1[1], kh1[2], kh1[3]);
      *reinterpret_cast<uint4*>(sm + OFF_KTT + ta) = make_uint4(kt0[0], kt0[1], kt0[2], kt0[3]);
      *reinterpret_cast<uint4*>(sm + OFF_KTT + tb) = make_uint4(kt1[0], kt1[1], kt1[2], kt1[3]);
      *reinterpret_cast<uint4*>(sm + OFF_VT + ta) = make_uint4(vt0[0], vt0[1], vt0[2], vt0[3]);
      *reinterpret_cast<uint4*>(sm + OFF_VT + tb) = make_uint4(vt1[0], vt1[1], vt1[2], vt1[3]);
    }
    fence_async_smem();
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

    // ---- MMA1: [A; M] = Xl Kb^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t xa = smem_u32(sm + OFF_XL), kb = smem_u32(sm + OFF_KB);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ss(tm + TM_D1, sw128_kdesc<2>(xa, 128, s), sw128_kdesc<2>(kb, kKbRows, s),
               idesc_n160, s > 0);
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!w) { ok = false; break; }
    tc_fence_after();

    // ---- read A (lanes 0..63) and M (lanes 64..127); warpgroup wg takes columns s of
    //      quarter q = wg.  Every tcgen05.ld address is warp-uniform.
    {
      const int r = ln & 63, R = r >> 4, q = wg;
      const int Rlo = 2 * ((warp & 3) & 1);  // the two row quarters this warp's lanes span
      float v[16];
      {
        float d16[16];
        tmem_ld16(tl + TM_D1 + 16 * q, d16);
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = (R == q) ? d16[m] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int Rp = Rlo + e;
        if (q < Rp) {  // warp-uniform
          const int offR = (Rp == 1) ? 64 : (Rp == 2) ? 80 : 112;
          float d16[16];
          tmem_ld16(tl + TM_D1 + offR + 16 * q, d16);
#pragma unroll
          for (int m = 0; m < 16; ++m) v[m] = (R == Rp) ? d16[m] : v[m];
        }
      }
      if (ln < 64) {
        const float br = s_beta[r];
        float* L = reinterpret_cast<float*>(sm + OFF_L) + r * LDL + 16 * q;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          float4 o;
          o.x = (16 * q + 4 * m4 + 0 < r) ? br * v[4 * m4 + 0] : 0.f;
          o.y = (16 * q + 4 * m4 + 1 < r) ? br * v[4 * m4 + 1] : 0.f;
          o.z = (16 * q + 4 * m4 + 2 < r) ? br * v[4 * m4 + 2] : 0.f;
          o.w = (16 * q + 4 * m4 + 3 < r) ? br * v[4 * m4 + 3] : 0.f;
          reinterpret_cast<float4*>(L)[m4] = o;
        }
      } else {
        uint32_t pk[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int s0 = 16 * q + 2 * p;
          pk[p] = pack_bf16((s0 <= r) ? v[2 * p] : 0.f, (s0 + 1 <= r) ? v[2 * p + 1] : 0.f);
        }
        *reinterpret_cast<uint4*>(sm + OFF_M + sw128_offset<2>(64, r, 16 * q)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(sm + OFF_M + sw128_offset<2>(64, r, 16 * q + 8)) =
            make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    __syncthreads();

    // ---- T = (I + L)^{-1} diag(beta), blocked by 16
    {
      const float* L = reinterpret_cast<const float*>(sm + OFF_L);
      float* X = reinterpret_cast<float*>(sm + OFF_X);
      float* Y = reinterpret_cast<float*>(sm + OFF_Y);
      // diagonal blocks: warp b inverts block b, lane s < 16 computes column s
      if (warp < 4 && lane < 16) {
        const int b0 = 16 * warp, s = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc = 0.f;
#pragma unroll
          for (int m4 = 0; m4 < r; m4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + (b0 + r) * LDL + b0 + m4);
            if (m4 + 0 < r) acc += l4.x * x[m4 + 0];
            if (m4 + 1 < r) acc += l4.y * x[m4 + 1];
            if (m4 + 2 < r) acc += l4.z * x[m4 + 2];
            if (m4 + 3 < r) acc += l4.w * x[m4 + 3];
          }
          x[r] = (r == s) ? 1.f : -acc;  // rows above s stay 0: all their terms are 0
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) X[(b0 + r) * LDL + b0 + s] = x[r];
      }
      __syncthreads();
      // off-diagonal blocks by distance d = i - j: Y = sum_k L_ik X_kj, X_ij = -X_ii Y.
      // Block (i, i - d) is handled by warpgroup (i - d); thread: row a, columns b, b + 1.
      const int a_ = ln >> 3, b_ = (ln & 7) * 2, jj = wg;
#pragma unroll
      for (int d = 1; d < 4; ++d) {
        const int ii = jj + d;
        if (ii < 4) {
          const float* Lr = L + (16 * ii + a_) * LDL + 16 * jj;
          const float* Xc = X + (16 * jj) * LDL + 16 * jj + b_;
          float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
#pragma unroll
          for (int m = 0; m < 16 * d; m += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(Lr + m);
            const float2 x0 = *reinterpret_cast<const float2*>(Xc + (m + 0) * LDL);
            const float2 x1 = *reinterpret_cast<const float2*>(Xc + (m + 1) * LDL);
            const float2 x2 = *reinterpret_cast<const float2*>(Xc + (m + 2) * LDL);
            const float2 x3 = *reinterpret_cast<const float2*>(Xc + (m + 3) * LDL);
            y0 += l4.x * x0.x + l4.z * x2.x;
            y1 += l4.x * x0.y + l4.z * x2.y;
            y2 += l4.y * x1.x + l4.w * x3.x;
            y3 += l4.y * x1.y + l4.w * x3.y;
          }
          Y[jj * 272 + a_ * 17 + b_] = y0 + y2;
          Y[jj * 272 + a_ * 17 + b_ + 1] = y1 + y3;
        }
        __syncthreads();
        if (ii < 4) {
          const float* Xr = X + (16 * ii + a_) * LDL + 16 * ii;
          float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
#pragma unroll
          for (int m = 0; m < 16; m += 4) {
            const float4 x4 = *reinterpret_cast<const float4*>(Xr + m);
            z0 += x4.x * Y[jj * 272 + (m + 0) * 17 + b_] + x4.z * Y[jj * 272 + (m + 2) * 17 + b_];
            z1 += x4.x * Y[jj * 272 + (m + 0) * 17 + b_ + 1] + x4.z * Y[jj * 272 + (m + 2) * 17 + b_ + 1];
            z2 += x4.y * Y[jj * 272 + (m + 1) * 17 + b_] + x4.w * Y[jj * 272 + (m + 3) * 17 + b_];
            z3 += x4.y * Y[jj * 272 + (m + 1) * 17 + b_ + 1] + x4.w * Y[jj * 272 + (m + 3) * 17 + b_ + 1];
          }
          *reinterpret_cast<float2*>(X + (16 * ii + a_) * LDL + 16 * jj + b_) =
              make_float2(-(z0 + z2), -(z1 + z3));
        }
        __syncthreads();
      }
      // T[r][s] = X[r][s] beta_s (s <= r): thread row r = tid >> 3, columns 8 (tid & 7) ..
      {
        const int r = tid >> 3, s0 = (tid & 7) * 8;
        uint32_t pk[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int s = s0 + 2 * p;
          const float t0v = (s <= r) ? X[r * LDL + s] * s_beta[s] : 0.f;
          const float t1v = (s + 1 <= r) ? X[r * LDL + s + 1] * s_beta[s + 1] : 0.f;
          pk[p] = pack_bf16(t0v, t1v);
        }
        *reinterpret_cast<uint4*>(sm + OFF_T + sw128_offset<2>(64, r, s0)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA2: W^T = K~^T T^T, U~^T = V^T T^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ts = smem_u32(sm + OFF_T), ks = smem_u32(sm + OFF_KTT),
                     vs = smem_u32(sm + OFF_VT);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t bd = sw128_kdesc<2>(ts, 64, s);
        mma_ss(tm + TM_DW, sw128_kdesc<2>(ks, 128, s), bd, idesc_n64, s > 0);
        mma_ss(tm + TM_DU, sw128_kdesc<2>(vs, 128, s), bd, idesc_n64, s > 0);
      }
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!w) { ok = false; break; }
    tc_fence_after();
    // -W into smem: thread (c = ln, rows 16 wg .. 16 wg + 15); row r has r & 7 == i & 7
    {
      float v16[16];
      tmem_ld16(tl + TM_DW + 16 * wg, v16);
      const uint32_t wkb = uint32_t(ln >> 6) * 8192u, wch = uint32_t(((ln & 63) * 2) >> 4),
                     wby = uint32_t(((ln & 63) * 2) & 15);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 16 * wg + i;
        const uint32_t off = wkb + uint32_t((r >> 3) * 1024 + (i & 7) * 128) +
                             (((wch ^ uint32_t(i & 7)) << 4) | wby);
        *reinterpret_cast<__nv_bfloat16*>(sm + OFF_W + off) = __float2bfloat16_rn(-v16[i]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA3: U^T += S^T (-W)^T, O^T = S^T Q~^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ws = smem_u32(sm + OFF_W), qs = smem_u32(sm + OFF_QT);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        mma_ts(tm + TM_DU, tm + TM_SA + 8 * s, sw128_kdesc<2>(ws, 64, s), idesc_n64, 1);
        mma_ts(tm + TM_DO, tm + TM_SA + 8 * s, sw128_kdesc<2>(qs, 64, s), idesc_n64, s > 0);
      }
      mma_commit(&bar_mma);
    }
    // meanwhile: decay the fp32 master state in place (TM_S is not read by MMA3)
    {
      float S[32];
      tmem_ld32(tl + TM_S + 32 * wg, S);
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] *= s_dec[32 * wg + i];
      tmem_st32(tl + TM_S + 32 * wg, S);
    }
    w = mma_wait();
    if (!w) { ok = false; break; }
    tc_fence_after();
    // ---- U^T -> bf16 A operand: thread (j = ln, tokens 16 wg .. 16 wg + 15)
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

    // ---- MMA4: O^T += U^T M^T, S^T += U^T K^
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ms = smem_u32(sm + OFF_M), ks = smem_u32(sm + OFF_KHT);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        mma_ts(tm + TM_DO, tm + TM_UA + 8 * s, sw128_kdesc<2>(ms, 64, s), idesc_n64, 1);
        mma_ts(tm + TM_S, tm + TM_UA + 8 * s, sw128_kdesc<2>(ks, 128, s), idesc_n128, 1);
      }
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!w) { ok = false; break; }
    tc_fence_after();
    // ---- bf16 copy of the new state and the output
    {
      float S[32];
      tmem_ld32(tl + TM_S + 32 * wg, S);
      uint32_t sp[16];
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
    // ---- end of chunk
  }

  if (!ok) {
    if (tid == 0) atomicOr(&g_tc_error, 1u);
    // let any copy still in flight land before the shared memory is released
    if (tma_pending) mbar_wait(&bar_tma, tma_parity, 1000000000ull);
    // and the last tensor-core batch, if its completion was what timed out
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  } else if (a.final_state) {
    tc_fence_after();
    float S[32];
    tmem_ld32(tl + TM_S + 32 * wg, S);
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
  CUtensorMap mq, mk, mv;
  const long long map_rows = rows > 0 ? rows : 1;  // empty inputs: the state still passes
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
