// Chunked KDA forward on the 5th-generation tensor cores (tcgen05) for bf16 q/k/v with
// dk = dv = 128 and 64-token chunks.
//
// One CTA of 512 threads (4 warpgroups) walks one (sequence, head) pair chunk by chunk.
// Per chunk (kernel_delta_attention page, "Algorithm modes: chunked"; decay-first
// recurrence), with G the in-chunk cumulative log-decay and the chunk cut into four
// 16-token sub-chunks R whose reference point P_R is G just before the sub-chunk:
//
//  prologue (SIMT, fused): gate activation and its cumulative sum, beta, and the
//    gate-scaled bf16 operands of the RAW q and k (K-major, 128-byte swizzle):
//      Xl  = [k_r e^{G_r - P_R}; q_r e^{G_r - P_R}]                  (128 x dk)
//      Kb  = [k_s e^{P_S - G_s} (diagonal sub-chunks);                (224 x dk)
//             the same times e^{P_R - P_S} for every later sub-chunk R;
//             q_s e^{P_S - G_s}]
//      Q~  = q e^{G},  K^^T = (k e^{G_C - G})^T,  K~^T = (k e^{G})^T,  V^T
//  MMA1  [A; M] = Xl Kb^T: gate-scaled K K^T and Q K^T, and on its diagonal |k_r|^2 and
//        |q_r|^2, from which the L2 norms rk = 1/|k|, rq = scale/|q| are taken.  The
//        norms are then applied as row / column factors instead of to every element:
//        A = diag(rk) A_raw diag(rk), W uses T diag(rk), U' = diag(rk) U, O = diag(rq) O'.
//  solve T = (I + diag(beta) tril(A, -1))^{-1} diag(beta)     (fp32, blocked by 16)
//  MMA2  W^T = K~^T (T diag(rk))^T,  U~^T = V^T T^T              (UT / WY transform)
//  MMA3  U^T = U~^T - S^T W^T,  O'^T = S^T Q~^T                  (S^T: bf16 copy in TMEM)
//  MMA4  O'^T += U'^T M_raw^T,  S^T <- S^T diag(e^{G_C}) + U'^T K^
//        (the fp32 master state lives in Tensor Memory; it is decayed in place before
//         MMA4 accumulates the chunk's update onto it)
//
// The sequential dependence is only through S.  The state-dependent products are
// oriented so that the value index j is the TMEM lane (M = dv = 128).  Every
// exponential factor lies in [e^{-80}, e^{80}] (lower_bound >= -5), inside the fp32 and
// bf16 exponent range.  Transcendentals use the fast hardware approximations (this path
// rounds every operand to bf16 anyway).
#include "kda_internal.cuh"
#include "tc_prims.cuh"
#include "chunk_common.cuh"

namespace kda {
namespace {

using namespace tc;
using namespace chunk;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kKbRows = 224;  // 64 diagonal + 16 + 32 + 48 off-diagonal key rows + 64 q rows

// Dynamic shared memory (byte offsets from a 1024-aligned base).
constexpr int OFF_Q = 0;                    // raw q tile, two SW128 boxes [64 tok x 64 ch]
constexpr int OFF_K = OFF_Q + 16384;        // raw k tile
constexpr int OFF_V = OFF_K + 16384;        // raw v tile
constexpr int OFF_XL = OFF_V + 16384;       // Xl [128 x 128] bf16, K-major SW128
constexpr int OFF_KB = OFF_XL + 32768;      // Kb [224 x 128]
constexpr int OFF_QT = OFF_KB + 57344;      // Q~ [64 x 128]
constexpr int OFF_KHT = OFF_QT + 16384;     // K^^T [128 x 64]
constexpr int OFF_KTT = OFF_KHT + 16384;    // K~^T [128 x 64]
constexpr int OFF_VT = OFF_KTT + 16384;     // V^T [128 x 64]
constexpr int OFF_OS = OFF_VT + 16384;      // output staging [64 tok x 128 ch] bf16 SW128
constexpr int OFF_END = OFF_OS + 16384;
// Re-used inside the Xl/Kb region once MMA1 has completed (everything below is consumed
// before the next chunk's prologue rewrites Xl/Kb).
constexpr int OFF_L = OFF_XL;               // fp32 [64][68] beta-scaled strict lower A
constexpr int OFF_X = OFF_L + 64 * LDL * 4; // fp32 [64][68] (I + L)^{-1}
constexpr int OFF_Y = OFF_X + 64 * LDL * 4; // fp32 [4][16][24] per-warp solve scratch
constexpr int OFF_T = OFF_XL + 40960;       // T [64 x 64] bf16 SW128
constexpr int OFF_TW = OFF_T + 8192;        // T diag(rk) [64 x 64]
constexpr int OFF_W = OFF_TW + 8192;        // -W [64 x 128]
constexpr int OFF_M = OFF_W + 16384;        // M_raw [64 x 64]
static_assert(OFF_Y + 4 * 16 * LDY * 4 <= OFF_T, "solve scratch overlaps T");
static_assert(OFF_M + 8192 <= OFF_QT, "reused tiles must stay inside the Xl/Kb region");
static_assert(OFF_T % 1024 == 0 && OFF_W % 1024 == 0 && OFF_M % 1024 == 0, "alignment");
constexpr size_t kSmemBytes = OFF_END + 1024;

// Tensor Memory columns (512 allocated).
constexpr uint32_t TM_D1 = 0;     // [A; M] accumulator, 224 columns
constexpr uint32_t TM_DW = 0;     // W^T accumulator (after D1 is consumed), 64
constexpr uint32_t TM_DU = 64;    // U~^T then U^T accumulator (after D1 is consumed), 64
constexpr uint32_t TM_UA = 128;   // U'^T A operand (bf16 pairs), 32
constexpr uint32_t TM_DO = 224;   // O'^T accumulator, 64
constexpr uint32_t TM_S = 288;    // fp32 master state S^T, 128
constexpr uint32_t TM_SA = 416;   // bf16 copy of S^T (A operand), 64
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kTxBytes = 3 * 16384;  // q, k, v tiles per chunk

__device__ unsigned int g_tc_error;  // bit 0: an mbarrier wait timed out

__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v,
                    const __grid_constant__ CUtensorMap map_o, const ChunkArgs a) {
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
  // prologue mapping: channel pair c0, c0 + 1 and tokens 8 tg .. 8 tg + 7 (quarter Rq)
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
    tma_prefetch_desc(&map_o);
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
  const uint32_t idesc_n224 = make_idesc(1, 128, kKbRows);
  const uint32_t idesc_n64 = make_idesc(1, 128, 64);
  const uint32_t idesc_n128 = make_idesc(1, 128, 128);
  // Addressing of this thread's channel pair in the K-major SW128 tiles: element
  // (8 tg + i + 8 k, c0) of a tile with `rows` rows lies at
  //   kb * rows * 128 + (tg + k) * 1024 + sw[i],  sw[i] = i * 128 + ((chunk ^ i) << 4 | byte)
  const uint32_t c_kb = uint32_t(c0 >> 6);
  const uint32_t c_chunk = uint32_t(((c0 & 63) * 2) >> 4);
  const uint32_t c_byte = uint32_t(((c0 & 63) * 2) & 15);
  uint32_t sw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sw[i] = uint32_t(i * 128) + (((c_chunk ^ uint32_t(i)) << 4) | c_byte);
  uint8_t* const p64 = sm + c_kb * 8192u + uint32_t(tg) * 1024u;    // 64-row tiles
  uint8_t* const p128 = sm + OFF_XL + c_kb * 16384u + uint32_t(tg) * 1024u;
  uint8_t* const p224 = sm + OFF_KB + c_kb * 28672u + uint32_t(tg) * 1024u;
  // transposed stores: lanes 4..7 of each 8-lane group write row c0 + 1 first, so that
  // the 8 lanes of one 128-bit wavefront hit 8 different swizzle phases
  const int tsw = (lane & 4) ? 1 : 0;

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

    // ---- gate prefix (thread: 2 channels x 8 tokens), beta, wait for q/k/v tiles
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
    if (tid < kC) {
      s_beta[tid] = tid < n ? sigmoidf_(blog) : 0.f;
      const int tn = t0 + kC + tid;
      blog = (tn < len) ? a.beta_logits[(bos + tn) * H + h] : 0.f;
    }
    bool w = block_wait(&bar_tma, ch & 1);
    if (!w) { ok = false; break; }
    tma_pending = false;
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
      float o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int g = 0; g < 8; g += 2)
        if (tg == g + 1) { o0 = tot[g].x; o1 = tot[g].y; }
      const float eP0 = fast_exp(Pm0), eP1 = fast_exp(Pm1);                // e^{P_R}
      const float eCP0 = fast_exp(Gc0 - Pm0), eCP1 = fast_exp(Gc1 - Pm1);  // e^{G_C - P_R}
      float cR0[4], cR1[4];  // e^{P_R' - P_R}, later sub-chunks R'
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        cR0[r] = (r > Rq) ? fast_exp(P0[r] - Pm0) : 0.f;
        cR1[r] = (r > Rq) ? fast_exp(P1[r] - Pm1) : 0.f;
      }
      if (tg == 0) *reinterpret_cast<float2*>(&s_dec[c0]) = make_float2(fast_exp(Gc0), fast_exp(Gc1));

      // Every operand is a product of raw bf16 pairs with per-channel factors, done as
      // packed bf16x2 multiplies (each operand is rounded to bf16 for the MMA anyway).
      const uint32_t eP2 = pack_bf16(eP0, eP1), eCP2 = pack_bf16(eCP0, eCP1);
      const uint32_t c12 = pack_bf16(cR0[1], cR1[1]), c22 = pack_bf16(cR0[2], cR1[2]),
                     c32 = pack_bf16(cR0[3], cR1[3]);
      uint32_t khw[8], ktw[8], vvw[8];  // per-token (c0, c0 + 1) words of the transposed tiles
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool live = 8 * tg + i < n;
        uint8_t* const r64 = p64 + sw[i];
        uint8_t* const r128 = p128 + sw[i];
        uint8_t* const r224 = p224 + sw[i];
        const uint32_t kw = live ? *reinterpret_cast<const uint32_t*>(r64 + OFF_K) : 0u;
        const uint32_t qw = live ? *reinterpret_cast<const uint32_t*>(r64 + OFF_Q) : 0u;
        vvw[i] = live ? *reinterpret_cast<const uint32_t*>(r64 + OFF_V) : 0u;
        const float e0 = fast_exp(loc0[i] + o0), e1 = fast_exp(loc1[i] + o1);  // e^{G_t - P_R}
        const uint32_t e2 = pack_bf16(e0, e1);
        const uint32_t i2 = pack_bf16(fast_rcp(e0), fast_rcp(e1));  // e^{P_R - G_t}
        const uint32_t xk = hmul2(kw, e2), xq = hmul2(qw, e2), kd = hmul2(kw, i2);
        *reinterpret_cast<uint32_t*>(r128) = xk;
        *reinterpret_cast<uint32_t*>(r128 + 8 * 1024) = xq;  // row 64 + t
        *reinterpret_cast<uint32_t*>(r224) = kd;
        if (Rq < 1) *reinterpret_cast<uint32_t*>(r224 + 8 * 1024) = hmul2(kd, c12);
        if (Rq < 2) *reinterpret_cast<uint32_t*>(r224 + 10 * 1024) = hmul2(kd, c22);
        if (Rq < 3) *reinterpret_cast<uint32_t*>(r224 + 14 * 1024) = hmul2(kd, c32);
        // q e^{P_R - G_t}: its product with the q rows of Xl puts |q_t|^2 on a diagonal
        *reinterpret_cast<uint32_t*>(r224 + 20 * 1024) = hmul2(qw, i2);
        *reinterpret_cast<uint32_t*>(r64 + OFF_QT) = hmul2(xq, eP2);  // q e^{G_t}
        khw[i] = hmul2(kd, eCP2);  // k e^{G_C - G_t}
        ktw[i] = hmul2(xk, eP2);   // k e^{G_t}
      }
      // transposed tiles: row c0 takes the low halves of tokens 8 tg .. 8 tg + 7, row
      // c0 + 1 the high halves; lanes 4..7 of each 8-lane group write row c0 + 1 first so
      // that one 128-bit wavefront covers 8 different swizzle phases
      uint4 lo[3], hi[3];
      {
        const uint32_t* src[3] = {khw, ktw, vvw};
#pragma unroll
        for (int m = 0; m < 3; ++m) {
          lo[m] = make_uint4(__byte_perm(src[m][0], src[m][1], 0x5410),
                             __byte_perm(src[m][2], src[m][3], 0x5410),
                             __byte_perm(src[m][4], src[m][5], 0x5410),
                             __byte_perm(src[m][6], src[m][7], 0x5410));
          hi[m] = make_uint4(__byte_perm(src[m][0], src[m][1], 0x7632),
                             __byte_perm(src[m][2], src[m][3], 0x7632),
                             __byte_perm(src[m][4], src[m][5], 0x7632),
                             __byte_perm(src[m][6], src[m][7], 0x7632));
        }
      }
      const uint32_t ta = trow_off(c0 + tsw, tg), tb = trow_off(c0 + 1 - tsw, tg);
      const int offs[3] = {OFF_KHT, OFF_KTT, OFF_VT};
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        *reinterpret_cast<uint4*>(sm + offs[m] + ta) = tsw ? hi[m] : lo[m];
        *reinterpret_cast<uint4*>(sm + offs[m] + tb) = tsw ? lo[m] : hi[m];
      }
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
               idesc_n224, s > 0);
      mma_commit(&bar_mma);
    }
    w = mma_wait();
    if (!w) { ok = false; break; }
    tc_fence_after();

    // ---- norms from the diagonals: |k_r|^2 = A_raw[r][r], |q_r|^2 = D1[64 + r][160 + r]
    if (wg == 0) {
      const int w4 = warp & 3, r = 32 * (w4 & 1) + lane;
      float v32[32];
      tmem_ld32(tl + TM_D1 + ((w4 < 2) ? 32 * w4 : 160 + 32 * (w4 - 2)), v32);
      float nn = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) nn = (i == lane) ? v32[i] : nn;
      if (w4 < 2)
        s_rk[r] = (r < n) ? rsqrtf(nn + kL2Eps) : 0.f;
      else
        s_rq[r] = (r < n) ? a.scale * rsqrtf(nn + kL2Eps) : 0.f;
    }
    __syncthreads();

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
        const float sr = s_beta[r] * s_rk[r];
        float* L = reinterpret_cast<float*>(sm + OFF_L) + r * LDL + 16 * q;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const float4 rk4 = *reinterpret_cast<const float4*>(&s_rk[16 * q + 4 * m4]);
          float4 o;
          o.x = (16 * q + 4 * m4 + 0 < r) ? sr * rk4.x * v[4 * m4 + 0] : 0.f;
          o.y = (16 * q + 4 * m4 + 1 < r) ? sr * rk4.y * v[4 * m4 + 1] : 0.f;
          o.z = (16 * q + 4 * m4 + 2 < r) ? sr * rk4.z * v[4 * m4 + 2] : 0.f;
          o.w = (16 * q + 4 * m4 + 3 < r) ? sr * rk4.w * v[4 * m4 + 3] : 0.f;
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
      // diagonal blocks: warp b inverts block b, lane s < 16 computes column s
      if (warp < 4 && lane < 16) {
        const int b0 = 16 * warp, s = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
          for (int m4 = 0; m4 < r; m4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + (b0 + r) * LDL + b0 + m4);
            if (m4 + 0 < r) acc0 += l4.x * x[m4 + 0];
            if (m4 + 1 < r) acc1 += l4.y * x[m4 + 1];
            if (m4 + 2 < r) acc0 += l4.z * x[m4 + 2];
            if (m4 + 3 < r) acc1 += l4.w * x[m4 + 3];
          }
          x[r] = (r == s) ? 1.f : -(acc0 + acc1);  // rows above s stay 0
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) X[(b0 + r) * LDL + b0 + s] = x[r];
      }
      __syncthreads();
      // Off-diagonal blocks level by level (distance d = i - j):
      //   X_ij = -X_ii sum_{k=j}^{i-1} L_ik X_kj,
      // one warp per block: the sum is one 16 x 16d x 16 product (tf32 warp MMAs), the
      // result goes through a per-warp scratch tile into a second product with X_ii.
      // ---- solve level d = 1
      solve_level<1>(L, X, reinterpret_cast<float*>(sm + OFF_Y), warp, lane);
      __syncthreads();
      // ---- solve level d = 2
      solve_level<2>(L, X, reinterpret_cast<float*>(sm + OFF_Y), warp, lane);
      __syncthreads();
      // ---- solve level d = 3
      solve_level<3>(L, X, reinterpret_cast<float*>(sm + OFF_Y), warp, lane);
      __syncthreads();
      // ---- T[r][s] = X[r][s] beta_s and T diag(rk) (s <= r): row r = tid >> 3, 8 columns
      {
        const int r = tid >> 3, s0 = (tid & 7) * 8;
        const float4 xa = *reinterpret_cast<const float4*>(X + r * LDL + s0);
        const float4 xb = *reinterpret_cast<const float4*>(X + r * LDL + s0 + 4);
        const float4 ba = *reinterpret_cast<const float4*>(&s_beta[s0]);
        const float4 bb = *reinterpret_cast<const float4*>(&s_beta[s0 + 4]);
        const float4 ka = *reinterpret_cast<const float4*>(&s_rk[s0]);
        const float4 kb = *reinterpret_cast<const float4*>(&s_rk[s0 + 4]);
        const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
        const float kv[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
        uint32_t pt[4], pw[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float t0v = (s0 + 2 * p <= r) ? xv[2 * p] * bv[2 * p] : 0.f;
          const float t1v = (s0 + 2 * p + 1 <= r) ? xv[2 * p + 1] * bv[2 * p + 1] : 0.f;
          pt[p] = pack_bf16(t0v, t1v);
          pw[p] = pack_bf16(t0v * kv[2 * p], t1v * kv[2 * p + 1]);
        }
        const uint32_t off = sw128_offset<2>(64, r, s0);
        *reinterpret_cast<uint4*>(sm + OFF_T + off) = make_uint4(pt[0], pt[1], pt[2], pt[3]);
        *reinterpret_cast<uint4*>(sm + OFF_TW + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA2: W^T = K~^T (T diag(rk))^T, U~^T = V^T T^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ts = smem_u32(sm + OFF_T), tw = smem_u32(sm + OFF_TW),
                     ks = smem_u32(sm + OFF_KTT), vs = smem_u32(sm + OFF_VT);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        mma_ss(tm + TM_DW, sw128_kdesc<2>(ks, 128, s), sw128_kdesc<2>(tw, 64, s), idesc_n64,
               s > 0);
        mma_ss(tm + TM_DU, sw128_kdesc<2>(vs, 128, s), sw128_kdesc<2>(ts, 64, s), idesc_n64,
               s > 0);
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

    // ---- MMA3: U^T += S^T (-W)^T, O'^T = S^T Q~^T
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
    // ---- U'^T = (diag(rk) U)^T -> bf16 A operand: thread (j = ln, tokens 16 wg .. + 15)
    {
      float v16[16];
      tmem_ld16(tl + TM_DU + 16 * wg, v16);
      uint32_t up[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        up[i] = pack_bf16(v16[2 * i] * s_rk[16 * wg + 2 * i],
                          v16[2 * i + 1] * s_rk[16 * wg + 2 * i + 1]);
      tmem_st8(tl + TM_UA + 8 * wg, up);
    }
    tc_fence_before();
    __syncthreads();

    // ---- MMA4: O'^T += U'^T M_raw^T, S^T += U'^T K^
    if (tid == 0) {
      bulk_wait_read_all();  // the previous chunk's output store has read its staging tile
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
    // ---- bf16 copy of the new state and the output O = diag(rq) O'
    {
      float S[32];
      tmem_ld32(tl + TM_S + 32 * wg, S);
      uint32_t sp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sp[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
      tmem_st16(tl + TM_SA + 16 * wg, sp);
      float o16[16];
      tmem_ld16(tl + TM_DO + 16 * wg, o16);
      if (n == kC) {
        // full chunk: stage the [64 x 128] bf16 tile for one TMA store (row r = 16 wg + i)
        const uint32_t ob = uint32_t(ln >> 6) * 8192u + uint32_t(wg) * 2048u;
        const uint32_t och = uint32_t(((ln & 63) * 2) >> 4), oby = uint32_t(((ln & 63) * 2) & 15);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t off = ob + uint32_t((i >> 3) * 1024 + (i & 7) * 128) +
                               (((och ^ uint32_t(i & 7)) << 4) | oby);
          *reinterpret_cast<__nv_bfloat16*>(sm + OFF_OS + off) =
              __float2bfloat16_rn(o16[i] * s_rq[16 * wg + i]);
        }
      } else {
        // last, partial chunk: plain stores of the live rows only (a full box would spill
        // into the next sequence)
        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) +
                            ((tok0 + 16 * wg) * H + h) * kD + ln;
        const long long stride = (long long)H * kD;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (16 * wg + i < n) op[i * stride] = __float2bfloat16_rn(o16[i] * s_rq[16 * wg + i]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && n == kC) {
      tma_store_3d(&map_o, sm + OFF_OS, 0, h, (int)tok0);
      tma_store_3d(&map_o, sm + OFF_OS + 8192, 64, h, (int)tok0);
      bulk_commit();
    }
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
  if (tid == 0) bulk_wait_all();  // output stores complete before the CTA retires
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kTmemCols);
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
  return bf16 && a.dk == kD && a.dv == kD && a.chunk == 64 && !a.gate_head && !a.beta_prob &&
         !a.no_l2norm && !a.literal;
}

cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t st) {
  const long long rows = a.cu_seqlens ? a.total_T : (long long)a.B * a.T;
  CUtensorMap mq, mk, mv, mo;
  const long long map_rows = rows > 0 ? rows : 1;  // empty inputs: the state still passes
  if (!make_map(&mq, a.q, map_rows, a.H) || !make_map(&mk, a.k, map_rows, a.H) ||
      !make_map(&mv, a.v, map_rows, a.H) || !make_map(&mo, a.out, map_rows, a.H))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.H, a.B);
  chunk_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, mo, a);
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
