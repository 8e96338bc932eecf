// Chunked form of the recurrent page's gated linear recurrence on the tensor cores: key-axis
// gates (g, gk, g_gamma) and the value-axis gate gv, bf16 q/k/v with head dim 128, 64-token
// chunks, forward order (ejkernel "recurrent" page, run / recurrent_attention: query, key,
// value, g, gk, gv, g_gamma, initial_state, cu_seqlens, softmax_scale).
//
// With a_t = g_t + gk_t + g_gamma per key channel, the recurrence
//     h_t = diag(e^{a_t}) h_{t-1} + k_t v_t^T,   o_t = h_t^T (scale q_t)
// over one chunk of tokens r = 1..C, with the in-chunk cumulative gate G_r = a_1 + .. + a_r
// and the state S entering the chunk, is
//     O = scale (Q~ S + M V),   S' = diag(e^{G_C}) S + K^^T V,
//     Q~_r = q_r e^{G_r},   K^_s = k_s e^{G_C - G_s},
//     M_rs = sum_c q_r[c] k_s[c] e^{G_r[c] - G_s[c]}  (s <= r; 0 above the diagonal).
// It is the KDA chunk form without the delta rule (no UT transform: the chunk writes V
// itself), and M is built the same way: the 16-token sub-chunk reference points P_R keep
// every factor within e^{16 |a|} inside a sub-chunk, which with a in [-5, 1] stays inside
// the fp32 / bf16 range over a whole 64-token chunk as well.
//
//  gla_prep_kernel   persistent, two CTAs per SM, one (chunk, query head) record at a time:
//                    gate prefix, the operand tiles, M on tcgen05, the records Q~, K^^T, M
//                    and e^{G_C}; the next record's q, k and gate tiles are staged by TMA
//                    while the current one finishes.
//  gla_scan_kernel   one CTA per (sequence, query head): per chunk O'^T = S^T Q~^T + V^T M^T
//                    and S^T <- S^T diag(e^{G_C}) + V^T K^ (V^T read as staged from the
//                    input, MN-major), the fp32 state in Tensor Memory with a bf16 copy as
//                    the A operand of the next chunk's output product.
//
// With a value-axis gate, b_t = gv_t per value column and h_t = diag(e^{a_t}) h_{t-1}
// diag(e^{b_t}) + k_t v_t^T.  With B_r = b_1 + .. + b_r in the chunk, the pair (r, s <= r)
// carries e^{B_r - B_s} per value column, so per chunk
//     O = scale (e^{B} o (Q~ S) + sum_s M_rs v_s e^{B_r - B_s}),
//     S' = diag(e^{G_C}) S diag(e^{B_C}) + K^^T V^,   V^_s = v_s e^{B_C - B_s},
// (o: elementwise over (r, value column)).  The in-chunk sum is split at the value side's
// own 16-token reference points Q_R (B just before sub-chunk R): for r in sub-chunk R and s
// in sub-chunk R' <= R, e^{B_r - B_s} = e^{B_r - Q_R} e^{Q_R - Q_R'} e^{Q_R' - B_s}, so with
// V~_s = v_s e^{Q_R(s) - B_s} and Y_R' = M[:, R'] V~[R'] (one K = 16 product per R'),
//     O_r = scale e^{B_r - Q_R} (e^{Q_R} (Q~ S)_r + sum_{R' <= R} e^{Q_R - Q_R'} Y_R',r),
// every factor within e^{16 |b|} like the key side's.
//  gla_vprep_kernel  (value gate only) per (chunk, query head): V^, V~, e^{B_r - Q_R} and the
//                    sub-chunk totals of b, for the scan.
#include "chunk_records.cuh"

namespace kda {
namespace {

using namespace tc;
using namespace chunk;

constexpr int kC = 64;
constexpr int kD = 128;

__device__ unsigned int g_gla_error;  // bit 4: a bounded wait of this path gave up;
                                      // bit 5: a sub-chunk's summed gate left this path's range
// Gates in [-5, 1] per token keep every factor e^{+-x} of a 16-token sub-chunk inside fp32:
// the sum of a sub-chunk's (or half sub-chunk's) gates then lies in [-80, 16] (resp.
// [-40, 8]).  The kernels check those sums (a little slack for rounding), one comparison per
// thread and record, and record bit 5 where one falls outside.
constexpr float kSubLo2 = -80.01f * kLog2E, kSubHi2 = 16.01f * kLog2E;  // log2 units
constexpr float kHalfLo = -40.01f, kHalfHi = 8.01f;

// Workspace records per (chunk slot, query head).
constexpr long long kGRecQ = 64LL * 128 * 2;   // Q~ [64 tok][128] bf16
constexpr long long kGRecK = 128LL * 64 * 2;   // K^^T [128][64 tok] bf16
constexpr long long kGRecM = 64LL * 64 * 2;    // M [64][64] bf16
constexpr long long kGRecVec = 256 * 4;        // e^{G_C} [128], scale per live row [64], pad
constexpr long long kGRecV = 64LL * 128 * 2;   // V^, V~ or e^{B - Q} [64 tok][128] bf16
constexpr long long kGRecVTot = 4 * 128 * 4;   // sub-chunk totals of b [4][128] fp32

struct GWs {
  __nv_bfloat16* qw;
  __nv_bfloat16* kt;
  __nv_bfloat16* m;
  float* vec;
  // value gate only: V^ and V~ [64 tok][128] bf16, e^{B_r - Q_R} [64 tok][128] bf16 and the
  // sub-chunk totals of b [4][128] fp32 per record
  __nv_bfloat16* vh;
  __nv_bfloat16* vt;
  __nv_bfloat16* eb;
  float* vtot;
  int32_t* coff;  // [nseq + 1] first chunk slot of each sequence (packed inputs only)
  long long recs;
  int nck_fixed;
};

long long gla_slots(const GlaArgs& a) {
  if (a.cu_seqlens) return (long long)a.T / kC + a.nseq;
  return (long long)a.nseq * ((a.T + kC - 1) / kC);
}

void gla_carve(const GlaArgs& a, void* base, GWs& w) {
  const long long recs = gla_slots(a) * a.Hq;
  uint8_t* p = static_cast<uint8_t*>(base);
  w.recs = recs;
  w.nck_fixed = a.cu_seqlens ? 0 : (a.T + kC - 1) / kC;
  w.qw = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kGRecQ;
  w.kt = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kGRecK;
  w.m = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kGRecM;
  w.vec = reinterpret_cast<float*>(p);
  p += recs * kGRecVec;
  if (a.gv || a.reverse) {  // (reverse order runs on the value records, gate or not)
    w.vh = reinterpret_cast<__nv_bfloat16*>(p);
    p += recs * kGRecV;
    w.vt = reinterpret_cast<__nv_bfloat16*>(p);
    p += recs * kGRecV;
    w.eb = reinterpret_cast<__nv_bfloat16*>(p);
    p += recs * kGRecV;
    w.vtot = reinterpret_cast<float*>(p);
    p += recs * kGRecVTot;
  }
  w.coff = reinterpret_cast<int32_t*>(p);
}

// Token range of sequence `seq` (packed offsets clamped into [0, T], as the SIMT kernel does).
__device__ __forceinline__ void gla_seq_range(const GlaArgs& a, int seq, long long& bos,
                                              int& len) {
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
}

// ------------------------------------------------------------------- prep kernel

constexpr int kGThreads = 256;
constexpr int kGKbRows = 160;        // 64 diagonal + 16 + 32 + 48 off-diagonal key rows
constexpr int G_XL = 0;              // Xl [128 x 128] bf16: rows 0..63 q e^{G - P_R}
constexpr int G_KB = 32768;          // Kb [160 x 128]
constexpr int G_KS = G_KB;           // K^^T record staging [128 x 64] (after MMA1)
constexpr int G_MS = G_KB + 16384;   // M record staging [64 x 64] (after MMA1)
constexpr int G_K = G_KB + 40960;    // staged k [64 tok x 128], two SW128 boxes
constexpr int G_Q = G_K + 16384;     // staged q
constexpr int G_END = G_Q + 16384;
constexpr int G_G = 0;               // staged gate [4][64 tok][32] fp32, inside Xl
constexpr size_t kGSmem = G_END + 1024;
constexpr uint32_t kGTmemCols = 256;  // D1 = Xl Kb^T: 160 columns
static_assert(G_MS + 8192 <= G_K, "record staging must stay inside Kb");

// Rows 64..127 of Xl are not written: the MMA's lanes 64..127 are never read.
// kRev: reverse order.  Every position p of a record is token p of the chunk walked
// backwards: chunk jc covers the tokens end - 64 (jc + 1) .. end - 64 jc - 1 of its sequence,
// staged as they lie (row 63 - p holds position p; rows before the sequence's first token
// are dead positions p >= n), so the records are those of the forward recurrence on the
// reversed sequence.
template <bool kRev>
__global__ void __launch_bounds__(kGThreads, 2)
    gla_prep_kernel(const __grid_constant__ CUtensorMap map_kt,
                    const __grid_constant__ CUtensorMap map_m,
                    const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_g, const GlaArgs a,
                    const float* gate2, const GWs w) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ __align__(16) float s_dec[kD];
  __shared__ __align__(16) float s_gtot[4][kD];
  __shared__ uint64_t bar_mma, bar_ld;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[2];
  __shared__ int s_gate_out;  // a sub-chunk's summed key-axis gate left [-80, 16]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7;
  const int ln = tid & 127;
  const int lane_base = 32 * (warp & 3);
  const int cp = tid & 63, R = tid >> 6;  // channel pair, sub-chunk
  const int c0 = 2 * cp;
  const int Hq = a.Hq;
  const int grp = a.Hq / a.Hkv;
  const bool tma_thread = tid == kGThreads - 32;
  const bool staged_gate = a.gk != nullptr || a.g != nullptr;

  // record walk: processing index p over (chunk DESCENDING, sequence, head) for fixed-length
  // inputs, the record index itself for packed ones (as in the KDA prep)
  const unsigned BH = (unsigned)a.nseq * (unsigned)Hq;
  long long cur_p = blockIdx.x;
  auto locate = [&](long long& rec_, int& h_, int& seq_, long long& tok0_, int& n_) -> bool {
    if (cur_p >= w.recs) return false;
    const unsigned p32 = (unsigned)cur_p;
    int seq, jc;
    if (a.cu_seqlens) {
      const unsigned slot = p32 / (unsigned)Hq;
      h_ = (int)(p32 - slot * (unsigned)Hq);
      rec_ = cur_p;
      const int N = a.nseq;
      if ((long long)slot >= w.coff[N]) return false;
      int lo = 0, hi = N;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((unsigned)w.coff[mid] <= slot) lo = mid; else hi = mid;
      }
      seq = lo;
      jc = (int)(slot - (unsigned)w.coff[lo]);
    } else {
      const unsigned jr = p32 / BH, rem = p32 - jr * BH;
      seq = (int)(rem / (unsigned)Hq);
      h_ = (int)(rem - (unsigned)seq * (unsigned)Hq);
      jc = w.nck_fixed - 1 - (int)jr;
      rec_ = ((long long)seq * w.nck_fixed + jc) * Hq + h_;
    }
    long long bos;
    int len;
    gla_seq_range(a, seq, bos, len);
    seq_ = seq;
    n_ = min(kC, len - jc * kC);
    // the first token of the staged tile (reverse: it may lie before the sequence's start)
    tok0_ = kRev ? bos + len - (long long)(jc + 1) * kC : bos + (long long)jc * kC;
    return true;
  };

  const uint64_t pol_in = policy_evict_first();  // inputs are read once
  // the next record's k and q (their bytes join bar_ld's phase without arriving) and its gate
  // tile (the arrival that closes the phase); lane 0 of the TMA warp issues them
  auto stage_kq = [&](int h_, long long tok0_) {
    mbar_expect_tx(&bar_ld, 2 * 16384);
    const int hk = h_ / grp;
    tma_load_3d_hint(sm + G_K, &map_k, &bar_ld, 0, hk, (int)tok0_, pol_in);
    tma_load_3d_hint(sm + G_K + 8192, &map_k, &bar_ld, 64, hk, (int)tok0_, pol_in);
    tma_load_3d_hint(sm + G_Q, &map_q, &bar_ld, 0, h_, (int)tok0_, pol_in);
    tma_load_3d_hint(sm + G_Q + 8192, &map_q, &bar_ld, 64, h_, (int)tok0_, pol_in);
  };
  auto stage_g = [&](int h_, long long tok0_) {
    if (!staged_gate) {
      mbar_arrive(&bar_ld);
      return;
    }
    mbar_arrive_expect_tx(&bar_ld, 32768);
    for (int qtr = 0; qtr < 4; ++qtr)
      tma_load_3d_hint(sm + G_G + qtr * 8192, &map_g, &bar_ld, 32 * qtr, h_, (int)tok0_,
                       pol_in);
  };

  if (warp == 0) {
    tmem_alloc(&s_tmem, kGTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    s_gate_out = 0;
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_ld, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_g);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(lane_base) << 16);
  uint32_t mma_phase = 0, wait_calls = 0;
  auto block_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t slot_w = wait_calls++ & 1;
    if (tid == 0) s_wait_ok[slot_w] = mbar_wait(bar, parity) ? 1 : 0;
    __syncthreads();
    return s_wait_ok[slot_w] != 0;
  };
  bool ok = true;

  int h = 0, n = 0, seq = 0, h_next = 0, n_next = 0, seq_next = 0;
  long long tok0 = 0, rec = 0, tok0_next = 0, rec_next = 0;
  bool have = locate(rec, h, seq, tok0, n);
  if (have && tma_thread) {
    stage_kq(h, tok0);
    stage_g(h, tok0);
  }
  uint32_t ld_parity = 0;
  bool ld_pending = have;   // a staging phase was started and not yet waited for
  bool arrive_owed = false;  // its k and q are issued, the gate tile's arrival not yet
  // element (row 16 R + i, channel c0) of a [64 x 128] bf16 tile of two SW128 boxes
  const uint32_t c_kb = uint32_t(c0 >> 6);
  const uint32_t c_chunk = uint32_t(((c0 & 63) * 2) >> 4);
  const uint32_t c_byte = uint32_t(((c0 & 63) * 2) & 15);
  // staged row of this thread's position 16 R + i (reverse: row 63 - 16 R - i)
  auto srow = [&](int i) -> int { return kRev ? 63 - 16 * R - i : 16 * R + i; };
  auto swz = [&](int i) -> uint32_t {
    const int rr = srow(i);
    return c_kb * 8192u + uint32_t((rr >> 3) * 1024 + (rr & 7) * 128) +
           (((c_chunk ^ uint32_t(rr & 7)) << 4) | c_byte);
  };
  while (have) {
    cur_p += gridDim.x;
    const bool have_next = locate(rec_next, h_next, seq_next, tok0_next, n_next);

    // ---- this record's staged k, q and gate tiles
    if (!(ok = block_wait(&bar_ld, ld_parity))) break;
    ld_parity ^= 1u;
    ld_pending = false;
    float2 graw[16];
    uint32_t kw[16], qw[16];
    const uint8_t* gsrc = sm + G_G + (c0 >> 5) * 8192 + (c0 & 31) * 4;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      graw[i] = staged_gate ? *reinterpret_cast<const float2*>(gsrc + srow(i) * 128)
                            : make_float2(0.f, 0.f);
      kw[i] = *reinterpret_cast<const uint32_t*>(sm + G_K + swz(i));
      qw[i] = *reinterpret_cast<const uint32_t*>(sm + G_Q + swz(i));
    }
    if (gate2) {  // both g and gk given: the second one straight from global memory
      const float* g2 = gate2 + (tok0 * Hq + h) * kD + c0;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (16 * R + i < n) {
          const float2 x =
              *reinterpret_cast<const float2*>(g2 + (long long)srow(i) * Hq * kD);
          graw[i] = __fadd2_rn(graw[i], x);
        }
    }
    if (n < kC) {  // partial chunk (uniform): rows past n belong to the next sequence
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (16 * R + i >= n) {
          graw[i] = make_float2(0.f, 0.f);
          kw[i] = 0u;
          qw[i] = 0u;
        }
    }

    // ---- gate prefix over this thread's sub-chunk, in log2 units (the same two-lane form
    //      as the KDA prep; the sub-chunk total stops at the last live token)
    float2 loc[16];
    {
      const float gam = a.g_gamma ? a.g_gamma[(a.cu_seqlens ? 0 : seq) * Hq + h] : 0.f;
      const float2 l2e = make_float2(kLog2E, kLog2E), gv2 = make_float2(gam, gam);
      float2 run = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        run = __ffma2_rn(l2e, __fadd2_rn(graw[i], gv2), run);
        loc[i] = run;
      }
      if (!(run.x >= kSubLo2 && run.x <= kSubHi2 && run.y >= kSubLo2 && run.y <= kSubHi2))
        s_gate_out = 1;
      if (n < kC) {
        const int live = n - 16 * R;
        run = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < live) run = loc[i];
      }
      *reinterpret_cast<float2*>(&s_gtot[R][c0]) = run;
    }
    // the previous record's M store has read its staging tile (inside Kb) before Kb is
    // rewritten; every thread has read the staged tiles before the next ones are issued
    if (tma_thread) bulk_wait_read_all();
    __syncthreads();
    if (tma_thread && have_next) stage_kq(h_next, tok0_next);
    if (have_next) ld_pending = arrive_owed = true;

    // ---- gate-scaled operands (channels c0, c0 + 1) x (tokens 16 R .. 16 R + 15): Xl q
    //      rows, Kb diagonal and off-diagonal key rows, the Q~ record, K^^T words
    uint4 khv[4];
    {
      float P0[4], P1[4];
      P0[0] = 0.f;
      P1[0] = 0.f;
#pragma unroll
      for (int r = 1; r < 4; ++r) {
        const float2 t2 = *reinterpret_cast<const float2*>(&s_gtot[r - 1][c0]);
        P0[r] = P0[r - 1] + t2.x;
        P1[r] = P1[r - 1] + t2.y;
      }
      const float2 t3 = *reinterpret_cast<const float2*>(&s_gtot[3][c0]);
      const float Gc0 = P0[3] + t3.x, Gc1 = P1[3] + t3.y;
      float Pm0 = P0[0], Pm1 = P1[0];
#pragma unroll
      for (int r = 1; r < 4; ++r)
        if (R == r) { Pm0 = P0[r]; Pm1 = P1[r]; }
      const float eP0 = fast_exp2(Pm0), eP1 = fast_exp2(Pm1);
      const float eCP0 = fast_exp2(Gc0 - Pm0), eCP1 = fast_exp2(Gc1 - Pm1);
      float cR0[4], cR1[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        cR0[r] = (r > R) ? fast_exp2(P0[r] - Pm0) : 0.f;
        cR1[r] = (r > R) ? fast_exp2(P1[r] - Pm1) : 0.f;
      }
      if (R == 0)
        *reinterpret_cast<float2*>(&s_dec[c0]) = make_float2(fast_exp2(Gc0), fast_exp2(Gc1));
      const uint32_t eP2 = pack_bf16(eP0, eP1), eCP2 = pack_bf16(eCP0, eCP1);
      const uint32_t c12 = pack_bf16(cR0[1], cR1[1]), c22 = pack_bf16(cR0[2], cR1[2]),
                     c32 = pack_bf16(cR0[3], cR1[3]);
      uint8_t* const p128 = sm + G_XL + c_kb * 16384u + uint32_t(R) * 2048u;
      uint8_t* const p160 = sm + G_KB + c_kb * 20480u + uint32_t(R) * 2048u;
      __nv_bfloat16* const qrec = w.qw + (rec * 64 + 16 * R) * kD + c0;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t khw[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int i = 8 * hf + ii;
          const uint32_t swi = uint32_t(hf * 1024 + ii * 128) +
                               (((c_chunk ^ uint32_t(ii)) << 4) | c_byte);
          const float e0 = fast_exp2(loc[i].x), e1 = fast_exp2(loc[i].y);  // e^{G_t - P_R}
          const uint32_t e2 = pack_bf16(e0, e1);
          const uint32_t i2 = pack_bf16(fast_rcp(e0), fast_rcp(e1));      // e^{P_R - G_t}
          const uint32_t xq = hmul2(qw[i], e2), kd = hmul2(kw[i], i2);
          *reinterpret_cast<uint32_t*>(p128 + swi) = xq;   // Xl row t: q e^{G_t - P_R}
          *reinterpret_cast<uint32_t*>(p160 + swi) = kd;   // Kb diagonal row t
          if (R < 1) *reinterpret_cast<uint32_t*>(p160 + swi + 8 * 1024) = hmul2(kd, c12);
          if (R < 2) *reinterpret_cast<uint32_t*>(p160 + swi + 10 * 1024) = hmul2(kd, c22);
          if (R < 3) *reinterpret_cast<uint32_t*>(p160 + swi + 14 * 1024) = hmul2(kd, c32);
          *reinterpret_cast<uint32_t*>(qrec + i * kD) = hmul2(xq, eP2);  // q e^{G_t}
          khw[ii] = hmul2(kd, eCP2);  // k e^{G_C - G_t}
        }
        khv[2 * hf] = make_uint4(__byte_perm(khw[0], khw[1], 0x5410), __byte_perm(khw[2], khw[3], 0x5410),
                                 __byte_perm(khw[4], khw[5], 0x5410), __byte_perm(khw[6], khw[7], 0x5410));
        khv[2 * hf + 1] = make_uint4(__byte_perm(khw[0], khw[1], 0x7632), __byte_perm(khw[2], khw[3], 0x7632),
                                     __byte_perm(khw[4], khw[5], 0x7632), __byte_perm(khw[6], khw[7], 0x7632));
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA1: D1 = Xl Kb^T (M = 128, N = 160, K = 128); lanes 0..63 hold M's blocks
    if (tid == 0) {
      tc_fence_after();
      const uint32_t xa = smem_u32(sm + G_XL), kb = smem_u32(sm + G_KB);
      const uint32_t idesc = make_idesc(1, 128, kGKbRows);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ss(tm, sw128_kdesc<2>(xa, 128, s), sw128_kdesc<2>(kb, kGKbRows, s), idesc, s > 0);
      mma_commit(&bar_mma);
    }
    if (!(ok = block_wait(&bar_mma, mma_phase & 1))) break;
    ++mma_phase;
    tc_fence_after();
    // Xl is free: the next record's gate tile goes there (closing bar_ld's phase)
    if (tma_thread && have_next) stage_g(h_next, tok0_next);
    arrive_owed = false;
    // K^^T record into its swizzled staging tile (inside Kb, free once MMA1 is done)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t piece = uint32_t(2 * R + hf);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = k ^ ((lane >> 2) & 1);
        const int c = c0 + e;
        *reinterpret_cast<uint4*>(sm + G_KS + (c >> 3) * 1024 + (c & 7) * 128 +
                                  ((piece ^ uint32_t(c & 7)) << 4)) =
            e ? khv[2 * hf + 1] : khv[2 * hf];
      }
    }
    // vector record: e^{G_C} [128], scale per live row [64]
    w.vec[rec * 256 + tid] = tid < 128 ? s_dec[tid] : tid < 192 ? ((tid - 128 < n) ? a.scale : 0.f)
                                                                : 0.f;

    // ---- read M (TMEM lanes 0..63: warps 0, 1, 4, 5); warpgroup wg takes the column
    //      quarters q = wg, wg + 2.  Every tcgen05.ld address is warp-uniform.
    if ((warp & 3) < 2) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int q = wg + 2 * qq;
        const int r = ln, Rr = r >> 4;
        const int Rlo = 2 * (warp & 1);  // the two row quarters this warp's lanes span
        float v[16];
        {
          float d16[16];
          tmem_ld16(tl + 16 * q, d16);
#pragma unroll
          for (int m = 0; m < 16; ++m) v[m] = (Rr == q) ? d16[m] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int Rp = Rlo + e;
          if (q < Rp) {  // warp-uniform
            const int offR = (Rp == 1) ? 64 : (Rp == 2) ? 80 : 112;
            float d16[16];
            tmem_ld16(tl + offR + 16 * q, d16);
#pragma unroll
            for (int m = 0; m < 16; ++m) v[m] = (Rr == Rp) ? d16[m] : v[m];
          }
        }
        uint32_t pk[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int s0 = 16 * q + 2 * p;
          pk[p] = pack_bf16((s0 <= r) ? v[2 * p] : 0.f, (s0 + 1 <= r) ? v[2 * p + 1] : 0.f);
        }
        uint8_t* const mrow = sm + G_MS + (r >> 3) * 1024 + (r & 7) * 128;
        const uint32_t sw = uint32_t(r & 7);
        *reinterpret_cast<uint4*>(mrow + ((uint32_t(2 * q) ^ sw) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(mrow + ((uint32_t(2 * q + 1) ^ sw) << 4)) =
            make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tma_thread) {
      tma_store_2d(&map_kt, sm + G_KS, 0, (int)(rec * 128));
      tma_store_2d(&map_m, sm + G_MS, 0, (int)(rec * 64));
      bulk_commit();
    }
    rec = rec_next;
    h = h_next;
    seq = seq_next;
    tok0 = tok0_next;
    n = n_next;
    have = have_next;
  }

  if (!ok) {
    if (tid == 0) {
      atomicOr(&g_gla_error, 16u);
      if (arrive_owed) mbar_arrive(&bar_ld);  // let the phase complete on its k and q bytes
      if (ld_pending) mbar_wait(&bar_ld, ld_parity, 1000000000ull);  // staging in flight
    }
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  }
  if (tma_thread) bulk_wait_read_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && s_gate_out) atomicOr(&g_gla_error, 32u);
  if (warp == 0) tmem_dealloc(tm, kGTmemCols);
}

// ------------------------------------------------------------- value-gate records

// Per (chunk, query head) record, thread (P, cp): value columns 2 cp and 2 cp + 1 (fp32 and
// bf16 pairs), the 8 tokens 8 P .. 8 P + 7 (half of sub-chunk R = P / 2).  The gate's prefix
// inside the sub-chunk, L_t = B_t - Q_R (b = gv, fp32; zero past a partial chunk's end, so
// the totals stop at its last token), and the sub-chunk totals T_R = Q_{R+1} - Q_R give
//   V^_s = v_s e^{B_C - B_s} = v_s e^{(T_R + .. + T_3) - L_s},  V~_s = v_s e^{-L_s},
//   E_r = e^{L_r}
// in bf16 (every row of the record: the rows past the end are zero) and the totals.  A
// thread's gate and v loads all go out before the one block barrier (the exchange of the
// 8-token totals).  Bound by its memory traffic; CTAs walk the records with a grid stride.
constexpr int kVThreads = 512;

// Without a value gate (reverse order routes every call through these records) b = 0:
// V^ = V~ = v, E = 1.  kRev: position p is token 63 - p of the staged tile, as in the prep.
template <bool kRev>
__global__ void __launch_bounds__(kVThreads, 2) gla_vprep_kernel(const GlaArgs a, const GWs w) {
  __shared__ float2 s_tot[8][kD / 2];
  const int cp = threadIdx.x & 63, P = threadIdx.x >> 6, R = P >> 1;
  const int c0 = 2 * cp;
  const int Hq = a.Hq, grp = a.Hq / a.Hkv;
  const long long gstride = (long long)Hq * kD, vstride = (long long)a.Hkv * kD;
  bool gate_out = false;  // a half sub-chunk's summed value-axis gate left [-40, 8]
  for (long long rec = blockIdx.x; rec < w.recs; rec += gridDim.x) {
    const int h = (int)(rec % Hq);
    const long long slot = rec / Hq;
    int seq, jc;
    if (a.cu_seqlens) {
      // records past the last chunk exist (their count is an upper bound); every later
      // record is past it too (uniform over the CTA)
      if (slot >= w.coff[a.nseq]) break;
      int lo = 0, hi = a.nseq;  // coff[lo] <= slot < coff[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (w.coff[mid] <= slot) lo = mid; else hi = mid;
      }
      seq = lo;
      jc = (int)(slot - w.coff[lo]);
    } else {
      seq = (int)(slot / w.nck_fixed);
      jc = (int)(slot % w.nck_fixed);
    }
    long long bos;
    int len;
    gla_seq_range(a, seq, bos, len);
    const int n = min(kC, len - jc * kC);  // live positions (>= 1)
    // token of position 0 (live) and the step between positions
    const long long ctok = kRev ? bos + len - 1 - (long long)jc * kC : bos + (long long)jc * kC;
    const int dir = kRev ? -1 : 1;
    const int hk = h / grp;
    // positions past the end read position 0 instead and are masked, so that the loads are
    // unconditional and all in flight at once
    const float* const gbase = a.gv ? a.gv + (ctok * Hq + h) * kD + c0 : nullptr;
    const __nv_bfloat16* const vbase =
        static_cast<const __nv_bfloat16*>(a.v) + (ctok * a.Hkv + hk) * kD + c0;
    float2 L[8];
    uint32_t vw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = 8 * P + i, tt = (t < n ? t : 0) * dir;
      L[i] = gbase ? *reinterpret_cast<const float2*>(gbase + tt * gstride)
                   : make_float2(0.f, 0.f);
      vw[i] = *reinterpret_cast<const uint32_t*>(vbase + tt * vstride);
    }
    float2 run = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (8 * P + i >= n) L[i] = make_float2(0.f, 0.f);
      run = __fadd2_rn(run, L[i]);
      L[i] = run;
    }
    s_tot[P][cp] = run;
    gate_out |= !(run.x >= kHalfLo && run.x <= kHalfHi && run.y >= kHalfLo && run.y <= kHalfHi);
    __syncthreads();
    // the sub-chunk's first half before this thread's tokens; the totals T_r; B_C - Q_R
    const float2 first = s_tot[2 * R][cp];
    if (P & 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) L[i] = __fadd2_rn(first, L[i]);
    }
    float2 tail = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float2 tr = __fadd2_rn(s_tot[2 * r][cp], s_tot[2 * r + 1][cp]);
      if (r >= R) tail = __fadd2_rn(tail, tr);
      if (P == 0) *reinterpret_cast<float2*>(w.vtot + rec * 512 + r * 128 + c0) = tr;
    }
    const long long row0 = (rec * kC + 8 * P) * kD + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool live = 8 * P + i < n;
      const float v0 = live ? bf16_lo(vw[i]) : 0.f, v1 = live ? bf16_hi(vw[i]) : 0.f;
      // e^{L} lies within e^{+-80} (16 gates in [-5, 1]): its reciprocal is e^{-L}
      const float e0 = __expf(L[i].x), e1 = __expf(L[i].y);
      *reinterpret_cast<uint32_t*>(w.vh + row0 + i * kD) =
          pack_bf16(v0 * __expf(tail.x - L[i].x), v1 * __expf(tail.y - L[i].y));
      *reinterpret_cast<uint32_t*>(w.vt + row0 + i * kD) =
          pack_bf16(v0 * fast_rcp(e0), v1 * fast_rcp(e1));
      *reinterpret_cast<uint32_t*>(w.eb + row0 + i * kD) = live ? pack_bf16(e0, e1) : 0u;
    }
    __syncthreads();  // s_tot is rewritten for the next record
  }
  if (__any_sync(0xffffffffu, gate_out) && (threadIdx.x & 31) == 0) atomicOr(&g_gla_error, 32u);
}

// ------------------------------------------------------------------- scan kernel

constexpr int kHThreads = 512;
// one stage = one chunk's record and its v tile
constexpr int H_Q = 0;          // Q~ [64 x 128] (two 64-channel boxes)
constexpr int H_KT = 16384;     // K^^T [128 x 64]
constexpr int H_M = 32768;      // M [64 x 64], right after K^^T: the B operand [K^^T; M]
constexpr int H_V = 40960;      // v [64 tok x 128] as staged (two SW128 boxes): V^T MN-major
constexpr int H_VEC = 57344;    // e^{G_C} [128], scale per live row [64]
constexpr int kHStage = 58368;
constexpr uint32_t kHStageTx = 58368;
constexpr int H_OS = 2 * kHStage;  // output staging [64 tok x 128] bf16 SW128
constexpr int H_END = H_OS + 16384;
constexpr size_t kHSmem = H_END + 1024;
static_assert(kHStage % 1024 == 0 && H_OS % 1024 == 0, "alignment");
// With a value gate the stage's v tile is V^ (same layout), followed by:
constexpr int H_VT = kHStage;        // V~ [64 tok x 128] (two SW128 boxes): V~^T MN-major
constexpr int H_EB = H_VT + 16384;   // e^{B_r - Q_R} [64 tok][128] bf16, row-major
constexpr int H_TOT = H_EB + 16384;  // sub-chunk totals of b [4][128] fp32
constexpr int kHStageVG = H_TOT + 2048;
constexpr int H_OS_VG = 2 * kHStageVG;
constexpr size_t kHSmemVG = H_OS_VG + 16384 + 1024;
static_assert(kHStageVG % 1024 == 0 && H_TOT % 1024 == 0, "alignment");
static_assert(kHSmemVG + 1024 <= 232448, "two value-gate stages fit one SM's shared memory");

constexpr uint32_t H_TM_S = 0;     // fp32 master state S^T [128 (value col) x 128 (key ch)]
constexpr uint32_t H_TM_DO = 128;  // O'^T [128 x 64 tok], right after S: one N = 192 update
constexpr uint32_t H_TM_SA = 192;  // bf16 copy of S^T (A operand), 64 columns
static_assert(H_TM_DO == H_TM_S + 128 && H_M == H_KT + 16384, "the N = 192 update's operands");
constexpr uint32_t kHTmemCols = 256;
// value gate: the in-chunk products Y_R' = M[:, R'] V~[R'] (R' = 0..3), [128 x 64 tok] each
constexpr uint32_t H_TM_Y = 256;
constexpr uint32_t kHTmemColsVG = 512;

// kVG: the value-axis gate (map_v then addresses the V^ records, map_vt the V~ records).
// kRev: reverse order (always with the V^ / V~ records, which hold the positions in the
// records' order): position p of chunk ch is token end - 64 ch - 1 - p, so the output tile's
// row 63 - p.
template <bool kVG, bool kRev>
__global__ void __launch_bounds__(kHThreads, 1)
    gla_scan_kernel(const __grid_constant__ CUtensorMap map_qw,
                    const __grid_constant__ CUtensorMap map_kt,
                    const __grid_constant__ CUtensorMap map_m,
                    const __grid_constant__ CUtensorMap map_v,
                    const __grid_constant__ CUtensorMap map_vt,
                    const __grid_constant__ CUtensorMap map_o, const GlaArgs a, const GWs w) {
  constexpr int kStg = kVG ? kHStageVG : kHStage;
  constexpr uint32_t kStgTx = kVG ? kHStageVG : kHStageTx;
  constexpr int kOS = kVG ? H_OS_VG : H_OS;
  constexpr uint32_t kTmCols = kVG ? kHTmemColsVG : kHTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ uint64_t bar_ld[2], bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[2];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int wg = tid >> 7;
  const int ln = tid & 127;
  const int lane_base = 32 * (warp & 3);
  const int h = blockIdx.x, seq = blockIdx.y;
  const int Hq = a.Hq;
  const int hk = h / (a.Hq / a.Hkv);
  long long bos;
  int len;
  gla_seq_range(a, seq, bos, len);
  long long slot0;
  int nck;
  if (a.cu_seqlens) {
    slot0 = w.coff[seq];
    nck = w.coff[seq + 1] - w.coff[seq];
  } else {
    slot0 = (long long)seq * w.nck_fixed;
    nck = w.nck_fixed;
  }
  const long long state_off = ((long long)seq * Hq + h) * kD * kD;

  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_ld[0], 1);
    mbar_init(&bar_ld[1], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_qw);
    tma_prefetch_desc(&map_kt);
    tma_prefetch_desc(&map_m);
    tma_prefetch_desc(&map_v);
    if (kVG) tma_prefetch_desc(&map_vt);
    tma_prefetch_desc(&map_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(lane_base) << 16);

  const uint64_t pol_rec = policy_evict_first();
  // chunk ch's record and v tile into stage st: its seven boxes from lane 0 of warps 1..7
  // (the expected bytes were registered by thread 0)
  // (value gate: the V^ record in place of the v tile, then V~, e^{B - Q} and the totals, from
  // lane 0 of warps 8..11)
  auto issue_load_spread = [&](int ch, int st) {
    if ((tid & 31) != 0 || warp == 0 || warp > (kVG ? 11 : 7)) return;
    const long long rec = (slot0 + ch) * Hq + h;
    const int tok = (int)(bos + (long long)ch * kC);
    uint8_t* b = sm + st * kStg;
    uint64_t* bar = &bar_ld[st];
    switch (warp) {
      case 1: tma_load_2d_hint(b + H_Q, &map_qw, bar, 0, (int)(rec * 64), pol_rec); break;
      case 2: tma_load_2d_hint(b + H_Q + 8192, &map_qw, bar, 64, (int)(rec * 64), pol_rec); break;
      case 3: tma_load_2d_hint(b + H_KT, &map_kt, bar, 0, (int)(rec * 128), pol_rec); break;
      case 4: tma_load_2d_hint(b + H_M, &map_m, bar, 0, (int)(rec * 64), pol_rec); break;
      case 5: bulk_load_hint(b + H_VEC, w.vec + rec * 256, 1024, bar, pol_rec); break;
      case 6:
        if (kVG) tma_load_2d_hint(b + H_V, &map_v, bar, 0, (int)(rec * 64), pol_rec);
        else tma_load_3d_hint(b + H_V, &map_v, bar, 0, hk, tok, pol_rec);
        break;
      case 7:
        if (kVG) tma_load_2d_hint(b + H_V + 8192, &map_v, bar, 64, (int)(rec * 64), pol_rec);
        else tma_load_3d_hint(b + H_V + 8192, &map_v, bar, 64, hk, tok, pol_rec);
        break;
      case 8: tma_load_2d_hint(b + H_VT, &map_vt, bar, 0, (int)(rec * 64), pol_rec); break;
      case 9: tma_load_2d_hint(b + H_VT + 8192, &map_vt, bar, 64, (int)(rec * 64), pol_rec); break;
      case 10: bulk_load_hint(b + H_EB, w.eb + rec * (kC * kD), 16384, bar, pol_rec); break;
      default: bulk_load_hint(b + H_TOT, w.vtot + rec * 512, 2048, bar, pol_rec); break;
    }
  };
  int inflight[2] = {nck > 0 ? 0 : -1, nck > 1 ? 1 : -1};
  if (tid == 0) {
    if (nck > 0) mbar_arrive_expect_tx(&bar_ld[0], kStgTx);
    if (nck > 1) mbar_arrive_expect_tx(&bar_ld[1], kStgTx);
  }
  __syncthreads();
  if (nck > 0) issue_load_spread(0, 0);
  if (nck > 1) issue_load_spread(1, 1);

  // initial state: thread (j = ln, warpgroup wg) owns S^T[j][32 wg .. 32 wg + 31]
  {
    float S[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      S[i] = a.initial_state ? a.initial_state[state_off + (long long)c * kD + ln] : 0.f;
    }
    tmem_st32(tl + H_TM_S + 32 * wg, S);
    uint32_t wv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
    tmem_st16(tl + H_TM_SA + 16 * wg, wv);
  }
  tc_fence_before();
  __syncthreads();

  const uint32_t idesc_n64 = make_idesc(1, 128, 64);
  const uint32_t idesc_n192_amn = make_idesc(1, 128, 192, true, false);
  const uint32_t idesc_n128_amn = make_idesc(1, 128, 128, true, false);
  const uint32_t idesc_n64_amn = make_idesc(1, 128, 64, true, false);
  uint32_t mma_phase = 0, wait_calls = 0;
  auto block_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t slot_w = wait_calls++ & 1;
    if (tid == 0) s_wait_ok[slot_w] = mbar_wait(bar, parity) ? 1 : 0;
    __syncthreads();
    return s_wait_ok[slot_w] != 0;
  };
  bool ok = true;

  for (int ch = 0; ch < nck; ++ch) {
    const int st = ch & 1;
    uint8_t* const b = sm + st * kStg;
    const int n = min(kC, len - ch * kC);
    // first token of the chunk's token tile (reverse: the tile ends at position 0)
    const long long tok0 = kRev ? bos + len - (long long)(ch + 1) * kC : bos + (long long)ch * kC;

    if (!(ok = block_wait(&bar_ld[st], (ch >> 1) & 1))) break;
    inflight[st] = -1;
    // e^{G_C} and the output scale, read from the stage itself (refilled after the output)
    const float* const s_vec = reinterpret_cast<const float*>(b + H_VEC);
    if (n < kC) {  // partial chunk: the v rows past n belong to the next sequence
      for (int u = tid; u < 1024; u += kHThreads) {
        const int row = (u >> 3) & 63;
        if (row >= n)
          *reinterpret_cast<uint4*>(b + H_V + (u >> 9) * 8192 + row * 128 + (u & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      fence_async_smem();
    }
    __syncthreads();

    // ---- output product O'^T = S^T Q~^T (M = 128, N = 64); its V^T M^T part joins the
    //      state update below
    const uint32_t vs = smem_u32(b + H_V);
    if (tid == 0) {
      tc_fence_after();
      const uint32_t qs = smem_u32(b + H_Q);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ts(tm + H_TM_DO, tm + H_TM_SA + 8 * s, sw128_kdesc<2>(qs, 64, s), idesc_n64, s > 0);
      if constexpr (kVG) {
        // Y_R'^T = V~^T[:, R'] M[:, R']^T: K = the 16 tokens of sub-chunk R' (one K step),
        // V~^T read MN-major from the staged V~ tile, M K-major
        const uint32_t vts = smem_u32(b + H_VT), ms = smem_u32(b + H_M);
#pragma unroll
        for (int r = 0; r < 4; ++r)
          mma_ss(tm + H_TM_Y + 64 * r,
                 make_sdesc(vts + uint32_t(r) * 2048u, 8192u, 1024u, kSwizzle128),
                 sw128_kdesc<2>(ms, 64, r), idesc_n64_amn, 0);
      }
    }
    // meanwhile: decay the fp32 master state in place (S^T diag(e^{G_C}), and with a value
    // gate diag(e^{B_C}) S^T: row j of S^T is value column j)
    {
      float S[32];
      tmem_ld32(tl + H_TM_S + 32 * wg, S);
      float eb_c = 1.f;
      if constexpr (kVG) {
        const float* tot = reinterpret_cast<const float*>(b + H_TOT) + ln;
        eb_c = __expf(tot[0] + tot[128] + tot[256] + tot[384]);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] *= s_vec[32 * wg + i] * eb_c;
      tmem_st32(tl + H_TM_S + 32 * wg, S);
    }
    tc_fence_before();
    __syncthreads();
    // ---- state update and the rest of the output: [S^T | O'^T] += V^T [K^^T; M]^T, one
    //      N = 192 MMA (M = 128, K = 64 tokens) over the adjacent K^^T and M tiles into the
    //      adjacent S and O' columns; the V^T operand is the staged v tile read MN-major (16
    //      tokens = 2 KB per K step, channel boxes 8 KB apart)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ks = smem_u32(b + H_KT);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if constexpr (kVG)  // S^T += V^^T K^ only (the output's in-chunk part is the Y's)
          mma_ss(tm + H_TM_S, make_sdesc(vs + uint32_t(s) * 2048u, 8192u, 1024u, kSwizzle128),
                 sw128_kdesc<2>(ks, 128, s), idesc_n128_amn, 1);
        else
          mma_ss(tm + H_TM_S, make_sdesc(vs + uint32_t(s) * 2048u, 8192u, 1024u, kSwizzle128),
                 sw128_kdesc<2>(ks, 192, s), idesc_n192_amn, 1);
      }
      mma_commit(&bar_mma);
      // the refill's bytes land on the stage's next phase
      if (ch + 2 < nck) mbar_arrive_expect_tx(&bar_ld[st], kStgTx);
    }
    if (!(ok = block_wait(&bar_mma, mma_phase & 1))) break;
    ++mma_phase;
    tc_fence_after();
    // ---- bf16 copy of the new state; the output O = scale O'
    {
      float S[32];
      tmem_ld32(tl + H_TM_S + 32 * wg, S);
      uint32_t sp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sp[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
      tmem_st16(tl + H_TM_SA + 16 * wg, sp);
      float o16[16];
      tmem_ld16(tl + H_TM_DO + 16 * wg, o16);
      if constexpr (kVG) {
        // O'_r = e^{B_r - Q_R} (e^{Q_R} (Q~ S)_r + sum_{R' <= R} e^{Q_R - Q_R'} Y_R',r) for
        // this thread's value column j = ln and the tokens of sub-chunk R = wg
        const float* tot = reinterpret_cast<const float*>(b + H_TOT) + ln;
        float qcum = 0.f;  // Q_R
#pragma unroll
        for (int r = 0; r < 3; ++r)
          if (r < wg) qcum += tot[128 * r];
        const float eq = __expf(qcum);
#pragma unroll
        for (int i = 0; i < 16; ++i) o16[i] *= eq;
        float qr = 0.f;  // Q_R'
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (r <= wg) {  // warp-uniform
            float y16[16];
            tmem_ld16(tl + H_TM_Y + 64 * r + 16 * wg, y16);
            const float f = __expf(qcum - qr);
#pragma unroll
            for (int i = 0; i < 16; ++i) o16[i] += f * y16[i];
          }
          qr += tot[128 * r];
        }
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(b + H_EB) +
                                 (16 * wg) * kD + ln;
#pragma unroll
        for (int i = 0; i < 16; ++i) o16[i] *= __bfloat162float(e[i * kD]);
      }
      if (tid == 0) bulk_wait_read_all();  // the previous output store has read its tile
      __syncthreads();
      if (n == kC) {
        const uint32_t ob = uint32_t(ln >> 6) * 8192u;
        const uint32_t och = uint32_t(((ln & 63) * 2) >> 4), oby = uint32_t(((ln & 63) * 2) & 15);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int rr = kRev ? 63 - 16 * wg - i : 16 * wg + i;  // the tile row of position
          const uint32_t off = ob + uint32_t((rr >> 3) * 1024 + (rr & 7) * 128) +
                               (((och ^ uint32_t(rr & 7)) << 4) | oby);
          *reinterpret_cast<__nv_bfloat16*>(sm + kOS + off) =
              __float2bfloat16_rn(o16[i] * s_vec[128 + 16 * wg + i]);
        }
      } else {
        // the token of position 16 wg; positions step by one token (backwards in reverse)
        const long long p0 = kRev ? tok0 + 63 - 16 * wg : tok0 + 16 * wg;
        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) + (p0 * Hq + h) * kD + ln;
        const long long stride = (kRev ? -1LL : 1LL) * Hq * kD;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (16 * wg + i < n) op[i * stride] = __float2bfloat16_rn(o16[i] * s_vec[128 + 16 * wg + i]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && n == kC) {
      tma_store_3d(&map_o, sm + kOS, 0, h, (int)tok0);
      tma_store_3d(&map_o, sm + kOS + 8192, 64, h, (int)tok0);
      bulk_commit();
    }
    // the stage is consumed (the MMAs, and the output's scale vector): refill it
    if (ch + 2 < nck) issue_load_spread(ch + 2, st);
    inflight[st] = (ch + 2 < nck) ? ch + 2 : -1;
  }

  if (!ok) {
    if (tid == 0) {
      atomicOr(&g_gla_error, 16u);
      for (int st = 0; st < 2; ++st)
        if (inflight[st] >= 0) mbar_wait(&bar_ld[st], (inflight[st] >> 1) & 1, 1000000000ull);
    }
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  } else if (a.final_state) {
    tc_fence_after();
    float S[32];
    tmem_ld32(tl + H_TM_S + 32 * wg, S);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      a.final_state[state_off + (long long)c * kD + ln] = S[i];
    }
  }
  if (tid == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kTmCols);
}

// ------------------------------------------------------------------------- host

// [rows, H, 128] bf16 (box {64, 1, 64}, 128-byte swizzle) or fp32 (box {32, 1, 64}).
bool map_in(CUtensorMap* m, const void* base, long long rows, int H, bool fp32) {
  return split::make_map_in(m, base, rows, H, fp32);
}

}  // namespace

bool gla_chunk_supported(const GlaArgs& a, bool bf16) {
  return bf16 && a.D == kD;
}

size_t gla_chunk_workspace(const GlaArgs& a) {
  const long long recs = gla_slots(a) * a.Hq;
  const size_t coff = a.cu_seqlens ? split::align_up(size_t(a.nseq + 1) * 4, 256) : 0;
  const long long vg = (a.gv || a.reverse) ? 3 * kGRecV + kGRecVTot : 0;
  return size_t(recs) * size_t(kGRecQ + kGRecK + kGRecM + kGRecVec + vg) + coff;
}

bool gla_chunk_index_ok(const GlaArgs& a) {
  return gla_slots(a) * a.Hq * 128 < 0x7fffffffLL;  // records' 32-bit TMA row coordinates
}

cudaError_t launch_gla_chunk(const GlaArgs& a, void* workspace, cudaStream_t st) {
  GWs w{};
  gla_carve(a, workspace, w);
  if (a.cu_seqlens) {  // the first chunk slot of every packed sequence
    ChunkArgs ca{};
    ca.cu_seqlens = a.cu_seqlens;
    ca.B = a.nseq;
    ca.total_T = a.T;
    split::Ws sw{};
    sw.coff = w.coff;
    const cudaError_t e = split::launch_chunk_offsets(ca, sw, st);
    if (e != cudaSuccess) return e;
  }
  const long long rows = a.cu_seqlens ? a.T : (long long)a.nseq * a.T;
  const long long map_rows = rows > 0 ? rows : 1;
  const long long rec_rows = w.recs > 0 ? w.recs : 1;
  const float* gstage = a.gk ? a.gk : a.g;                 // staged by TMA
  const float* gate2 = (a.gk && a.g) ? a.g : nullptr;      // read from global memory
  const bool rev = a.reverse != 0;
  const bool vg = a.gv != nullptr || rev;  // reverse order runs on the value records
  CUtensorMap mqw, mkt, mm, mv, mvt, mo, mq, mk, mg;
  if (!split::make_map_2d(&mqw, w.qw, rec_rows * 64, 128, 64) ||
      !split::make_map_2d(&mkt, w.kt, rec_rows * 128, 64, 128) ||
      !split::make_map_2d(&mm, w.m, rec_rows * 64, 64, 64) ||
      !map_in(&mq, a.q, map_rows, a.Hq, false) || !map_in(&mk, a.k, map_rows, a.Hkv, false) ||
      // value gate: the scan's v tile is the V^ record, its V~ tile the V~ record
      !(vg ? split::make_map_2d(&mv, w.vh, rec_rows * 64, 128, 64)
           : map_in(&mv, a.v, map_rows, a.Hkv, false)) ||
      !split::make_map_2d(&mvt, vg ? (const void*)w.vt : (const void*)w.qw, rec_rows * 64, 128,
                          64) ||
      // (without a gate tensor the unused gate map is laid over q)
      !map_in(&mg, gstage ? (const void*)gstage : a.q, map_rows, a.Hq, gstage != nullptr) ||
      !split::make_map_out(&mo, a.out, map_rows, a.Hq))
    return cudaErrorInvalidValue;
  auto prep = rev ? gla_prep_kernel<true> : gla_prep_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(prep,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
  if (e != cudaSuccess) return e;
  auto scan = rev ? gla_scan_kernel<true, true>
                 : vg ? gla_scan_kernel<true, false> : gla_scan_kernel<false, false>;
  const size_t scan_smem = vg ? kHSmemVG : kHSmem;
  e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem);
  if (e != cudaSuccess) return e;
  if (w.recs > 0) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const long long grid = std::min<long long>(w.recs, 2LL * sms);
    prep<<<(unsigned)grid, kGThreads, kGSmem, st>>>(mkt, mm, mq, mk, mg, a, gate2, w);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (vg) {
      const long long vgrid = std::min<long long>(w.recs, 2LL * sms);
      (rev ? gla_vprep_kernel<true> : gla_vprep_kernel<false>)<<<(unsigned)vgrid, kVThreads, 0,
                                                                 st>>>(a, w);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  scan<<<dim3(a.Hq, a.nseq), kHThreads, scan_smem, st>>>(mqw, mkt, mm, mv, mvt, mo, a, w);
  return cudaGetLastError();
}

unsigned int gla_chunk_read_error(bool reset) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_gla_error, sizeof(v));
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_gla_error, &z, sizeof(z));
  }
  return v;
}

}  // namespace kda
