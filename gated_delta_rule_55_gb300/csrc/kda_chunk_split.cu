// Chunked KDA forward in two launches, for bf16 q/k/v with dk = dv = 128 and 64-token
// chunks (kernel_delta_attention page, "Algorithm modes: chunked"; decay-first recurrence).
//
// Everything in a chunk except the state is independent of every other chunk.  The work
// is therefore cut at the state:
//
//  chunk_prep_kernel   one CTA per (chunk, head), all chunks of all sequences at once (two
//                      CTAs per SM).  Gate activation and in-chunk cumulative sum, beta, L2
//                      norms, the gate-scaled products A and M (tcgen05, 16-token sub-chunk
//                      reference points), the UT solve T = (I + diag(beta) tril(A,-1))^{-1}
//                      diag(beta) and the transform W = T diag(rk) K~, U~ = T V (tcgen05).
//                      It writes one workspace record per (chunk, head):
//                        Q~^T = (q e^{G})^T                 [128][64 tok]  bf16
//                               (the backward's records: Q~ [64 tok][128])
//                        K^^T = (k e^{G_C - G})^T           [128][64 tok]  bf16
//                        U~^T  16-byte pieces, piece-major  [8][128][8 tok] bf16
//                        -W^T                               [128][64 tok]  bf16
//                        M_raw (gate-scaled q k^T, s <= r)  [64][64]       bf16
//                        e^{G_C} [128], rk [64], rq [64]                    fp32
//  chunk_scan_kernel   one CTA per (sequence, head) walks its chunks in order, records
//                      double-buffered through TMA, with only the state-dependent products:
//                        U^T  = U~^T - S^T W^T,  O'^T = S^T Q~^T
//                        O'^T += U'^T M_raw^T,   S^T <- S^T diag(e^{G_C}) + U'^T K^
//                      (U' = diag(rk) U, O = diag(rq) O'; S^T lives in Tensor Memory in fp32,
//                      with a bf16 copy as the A operand of the next chunk's products).  Each
//                      line is one tcgen05.mma per K step over adjacent B tiles.
//
// The algebra is that of the single-pass kernel (kda_chunk_tc.cu); here the key side of
// every chunk runs on all SMs at once instead of inside the per-sequence scan.
#include "chunk_records.cuh"

namespace kda {
namespace {

using namespace tc;
using namespace chunk;
using namespace split;

// ------------------------------------------------------------------- prep kernel

constexpr int kPThreads = 256;
constexpr int kPKbRows = 160;  // 64 diagonal + 16 + 32 + 48 off-diagonal key rows
// Dynamic shared memory of the prep kernel (1024-aligned base).
constexpr int P_XL = 0;                 // Xl [128 x 128] bf16 (k rows, then q rows)
constexpr int P_KB = P_XL + 32768;      // Kb [160 x 128]
constexpr int P_KTT = P_KB + 40960;     // K~^T [128 x 64]
constexpr int P_V = P_KTT + 16384;      // v [64 tok x 128] as staged (MMA2's MN-major A)
constexpr int P_END = P_V + 16384;
// re-used inside Xl/Kb once MMA1 has completed
constexpr int P_L = 0;                  // fp32 [64][LDL] beta-scaled strict lower A
constexpr int P_X = P_L + 64 * LDL * 4; // fp32 [64][LDL] (I + L)^{-1}
constexpr int P_Y = P_X + 64 * LDL * 4; // fp32 [4][16][LDY] per-warp scratch
constexpr int P_T = 40960;              // T [64 x 64] bf16 SW128
constexpr int P_TW = P_T + 8192;        // -T diag(rk)
constexpr int P_KS = P_TW + 8192;       // K^^T [128 x 64] staging (after MMA1)
constexpr int P_MS = P_T;               // M record [64 x 64] staging (readback to T write)
constexpr int P_W = P_T;                // -W [64 x 128] or -W^T [128 x 64] staging (T and
                                        // T diag(rk), after MMA2)
static_assert(P_Y + 4 * 16 * LDY * 4 <= P_T, "solve scratch overlaps T");
static_assert(P_KS + 16384 <= P_KTT, "re-used tiles must stay inside Xl/Kb");
// Staging of the NEXT record's raw inputs (TMA), each tile issued as soon as its space is
// free: k into the K^^T staging tile once the K^^T store has read it (after the A/M
// readback), g into L and X once the T tiles are written, q into K~^T and v into its own
// tile (where MMA2 reads it as staged) once MMA2 is done.  k and g land on one barrier, q
// and v on a second, so that the next record's gate prefix can start before q and v arrive.
constexpr int ST_K = P_KS;              // k [64 tok x 128] bf16, two SW128 boxes
constexpr int ST_G = 0;                 // g [4 quarters][64 tok][32] fp32, no swizzle
constexpr int ST_Q = P_KTT;             // q, two SW128 boxes
constexpr int ST_V = P_V;               // v
static_assert(ST_G + 32768 <= P_T, "g staging must stay inside the solve area");
constexpr uint32_t kStageBytes = 3 * 16384 + 32768;  // one record's staged tiles
static_assert(kStageBytes == (16384 + 32768) + 2 * 16384, "k + g batch and q + v batch");
constexpr size_t kPSmem = P_END + 1024;

// Tensor Memory of the prep kernel (256 columns: two CTAs per SM).
constexpr uint32_t P_TM_D1 = 0;   // [A; M] accumulator, 160 columns
constexpr uint32_t P_TM_DW = 0;    // after D1 is consumed: [T K~; -W] (forward, 128) or
                                   // -W^T (backward records, 64)
constexpr uint32_t P_TM_DU = 128;  // U~^T, 64
constexpr uint32_t kPTmemCols = 256;

__device__ unsigned int g_split_error;  // bit 1: a bounded wait of the split path gave up;
                                        // bit 5: the attention mode met a decay whose
                                        // 16-token sum left [-80, 16]

// kBwd: also the backward's records (rq folded into Q~ and M, and N).
// kAttn: the kernel_delta_attention call's own variants (ChunkArgs gate_head): a per-head
// log-decay decay[t, h] on every channel instead of the raw per-channel gate (no g tiles are
// staged), beta used as given, and the runtime choices no_l2norm (q and k as given, scale
// still on q) and literal (the key side of A and K~ takes the decay up to the token before:
// e^{G_{t-1}} instead of e^{G_t}; with one decay per token |k|^2 = A_tt e^{gamma_t}).
template <bool kBwd, bool kAttn>
__global__ void __launch_bounds__(kPThreads, 2)
    chunk_prep_kernel(const __grid_constant__ CUtensorMap map_ku,
                      const __grid_constant__ CUtensorMap map_wr,
                      const __grid_constant__ CUtensorMap map_m,
                      const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_g, const ChunkArgs a,
                      const Ws ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ __align__(16) float s_rk[kC];
  __shared__ __align__(16) float s_rq[kC];
  __shared__ __align__(16) float s_beta[kC];
  __shared__ __align__(16) float s_dec[kD];
  __shared__ __align__(16) float s_gtot[4][kD];
  __shared__ __align__(16) float s_qq[2][kC];
  __shared__ __align__(16) float s_gam[kC];  // kAttn: this record's per-token log2-decay
  __shared__ uint64_t bar_mma, bar_ld, bar_qv;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[2];
  __shared__ int s_decay_out;  // kAttn: a sub-chunk's summed decay left [-80, 16]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7;        // warpgroup (0, 1)
  const int ln = tid & 127;       // TMEM lane
  const int lane_base = 32 * (warp & 3);
  // SIMT mapping: channel pair c0, c0 + 1 and the 16 tokens of sub-chunk R
  const int cp = tid & 63, R = tid >> 6;
  const int c0 = 2 * cp;
  const int H = a.H;
  // lane 0 of the last warp issues the bulk stores of the records (and waits for their
  // reads) and the early staging of the next record: that warp is idle during the solve,
  // which warp 0 leads
  const bool tma_thread = tid == kPThreads - 32;

  // The CTA walks processing indices p = blockIdx.x, blockIdx.x + gridDim.x, ...  For
  // fixed-length inputs p runs over (chunk, sequence, head), head fastest, with the chunk
  // index DESCENDING: the records the scan reads first (every sequence's first chunks) are
  // the last ones written, so they are still in L2 when the scan starts.  For packed inputs
  // p is the record index itself (record r = slot * H + h).
  const unsigned BH = (unsigned)a.B * (unsigned)H;  // fixed-length: records per chunk index
  long long cur_p = blockIdx.x;
  auto advance = [&]() { cur_p += gridDim.x; };
  // the current processing index -> (record, head, first token, live tokens); false past
  // the last record, and past the last chunk of packed inputs (the record count is an upper
  // bound there).  Record counts stay below 2^31 (the records' TMA row coordinates are
  // 32-bit), so the index arithmetic is 32-bit.
  auto locate = [&](long long& rec_, int& h_, long long& tok0_, int& n_) -> bool {
    if (cur_p >= ws.recs) return false;
    const unsigned p32 = (unsigned)cur_p;
    int seq, jc;
    if (a.cu_seqlens) {
      const unsigned slot = p32 / (unsigned)H;
      h_ = (int)(p32 - slot * (unsigned)H);
      rec_ = cur_p;
      const int N = a.B;
      if ((long long)slot >= ws.coff[N]) return false;
      int lo = 0, hi = N;  // coff[lo] <= slot < coff[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((unsigned)ws.coff[mid] <= slot) lo = mid; else hi = mid;
      }
      seq = lo;
      jc = (int)(slot - (unsigned)ws.coff[lo]);
    } else {
      const unsigned jr = p32 / BH, rem = p32 - jr * BH;
      seq = (int)(rem / (unsigned)H);
      h_ = (int)(rem - (unsigned)seq * (unsigned)H);
      jc = ws.nck_fixed - 1 - (int)jr;
      rec_ = ((long long)seq * ws.nck_fixed + jc) * H + h_;
    }
    long long bos;
    int len;
    seq_range(a, seq, bos, len);
    n_ = min(kC, len - jc * kC);  // live tokens of this chunk (>= 1)
    tok0_ = bos + (long long)jc * kC;
    return true;
  };
  // a record's raw q / k / v / g tiles into the staging area (one thread)
  // The ten box loads of a record are issued by lane 0 of the eight warps (loads w and
  // w + 8), so that no single thread spends the issue time; the barrier's expected bytes are
  // registered beforehand by thread 0 (stage_expect), with a block barrier in between.
  // the first record: k and g on bar_ld, q and v on bar_qv
  auto stage_expect = [&]() {
    mbar_arrive_expect_tx(&bar_ld, kAttn ? 16384 : 16384 + 32768);
    mbar_arrive_expect_tx(&bar_qv, 2 * 16384);
  };
  // the next record's k (thread 0; its bytes join the barrier phase without arriving)
  // (the inputs are read once: they are loaded with an evict-first L2 policy, so that the
  // L2 keeps the records instead)
  const uint64_t pol_in = policy_evict_first();
  auto stage_k = [&](int h_, long long tok0_) {
    mbar_expect_tx(&bar_ld, 16384);
    tma_load_3d_hint(sm + ST_K, &map_k, &bar_ld, 0, h_, (int)tok0_, pol_in);
    tma_load_3d_hint(sm + ST_K + 8192, &map_k, &bar_ld, 64, h_, (int)tok0_, pol_in);
  };
  // the next record's g (thread 0), with the arrival that closes bar_ld's batch
  auto stage_g = [&](int h_, long long tok0_) {
    if constexpr (kAttn) {  // no gate tiles: the arrival alone closes the batch
      mbar_arrive(&bar_ld);
      return;
    }
    mbar_arrive_expect_tx(&bar_ld, 32768);
    for (int qtr = 0; qtr < 4; ++qtr)
      tma_load_3d_hint(sm + ST_G + qtr * 8192, &map_g, &bar_ld, 32 * qtr, h_, (int)tok0_,
                       pol_in);
  };
  // the next record's q and v halves (lane 0 of warps 0..3), after thread 0's arrival
  // registered their bytes
  auto stage_qv = [&](int h_, long long tok0_) {
    if (lane != 0 || warp >= 4) return;
    const int half = warp & 1;
    if (warp < 2)
      tma_load_3d_hint(sm + ST_Q + half * 8192, &map_q, &bar_qv, 64 * half, h_, (int)tok0_,
                       pol_in);
    else
      tma_load_3d_hint(sm + ST_V + half * 8192, &map_v, &bar_qv, 64 * half, h_, (int)tok0_,
                       pol_in);
  };
  auto stage_issue = [&](int h_, long long tok0_) {
    if (lane != 0) return;
    const int r0 = (int)tok0_;
    for (int box = warp; box < (kAttn ? 6 : 10); box += 8) {
      if (box < 6) {
        const int half = box & 1, which = box >> 1;  // q, k, v halves
        const CUtensorMap* m = which == 0 ? &map_q : which == 1 ? &map_k : &map_v;
        const int dst = (which == 0 ? ST_Q : which == 1 ? ST_K : ST_V) + half * 8192;
        tma_load_3d_hint(sm + dst, m, which == 1 ? &bar_ld : &bar_qv, 64 * half, h_, r0,
                         pol_in);
      } else {
        const int qtr = box - 6;  // g quarters
        tma_load_3d_hint(sm + ST_G + qtr * 8192, &map_g, &bar_ld, 32 * qtr, h_, r0, pol_in);
      }
    }
  };

  if (warp == 0) {
    tmem_alloc(&s_tmem, kPTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    if constexpr (kAttn) s_decay_out = 0;
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_qv, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_g);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(lane_base) << 16);
  uint32_t mma_phase = 0;
  uint32_t wait_calls = 0;
  auto mma_wait = [&]() -> bool {
    const uint32_t slot_w = wait_calls++ & 1;
    if (tid == 0) s_wait_ok[slot_w] = mbar_wait(&bar_mma, mma_phase & 1) ? 1 : 0;
    ++mma_phase;
    __syncthreads();
    return s_wait_ok[slot_w] != 0;
  };
  bool ok = true;

  int h, n, h_next = 0, n_next = 0;
  long long tok0, tok0_next = 0, rec = 0, rec_next = 0;
  bool have = locate(rec, h, tok0, n);
  if (have && tid == 0) stage_expect();
  __syncthreads();
  if (have) stage_issue(h, tok0);
  uint32_t ld_parity = 0;
  bool ld_pending = have;  // a staging batch was issued and not yet waited for (k, g)
  bool qv_pending = have;  // (q, v)
  // element (row 16 R + i, channel c0) of a [64 x 128] bf16 tile of two SW128 boxes:
  //   (c0 / 64) * 8192 + 2 R * 1024 + swz(i)
  const uint32_t c_kb = uint32_t(c0 >> 6);
  const uint32_t c_chunk = uint32_t(((c0 & 63) * 2) >> 4);
  const uint32_t c_byte = uint32_t(((c0 & 63) * 2) & 15);
  auto swz = [&](int i) -> uint32_t {
    return uint32_t((i >> 3) * 1024 + (i & 7) * 128) +
           (((c_chunk ^ uint32_t(i & 7)) << 4) | c_byte);
  };
  const uint32_t tile_base = c_kb * 8192u + uint32_t(R) * 2048u;
  float blog = (have && tid < n) ? a.beta_logits[(tok0 + tid) * H + h] : 0.f;  // tid < 64
  // kAttn: the per-token decay in log2 units (0 past the chunk's end), read by every thread
  // after the next block barrier (the staged-tile wait)
  if constexpr (kAttn)
    if (tid < kC)
      s_gam[tid] = (have && tid < n && a.decay) ? a.decay[(tok0 + tid) * H + h] * kLog2E : 0.f;
  const bool lit = kAttn && a.literal != 0;
  const bool norm = !kAttn || a.no_l2norm == 0;
  while (have) {
    advance();
    const bool have_next = locate(rec_next, h_next, tok0_next, n_next);

    // ---- loads: this record's staged k and g tiles; raw gates and k words of (16 tokens,
    //      channels c0, c0 + 1).  q and v may still be in flight.
    {
      const uint32_t slot_w = wait_calls++ & 1;
      if (tid == 0) s_wait_ok[slot_w] = mbar_wait(&bar_ld, ld_parity) ? 1 : 0;
      __syncthreads();
      if (!s_wait_ok[slot_w]) { ok = false; break; }
      ld_pending = false;
    }
    float2 graw[16];
    uint32_t kw[16], qw[16];
    const uint8_t* gsrc = sm + ST_G + (c0 >> 5) * 8192 + (16 * R) * 128 + (c0 & 31) * 4;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if constexpr (!kAttn) graw[i] = *reinterpret_cast<const float2*>(gsrc + i * 128);
      kw[i] = *reinterpret_cast<const uint32_t*>(sm + ST_K + tile_base + swz(i));
    }
    if (n < kC) {  // partial chunk (uniform): rows past n belong to the next sequence
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (16 * R + i >= n) {
          graw[i] = make_float2(0.f, 0.f);
          kw[i] = 0u;
        }
    }

    // ---- gate prefix over this thread's sub-chunk, beta
    float2 loc[16];  // (G_t - P_R) log2 e for channels (c0, c0 + 1), packed pairs
    if constexpr (kAttn) {  // one decay per token, the same on both channels
      float run = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        run += s_gam[16 * R + i];
        loc[i] = make_float2(run, run);
      }
      *reinterpret_cast<float2*>(&s_gtot[R][c0]) = make_float2(run, run);
      // decays in [-5, 1] keep a sub-chunk's sum in [-80, 16], where its factors stay
      // inside fp32; a sum outside it is reported (bit 5 of the device error mask)
      if (!(run >= -80.01f * kLog2E && run <= 16.01f * kLog2E)) s_decay_out = 1;
    } else {
      // the gate in log2 units: gamma log2 e = lb2 / (1 + 2^(na2 (g + dt_bias)))
      const float na2 = -__expf(a.a_log[h]) * kLog2E;
      const float cb0 = na2 * a.dt_bias[c0 * H + h], cb1 = na2 * a.dt_bias[(c0 + 1) * H + h];
      const float lb2 = a.lower_bound * kLog2E;
      // channel pairs ride Blackwell's two-lane fp32 instructions.  Tokens past a partial
      // chunk's end (their raw gate zeroed above, their k and q zero) run through the same
      // instructions: their gates lie in [lower_bound, 0] like every other, so their factors
      // stay in range, and the sub-chunk total stops at the last live token.
      const float2 na2v = make_float2(na2, na2), cbv = make_float2(cb0, cb1);
      const float2 one = make_float2(1.f, 1.f), lbv = make_float2(lb2, lb2);
      float2 run = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 x = __ffma2_rn(na2v, graw[i], cbv);
        const float2 den = __fadd2_rn(one, make_float2(fast_exp2(x.x), fast_exp2(x.y)));
        run = __ffma2_rn(lbv, make_float2(fast_rcp(den.x), fast_rcp(den.y)), run);
        loc[i] = run;
      }
      if (n < kC) {
        const int live = n - 16 * R;  // live tokens of this sub-chunk (may be <= 0)
        run = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < live) run = loc[i];
      }
      *reinterpret_cast<float2*>(&s_gtot[R][c0]) = run;
    }
    if (tid < kC) s_beta[tid] = (tid < n) ? (kAttn ? blog : sigmoidf_(blog)) : 0.f;

    // transposed [128 x 64] tile rows c0, c0 + 1 (tokens contiguous): row c0 takes the low
    // halves, row c0 + 1 the high halves; lanes 4..7 of every 8-lane group write row c0 + 1
    // first so that one 128-bit wavefront covers 8 swizzle phases.
    const int tsw = (lane & 4) ? 1 : 0;
    auto store_t8 = [&](int off, const uint32_t* w8, int g8) {
      const uint4 lo = make_uint4(__byte_perm(w8[0], w8[1], 0x5410), __byte_perm(w8[2], w8[3], 0x5410),
                                  __byte_perm(w8[4], w8[5], 0x5410), __byte_perm(w8[6], w8[7], 0x5410));
      const uint4 hi = make_uint4(__byte_perm(w8[0], w8[1], 0x7632), __byte_perm(w8[2], w8[3], 0x7632),
                                  __byte_perm(w8[4], w8[5], 0x7632), __byte_perm(w8[6], w8[7], 0x7632));
      *reinterpret_cast<uint4*>(sm + off + trow_off(c0 + tsw, g8)) = tsw ? hi : lo;
      *reinterpret_cast<uint4*>(sm + off + trow_off(c0 + 1 - tsw, g8)) = tsw ? lo : hi;
    };

    // ---- the staged q and v tiles; q words
    {
      const uint32_t slot_w = wait_calls++ & 1;
      if (tid == 0) s_wait_ok[slot_w] = mbar_wait(&bar_qv, ld_parity) ? 1 : 0;
      __syncthreads();
      if (!s_wait_ok[slot_w]) { ok = false; break; }
      qv_pending = false;
      ld_parity ^= 1u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
      qw[i] = *reinterpret_cast<const uint32_t*>(sm + ST_Q + tile_base + swz(i));
    if (n < kC) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (16 * R + i >= n) qw[i] = 0u;
      // the v tile's rows past n are zeroed where MMA2 reads them (whole 128-byte rows, so
      // the swizzle does not matter)
      for (int u = tid; u < 1024; u += kPThreads) {
        const int row = (u >> 3) & 63;
        if (row >= n)
          *reinterpret_cast<uint4*>(sm + ST_V + (u >> 9) * 8192 + row * 128 + (u & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
    }

    // ---- |q_t|^2: this thread's two channels, then a reduce-scatter over the warp's 32
    //      channel pairs (lanes l and l ^ 1 end with the same token); two warps per token.
    if (norm) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x = bf16_lo(qw[i]), y = bf16_hi(qw[i]);
        v[i] = x * x + y * y;
      }
#pragma unroll
      for (int half = 8, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
        const bool up = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = up ? v[i] : v[i + half];
          const float keep = up ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      const int tq = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                     ((lane >> 1) & 1);
      if ((lane & 1) == 0) s_qq[warp & 1][16 * R + tq] = v[0];
    }
    // the previous record's -W^T store has read its staging tile (inside Kb) before Kb is
    // rewritten below
    if (tma_thread) bulk_wait_read_all();
    __syncthreads();

    // ---- gate-scaled operands of (channels c0, c0 + 1) x (tokens 16 R .. 16 R + 15)
    // K^^T words (rows c0, c0 + 1, tokens 16 R + 8 hf .. + 7): staged once MMA1 is done
    uint4 khv[4];
    {
      float P0[4], P1[4];  // P_R: G just before sub-chunk R
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
      const float eP0 = fast_exp2(Pm0), eP1 = fast_exp2(Pm1);                // e^{P_R}
      const float eCP0 = fast_exp2(Gc0 - Pm0), eCP1 = fast_exp2(Gc1 - Pm1);  // e^{G_C - P_R}
      float cR0[4], cR1[4];  // e^{P_R' - P_R} for later sub-chunks R'
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        cR0[r] = (r > R) ? fast_exp2(P0[r] - Pm0) : 0.f;
        cR1[r] = (r > R) ? fast_exp2(P1[r] - Pm1) : 0.f;
      }
      if (R == 0) *reinterpret_cast<float2*>(&s_dec[c0]) = make_float2(fast_exp2(Gc0), fast_exp2(Gc1));

      const uint32_t eP2 = pack_bf16(eP0, eP1), eCP2 = pack_bf16(eCP0, eCP1);
      const uint32_t c12 = pack_bf16(cR0[1], cR1[1]), c22 = pack_bf16(cR0[2], cR1[2]),
                     c32 = pack_bf16(cR0[3], cR1[3]);
      // element (row 16 R + i, channel c0) of a K-major SW128 tile with `rows` rows:
      //   (c0 / 64) * rows * 128 + 2 R * 1024 + sw[i]
      uint8_t* const p128 = sm + P_XL + c_kb * 16384u + uint32_t(R) * 2048u;
      uint8_t* const p160 = sm + P_KB + c_kb * 20480u + uint32_t(R) * 2048u;
      __nv_bfloat16* const qrec = ws.qw + (rec * 64 + 16 * R) * kD + c0;  // Q~ row 16 R
      // literal order: the key side takes e^{G_{t-1} - P_R}, the previous token's factor
      // (1 for the sub-chunk's first token)
      uint32_t e2_prev = 0x3F803F80u;  // bf16 pair (1, 1)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t khw[8], ktw[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int i = 8 * hf + ii;
          const uint32_t swi = uint32_t(hf * 1024 + ii * 128) +
                               (((c_chunk ^ uint32_t(ii)) << 4) | c_byte);
          const float e0 = fast_exp2(loc[i].x), e1 = fast_exp2(loc[i].y);  // e^{G_t - P_R}
          const uint32_t e2 = pack_bf16(e0, e1);
          const uint32_t i2 = pack_bf16(fast_rcp(e0), fast_rcp(e1));  // e^{P_R - G_t}
          const uint32_t xk = hmul2(kw[i], lit ? e2_prev : e2);
          const uint32_t xq = hmul2(qw[i], e2), kd = hmul2(kw[i], i2);
          e2_prev = e2;
          *reinterpret_cast<uint32_t*>(p128 + swi) = xk;             // Xl row t
          *reinterpret_cast<uint32_t*>(p128 + swi + 8 * 1024) = xq;  // Xl row 64 + t
          *reinterpret_cast<uint32_t*>(p160 + swi) = kd;             // Kb diagonal row t
          if (R < 1) *reinterpret_cast<uint32_t*>(p160 + swi + 8 * 1024) = hmul2(kd, c12);
          if (R < 2) *reinterpret_cast<uint32_t*>(p160 + swi + 10 * 1024) = hmul2(kd, c22);
          if (R < 3) *reinterpret_cast<uint32_t*>(p160 + swi + 14 * 1024) = hmul2(kd, c32);
          if constexpr (kBwd) {  // q^ e^{G_t} = rq q e^{G_t}
            const int t = 16 * R + i;
            const float rqt =
                (t < n) ? a.scale * rsqrtf(s_qq[0][t] + s_qq[1][t] + kL2Eps) : 0.f;
            *reinterpret_cast<uint32_t*>(qrec + i * kD) =
                pack_bf16(bf16_lo(qw[i]) * e0 * eP0 * rqt, bf16_hi(qw[i]) * e1 * eP1 * rqt);
          } else {
            *reinterpret_cast<uint32_t*>(qrec + i * kD) = hmul2(xq, eP2);  // q e^{G_t}
          }
          khw[ii] = hmul2(kd, eCP2);  // k e^{G_C - G_t}
          ktw[ii] = hmul2(xk, eP2);   // k e^{G_t} (literal order: k e^{G_{t-1}})
        }
        store_t8(P_KTT, ktw, 2 * R + hf);
        // K^^T record rows c0, c0 + 1, tokens 16 R + 8 hf .. + 7
        const uint4 lo = make_uint4(__byte_perm(khw[0], khw[1], 0x5410), __byte_perm(khw[2], khw[3], 0x5410),
                                    __byte_perm(khw[4], khw[5], 0x5410), __byte_perm(khw[6], khw[7], 0x5410));
        const uint4 hi = make_uint4(__byte_perm(khw[0], khw[1], 0x7632), __byte_perm(khw[2], khw[3], 0x7632),
                                    __byte_perm(khw[4], khw[5], 0x7632), __byte_perm(khw[6], khw[7], 0x7632));
        khv[2 * hf] = lo;
        khv[2 * hf + 1] = hi;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA1: [A; M] = Xl Kb^T  (M = 128, N = 160, K = 128)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t xa = smem_u32(sm + P_XL), kb = smem_u32(sm + P_KB);
      const uint32_t idesc = make_idesc(1, 128, kPKbRows);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ss(tm + P_TM_D1, sw128_kdesc<2>(xa, 128, s), sw128_kdesc<2>(kb, kPKbRows, s), idesc,
               s > 0);
      mma_commit(&bar_mma);
    }
    if (!(ok = mma_wait())) break;
    tc_fence_after();
    // K^^T record into the swizzled [128 x 64] staging tile (inside Kb, free once MMA1 is
    // done); stored by TMA after the next block barrier
    // (lanes 4..7 of every 8-lane group take row c0 + 1 first: one wavefront covers all
    // eight swizzle phases)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t piece = uint32_t(2 * R + hf);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = k ^ ((lane >> 2) & 1);
        const int c = c0 + e;
        *reinterpret_cast<uint4*>(sm + P_KS + (c >> 3) * 1024 + (c & 7) * 128 +
                                  ((piece ^ uint32_t(c & 7)) << 4)) =
            e ? khv[2 * hf + 1] : khv[2 * hf];
      }
    }
    fence_async_smem();

    // ---- norms: |k_r|^2 = A_raw[r][r] (diagonal of D1); |q_r|^2 from the reduction
    //      (kAttn without L2 norm: rk = 1, rq = scale; literal order: the diagonal holds
    //      |k_r|^2 e^{-gamma_r})
    if (warp < 2) {
      const int r = 32 * warp + lane;
      if (norm) {
        float v32[32];
        tmem_ld32(tl + P_TM_D1 + 32 * warp, v32);
        float nn = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) nn = (i == lane) ? v32[i] : nn;
        if (lit) nn *= fast_exp2(s_gam[r]);
        s_rk[r] = (r < n) ? rsqrtf(nn + kL2Eps) : 0.f;
      } else {
        s_rk[r] = (r < n) ? 1.f : 0.f;
      }
    } else if (warp < 4) {
      const int r = tid - 64;
      s_rq[r] = (r < n) ? a.scale * (norm ? rsqrtf(s_qq[0][r] + s_qq[1][r] + kL2Eps) : 1.f)
                        : 0.f;
    }
    __syncthreads();
    if (tma_thread) {
      tma_store_2d(&map_ku, sm + P_KS, 0, (int)(rec * 128));
      bulk_commit();
    }
    // vector record: e^{G_C}, rk, rq
    ws.vec[rec * 256 + tid] = tid < 128 ? s_dec[tid] : tid < 192 ? s_rk[tid - 128] : s_rq[tid - 192];

    // ---- read A (TMEM lanes 0..63) and M (lanes 64..127); warpgroup wg takes the column
    //      quarters q = wg, wg + 2.  Every tcgen05.ld address is warp-uniform.
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int q = wg + 2 * qq;
      const int r = ln & 63, Rr = r >> 4;
      const int Rlo = 2 * ((warp & 3) & 1);  // the two row quarters this warp's lanes span
      float v[16];
      {
        float d16[16];
        tmem_ld16(tl + P_TM_D1 + 16 * q, d16);
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = (Rr == q) ? d16[m] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int Rp = Rlo + e;
        if (q < Rp) {  // warp-uniform
          const int offR = (Rp == 1) ? 64 : (Rp == 2) ? 80 : 112;
          float d16[16];
          tmem_ld16(tl + P_TM_D1 + offR + 16 * q, d16);
#pragma unroll
          for (int m = 0; m < 16; ++m) v[m] = (Rr == Rp) ? d16[m] : v[m];
        }
      }
      if (ln < 64) {
        // L = diag(beta rk) A diag(rk).  The solve reads only L's strictly lower triangle,
        // so the entries on and above the diagonal are written as they come (finite), with
        // no mask.
        const float sr = s_beta[r] * s_rk[r];
        const float2 srv = make_float2(sr, sr);
        float* L = reinterpret_cast<float*>(sm + P_L) + r * LDL + 16 * q;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const float4 rk4 = *reinterpret_cast<const float4*>(&s_rk[16 * q + 4 * m4]);
          const float2 lo = __fmul2_rn(__fmul2_rn(srv, make_float2(rk4.x, rk4.y)),
                                       make_float2(v[4 * m4 + 0], v[4 * m4 + 1]));
          const float2 hi = __fmul2_rn(__fmul2_rn(srv, make_float2(rk4.z, rk4.w)),
                                       make_float2(v[4 * m4 + 2], v[4 * m4 + 3]));
          reinterpret_cast<float4*>(L)[m4] = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
      } else {
        uint32_t pk[8];
        const float mf = kBwd ? s_rq[r] : 1.f;  // backward records: rows of rq_r M_raw
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int s0 = 16 * q + 2 * p;
          pk[p] = pack_bf16((s0 <= r) ? mf * v[2 * p] : 0.f,
                            (s0 + 1 <= r) ? mf * v[2 * p + 1] : 0.f);
        }
        // row r, 16-byte chunks 2 q and 2 q + 1 of the swizzled [64 x 64] staging tile
        uint8_t* const mrow = sm + P_MS + (r >> 3) * 1024 + (r & 7) * 128;
        const uint32_t sw = uint32_t(r & 7);
        *reinterpret_cast<uint4*>(mrow + ((uint32_t(2 * q) ^ sw) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(mrow + ((uint32_t(2 * q + 1) ^ sw) << 4)) =
            make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tma_thread) {
      if (have_next) {
        bulk_wait_read_all();  // the K^^T store has read its staging tile: k goes there
        stage_k(h_next, tok0_next);
      }
      tma_store_2d(&map_m, sm + P_MS, 0, (int)(rec * 64));
      bulk_commit();
    }
    if (have_next) ld_pending = true;

    // ---- T = (I + L)^{-1} diag(beta), blocked by 16
    {
      const float* L = reinterpret_cast<const float*>(sm + P_L);
      float* X = reinterpret_cast<float*>(sm + P_X);
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
          x[r] = (r == s) ? 1.f : -(acc0 + acc1);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) X[(b0 + r) * LDL + b0 + s] = x[r];
      }
      __syncthreads();
      solve_level<1>(L, X, reinterpret_cast<float*>(sm + P_Y), warp, lane);
      __syncthreads();
      solve_level<2>(L, X, reinterpret_cast<float*>(sm + P_Y), warp, lane);
      __syncthreads();
      solve_level<3>(L, X, reinterpret_cast<float*>(sm + P_Y), warp, lane);
      if (tma_thread) bulk_wait_read_all();  // the M store has read its staging tile (T's)
      __syncthreads();
      // T[r][s] = X[r][s] beta_s and T diag(rk) (s <= r): row r, 8 columns per thread
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int r = (tid >> 3) + 32 * it, s0 = (tid & 7) * 8;
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
        // X is exactly zero above the diagonal inside its diagonal 16 x 16 blocks (forward
        // substitution) and unwritten in the blocks above them: one test per 8 columns
        const bool above = (s0 >> 4) > (r >> 4);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float t0v = above ? 0.f : xv[2 * p] * bv[2 * p];
          const float t1v = above ? 0.f : xv[2 * p + 1] * bv[2 * p + 1];
          pt[p] = pack_bf16(t0v, t1v);
          // -T diag(rk): MMA2 then yields -W^T, the record's sign, directly
          pw[p] = pack_bf16(-t0v * kv[2 * p], -t1v * kv[2 * p + 1]);
        }
        const uint32_t off = sw128_offset<2>(64, r, s0);
        if constexpr (kBwd) {  // N = (I + L)^{-1}, lower triangle, row r, columns s0 .. s0 + 7
          uint32_t pn[4];
#pragma unroll
          for (int p = 0; p < 4; ++p)
            pn[p] = pack_bf16(above ? 0.f : xv[2 * p], above ? 0.f : xv[2 * p + 1]);
          *reinterpret_cast<uint4*>(ws.nrec + (rec * 64 + r) * 64 + s0) =
              make_uint4(pn[0], pn[1], pn[2], pn[3]);
        }
        *reinterpret_cast<uint4*>(sm + P_T + off) = make_uint4(pt[0], pt[1], pt[2], pt[3]);
        *reinterpret_cast<uint4*>(sm + P_TW + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA2: U~^T = V^T T^T (M = 128, N = 64, K = 64) and
    //      forward records: [T; -T diag(rk)] K~ (M = 128: the T and -T diag(rk) tiles are
    //        adjacent, N = 128 channels): its rows 64..127 are -W, token-major;
    //      backward records: -W^T = K~^T (-T diag(rk))^T (M = 128 channels, N = 64)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ts = smem_u32(sm + P_T), tw = smem_u32(sm + P_TW),
                     ks = smem_u32(sm + P_KTT), vs = smem_u32(sm + P_V);
      const uint32_t idesc = make_idesc(1, 128, 64), idesc_n128 = make_idesc(1, 128, 128);
      // V^T as the A operand is v as staged ([64 tok][128] in two 64-channel boxes), read
      // MN-major: 16 tokens (2 KB) per K step, the channel boxes 8 KB apart
      const uint32_t idesc_amn = make_idesc(1, 128, 64, true, false);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if constexpr (kBwd)
          mma_ss(tm + P_TM_DW, sw128_kdesc<2>(ks, 128, s), sw128_kdesc<2>(tw, 64, s), idesc,
                 s > 0);
        else
          mma_ss(tm + P_TM_DW, sw128_kdesc<2>(ts, 128, s), sw128_kdesc<2>(ks, 128, s),
                 idesc_n128, s > 0);
        mma_ss(tm + P_TM_DU, make_sdesc(vs + uint32_t(s) * 2048u, 8192u, 1024u, kSwizzle128),
               sw128_kdesc<2>(ts, 64, s), idesc_amn, s > 0);
      }
      mma_commit(&bar_mma);
    }
    if (tma_thread && have_next) {
      stage_g(h_next, tok0_next);                // L and X are free (T tiles written)
      mbar_arrive_expect_tx(&bar_qv, 2 * 16384);  // q and v, issued once MMA2 is done
    }
    if (!(ok = mma_wait())) break;
    tc_fence_after();
    // K~^T and the v tile are free now (MMA2 was their last reader)
    if (have_next) {
      stage_qv(h_next, tok0_next);
      qv_pending = true;
    }

    // ---- records.  U~^T: thread (j = ln, wg) holds row j for tokens 32 wg .. + 31, stored
    //      piece-major (read only by the scan's threads), coalesced as it stands.
    //      Forward: -W row t = ln - 64 (TMEM lanes 64..127), channels 64 wg .. + 63, into a
    //      swizzled [64 x 128] staging tile (two 64-channel boxes) and two bulk-tensor stores.
    //      Backward records: -W^T row j, tokens 32 wg .. + 31, into a swizzled [128 x 64]
    //      staging tile and one bulk-tensor store.
    {
      float w32[32];
      if constexpr (kBwd) {
        tmem_ld32(tl + P_TM_DW + 32 * wg, w32);
        // row ln of the swizzled [128 x 64] staging tile: 16-byte pieces 4 wg .. 4 wg + 3
        uint8_t* const wrow = sm + P_W + (ln >> 3) * 1024 + (ln & 7) * 128;
#pragma unroll
        for (int p = 0; p < 4; ++p)
          *reinterpret_cast<uint4*>(wrow + (((4 * wg + p) ^ (ln & 7)) << 4)) =
              make_uint4(pack_bf16(w32[8 * p + 0], w32[8 * p + 1]),
                         pack_bf16(w32[8 * p + 2], w32[8 * p + 3]),
                         pack_bf16(w32[8 * p + 4], w32[8 * p + 5]),
                         pack_bf16(w32[8 * p + 6], w32[8 * p + 7]));
      } else if (ln >= 64) {  // warp-uniform: warps 2, 3, 6, 7
        const int t = ln - 64;
        uint8_t* const wrow = sm + P_W + wg * 8192 + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(tl + P_TM_DW + 64 * wg + 32 * half, w32);
#pragma unroll
          for (int p = 0; p < 4; ++p)
            *reinterpret_cast<uint4*>(wrow + (((4 * half + p) ^ (t & 7)) << 4)) =
                make_uint4(pack_bf16(w32[8 * p + 0], w32[8 * p + 1]),
                           pack_bf16(w32[8 * p + 2], w32[8 * p + 3]),
                           pack_bf16(w32[8 * p + 4], w32[8 * p + 5]),
                           pack_bf16(w32[8 * p + 6], w32[8 * p + 7]));
        }
      }
      float u32[32];
      tmem_ld32(tl + P_TM_DU + 32 * wg, u32);
      // piece P = 4 wg + p of row ln (tokens 8 P .. 8 P + 7) at piece-major position
      // P * 128 + ln: a warp's store covers 512 contiguous bytes
      uint4* urec = reinterpret_cast<uint4*>(ws.ku + (ws.recs + rec) * 8192);
#pragma unroll
      for (int p = 0; p < 4; ++p)
        urec[(4 * wg + p) * 128 + ln] = make_uint4(pack_bf16(u32[8 * p + 0], u32[8 * p + 1]),
                             pack_bf16(u32[8 * p + 2], u32[8 * p + 3]),
                             pack_bf16(u32[8 * p + 4], u32[8 * p + 5]),
                             pack_bf16(u32[8 * p + 6], u32[8 * p + 7]));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tma_thread) {
      if constexpr (kBwd) {
        tma_store_2d(&map_ku, sm + P_W, 0, (int)((2 * ws.recs + rec) * 128));
      } else {
        tma_store_2d(&map_wr, sm + P_W, 0, (int)(rec * 64));
        tma_store_2d(&map_wr, sm + P_W + 8192, 64, (int)(rec * 64));
      }
      bulk_commit();
    }
    rec = rec_next;
    h = h_next;
    tok0 = tok0_next;
    n = n_next;
    have = have_next;
    blog = (have && tid < n) ? a.beta_logits[(tok0 + tid) * H + h] : 0.f;
    if constexpr (kAttn)
      if (tid < kC)
        s_gam[tid] = (have && tid < n && a.decay) ? a.decay[(tok0 + tid) * H + h] * kLog2E
                                                  : 0.f;
  }

  if (!ok) {
    if (tid == 0) {
      atomicOr(&g_split_error, 2u);
      if (ld_pending) mbar_wait(&bar_ld, ld_parity, 1000000000ull);  // staging in flight
      if (qv_pending) mbar_wait(&bar_qv, ld_parity, 1000000000ull);
    }
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  }
  if (tma_thread) bulk_wait_read_all();  // the last staging tile is read before exit
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (kAttn)
    if (tid == 0 && s_decay_out) atomicOr(&g_split_error, 32u);
  if (warp == 0) tmem_dealloc(tm, kPTmemCols);
}

// ------------------------------------------------------------------- scan kernel

constexpr int kSThreads = 512;
// one stage = one chunk's record
// Forward records: [Q~ box 0 | -W box 0 | Q~ box 1 | -W box 1], each [64 tok x 64 ch] bf16
// with 128-byte swizzle: the K-major B operand [Q~; -W] (channels 0..63 in the first 16 KB,
// 64..127 in the second) of one N = 128 MMA for the output and U products.  Backward records:
// Q~ boxes 0 and 1, then -W^T [128 x 64].  K^^T and M_raw are adjacent: the B operand
// [K^^T; M_raw] of one N = 192 MMA for the state and output updates.
constexpr int S_Q = 0;          // Q~ [64 x 128] (two 64-channel boxes), with -W (forward)
constexpr int S_KT = 32768;     // K^^T [128 x 64]
constexpr int S_M = 49152;      // M_raw [64 x 64]
constexpr int S_UT = 57344;     // U~^T, piece-major [8][128][8 tok]
constexpr int S_V = 73728;      // e^{G_C}, rk, rq
static_assert(S_M == S_KT + 16384, "the wide MMA's operand pair");
constexpr int kStage = 74752;
constexpr uint32_t kStageTx = 74752;
constexpr uint32_t kStageTxBwd = kStageTx - 2 * 8192 - 8192;  // no Q~, no M
constexpr int S_OS = 2 * kStage;  // output staging [64 tok x 128] bf16 SW128
constexpr int S_END = S_OS + 16384;
// backward records only (the launch asks for this shared memory only then):
constexpr int S_SD = S_END;         // staged S^T image [128 x 128] (two boxes)
constexpr int S_UD = S_SD + 32768;  // staged U^T image [128 x 64]
constexpr int S_END_BWD = S_UD + 16384;
static_assert(kStage % 1024 == 0 && S_OS % 1024 == 0 && S_SD % 1024 == 0, "alignment");
constexpr size_t kSSmem = S_END + 1024;
constexpr size_t kSSmemBwd = S_END_BWD + 1024;

constexpr uint32_t S_TM_S = 0;     // fp32 master state S^T, 128
constexpr uint32_t S_TM_DO = 128;  // O'^T, 64 (right after S: one N = 192 accumulator)
constexpr uint32_t S_TM_DU = 192;  // S^T (-W)^T, 64 (right after O': one N = 128 accumulator)
constexpr uint32_t S_TM_SA = 256;  // bf16 copy of S^T (A operand), 64
constexpr uint32_t S_TM_UA = 320;  // U'^T A operand (bf16 pairs), 32
constexpr uint32_t kSTmemCols = 512;
static_assert(S_TM_DO == S_TM_S + 128 && S_TM_DU == S_TM_DO + 64, "the wide MMAs' accumulators");

// kMode 0: the forward; 1: the backward's own forward pass (per-chunk images, no output);
// 2: the training forward (output and per-chunk images)
template <int kMode>
__global__ void __launch_bounds__(kSThreads, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap map_qw,
                      const __grid_constant__ CUtensorMap map_ku,
                      const __grid_constant__ CUtensorMap map_wr,
                      const __grid_constant__ CUtensorMap map_m,
                      const __grid_constant__ CUtensorMap map_o,
                      const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_s0,
                      const __grid_constant__ CUtensorMap map_ut, const ChunkArgs a,
                      const Ws ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ uint64_t bar_ld[2], bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[2];
  __shared__ __align__(16) float s_one[64];   // unit output scale (rq folded into the records)
  constexpr bool bwd = kMode != 0;
  constexpr bool want_out = kMode != 1;
  constexpr bool fwd = kMode == 0;  // -W records token-major, interleaved with Q~
  constexpr int q_box1 = fwd ? 16384 : 8192;  // Q~'s second 64-channel box
  constexpr int w_at = fwd ? 8192 : 16384;    // -W's first box, or -W^T
  if (threadIdx.x < 64) s_one[threadIdx.x] = 1.f;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int wg = tid >> 7;
  const int ln = tid & 127;
  const int lane_base = 32 * (warp & 3);
  const int h = blockIdx.x;
  const int H = a.H;
  // The chain this CTA scans: a sequence's chunks [c0, nck), from its initial state (kind
  // 0 or 1), from zero (kind 2) or from the identity with the chunk writes dropped (kind 3).
  // The planned forward of packed inputs reads it from the chain table (longest first).
  int seq = blockIdx.y, c0 = 0, kind = 0, slot = 0, c_end = -1;
  if (fwd && ws.chains) {
    if ((int)blockIdx.y >= ws.nchains[0]) return;  // uniform: no chain for this CTA
    const int4 e = ws.chains[blockIdx.y];
    seq = e.x;
    c0 = e.y;
    c_end = e.z;
    kind = e.w & 3;
    slot = e.w >> 2;
  }
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  long long slot0;
  int nck;
  if (a.cu_seqlens) {
    slot0 = ws.coff[seq];
    nck = ws.coff[seq + 1] - ws.coff[seq];
  } else {
    slot0 = (long long)seq * ws.nck_fixed;
    nck = ws.nck_fixed;
  }
  if (c_end >= 0) nck = c_end;
  const int nrun = nck - c0;  // chunks this CTA scans
  const long long state_off = ((long long)seq * H + h) * kD * kD;
  const bool drop_u = kind == 3;
  const float* const st_in = kind <= 1 ? (a.initial_state ? a.initial_state + state_off : nullptr)
                                       : nullptr;
  float* const st_out =
      kind == 0 ? (a.final_state ? a.final_state + state_off : nullptr)
                : ws.split_st + ((long long)(3 * slot + kind - 1) * H + h) * kD * kD;
  const CUtensorMap* const omap = kind == 3 ? &map_x : &map_o;
  __nv_bfloat16* const obase = static_cast<__nv_bfloat16*>(kind == 3 ? (void*)ws.xbuf : a.out);

  if (warp == 0) {
    tmem_alloc(&s_tmem, kSTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_ld[0], 1);
    mbar_init(&bar_ld[1], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_qw);
    tma_prefetch_desc(&map_ku);
    if (fwd) tma_prefetch_desc(&map_wr);
    tma_prefetch_desc(&map_m);
    tma_prefetch_desc(omap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(lane_base) << 16);

  // the refill of stage st with chunk ch, its boxes spread over lane 0 of warps 1..7 (the
  // expected bytes were registered by thread 0 with the MMAs that last read the stage)
  auto issue_load_spread = [&](int ch, int st) {
    if ((tid & 31) != 0 || warp == 0 || warp > 7) return;
    const long long rec = (slot0 + ch) * H + h;
    uint8_t* b = sm + st * kStage;
    uint64_t* bar = &bar_ld[st];
    switch (warp) {
      case 1:
        if (fwd) {
          tma_load_2d(b + w_at, &map_wr, bar, 0, (int)(rec * 64));
          tma_load_2d(b + w_at + 16384, &map_wr, bar, 64, (int)(rec * 64));
        } else {
          tma_load_2d(b + w_at, &map_ku, bar, 0, (int)((2 * ws.recs + rec) * 128));
        }
        break;
      case 2: tma_load_2d(b + S_KT, &map_ku, bar, 0, (int)(rec * 128)); break;
      case 3: bulk_load(b + S_UT, ws.ku + (ws.recs + rec) * 8192, 16384, bar); break;
      case 4: bulk_load(b + S_V, ws.vec + rec * 256, 1024, bar); break;
      case 5: if (want_out) tma_load_2d(b + S_Q, &map_qw, bar, 0, (int)(rec * 64)); break;
      case 6: if (want_out) tma_load_2d(b + S_Q + q_box1, &map_qw, bar, 64, (int)(rec * 64)); break;
      default: if (want_out) tma_load_2d(b + S_M, &map_m, bar, 0, (int)(rec * 64)); break;
    }
  };
  // one chunk record into stage st
  auto issue_load = [&](int ch, int st) {
    const long long rec = (slot0 + ch) * H + h;
    uint8_t* b = sm + st * kStage;
    uint64_t* bar = &bar_ld[st];
    mbar_arrive_expect_tx(bar, want_out ? kStageTx : kStageTxBwd);
    const int rq = (int)(rec * 64), rw = (int)((2 * ws.recs + rec) * 128);
    if (want_out) {  // the backward's own forward pass computes no output
      tma_load_2d(b + S_Q, &map_qw, bar, 0, rq);
      tma_load_2d(b + S_Q + q_box1, &map_qw, bar, 64, rq);
      tma_load_2d(b + S_M, &map_m, bar, 0, (int)(rec * 64));
    }
    if (fwd) {
      tma_load_2d(b + w_at, &map_wr, bar, 0, rq);
      tma_load_2d(b + w_at + 16384, &map_wr, bar, 64, rq);
    } else {
      tma_load_2d(b + w_at, &map_ku, bar, 0, rw);
    }
    tma_load_2d(b + S_KT, &map_ku, bar, 0, (int)(rec * 128));
    bulk_load(b + S_UT, ws.ku + (ws.recs + rec) * 8192, 16384, bar);
    bulk_load(b + S_V, ws.vec + rec * 256, 1024, bar);
  };
  // step (chunk - c0) whose record is in flight into each stage (-1: none); same on every
  // thread
  int inflight[2] = {nrun > 0 ? 0 : -1, nrun > 1 ? 1 : -1};
  if (tid == 0) {
    if (nrun > 0) issue_load(c0, 0);
    if (nrun > 1) issue_load(c0 + 1, 1);
  }

  // Initial state: thread (j = ln, warpgroup wg) owns S^T[j][32 wg .. 32 wg + 31].
  {
    float S[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      S[i] = kind == 3 ? (c == ln ? 1.f : 0.f)
                       : st_in ? st_in[(long long)c * kD + ln] : 0.f;
    }
    tmem_st32(tl + S_TM_S + 32 * wg, S);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
    tmem_st16(tl + S_TM_SA + 16 * wg, w);
    if (bwd && nck > 0) {  // the state entering chunk 0
      uint4* d = reinterpret_cast<uint4*>(ws.s0 + ((slot0 * H + h) * 128 + ln) * 128 + 32 * wg);
#pragma unroll
      for (int p = 0; p < 4; ++p)
        d[p] = make_uint4(w[4 * p], w[4 * p + 1], w[4 * p + 2], w[4 * p + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();

  const uint32_t idesc_n64 = make_idesc(1, 128, 64);
  const uint32_t idesc_n64_bmn = make_idesc(1, 128, 64, false, true);
  const uint32_t idesc_n128 = make_idesc(1, 128, 128);
  const uint32_t idesc_n192 = make_idesc(1, 128, 192);
  uint32_t mma_phase = 0;
  uint32_t wait_calls = 0;
  auto block_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t slot_w = wait_calls++ & 1;
    if (tid == 0) s_wait_ok[slot_w] = mbar_wait(bar, parity) ? 1 : 0;
    __syncthreads();
    return s_wait_ok[slot_w] != 0;
  };
  auto mma_wait = [&]() -> bool {
    const bool w = block_wait(&bar_mma, mma_phase & 1);
    ++mma_phase;
    return w;
  };
  bool ok = true;

  for (int ch = c0; ch < nck; ++ch) {
    const int it = ch - c0;  // step of this CTA's chain
    const int st = it & 1;
    uint8_t* const b = sm + st * kStage;
    // e^{G_C}, rk, rq, read from the stage itself (it is refilled after the output phase)
    const float* const vec = reinterpret_cast<const float*>(b + S_V);
    const int n = min(kC, len - ch * kC);
    const long long tok0 = bos + (long long)ch * kC;

    // the previous step's image stores have read their staging tiles before they are rewritten
    if (tid == 0 && bwd) bulk_wait_read_all();
    if (!(ok = block_wait(&bar_ld[st], (it >> 1) & 1))) break;
    inflight[st] = -1;

    // ---- MMA3: O'^T = S^T Q~^T, D_U = S^T (-W)^T  (M = 128, K = 128).  Forward records:
    //      one N = 128 MMA over the K-major B operand [Q~; -W] into the adjacent O' and D_U
    //      columns.  Backward records: the -W^T record read MN-major (16 channel rows per K
    //      step) and Q~ K-major, N = 64 each.
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ws_ = smem_u32(b + w_at), qs = smem_u32(b + S_Q);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        if constexpr (fwd) {
          mma_ts(tm + S_TM_DO, tm + S_TM_SA + 8 * s, sw128_kdesc<2>(qs, 128, s), idesc_n128,
                 s > 0);
        } else {
          mma_ts(tm + S_TM_DU, tm + S_TM_SA + 8 * s,
                 make_sdesc(ws_ + uint32_t(s) * 2048u, 8192u, 1024u, kSwizzle128),
                 idesc_n64_bmn, s > 0);
          if (want_out)
            mma_ts(tm + S_TM_DO, tm + S_TM_SA + 8 * s, sw128_kdesc<2>(qs, 64, s), idesc_n64,
                   s > 0);
        }
      }
      mma_commit(&bar_mma);
    }
    // meanwhile: decay the fp32 master state in place (S^T diag(e^{G_C}))
    {
      float S[32];
      tmem_ld32(tl + S_TM_S + 32 * wg, S);
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] *= vec[32 * wg + i];
      tmem_st32(tl + S_TM_S + 32 * wg, S);
    }
    if (!(ok = mma_wait())) break;
    tc_fence_after();
    // ---- U'^T = diag(rk) (U~ + D_U) -> bf16 A operand: thread (j = ln, tokens 16 wg .. + 15)
    {
      float v16[16];
      tmem_ld16(tl + S_TM_DU + 16 * wg, v16);
      const uint4 ua = *reinterpret_cast<const uint4*>(b + S_UT + ((2 * wg) * 128 + ln) * 16);
      const uint4 ub = *reinterpret_cast<const uint4*>(b + S_UT + ((2 * wg + 1) * 128 + ln) * 16);
      // (the identity-start chain drops the chunk's write: U~ = 0)
      const uint32_t uw[8] = {drop_u ? 0u : ua.x, drop_u ? 0u : ua.y, drop_u ? 0u : ua.z,
                              drop_u ? 0u : ua.w, drop_u ? 0u : ub.x, drop_u ? 0u : ub.y,
                              drop_u ? 0u : ub.z, drop_u ? 0u : ub.w};
      uint32_t up[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        up[i] = pack_bf16((bf16_lo(uw[i]) + v16[2 * i]) * vec[128 + 16 * wg + 2 * i],
                          (bf16_hi(uw[i]) + v16[2 * i + 1]) * vec[128 + 16 * wg + 2 * i + 1]);
      tmem_st8(tl + S_TM_UA + 8 * wg, up);
      if (bwd) {  // U^T of this chunk (before the rk row factor), staged for a TMA store
        uint32_t u8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          u8[i] = pack_bf16(bf16_lo(uw[i]) + v16[2 * i], bf16_hi(uw[i]) + v16[2 * i + 1]);
        uint8_t* row = sm + S_UD + (ln >> 3) * 1024 + (ln & 7) * 128;
        *reinterpret_cast<uint4*>(row + (((2 * wg) ^ (ln & 7)) << 4)) =
            make_uint4(u8[0], u8[1], u8[2], u8[3]);
        *reinterpret_cast<uint4*>(row + (((2 * wg + 1) ^ (ln & 7)) << 4)) =
            make_uint4(u8[4], u8[5], u8[6], u8[7]);
        fence_async_smem();
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- MMA4: S^T += U'^T K^, O'^T += U'^T M_raw^T: one N = 192 MMA over [K^^T; M_raw]
    //      (K-major, adjacent) into the adjacent S and O' columns
    if (tid == 0) {
      bulk_wait_read_all();  // the previous chunk's output store has read its staging tile
      if (bwd) {
        tma_store_2d(&map_ut, sm + S_UD, 0, (int)(((slot0 + ch) * H + h) * 128));
        bulk_commit();
      }
      tc_fence_after();
      const uint32_t ks = smem_u32(b + S_KT);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (want_out)
          mma_ts(tm + S_TM_S, tm + S_TM_UA + 8 * s, sw128_kdesc<2>(ks, 192, s), idesc_n192, 1);
        else
          mma_ts(tm + S_TM_S, tm + S_TM_UA + 8 * s, sw128_kdesc<2>(ks, 128, s), idesc_n128, 1);
      }
      mma_commit(&bar_mma);
      // the refill's bytes land on the stage's next phase (its current phase completed at
      // the top of this chunk)
      if (ch + 2 < nck) mbar_arrive_expect_tx(&bar_ld[st], want_out ? kStageTx : kStageTxBwd);
    }
    if (!(ok = mma_wait())) break;
    tc_fence_after();
    // ---- bf16 copy of the new state and the output O = diag(rq) O' (O' itself when the
    //      records carry rq)
    {
      float S[32];
      tmem_ld32(tl + S_TM_S + 32 * wg, S);
      uint32_t sp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sp[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
      tmem_st16(tl + S_TM_SA + 16 * wg, sp);
      if (bwd && ch + 1 < nck) {  // the state entering the next chunk, staged
        uint8_t* row = sm + S_SD + (wg >> 1) * 16384 + (ln >> 3) * 1024 + (ln & 7) * 128;
#pragma unroll
        for (int p = 0; p < 4; ++p)
          *reinterpret_cast<uint4*>(row + (((4 * (wg & 1) + p) ^ (ln & 7)) << 4)) =
              make_uint4(sp[4 * p], sp[4 * p + 1], sp[4 * p + 2], sp[4 * p + 3]);
      }
      if (want_out) {
        // backward records carry rq inside Q~ and M: O' is the output itself
        const float* const rqv = bwd ? s_one : vec + 192;
        float o16[16];
        tmem_ld16(tl + S_TM_DO + 16 * wg, o16);
        if (n == kC) {
          const uint32_t ob = uint32_t(ln >> 6) * 8192u + uint32_t(wg) * 2048u;
          const uint32_t och = uint32_t(((ln & 63) * 2) >> 4), oby = uint32_t(((ln & 63) * 2) & 15);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t off = ob + uint32_t((i >> 3) * 1024 + (i & 7) * 128) +
                                 (((och ^ uint32_t(i & 7)) << 4) | oby);
            *reinterpret_cast<__nv_bfloat16*>(sm + S_OS + off) =
                __float2bfloat16_rn(o16[i] * rqv[16 * wg + i]);
          }
        } else {
          __nv_bfloat16* op = obase + ((tok0 + 16 * wg) * H + h) * kD + ln;
          const long long stride = (long long)H * kD;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (16 * wg + i < n) op[i * stride] = __float2bfloat16_rn(o16[i] * rqv[16 * wg + i]);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && want_out) {
      if (n == kC) {
        tma_store_3d(omap, sm + S_OS, 0, h, (int)tok0);
        tma_store_3d(omap, sm + S_OS + 8192, 64, h, (int)tok0);
        bulk_commit();
      }
    }
    // the stage is consumed (its last readers were MMA4, the U' pack and the output's rq):
    // refill it
    if (ch + 2 < nck) issue_load_spread(ch + 2, st);
    inflight[st] = (ch + 2 < nck) ? it + 2 : -1;
    if (tid == 0 && bwd && ch + 1 < nck) {
      const int row = (int)(((slot0 + ch + 1) * H + h) * 128);
      tma_store_2d(&map_s0, sm + S_SD, 0, row);
      tma_store_2d(&map_s0, sm + S_SD + 16384, 64, row);
      bulk_commit();
    }
    // ---- end of chunk
  }

  if (!ok) {
    if (tid == 0) {
      atomicOr(&g_split_error, 2u);
      // records still in flight land before the shared memory is released
      for (int st = 0; st < 2; ++st)
        if (inflight[st] >= 0) mbar_wait(&bar_ld[st], (inflight[st] >> 1) & 1, 1000000000ull);
    }
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  } else if (st_out) {
    tc_fence_after();
    float S[32];
    tmem_ld32(tl + S_TM_S + 32 * wg, S);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      st_out[(long long)c * kD + ln] = S[i];
    }
  }
  if (tid == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kSTmemCols);
}

// ------------------------------------------------------------ split-chain fix-up

// After the scan of a planned packed forward: for each split sequence (slot s, cut at chunk
// mid) and head h, the end state S0 + P S_mid and, for the tokens of the second part,
// out += X S_mid (X: the identity-start chain's outputs, tokens x key channels).  Both are
// tcgen05 products with S_mid as the MN-major B operand; the end state takes P and S_mid
// each as a bf16 pair (hi, lo = x - hi) and sums Ph Sh + Ph Sl + Pl Sh, about 2^-16 from
// the fp32 product.  Work units per (s, h): the end state, then the 128-token tiles of the
// second part; each CTA takes a contiguous range of units, so consecutive units share the
// staged S_mid, and the next tile's X rows load while the current unit finishes.
constexpr int kFThreads = 256;
constexpr int F_X = 0;        // X tile [128 tok x 128] bf16: two 64-channel boxes of 128 rows
constexpr int F_B = 32768;    // S_mid hi (bf16) as the MN-major B operand [128 k][128 n]
constexpr int F_BL = 65536;   // S_mid lo
constexpr int F_PH = 98304;   // P hi (bf16) as the K-major A operand [128 i][128 k]
constexpr int F_PL = 131072;  // P lo
constexpr size_t kFSmem = 163840 + 1024;

__global__ void __launch_bounds__(kFThreads, 1)
    chunk_fixup_kernel(const __grid_constant__ CUtensorMap map_x, const ChunkArgs a,
                       const Ws ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ uint64_t bar_x, bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_ok;
  const int k = ws.nchains[1];
  if (k == 0) return;  // uniform
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
  const int H = a.H;
  // per split: first token of the second part, its end, and its 128-token tile count
  long long t_first[kMaxSplit], t_end[kMaxSplit], u_first[kMaxSplit + 1];
  int ntile[kMaxSplit];
  u_first[0] = 0;
  for (int s2 = 0; s2 < kMaxSplit; ++s2) {
    ntile[s2] = 0;
    t_first[s2] = t_end[s2] = 0;
    if (s2 < k) {
      const int4 sp = ws.splits[s2];
      long long bos;
      int len;
      seq_range(a, sp.x, bos, len);
      t_first[s2] = bos + (long long)sp.y * kC;
      t_end[s2] = bos + len;
      ntile[s2] = (int)((t_end[s2] - t_first[s2] + 127) / 128);
    }
    u_first[s2 + 1] = u_first[s2] + (long long)H * (1 + ntile[s2]);
  }
  const long long total = u_first[k];
  const long long u_lo = total * blockIdx.x / gridDim.x;
  const long long u_hi = total * (blockIdx.x + 1) / gridDim.x;
  if (u_lo >= u_hi) return;  // uniform
  if (warp == 0) {
    tmem_alloc(&s_tmem, 128);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_x, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(32 * (warp & 3)) << 16);
  const long long sq = (long long)kD * kD;
  // unit -> (split, head, u): u = 0 the end state, else tile u - 1
  auto decode = [&](long long unit, int& s2, int& h, int& u) {
    s2 = 0;
    while (s2 < k - 1 && unit >= u_first[s2 + 1]) ++s2;
    const long long r = unit - u_first[s2];
    const int per = 1 + ntile[s2];
    h = (int)(r / per);
    u = (int)(r % per);
  };
  auto issue_x = [&](int s2, int h, int tile) {  // thread 0
    const long long t_lo = t_first[s2] + 128LL * tile;
    mbar_arrive_expect_tx(&bar_x, 32768);
    for (int q2 = 0; q2 < 4; ++q2)  // (tokens 0..63 | 64..127) x (channels 0..63 | 64..127)
      tma_load_3d(sm + F_X + (q2 >> 1) * 16384 + (q2 & 1) * 8192, &map_x, &bar_x,
                  64 * (q2 >> 1), h, (int)(t_lo + 64 * (q2 & 1)));
  };
  // a [128][128] fp32 matrix as bf16 (hi, lo) pairs, in the layout shared by the MN-major
  // B operand (rows = k, columns = n) and the K-major A operand (rows = m, columns = k)
  auto stage_pair = [&](const float* src, uint32_t hi_off, uint32_t lo_off) {
    // all of this thread's loads first (one round trip), then the conversions and stores
    constexpr int kIt = kD * kD / 8 / kFThreads;
    float4 ld[2 * kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int q2 = tid + it * kFThreads;
      const int row = q2 >> 4, c8 = (q2 & 15) * 8;
      ld[2 * it] = *reinterpret_cast<const float4*>(src + row * kD + c8);
      ld[2 * it + 1] = *reinterpret_cast<const float4*>(src + row * kD + c8 + 4);
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int q2 = tid + it * kFThreads;
      const int row = q2 >> 4, c8 = (q2 & 15) * 8;
      const float4 x0 = ld[2 * it], x1 = ld[2 * it + 1];
      const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hw[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        lw[e] = pack_bf16(x[2 * e] - bf16_lo(hw[e]), x[2 * e + 1] - bf16_hi(hw[e]));
      }
      // 64-column block c8 / 64 at 16 KB, rows of 128 bytes in 8-row swizzled groups
      const uint32_t off = uint32_t(c8 >> 6) * 16384u + uint32_t(row >> 3) * 1024u +
                           uint32_t(row & 7) * 128u +
                           ((uint32_t((c8 & 63) >> 3) ^ uint32_t(row & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + hi_off + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      if (lo_off) *reinterpret_cast<uint4*>(sm + lo_off + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  };
  int staged = -1;  // (s2 * H + h) whose S_mid (hi, lo) is staged
  uint32_t xphase = 0, mphase = 0;
  bool x_issued = false;  // the current unit's X rows are already in flight
  bool ok = true;
  const uint32_t idesc = make_idesc(1, 128, 128, false, true);
  for (long long unit = u_lo; unit < u_hi; ++unit) {
    int s2, h, u;
    decode(unit, s2, h, u);
    const int key = s2 * H + h;
    const float* smid = ws.split_st + ((long long)(3 * s2) * H + h) * sq;
    const bool state = u == 0;
    if (state && !a.final_state) continue;  // uniform
    const int tile = u - 1;
    const long long t_lo = state ? 0 : t_first[s2] + 128LL * tile;
    const long long t_hi = state ? 0 : min(t_lo + 128, t_end[s2]);
    if (!state && tid == 0 && !x_issued) issue_x(s2, h, tile);
    x_issued = false;
    // this thread's row of the result: TMEM lane r, columns 64 wg .. + 63; its addend (the
    // output rows of the tile, or the rows of S0) is loaded while the products run
    const int r_row = 32 * (warp & 3) + lane;
    const long long t_row = t_lo + r_row;
    float* const st_row = a.final_state + ((long long)ws.splits[s2].x * H + h) * sq +
                          r_row * kD + 64 * wg;
    uint4* const o4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                               (t_row * H + h) * kD + 64 * wg);
    uint4 ov[8];
    if (!state && t_row < t_hi) {
#pragma unroll
      for (int q2 = 0; q2 < 8; ++q2) ov[q2] = o4[q2];
    }
    if (staged != key) {  // (the previous unit's products, their last reader, are complete)
      stage_pair(smid, F_B, F_BL);
      staged = key;
    }
    if (state)
      stage_pair(ws.split_st + ((long long)(3 * s2 + 2) * H + h) * sq, F_PH, F_PL);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      s_ok = state ? 1 : (mbar_wait(&bar_x, xphase & 1) ? 1 : 0);
      if (s_ok) {
        tc_fence_after();
        const uint32_t bh = smem_u32(sm + F_B), bl = smem_u32(sm + F_BL);
        auto bdesc = [&](uint32_t base, int s3) {
          return make_sdesc(base + uint32_t(s3) * 2048u, 16384u, 1024u, kSwizzle128);
        };
        if (state) {
          const uint32_t ph = smem_u32(sm + F_PH), pl = smem_u32(sm + F_PL);
#pragma unroll
          for (int s3 = 0; s3 < 8; ++s3)
            mma_ss(tm, sw128_kdesc<2>(ph, 128, s3), bdesc(bh, s3), idesc, s3 > 0);
#pragma unroll
          for (int s3 = 0; s3 < 8; ++s3) mma_ss(tm, sw128_kdesc<2>(ph, 128, s3), bdesc(bl, s3), idesc, 1);
#pragma unroll
          for (int s3 = 0; s3 < 8; ++s3) mma_ss(tm, sw128_kdesc<2>(pl, 128, s3), bdesc(bh, s3), idesc, 1);
        } else {
          const uint32_t xs = smem_u32(sm + F_X);
#pragma unroll
          for (int s3 = 0; s3 < 8; ++s3)
            mma_ss(tm, sw128_kdesc<2>(xs, 128, s3), bdesc(bh, s3), idesc, s3 > 0);
        }
        mma_commit(&bar_mma);
        s_ok = mbar_wait(&bar_mma, mphase & 1) ? 1 : 0;
        // the X tile is free: the next unit's rows, when it is a tile
        if (s_ok && unit + 1 < u_hi) {
          int ns, nh, nu;
          decode(unit + 1, ns, nh, nu);
          if (nu >= 1) {
            issue_x(ns, nh, nu - 1);
            s_ok = 3;
          }
        }
      }
    }
    if (!state) ++xphase;
    ++mphase;
    __syncthreads();
    if (!s_ok) {
      ok = false;
      break;
    }
    x_issued = s_ok == 3;
    tc_fence_after();
    {
      float d[64];
      tmem_ld32(tl + 64 * wg, *reinterpret_cast<float(*)[32]>(d));
      tmem_ld32(tl + 64 * wg + 32, *reinterpret_cast<float(*)[32]>(d + 32));
      if (state) {
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          const float4 s0v = *reinterpret_cast<const float4*>(
              ws.split_st + ((long long)(3 * s2 + 1) * H + h) * sq + r_row * kD + 64 * wg + j);
          *reinterpret_cast<float4*>(st_row + j) =
              make_float4(s0v.x + d[j], s0v.y + d[j + 1], s0v.z + d[j + 2], s0v.w + d[j + 3]);
        }
      } else if (t_row < t_hi) {
#pragma unroll
        for (int q2 = 0; q2 < 8; ++q2) {
          const uint32_t w[4] = {ov[q2].x, ov[q2].y, ov[q2].z, ov[q2].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_bf16(bf16_lo(w[e]) + d[8 * q2 + 2 * e],
                             bf16_hi(w[e]) + d[8 * q2 + 2 * e + 1]);
          o4[q2] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (!ok && tid == 0) {
    atomicOr(&g_split_error, 2u);
    // the unit's loads and products land before the shared memory is released
    if (xphase > 0) mbar_wait(&bar_x, (xphase - 1) & 1, 1000000000ull);
    mbar_wait(&bar_mma, (mphase - 1) & 1, 1000000000ull);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 128);
}

// ------------------------------------------------------------ varlen chunk offsets

// coff[0] = 0, coff[i + 1] = coff[i] + ceil(len_i / 64) (lengths clamped as seq_range does);
// the whole block (a multiple of 32 threads, at most 1024) takes part.
__device__ void chunk_offsets_body(const int32_t* cu, int N, int total_T, int32_t* coff) {
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = blockDim.x, nw = nt >> 5;
  if (tid == 0) {
    s_carry = 0;
    coff[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < N; base += nt) {
    const int i = base + tid;
    int c = 0;
    if (i < N) {
      int lo = cu[i], hi = cu[i + 1];
      lo = min(max(lo, 0), total_T);
      hi = min(max(hi, lo), total_T);
      c = (hi - lo + kC - 1) / kC;
    }
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nw) s_warp[lane] = w;
    }
    __syncthreads();
    const int carry = s_carry;
    const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0);
    if (i < N) coff[i + 1] = carry + incl;
    __syncthreads();
    if (tid == nt - 1) s_carry = carry + incl;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024) chunk_offsets_kernel(const int32_t* cu, int N,
                                                             int total_T, int32_t* coff) {
  chunk_offsets_body(cu, N, total_T, coff);
}

// The chunk offsets of packed inputs, then the forward scan's plan: which sequences' chains
// are split (the longest ones, one at a time, while that shortens the longest chain and the
// chain count stays within `budget` CTAs per head-group), and the chain table in
// longest-first order, so that a scan with more chains than SMs starts the long ones first.
constexpr int kPlanSort = 4096;  // chain tables up to this size are sorted
constexpr int kPlanCache = 2048;  // chunk counts of up to this many sequences kept on chip
constexpr int kPlanThreads = 256;

// chunks of packed sequence i (its length clamped as seq_range does)
__device__ __forceinline__ int chunk_count(const int32_t* cu, int i, int total_T) {
  int lo = cu[i], hi = cu[i + 1];
  lo = min(max(lo, 0), total_T);
  hi = min(max(hi, lo), total_T);
  return (hi - lo + kC - 1) / kC;
}

// The plan of chunk_plan_kernel for at most kPlanThreads sequences, one per thread: every
// sequence's rank by length (longer first, ties by index) and every chain's rank in the
// table are counted directly (a few block barriers instead of selection rounds and a sort).
__device__ void plan_small(const int32_t* cu, int N, int total_T, int H, int budget,
                           int4* chains, int32_t* counts, int4* splits) {
  __shared__ int s_len[kPlanThreads + 2 * kMaxSplit];
  __shared__ int s_top_seq[kMaxSplit + 1], s_top_len[kMaxSplit + 1];
  __shared__ int s_slot[kPlanThreads];  // split slot of each sequence, -1 if whole
  __shared__ int s_k;
  const int tid = threadIdx.x;
  const int nck = tid < N ? chunk_count(cu, tid, total_T) : 0;
  if (tid < N) s_len[tid] = nck;
  __syncthreads();
  if (tid < N) {
    int r = 0;
    for (int j = 0; j < N; ++j) r += (s_len[j] > nck) || (s_len[j] == nck && j < tid);
    if (r <= kMaxSplit) {
      s_top_seq[r] = tid;
      s_top_len[r] = nck;
    }
    s_slot[tid] = -1;
  }
  __syncthreads();
  if (tid == 0) {
    int k = 0, crit = N > 0 ? s_top_len[0] : 0;
    for (int kk = 1; kk <= min(kMaxSplit, N); ++kk) {
      if (s_top_len[kk - 1] < kSplitMinChunks) break;
      if ((long long)(N + 2 * kk) * H > (long long)budget) break;
      const int nc = max((s_top_len[0] + 1) / 2, kk < N ? s_top_len[kk] : 0);
      if (nc < crit) {
        k = kk;
        crit = nc;
      }
    }
    for (int s2 = 0; s2 < k; ++s2) {
      splits[s2] = make_int4(s_top_seq[s2], (s_top_len[s2] + 1) / 2, s_top_len[s2], 0);
      s_slot[s_top_seq[s2]] = s2;
      // the second parts' lengths: entries N + 2 s2 (from zero) and N + 2 s2 + 1 (identity)
      s_len[N + 2 * s2] = s_len[N + 2 * s2 + 1] = s_top_len[s2] - (s_top_len[s2] + 1) / 2;
    }
    s_k = k;
    counts[0] = N + 2 * k;
    counts[1] = k;
  }
  __syncthreads();
  const int k = s_k, count = N + 2 * k;
  if (tid < N && s_slot[tid] >= 0) s_len[tid] = (nck + 1) / 2;  // a split sequence's first part
  __syncthreads();
  for (int e = tid; e < count; e += kPlanThreads) {
    const int len = s_len[e];
    int r = 0;
    for (int j = 0; j < count; ++j) r += (s_len[j] > len) || (s_len[j] == len && j < e);
    int4 c;
    if (e < N) {
      const int s2 = s_slot[e];
      c = s2 >= 0 ? make_int4(e, 0, len, 1 | (s2 << 2)) : make_int4(e, 0, len, 0);
    } else {
      const int s2 = (e - N) >> 1, part = (e - N) & 1;
      const int mid = (s_top_len[s2] + 1) / 2;
      c = make_int4(s_top_seq[s2], mid, s_top_len[s2], (2 + part) | (s2 << 2));
    }
    chains[r] = c;
  }
}
__global__ void __launch_bounds__(kPlanThreads) chunk_plan_kernel(const int32_t* cu, int N, int total_T,
                                                          int H, int budget, int32_t* coff,
                                                          int4* chains, int32_t* counts,
                                                          int4* splits) {
  __shared__ unsigned long long s_key[kPlanSort];
  __shared__ int s_nck[kPlanCache];
  __shared__ unsigned long long s_red[32];
  __shared__ int s_top_seq[kMaxSplit + 1], s_top_len[kMaxSplit + 1];
  __shared__ int s_k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nt = kPlanThreads, nw = kPlanThreads / 32;
  chunk_offsets_body(cu, N, total_T, coff);
  if (N <= nt) {  // one sequence per thread: ranks by counting, no sort network
    plan_small(cu, N, total_T, H, budget, chains, counts, splits);
    return;
  }
  __syncthreads();  // coff (global memory) written by this block is visible to it
  const bool cached = N <= kPlanCache;
  if (cached)
    for (int i = tid; i < N; i += nt) s_nck[i] = coff[i + 1] - coff[i];
  __syncthreads();
  auto nck_of = [&](int i) { return cached ? s_nck[i] : coff[i + 1] - coff[i]; };
  // the r-th longest sequence (ties: the lower index) by a block maximum over the others
  auto select = [&](int r) {
    unsigned long long best = 0;
    for (int i = tid; i < N; i += nt) {
      bool taken = false;
      for (int j = 0; j < r; ++j) taken |= (s_top_seq[j] == i);
      if (taken) continue;
      const unsigned long long key =
          ((unsigned long long)(unsigned)nck_of(i) << 32) | (0xffffffffu - (unsigned)i);
      best = key > best ? key : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
      best = y > best ? y : best;
    }
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = 0;
      for (int w = 0; w < nw; ++w) b = s_red[w] > b ? s_red[w] : b;
      s_top_seq[r] = (int)(0xffffffffu - (unsigned)(b & 0xffffffffu));
      s_top_len[r] = (int)(b >> 32);
    }
    __syncthreads();
  };
  // split the kk longest sequences, kk chosen to minimise the longest chain, which is then
  // max(ceil(L_0 / 2), L_kk) (L sorted descending); the fewest splits on a tie
  const int ranks = min(kMaxSplit + 1, N);
  for (int r = 0; r < ranks; ++r) select(r);
  if (tid == 0) {
    int k = 0, crit = N > 0 ? s_top_len[0] : 0;
    for (int kk = 1; kk <= min(kMaxSplit, N); ++kk) {
      if (s_top_len[kk - 1] < kSplitMinChunks) break;
      if ((long long)(N + 2 * kk) * H > (long long)budget) break;
      const int nc = max((s_top_len[0] + 1) / 2, kk < N ? s_top_len[kk] : 0);
      if (nc < crit) {
        k = kk;
        crit = nc;
      }
    }
    s_k = k;
  }
  __syncthreads();
  if (tid == 0) {
    const int k = s_k;
    for (int s2 = 0; s2 < k; ++s2)
      splits[s2] = make_int4(s_top_seq[s2], (s_top_len[s2] + 1) / 2, s_top_len[s2], 0);
    counts[0] = N + 2 * k;
    counts[1] = k;
  }
  __syncthreads();
  const int k = s_k;
  const int count = N + 2 * k;
  // entry e < N: sequence e (whole, or its first part when split); e >= N: the second
  // part of split slot (e - N) / 2, from zero (even) or from the identity (odd)
  auto entry = [&](int e) -> int4 {
    if (e < N) {
      for (int s2 = 0; s2 < k; ++s2)
        if (s_top_seq[s2] == e) return make_int4(e, 0, (s_top_len[s2] + 1) / 2, 1 | (s2 << 2));
      return make_int4(e, 0, nck_of(e), 0);
    }
    const int s2 = (e - N) >> 1, part = (e - N) & 1;
    const int mid = (s_top_len[s2] + 1) / 2;
    return make_int4(s_top_seq[s2], mid, s_top_len[s2], (2 + part) | (s2 << 2));
  };
  if (count <= kPlanSort) {
    int n2 = 1;
    while (n2 < count) n2 <<= 1;
    for (int e = tid; e < n2; e += nt) {
      unsigned long long key = ~0ull;  // padding sorts last
      if (e < count) {
        const int4 c = entry(e);
        key = ((unsigned long long)(0x7fffffffu - (unsigned)(c.z - c.y)) << 32) | (unsigned)e;
      }
      s_key[e] = key;
    }
    __syncthreads();
    // bitonic sort, ascending: the longest chains first, ties in entry order
    for (int size = 2; size <= n2; size <<= 1)
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < n2; i += nt) {
          const int j = i ^ stride;
          if (j > i) {
            const bool up = (i & size) == 0;
            const unsigned long long a = s_key[i], b = s_key[j];
            if ((a > b) == up) {
              s_key[i] = b;
              s_key[j] = a;
            }
          }
        }
        __syncthreads();
      }
    for (int i = tid; i < count; i += nt) chains[i] = entry((int)(s_key[i] & 0xffffffffu));
  } else {
    // too many to sort here: the split chains' second parts first, then sequence order
    for (int i = tid; i < count; i += nt) chains[i] = entry(i < 2 * k ? N + i : i - 2 * k);
  }
}

// ------------------------------------------------------------------------- host

}  // namespace

// The split area of a planned packed forward: chain table, counts, split list, the three
// fp32 states per split and head, and X rows for every token (an upper bound).
static size_t split_area_bytes(const ChunkArgs& a) {
  if (!a.cu_seqlens) return 0;
  return align_up(size_t(a.B + 2 * kMaxSplit) * sizeof(int4), 256) + 256 +
         align_up(size_t(kMaxSplit) * sizeof(int4), 256) +
         size_t(kMaxSplit) * 3 * size_t(a.H) * kD * kD * 4 +
         align_up(size_t(a.total_T) * a.H * kD * 2, 256);
}

static void carve_split(const ChunkArgs& a, uint8_t* p, Ws& ws) {
  ws.chains = reinterpret_cast<int4*>(p);
  p += align_up(size_t(a.B + 2 * kMaxSplit) * sizeof(int4), 256);
  ws.nchains = reinterpret_cast<int32_t*>(p);
  p += 256;
  ws.splits = reinterpret_cast<int4*>(p);
  p += align_up(size_t(kMaxSplit) * sizeof(int4), 256);
  ws.split_st = reinterpret_cast<float*>(p);
  p += size_t(kMaxSplit) * 3 * size_t(a.H) * kD * kD * 4;
  ws.xbuf = reinterpret_cast<__nv_bfloat16*>(p);
}

size_t chunk_split_workspace(const ChunkArgs& a) {
  const long long recs = slots_for(a) * a.H;
  const size_t coff = a.cu_seqlens ? align_up(size_t(a.B + 1) * 4, 256) : 0;
  return record_bytes(recs) + coff + split_area_bytes(a);
}

bool chunk_split_index_ok(const ChunkArgs& a) {
  // TMA row coordinates of the records are 32-bit: 3 * recs * 128 < 2^31
  return slots_for(a) * a.H * 384 < 0x7fffffffLL;
}

cudaError_t split::launch_prep_scan(const ChunkArgs& a, const Ws& ws, cudaStream_t st) {
  const long long rows = a.cu_seqlens ? a.total_T : (long long)a.B * a.T;
  const long long map_rows = rows > 0 ? rows : 1;
  const long long rec_rows = ws.recs > 0 ? ws.recs : 1;
  CUtensorMap mqw, mku, mwr, mm, mo, mx, mq, mk, mv, mg, ms0, mut;
  // the backward's scan writes no output: its (unused) output map is laid over q
  // -W: the forward's records hold it token-major ([64 x 128] per record), in the space the
  // backward's -W^T records take ([128 x 64], the third part of ku)
  if (!make_map_2d(&mqw, ws.qw, rec_rows * 64, 128, 64) ||
      !make_map_2d(&mku, ws.ku, 3 * rec_rows * 128, 64, 128) ||
      !make_map_2d(&mwr, ws.ku + 2 * ws.recs * 8192, rec_rows * 64, 128, 64) ||
      !make_map_2d(&mm, ws.m, rec_rows * 64, 64, 64) ||
      !make_map_out(&mo, ws.bwd == 1 ? a.q : a.out, map_rows, a.H) ||
      // X rows of the split chains (laid over q when the call plans no splits)
      !make_map_out(&mx, ws.xbuf ? (const void*)ws.xbuf : a.q, map_rows, a.H) ||
      !make_map_in(&mq, a.q, map_rows, a.H, false) ||
      !make_map_in(&mk, a.k, map_rows, a.H, false) ||
      !make_map_in(&mv, a.v, map_rows, a.H, false) ||
      // (the attention variant stages no gate tiles: its unused map is laid over q)
      !make_map_in(&mg, a.g ? (const void*)a.g : a.q, map_rows, a.H, a.g != nullptr))
    return cudaErrorInvalidValue;
  // the per-chunk images of the backward records (laid over q when there are none)
  if (!make_map_2d(&ms0, ws.bwd ? (const void*)ws.s0 : a.q, ws.bwd ? rec_rows * 128 : 1, 128,
                   128) ||
      !make_map_2d(&mut, ws.bwd ? (const void*)ws.ut : a.q, ws.bwd ? rec_rows * 128 : 1, 64, 128))
    return cudaErrorInvalidValue;
  auto prep = ws.bwd ? chunk_prep_kernel<true, false>
                     : a.gate_head ? chunk_prep_kernel<false, true>
                                   : chunk_prep_kernel<false, false>;
  auto scan = ws.bwd == 0 ? chunk_scan_kernel<0> : ws.bwd == 1 ? chunk_scan_kernel<1>
                                                                : chunk_scan_kernel<2>;
  const size_t scan_smem = ws.bwd ? kSSmemBwd : kSSmem;
  cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kPSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem);
  if (e != cudaSuccess) return e;
  if (ws.recs > 0) {
    // persistent: two CTAs per SM (shared memory and Tensor Memory admit no more)
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const long long grid = std::min<long long>(ws.recs, 2LL * sms);
    prep<<<(unsigned)grid, kPThreads, kPSmem, st>>>(mku, mwr, mm, mq, mk, mv, mg, a, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // a planned scan has up to 2 kMaxSplit chains more than sequences (the unused CTAs exit);
  // the grid's y extent stops at 65535, which only binds when no sequence can be split (the
  // plan splits only while all chains fit in two per SM)
  const unsigned ny = std::min(65535u, (unsigned)a.B + (ws.chains ? 2u * kMaxSplit : 0u));
  scan<<<dim3(a.H, ny), kSThreads, scan_smem, st>>>(mqw, mku, mwr, mm, mo, mx, ms0, mut, a, ws);
  if ((e = cudaGetLastError()) != cudaSuccess || !ws.chains) return e;
  // the split chains' correction (no work, and an immediate return, when nothing was split)
  if ((e = cudaFuncSetAttribute(chunk_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kFSmem)) != cudaSuccess)
    return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  chunk_fixup_kernel<<<sms, kFThreads, kFSmem, st>>>(mx, a, ws);
  return cudaGetLastError();
}

cudaError_t split::launch_chunk_offsets(const ChunkArgs& a, const Ws& ws, cudaStream_t st) {
  chunk_offsets_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.B, a.total_T, ws.coff);
  return cudaGetLastError();
}

cudaError_t launch_chunk_split(const ChunkArgs& a, void* workspace, cudaStream_t st) {
  Ws ws{};
  uint8_t* p = carve_records(a, workspace, ws);
  if (a.cu_seqlens) {
    // packed inputs: the chunk offsets and the scan's plan (chains, longest first, with the
    // longest sequences split while that shortens the longest chain)
    carve_split(a, p + align_up(size_t(a.B + 1) * 4, 256), ws);
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    chunk_plan_kernel<<<1, kPlanThreads, 0, st>>>(a.cu_seqlens, a.B, a.total_T, a.H, 2 * sms, ws.coff,
                                          ws.chains, ws.nchains, ws.splits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return split::launch_prep_scan(a, ws, st);
}

unsigned int chunk_split_read_error(bool reset) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_split_error, sizeof(v));
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_split_error, &z, sizeof(z));
  }
  return v;
}

}  // namespace kda
