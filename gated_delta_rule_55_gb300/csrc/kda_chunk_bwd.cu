// Chunked backward of the KDA forward on the tensor cores (bf16 q/k/v/d_out, dk = dv = 128,
// 64-token chunks, fixed-length or packed sequences, decay-first recurrence with the kda_tkg
// gate and beta logits).  The pages give no backward ("Algorithm modes: chunked" is named as the
// training path); this is reverse-mode differentiation of the chunk form of the forward,
//
//   U = T (V - K~ S),   O = Q~ S + M U,   S' = diag(e^{G_C}) S + Kd^T U,
//   T = N diag(beta),   N = (I + diag(beta) tril(A, -1))^{-1},
//
// with K~ = k^ e^{G}, Q~ = q^ e^{G}, Kd = k^ e^{G_C - G}, A / M the gate-scaled k^ k^T and
// q^ k^T of the chunk.  Given the adjoint dS' of the state leaving a chunk and d_out:
//
//   dU  = Kd dS' + M^T dO                            (sequential over chunks, reversed)
//   dS  = diag(e^{G_C}) dS' + Q~^T dO - W^T dU
//   lam = N^T dU,  dV = diag(beta) lam,  dK~ = -dV S^T,  dQ~ = dO S^T,  dKd = U dS'^T
//   dA  = -dV U^T (s < r),  dM = dO U^T (s <= r),  dbeta_logit_r = (1 - beta_r) lam_r . u_r
//
// and the gate-scaled products A, M are differentiated through the same 16-token sub-chunk
// operand tiles (Xl, Kb) that form them in the forward.  Launches:
//
//   chunk_prep_kernel / chunk_scan_kernel (kda_chunk_split.cu, backward mode): the forward
//       records with rq folded into Q~ and M, N, and per chunk the entering state S and U;
//   bwd_scan_kernel: one CTA per (sequence, head) walks the chunks in reverse with dS' in
//       Tensor Memory, writing per chunk dS' and dU (bf16) and finally d_initial_state;
//   bwd_chunk_kernel: one CTA per (chunk, head), all at once: every other product above,
//       then the gate, L2-norm and sigmoid chain rules, writing dq, dk, dv, dg, dbeta_logits
//       and adding into da_log and ddt_bias.
//
// The training forward (launch_chunk_fwd_train) runs the first two launches with the output
// written as well; a backward on its workspace then starts at bwd_scan_kernel.
//
// Operands are the row-major 128-byte-swizzled tiles that TMA moves; a tile [lines][64] is
// read K-major when the contraction runs along its rows' elements and MN-major when it runs
// across its lines, so no operand is transposed in memory.
#include "chunk_records.cuh"

namespace kda {
namespace {

using namespace tc;
using namespace chunk;
using namespace split;

__device__ unsigned int g_bwd_error;  // bit 2: a bounded wait of the chunked backward gave up

struct BwdWs {
  Ws f;                // forward records (backward mode) and the forward scan's S, U
  __nv_bfloat16* ds;   // [recs * 128][128]: dS'^T of each chunk (row = value column j)
  __nv_bfloat16* dut;  // [recs * 128][64]: dU^T of each chunk
};

struct BwdOut {
  const float* d_final;  // [B, H, 128, 128] or NULL
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dg;
  float* dbeta_logits;
  float* da_log;
  float* ddt_bias;
  float* d_initial;      // [B, H, 128, 128] or NULL
};

// Byte offset of element e (bf16) of line `line` of a tile cut into 64-element boxes
// ([lines][64] each, `bs` bytes apart), 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_off(int line, int e, uint32_t bs) {
  const uint32_t byte = uint32_t(e & 63) * 2u;
  return uint32_t(e >> 6) * bs + uint32_t(line >> 3) * 1024u + uint32_t(line & 7) * 128u +
         ((((byte >> 4) ^ uint32_t(line & 7)) << 4) | (byte & 15u));
}

// MN-major operand descriptor of K-step s (16 lines) of such a tile: 64-element blocks of
// the M / N extent `bs` bytes apart, 8-line groups 1024 bytes apart.
__device__ __forceinline__ uint64_t mn_desc(uint32_t tile, uint32_t bs, int s) {
  return make_sdesc(tile + uint32_t(s) * 2048u, bs, 1024u, kSwizzle128);
}

// Zeroes rows n .. 63 of a [64 x 128] bf16 tile of two boxes 8192 bytes apart (rows that
// belong to the next sequence or lie past the tensor); 8 threads per row.
__device__ __forceinline__ void zero_rows(uint8_t* tile, int n, int tid) {
  const int row = tid >> 3, piece = tid & 7;
  if (row < 64 && row >= n) {
    const uint32_t base = uint32_t(piece >> 2) * 8192u + uint32_t(row >> 3) * 1024u +
                          uint32_t(row & 7) * 128u;
    const uint32_t c0 = uint32_t(piece & 3) * 2u;
    *reinterpret_cast<uint4*>(tile + base + ((c0 ^ uint32_t(row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(tile + base + (((c0 + 1) ^ uint32_t(row & 7)) << 4)) =
        make_uint4(0, 0, 0, 0);
  }
}

// Sum over the 32 lanes of eight per-lane values v[0..7]; the sum for index
// tq = 4 b4 + 2 b3 + b2 (bits of the lane) ends in v[0] of lanes with (lane & 3) == 0.
__device__ __forceinline__ float reduce_scatter8(float (&v)[8], int lane, int& tq) {
#pragma unroll
  for (int half = 4, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  tq = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
  return v[0];
}

// Both lanes of x rounded to the nearest bf16 value (kept in fp32), through one bf16x2
// conversion.
__device__ __forceinline__ float2 bf16_round2(float2 x) {
  const uint32_t p = pack_bf16(x.x, x.y);
  return make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------ reverse chunk scan

constexpr int kBSThreads = 512;
// one stage = one chunk: the forward records it needs and the chunk's d_out tile
constexpr int B_Q = 0;          // Q~ = q^ e^{G} [64 tok][128] (two boxes)
constexpr int B_W = 16384;      // -W^T [128][64 tok]
constexpr int B_KT = 32768;     // K^^T = (k e^{G_C - G})^T [128][64 tok]
constexpr int B_M = 49152;      // rq_r M_raw[r][s] [64][64]
constexpr int B_DO = 57344;     // d_out [64 tok][128] (two boxes)
constexpr int B_V = 73728;      // e^{G_C}, rk, rq
constexpr int kBStage = 74752;
constexpr uint32_t kBStageTx = 74752;
static_assert(kBStage % 1024 == 0, "alignment");
constexpr int B_SDS = 2 * kBStage;   // staged dS'^T image [128 x 128] (two boxes)
constexpr int B_SDU = B_SDS + 32768;  // staged dU^T image [128 x 64]
constexpr size_t kBSSmem = B_SDU + 16384 + 1024;

constexpr uint32_t BT_DU = 0;    // dU^T accumulator, 64 columns
constexpr uint32_t BT_S = 128;   // fp32 dS^T, 128
constexpr uint32_t BT_SA = 256;  // bf16 copy of dS^T (A operand), 64
constexpr uint32_t BT_UA = 320;  // bf16 dU^T (A operand), 32
constexpr uint32_t kBTmemCols = 512;

__global__ void __launch_bounds__(kBSThreads, 1)
    bwd_scan_kernel(const __grid_constant__ CUtensorMap map_qw,
                    const __grid_constant__ CUtensorMap map_ku,
                    const __grid_constant__ CUtensorMap map_m,
                    const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_ds,
                    const __grid_constant__ CUtensorMap map_dut, const ChunkArgs a,
                    const BwdWs bw, const BwdOut o) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ uint64_t bar_ld[2], bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[2];
  __shared__ __align__(16) float s_vec[256];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int wg = tid >> 7;
  const int ln = tid & 127;
  const int lane_base = 32 * (warp & 3);
  const int h = blockIdx.x, seq = blockIdx.y;
  const int H = a.H;
  long long bos;
  int len;
  seq_range(a, seq, bos, len);
  long long slot0;
  int nck;
  if (a.cu_seqlens) {
    slot0 = bw.f.coff[seq];
    nck = bw.f.coff[seq + 1] - bw.f.coff[seq];
  } else {
    slot0 = (long long)seq * bw.f.nck_fixed;
    nck = bw.f.nck_fixed;
  }
  const long long state_off = ((long long)seq * H + h) * kD * kD;
  auto rec_of = [&](int ch) -> long long { return (slot0 + ch) * H + h; };

  if (warp == 0) {
    tmem_alloc(&s_tmem, kBTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_ld[0], 1);
    mbar_init(&bar_ld[1], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_qw);
    tma_prefetch_desc(&map_ku);
    tma_prefetch_desc(&map_m);
    tma_prefetch_desc(&map_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(lane_base) << 16);

  // the refill of stage st for step it, its boxes spread over lane 0 of warps 1..8 (the
  // expected bytes were registered by thread 0 with the MMAs that last read the stage)
  auto issue_load_spread = [&](int it, int st) {
    if ((tid & 31) != 0 || warp == 0 || warp > 8) return;
    const int ch = nck - 1 - it;
    const long long rec = rec_of(ch);
    uint8_t* b = sm + st * kBStage;
    uint64_t* bar = &bar_ld[st];
    const int tok0 = (int)(bos + (long long)ch * kC);
    switch (warp) {
      case 1: tma_load_2d(b + B_Q, &map_qw, bar, 0, (int)(rec * 64)); break;
      case 2: tma_load_2d(b + B_Q + 8192, &map_qw, bar, 64, (int)(rec * 64)); break;
      case 3: tma_load_2d(b + B_W, &map_ku, bar, 0, (int)((2 * bw.f.recs + rec) * 128)); break;
      case 4: tma_load_2d(b + B_KT, &map_ku, bar, 0, (int)(rec * 128)); break;
      case 5: tma_load_2d(b + B_M, &map_m, bar, 0, (int)(rec * 64)); break;
      case 6: tma_load_3d(b + B_DO, &map_do, bar, 0, h, tok0); break;
      case 7: tma_load_3d(b + B_DO + 8192, &map_do, bar, 64, h, tok0); break;
      default: bulk_load(b + B_V, bw.f.vec + rec * 256, 1024, bar); break;
    }
  };
  // step `it` handles chunk nck - 1 - it
  auto issue_load = [&](int it, int st) {
    const int ch = nck - 1 - it;
    const long long rec = rec_of(ch);
    uint8_t* b = sm + st * kBStage;
    uint64_t* bar = &bar_ld[st];
    mbar_arrive_expect_tx(bar, kBStageTx);
    const int rq = (int)(rec * 64), rw = (int)((2 * bw.f.recs + rec) * 128);
    const int tok0 = (int)(bos + (long long)ch * kC);
    tma_load_2d(b + B_Q, &map_qw, bar, 0, rq);
    tma_load_2d(b + B_Q + 8192, &map_qw, bar, 64, rq);
    tma_load_2d(b + B_W, &map_ku, bar, 0, rw);
    tma_load_2d(b + B_KT, &map_ku, bar, 0, (int)(rec * 128));
    tma_load_2d(b + B_M, &map_m, bar, 0, (int)(rec * 64));
    tma_load_3d(b + B_DO, &map_do, bar, 0, h, tok0);
    tma_load_3d(b + B_DO + 8192, &map_do, bar, 64, h, tok0);
    bulk_load(b + B_V, bw.f.vec + rec * 256, 1024, bar);
  };
  int inflight[2] = {nck > 0 ? 0 : -1, nck > 1 ? 1 : -1};
  if (tid == 0) {
    if (nck > 0) issue_load(0, 0);
    if (nck > 1) issue_load(1, 1);
  }

  // dS' of the last chunk = d_final_state: thread (j = ln, wg) owns dS^T[j][32 wg .. + 31]
  {
    float S[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      S[i] = o.d_final ? o.d_final[state_off + (long long)c * kD + ln] : 0.f;
    }
    tmem_st32(tl + BT_S + 32 * wg, S);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
    tmem_st16(tl + BT_SA + 16 * wg, w);
    if (nck > 0) {
      uint4* d = reinterpret_cast<uint4*>(bw.ds + (rec_of(nck - 1) * 128 + ln) * 128 + 32 * wg);
#pragma unroll
      for (int p = 0; p < 4; ++p) d[p] = make_uint4(w[4 * p], w[4 * p + 1], w[4 * p + 2], w[4 * p + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();

  const uint32_t idesc_du_ts = make_idesc(1, 128, 64, false, true);
  const uint32_t idesc_du_ss = make_idesc(1, 128, 64, true, true);
  const uint32_t idesc_s_ss = make_idesc(1, 128, 128, true, true);
  const uint32_t idesc_s_ts = make_idesc(1, 128, 128, false, false);
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

  for (int it = 0; it < nck; ++it) {
    const int ch = nck - 1 - it;
    const int st = it & 1;
    uint8_t* const b = sm + st * kBStage;
    const int n = min(kC, len - ch * kC);
    const long long rec = rec_of(ch);

    // the previous step's image stores have read their staging tiles before they are rewritten
    if (tid == 0) bulk_wait_read_all();
    if (!(ok = block_wait(&bar_ld[st], (it >> 1) & 1))) break;
    inflight[st] = -1;
    if (tid < 256) s_vec[tid] = reinterpret_cast<const float*>(b + B_V)[tid];
    if (n < kC) {
      zero_rows(b + B_DO, n, tid);
      fence_async_smem();
    }
    __syncthreads();

    // ---- dU^T = dS'^T K^ + dO^T (rq M_raw)  (the rk column factor is applied below)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kt = smem_u32(b + B_KT), ms = smem_u32(b + B_M), dos = smem_u32(b + B_DO);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_ts(tm + BT_DU, tm + BT_SA + 8 * s, mn_desc(kt, 8192, s), idesc_du_ts, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tm + BT_DU, mn_desc(dos, 8192, s), mn_desc(ms, 8192, s), idesc_du_ss, 1);
      mma_commit(&bar_mma);
    }
    // meanwhile: dS'^T diag(e^{G_C}) in place
    {
      float S[32];
      tmem_ld32(tl + BT_S + 32 * wg, S);
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] *= s_vec[32 * wg + i];
      tmem_st32(tl + BT_S + 32 * wg, S);
    }
    if (!(ok = mma_wait())) break;
    tc_fence_after();
    // ---- dU^T (rk column factor) -> bf16 A operand and the dU^T record: thread
    //      (j = ln, tokens 16 wg .. + 15)
    {
      float v16[16];
      tmem_ld16(tl + BT_DU + 16 * wg, v16);
      uint32_t up[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        up[i] = pack_bf16(v16[2 * i] * s_vec[128 + 16 * wg + 2 * i],
                          v16[2 * i + 1] * s_vec[128 + 16 * wg + 2 * i + 1]);
      tmem_st8(tl + BT_UA + 8 * wg, up);
      uint8_t* row = sm + B_SDU + (ln >> 3) * 1024 + (ln & 7) * 128;
      *reinterpret_cast<uint4*>(row + (((2 * wg) ^ (ln & 7)) << 4)) =
          make_uint4(up[0], up[1], up[2], up[3]);
      *reinterpret_cast<uint4*>(row + (((2 * wg + 1) ^ (ln & 7)) << 4)) =
          make_uint4(up[4], up[5], up[6], up[7]);
      fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();

    // ---- dS^T += dO^T Q~ + dU^T (-W)
    if (tid == 0) {
      tma_store_2d(&map_dut, sm + B_SDU, 0, (int)(rec * 128));
      bulk_commit();
      tc_fence_after();
      const uint32_t qs = smem_u32(b + B_Q), wsm = smem_u32(b + B_W), dos = smem_u32(b + B_DO);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tm + BT_S, mn_desc(dos, 8192, s), mn_desc(qs, 8192, s), idesc_s_ss, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ts(tm + BT_S, tm + BT_UA + 8 * s, sw128_kdesc<2>(wsm, 128, s), idesc_s_ts, 1);
      mma_commit(&bar_mma);
      // the refill's bytes land on the stage's next phase (its current phase completed at
      // the top of this step)
      if (it + 2 < nck) mbar_arrive_expect_tx(&bar_ld[st], kBStageTx);
    }
    if (!(ok = mma_wait())) break;
    tc_fence_after();
    if (it + 2 < nck) issue_load_spread(it + 2, st);
    inflight[st] = (it + 2 < nck) ? it + 2 : -1;
    // ---- bf16 copy of dS (= dS' of the previous chunk) and its record
    {
      float S[32];
      tmem_ld32(tl + BT_S + 32 * wg, S);
      uint32_t sp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sp[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
      tmem_st16(tl + BT_SA + 16 * wg, sp);
      if (ch > 0) {  // staged for a TMA store
        uint8_t* row = sm + B_SDS + (wg >> 1) * 16384 + (ln >> 3) * 1024 + (ln & 7) * 128;
#pragma unroll
        for (int p = 0; p < 4; ++p)
          *reinterpret_cast<uint4*>(row + (((4 * (wg & 1) + p) ^ (ln & 7)) << 4)) =
              make_uint4(sp[4 * p], sp[4 * p + 1], sp[4 * p + 2], sp[4 * p + 3]);
        fence_async_smem();
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ch > 0) {
      const int row = (int)(rec_of(ch - 1) * 128);
      tma_store_2d(&map_ds, sm + B_SDS, 0, row);
      tma_store_2d(&map_ds, sm + B_SDS + 16384, 64, row);
      bulk_commit();
    }
  }

  if (!ok) {
    if (tid == 0) {
      atomicOr(&g_bwd_error, 4u);
      for (int st = 0; st < 2; ++st)
        if (inflight[st] >= 0) mbar_wait(&bar_ld[st], (inflight[st] >> 1) & 1, 1000000000ull);
    }
    mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  } else if (o.d_initial) {
    tc_fence_after();
    float S[32];
    tmem_ld32(tl + BT_S + 32 * wg, S);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * wg + i;
      o.d_initial[state_off + (long long)c * kD + ln] = S[i];
    }
  }
  if (tid == 0) bulk_wait_all();  // the image stores are done before the CTA leaves
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kBTmemCols);
}

// ------------------------------------------------------------ per-chunk products

constexpr int kKThreads = 512;
// Dynamic shared memory (1024-aligned offsets).  Loaded at the start:
constexpr int K_DUT = 0;        // dU^T [128 j][64 r]; dV^T once lam is read
constexpr int K_NN = 16384;     // N [64][64]
constexpr int K_UT = 24576;     // U^T [128 j][64 s]
constexpr int K_DO = 40960;     // d_out [64 r][128 j] (two boxes, 8192 apart)
constexpr int K_S0 = 57344;     // S^T [128 j][128 c] (two boxes, 16384 apart)
constexpr int K_DS = 90112;     // dS'^T [128 j][128 c]
constexpr int K_RQ = 122880;    // raw q [64 tok][128] bf16 (two boxes, 8192 apart)
constexpr int K_RK = 139264;    // raw k
constexpr int K_RG = 155648;    // raw g fp32 [4 quarters][64 tok][32] (8192 apart)
constexpr int K_END = 188416;
// Built later, in tiles whose readers are done:
constexpr int K_XL = K_DS;      // Xl [128 rows][128 c] (two boxes, 16384 apart): after dKd^T
constexpr int K_KB = 0;         // Kb [160 rows][128 c] (two boxes, 20480 apart): after dA, dM
constexpr int K_D1 = K_DO;      // dD1 [128 rows][192] (three boxes, 16384 apart): after dA, dM
// The epilogue reads only the raw tiles and Tensor Memory, so the next record's loaded tiles
// (everything below K_RQ) go out once the last MMA group is done, and its raw tiles once the
// epilogue's first half has read them.
static_assert(K_KB + 2 * 20480 <= K_D1 && K_D1 + 3 * 16384 <= K_XL, "late tiles overlap");
static_assert(K_XL + 32768 <= K_RQ, "late tiles overlap the raw tiles");
static_assert(K_DO + 3 * 8192 <= K_END, "rows 64..127 of the d_out A operand read in bounds");
static_assert(K_DUT + 2 * 16384 <= K_DO, "second M block of the dV^T A operand in bounds");
constexpr uint32_t kKLoadTx = 16384 + 8192 + 16384 + 16384 + 32768 + 32768;
constexpr uint32_t kKRawTx = 16384 + 16384 + 32768;
constexpr size_t kKSmem = K_END + 1024;

// Tensor Memory (512 columns, one CTA per SM).
constexpr uint32_t KT_P1 = 0;    // dQ~^T [c][r]
constexpr uint32_t KT_P3 = 64;   // dKd^T [c][s]
constexpr uint32_t KT_P2 = 128;  // (dV S^T)^T [c][r] = -dK~^T
constexpr uint32_t KT_L = 192;   // lam^T [j][r]
constexpr uint32_t KT_DA = 256;  // dV U^T [r][s] (lanes 0..63)
constexpr uint32_t KT_DM = 320;  // dO U^T [r][s] (lanes 0..63)
constexpr uint32_t KT_P6 = 192;  // dXl^T [c][row], 128 (after lam, dA, dM are read)
constexpr uint32_t KT_P7 = 320;  // dKb^T [c][col], 160
constexpr uint32_t kKTmemCols = 512;
// Between the epilogue's halves each thread keeps its 16 tokens' dq^, dk^, q^, k^ and gate
// argument in Tensor Memory cells that only it reads, once it has read them: the columns
// 16 R .. 16 R + 15 of P1, P2, P3 and of both halves of P6, in its own lane.
constexpr uint32_t KT_KEEP_AQ = KT_P1, KT_KEEP_DKH = KT_P2, KT_KEEP_QH = KT_P3,
                   KT_KEEP_KH = KT_P6, KT_KEEP_X = KT_P6 + 64;

// Store 8 consecutive 32-bit columns of this thread's lane; completion is waited for by
// tmem_wait_st.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// first Kb row (and dD1 column) of the block that refers the earlier tokens to P_g
__device__ __forceinline__ int kb_base(int g) { return g == 1 ? 64 : g == 2 ? 80 : 112; }

__global__ void __launch_bounds__(kKThreads, 1)
    bwd_chunk_kernel(const __grid_constant__ CUtensorMap map_dut,
                     const __grid_constant__ CUtensorMap map_n,
                     const __grid_constant__ CUtensorMap map_ut,
                     const __grid_constant__ CUtensorMap map_do,
                     const __grid_constant__ CUtensorMap map_s0,
                     const __grid_constant__ CUtensorMap map_ds,
                     const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_g, const ChunkArgs a,
                     const BwdWs bw, const BwdOut o) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  __shared__ uint64_t bar_ld, bar_raw, bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_wait_ok[4];
  __shared__ __align__(16) float s_half[8][kD];  // gate total of each half sub-chunk
  __shared__ __align__(16) float s_beta[kC], s_rk[kC], s_rq[kC];
  __shared__ __align__(16) float s_lu[4][kC];
  __shared__ __align__(16) float s_sdot[4][kD];
  __shared__ __align__(16) float s_dgs[8][kD];  // sum of dG over each half sub-chunk
  __shared__ __align__(16) float s_dgc[4][kD];
  __shared__ __align__(16) float s_qd[4][kC], s_kd[4][kC];
  __shared__ __align__(16) float4 s_tf[kC];  // per token: rq, q^.dq^ / scale^2, rk, k^.dk^
  __shared__ __align__(16) float s_ddb[4][kD];
  __shared__ float s_dal[16];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int R = tid >> 7;      // warpgroup: a quarter of the work in the split phases
  const int c = tid & 127;     // channel (Tensor Memory lane)
  // The token-wise phases give each warpgroup two half sub-chunks ("units": 8 tokens of
  // sub-chunk uR[u], half uh), paired so that every warpgroup carries the same off-diagonal
  // work (sub-chunk r has 3 - r off-diagonal blocks): warpgroups 0, 1 take sub-chunks 0 and
  // 3, warpgroups 2, 3 sub-chunks 1 and 2, each one half of both.
  const int uh = R & 1;
  const int uR[2] = {R < 2 ? 0 : 1, R < 2 ? 3 : 2};
  const int ut0[2] = {16 * uR[0] + 8 * uh, 16 * uR[1] + 8 * uh};  // first token of each unit
  const int sp = warp & 3;     // Tensor Memory sub-partition
  const int H = a.H;
  if (warp == 0) {
    tmem_alloc(&s_tmem, kKTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_raw, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t tl = tm + (uint32_t(32 * sp) << 16);
  uint32_t mma_phase = 0;
  uint32_t wait_calls = 0;
  auto block_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t slot_w = wait_calls++ & 3;
    if (tid == 0) s_wait_ok[slot_w] = mbar_wait(bar, parity) ? 1 : 0;
    __syncthreads();
    return s_wait_ok[slot_w] != 0;
  };
  // Loads go out from thread 0: raw_armed / ld_armed count the phases it has armed on
  // bar_raw / bar_ld, raw_seen / ld_seen the phases the block has waited for.  Every record
  // takes one phase of each, so the record's phase is the count of records processed.
  uint32_t raw_armed = 0, ld_armed = 0, raw_seen = 0, ld_seen = 0;
  long long early = -1;  // thread 0: the record whose loads went out during the previous one
  // record -> first token and token count; false for the slots past the last chunk of packed
  // sequences (their count is an upper bound), which come after every live slot
  auto locate = [&](long long r, long long& t0, int& cnt) -> bool {
    const long long slot = r / H;
    int seq, jc;
    if (a.cu_seqlens) {
      const int N = a.B;
      if (slot >= bw.f.coff[N]) return false;
      int lo = 0, hi = N;  // coff[lo] <= slot < coff[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (bw.f.coff[mid] <= slot) lo = mid; else hi = mid;
      }
      seq = lo;
      jc = (int)(slot - bw.f.coff[lo]);
    } else {
      seq = (int)(slot / bw.f.nck_fixed);
      jc = (int)(slot % bw.f.nck_fixed);
    }
    long long bos;
    int len;
    seq_range(a, seq, bos, len);
    t0 = bos + (long long)jc * kC;
    cnt = min(kC, len - jc * kC);
    return true;
  };
  // the chunk's raw q, k, g (thread 0)
  auto issue_raw = [&](long long r, long long t0) {
    const int hr = (int)(r % H);
    mbar_arrive_expect_tx(&bar_raw, kKRawTx);
    tma_load_3d(sm + K_RQ, &map_q, &bar_raw, 0, hr, (int)t0);
    tma_load_3d(sm + K_RQ + 8192, &map_q, &bar_raw, 64, hr, (int)t0);
    tma_load_3d(sm + K_RK, &map_k, &bar_raw, 0, hr, (int)t0);
    tma_load_3d(sm + K_RK + 8192, &map_k, &bar_raw, 64, hr, (int)t0);
#pragma unroll
    for (int qt = 0; qt < 4; ++qt)
      tma_load_3d(sm + K_RG + qt * 8192, &map_g, &bar_raw, 32 * qt, hr, (int)t0);
    ++raw_armed;
  };
  // the record's tiles, states and d_out (thread 0)
  auto issue_ld = [&](long long r, long long t0) {
    const int hr = (int)(r % H);
    mbar_arrive_expect_tx(&bar_ld, kKLoadTx);
    tma_load_2d(sm + K_DUT, &map_dut, &bar_ld, 0, (int)(r * 128));
    tma_load_2d(sm + K_NN, &map_n, &bar_ld, 0, (int)(r * 64));
    tma_load_2d(sm + K_UT, &map_ut, &bar_ld, 0, (int)(r * 128));
    tma_load_3d(sm + K_DO, &map_do, &bar_ld, 0, hr, (int)t0);
    tma_load_3d(sm + K_DO + 8192, &map_do, &bar_ld, 64, hr, (int)t0);
    tma_load_2d(sm + K_S0, &map_s0, &bar_ld, 0, (int)(r * 128));
    tma_load_2d(sm + K_S0 + 16384, &map_s0, &bar_ld, 64, (int)(r * 128));
    tma_load_2d(sm + K_DS, &map_ds, &bar_ld, 0, (int)(r * 128));
    tma_load_2d(sm + K_DS + 16384, &map_ds, &bar_ld, 64, (int)(r * 128));
    ++ld_armed;
  };
  // Persistent: the CTA (one per SM) walks records blockIdx.x, + gridDim.x, ...; the TMEM
  // allocation and the barriers are set up once, and each next record's loads go out while
  // the current record's epilogue runs.
  for (long long rec = blockIdx.x; rec < bw.f.recs; rec += gridDim.x) {
  const int h = (int)(rec % H);
  long long tok0;
  int n;
  if (!locate(rec, tok0, n)) continue;  // uniform over the CTA
  if (tid == 0 && early != rec) {
    issue_raw(rec, tok0);
    issue_ld(rec, tok0);
  }
  if (tid < kC) {
    s_beta[tid] = (tid < n) ? sigmoidf_(a.beta_logits[(tok0 + tid) * H + h]) : 0.f;
    s_rk[tid] = bw.f.vec[rec * 256 + 128 + tid];
    s_rq[tid] = bw.f.vec[rec * 256 + 192 + tid];
  }
  const float ea = __expf(a.a_log[h]);
  const float db = a.dt_bias[c * H + h];
  // the gate in log2 units: gamma log2 e = lb2 / (1 + 2^(nea2 (g + dt_bias))); every
  // cumulative gate below (loc, P, PR, GC, the half totals) is in log2 units, so each
  // factor e^{G} is one 2^x
  const float lb2 = a.lower_bound * kLog2E, nea2 = -ea * kLog2E;
  __syncthreads();
  float loc[16], P[4], fg[2][4], GC, PR[2];

  // element (t, c) of the staged tiles
  const uint8_t* const rq_t = sm + K_RQ;
  const uint8_t* const rk_t = sm + K_RK;
  const float* const rg_t = reinterpret_cast<const float*>(sm + K_RG) + (c >> 5) * 2048 + (c & 31);
  auto raw_q = [&](int t) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(rq_t + sw_off(t, c, 8192)));
  };
  auto raw_k = [&](int t) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(rk_t + sw_off(t, c, 8192)));
  };
  auto row_of = [&](int t) -> long long { return (tok0 + t) * H + h; };

  // ---- gates: the prefix inside each of this thread's units (completed to G_t - P_R once
  //      the first halves' totals are known)
  if (!block_wait(&bar_raw, raw_seen & 1)) goto fail;
  ++raw_seen;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = ut0[u] + i;
      float gm = 0.f;
      if (t < n) gm = lb2 * fast_rcp(1.f + fast_exp2(nea2 * (rg_t[t * 32] + db)));
      run += gm;
      loc[8 * u + i] = run;
    }
    s_half[2 * uR[u] + uh][c] = run;
  }

  // ---- loaded tiles: clear d_out rows past the chunk, S . dS' per channel (quarter of j)
  if (!block_wait(&bar_ld, ld_seen & 1)) goto fail;
  ++ld_seen;
  if (uh) {  // second halves: add the first half's total
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float first = s_half[2 * uR[u]][c];
#pragma unroll
      for (int i = 0; i < 8; ++i) loc[8 * u + i] += first;
    }
  }
  if (n < kC) zero_rows(sm + K_DO, n, tid);
  {
    float acc = 0.f;
#pragma unroll 8
    for (int jj = 0; jj < 32; ++jj) {
      const int j = 32 * R + jj;
      const uint32_t off = sw_off(j, c, 16384);
      acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + K_S0 + off)) *
             __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + K_DS + off));
    }
    s_sdot[R][c] = acc;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- lam^T = dU^T N;  dQ~^T = S^T-as-MN x d_out;  dKd^T = dS'^T-as-MN x U^T-as-MN
  if (tid == 0) {
    tc_fence_after();
    const uint32_t dut = smem_u32(sm + K_DUT), nn = smem_u32(sm + K_NN), ut = smem_u32(sm + K_UT),
                   dos = smem_u32(sm + K_DO), s0 = smem_u32(sm + K_S0), ds = smem_u32(sm + K_DS);
    const uint32_t id_l = make_idesc(1, 128, 64, false, true);
    const uint32_t id_p1 = make_idesc(1, 128, 64, true, false);
    const uint32_t id_p3 = make_idesc(1, 128, 64, true, true);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      mma_ss(tm + KT_L, sw128_kdesc<2>(dut, 128, s), mn_desc(nn, 8192, s), id_l, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      mma_ss(tm + KT_P1, mn_desc(s0, 16384, s), sw128_kdesc<2>(dos, 64, s), id_p1, s > 0);
      mma_ss(tm + KT_P3, mn_desc(ds, 16384, s), mn_desc(ut, 8192, s), id_p3, s > 0);
    }
    mma_commit(&bar_mma);
  }
  // meanwhile: the sub-chunk reference points, and each unit's P_R and e^{P_g - P_R}
  P[0] = 0.f;
#pragma unroll
  for (int r = 1; r < 4; ++r) P[r] = P[r - 1] + (s_half[2 * r - 2][c] + s_half[2 * r - 1][c]);
  GC = P[3] + (s_half[6][c] + s_half[7][c]);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    PR[u] = P[0];
#pragma unroll
    for (int r = 1; r < 4; ++r) PR[u] = (uR[u] == r) ? P[r] : PR[u];
#pragma unroll
    for (int g = 0; g < 4; ++g) fg[u][g] = (g > uR[u]) ? fast_exp2(P[g] - PR[u]) : 0.f;
  }
  if (!block_wait(&bar_mma, mma_phase++ & 1)) goto fail;
  tc_fence_after();

  // ---- lam -> dV (output and dV^T operand), lam . u per token
  {
    const int j = c;
    float lam[16];
    tmem_ld16(tl + KT_L + 16 * R, lam);
    const uint32_t rowb = uint32_t(j >> 3) * 1024u + uint32_t(j & 7) * 128u;
    const uint32_t ca = uint32_t(2 * R) ^ uint32_t(j & 7), cb = uint32_t(2 * R + 1) ^ uint32_t(j & 7);
    const uint4 ua = *reinterpret_cast<const uint4*>(sm + K_UT + rowb + (ca << 4));
    const uint4 ub = *reinterpret_cast<const uint4*>(sm + K_UT + rowb + (cb << 4));
    const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
    uint32_t dw[8];
    float lu0[8], lu1[8];
    __nv_bfloat16* const dv_p = o.dv + row_of(16 * R) * kD + j;  // token 16 R; H * 128 apart
    const long long tstride = (long long)H * kD;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int t0 = 16 * R + 2 * p;
      const float v0 = s_beta[t0] * lam[2 * p], v1 = s_beta[t0 + 1] * lam[2 * p + 1];
      dw[p] = pack_bf16(v0, v1);
      if (t0 < n) dv_p[(2 * p) * tstride] = __float2bfloat16_rn(v0);
      if (t0 + 1 < n) dv_p[(2 * p + 1) * tstride] = __float2bfloat16_rn(v1);
      const float l0 = lam[2 * p] * bf16_lo(uw[p]), l1 = lam[2 * p + 1] * bf16_hi(uw[p]);
      if (p < 4) { lu0[2 * p] = l0; lu0[2 * p + 1] = l1; }
      else { lu1[2 * (p - 4)] = l0; lu1[2 * (p - 4) + 1] = l1; }
    }
    *reinterpret_cast<uint4*>(sm + K_DUT + rowb + (ca << 4)) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
    *reinterpret_cast<uint4*>(sm + K_DUT + rowb + (cb << 4)) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
    int tq;
    const float s0v = reduce_scatter8(lu0, lane, tq);
    const float s1v = reduce_scatter8(lu1, lane, tq);
    if ((lane & 3) == 0) {
      s_lu[sp][16 * R + tq] = s0v;
      s_lu[sp][16 * R + 8 + tq] = s1v;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- -dK~^T (as dV S^T), dV U^T and dO U^T (rows 64..127 of the last two A operands
  //      are unused)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t dvt = smem_u32(sm + K_DUT), ut = smem_u32(sm + K_UT),
                   dos = smem_u32(sm + K_DO), s0 = smem_u32(sm + K_S0);
    const uint32_t id_p2 = make_idesc(1, 128, 64, true, true);
    const uint32_t id_dm = make_idesc(1, 128, 64, false, true);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      mma_ss(tm + KT_P2, mn_desc(s0, 16384, s), mn_desc(dvt, 8192, s), id_p2, s > 0);
      mma_ss(tm + KT_DA, mn_desc(dvt, 16384, s), mn_desc(ut, 8192, s), id_p2, s > 0);
      mma_ss(tm + KT_DM, sw128_kdesc<2>(dos, 64, s), mn_desc(ut, 8192, s), id_dm, s > 0);
    }
    mma_commit(&bar_mma);
  }
  // meanwhile: Xl rows t (k^ e^{G_t - P_R}) and 64 + t (q^ e^{G_t - P_R}) into the dS' tile,
  // whose readers (dKd^T and the S . dS' sums) are done
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int t = ut0[i >> 3] + (i & 7);
    const bool live = t < n;
    const float kh = live ? raw_k(t) * s_rk[t] : 0.f;
    const float qh = live ? raw_q(t) * s_rq[t] : 0.f;
    const float e = fast_exp2(loc[i]);
    *reinterpret_cast<__nv_bfloat16*>(sm + K_XL + sw_off(t, c, 16384)) = __float2bfloat16_rn(kh * e);
    *reinterpret_cast<__nv_bfloat16*>(sm + K_XL + sw_off(64 + t, c, 16384)) =
        __float2bfloat16_rn(qh * e);
  }
  if (!block_wait(&bar_mma, mma_phase++ & 1)) goto fail;
  tc_fence_after();

  // ---- dD1 = [dA; dM] in the column layout of the Kb rows (over d_out and S); Kb rows t
  //      (k^ e^{P_R - G_t}) and base_g + t (k^ e^{P_g - G_t}) over dU^T, N and U^T;
  //      dbeta_logits
  if (sp < 2) {
    // row r of dA and dM; the columns of this thread's two units (8 tokens s of sub-chunk
    // uR[u]), placed in the diagonal block and the off-diagonal blocks that refer them
    const int r = 32 * sp + lane, Rr = r >> 4;
    const bool live = r < n;
    auto put = [&](int row, int col0, bool on, uint4 w) {
      *reinterpret_cast<uint4*>(sm + K_D1 + sw_off(row, col0, 16384)) =
          on ? w : make_uint4(0, 0, 0, 0);
    };
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float da[8], dm[8];
      tmem_ld8(tl + KT_DA + ut0[u], da);
      tmem_ld8(tl + KT_DM + ut0[u], dm);
      uint32_t pa[4], pm[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int s0 = ut0[u] + 2 * p;
        pa[p] = pack_bf16((live && s0 < r) ? -da[2 * p] : 0.f, (live && s0 + 1 < r) ? -da[2 * p + 1] : 0.f);
        pm[p] = pack_bf16((live && s0 <= r) ? dm[2 * p] : 0.f, (live && s0 + 1 <= r) ? dm[2 * p + 1] : 0.f);
      }
      const uint4 wa = make_uint4(pa[0], pa[1], pa[2], pa[3]);
      const uint4 wm = make_uint4(pm[0], pm[1], pm[2], pm[3]);
      put(r, ut0[u], uR[u] == Rr, wa);
      put(64 + r, ut0[u], uR[u] == Rr, wm);
#pragma unroll
      for (int g = 1; g < 4; ++g)
        if (g > uR[u]) {
          put(r, kb_base(g) + ut0[u], Rr == g, wa);
          put(64 + r, kb_base(g) + ut0[u], Rr == g, wm);
        }
    }
  } else if (tid >= 64 && tid < 64 + kC) {  // warps 2 and 3 (sub-partitions 2, 3)
    const int t = tid - 64;
    if (t < n)
      o.dbeta_logits[row_of(t)] =
          (1.f - s_beta[t]) * (s_lu[0][t] + s_lu[1][t] + s_lu[2][t] + s_lu[3][t]);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int u = i >> 3, t = ut0[u] + (i & 7);
    const float kd = (t < n) ? raw_k(t) * s_rk[t] * fast_exp2(-loc[i]) : 0.f;
    *reinterpret_cast<__nv_bfloat16*>(sm + K_KB + sw_off(t, c, 20480)) = __float2bfloat16_rn(kd);
#pragma unroll
    for (int g = 1; g < 4; ++g)
      if (g > uR[u])
        *reinterpret_cast<__nv_bfloat16*>(sm + K_KB + sw_off(kb_base(g) + t, c, 20480)) =
            __float2bfloat16_rn(kd * fg[u][g]);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- dXl^T = Kb-as-MN x dD1 (K = 160 Kb rows), dKb^T = Xl-as-MN x dD1-as-MN
  if (tid == 0) {
    tc_fence_after();
    const uint32_t kb = smem_u32(sm + K_KB), xl = smem_u32(sm + K_XL), d1 = smem_u32(sm + K_D1);
    const uint32_t id_p6 = make_idesc(1, 128, 128, true, false);
    const uint32_t id_p7 = make_idesc(1, 128, 160, true, true);
#pragma unroll
    for (int s = 0; s < 10; ++s)
      mma_ss(tm + KT_P6, mn_desc(kb, 20480, s), sw128_kdesc<2>(d1, 128, s), id_p6, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      mma_ss(tm + KT_P7, mn_desc(xl, 16384, s), mn_desc(d1, 16384, s), id_p7, s > 0);
    mma_commit(&bar_mma);
  }
  if (!block_wait(&bar_mma, mma_phase++ & 1)) goto fail;
  tc_fence_after();
  // the next record's tiles, states and d_out: nothing below K_RQ is read from here on
  if (tid == 0 && rec + gridDim.x < bw.f.recs) {
    long long nt0;
    int ncnt;
    if (locate(rec + gridDim.x, nt0, ncnt)) issue_ld(rec + gridDim.x, nt0);
  }

  // ---- epilogue: per (channel c, token t of each of this thread's units)
  {
    float dG[16];
    float2 dgc2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // (unit hh: sub-chunk uR[hh])
      const int cb = ut0[hh];  // first token of this unit
      const float eP = fast_exp2(PR[hh]), eCP = fast_exp2(GC - PR[hh]);
      // token pairs (t, t + 1) ride Blackwell's two-lane fp32 instructions; every pair
      // operation rounds exactly as the two scalar ones would
      const float2 ePv = make_float2(eP, eP), neP = make_float2(-eP, -eP);
      const float2 eCPv = make_float2(eCP, eCP);
      float2 E[4], EI[4], KH[4], QH[4], AQ2[4], POS[4], NEG[4], DG[4], T[4];
      float t8[8];
      auto load_t = [&](uint32_t col) {
        tmem_ld8(tl + col, t8);
#pragma unroll
        for (int p = 0; p < 4; ++p) T[p] = make_float2(t8[2 * p], t8[2 * p + 1]);
      };
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int t = cb + 2 * p;
        const float l0 = loc[8 * hh + 2 * p], l1 = loc[8 * hh + 2 * p + 1];
        E[p] = make_float2(fast_exp2(l0), fast_exp2(l1));
        EI[p] = make_float2(fast_exp2(-l0), fast_exp2(-l1));
        const float2 rk2 = *reinterpret_cast<const float2*>(&s_rk[t]);
        const float2 rq2 = *reinterpret_cast<const float2*>(&s_rq[t]);
        KH[p] = __fmul2_rn(make_float2(raw_k(t), raw_k(t + 1)), rk2);
        QH[p] = __fmul2_rn(make_float2(raw_q(t), raw_q(t + 1)), rq2);
        if (t >= n) { KH[p].x = 0.f; QH[p].x = 0.f; }
        if (t + 1 >= n) { KH[p].y = 0.f; QH[p].y = 0.f; }
      }
      // dq^, dk^ (exact gate factors) and dG; each Xl / Kb term of dG is weighted by the bf16
      // operand value the product used, so that the +G and -G terms of a pair (r, s) of the
      // gate-scaled products cancel as they do in exact arithmetic
      load_t(KT_P1 + cb);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        AQ2[p] = __fmul2_rn(__fmul2_rn(ePv, E[p]), T[p]);
        DG[p] = __fmul2_rn(QH[p], AQ2[p]);
      }
      load_t(KT_P6 + 64 + cb);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        AQ2[p] = __ffma2_rn(E[p], T[p], AQ2[p]);
        DG[p] = __ffma2_rn(bf16_round2(__fmul2_rn(QH[p], E[p])), T[p], DG[p]);
      }
      load_t(KT_P2 + cb);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        POS[p] = __fmul2_rn(__fmul2_rn(neP, E[p]), T[p]);
        DG[p] = __ffma2_rn(KH[p], POS[p], DG[p]);
      }
      load_t(KT_P6 + cb);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        POS[p] = __ffma2_rn(E[p], T[p], POS[p]);
        DG[p] = __ffma2_rn(bf16_round2(__fmul2_rn(KH[p], E[p])), T[p], DG[p]);
      }
      load_t(KT_P3 + cb);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        NEG[p] = __fmul2_rn(__fmul2_rn(eCPv, EI[p]), T[p]);
        dgc2 = __ffma2_rn(KH[p], NEG[p], dgc2);
        DG[p] = __ffma2_rn(make_float2(-KH[p].x, -KH[p].y), NEG[p], DG[p]);
      }
      // with -k (the bf16 rounding is symmetric: round(-x) = -round(x))
      float2 NKD[4];
      load_t(KT_P7 + cb);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        NKD[p] = __fmul2_rn(make_float2(-KH[p].x, -KH[p].y), EI[p]);
        NEG[p] = __ffma2_rn(EI[p], T[p], NEG[p]);
        DG[p] = __ffma2_rn(bf16_round2(NKD[p]), T[p], DG[p]);
      }
#pragma unroll
      for (int g = 1; g < 4; ++g)
        if (g > uR[hh]) {
          const float2 fgv = make_float2(fg[hh][g], fg[hh][g]);
          load_t(KT_P7 + kb_base(g) + cb);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            NEG[p] = __ffma2_rn(__fmul2_rn(EI[p], fgv), T[p], NEG[p]);
            DG[p] = __ffma2_rn(bf16_round2(__fmul2_rn(NKD[p], fgv)), T[p], DG[p]);
          }
        }
      float qd[8], kd[8], keep[8];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 dkh = __fadd2_rn(POS[p], NEG[p]);
        const int i = 2 * p;
        dG[8 * hh + i] = DG[p].x;
        dG[8 * hh + i + 1] = DG[p].y;
        const float2 q2 = __fmul2_rn(QH[p], AQ2[p]), k2 = __fmul2_rn(KH[p], dkh);
        qd[i] = q2.x;
        qd[i + 1] = q2.y;
        kd[i] = k2.x;
        kd[i + 1] = k2.y;
        keep[i] = dkh.x;
        keep[i + 1] = dkh.y;
      }
      // kept for the second half: dq^, dk^, q^, k^ and the gate argument of these tokens
      tmem_st8(tl + KT_KEEP_DKH + cb, keep);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        keep[2 * p] = AQ2[p].x;
        keep[2 * p + 1] = AQ2[p].y;
      }
      tmem_st8(tl + KT_KEEP_AQ + cb, keep);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        keep[2 * p] = QH[p].x;
        keep[2 * p + 1] = QH[p].y;
      }
      tmem_st8(tl + KT_KEEP_QH + cb, keep);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        keep[2 * p] = KH[p].x;
        keep[2 * p + 1] = KH[p].y;
      }
      tmem_st8(tl + KT_KEEP_KH + cb, keep);
#pragma unroll
      for (int i = 0; i < 8; ++i) keep[i] = ea * (rg_t[(cb + i) * 32] + db);
      tmem_st8(tl + KT_KEEP_X + cb, keep);
      int tq;
      const float qs = reduce_scatter8(qd, lane, tq);
      const float ks = reduce_scatter8(kd, lane, tq);
      if ((lane & 3) == 0) {
        s_qd[sp][cb + tq] = qs;
        s_kd[sp][cb + tq] = ks;
      }
    }
    const float dgc = dgc2.x + dgc2.y;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float sg = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) sg += dG[8 * u + i];
      s_dgs[2 * uR[u] + uh][c] = sg;
    }
    s_dgc[R][c] = dgc;
    tmem_wait_st();
    __syncthreads();
    // the next record's raw q, k, g: the raw tiles are not read from here on
    if (tid == 0 && rec + gridDim.x < bw.f.recs) {
      long long nt0;
      int ncnt;
      if (locate(rec + gridDim.x, nt0, ncnt)) {
        issue_raw(rec + gridDim.x, nt0);
        early = rec + gridDim.x;
      }
    }
    // dgamma_t = sum_{r >= t} dG_r + dG_C
    const float dGC = s_dgc[0][c] + s_dgc[1][c] + s_dgc[2][c] + s_dgc[3][c] +
                      fast_exp2(GC) * (s_sdot[0][c] + s_sdot[1][c] + s_sdot[2][c] + s_sdot[3][c]);
    // per token: the sums of q^ . dq^ and k^ . dk^ over the four warps that hold its
    // channels, beside the norms' factors, for one 16-byte read per token below
    const float inv_s2 = 1.f / (a.scale * a.scale);
    if (tid < kC) {
      const float qs = s_qd[0][tid] + s_qd[1][tid] + s_qd[2][tid] + s_qd[3][tid];
      const float ks = s_kd[0][tid] + s_kd[1][tid] + s_kd[2][tid] + s_kd[3][tid];
      s_tf[tid] = make_float4(s_rq[tid], qs * inv_s2, s_rk[tid], ks);
    }
    __syncthreads();
    // dx_t = carry_t lb sg (1 - sg) with sg = sigmoid(x_t): sw sums carry sg (1 - sg) and swx
    // the same times x_t, so that ddt_bias = lb ea sw and da_log = lb swx
    float sw = 0.f, swx = 0.f;
    const float lb = a.lower_bound, lbea = a.lower_bound * ea;
    const long long tstride = (long long)H * kD;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
    // the sum of dG over every later half sub-chunk, then this unit's tokens backwards
    float carry = dGC;
#pragma unroll
    for (int x = 1; x < 8; ++x)
      if (x > 2 * uR[u] + uh) carry += s_dgs[x][c];
    // this thread's element of the unit's first token in each [B, T, H, 128] output; tokens
    // H * 128 apart
    const long long base = row_of(ut0[u]) * kD + c;
    float* const dg_p = o.dg + base;
    __nv_bfloat16* const dq_p = o.dq + base;
    __nv_bfloat16* const dk_p = o.dk + base;
#pragma unroll
    for (int qq = 1; qq >= 0; --qq) {
      const int cb = ut0[u] + 4 * qq;
      float aq[4], dkh[4], qh[4], kh[4], xg[4];
      tmem_ld4(tl + KT_KEEP_AQ + cb, aq);
      tmem_ld4(tl + KT_KEEP_DKH + cb, dkh);
      tmem_ld4(tl + KT_KEEP_QH + cb, qh);
      tmem_ld4(tl + KT_KEEP_KH + cb, kh);
      tmem_ld4(tl + KT_KEEP_X + cb, xg);
#pragma unroll
      for (int i = 3; i >= 0; --i) {
        carry += dG[8 * u + 4 * qq + i];
        const int t = cb + i;
        if (t < n) {
          // gate: gamma = lb sigmoid(x), x = e^{a_log} (g + dt_bias)
          const float x = xg[i];
          const float sg = fast_rcp(1.f + fast_exp(-x));
          const float cw = carry * fmaf(-sg, sg, sg);  // carry sg (1 - sg)
          dg_p[(4 * qq + i) * tstride] = cw * lbea;
          sw += cw;
          swx = fmaf(cw, x, swx);
          // L2 norms: q^ = rq q with rq = scale / |q|, k^ = rk k:
          //   dq = rq (dq^ - q^ (q^ . dq^) / scale^2),  dk = rk (dk^ - k^ (k^ . dk^))
          const float4 f = s_tf[t];
          dq_p[(4 * qq + i) * tstride] = __float2bfloat16_rn(f.x * fmaf(-qh[i], f.y, aq[i]));
          dk_p[(4 * qq + i) * tstride] = __float2bfloat16_rn(f.z * fmaf(-kh[i], f.w, dkh[i]));
        }
      }
    }
    }  // units
    s_ddb[R][c] = lbea * sw;
    const float dal = warp_sum(lb * swx);
    if (lane == 0) s_dal[warp] = dal;
    __syncthreads();
    if (R == 0) atomicAdd(&o.ddt_bias[c * H + h], s_ddb[0][c] + s_ddb[1][c] + s_ddb[2][c] + s_ddb[3][c]);
    if (tid == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < 16; ++w) t += s_dal[w];
      atomicAdd(&o.da_log[h], t);
    }
  }
  __syncthreads();  // this record's last readers of Tensor Memory and of the small arrays are
                    // done before the next record writes them
  }  // records
  goto done;

fail:
  if (tid == 0) {
    atomicOr(&g_bwd_error, 4u);
    // at most one phase of each is in flight: the next is armed only after the block has
    // waited for the current one
    if (raw_armed > raw_seen) mbar_wait(&bar_raw, raw_seen & 1, 1000000000ull);
    if (ld_armed > ld_seen) mbar_wait(&bar_ld, ld_seen & 1, 1000000000ull);
    if (mma_phase > 0) mbar_wait(&bar_mma, (mma_phase - 1) & 1, 1000000000ull);
  }
done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kKTmemCols);
}

}  // namespace

// Bytes of the forward records and, for packed sequences, the chunk offsets after them.
size_t head_bytes(const ChunkArgs& a, long long recs) {
  const size_t coff = a.cu_seqlens ? size_t(a.B + 1) * 4 : 0;
  return align_up(record_bytes(recs) + coff, 256);
}

size_t chunk_bwd_workspace(const ChunkArgs& a) {
  const long long recs = slots_for(a) * a.H;
  return head_bytes(a, recs) +
         size_t(recs) * size_t(kRecM + kRecState + kRecTile + kRecState + kRecTile);
}

bool chunk_bwd_supported(const ChunkArgs& a, bool bf16) {
  return bf16 && a.dk == 128 && a.dv == 128 && a.chunk == 64 && !a.gate_head && !a.beta_prob &&
         !a.no_l2norm && !a.literal && (a.cu_seqlens || a.T > 0) &&
         slots_for(a) * a.H * 384 < 0x7fffffffLL;
}

namespace {

// The backward workspace: the forward records, N, the per-chunk entering state and U, then
// the reverse scan's dS' and dU per chunk.
void carve_bwd(const ChunkArgs& a, void* workspace, BwdWs& bw) {
  uint8_t* p = static_cast<uint8_t*>(workspace);
  carve_records(a, p, bw.f);
  const long long recs = bw.f.recs;
  p += head_bytes(a, recs);
  bw.f.nrec = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kRecM;
  bw.f.s0 = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kRecState;
  bw.f.ut = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kRecTile;
  bw.ds = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kRecState;
  bw.dut = reinterpret_cast<__nv_bfloat16*>(p);
}

}  // namespace

cudaError_t launch_chunk_fwd_train(const ChunkArgs& a, void* workspace, cudaStream_t st) {
  BwdWs bw{};
  carve_bwd(a, workspace, bw);
  bw.f.bwd = 2;
  if (a.cu_seqlens) {
    const cudaError_t e = split::launch_chunk_offsets(a, bw.f, st);
    if (e != cudaSuccess) return e;
  }
  return split::launch_prep_scan(a, bw.f, st);
}

cudaError_t launch_chunk_bwd(const ChunkArgs& a, const void* d_out, const float* d_final,
                             void* dq, void* dk, void* dv, float* dg, float* dbeta_logits,
                             float* da_log, float* ddt_bias, float* d_initial, void* workspace,
                             bool saved, cudaStream_t st) {
  BwdWs bw{};
  carve_bwd(a, workspace, bw);
  const long long recs = bw.f.recs;
  BwdOut o{};
  o.d_final = d_final;
  o.dq = static_cast<__nv_bfloat16*>(dq);
  o.dk = static_cast<__nv_bfloat16*>(dk);
  o.dv = static_cast<__nv_bfloat16*>(dv);
  o.dg = dg;
  o.dbeta_logits = dbeta_logits;
  o.da_log = da_log;
  o.ddt_bias = ddt_bias;
  o.d_initial = d_initial;

  cudaError_t e = cudaMemsetAsync(da_log, 0, sizeof(float) * a.H, st);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * kD * a.H, st)) != cudaSuccess) return e;
  if (!saved) {  // the forward's records and states, without its output
    ChunkArgs f = a;
    f.out = nullptr;
    f.final_state = nullptr;
    bw.f.bwd = 1;
    if (a.cu_seqlens && (e = split::launch_chunk_offsets(a, bw.f, st)) != cudaSuccess) return e;
    if ((e = split::launch_prep_scan(f, bw.f, st)) != cudaSuccess) return e;
  }

  const long long tok_rows = a.cu_seqlens ? a.total_T : (long long)a.B * a.T;
  const long long rows = tok_rows > 0 ? tok_rows : 1;
  CUtensorMap mqw, mku, mm, mdo, mdut, mn, mut, ms0, mds, mq, mk, mg;
  if (!make_map_2d(&mqw, bw.f.qw, recs * 64, 128, 64) ||
      !make_map_2d(&mku, bw.f.ku, 3 * recs * 128, 64, 128) ||
      !make_map_2d(&mm, bw.f.m, recs * 64, 64, 64) || !make_map_in(&mdo, d_out, rows, a.H, false) ||
      !make_map_2d(&mdut, bw.dut, recs * 128, 64, 128) ||
      !make_map_2d(&mn, bw.f.nrec, recs * 64, 64, 64) ||
      !make_map_2d(&mut, bw.f.ut, recs * 128, 64, 128) ||
      !make_map_2d(&ms0, bw.f.s0, recs * 128, 128, 128) ||
      !make_map_2d(&mds, bw.ds, recs * 128, 128, 128) ||
      !make_map_in(&mq, a.q, rows, a.H, false) || !make_map_in(&mk, a.k, rows, a.H, false) ||
      !make_map_in(&mg, a.g, rows, a.H, true))
    return cudaErrorInvalidValue;
  if ((e = cudaFuncSetAttribute(bwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kBSSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kKSmem)) != cudaSuccess)
    return e;
  bwd_scan_kernel<<<dim3(a.H, a.B), kBSThreads, kBSSmem, st>>>(mqw, mku, mm, mdo, mds, mdut, a,
                                                                 bw, o);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // persistent: one CTA per SM walks the records
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long grid = std::min<long long>(recs, sms);
  bwd_chunk_kernel<<<(unsigned)grid, kKThreads, kKSmem, st>>>(mdut, mn, mut, mdo, ms0, mds, mq,
                                                               mk, mg, a, bw, o);
  return cudaGetLastError();
}

unsigned int chunk_bwd_read_error(bool reset) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof(v));
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_bwd_error, &z, sizeof(z));
  }
  return v;
}

}  // namespace kda
