// Workspace records of the two-launch tensor-core chunk path (bf16, dk = dv = 128, 64-token
// chunks), shared by the forward (kda_chunk_split.cu) and the chunked backward
// (kda_chunk_bwd.cu): the per-(chunk, head) record layout, the tensor maps that move records
// and token tiles, and the host-side carving of the workspace.
#pragma once

#include <algorithm>

#include "chunk_common.cuh"

namespace kda {
namespace split {

constexpr int kC = 64;
constexpr int kD = 128;

constexpr long long kRecTile = 64LL * 128 * 2;  // one [64 x 128] (or [128 x 64]) bf16 tile
constexpr long long kRecM = 64LL * 64 * 2;
constexpr long long kRecVec = 256 * 4;          // e^{G_C}[128], rk[64], rq[64]
constexpr long long kRecState = 128LL * 128 * 2;  // a bf16 [128 x 128] state image

struct Ws {
  __nv_bfloat16* qw;   // [recs * 64][128]: Q~ records
  // [3 * recs * 128][64]: K^^T records ([128][64] each), then U~^T records (16-byte pieces
  // stored piece-major, [8][128][8]), then the -W records: token-major [64][128] each for
  // the forward, -W^T [128][64] for the backward's records (the same bytes)
  __nv_bfloat16* ku;
  __nv_bfloat16* m;    // [recs * 64][64]
  float* vec;          // [recs][256]
  int32_t* coff;       // [N + 1] first chunk slot of each sequence (packed inputs only)
  long long recs;      // chunk slots x heads
  int nck_fixed;       // chunks per sequence (fixed-length inputs)
  // Chain splitting of the packed forward (null otherwise).  A sequence's scan is a chain
  // of per-chunk affine maps S' = A_c S + B_c; a long one is cut at chunk `mid` into three
  // chains that run at once: [0, mid) from the initial state (its end state is S_mid),
  // [mid, nck) from S = 0 (end state S0, outputs O0) and [mid, nck) from S = I with the
  // chunk writes dropped (end state P = A_{nck-1} ... A_mid, outputs X).  Then the true
  // outputs of the second part are O0 + X S_mid and its end state S0 + P S_mid.
  int4* chains;        // [N + 2 kMaxSplit] scan work, longest first: seq, first chunk,
                       // end chunk, kind | slot << 2 (kind 0 whole, 1 first part, 2 from
                       // zero, 3 from identity)
  int32_t* nchains;    // [2]: chain count, split count
  int4* splits;        // [kMaxSplit]: seq, mid, nck of each split sequence
  float* split_st;     // [kMaxSplit][3][H][128][128]: S_mid, S0, P (fp32, [dk][dv])
  __nv_bfloat16* xbuf; // [total_T][H][128]: X rows of the second parts
  // Records kept for the backward (bwd != 0).  The prep then folds rq into Q~ and into the
  // rows of M (Q~ = q^ e^{G}, M[r][s] = rq_r M_raw[r][s]) and writes N; the scan writes,
  // per chunk, the state entering it and the chunk's U, and computes the output only in
  // the training forward (bwd == 2), not in the backward's own forward pass (bwd == 1).
  __nv_bfloat16* nrec;  // [recs * 64][64]: N = (I + diag(beta) tril(A, -1))^{-1}, s <= r
  __nv_bfloat16* s0;    // [recs * 128][128]: S^T entering the chunk (row = value column j)
  __nv_bfloat16* ut;    // [recs * 128][64]: U^T of the chunk (row j, column = token)
  int bwd;
};

constexpr int kMaxSplit = 8;      // sequences whose chain may be split, per call
constexpr int kSplitMinChunks = 16;  // shortest chain worth splitting

inline long long slots_for(const ChunkArgs& a) {
  if (a.cu_seqlens) return (long long)a.total_T / kC + a.B;
  return (long long)a.B * ((a.T + kC - 1) / kC);
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of the forward records for `recs` records.
inline size_t record_bytes(long long recs) {
  return size_t(recs) * size_t(4 * kRecTile + kRecM + kRecVec);
}

// Lays the forward records out from `base` (the varlen chunk offsets follow them).
inline uint8_t* carve_records(const ChunkArgs& a, void* base, Ws& ws) {
  const long long recs = slots_for(a) * a.H;
  uint8_t* p = static_cast<uint8_t*>(base);
  ws.recs = recs;
  ws.nck_fixed = a.cu_seqlens ? 0 : (a.T + kC - 1) / kC;
  ws.qw = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kRecTile;
  ws.ku = reinterpret_cast<__nv_bfloat16*>(p);
  p += 3 * recs * kRecTile;
  ws.m = reinterpret_cast<__nv_bfloat16*>(p);
  p += recs * kRecM;
  ws.vec = reinterpret_cast<float*>(p);
  p += recs * kRecVec;
  ws.coff = reinterpret_cast<int32_t*>(p);
  return p;
}

// [rows][inner] bf16, box {64, box_rows}, 128-byte swizzle.
inline bool make_map_2d(CUtensorMap* m, const void* base, long long rows, int inner,
                        int box_rows) {
  auto enc = chunk::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// [rows, H, 128] bf16 output, box {64 ch, 1 head, 64 tokens}, 128-byte swizzle.
inline bool make_map_out(CUtensorMap* m, const void* base, long long rows, int H) {
  auto enc = chunk::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// [rows, H, 128] inputs, box {64 ch, 1 head, 64 tokens} bf16 with 128-byte swizzle, or
// {32 ch, 1, 64} fp32 without swizzle; rows past the end read as zeros.
inline bool make_map_in(CUtensorMap* m, const void* base, long long rows, int H, bool fp32) {
  auto enc = chunk::encode_fn();
  if (!enc) return false;
  const int es = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * es, (cuuint64_t)H * kD * es};
  cuuint32_t box[3] = {fp32 ? 32u : 64u, 1, 64};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
             fp32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Prep and scan launches over records carved into `ws` (the chunk offsets of packed inputs
// must already be in ws.coff).  With ws.bwd set they keep the backward's records instead
// of producing the output.
cudaError_t launch_prep_scan(const ChunkArgs& a, const Ws& ws, cudaStream_t st);
// The first chunk slot of every packed sequence into ws.coff (one CTA).
cudaError_t launch_chunk_offsets(const ChunkArgs& a, const Ws& ws, cudaStream_t st);

}  // namespace split
}  // namespace kda
