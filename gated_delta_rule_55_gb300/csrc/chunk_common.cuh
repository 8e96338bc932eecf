// Device helpers shared by the tensor-core chunk kernels: bf16 packing, single-instruction
// exponential / reciprocal approximations, Tensor Memory stores, the warp-level tf32 block
// solve of the UT transform, bulk-tensor stores, and the host-side tensor-map encoder.
#pragma once

#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "tc_prims.cuh"

namespace kda {
namespace chunk {

using namespace tc;

constexpr int LDL = 68;  // fp32 row pitch of the 64 x 64 solve matrices (16-byte aligned rows)
constexpr int LDY = 24;  // pitch of the per-warp 16 x 16 solve scratch

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// e^x as 2^(x log2 e) on the approximate exponential unit, and an approximate reciprocal:
// single instructions; their relative error (~2^-22) is far below the bf16 rounding of
// every operand they feed.
__device__ __forceinline__ float fast_exp(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}
// 2^x on the approximate exponential unit (x already in log2 units).
constexpr float kLog2E = 1.4426950408889634f;
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed bf16 x bf16 -> bf16 products (round to nearest even).
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                   *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// tcgen05.st of 8 columns (shape 32x32b, x8), waited for.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// tcgen05.st of 32 fp32 columns, waited for.
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

// Warp-level tf32 MMA (m16n8k8, fp32 accumulate) for the small 16 x 16 block products of
// the triangular solve.  Fragment ownership (g = lane / 4, t = lane % 4):
//   A 16x8: a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4)
//   B 8x8:  b0 (t, g), b1 (t + 4, g)
//   C 16x8: c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t), c3 (g + 8, 2t + 1)
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// C[16 x 16] += A[16 x K] B[K x 16] for fp32 matrices in shared memory (row pitches
// lda, ldb in floats), one warp.  C is two 16 x 8 accumulator tiles.
template <int K>
__device__ __forceinline__ void warp_gemm16(const float* A, int lda, const float* B, int ldb,
                                            float (&c)[2][4], int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    const uint32_t a[4] = {__float_as_uint(A[g * lda + k0 + t]),
                           __float_as_uint(A[(g + 8) * lda + k0 + t]),
                           __float_as_uint(A[g * lda + k0 + t + 4]),
                           __float_as_uint(A[(g + 8) * lda + k0 + t + 4])};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t b[2] = {__float_as_uint(B[(k0 + t) * ldb + 8 * nt + g]),
                             __float_as_uint(B[(k0 + t + 4) * ldb + 8 * nt + g])};
      mma_tf32(c[nt], a, b);
    }
  }
}

// Store a 16 x 16 accumulator (times `sign`) to a row-major fp32 matrix (pitch ld).
__device__ __forceinline__ void warp_store16(float* D, int ld, const float (&c)[2][4],
                                             float sign, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2*>(D + g * ld + 8 * nt + 2 * t) =
        make_float2(sign * c[nt][0], sign * c[nt][1]);
    *reinterpret_cast<float2*>(D + (g + 8) * ld + 8 * nt + 2 * t) =
        make_float2(sign * c[nt][2], sign * c[nt][3]);
  }
}

// One level (block distance D) of the blocked triangular inverse: warp jj computes
// X_{jj+D, jj} = -X_ii sum_{k=jj}^{jj+D-1} L_{jj+D, k} X_{k, jj} (16 x 16 blocks, fp32
// storage with pitch LDL, tf32 products), through its own 16 x 16 scratch tile.
template <int D>
__device__ __forceinline__ void solve_level(const float* L, float* X, float* Y, int warp,
                                            int lane) {
  const int jj = warp, ii = warp + D;
  if (ii >= 4) return;  // warp-uniform
  float* Yw = Y + jj * 16 * LDY;
  float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  warp_gemm16<16 * D>(L + (16 * ii) * LDL + 16 * jj, LDL, X + (16 * jj) * LDL + 16 * jj, LDL,
                      c, lane);
  warp_store16(Yw, LDY, c, 1.f, lane);
  __syncwarp();
  float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  warp_gemm16<16>(X + (16 * ii) * LDL + 16 * ii, LDL, Yw, LDY, z, lane);
  warp_store16(X + (16 * ii) * LDL + 16 * jj, LDL, z, -1.f, lane);
}

// 3-D tiled store of a shared-memory box to global memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Byte offset of the 16-byte chunk holding tokens 8 tg .. 8 tg + 7 of row c of a
// transposed [128 x 64] tile (rows = channels, tokens contiguous, one 128-byte block).
__device__ __forceinline__ uint32_t trow_off(int c, int tg) {
  return uint32_t((c >> 3) * 1024 + (c & 7) * 128 + ((tg ^ (c & 7)) << 4));
}

// 2-D tiled load / store of a shared-memory box (coordinates c0 innermost, c1).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0,
                                             int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}
// Plain (untiled) bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch `bytes` (multiple of 16, 16-byte aligned address) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// L2 eviction-priority policy for data read once (createpolicy; every access that carries
// it is among the first candidates for eviction).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The tiled / plain bulk loads above with an L2 cache-policy hint.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Host: the driver's cuTensorMapEncodeTiled, looked up once through the runtime.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace chunk
}  // namespace kda
