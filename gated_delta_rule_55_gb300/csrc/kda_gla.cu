// Gated linear recurrent attention (ejkernel "recurrent" page, recurrent_attention): per
// (sequence, query head) a state h in R^{D x D} advanced token by token,
//
//   a_t = g_t + gk_t + g_gamma   (log-decay along the key axis; each term when given)
//   h_t = diag(e^{a_t}) h_{t-1} diag(e^{gv_t}) + k_t v_t^T,        o_t = h_t^T (scale q_t)
//
// (the page names the gates but prints no formula: this is the reading stated with the
// oracle).  Query head h reads key / value head h / (Hq / Hkv); `reverse` walks each
// sequence from its last token to its first.
//
// One CTA per (sequence, query head, 32-wide slice of the value axis): thread (r, c) =
// (tid / 8, tid % 8) owns columns 4 c .. 4 c + 3 on the row pairs (2 p, 2 p + 1),
// p = r, r + G, ... (G = threads / 8 row groups); the state slice stays in registers as pairs of adjacent key channels,
// so that every update is a packed two-lane fp32 multiply or fma (Blackwell's f32x2) whose
// key-channel operands (k, e^{a}, scale q) load as pairs and whose value-column operands
// (v, e^{gv}) are broadcast once per token.  The
// state update needs no other thread's data, and no token needs an earlier token's output,
// so tokens go in blocks of kTB: the block's inputs are staged in shared memory (gate
// exponentials applied), every thread advances its state through the whole block keeping one
// partial output per token, and the outputs are reduced over the key axis once per block.
// The raw inputs of the next block are copied global -> shared with cp.async (no registers)
// while the current block is computed.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDVS = 32;
// Threads per CTA: 8 column groups x 16 row groups (256 threads measured slower: the
// per-block staging and output reduction grow while the work per thread halves).
template <int D>
__host__ __device__ constexpr int gla_threads() { return 128; }
constexpr int kTB = 8;  // tokens per staged block (4 CTAs per SM fit with the double buffer)

// 16-byte asynchronous global -> shared copy (cp.async, cache-global), and its group fences.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_one() {  // all but the newest group landed
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Raw inputs of one block of tokens as they sit in memory.
template <typename Tin, int D>
struct RawBlock {
  Tin q[kTB][D], k[kTB][D];
  float a[kTB][D];            // g + gk (g_gamma is added on conversion)
  float gk2[kTB][D];          // the second key gate when both g and gk are given
  Tin v[kTB][kDVS];
  float gv[kTB][kDVS];
};

// Packed two-lane fp32 arithmetic (sm_100 family): a 64-bit register holds (lo, hi).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <typename Tin, int D>
__global__ void __launch_bounds__(gla_threads<D>()) gla_kernel(GlaArgs a) {
  constexpr int kThreads = gla_threads<D>();
  constexpr int NRG = kThreads / 8;    // row groups
  constexpr int NW = kThreads / 32;    // warps
  constexpr int PPT = D / (2 * NRG);   // row pairs per thread
  extern __shared__ __align__(16) uint8_t dyn[];
  RawBlock<Tin, D>* raw = reinterpret_cast<RawBlock<Tin, D>*>(dyn);  // [2], double-buffered
  // per token and key channel: k, e^{a}, scale q
  __shared__ __align__(16) float s_k[kTB][D], s_ea[kTB][D], s_q[kTB][D];
  __shared__ __align__(16) float2 s_vb[kTB][kDVS];   // (v, e^{gv}) per token and column
  __shared__ __align__(16) float s_o[kTB][NW][kDVS];  // per-warp partial outputs

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int rg = tid >> 3, c4 = tid & 7;
  const int j0 = blockIdx.x * kDVS, h = blockIdx.y, seq = blockIdx.z;
  const int Hq = a.Hq, Hkv = a.Hkv, hk = h / (Hq / Hkv);
  long long bos;
  int len;
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
  const int bidx = a.cu_seqlens ? 0 : seq;  // batch row of g_gamma
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  Tin* out = static_cast<Tin*>(a.out);
  const long long st_off = ((long long)seq * Hq + h) * D * D;
  const float gamma = a.g_gamma ? a.g_gamma[bidx * Hq + h] : 0.f;

  // S2[i][jj] = (S[2 p][j], S[2 p + 1][j]) with p = rg + NRG i, j = j0 + 4 c4 + jj
  uint64_t S2[PPT][4];
#pragma unroll
  for (int i = 0; i < PPT; ++i)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const long long e0 = st_off + (long long)(2 * (rg + NRG * i)) * D + j0 + 4 * c4 + jj;
      S2[i][jj] = a.initial_state ? f2pack(a.initial_state[e0], a.initial_state[e0 + D])
                                  : f2pack(0.f, 0.f);
    }

  // token slot u of a block starting at position p0 is position p0 + u (forward) or
  // p0 - u (reverse)
  const int dir = a.reverse ? -1 : 1;
  const int nblocks = (len + kTB - 1) / kTB;
  // copies block bi's raw rows into raw[bi & 1] (16-byte pieces; one commit group)
  auto fetch = [&](int bi) {
    if (bi < nblocks) {
      RawBlock<Tin, D>& r = raw[bi & 1];
      const int b0 = bi * kTB, nb = min(kTB, len - b0);
      const int p0 = a.reverse ? len - 1 - b0 : b0;
      constexpr int QP = D * sizeof(Tin) / 16;    // 16-byte pieces per q / k row
      constexpr int FP = D * 4 / 16;              // per fp32 gate row
      constexpr int VP = kDVS * sizeof(Tin) / 16; // per v slice row
      constexpr int GP = kDVS * 4 / 16;           // per gv slice row
      for (int e = tid; e < nb * QP; e += kThreads) {
        const int u = e / QP, pc = e % QP;
        const long long tok = bos + p0 + dir * u;
        cp_async16(reinterpret_cast<uint8_t*>(r.q[u]) + 16 * pc,
                   reinterpret_cast<const uint8_t*>(q + (tok * Hq + h) * D) + 16 * pc);
        cp_async16(reinterpret_cast<uint8_t*>(r.k[u]) + 16 * pc,
                   reinterpret_cast<const uint8_t*>(k + (tok * Hkv + hk) * D) + 16 * pc);
      }
      const float* ga = a.g ? a.g : a.gk;          // first key gate, if any
      const float* gb = (a.g && a.gk) ? a.gk : nullptr;
      for (int e = tid; e < nb * FP; e += kThreads) {
        const int u = e / FP, pc = e % FP;
        const long long rq = (bos + p0 + dir * u) * Hq + h;
        if (ga) cp_async16(reinterpret_cast<uint8_t*>(r.a[u]) + 16 * pc,
                           reinterpret_cast<const uint8_t*>(ga + rq * D) + 16 * pc);
        if (gb) cp_async16(reinterpret_cast<uint8_t*>(r.gk2[u]) + 16 * pc,
                           reinterpret_cast<const uint8_t*>(gb + rq * D) + 16 * pc);
      }
      for (int e = tid; e < nb * VP; e += kThreads) {
        const int u = e / VP, pc = e % VP;
        const long long tok = bos + p0 + dir * u;
        cp_async16(reinterpret_cast<uint8_t*>(r.v[u]) + 16 * pc,
                   reinterpret_cast<const uint8_t*>(v + (tok * Hkv + hk) * D + j0) + 16 * pc);
      }
      if (a.gv) {
        for (int e = tid; e < nb * GP; e += kThreads) {
          const int u = e / GP, pc = e % GP;
          const long long rq = (bos + p0 + dir * u) * Hq + h;
          cp_async16(reinterpret_cast<uint8_t*>(r.gv[u]) + 16 * pc,
                     reinterpret_cast<const uint8_t*>(a.gv + rq * D + j0) + 16 * pc);
        }
      }
    }
    cp_async_commit();  // (an empty group past the last block keeps the counting uniform)
  };
  fetch(0);
  for (int bi = 0; bi < nblocks; ++bi) {
    const int b0 = bi * kTB, nb = min(kTB, len - b0);
    const int p0 = a.reverse ? len - 1 - b0 : b0;
    fetch(bi + 1);      // in flight while this block is converted and computed
    cp_async_wait_one();  // this block's copies have landed (for this thread)
    __syncthreads();      // ... and for every thread
    const RawBlock<Tin, D>& r = raw[bi & 1];
    const bool has_a = a.g || a.gk, has_b = a.g && a.gk;
    for (int e = tid; e < nb * D; e += kThreads) {
      const int u = e / D, c = e % D;
      float x = gamma;
      if (has_a) x += r.a[u][c];
      if (has_b) x += r.gk2[u][c];
      s_k[u][c] = load_as_float(&r.k[u][c]);
      s_ea[u][c] = __expf(x);
      s_q[u][c] = a.scale * load_as_float(&r.q[u][c]);
    }
    for (int e = tid; e < nb * kDVS; e += kThreads) {
      const int u = e / kDVS, jj = e % kDVS;
      s_vb[u][jj] = make_float2(load_as_float(&r.v[u][jj]), a.gv ? __expf(r.gv[u][jj]) : 1.f);
    }
    __syncthreads();
    // every token of the block advances the state and leaves this thread's partial output
    // (its row pairs, four columns); the partials are summed over the warp's row groups once
    // per block.  Unrolled over the block, so that the next token's operand loads go out
    // while the current token's products run.
    float po[kTB * 4];
#pragma unroll
    for (int u = 0; u < kTB; ++u) {
      if (u < nb) {  // uniform
        const float4 vb01 = *reinterpret_cast<const float4*>(&s_vb[u][4 * c4]);
        const float4 vb23 = *reinterpret_cast<const float4*>(&s_vb[u][4 * c4 + 2]);
        const uint64_t vv2[4] = {f2pack(vb01.x, vb01.x), f2pack(vb01.z, vb01.z),
                                 f2pack(vb23.x, vb23.x), f2pack(vb23.z, vb23.z)};
        const uint64_t bb2[4] = {f2pack(vb01.y, vb01.y), f2pack(vb01.w, vb01.w),
                                 f2pack(vb23.y, vb23.y), f2pack(vb23.w, vb23.w)};
        uint64_t o2[4] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f),
                          f2pack(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
          const int c = 2 * (rg + NRG * i);
          const uint64_t k2 = *reinterpret_cast<const uint64_t*>(&s_k[u][c]);
          const uint64_t ea2 = *reinterpret_cast<const uint64_t*>(&s_ea[u][c]);
          const uint64_t q2 = *reinterpret_cast<const uint64_t*>(&s_q[u][c]);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            // S = (e^{a} e^{gv}) S + k v, then the output partial q . S over the two rows
            S2[i][jj] = f2fma(f2mul(ea2, bb2[jj]), S2[i][jj], f2mul(k2, vv2[jj]));
            o2[jj] = f2fma(S2[i][jj], q2, o2[jj]);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float lo, hi;
          f2unpack(o2[jj], lo, hi);
          po[4 * u + jj] = lo + hi;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) po[4 * u + jj] = 0.f;
      }
    }
    // sums over the warp's four row groups (lanes c4, c4 + 8, c4 + 16, c4 + 24), scattered:
    // lane bit 3 picks a half of the 32 (token, column) partials, lane bit 4 a quarter, so
    // that every lane ends with the totals of two tokens (same pairing of the additions as
    // a per-token butterfly)
    {
      const bool up1 = (lane & 8) != 0, up2 = (lane & 16) != 0;
      float h1[kTB * 2];
#pragma unroll
      for (int i = 0; i < kTB * 2; ++i) {
        const float send = up1 ? po[i] : po[i + kTB * 2];
        const float keep = up1 ? po[i + kTB * 2] : po[i];
        h1[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      float h2[kTB];
#pragma unroll
      for (int i = 0; i < kTB; ++i) {
        const float send = up2 ? h1[i] : h1[i + kTB];
        const float keep = up2 ? h1[i + kTB] : h1[i];
        h2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
      // this lane's totals: partial indices 2 kTB up1 + kTB up2 + (0 .. kTB - 1)
      const int u0 = (2 * kTB * (up1 ? 1 : 0) + kTB * (up2 ? 1 : 0)) / 4;
#pragma unroll
      for (int m = 0; m < kTB / 4; ++m)
        *reinterpret_cast<float4*>(&s_o[u0 + m][w][4 * c4]) =
            make_float4(h2[4 * m], h2[4 * m + 1], h2[4 * m + 2], h2[4 * m + 3]);
    }
    __syncthreads();
    for (int e = tid; e < nb * kDVS; e += kThreads) {
      const int u = e / kDVS, jj = e % kDVS;
      float tot = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) tot += s_o[u][ww][jj];
      store_from_float(out + ((bos + p0 + dir * u) * Hq + h) * D + j0 + jj, tot);
    }
    __syncthreads();  // the staged block, the partials and raw[bi & 1] are rewritten next
  }
  if (a.final_state) {
#pragma unroll
    for (int i = 0; i < PPT; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const long long e0 = st_off + (long long)(2 * (rg + NRG * i)) * D + j0 + 4 * c4 + jj;
        float lo, hi;
        f2unpack(S2[i][jj], lo, hi);
        a.final_state[e0] = lo;
        a.final_state[e0 + D] = hi;
      }
  }
}

template <typename Tin, int D>
cudaError_t launch_t(const GlaArgs& a, cudaStream_t st) {
  const dim3 grid(D / kDVS, a.Hq, a.nseq);
  const int dyn = 2 * (int)sizeof(RawBlock<Tin, D>);
  cudaError_t e = cudaFuncSetAttribute(gla_kernel<Tin, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  gla_kernel<Tin, D><<<grid, gla_threads<D>(), dyn, st>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dtype(const GlaArgs& a, cudaStream_t st) {
  switch (a.D) {
    case 32: return launch_t<Tin, 32>(a, st);
    case 64: return launch_t<Tin, 64>(a, st);
    default: return launch_t<Tin, 128>(a, st);
  }
}

}  // namespace

cudaError_t launch_gla(const GlaArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? launch_dtype<__nv_bfloat16>(a, st) : launch_dtype<float>(a, st);
}

}  // namespace kda
