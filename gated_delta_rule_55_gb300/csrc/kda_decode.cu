// Single-token KDA decode step (NKI "KDA TKG Kernel API Reference", kda_tkg): for every
// (request b, head h) the fp32 memory S[b, h] ([dk, dv]) is streamed from HBM exactly
// once, decayed, given the delta-rule write and written back in place, while the output
// o = S_new^T q^ is formed from the same data.
//
// Per (b, h), with S' = diag(exp(gamma)) S:
//   p_k = S'^T k^,  p_q = S'^T q^            (reductions over the dk rows)
//   u   = beta (v - p_k)
//   S   = S' + k^ u^T
//   o   = S^T q^ = p_q + u (k^ . q^)
// Every value column is independent (the reductions run over dk only), so one pass over
// S suffices.  The step is bound by HBM: 2 * dk * dv * 4 bytes of state traffic against
// ~6 flops per state element.
//
// Work layout: a persistent grid of one 256-thread CTA per SM.  Each CTA walks the
// (b, h) units u = blockIdx.x, blockIdx.x + gridDim.x, ... and streams every unit's state
// tile (contiguous, dk * dv * 4 bytes) through a 3-deep ring of shared-memory buffers
// with 1-D bulk async copies: the load of unit i + 2 and the store of unit i - 1 are in
// flight while unit i is computed.  The small per-unit inputs (q, k, g, v, beta) are
// prefetched into registers one unit ahead.
#include "kda_internal.cuh"
#include "tc_prims.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kDecodeThreads = 256;
constexpr int kBufs = 3;

__device__ unsigned int g_decode_error;  // bit 1: a bounded wait gave up

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Per-unit small inputs of one thread: channel c = tid < DK and value column tid < DV.
struct UnitIn {
  float q, k, g, v, beta_logit;
};

template <int DK, int DV>
__device__ __forceinline__ UnitIn load_unit(const DecodeArgs& a, long long bh, int tid) {
  UnitIn x{0.f, 0.f, 0.f, 0.f, 0.f};
  const int b = (int)(bh / a.H), h = (int)(bh % a.H);
  if (tid < DK) {
    const long long off = ((long long)b * DK + tid) * a.H + h;  // [B, dk, H]
    x.q = a.q[off];
    x.k = a.k[off];
    x.g = a.g[off];
  }
  if (tid < DV) x.v = a.v[bh * DV + tid];  // [B, H, dv]
  if (tid == 0) x.beta_logit = a.beta_logits[bh];  // [B, 1, H]
  return x;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(DecodeArgs a) {
  constexpr int NCG = DV / 4;                  // 16-byte column groups per row
  constexpr int NRG = kDecodeThreads / NCG;    // row groups
  constexpr int RPT = DK / NRG;                // rows per thread
  constexpr uint32_t kTile = DK * DV * 4;      // bytes of one state tile
  static_assert(DK % NRG == 0 && RPT >= 1, "tile shape");

  extern __shared__ __align__(128) uint8_t smem[];
  float* sbuf = reinterpret_cast<float*>(smem);  // kBufs tiles
  __shared__ float s_k[DK], s_q[DK], s_dec[DK];
  __shared__ float s_u[DV];
  __shared__ __align__(16) float s_red_k[NRG][DV + 4];
  __shared__ __align__(16) float s_red_q[NRG][DV + 4];
  __shared__ float s_norm[3][4];
  __shared__ float s_beta;
  __shared__ uint64_t full[kBufs];

  const int tid = threadIdx.x;
  const int cg = tid % NCG;
  const int rg = tid / NCG;
  const long long units = (long long)a.B * a.H;
  const long long first = blockIdx.x, stride = gridDim.x;
  const long long my_units = (units - first + stride - 1) / stride;

  if (tid == 0) {
    for (int i = 0; i < kBufs; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // prime the ring with the first two units
  if (tid == 0) {
    for (int i = 0; i < 2 && i < my_units; ++i) {
      const long long bh = first + i * stride;
      mbar_arrive_expect_tx(&full[i], kTile);
      bulk_load(sbuf + i * (kTile / 4), a.S + bh * (long long)(DK * DV), kTile, &full[i]);
    }
  }
  UnitIn nxt = my_units > 0 ? load_unit<DK, DV>(a, first, tid) : UnitIn{};
  bool ok = true;
  long long failed_at = -1;

  for (long long i = 0; i < my_units; ++i) {
    const long long bh = first + i * stride;
    const int h = (int)(bh % a.H);
    const int buf = (int)(i % kBufs);
    float* S = sbuf + buf * (kTile / 4);
    const UnitIn cur = nxt;
    if (i + 1 < my_units) nxt = load_unit<DK, DV>(a, bh + stride, tid);

    // prologue: gate, norms, beta (from the prefetched registers)
    float kq = 0.f;
    if (tid < DK) {
      const float gamma = gate_gamma(cur.g, a.dt_bias[tid * a.H + h], expf(a.a_log[h]),
                                     a.lower_bound);
      s_dec[tid] = expf(gamma);
      const float kk = warp_sum(cur.k * cur.k), qq = warp_sum(cur.q * cur.q),
                  kqs = warp_sum(cur.k * cur.q);
      if ((tid & 31) == 0) {
        s_norm[0][tid >> 5] = kk;
        s_norm[1][tid >> 5] = qq;
        s_norm[2][tid >> 5] = kqs;
      }
    }
    if (tid == 0) s_beta = sigmoidf_(cur.beta_logit);
    __syncthreads();
    const float beta = s_beta;
    {
      float k2 = 0.f, q2 = 0.f, kq2 = 0.f;
#pragma unroll
      for (int w = 0; w < DK / 32; ++w) {
        k2 += s_norm[0][w];
        q2 += s_norm[1][w];
        kq2 += s_norm[2][w];
      }
      const float rk = 1.0f / sqrtf(k2 + kL2Eps);
      const float rq = a.scale / sqrtf(q2 + kL2Eps);
      kq = kq2 * rk * rq;  // k^ . q^ (scale included)
      if (tid < DK) {
        s_k[tid] = cur.k * rk;
        s_q[tid] = cur.q * rq;
      }
    }
    // the tile of this unit
    const bool w = mbar_wait(&full[buf], (uint32_t)((i / kBufs) & 1));
    if (!__syncthreads_and(w)) { ok = false; failed_at = i; break; }

    // decay and the two partial reductions over this thread's rows
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int row = r * NRG + rg;
      float4 s = reinterpret_cast<const float4*>(S)[row * NCG + cg];
      const float d = s_dec[row], kr = s_k[row], qr = s_q[row];
      s.x *= d; s.y *= d; s.z *= d; s.w *= d;
      pk.x += s.x * kr; pk.y += s.y * kr; pk.z += s.z * kr; pk.w += s.w * kr;
      pq.x += s.x * qr; pq.y += s.y * qr; pq.z += s.z * qr; pq.w += s.w * qr;
    }
    *reinterpret_cast<float4*>(&s_red_k[rg][4 * cg]) = pk;
    *reinterpret_cast<float4*>(&s_red_q[rg][4 * cg]) = pq;
    __syncthreads();
    if (tid < DV) {
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int r = 0; r < NRG; ++r) {
        sk += s_red_k[r][tid];
        sq += s_red_q[r][tid];
      }
      const float u = beta * (cur.v - sk);
      s_u[tid] = u;
      a.out[bh * DV + tid] = sq + u * kq;  // [B, H, dv]
    }
    __syncthreads();
    // rank-1 delta write, back into the same buffer
    {
      const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * cg]);
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const int row = r * NRG + rg;
        float4* p = reinterpret_cast<float4*>(S) + row * NCG + cg;
        float4 s = *p;
        const float d = s_dec[row], kr = s_k[row];
        s.x = s.x * d + kr * u4.x;
        s.y = s.y * d + kr * u4.y;
        s.z = s.z * d + kr * u4.z;
        s.w = s.w * d + kr * u4.w;
        *p = s;
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(a.S + bh * (long long)(DK * DV), S, kTile);
      bulk_commit();
      // the buffer of unit i + 2 was last used by unit i - 1: its store must be done
      // reading before the next load lands there
      if (i + 2 < my_units) {
        bulk_wait_read<1>();
        const int nb = (int)((i + 2) % kBufs);
        mbar_arrive_expect_tx(&full[nb], kTile);
        bulk_load(sbuf + nb * (kTile / 4), a.S + (bh + 2 * stride) * (long long)(DK * DV),
                  kTile, &full[nb]);
      }
    }
  }
  if (tid == 0) {
    if (!ok) {
      atomicOr(&g_decode_error, 2u);
      // loads issued for units failed_at and failed_at + 1 may still be in flight: let
      // them land (bounded) before the shared memory is released
      for (long long j = failed_at; j < failed_at + 2 && j < my_units; ++j)
        mbar_wait(&full[j % kBufs], (uint32_t)((j / kBufs) & 1), 1000000000ull);
    }
    bulk_wait_all();
  }
  __syncthreads();
}

int g_num_sms = 0;

template <int DK, int DV>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  const size_t smem = (size_t)kBufs * DK * DV * 4;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.B * a.H;
  const int grid = (int)(units < g_num_sms ? units : g_num_sms);
  decode_kernel<DK, DV><<<grid, kDecodeThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const DecodeArgs& a, cudaStream_t st) {
  switch (a.dv) {
    case 32: return launch_t<DK, 32>(a, st);
    case 64: return launch_t<DK, 64>(a, st);
    default: return launch_t<DK, 128>(a, st);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  switch (a.dk) {
    case 32: return launch_dk<32>(a, st);
    case 64: return launch_dk<64>(a, st);
    default: return launch_dk<128>(a, st);
  }
}

unsigned int decode_read_error(bool reset) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v));
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_decode_error, &z, sizeof(z));
  }
  return v;
}

}  // namespace kda
