// query_lowrank.cu -- MFA's low-rank query path on the tensor cores.
//
// "Step-3 is Large yet Affordable" (paper summary page), section 2 / Table 1:
// the query is projected down from the model width (7168) to rank 2048,
// normalised, then projected up to 64 heads x 256. Read as
//     y = x W_down (fp32),  h = bf16(y / sqrt(mean(y^2) + eps) * gamma),
//     q = bf16(h W_up)
// Both products are skinny (M = the batch): every weight element is used once
// per call, so the path streams the weights (96 MB at the Step-3 shape) and
// is bound by HBM bandwidth.
//
// lowrank_gemm_kernel computes the transposed product for 128 output
// features and a range of K per CTA:
//     Y^T[feature, b] = W[k, feature]^T . X[b, k]^T    (M=128, N=batch padded
//                                                      to 16, K=16 per MMA)
// A = a W tile [64 k rows x 128 features] (two [64 x 64] TMA boxes, 128-byte
// swizzle, MN-major), B = an X tile [batch rows x 64 k] (K-major), D in TMEM
// (lane = feature, column = batch entry). Warps 0-3 write the result (lane =
// feature, so consecutive lanes store consecutive features), warp 4 issues the
// TMA copies through a 4-stage mbarrier ring, one thread of warp 5 issues the
// MMAs. The down-projection splits K over the CTAs (its 16 feature blocks
// alone would leave most SMs idle) and adds the partial sums with fp32
// atomics; the up-projection writes bf16 directly. Every wait is bounded.
#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kGemmThreads = 192;
constexpr int kGemmStages = 4;
constexpr int kKChunk = 64;            // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kWStageBytes = 16384;    // [64 k rows x 128 features] bf16
constexpr int kTmemColsGemm = 256;     // D: up to 256 batch columns
constexpr int kNormThreads = 256;

struct GemmParams {
  float* y;          // [B][N] fp32, accumulated with atomics (K split over CTAs), or null
  uint16_t* out;     // [B][N] bf16 bits, written directly (one K range per feature block), or null
  uint32_t* err;
  uint64_t budget;
  int B, Bp, N, K, splits;
};

__host__ __device__ constexpr uint32_t x_stage_bytes(int Bp) { return (uint32_t)Bp * 128u; }
__host__ __device__ constexpr uint32_t gemm_stage_bytes(int Bp) {
  return ((uint32_t)kWStageBytes + x_stage_bytes(Bp) + 1023u) & ~1023u;
}
__host__ __device__ constexpr size_t gemm_smem_bytes(int Bp) { return 1024 + (size_t)kGemmStages * gemm_stage_bytes(Bp); }

template <bool kAtomic>
__global__ void __launch_bounds__(kGemmThreads, 1)
    lowrank_gemm_kernel(const __grid_constant__ GemmParams g, const __grid_constant__ CUtensorMap wmap,
                        const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t bars[2 * kGemmStages + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const uint32_t raw = smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = gemm_stage_bytes(g.Bp);
  const int chunks = g.K / kKChunk;
  const int c0 = (int)((long long)blockIdx.y * chunks / g.splits);
  const int c1 = (int)((long long)(blockIdx.y + 1) * chunks / g.splits);
  const int f0 = blockIdx.x * 128;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kGemmStages]);
  const uint32_t done = smem_u32(&bars[2 * kGemmStages]);
  volatile int* abort = &abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGemmStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    mbar_init(done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&wmap);
    prefetch_tensormap(&xmap);
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "n"(kTmemColsGemm)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    if (lane == 0) {  // producer: W tile (streamed once) and X tile (re-read by every feature block)
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      int i = 0;
      for (int c = c0; c < c1; ++c, ++i) {
        const int s = i % kGemmStages, n = i / kGemmStages;
        if (!mbar_wait(empty0 + 8 * s, (n & 1) ^ 1, g.budget, abort, g.err)) break;
        const uint32_t dst = base + s * sb, bar = full0 + 8 * s;
        mbar_arrive_expect_tx(bar, (uint32_t)kWStageBytes + x_stage_bytes(g.Bp));
        tma_load_2d(dst, &wmap, f0, c * kKChunk, bar, pol_w);
        tma_load_2d(dst + 8192, &wmap, f0 + 64, c * kKChunk, bar, pol_w);
        tma_load_2d(dst + kWStageBytes, &xmap, c * kKChunk, 0, bar, pol_x);
      }
      // every copy this thread issued must land before the CTA exits
      for (int k = (i > kGemmStages ? i - kGemmStages : 0); k < i; ++k)
        (void)mbar_wait(full0 + 8 * (k % kGemmStages), (k / kGemmStages) & 1, g.budget, nullptr, g.err);
    }
  } else if (warp == 5) {
    if (lane == 0 && c0 < c1) {  // MMA issue: 4 MMAs of K=16 per stage
      const uint32_t idesc = idesc_f16(128, g.Bp, 1, 1, 0);  // bf16; A (W^T) MN-major, B (X) K-major
      int i = 0;
      bool ok = true;
      for (int c = c0; c < c1; ++c, ++i) {
        const int s = i % kGemmStages, n = i / kGemmStages;
        if (!(ok = mbar_wait(full0 + 8 * s, n & 1, g.budget, abort, g.err))) break;
        tc_fence_after();
        const uint32_t a = base + s * sb, b = a + kWStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tmem, smem_desc_sw128(a + kk * 2048, 8192, 1024), smem_desc_sw128(b + kk * 32, 16, 1024), idesc,
                 (i | kk) != 0);
        tc_commit(empty0 + 8 * s);
      }
      tc_commit(done);  // also tracks the MMAs of an abandoned range, so TMEM is quiet before release
      (void)ok;
    }
  } else {  // warps 0-3: lane = feature f0 + 32 warp + lane; TMEM columns = batch entries
    if (c0 < c1 && mbar_wait(done, 0, g.budget, abort, g.err)) {
      tc_fence_after();
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      const int f = f0 + 32 * warp + lane;
      for (int j = 0; j < g.Bp; j += 32) {
        float v[32];
        tmem_ld32(tmem + lane_base + j, v);
        tc_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int b = j + u;
          if (b < g.B) {
            if constexpr (kAtomic)
              atomicAdd(g.y + (size_t)b * g.N + f, v[u]);
            else
              g.out[(size_t)b * g.N + f] = __bfloat16_as_ushort(__float2bfloat16_rn(v[u]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemColsGemm) : "memory");
}

// h[b][i] = bf16(y[b][i] / sqrt(mean_i y[b][i]^2 + eps) * gamma[i]); one CTA per batch row.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float* y, const uint16_t* gamma, uint16_t* h,
                                                                int R, float eps) {
  __shared__ float part[kNormThreads / 32];
  const float* row = y + (size_t)blockIdx.x * R;
  float ss = 0.0f;
  for (int i = threadIdx.x; i < R; i += kNormThreads) {
    const float v = row[i];
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += part[w];
  const float r = rsqrtf(tot / (float)R + eps);
  uint16_t* out = h + (size_t)blockIdx.x * R;
  for (int i = threadIdx.x; i < R; i += kNormThreads) {
    const float gi = __uint_as_float((uint32_t)gamma[i] << 16);
    out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(row[i] * r * gi));
  }
}

template <bool kAtomic>
cudaError_t launch_gemm(const GemmParams& g, const CUtensorMap& wmap, const CUtensorMap& xmap, int features,
                        cudaStream_t s) {
  const size_t smem = gemm_smem_bytes(g.Bp);
  static int configured = 0;
  if ((int)smem > configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(lowrank_gemm_kernel<kAtomic>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = (int)smem;
  }
  lowrank_gemm_kernel<kAtomic><<<dim3(features / 128, g.splits), kGemmThreads, smem, s>>>(g, wmap, xmap);
  return cudaGetLastError();
}

}  // namespace

size_t query_lowrank_gemm_smem_bytes(int Bp) { return gemm_smem_bytes(Bp); }

cudaError_t launch_query_lowrank(const QueryLowrankParams& p, const CUtensorMap& wd_map, const CUtensorMap& x_map,
                                 const CUtensorMap& wu_map, const CUtensorMap& h_map, cudaStream_t s) {
  const int Bp = (p.B + 15) & ~15;
  cudaError_t e = cudaMemsetAsync(p.y, 0, (size_t)p.B * p.rank * sizeof(float), s);
  if (e != cudaSuccess) return e;
  GemmParams g1{p.y, nullptr, p.err, p.budget, p.B, Bp, p.rank, p.d_model, p.splits_down};
  if ((e = launch_gemm<true>(g1, wd_map, x_map, p.rank, s)) != cudaSuccess) return e;
  rmsnorm_kernel<<<p.B, kNormThreads, 0, s>>>(p.y, p.gamma, p.h, p.rank, p.eps);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  GemmParams g2{nullptr, p.q, p.err, p.budget, p.B, Bp, p.n_out, p.rank, 1};
  return launch_gemm<false>(g2, wu_map, h_map, p.n_out, s);
}

}  // namespace mfa
