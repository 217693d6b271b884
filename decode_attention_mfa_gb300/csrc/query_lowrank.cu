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
// TMA copies through an mbarrier ring and prefetches the weight chunks beyond
// the ring into L2, one thread of warp 5 issues the MMAs. Every wait is bounded.
//
// Two launches, chained by programmatic dependent launch:
//   down (kDown): the K of W_down is split over the CTAs of a feature block
//     (its 16 feature blocks alone would leave most SMs idle). Each CTA stages
//     its [B x 128] fp32 sum in shared memory and adds it into y with one TMA
//     bulk reduce-add; the last CTA of the block to arrive (a byte counter in
//     the workspace header) reads the finished y block, writes
//     h' = bf16(y * gamma) and the block's sums of y^2 per row, and zeroes its
//     y block for the next call.
//   up: q[b] = bf16(r_b * (h' W_up)[b]) with r_b = 1 / sqrt(mean(y_b^2) + eps)
//     -- the row scale of the RMSNorm commutes with the product and is applied
//     in the epilogue. W_up does not depend on the down launch, so the up CTAs
//     fill their ring with W_up tiles and prefetch more of it into L2 while
//     the down launch runs, and wait for it only before loading h'.
#include <algorithm>

#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kGemmThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kDownStages = 4;         // the down launch's ring (>= 4: it also stages the [B x 128] fp32 sum)
constexpr int kUpPrefetch = 12;        // W_up chunks read ahead into L2 beyond the ring
constexpr int kDownGroup = 4;          // feature blocks per K order (down)
constexpr int kUpGroup = 16;           // feature blocks per K order (up)
constexpr int kKChunk = 64;            // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kWStageBytes = 16384;    // [64 k rows x 128 features] bf16
constexpr int kTmemColsGemm = 256;     // D: up to 256 batch columns
constexpr int kEpiThreads = 128;       // warps 0-3
// dynamic shared memory of one down CTA plus one up CTA, so that both fit on one SM
constexpr size_t kPairSmemBudget = 220 * 1024;

struct GemmParams {
  float* y;                 // down: [R/128][B][128] fp32 sums (zero between calls)
  uint16_t* h;              // down out, up operand: [B][R] bf16 h' = bf16(y * gamma)
  float* ssq;               // down out, up in: [R/128][B] sums of y^2 per feature block
  const uint16_t* gamma;    // [R] bf16 bits
  uint32_t* counters;       // down: one byte per feature block (arrivals)
  uint16_t* out;            // up: q [B][N] bf16 bits
  uint32_t* err;
  uint64_t budget;
  float eps;
  int B, Bp, N, K, splits, stages, prefetch, rank;
  int group;                // feature blocks that walk their K range in the same order (see chunk rotation)
};

__host__ __device__ constexpr uint32_t x_stage_bytes(int Bp) { return (uint32_t)Bp * 128u; }
__host__ __device__ constexpr uint32_t gemm_stage_bytes(int Bp) {
  return ((uint32_t)kWStageBytes + x_stage_bytes(Bp) + 1023u) & ~1023u;
}
__host__ __device__ constexpr size_t gemm_smem_bytes(int Bp, int stages) {
  return 1024 + (size_t)stages * gemm_stage_bytes(Bp);
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}
// dst[i] += src[i] for `bytes` / 4 floats, performed at L2 by the TMA unit; returns once the adds are complete.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

template <bool kDown>
__global__ void __launch_bounds__(kGemmThreads, 1)
    lowrank_gemm_kernel(const __grid_constant__ GemmParams g, const __grid_constant__ CUtensorMap wmap,
                        const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag, last_flag;
  __shared__ float row_scale[kMaxQueryBatch];
  const uint32_t raw = smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = gemm_stage_bytes(g.Bp);
  const int S = g.stages;
  const int chunks = g.K / kKChunk;
  const int c0 = (int)((long long)blockIdx.y * chunks / g.splits);
  const int c1 = (int)((long long)(blockIdx.y + 1) * chunks / g.splits);
  const int n = c1 - c0;
  const int fb = blockIdx.x, f0 = fb * 128;
  // Every feature block reads the same X tile at each K step. Walking K in lockstep would send all of
  // them to the same 4 KB of L2 at once; instead each group of g.group blocks starts at its own offset
  // of the CTA's K range (the sum is order-independent up to fp32 rounding).
  const int groups = (int)((gridDim.x + g.group - 1) / g.group);
  const int rot = n > 0 ? (int)((long long)(fb / g.group) * n / groups) % n : 0;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kMaxStages]);
  const uint32_t done = smem_u32(&bars[2 * kMaxStages]);
  volatile int* abort = &abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
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
  if constexpr (kDown) {
    // x and the weights may come from the previous kernel: wait for it, then let the up launch start
    pdl_wait_prior_grid();
    pdl_launch_dependents();
  } else {
    // whatever follows may be scheduled once every CTA of this grid is resident; its own grid dependency
    // wait still covers this grid's results
    pdl_launch_dependents();
  }

  if (warp == 4) {
    if (lane == 0) {  // producer: W tile (streamed once) and X tile (re-read by every feature block)
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      const uint32_t tx = (uint32_t)kWStageBytes + x_stage_bytes(g.Bp);
      auto krow = [&](int i) { return (c0 + (i + rot) % n) * kKChunk; };  // K row of the i-th chunk
      auto load_w = [&](int i) {
        const uint32_t dst = base + (i % S) * sb, bar = full0 + 8 * (i % S);
        tma_load_2d(dst, &wmap, f0, krow(i), bar, pol_w);
        tma_load_2d(dst + 8192, &wmap, f0 + 64, krow(i), bar, pol_w);
      };
      auto load_x = [&](int i) {
        tma_load_2d(base + (i % S) * sb + kWStageBytes, &xmap, krow(i), 0, full0 + 8 * (i % S), pol_x);
      };
      auto prefetch_w = [&](int i) {
        tma_prefetch_2d(&wmap, f0, krow(i));
        tma_prefetch_2d(&wmap, f0 + 64, krow(i));
      };
      // The ring's first copies go first (the TMA unit works through its queue in order), then the
      // read-ahead of the following weight chunks into L2.
      const int pre = min(n, S);
      int pf = pre;  // next chunk to read ahead into L2
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(full0 + 8 * i, tx);
        load_w(i);
        if constexpr (kDown) load_x(i);
      }
      for (; pf < min(n, pre + g.prefetch); ++pf) prefetch_w(pf);
      if constexpr (!kDown) {
        // the weights do not depend on the down launch: the ring is full and the read-ahead issued
        pdl_wait_prior_grid();  // h' is the down launch's output
        for (int k = 0; k < pre; ++k) load_x(k);
      }
      int i = pre;
      for (; i < n; ++i) {
        const int s = i % S, ph = i / S;
        if (!mbar_wait(empty0 + 8 * s, (ph & 1) ^ 1, g.budget, abort, g.err)) break;
        mbar_arrive_expect_tx(full0 + 8 * s, tx);
        load_w(i);
        load_x(i);
        if (pf < n) prefetch_w(pf++);
      }
      // every copy this thread issued must land before the CTA exits
      for (int k = (i > S ? i - S : 0); k < i; ++k)
        (void)mbar_wait(full0 + 8 * (k % S), (k / S) & 1, g.budget, nullptr, g.err);
    }
  } else if (warp == 5) {
    if (lane == 0 && n > 0) {  // MMA issue: 4 MMAs of K=16 per stage
      const uint32_t idesc = idesc_f16(128, g.Bp, 1, 1, 0);  // bf16; A (W^T) MN-major, B (X) K-major
      for (int i = 0; i < n; ++i) {
        const int s = i % S, ph = i / S;
        if (!mbar_wait(full0 + 8 * s, ph & 1, g.budget, abort, g.err)) break;
        tc_fence_after();
        const uint32_t a = base + s * sb, b = a + kWStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tmem, smem_desc_sw128(a + kk * 2048, 8192, 1024), smem_desc_sw128(b + kk * 32, 16, 1024), idesc,
                 (i | kk) != 0);
        tc_commit(empty0 + 8 * s);
      }
      tc_commit(done);  // also tracks the MMAs of an abandoned range, so TMEM is quiet before release
    }
  } else {  // warps 0-3: lane = feature f0 + 32 warp + lane; TMEM columns = batch entries
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const int fl = 32 * warp + lane;
    if constexpr (kDown) {
      float* stage = reinterpret_cast<float*>(dyn_smem + (base - raw));  // [B][128] fp32, over the idle ring
      if (n > 0 && mbar_wait(done, 0, g.budget, abort, g.err)) {
        tc_fence_after();
        for (int j = 0; j < g.Bp; j += 32) {
          float v[32];
          tmem_ld32(tmem + lane_base + j, v);
          tc_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u)
            if (j + u < g.B) stage[(j + u) * 128 + fl] = v[u];
        }
        fence_proxy_async_smem();
      }
      epi_sync();
      if (threadIdx.x == 0 && n > 0 && *abort == 0)
        bulk_reduce_add_f32(g.y + (size_t)fb * g.B * 128, base, (uint32_t)g.B * 512u);
    } else {
      pdl_wait_prior_grid();  // the sums of y^2 come from the down launch
      const int nfb = g.rank / 128;
      for (int b = threadIdx.x; b < g.B; b += kEpiThreads) {
        float ss = 0.0f;
        for (int k = 0; k < nfb; ++k) ss += __ldcg(g.ssq + (size_t)k * g.B + b);
        row_scale[b] = rsqrtf(ss / (float)g.rank + g.eps);
      }
      epi_sync();
      if (n > 0 && mbar_wait(done, 0, g.budget, abort, g.err)) {
        tc_fence_after();
        const int f = f0 + fl;
        for (int j = 0; j < g.Bp; j += 32) {
          float v[32];
          tmem_ld32(tmem + lane_base + j, v);
          tc_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int b = j + u;
            if (b < g.B) g.out[(size_t)b * g.N + f] = __bfloat16_as_ushort(__float2bfloat16_rn(v[u] * row_scale[b]));
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

  if constexpr (kDown) {
    // Every CTA arrives, even one that gave up (its sum is missing and the error word says so), so the
    // counter returns to zero and the block's y is zeroed whatever happened.
    if (threadIdx.x == 0) {
      const int shift = 8 * (fb & 3);
      uint32_t old;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                   : "=r"(old)
                   : "l"(g.counters + (fb >> 2)), "r"(1u << shift)
                   : "memory");
      const bool last = (int)((old >> shift) & 0xffu) == g.splits - 1;
      if (last) atomicSub(g.counters + (fb >> 2), (uint32_t)g.splits << shift);
      last_flag = last;
    }
    __syncthreads();
    if (last_flag) {
      __threadfence();  // every thread: the other CTAs' sums are visible (thread 0 acquired them)
      // finish the block: h' = bf16(y * gamma), sums of y^2 per row, y back to zero. Warp w takes rows
      // w, w + 6, ...; lane l features 4l .. 4l + 3 of the block.
      float4* yb = reinterpret_cast<float4*>(g.y + (size_t)fb * g.B * 128);
      const uint16_t* gm = g.gamma + f0 + 4 * lane;
      const float ga = __uint_as_float((uint32_t)gm[0] << 16), gb = __uint_as_float((uint32_t)gm[1] << 16);
      const float gc = __uint_as_float((uint32_t)gm[2] << 16), gd = __uint_as_float((uint32_t)gm[3] << 16);
      constexpr int kWarps = kGemmThreads / 32, kBatch = 8;
      for (int b0 = warp; b0 < g.B; b0 += kWarps * kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int b = b0 + k * kWarps;
          if (b < g.B) v[k] = __ldcg(yb + b * 32 + lane);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int b = b0 + k * kWarps;
          if (b < g.B) {
            __stcg(yb + b * 32 + lane, make_float4(0.f, 0.f, 0.f, 0.f));
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v[k].x * ga, v[k].y * gb);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v[k].z * gc, v[k].w * gd);
            uint2 hv;
            hv.x = *reinterpret_cast<const uint32_t*>(&lo);
            hv.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(g.h + (size_t)b * g.N + f0 + 4 * lane) = hv;
            float ss = v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) g.ssq[(size_t)fb * g.B + b] = ss;
          }
        }
      }
    }
  }
}

template <bool kDown>
cudaError_t launch_gemm(const GemmParams& g, const CUtensorMap& wmap, const CUtensorMap& xmap, int features,
                        cudaStream_t s) {
  const size_t smem = gemm_smem_bytes(g.Bp, g.stages);
  // the full carve-out: a down CTA and an up CTA then fit on one SM together (the carve-out an SM runs
  // with is set by the first kernel placed on it)
  static int configured[kTrackedDevices] = {};
  const cudaError_t e = ensure_dynamic_smem(lowrank_gemm_kernel<kDown>, smem, configured, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(lowrank_gemm_kernel<kDown>, dim3(features / 128, g.splits), dim3(kGemmThreads), smem, s, g, wmap,
                    xmap);
}

}  // namespace

size_t query_lowrank_gemm_smem_bytes(int Bp) { return gemm_smem_bytes(Bp, kDownStages); }

cudaError_t launch_query_lowrank(const QueryLowrankParams& p, const CUtensorMap& wd_map, const CUtensorMap& x_map,
                                 const CUtensorMap& wu_map, const CUtensorMap& h_map, cudaStream_t s) {
  const int Bp = (p.B + 15) & ~15;
  GemmParams g1{};
  g1.y = p.y;
  g1.h = p.h;
  g1.ssq = p.ssq;
  g1.gamma = p.gamma;
  g1.counters = p.counters;
  g1.err = p.err;
  g1.budget = p.budget;
  g1.eps = p.eps;
  g1.B = p.B;
  g1.Bp = Bp;
  g1.N = p.rank;
  g1.K = p.d_model;
  g1.splits = p.splits_down;
  g1.stages = kDownStages;
  g1.prefetch = kKChunk * 1024;  // the whole K range of the CTA
  g1.rank = p.rank;
  g1.group = kDownGroup;
  cudaError_t e = launch_gemm<true>(g1, wd_map, x_map, p.rank, s);
  if (e != cudaSuccess) return e;
  // the up launch's ring: as deep as fits beside one down CTA (so both run on an SM at once), at least 2
  const size_t sb = gemm_stage_bytes(Bp);
  const size_t down = gemm_smem_bytes(Bp, kDownStages);
  int up_stages = down + 1024 + 2 * sb <= kPairSmemBudget ? (int)((kPairSmemBudget - down - 1024) / sb) : 2;
  up_stages = std::max(2, std::min(kMaxStages, up_stages));
  while (up_stages > 2 && gemm_smem_bytes(Bp, up_stages) > 227 * 1024) --up_stages;
  GemmParams g2{};
  g2.ssq = p.ssq;
  g2.out = p.q;
  g2.err = p.err;
  g2.budget = p.budget;
  g2.eps = p.eps;
  g2.B = p.B;
  g2.Bp = Bp;
  g2.N = p.n_out;
  g2.K = p.rank;
  g2.splits = 1;
  g2.stages = up_stages;
  g2.prefetch = kUpPrefetch;
  g2.rank = p.rank;
  g2.group = kUpGroup;
  return launch_gemm<false>(g2, wu_map, h_map, p.n_out, s);
}

}  // namespace mfa
