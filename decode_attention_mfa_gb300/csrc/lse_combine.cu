// lse_combine.cu -- merges the split-KV partial results of each sequence.
//
// Each partial s of sequence b holds O_s = attention over its own pages
// (already normalised) and lse_s = ln of its softmax denominator. With
// M = max_s lse_s and w_s = exp(lse_s - M):
//     out = sum_s w_s O_s / sum_s w_s,   lse = M + ln sum_s w_s,
// which equals attention over the whole sequence (the splits partition the
// softmax sum exactly). One warp per (sequence, head): lane s reads lse_s,
// the maximum and the sum go through warp shuffles, and each lane then
// accumulates 8 of the 256 output dimensions.
#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kCombineThreads = 256;  // 8 warps = 8 heads of one sequence
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ bool cta_range_nonempty(int c, long long C, int G) {
  return cta_cost_lo(c, C, G) < cta_cost_lo(c + 1, C, G);
}

__global__ void __launch_bounds__(kCombineThreads) lse_combine_kernel(DecodeParams p) {
  extern __shared__ int smem_i[];
  int* s_len = smem_i;
  int* s_cost = smem_i + p.B;
  // seq_lens is final before the split kernel starts; the partials are not
  build_cost_prefix(p.seq_lens, p.B, p.max_pages * kPageSize, nullptr, p.piece_cost, s_len, s_cost);
  pdl_wait_prior_grid();
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * (kCombineThreads / 32) + warp;
  const long long C = s_cost[p.B];
  const int G = p.grid;
  const int np = pages_of_len(s_len[b]);
  uint16_t* out = p.out + ((size_t)b * kHeads + h) * kHeadDim;
  if (np == 0) {  // empty sequence
    reinterpret_cast<uint2*>(out)[lane] = make_uint2(0u, 0u);
    reinterpret_cast<uint2*>(out + 128)[lane] = make_uint2(0u, 0u);
    if (lane == 0) p.lse[(size_t)b * kHeads + h] = -INFINITY;
    return;
  }
  // the CTAs holding the first and the last page of b; every CTA between
  // them with a non-empty range holds a piece of b
  const long long first = (long long)s_cost[b] + p.piece_cost;
  const int c_first = cta_of_cost(first, C, G);
  const int c_last = cta_of_cost(first + np - 1, C, G);
  // maximum of the partial LSEs
  float mx = -INFINITY;
  for (int c = c_first + lane; c <= c_last; c += 32)
    if (cta_range_nonempty(c, C, G)) mx = fmaxf(mx, __ldcg(p.part_lse + (size_t)(c + b) * kHeads + h));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  float den = 0.0f;
  for (int base = c_first; base <= c_last; base += 32) {
    const int c = base + lane;
    float w = 0.0f;
    if (c <= c_last && cta_range_nonempty(c, C, G))
      w = exp2f((__ldcg(p.part_lse + (size_t)(c + b) * kHeads + h) - mx) * kLog2e);
    den += w;
    const int n = min(32, c_last - base + 1);
    // four partials per round: their eight loads are in flight together; a slot
    // of an empty CTA range (weight 0) is never read (it may hold stale data)
    for (int j = 0; j < n; j += 4) {
      float wj[4];
      float4 x0[4], x1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wj[u] = __shfl_sync(0xffffffffu, w, (j + u) & 31);
        if (j + u >= n) wj[u] = 0.0f;
        x0[u] = x1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (wj[u] != 0.0f) {
          const float* src = p.part_o + ((size_t)(base + j + u + b) * kHeads + h) * kHeadDim;
          x0[u] = __ldcg(reinterpret_cast<const float4*>(src) + lane);
          x1[u] = __ldcg(reinterpret_cast<const float4*>(src + 128) + lane);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a0.x += wj[u] * x0[u].x; a0.y += wj[u] * x0[u].y; a0.z += wj[u] * x0[u].z; a0.w += wj[u] * x0[u].w;
        a1.x += wj[u] * x1[u].x; a1.y += wj[u] * x1[u].y; a1.z += wj[u] * x1[u].z; a1.w += wj[u] * x1[u].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = 1.0f / den;
  __nv_bfloat162 r0 = __floats2bfloat162_rn(a0.x * inv, a0.y * inv);
  __nv_bfloat162 r1 = __floats2bfloat162_rn(a0.z * inv, a0.w * inv);
  __nv_bfloat162 r2 = __floats2bfloat162_rn(a1.x * inv, a1.y * inv);
  __nv_bfloat162 r3 = __floats2bfloat162_rn(a1.z * inv, a1.w * inv);
  reinterpret_cast<uint2*>(out)[lane] =
      make_uint2(*reinterpret_cast<uint32_t*>(&r0), *reinterpret_cast<uint32_t*>(&r1));
  reinterpret_cast<uint2*>(out + 128)[lane] =
      make_uint2(*reinterpret_cast<uint32_t*>(&r2), *reinterpret_cast<uint32_t*>(&r3));
  if (lane == 0) p.lse[(size_t)b * kHeads + h] = mx + log2f(den) * kLn2;
}

}  // namespace

cudaError_t launch_lse_combine(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(kHeads / (kCombineThreads / 32), p.B);
  const size_t smem = sizeof(int) * (2 * (size_t)p.B + 1);
  return launch_pdl(lse_combine_kernel, grid, dim3(kCombineThreads), smem, stream, p);
}

}  // namespace mfa
