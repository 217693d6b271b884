// lse_combine.cu -- merges the split-KV partial results of each sequence.
//
// Each partial s of sequence b holds O_s = attention over its own pages
// (already normalised) and lse_s = ln of its softmax denominator. With
// M = max_s lse_s and w_s = exp(lse_s - M):
//     out = sum_s w_s O_s / sum_s w_s,   lse = M + ln sum_s w_s,
// which equals attention over the whole sequence (the splits partition the
// softmax sum exactly).
//
// With several query tokens per sequence (multi-token decode) every token t
// is merged on its own, over the partials of its token group (a slot holds
// [token of the group][head][dim]); token t of a sequence of length L sees the
// first L - (n_query - 1 - t) positions.
//
// One CTA of 256 threads per (sequence, token, group of kH heads); kH is chosen from
// the batch so that small batches still spread over the SMs. Per head,
// 256 / kH threads split the 256 output dimensions (4 or 8 each) and, when
// there are more than 64 of them, also the partials (S interleaved subsets,
// summed through shared memory at the end). Warp i < kH turns the partial
// LSEs of head i into normalised weights (maximum and sum by warp shuffles).
// The first round of partial-O loads is issued before the weights are known,
// so the LSE and O reads overlap; a value read from a slot whose weight turns
// out to be 0 (an empty CTA range, whose slot may hold data of an earlier
// call, or an underflowed exponent) is discarded by a select, never scaled.
#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kRound = 4;  // partials per thread and round (loads in flight)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ bool cta_range_nonempty(int c, long long C, int G) {
  return cta_cost_lo(c, C, G) < cta_cost_lo(c + 1, C, G);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int kH>
struct CombineShape {
  static constexpr int kThreadsPerHead = kCombineThreads / kH;
  static constexpr int kDimThreads = kThreadsPerHead < 64 ? kThreadsPerHead : 64;  // threads across the 256 dims
  static constexpr int kVec = kHeadDim / (4 * kDimThreads);                      // float4s per thread
  static constexpr int kSubsets = kThreadsPerHead / kDimThreads;                 // partial subsets per head
  static_assert(kDimThreads * kVec * 4 == kHeadDim, "dims per thread");
  static_assert(kH <= 8, "weights are computed by warps 0 .. kH-1");
};

// At most 64 registers a thread, so four CTAs share an SM (608 on 152 SMs), which holds the whole
// grid of batches up to 64 sequences in one wave (at 80 registers, three a SM, B = 64 took two).
template <int kH>
__global__ void __launch_bounds__(kCombineThreads, 4) lse_combine_kernel(DecodeParams p) {
  using Sh = CombineShape<kH>;
  extern __shared__ int smem_i[];
  int* s_len = smem_i;
  int* s_cost = smem_i + p.B;
  float* s_w = reinterpret_cast<float*>(smem_i + 2 * p.B + 1);  // [kH][G] normalised weights
  __shared__ float s_lse[kH];
  __shared__ float4 s_acc[Sh::kSubsets > 1 ? kCombineThreads * Sh::kVec : 1];
  // seq_lens is final before the split kernel starts; the partials are not
  build_cost_prefix(p.seq_lens, p.B, p.max_pages * kPageSize, nullptr, p.piece_cost, s_len, s_cost, p.n_blocks,
                    p.max_blocks);
  const int nq = p.n_query;
  const int b = blockIdx.y / nq, tq = blockIdx.y % nq;  // sequence, query token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = threadIdx.x / Sh::kThreadsPerHead;
  const int r = threadIdx.x % Sh::kThreadsPerHead;
  const int dt = r % Sh::kDimThreads, sub = r / Sh::kDimThreads;
  const int h = blockIdx.x * kH + hl;
  // token groups: the split ran q_groups copies of a partition into G ranges; token tq sits in group grp
  // at position t, and range c's partial of it is row ((c + b) * q_groups + grp) * q_per_cta + t
  const int P = p.q_groups, kq = p.q_per_cta, grp = tq / kq, t = tq % kq;
  const int G = p.grid / P;
  const long long C = s_cost[p.B];
  const int np = pages_of_len(s_len[b]);
  uint16_t* out = p.out + ((size_t)blockIdx.y * kHeads + h) * kHeadDim;
  if (np == 0 || s_len[b] - (nq - 1 - tq) <= 0) {  // empty sequence, or a token that sees no position
    if (sub == 0) {
#pragma unroll
      for (int v = 0; v < Sh::kVec; ++v) reinterpret_cast<uint2*>(out)[dt * Sh::kVec + v] = make_uint2(0u, 0u);
      if (dt == 0) p.lse[(size_t)blockIdx.y * kHeads + h] = -INFINITY;
    }
    return;
  }
  // the CTAs holding the first and the last page of b; every CTA between
  // them with a non-empty range holds a piece of b
  const long long first = (long long)s_cost[b] + p.piece_cost;
  const int c_first = cta_of_cost(first, C, G);
  const int n = cta_of_cost(first + np - 1, C, G) - c_first + 1;
  const size_t kSlotStride = (size_t)P * kq * kHeads * kHeadDim;  // floats from one range's slot to the next
  const float* src =
      p.part_o + ((((size_t)(c_first + b) * P + grp) * kq + t) * kHeads + h) * kHeadDim + 4 * Sh::kVec * dt;

  pdl_wait_prior_grid();
  // first round of O loads (partials sub, sub + S, ...), before the weights
  float4 x[kRound][Sh::kVec];
#pragma unroll
  for (int u = 0; u < kRound; ++u) {
    const int i = sub + u * Sh::kSubsets;
#pragma unroll
    for (int v = 0; v < Sh::kVec; ++v)
      x[u][v] = (i < n) ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)i * kSlotStride) + v)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (warp < kH) {
    const int hh = blockIdx.x * kH + warp;
    float* w = s_w + warp * G;
    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32) {
      const int c = c_first + i;
      const float v =
          cta_range_nonempty(c, C, G) ? __ldcg(p.part_lse + ((((size_t)(c + b) * P + grp) * kq + t) * kHeads + hh))
                                      : -INFINITY;
      w[i] = v;
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.0f;
    for (int i = lane; i < n; i += 32) {
      const float e = exp2f((w[i] - mx) * kLog2e);  // 0 for an empty range
      w[i] = e;
      den += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = 1.0f / den;
    for (int i = lane; i < n; i += 32) w[i] *= inv;
    if (lane == 0) s_lse[warp] = mx + log2f(den) * kLn2;
  }
  __syncthreads();

  const float* w = s_w + hl * G;
  float4 acc[Sh::kVec];
#pragma unroll
  for (int v = 0; v < Sh::kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < n; i0 += kRound * Sh::kSubsets) {
    if (i0 > 0) {
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        const int i = i0 + sub + u * Sh::kSubsets;
#pragma unroll
        for (int v = 0; v < Sh::kVec; ++v)
          x[u][v] = (i < n && w[i] != 0.0f)
                        ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)i * kSlotStride) + v)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int i = i0 + sub + u * Sh::kSubsets;
      const float wi = (i < n) ? w[i] : 0.0f;
      if (wi != 0.0f) {
#pragma unroll
        for (int v = 0; v < Sh::kVec; ++v) {
          acc[v].x += wi * x[u][v].x;
          acc[v].y += wi * x[u][v].y;
          acc[v].z += wi * x[u][v].z;
          acc[v].w += wi * x[u][v].w;
        }
      }
    }
  }
  if constexpr (Sh::kSubsets > 1) {
#pragma unroll
    for (int v = 0; v < Sh::kVec; ++v) s_acc[threadIdx.x * Sh::kVec + v] = acc[v];
    __syncthreads();
    if (sub == 0) {
      for (int k = 1; k < Sh::kSubsets; ++k) {
#pragma unroll
        for (int v = 0; v < Sh::kVec; ++v) {
          const float4 y = s_acc[(threadIdx.x + k * Sh::kDimThreads) * Sh::kVec + v];
          acc[v].x += y.x;
          acc[v].y += y.y;
          acc[v].z += y.z;
          acc[v].w += y.w;
        }
      }
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int v = 0; v < Sh::kVec; ++v)
      reinterpret_cast<uint2*>(out)[dt * Sh::kVec + v] =
          make_uint2(pack_bf16x2(acc[v].x, acc[v].y), pack_bf16x2(acc[v].z, acc[v].w));
    if (dt == 0) p.lse[(size_t)blockIdx.y * kHeads + h] = s_lse[hl];
  }
}

template <int kH>
cudaError_t launch_kh(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(kHeads / kH, p.B * p.n_query);
  const size_t smem = sizeof(int) * (2 * (size_t)p.B + 1) + sizeof(float) * (size_t)kH * p.grid;
  return launch_pdl(lse_combine_kernel<kH>, grid, dim3(kCombineThreads), smem, stream, p);
}

}  // namespace

// Heads per CTA: the grid (64 / kH) x B should be about 2-4 CTAs per SM, so
// fewer heads per CTA (and partial subsets) for small batches.
cudaError_t launch_lse_combine(const DecodeParams& p, cudaStream_t stream) {
  if (p.B <= 8) return launch_kh<1>(p, stream);
  if (p.B <= 16) return launch_kh<2>(p, stream);
  if (p.B <= 48) return launch_kh<4>(p, stream);
  return launch_kh<8>(p, stream);
}

}  // namespace mfa
