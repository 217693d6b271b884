// decode_split_simt.cu -- split-KV MFA decode on the CUDA cores (bf16 cache,
// or FP8 E4M3 cache with per-token scales).
//
// Work partition: the pages of all sequences are cut into `grid` equal,
// contiguous ranges (see mfa_plan_decode); CTA c walks its range and, for
// every sequence it touches, writes one partial result (attention over those
// pages, normalised, plus its natural-log LSE) into slot c + b. The LSE
// combine kernel merges the partials.
//
// Inside a CTA, warp w owns heads [8w, 8w + 8) and lane i owns dimensions
// [8i, 8i + 8): a logit is a warp-wide sum, and the softmax runs online in
// fp32 (the "DuckLLM decode fixed-cost reduction" page, section 7.6, found
// that fp32 intermediates are required in its decode-context kernel).
#include <cuda_fp8.h>

#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kSimtThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Dimensions [8 lane, 8 lane + 8) of one cached E4M3 row, dequantised to fp32.
__device__ __forceinline__ void load_row_fp8(const uint8_t* __restrict__ cache, const float* __restrict__ scales,
                                             size_t row, int lane, float* x) {
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(cache + row * kHeadDim) + lane);
  const float s = __ldg(scales + row);
  const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __nv_fp8x2_storage_t c2 = (__nv_fp8x2_storage_t)((w[i] >> (16 * j)) & 0xFFFFu);
      const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(c2, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      x[4 * i + 2 * j] = f.x * s;
      x[4 * i + 2 * j + 1] = f.y * s;
    }
  }
}

// Dimensions [8 lane, 8 lane + 8) of one cached bf16 row, widened to fp32.
__device__ __forceinline__ void load_row_bf16(const uint16_t* __restrict__ cache, size_t row, int lane, float* x) {
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(cache + row * kHeadDim) + lane);
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(kSimtThreads) decode_split_simt_kernel(DecodeParams p) {
  extern __shared__ int smem_i[];
  int* s_len = smem_i;
  int* s_prefix = smem_i + p.B;
  pdl_wait_prior_grid();    // previous kernel (the KV append) complete
  pdl_launch_dependents();  // the combine may be scheduled; it waits for this grid
  build_page_prefix(p.seq_lens, p.B, p.max_pages * kPageSize, p.err, s_len, s_prefix);
  const long long P = s_prefix[p.B];
  const int c = blockIdx.x, G = p.grid;
  const long long lo = cta_page_lo(c, P, G), hi = cta_page_lo(c + 1, P, G);
  if (lo >= hi) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = warp * 8;
  const float c2 = p.scale * kLog2e;
  for (int b = seq_of_page(s_prefix, p.B, lo); b < p.B && s_prefix[b] < hi; ++b) {
    const long long sp0 = s_prefix[b], sp1 = s_prefix[b + 1];
    if (sp1 == sp0) continue;
    const int pg0 = (int)(max(sp0, lo) - sp0), pg1 = (int)(min(sp1, hi) - sp0);
    const int L = s_len[b];
    float q[8][8], o[8][8], m[8], l[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)b * kHeads + h0 + h) * kHeadDim) + lane);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        q[h][2 * i] = __uint_as_float(w[i] << 16);
        q[h][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) o[h][i] = 0.0f;
      m[h] = -INFINITY;
      l[h] = 0.0f;
    }
    for (int pg = pg0; pg < pg1; ++pg) {
      int page = p.page_table[(size_t)b * p.max_pages + pg];
      if (page < 0 || page >= p.num_pages) {
        raise_error(p.err, MFA_DEVERR_PAGE);
        page = 0;
      }
      const int ntok = min(kPageSize, L - pg * kPageSize);
      for (int t = 0; t < ntok; ++t) {
        const size_t row = (size_t)page * kPageSize + t;
        float k[8], v[8];
        if constexpr (kFp8) {
          load_row_fp8(static_cast<const uint8_t*>(p.k_cache), p.k_scale, row, lane, k);
          load_row_fp8(static_cast<const uint8_t*>(p.v_cache), p.v_scale, row, lane, v);
        } else {
          load_row_bf16(static_cast<const uint16_t*>(p.k_cache), row, lane, k);
          load_row_bf16(static_cast<const uint16_t*>(p.v_cache), row, lane, v);
        }
        float s[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          float acc = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) acc = fmaf(q[h][i], k[i], acc);
          s[h] = acc;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int h = 0; h < 8; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], off);
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float x = s[h] * c2;
          const float mn = fmaxf(m[h], x);
          const float alpha = exp2f(m[h] - mn);
          const float pr = exp2f(x - mn);
          l[h] = l[h] * alpha + pr;
#pragma unroll
          for (int i = 0; i < 8; ++i) o[h][i] = fmaf(o[h][i], alpha, pr * v[i]);
          m[h] = mn;
        }
      }
    }
    const size_t slot = (size_t)c + b;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float inv = 1.0f / l[h];
      float* dst = p.part_o + (slot * kHeads + h0 + h) * kHeadDim + lane * 8;
      reinterpret_cast<float4*>(dst)[0] = make_float4(o[h][0] * inv, o[h][1] * inv, o[h][2] * inv, o[h][3] * inv);
      reinterpret_cast<float4*>(dst)[1] = make_float4(o[h][4] * inv, o[h][5] * inv, o[h][6] * inv, o[h][7] * inv);
      if (lane == 0) p.part_lse[slot * kHeads + h0 + h] = (m[h] + log2f(l[h])) * kLn2;
    }
  }
}

}  // namespace

cudaError_t launch_decode_split_simt(const DecodeParams& p, bool fp8, cudaStream_t stream) {
  const size_t smem = sizeof(int) * (2 * (size_t)p.B + 1);
  if (fp8) return launch_pdl(decode_split_simt_kernel<true>, dim3(p.grid), dim3(kSimtThreads), smem, stream, p);
  return launch_pdl(decode_split_simt_kernel<false>, dim3(p.grid), dim3(kSimtThreads), smem, stream, p);
}

}  // namespace mfa
