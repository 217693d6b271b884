// kv_append.cu -- in-place KV append into the paged cache (bf16 copy or
// per-token E4M3 or E2M1 quantisation), advancing the device-owned length
// counter.
//
// Semantics: "DuckLLM decode fixed-cost reduction" page, sections 7.2 (static
// KV cache written at a fixed slot, never re-materialised) and 7.6 (the append
// offset and the attention length come from one device-owned counter, and the
// attention after an append includes the new token). FP8 storage: "Step-3 is
// Large yet Affordable" (paper summary page), section 7 (8-bit KV, 512 bytes
// per token per layer); one fp32 scale per token (absmax / 448) because the
// pages do not fix the granularity. 4-bit storage: same page, section 5.2 (KV
// kept in 4 bits, attention computed in 8 bits), as OCP MX FP4 (E2M1) codes
// with one fp32 scale per token (absmax / 6), two codes per byte.
#include <cuda_fp8.h>

#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kAppendThreads = 256;  // 8 warps, one token row (K or V) per warp at a time

// Rows are 512 bytes of bf16: lane i holds elements [8i, 8i + 8).
// Quantise one bf16 row to E4M3 with scale = absmax / 448 (1 for a zero row).
// Divisions are IEEE round-to-nearest; the conversion rounds to nearest even
// and saturates to +-448.
__device__ __forceinline__ void quantise_row_e4m3(const uint4 raw, uint8_t* __restrict__ dst,
                                                  float* __restrict__ scale_out, int lane) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t packed[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float2 pr = make_float2(__fdiv_rn(x[4 * i + 2 * j], s), __fdiv_rn(x[4 * i + 2 * j + 1], s));
      const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(pr, __NV_SATFINITE, __NV_E4M3);
      word |= (uint32_t)c2 << (16 * j);
    }
    packed[i] = word;
  }
  reinterpret_cast<uint2*>(dst)[lane] = make_uint2(packed[0], packed[1]);
  if (lane == 0) *scale_out = s;
}

// Nearest E2M1 code to y, a tie going to the code with mantissa bit 0, beyond 6
// saturating; the sign is kept (sign bit 3, also on zero). The candidate
// magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6: the comparisons are against the
// midpoints, each tie resolved toward the even code.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t c = a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
                   : a <= 2.5f ? 4u : a < 3.5f ? 5u : a <= 5.0f ? 6u : 7u;
  return c | (signbit(y) ? 8u : 0u);
}

// Quantise one bf16 row to E2M1 with scale = absmax / 6 (1 for a zero row):
// lane i packs elements [8i, 8i + 8) into 4 bytes, element 2k in the low nibble.
__device__ __forceinline__ void quantise_row_e2m1(const uint4 raw, uint8_t* __restrict__ dst,
                                                  float* __restrict__ scale_out, int lane) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = (amax > 0.0f) ? __fdiv_rn(amax, 6.0f) : 1.0f;
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) word |= e2m1_code(__fdiv_rn(x[i], s)) << (4 * i);
  reinterpret_cast<uint32_t*>(dst)[lane] = word;
  if (lane == 0) *scale_out = s;
}

constexpr int kMaxStagedPages = 64;  // page ids validated once and kept in shared memory

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(AppendParams p) {
  __shared__ int s_start;
  __shared__ int s_bad;
  __shared__ int s_pages[kMaxStagedPages];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kAppendThreads / 32;
  pdl_launch_dependents();  // the decode kernel may run its prologue meanwhile
  pdl_wait_prior_grid();    // launched early too: whatever ran before must be complete and visible
  // the row of this warp's first work item (token t = i / 2, K or V) is read
  // while warp 0 looks up and checks where the tokens go
  const int first = warp;
  uint4 first_row = make_uint4(0u, 0u, 0u, 0u);
  if (first < 2 * p.n_new) {
    const uint16_t* src = ((first & 1) ? p.v_new : p.k_new) + ((size_t)b * p.n_new + (first >> 1)) * kHeadDim;
    first_row = __ldg(reinterpret_cast<const uint4*>(src) + lane);
  }
  if (warp == 0) {
    const int start = p.seq_lens[b];
    const long long cap = (long long)p.max_pages * kPageSize;
    bool bad_cap = start < 0 || (long long)start + p.n_new > cap;
    bool bad_page = false;
    if (!bad_cap) {
      // every page id the new tokens land in is checked before anything is written
      const int pg_first = start / kPageSize, pg_last = (start + p.n_new - 1) / kPageSize;
      for (int pg = pg_first + lane; pg <= pg_last; pg += 32) {
        const int page = p.page_table[(size_t)b * p.max_pages + pg];
        if (page < 0 || page >= p.num_pages) bad_page = true;
        if (pg - pg_first < kMaxStagedPages) s_pages[pg - pg_first] = page;
      }
      bad_page = __any_sync(0xffffffffu, bad_page);
    }
    if (lane == 0) {
      if (bad_cap) raise_error(p.err, MFA_DEVERR_CAPACITY);
      if (bad_page) raise_error(p.err, MFA_DEVERR_PAGE);
      s_bad = (bad_cap || bad_page) ? 1 : 0;
      s_start = start;
    }
  }
  __syncthreads();
  if (s_bad) return;
  const int start = s_start;
  const int pg_first = start / kPageSize;
  for (int i = warp; i < 2 * p.n_new; i += kWarps) {
    const int t = i >> 1;
    const bool is_v = i & 1;
    const int pos = start + t;
    const int pg = pos / kPageSize;
    const int page = (pg - pg_first < kMaxStagedPages) ? s_pages[pg - pg_first]
                                                        : p.page_table[(size_t)b * p.max_pages + pg];
    const size_t slot = (size_t)page * kPageSize + (pos % kPageSize);
    const uint16_t* src = (is_v ? p.v_new : p.k_new) + ((size_t)b * p.n_new + t) * kHeadDim;
    const uint4 row = (i == first) ? first_row : __ldg(reinterpret_cast<const uint4*>(src) + lane);
    if (p.fmt == kKvE2M1) {
      uint8_t* dst = static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + slot * (kHeadDim / 2);
      float* sc = (is_v ? p.v_scale : p.k_scale) + slot;
      quantise_row_e2m1(row, dst, sc, lane);
    } else if (p.fmt == kKvE4M3) {
      uint8_t* dst = static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + slot * kHeadDim;
      float* sc = (is_v ? p.v_scale : p.k_scale) + slot;
      quantise_row_e4m3(row, dst, sc, lane);
    } else {
      uint16_t* dst = static_cast<uint16_t*>(is_v ? p.v_cache : p.k_cache) + slot * kHeadDim;
      reinterpret_cast<uint4*>(dst)[lane] = row;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) p.seq_lens[b] = start + p.n_new;
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  return launch_pdl(kv_append_kernel, dim3(p.B), dim3(kAppendThreads), 0, stream, p);
}

}  // namespace mfa
