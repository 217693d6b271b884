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
// The partial-O rows come into shared memory by TMA bulk copies issued right
// after the grid dependency wait, so they travel while the LSEs are read and
// the weights formed; a row whose weight turns out to be 0 (an empty CTA
// range, whose slot may hold data of an earlier call, or an underflowed
// exponent) is skipped, never scaled.
#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kCombineThreads = 256;
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

// Partial-O rows staged in shared memory per round: the rows of chunk_bytes / (kH KB) partials, brought
// by TMA bulk copies issued right after the grid dependency wait, while warps 0 .. kH-1 read the LSEs.
// One round covers every partial of the configurations' sequences (4K context: about 6 partials of 4
// heads; 128K context: about 20 of one head), so the merge waits on L2 once.
// Eight heads a CTA take 8 KB a partial: 48 KB keep a sequence of six pieces in one round; four CTAs of
// that size still share an SM.
template <int kH>
__host__ __device__ constexpr int chunk_bytes() { return kH == 8 ? 48 * 1024 : 32 * 1024; }

// At most 64 registers a thread and about 36 KB of shared memory, so four CTAs share an SM (608 on 152
// SMs), which holds the whole grid of batches up to 64 sequences in one wave.
template <int kH>
__global__ void __launch_bounds__(kCombineThreads, 4) lse_combine_kernel(DecodeParams p) {
  using Sh = CombineShape<kH>;
  constexpr int kPartBytes = kH * 1024;            // the kH heads' rows of one partial
  constexpr int kChunkBytes = chunk_bytes<kH>();
  constexpr int kChunk = kChunkBytes / kPartBytes;  // partials per round
  extern __shared__ __align__(128) uint8_t smem_raw[];
  int* s_len = reinterpret_cast<int*>(smem_raw + kChunkBytes);
  int* s_cost = s_len + p.B;
  float* s_w = reinterpret_cast<float*>(s_cost + p.B + 1);  // [kH][G] normalised weights
  __shared__ float s_lse[kH];
  __shared__ float4 s_acc[Sh::kSubsets > 1 ? kCombineThreads * Sh::kVec : 1];
  __shared__ __align__(8) uint64_t s_bar;
  const uint32_t o_base = smem_u32(smem_raw), bar = smem_u32(&s_bar);
  // whatever follows on the stream may be scheduled once every CTA of this grid is resident (its grid
  // dependency wait still covers this grid's results): it then starts as these CTAs leave their SMs,
  // without a launch gap after the last one
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // seq_lens is final before the split kernel starts; the partials are not (ends with a barrier)
  build_cost_prefix(p.seq_lens, p.B, p.max_pages * kPageSize, nullptr, p.piece_cost, s_len, s_cost, p.n_blocks,
                    p.max_blocks);
  const int nq = p.n_query;
  const int b = blockIdx.y / nq, tq = blockIdx.y % nq;  // sequence, query token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = threadIdx.x / Sh::kThreadsPerHead;
  const int r = threadIdx.x % Sh::kThreadsPerHead;
  const int dt = r % Sh::kDimThreads, sub = r / Sh::kDimThreads;
  const int h0 = blockIdx.x * kH, h = h0 + hl;
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
  // the kH heads' rows of range c_first + i's partial (kH KB, contiguous)
  auto part_rows = [&](int i) -> const float* {
    return p.part_o + ((((size_t)(c_first + i + b) * P + grp) * kq + t) * kHeads + h0) * kHeadDim;
  };
  // round k brings partials [k kChunk, min(n, (k + 1) kChunk)); a slot of an empty range holds stale data
  // and is copied all the same (its weight is 0)
  // issued by warp 0, one copy a lane (kChunk <= 32), after lane 0 has announced the round's bytes
  auto issue_round = [&](int k) {
    const int i0 = k * kChunk, cnt = min(kChunk, n - i0);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(cnt * kPartBytes));
    __syncwarp();
    if (lane < cnt) bulk_load(o_base + (uint32_t)(lane * kPartBytes), part_rows(i0 + lane), kPartBytes, bar);
  };
  static_assert(kChunk <= 32, "one copy a lane");

  pdl_wait_prior_grid();
  if (warp == 0) issue_round(0);
  if (warp < kH) {
    const int hh = h0 + warp;
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
  const int rounds = (n + kChunk - 1) / kChunk;
  for (int k = 0; k < rounds; ++k) {
    if (k > 0) {
      __syncthreads();  // every thread is done with the previous round's rows
      if (warp == 0) issue_round(k);
    }
    // bounded; on expiry the error word records it and the output is meaningless, but every thread
    // still reaches the barriers below
    (void)mbar_wait(bar, k & 1, p.wait_budget_ns, nullptr, p.err);
    const int i0 = k * kChunk, cnt = min(kChunk, n - i0);
    for (int i = sub; i < cnt; i += Sh::kSubsets) {
      const float wi = w[i0 + i];
      if (wi != 0.0f) {  // a zero weight (empty range, underflow) is skipped, never scaled
        const float4* row =
            reinterpret_cast<const float4*>(smem_raw + i * kPartBytes + hl * 1024) + dt * Sh::kVec;
#pragma unroll
        for (int v = 0; v < Sh::kVec; ++v) {
          const float4 y = row[v];
          acc[v].x = fmaf(wi, y.x, acc[v].x);
          acc[v].y = fmaf(wi, y.y, acc[v].y);
          acc[v].z = fmaf(wi, y.z, acc[v].z);
          acc[v].w = fmaf(wi, y.w, acc[v].w);
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
  const size_t smem = chunk_bytes<kH>() + sizeof(int) * (2 * (size_t)p.B + 1) + sizeof(float) * (size_t)kH * p.grid;
  static int configured[kTrackedDevices] = {};
  const cudaError_t e = ensure_dynamic_smem(lse_combine_kernel<kH>, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(lse_combine_kernel<kH>, grid, dim3(kCombineThreads), smem, stream, p);
}

}  // namespace

// Heads per CTA: the grid (64 / kH) x rows, rows = B x query tokens, should be about 2-4 CTAs per SM, so
// fewer heads per CTA (and partial subsets) for few rows, and one wave up to 64 rows.
cudaError_t launch_lse_combine(const DecodeParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.n_query;
  if (rows <= 8) return launch_kh<1>(p, stream);
  if (rows <= 16) return launch_kh<2>(p, stream);
  if (rows <= 48) return launch_kh<4>(p, stream);
  return launch_kh<8>(p, stream);
}

}  // namespace mfa
