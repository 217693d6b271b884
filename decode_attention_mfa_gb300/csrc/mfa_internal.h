// mfa_internal.h -- constants, kernel parameter blocks and launch entry points
// shared by the host side (mfa_api.cu) and the kernels of libmfa.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mfa.h"

namespace mfa {

constexpr int kHeads = MFA_HEADS;        // query heads sharing one K and one V head
constexpr int kHeadDim = MFA_HEAD_DIM;   // head dimension
constexpr int kPageSize = MFA_PAGE_SIZE; // tokens per cache page
constexpr int kMaxBatch = MFA_MAX_BATCH;
constexpr int kMaxQueryBatch = MFA_MAX_QUERY_BATCH;  // the query path's N = batch (one MMA, <= 256)

// Workspace layout: [header 256 B][partial O: slots x 64 x 256 fp32][partial lse: slots x 64 fp32]
constexpr size_t kWsHeaderBytes = 256;
constexpr size_t kPartialOBytes = (size_t)kHeads * kHeadDim * sizeof(float);
constexpr size_t kPartialLseBytes = (size_t)kHeads * sizeof(float);

// Work partition of the split kernel: besides its pages, every sequence piece
// is charged this many page-equivalents (a CTA pays for loading Q and page
// ids and for writing the partial result of each piece it holds, during which
// its softmax warps stream nothing). Measured per kernel variant (a sweep of
// 1, 2 and 3 on the bf16 workloads): the bf16 kernel's best is 2 (ragged
// 112.8 -> 111.5 us, ctx4k unchanged) and the two-token kernel's 3 (its pieces
// write two partials: mtp4k 41.2 -> 39.4 us). Block gather measured best at 1
// (blocks32k 33.5 against 34.1 us) but keeps the bf16 kernel's charge, so that
// selecting every block splits exactly like the dense call and gives the same
// bits (a parity test relies on it).
constexpr int kPieceCostPages = 2;
constexpr int kPieceCostPagesTwoTokens = 3;
// E4M3: a piece also splits Q into E4M3 terms and finds the largest V scale,
// and a tile (two pages) streams in about half the time of a bf16 tile, so a
// piece is worth more pages.
constexpr int kPieceCostPagesFp8 = 3;

// Cache formats: bf16 rows, E4M3 codes + per-token scale, packed E2M1 codes + per-token scale.
constexpr int kKvBf16 = 0, kKvE4M3 = 1, kKvE2M1 = 2;

struct AppendParams {
  const uint16_t* k_new;  // [B][n_new][256] bf16 bits
  const uint16_t* v_new;
  void* k_cache;          // bf16 or E4M3 pages
  void* v_cache;
  float* k_scale;         // E4M3 only
  float* v_scale;
  const int32_t* page_table;
  int32_t* seq_lens;
  uint32_t* err;
  int n_new, B, max_pages, num_pages;
  int fmt;                // kKvBf16, kKvE4M3 or kKvE2M1
};

struct DecodeParams {
  const uint16_t* q;       // [B][64][256] bf16 bits
  const void* k_cache;     // [num_pages][64][256] bf16 bits or E4M3 codes
  const void* v_cache;
  const float* k_scale;    // [num_pages][64] (E4M3 only)
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  // Block gather (null block_idx: the whole sequence): sequence b attends to
  // the 8-token blocks block_idx[b][0 .. n_blocks[b]) and to its own last block
  // up to its last token; k/v tensor maps then use 8-row boxes.
  const int32_t* block_idx;  // [B][max_blocks]
  const int32_t* n_blocks;   // [B]
  int max_blocks;
  int kv_fp4;              // E4M3 kernel: the cache holds packed E2M1 codes ([num_pages][64][128] bytes)
  uint16_t* out;           // [B][n_query][64][256] bf16 bits
  float* lse;              // [B][n_query][64]
  float* part_o;           // [slots][n_query][64][256]
  float* part_lse;         // [slots][n_query][64]
  uint32_t* err;
  float scale;
  int B, max_pages, num_pages, grid;
  int piece_cost;          // cost units charged per sequence piece (work partition)
  int n_query;             // query tokens per sequence (T, multi-token decode); q is [B][T][64][256]
  // Token groups (multi-token decode): a CTA serves q_per_cta consecutive query tokens (2 on the
  // two-token bf16 kernel, else 1), so the T tokens form q_groups = ceil(T / q_per_cta) groups. The grid
  // is q_groups interleaved copies of the stream-K partition: CTA c works on range c / q_groups of the
  // partition for token group c % q_groups, so the CTAs of one range read the same pages at the
  // same time and the cache comes from HBM about once. Partial slot of (range i, sequence b, group r):
  // (i + b) * q_groups + r, holding q_per_cta tokens.
  int q_per_cta, q_groups;
  uint64_t wait_budget_ns;
};

// Launch with programmatic stream serialisation (the kernel calls
// pdl_wait_prior_grid before it reads anything an earlier kernel writes).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory opt-in (and, with full_carveout, its preferred carve-out to all
// of the unified L1 / shared array) on the current device before a launch that needs `bytes`. The
// attributes belong to each device's context, so `record` keeps the largest value set per device
// ordinal. One process-wide lock covers the check, the attribute calls and the record, so host
// threads that launch with different sizes at once can never lower the opt-in below what another
// launch was promised: the value only ever grows. A device past the record's end reads the
// attribute back and raises it only when needed.
inline std::mutex& smem_attr_mutex() {
  static std::mutex m;
  return m;
}
constexpr int kTrackedDevices = 64;
template <typename... KArgs>
inline cudaError_t ensure_dynamic_smem(void (*kernel)(KArgs...), size_t bytes, int (&record)[kTrackedDevices],
                                       bool full_carveout = false) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(smem_attr_mutex());
  int* rec = (dev >= 0 && dev < kTrackedDevices) ? &record[dev] : nullptr;
  if (rec && (int)bytes <= *rec) return cudaSuccess;
  if (!rec) {
    cudaFuncAttributes a{};
    if ((e = cudaFuncGetAttributes(&a, kernel)) != cudaSuccess) return e;
    if ((int)bytes <= a.maxDynamicSharedSizeBytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && full_carveout)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess && rec) *rec = (int)bytes;
  return e;
}

// Kernel launchers (each returns the launch's cudaError_t).
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_decode_split_tc(const DecodeParams& p, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                   const CUtensorMap& q_map, cudaStream_t stream);
cudaError_t launch_decode_split_tc_fp8(const DecodeParams& p, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                       const CUtensorMap& q_map, cudaStream_t stream);
// Block gather over an E4M3 cache: an instantiation of its own, so the dense kernel's code stays as it is.
cudaError_t launch_decode_split_tc_fp8_blocks(const DecodeParams& p, const CUtensorMap& k_map,
                                              const CUtensorMap& v_map, const CUtensorMap& q_map, cudaStream_t stream);
size_t decode_split_tc_smem_bytes(int B);
size_t decode_split_tc_fp8_smem_bytes(int B);
// Two query tokens per sequence (multi-token decode), bf16 cache.
cudaError_t launch_decode_split_tc_mtp(const DecodeParams& p, const CUtensorMap& k_map, const CUtensorMap& v_map,
                                       const CUtensorMap& q_map, cudaStream_t stream);
size_t decode_split_tc_mtp_smem_bytes(int B);

// Host-side services of mfa_api.cu for other entry points of the library.
void set_last_error_message(const char* msg);
uint64_t current_wait_budget_ns();
cudaError_t launch_lse_combine(const DecodeParams& p, cudaStream_t stream);

// Low-rank query path: y = x W_down (fp32, K split over `splits_down` CTAs per
// feature block), h = bf16(RMSNorm(y) * gamma), q = bf16(h W_up).
constexpr size_t kQueryCounterOffset = 128;  // header bytes 128..255: one arrival byte per feature block
constexpr int kMaxQueryRank = MFA_MAX_QUERY_RANK;  // 128 feature blocks: one arrival byte each
constexpr int kMaxQuerySplits = 128;         // a byte holds every arrival
struct QueryLowrankParams {
  const uint16_t* gamma;   // [rank] bf16 bits
  float* y;                // [rank/128][B][128] fp32 scratch, zero between calls
  uint16_t* h;             // [B][rank] bf16 scratch: bf16(y * gamma)
  float* ssq;              // [rank/128][B] fp32 scratch: sums of y^2 per feature block
  uint32_t* counters;      // arrival bytes in the workspace header
  uint16_t* q;             // [B][n_out] bf16 bits
  uint32_t* err;
  uint64_t budget;
  float eps;
  int B, d_model, rank, n_out, splits_down;
};
// wd_map: W_down [d_model][rank]; x_map: x [B][d_model]; wu_map: W_up [rank][n_out]; h_map: h [B][rank]
// (bf16, 64 x 64 boxes for the weights, 64 x Bp boxes for the activations, 128-byte swizzle).
// Two launches with programmatic stream serialisation.
cudaError_t launch_query_lowrank(const QueryLowrankParams& p, const CUtensorMap& wd_map, const CUtensorMap& x_map,
                                 const CUtensorMap& wu_map, const CUtensorMap& h_map, cudaStream_t stream);
size_t query_lowrank_gemm_smem_bytes(int Bp);
cudaError_t launch_selftest_wait(uint32_t* err, uint64_t budget_ns, cudaStream_t stream);

}  // namespace mfa
