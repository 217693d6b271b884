// mfa_api.cu -- host side of the libmfa C ABI: argument checks, split
// planning and kernel launches. No call here allocates device memory or
// synchronises, except mfa_check_device_errors.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "mfa_internal.h"

namespace {

using namespace mfa;

thread_local std::string g_last_error;
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;
std::atomic<uint64_t> g_wait_budget_ns{2000000000ull};

mfa_status_t fail(mfa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mfa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MFA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------ device info
struct DeviceInfo {
  int num_sms = 0;
  int major = 0, minor = 0;
  bool valid = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

mfa_status_t current_device(int* dev_out, DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MFA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.valid) {
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.valid = true;
  }
  if (dev_out) *dev_out = dev;
  if (info) *info = d;
  if (!(d.major == 10 && d.minor == 3))
    return fail(MFA_ERR_UNSUPPORTED, "libmfa is built for sm_103a; device is sm_%d%d", d.major, d.minor);
  return MFA_OK;
}

// ------------------------------------------------------------ planning
// Grid of the split kernel: one CTA per SM, fewer when there is too little
// work (at least kMinPagesPerCta pages per CTA for the expected lengths).
constexpr int kMinPagesPerCta = 2;

int plan_grid(int batch, int max_len_hint, int num_sms) {
  const long long pages = (long long)batch * ((max_len_hint + kPageSize - 1) / kPageSize);
  long long g = (pages + kMinPagesPerCta - 1) / kMinPagesPerCta;
  if (g < 1) g = 1;
  if (g > num_sms) g = num_sms;
  return (int)g;
}

// Token groups of multi-token decode: a CTA serves q_per_cta query tokens, so the T tokens form
// q_groups = ceil(T / q_per_cta) groups, and the grid holds q_groups copies of a partition of the
// work into `ranges` ranges (q_groups CTAs read each range's pages together). A partial slot holds
// the results of the q_per_cta tokens of its group for one sequence piece.
struct TokenGroups {
  int q_per_cta, q_groups;
};
TokenGroups token_groups(int n_query, bool quantised) {
  TokenGroups g;
  g.q_per_cta = (!quantised && n_query >= 2) ? 2 : 1;
  g.q_groups = (n_query + g.q_per_cta - 1) / g.q_per_cta;
  return g;
}

void fill_plan(int batch, int max_len_hint, int num_sms, mfa_plan_t* plan, TokenGroups tg = {1, 1}) {
  int ranges = plan_grid(batch, max_len_hint, num_sms);
  if (tg.q_groups > 1) ranges = std::max(1, std::min(ranges, num_sms / tg.q_groups));
  plan->grid_ctas = ranges * tg.q_groups;
  plan->partial_slots = (ranges + batch - 1) * tg.q_groups;
  plan->workspace_bytes =
      kWsHeaderBytes + (size_t)plan->partial_slots * tg.q_per_cta * (kPartialOBytes + kPartialLseBytes);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------ TMA descriptors
// Tensor maps are encoded on the host per call (a pure host computation) and
// passed to the kernel as __grid_constant__ parameters, so a captured graph
// keeps them with its node.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

mfa_status_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!g_encode) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  *fn = g_encode;
  return MFA_OK;
}

// 2-D bf16 tensor [rows][256] read in [box_rows x 64 columns] boxes with the
// 128-byte swizzle (128-byte box rows).
mfa_status_t encode_rows_bf16(CUtensorMap* map, const void* base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  mfa_status_t st = get_encoder(&enc);
  if (st != MFA_OK) return st;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MFA_OK;
}

// 2-D bf16 tensor [rows][cols] read in [box_rows x 64 columns] boxes with the
// 128-byte swizzle; rows past the end read as zeros.
mfa_status_t encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  mfa_status_t st = get_encoder(&enc);
  if (st != MFA_OK) return st;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MFA_OK;
}

// Block gather: the bf16 cache [rows][256] viewed as 3-D -- x = 64 columns of
// a 128-byte column block, y = row (512-byte stride), z = column block
// (128-byte stride) -- read in boxes of 8 rows x `zbox` column blocks, which
// land as zbox swizzle atoms of [8 rows x 128 B], one column block after the
// other.
mfa_status_t encode_blocks_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint32_t zbox) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  mfa_status_t st = get_encoder(&enc);
  if (st != MFA_OK) return st;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(kHeadDim / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, 128};
  const cuuint32_t box[3] = {64, 8, zbox};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled (block view) failed (%d)", (int)r);
  return MFA_OK;
}

// Block gather on an E4M3 cache: the cache [rows][256] bytes viewed as 3-D -- x = the 128 bytes of a
// 128-dim half, y = row (256-byte stride), z = half (128-byte stride) -- read in boxes of 8 rows x both
// halves, which land as two swizzle atoms [8 rows x 128 B], half 0 then half 1 (2 KB per block).
mfa_status_t encode_blocks_e4m3(CUtensorMap* map, const void* base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  mfa_status_t st = get_encoder(&enc);
  if (st != MFA_OK) return st;
  const cuuint64_t dims[3] = {128, (cuuint64_t)rows, 2};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim, 128};
  const cuuint32_t box[3] = {128, 8, 2};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled (E4M3 block view) failed (%d)", (int)r);
  return MFA_OK;
}

// 2-D byte tensor [rows][256] (E4M3 codes) read in [64 rows x 128 bytes]
// boxes with the 128-byte swizzle.
mfa_status_t encode_rows_e4m3(CUtensorMap* map, const void* base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  mfa_status_t st = get_encoder(&enc);
  if (st != MFA_OK) return st;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
  const cuuint32_t box[2] = {128, 64};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MFA_OK;
}

// 4-bit cache: 2-D [rows][256] E2M1 codes packed two per byte (128-byte rows)
// read in [64 rows x 128 codes] boxes; TMA expands each 16 codes (8 bytes) to
// 16 bytes of shared memory (8-byte gap), which is the operand layout of the
// 4-bit formats in kind::f8f6f4 MMAs, with the 128-byte swizzle. The box then
// has the shared-memory geometry of a [64 x 128] E4M3 box.
mfa_status_t encode_rows_e2m1(CUtensorMap* map, const void* base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  mfa_status_t st = get_encoder(&enc);
  if (st != MFA_OK) return st;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim / 2};
  const cuuint32_t box[2] = {128, 64};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box,
                         elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MFA_ERR_CUDA, "cuTensorMapEncodeTiled (4-bit) failed (%d)", (int)r);
  return MFA_OK;
}

// ------------------------------------------------------------ common checks
mfa_status_t check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* page_table, const int32_t* seq_lens, const void* out,
                               const float* lse, int batch, int max_pages, int num_pages,
                               int max_len_hint, const void* workspace, size_t workspace_bytes,
                               int num_sms, mfa_plan_t* plan, TokenGroups tg = {1, 1}) {
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out || !lse)
    return fail(MFA_ERR_INVALID_ARG, "null pointer argument");
  if (batch < 1 || batch > kMaxBatch) return fail(MFA_ERR_INVALID_ARG, "batch %d outside [1, %d]", batch, kMaxBatch);
  if (max_pages < 1 || num_pages < 1) return fail(MFA_ERR_INVALID_ARG, "max_pages and num_pages must be >= 1");
  if (max_len_hint < 0) return fail(MFA_ERR_INVALID_ARG, "negative max_len_hint");
  if ((long long)max_pages * kPageSize > 0x7fffffffLL) return fail(MFA_ERR_INVALID_ARG, "max_pages too large");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(seq_lens, 4))
    return fail(MFA_ERR_INVALID_ARG, "misaligned pointer (q, caches, out need 16 bytes)");
  if (!workspace || !aligned(workspace, 256))
    return fail(MFA_ERR_WORKSPACE, "workspace missing or not 256-byte aligned");
  fill_plan(batch, max_len_hint, num_sms, plan, tg);
  if (workspace_bytes < plan->workspace_bytes)
    return fail(MFA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, plan->workspace_bytes);
  return MFA_OK;
}

DecodeParams make_decode_params(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                const float* v_scale, const int32_t* page_table, const int32_t* seq_lens,
                                void* out, float* lse, float scale, int batch, int max_pages, int num_pages,
                                void* workspace, const mfa_plan_t& plan, int n_query = 1, TokenGroups tg = {1, 1}) {
  DecodeParams p{};
  char* ws = static_cast<char*>(workspace);
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.part_o = reinterpret_cast<float*>(ws + kWsHeaderBytes);
  p.part_lse =
      reinterpret_cast<float*>(ws + kWsHeaderBytes + (size_t)plan.partial_slots * tg.q_per_cta * kPartialOBytes);
  p.scale = scale;
  p.B = batch;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.grid = plan.grid_ctas;
  p.piece_cost = kPieceCostPages;
  p.n_query = n_query;
  p.q_per_cta = tg.q_per_cta;
  p.q_groups = tg.q_groups;
  p.wait_budget_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  return p;
}

mfa_status_t append_common(const void* k_new, const void* v_new, int n_new, void* k_cache, void* v_cache,
                           float* k_scale, float* v_scale, int fmt, const int32_t* page_table,
                           int32_t* seq_lens, int batch, int max_pages, int num_pages, void* workspace,
                           void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !seq_lens)
    return fail(MFA_ERR_INVALID_ARG, "null pointer argument");
  if (fmt != kKvBf16 && (!k_scale || !v_scale)) return fail(MFA_ERR_INVALID_ARG, "null scale pointer");
  if (fmt != kKvBf16 && (!aligned(k_scale, 4) || !aligned(v_scale, 4))) return fail(MFA_ERR_INVALID_ARG, "misaligned scales");
  if (batch < 1 || batch > kMaxBatch) return fail(MFA_ERR_INVALID_ARG, "batch %d outside [1, %d]", batch, kMaxBatch);
  if (n_new < 0) return fail(MFA_ERR_INVALID_ARG, "negative n_new");
  if (max_pages < 1 || num_pages < 1) return fail(MFA_ERR_INVALID_ARG, "max_pages and num_pages must be >= 1");
  if ((long long)max_pages * kPageSize > 0x7fffffffLL) return fail(MFA_ERR_INVALID_ARG, "max_pages too large");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(page_table, 4) || !aligned(seq_lens, 4))
    return fail(MFA_ERR_INVALID_ARG, "misaligned pointer (rows and caches need 16 bytes)");
  if (!workspace || !aligned(workspace, 256))
    return fail(MFA_ERR_WORKSPACE, "workspace missing or not 256-byte aligned");
  mfa_status_t st = current_device(nullptr, nullptr);
  if (st != MFA_OK) return st;
  if (n_new == 0) return MFA_OK;
  AppendParams p{};
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.err = static_cast<uint32_t*>(workspace);
  p.n_new = n_new;
  p.B = batch;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.fmt = fmt;
  const cudaError_t e = launch_kv_append(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return MFA_OK;
}

mfa_status_t decode_common(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, bool fp8, const int32_t* page_table, const int32_t* seq_lens,
                           void* out, float* lse, float scale, int batch, int max_pages, int num_pages,
                           int max_len_hint, void* workspace, size_t workspace_bytes, void* stream,
                           int n_query = 1, const int32_t* block_idx = nullptr, const int32_t* n_blocks = nullptr,
                           int max_blocks = 0, int kv_fp4 = 0) {
  DeviceInfo info;
  mfa_status_t st = current_device(nullptr, &info);
  if (st != MFA_OK) return st;
  if (fp8 && (!k_scale || !v_scale)) return fail(MFA_ERR_INVALID_ARG, "null scale pointer");
  if (fp8 && (!aligned(k_scale, 16) || !aligned(v_scale, 16)))
    return fail(MFA_ERR_INVALID_ARG, "misaligned scales (16 bytes needed)");
  mfa_plan_t plan;
  const TokenGroups tg = token_groups(n_query, fp8);
  st = check_decode_args(q, k_cache, v_cache, page_table, seq_lens, out, lse, batch, max_pages, num_pages,
                         max_len_hint, workspace, workspace_bytes, info.num_sms, &plan, tg);
  if (st != MFA_OK) return st;
  DecodeParams p = make_decode_params(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, out, lse,
                                      scale, batch, max_pages, num_pages, workspace, plan, n_query, tg);
  p.piece_cost = fp8 ? kPieceCostPagesFp8 : tg.q_per_cta == 2 ? kPieceCostPagesTwoTokens : kPieceCostPages;
  p.kv_fp4 = kv_fp4;
  p.block_idx = block_idx;
  p.n_blocks = n_blocks;
  p.max_blocks = max_blocks;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (g_prof_start && (e = cudaEventRecordWithFlags(g_prof_start, s, cudaEventRecordExternal)) != cudaSuccess)
    return cuda_fail(e, "profile event record");
  CUtensorMap kmap, vmap, qmap;
  const uint64_t rows = (uint64_t)num_pages * kPageSize;
  if ((st = encode_rows_bf16(&qmap, q, (uint64_t)batch * n_query * kHeads)) != MFA_OK) return st;
  if (fp8) {
    if (kv_fp4) {
      if ((st = encode_rows_e2m1(&kmap, k_cache, rows)) != MFA_OK ||
          (st = encode_rows_e2m1(&vmap, v_cache, rows)) != MFA_OK)
        return st;
    } else if (block_idx) {  // block gather: one 8-row box of both halves per block
      if ((st = encode_blocks_e4m3(&kmap, k_cache, rows)) != MFA_OK ||
          (st = encode_blocks_e4m3(&vmap, v_cache, rows)) != MFA_OK)
        return st;
    } else if ((st = encode_rows_e4m3(&kmap, k_cache, rows)) != MFA_OK ||
               (st = encode_rows_e4m3(&vmap, v_cache, rows)) != MFA_OK) {
      return st;
    }
    e = block_idx ? launch_decode_split_tc_fp8_blocks(p, kmap, vmap, qmap, s) : launch_decode_split_tc_fp8(p, kmap, vmap, qmap, s);
  } else {
    if (block_idx) {  // block gather: one 8-token block per box, K by column-block pairs, V whole
      if ((st = encode_blocks_bf16(&kmap, k_cache, rows, 2)) != MFA_OK ||
          (st = encode_blocks_bf16(&vmap, v_cache, rows, 4)) != MFA_OK)
        return st;
    } else if ((st = encode_rows_bf16(&kmap, k_cache, rows)) != MFA_OK ||
               (st = encode_rows_bf16(&vmap, v_cache, rows)) != MFA_OK) {
      return st;
    }
    e = tg.q_per_cta == 2 ? launch_decode_split_tc_mtp(p, kmap, vmap, qmap, s)
                          : launch_decode_split_tc(p, kmap, vmap, qmap, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode split launch");
  if (g_prof_stop && (e = cudaEventRecordWithFlags(g_prof_stop, s, cudaEventRecordExternal)) != cudaSuccess)
    return cuda_fail(e, "profile event record");
  e = launch_lse_combine(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "lse combine launch");
  return MFA_OK;
}

}  // namespace

namespace mfa {
void set_last_error_message(const char* msg) { g_last_error = msg; }
uint64_t current_wait_budget_ns() { return g_wait_budget_ns.load(std::memory_order_relaxed); }
}  // namespace mfa

extern "C" {

mfa_status_t mfa_plan_decode(int batch, int max_len_hint, int num_sms, mfa_plan_t* plan) {
  if (!plan) return fail(MFA_ERR_INVALID_ARG, "null plan");
  if (batch < 1 || batch > kMaxBatch) return fail(MFA_ERR_INVALID_ARG, "batch %d outside [1, %d]", batch, kMaxBatch);
  if (max_len_hint < 0) return fail(MFA_ERR_INVALID_ARG, "negative max_len_hint");
  if (num_sms <= 0) {
    DeviceInfo info;
    const mfa_status_t st = current_device(nullptr, &info);
    if (st != MFA_OK) return st;
    num_sms = info.num_sms;
  }
  fill_plan(batch, max_len_hint, num_sms, plan);
  return MFA_OK;
}

size_t mfa_decode_workspace_bytes(int batch, int max_len_hint) {
  mfa_plan_t plan;
  if (mfa_plan_decode(batch, max_len_hint, 0, &plan) != MFA_OK) return 0;
  return plan.workspace_bytes;
}

size_t mfa_decode_mtp_workspace_bytes(int batch, int n_query, int max_len_hint) {
  mfa_plan_t plan;
  if (n_query < 1 || n_query > MFA_MAX_QUERY_TOKENS || mfa_plan_decode(batch, max_len_hint, 0, &plan) != MFA_OK)
    return 0;
  DeviceInfo info;
  if (current_device(nullptr, &info) != MFA_OK) return 0;
  // enough for the bf16 kernels (two tokens a CTA) and the quantised ones (one token a CTA)
  size_t need = 0;
  for (const bool quantised : {false, true}) {
    fill_plan(batch, max_len_hint, info.num_sms, &plan, token_groups(n_query, quantised));
    need = std::max(need, plan.workspace_bytes);
  }
  return need;
}

mfa_status_t mfa_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kWsHeaderBytes || !aligned(workspace, 256))
    return fail(MFA_ERR_WORKSPACE, "workspace missing, misaligned or smaller than its header");
  const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return MFA_OK;
}

mfa_status_t mfa_kv_append(const void* k_new, const void* v_new, int n_new, void* k_cache, void* v_cache,
                           const int32_t* page_table, int32_t* seq_lens, int batch, int max_pages, int num_pages,
                           void* workspace, void* stream) {
  return append_common(k_new, v_new, n_new, k_cache, v_cache, nullptr, nullptr, 0, page_table, seq_lens, batch,
                       max_pages, num_pages, workspace, stream);
}

mfa_status_t mfa_kv_append_fp8(const void* k_new, const void* v_new, int n_new, void* k_cache, void* v_cache,
                               float* k_scale, float* v_scale, const int32_t* page_table, int32_t* seq_lens,
                               int batch, int max_pages, int num_pages, void* workspace, void* stream) {
  return append_common(k_new, v_new, n_new, k_cache, v_cache, k_scale, v_scale, kKvE4M3, page_table, seq_lens, batch,
                       max_pages, num_pages, workspace, stream);
}

mfa_status_t mfa_kv_append_fp4(const void* k_new, const void* v_new, int n_new, void* k_cache, void* v_cache,
                               float* k_scale, float* v_scale, const int32_t* page_table, int32_t* seq_lens,
                               int batch, int max_pages, int num_pages, void* workspace, void* stream) {
  if (!aligned(k_cache, 32) || !aligned(v_cache, 32))
    return fail(MFA_ERR_INVALID_ARG, "misaligned 4-bit cache (32 bytes needed)");
  return append_common(k_new, v_new, n_new, k_cache, v_cache, k_scale, v_scale, kKvE2M1, page_table, seq_lens, batch,
                       max_pages, num_pages, workspace, stream);
}

mfa_status_t mfa_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* page_table, const int32_t* seq_lens, void* out, float* lse,
                                  float scale, int batch, int max_pages, int num_pages, int max_len_hint,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common(q, k_cache, v_cache, nullptr, nullptr, false, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream);
}

mfa_status_t mfa_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale, const int32_t* page_table,
                                      const int32_t* seq_lens, void* out, float* lse, float scale, int batch,
                                      int max_pages, int num_pages, int max_len_hint, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return decode_common(q, k_cache, v_cache, k_scale, v_scale, true, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream);
}

mfa_status_t mfa_decode_attention_fp4(const void* q, const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale, const int32_t* page_table,
                                      const int32_t* seq_lens, void* out, float* lse, float scale, int batch,
                                      int max_pages, int num_pages, int max_len_hint, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (!aligned(k_cache, 32) || !aligned(v_cache, 32))
    return fail(MFA_ERR_INVALID_ARG, "misaligned 4-bit cache (32 bytes needed)");
  return decode_common(q, k_cache, v_cache, k_scale, v_scale, true, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream, 1, nullptr, nullptr,
                       0, 1);
}

// Query-path workspace for up to `cap` rows: header (arrival counters at bytes 128-255) |
// y fp32 [cap * rank] | h bf16 [cap * rank] | ssq fp32 [rank/128 * cap].
// A call with batch B <= cap uses the first B * rank floats of y, which it leaves zero, so y is zero on
// entry whatever batch the previous call had.
namespace {
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
struct QueryWs {
  size_t y, h, ssq, total;
};
QueryWs query_ws(int cap, int rank) {
  QueryWs w;
  w.y = kWsHeaderBytes;
  w.h = w.y + (size_t)cap * rank * sizeof(float);
  w.ssq = w.h + round256((size_t)cap * rank * sizeof(uint16_t));
  w.total = w.ssq + round256((size_t)(rank / 128) * cap * sizeof(float));
  return w;
}
}  // namespace

size_t mfa_query_lowrank_workspace_bytes(int batch, int rank, int n_out) {
  if (batch < 1 || batch > kMaxQueryBatch || rank < 128 || rank > kMaxQueryRank || rank % 128 || n_out < 128 ||
      n_out % 128)
    return 0;
  return query_ws(batch, rank).total;
}

mfa_status_t mfa_query_lowrank(const void* x, const void* w_down, const void* gamma, const void* w_up, void* q,
                               int batch, int d_model, int rank, int n_out, float eps, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!x || !w_down || !gamma || !w_up || !q) return fail(MFA_ERR_INVALID_ARG, "null pointer argument");
  if (batch < 1 || batch > kMaxQueryBatch)
    return fail(MFA_ERR_INVALID_ARG, "batch %d outside [1, %d]", batch, kMaxQueryBatch);
  if (d_model < 64 || d_model % 64 || rank < 128 || rank % 128 || n_out < 128 || n_out % 128)
    return fail(MFA_ERR_INVALID_ARG, "d_model must be a multiple of 64, rank and n_out multiples of 128");
  if (rank > kMaxQueryRank) return fail(MFA_ERR_INVALID_ARG, "rank %d above %d", rank, kMaxQueryRank);
  if (!(eps >= 0.0f)) return fail(MFA_ERR_INVALID_ARG, "eps must be >= 0");
  if (!aligned(x, 16) || !aligned(w_down, 16) || !aligned(w_up, 16) || !aligned(q, 16) || !aligned(gamma, 2))
    return fail(MFA_ERR_INVALID_ARG, "misaligned pointer (x, weights, q need 16 bytes)");
  if (!workspace || !aligned(workspace, 256)) return fail(MFA_ERR_WORKSPACE, "workspace missing or not 256-byte aligned");
  const size_t need = mfa_query_lowrank_workspace_bytes(batch, rank, n_out);
  if (workspace_bytes < need) return fail(MFA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  DeviceInfo info;
  mfa_status_t st = current_device(nullptr, &info);
  if (st != MFA_OK) return st;
  char* ws = static_cast<char*>(workspace);
  QueryLowrankParams p{};
  p.gamma = static_cast<const uint16_t*>(gamma);
  int cap = kMaxQueryBatch;  // the most rows this workspace holds
  while (cap > batch && query_ws(cap, rank).total > workspace_bytes) --cap;
  const QueryWs lay = query_ws(cap, rank);
  p.y = reinterpret_cast<float*>(ws + lay.y);
  p.h = reinterpret_cast<uint16_t*>(ws + lay.h);
  p.ssq = reinterpret_cast<float*>(ws + lay.ssq);
  p.counters = reinterpret_cast<uint32_t*>(ws + kQueryCounterOffset);
  p.q = static_cast<uint16_t*>(q);
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.budget = g_wait_budget_ns.load(std::memory_order_relaxed);
  p.eps = eps;
  p.B = batch;
  p.d_model = d_model;
  p.rank = rank;
  p.n_out = n_out;
  // K split of the down-projection: about one CTA per SM, at least one 64-wide K block per CTA
  const int blocks = rank / 128, kchunks = d_model / 64;
  p.splits_down = std::max(1, std::min({kchunks, info.num_sms / blocks, kMaxQuerySplits}));
  const uint32_t Bp = (uint32_t)((batch + 15) & ~15);
  CUtensorMap wd_map, x_map, wu_map, h_map;
  if ((st = encode_bf16_2d(&wd_map, w_down, (uint64_t)rank, (uint64_t)d_model, 64)) != MFA_OK ||
      (st = encode_bf16_2d(&x_map, x, (uint64_t)d_model, (uint64_t)batch, Bp)) != MFA_OK ||
      (st = encode_bf16_2d(&wu_map, w_up, (uint64_t)n_out, (uint64_t)rank, 64)) != MFA_OK ||
      (st = encode_bf16_2d(&h_map, p.h, (uint64_t)rank, (uint64_t)batch, Bp)) != MFA_OK)
    return st;
  const cudaError_t e = launch_query_lowrank(p, wd_map, x_map, wu_map, h_map, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "query path launch");
  return MFA_OK;
}

mfa_status_t mfa_decode_attention_mtp(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* page_table, const int32_t* seq_lens, void* out, float* lse,
                                      float scale, int batch, int n_query, int max_pages, int num_pages,
                                      int max_len_hint, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_query < 1 || n_query > MFA_MAX_QUERY_TOKENS)
    return fail(MFA_ERR_INVALID_ARG, "n_query %d outside [1, %d]", n_query, MFA_MAX_QUERY_TOKENS);
  return decode_common(q, k_cache, v_cache, nullptr, nullptr, false, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream, n_query);
}

mfa_status_t mfa_decode_attention_mtp_fp8(const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale, const int32_t* page_table,
                                          const int32_t* seq_lens, void* out, float* lse, float scale, int batch,
                                          int n_query, int max_pages, int num_pages, int max_len_hint,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  if (n_query < 1 || n_query > MFA_MAX_QUERY_TOKENS)
    return fail(MFA_ERR_INVALID_ARG, "n_query %d outside [1, %d]", n_query, MFA_MAX_QUERY_TOKENS);
  return decode_common(q, k_cache, v_cache, k_scale, v_scale, true, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream, n_query);
}

mfa_status_t mfa_decode_attention_mtp_fp4(const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale, const int32_t* page_table,
                                          const int32_t* seq_lens, void* out, float* lse, float scale, int batch,
                                          int n_query, int max_pages, int num_pages, int max_len_hint,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  if (n_query < 1 || n_query > MFA_MAX_QUERY_TOKENS)
    return fail(MFA_ERR_INVALID_ARG, "n_query %d outside [1, %d]", n_query, MFA_MAX_QUERY_TOKENS);
  if (!aligned(k_cache, 32) || !aligned(v_cache, 32))
    return fail(MFA_ERR_INVALID_ARG, "misaligned 4-bit cache (32 bytes needed)");
  return decode_common(q, k_cache, v_cache, k_scale, v_scale, true, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream, n_query, nullptr,
                       nullptr, 0, 1);
}

mfa_status_t mfa_decode_attention_blocks(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* page_table, const int32_t* seq_lens, const int32_t* block_idx,
                                         const int32_t* n_blocks, int max_blocks, void* out, float* lse, float scale,
                                         int batch, int max_pages, int num_pages, int max_len_hint, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (!block_idx || !n_blocks) return fail(MFA_ERR_INVALID_ARG, "null block_idx or n_blocks");
  if (!aligned(block_idx, 4) || !aligned(n_blocks, 4)) return fail(MFA_ERR_INVALID_ARG, "misaligned block lists");
  if (max_blocks < 1 || (long long)max_blocks > (long long)max_pages * (kPageSize / 8))
    return fail(MFA_ERR_INVALID_ARG, "max_blocks %d outside [1, 8 * max_pages]", max_blocks);
  return decode_common(q, k_cache, v_cache, nullptr, nullptr, false, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream, 1, block_idx,
                       n_blocks, max_blocks);
}

mfa_status_t mfa_decode_attention_blocks_fp8(const void* q, const void* k_cache, const void* v_cache,
                                             const float* k_scale, const float* v_scale, const int32_t* page_table,
                                             const int32_t* seq_lens, const int32_t* block_idx,
                                             const int32_t* n_blocks, int max_blocks, void* out, float* lse,
                                             float scale, int batch, int max_pages, int num_pages, int max_len_hint,
                                             void* workspace, size_t workspace_bytes, void* stream) {
  if (!block_idx || !n_blocks) return fail(MFA_ERR_INVALID_ARG, "null block_idx or n_blocks");
  if (!aligned(block_idx, 4) || !aligned(n_blocks, 4)) return fail(MFA_ERR_INVALID_ARG, "misaligned block lists");
  if (max_blocks < 1 || (long long)max_blocks > (long long)max_pages * (kPageSize / 8))
    return fail(MFA_ERR_INVALID_ARG, "max_blocks %d outside [1, 8 * max_pages]", max_blocks);
  return decode_common(q, k_cache, v_cache, k_scale, v_scale, true, page_table, seq_lens, out, lse, scale, batch,
                       max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream, 1, block_idx,
                       n_blocks, max_blocks);
}

mfa_status_t mfa_check_device_errors(void* workspace, int clear, void* stream) {
  if (!workspace) return fail(MFA_ERR_WORKSPACE, "null workspace");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
  if (clear) {
    e = cudaMemsetAsync(workspace, 0, sizeof word, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
  }
  if (word & MFA_DEVERR_PAGE) return fail(MFA_ERR_DEVICE_PAGE, "device error word 0x%x", word);
  if (word & MFA_DEVERR_CAPACITY) return fail(MFA_ERR_DEVICE_CAPACITY, "device error word 0x%x", word);
  if (word & MFA_DEVERR_TIMEOUT) return fail(MFA_ERR_DEVICE_TIMEOUT, "device error word 0x%x", word);
  return MFA_OK;
}

void mfa_set_wait_budget_ns(uint64_t budget_ns) { g_wait_budget_ns.store(budget_ns, std::memory_order_relaxed); }

mfa_status_t mfa_selftest_wait_timeout(void* workspace, uint64_t budget_ns, void* stream) {
  if (!workspace || !aligned(workspace, 256)) return fail(MFA_ERR_WORKSPACE, "workspace missing or misaligned");
  const mfa_status_t st = current_device(nullptr, nullptr);
  if (st != MFA_OK) return st;
  const cudaError_t e =
      launch_selftest_wait(static_cast<uint32_t*>(workspace), budget_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return MFA_OK;
}

void mfa_profile_split_events(void* start_event, void* stop_event) {
  if (start_event && stop_event) {
    g_prof_start = static_cast<cudaEvent_t>(start_event);
    g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  } else {
    g_prof_start = g_prof_stop = nullptr;
  }
}

const char* mfa_status_string(mfa_status_t status) {
  switch (status) {
    case MFA_OK: return "MFA_OK";
    case MFA_ERR_INVALID_ARG: return "MFA_ERR_INVALID_ARG";
    case MFA_ERR_UNSUPPORTED: return "MFA_ERR_UNSUPPORTED";
    case MFA_ERR_CUDA: return "MFA_ERR_CUDA";
    case MFA_ERR_WORKSPACE: return "MFA_ERR_WORKSPACE";
    case MFA_ERR_DEVICE_PAGE: return "MFA_ERR_DEVICE_PAGE";
    case MFA_ERR_DEVICE_CAPACITY: return "MFA_ERR_DEVICE_CAPACITY";
    case MFA_ERR_DEVICE_TIMEOUT: return "MFA_ERR_DEVICE_TIMEOUT";
  }
  return "MFA_ERR_UNKNOWN";
}

const char* mfa_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
