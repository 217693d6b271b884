// decode_noalloc.cu -- bf16 decode attention that needs no caller workspace.
//
// The regular entry point takes a caller-allocated workspace for the split
// results. Some callers cannot hand one over: a plugin or foreign-function
// host that passes the library only tensors it already owns and gives it no
// allocator, or a latency-bound serving loop that must not call cudaMalloc
// (which can synchronise the whole device) once it is running. For them this
// file keeps the scratch in a fixed, file-scope device array and launches the
// same split and combine kernels on it.
//
// The array is kStaticScratchBytes (24 MiB) on every GPU that loads the
// library, for the life of the process. All calls share it, so calls that can
// overlap on the GPU (other streams, other host threads) race on it. Only the
// error word at its start must begin at zero; every split result is written
// before it is read.
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "mfa_internal.h"

namespace {

using namespace mfa;

constexpr size_t kStaticScratchBytes = (size_t)24 << 20;

// Scratch for the split results of mfa_decode_attention_noalloc. In host code
// this name is only a stand-in: kernels get the device address from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

mfa_status_t report(mfa_status_t st, const char* fmt, size_t a = 0, size_t b = 0) {
  char buf[320];
  snprintf(buf, sizeof buf, fmt, a, b);
  set_last_error_message(buf);
  return st;
}

// Device address of the scratch on the current device, looked up once per
// device (with that device current) on its first call.
mfa_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report(MFA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return report(MFA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      set_last_error_message(cudaGetErrorString(e));
      return MFA_ERR_CUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return MFA_OK;
}

mfa_status_t encode_map(CUtensorMap* map, const void* base, uint64_t rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!enc) return report(MFA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t elem[2] = {1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return report(MFA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return MFA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" mfa_status_t mfa_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                     const int32_t* page_table, const int32_t* seq_lens, void* out,
                                                     float* lse, float scale, int batch, int max_pages,
                                                     int num_pages, int max_len_hint, uint32_t* device_error_word,
                                                     void* stream) {
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out || !lse)
    return report(MFA_ERR_INVALID_ARG, "null pointer argument");
  if (max_pages < 1 || num_pages < 1 || (long long)max_pages * kPageSize > 0x7fffffffLL)
    return report(MFA_ERR_INVALID_ARG, "max_pages and num_pages must be >= 1 (and max_pages * 64 < 2^31)");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(device_error_word, 4))
    return report(MFA_ERR_INVALID_ARG, "misaligned pointer (q, caches, out need 16 bytes)");
  mfa_plan_t plan;
  mfa_status_t st = mfa_plan_decode(batch, max_len_hint, 0, &plan);  // also checks batch, hint and the device
  if (st != MFA_OK) return st;
  if (plan.workspace_bytes > kStaticScratchBytes)
    return report(MFA_ERR_WORKSPACE,
                  "this batch needs %zu bytes of split scratch; the allocation-free entry point has %zu "
                  "(use mfa_decode_attention with a workspace, or a smaller batch)",
                  plan.workspace_bytes, kStaticScratchBytes);
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != MFA_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(scratch);
  uint32_t* err = device_error_word ? device_error_word : reinterpret_cast<uint32_t*>(ws);
  if (!device_error_word) {
    // the error word in the shared scratch must start each call at zero
    const cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return report(MFA_ERR_CUDA, "clearing the scratch error word failed");
  }
  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = err;
  p.part_o = reinterpret_cast<float*>(ws + kWsHeaderBytes);
  p.part_lse = reinterpret_cast<float*>(ws + kWsHeaderBytes + (size_t)plan.partial_slots * kPartialOBytes);
  p.scale = scale;
  p.B = batch;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.grid = plan.grid_ctas;
  p.piece_cost = kPieceCostPages;
  p.n_query = 1;
  p.q_per_cta = 1;
  p.q_groups = 1;
  p.wait_budget_ns = current_wait_budget_ns();
  CUtensorMap kmap, vmap, qmap;
  if ((st = encode_map(&kmap, k_cache, (uint64_t)num_pages * kPageSize)) != MFA_OK ||
      (st = encode_map(&vmap, v_cache, (uint64_t)num_pages * kPageSize)) != MFA_OK ||
      (st = encode_map(&qmap, q, (uint64_t)batch * kHeads)) != MFA_OK)
    return st;
  cudaError_t e = launch_decode_split_tc(p, kmap, vmap, qmap, s);
  if (e == cudaSuccess) e = launch_lse_combine(p, s);
  if (e != cudaSuccess) {
    set_last_error_message(cudaGetErrorString(e));
    return MFA_ERR_CUDA;
  }
  return MFA_OK;
}
