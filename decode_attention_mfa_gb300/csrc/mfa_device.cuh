// mfa_device.cuh -- device-side building blocks shared by the libmfa kernels:
// the work partition over pages, the device error word, bounded mbarrier waits,
// TMA bulk-tensor loads and the tcgen05 (5th-generation tensor core) wrappers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mfa_internal.h"

namespace mfa {

// ---------------------------------------------------------------- error word
__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- partition
// Pages of one sequence: ceil(L / 64) with L clamped to [0, capacity].
__device__ __forceinline__ int pages_of_len(int len) { return (len + kPageSize - 1) / kPageSize; }

__device__ __forceinline__ int clamp_len(int len, int cap_tokens, uint32_t* err) {
  if (len < 0) {
    raise_error(err, MFA_DEVERR_CAPACITY);
    return 0;
  }
  if (len > cap_tokens) {
    raise_error(err, MFA_DEVERR_CAPACITY);
    return cap_tokens;
  }
  return len;
}

// Work partition of one decode step. Sequence b with n_b > 0 pages costs
// n_b + piece_cost units (an empty one costs nothing): the fixed part stands
// for what a sequence piece costs a CTA besides its pages (loading Q, the page
// table row, writing the partial result). Page k of b sits at cost position
// s_cost[b] + piece_cost + k; the first piece_cost positions of b hold no page.
// The G CTAs split the C = s_cost[B] units into equal ranges and each works on
// the pages whose positions fall in its range.
//
// Block gather: a sequence of length L > 0 holds c = floor((L - 1) / 8)
// complete blocks before the one with its last token. With nb of them
// selected (clamped to [0, min(c, max_blocks)], out of range recorded as a
// capacity error) it is read as a virtual sequence of the selected blocks,
// in the caller's order, followed by the L - 8c tokens of its last block.
__device__ __forceinline__ int selected_blocks(int len, const int32_t* n_blocks, int b, int max_blocks,
                                               uint32_t* err) {
  if (len <= 0) return 0;
  const int lim = min((len - 1) >> 3, max_blocks);
  const int nb = __ldg(n_blocks + b);
  if (nb < 0 || nb > lim) {
    raise_error(err, MFA_DEVERR_CAPACITY);
    return nb < 0 ? 0 : lim;
  }
  return nb;
}
__device__ __forceinline__ int virtual_len(int len, int nb) {
  return len <= 0 ? 0 : 8 * nb + len - 8 * ((len - 1) >> 3);
}

// Fill s_len[b] (clamped lengths; virtual lengths under block gather, when
// n_blocks is not null) and s_cost[b] = sum_{c<b} cost(c) for b <= B, using
// every thread of the block. s_cost has B + 1 entries.
// Must be called by all threads of the block; ends with __syncthreads().
__device__ __forceinline__ void build_cost_prefix(const int32_t* __restrict__ seq_lens, int B,
                                                  int cap_tokens, uint32_t* err, int piece_cost, int* s_len,
                                                  int* s_cost, const int32_t* n_blocks = nullptr,
                                                  int max_blocks = 0) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int len = clamp_len(__ldg(seq_lens + b), cap_tokens, err);
    s_len[b] = n_blocks ? virtual_len(len, selected_blocks(len, n_blocks, b, max_blocks, err)) : len;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int running = 0;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      const int np = (b < B) ? pages_of_len(s_len[b]) : 0;
      const int v = np > 0 ? np + piece_cost : 0;
      int x = v;  // inclusive warp scan
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (b < B) s_cost[b] = running + x - v;
      running += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_cost[B] = running;
  }
  __syncthreads();
}

// Range start of CTA c over C cost units split into G equal parts.
__host__ __device__ __forceinline__ long long cta_cost_lo(int c, long long C, int G) {
  return (long long)c * C / G;
}
// The CTA whose range holds cost position x (0 <= x < C).
__host__ __device__ __forceinline__ int cta_of_cost(long long x, long long C, int G) {
  return (int)(((x + 1) * (long long)G - 1) / C);
}
// Largest b in [0, B) with s_cost[b] <= x (no sequence before it reaches x).
__device__ __forceinline__ int seq_of_cost(const int* s_cost, int B, long long x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)s_cost[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- dependent launch
// Kernels of one decode step are launched with programmatic stream
// serialisation: a kernel lets the next one be scheduled early
// (launch_dependents) and the next one runs its prologue, then waits for the
// previous grid's completion and memory (wait) before reading its results.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// `budget_ns`. On expiry (or when another role already gave up, `*abort` != 0)
// it records MFA_DEVERR_TIMEOUT, raises *abort and returns false; it never traps.
// The polling loop is out of line: a wait whose phase has already completed
// (the common case in a running pipeline) costs one try_wait.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint64_t budget_ns,
                                                   volatile int* abort, uint32_t* err) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (globaltimer_ns() - t0 > budget_ns) {
      raise_error(err, MFA_DEVERR_TIMEOUT);
      if (abort) *abort = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t budget_ns,
                                          volatile int* abort, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, budget_ns, abort, err);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(cache_hint)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(cache_hint)
      : "memory");
}
// 1-D bulk copy (addresses 16-byte aligned, size a multiple of 16) completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Hint: bring [src, src + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Block `blk` of `nblk` prefetches its share of a buffer of `bytes` bytes
// into L2, in pieces of at most 64 KB (nothing if the buffer is not 16-byte
// aligned: the bulk prefetch requires it).
__device__ __forceinline__ void prefetch_l2_share(const void* base, size_t bytes, int blk, int nblk) {
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return;
  const size_t per = ((bytes + (size_t)nblk - 1) / nblk + 15) & ~(size_t)15;
  size_t lo = per * (size_t)blk;
  const size_t hi = min(bytes & ~(size_t)15, lo + per);
  for (; lo < hi; lo += 65536)
    prefetch_l2(static_cast<const uint8_t*>(base) + lo, (uint32_t)min((size_t)65536, hi - lo));
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bit 46, swizzle
// mode at bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
// ab_format: 0 = f16, 1 = bf16 (A and B always share it).
__host__ __device__ __forceinline__ constexpr uint32_t idesc_f16(int M, int N, int ab_format, int a_mn_major,
                                                                 int b_mn_major) {
  return (1u << 4) | ((uint32_t)ab_format << 7) | ((uint32_t)ab_format << 10) |
         ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with the A operand read from tensor memory (row i of A in lane i,
// 16-bit elements 2j and 2j+1 in the low and high halves of column j).
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 8-bit operands (kind::f8f6f4), both from shared memory.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Shared-memory matrix descriptor with a given swizzle mode (2: 128-byte, 4: 64-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t mode) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)mode << 61;
  return d;
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns (one lane per thread of the warp).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v);
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// kN (16 or 32) consecutive columns of this thread's lane
template <int kN>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v) {
  static_assert(kN == 16 || kN == 32, "tcgen05.ld width");
  if constexpr (kN == 32) tmem_ld32(taddr, v); else tmem_ld16(taddr, v);
}
template <int kN>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float* v) {
  static_assert(kN == 16 || kN == 32, "tcgen05.st width");
  if constexpr (kN == 32) tmem_st32(taddr, v); else tmem_st16(taddr, v);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Byte offset of element (row r, column c) of a [rows x 64] 16-bit tile stored
// with the 128-byte swizzle (128-byte rows, 16-byte chunks XOR-ed with r % 8);
// the tile base must be 1024-byte aligned.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)(r * 128 + ((((c * 2) >> 4) ^ (r & 7)) << 4) + ((c * 2) & 15));
}

}  // namespace mfa
