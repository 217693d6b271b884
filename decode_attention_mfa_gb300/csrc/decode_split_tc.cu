// decode_split_tc.cu -- split-KV MFA decode on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators) with TMA streaming: a bf16 cache, an FP8-E4M3
// cache with per-token fp32 scales, and a bf16 cache read once for two query
// tokens per sequence (multi-token decode).
//
// MFA ("Step-3 is Large yet Affordable", paper summary page, section 2 /
// Table 1) gives all 64 query heads one shared K head and one shared V head
// (d = 256), so for one sequence the logits of every head against a tile of
// keys form one dense contraction. The kernel computes, per 128-token tile
// (two 64-token pages), the transposed products
//     S^T[tok, col] = K_tile[tok, :] . Q[col, :]^T        (M=128, N=64 or 128)
//     O^T[dim, col] += V_tile[:, dim]^T . P^T[tok, col]   (two 128-dim halves)
// so every MMA uses the full 128-lane data path (an M=64 MMA costs as much as
// an M=128 one on sm_103a), and softmax statistics are reduced across the 128
// TMEM lanes. The columns are the 64 heads (bf16), [token][head] (two query
// tokens), or [E4M3 term][head] (E4M3, where the softmax adds the terms).
//
// Work split: a stream-K partition of cost units (each non-empty sequence
// costs its pages plus a fixed charge per piece, see build_cost_prefix); CTA
// c owns units [c*C/G, (c+1)*C/G) and writes one normalised partial result
// plus its natural-log LSE per sequence piece (and query token) into slot
// c + b; the LSE combine kernel merges the pieces.
//
// Warp roles (one CTA per SM):
//   warps 0-7  softmax, two warpgroups: warpgroup g owns heads [32g, 32g+32)
//              (with two query tokens: query token g); TMEM lane = token of
//              the tile; online softmax in fp32 with a lazily updated
//              reference maximum (only when a logit exceeds it by
//              2^threshold are the row sums and O^T rescaled); then the
//              epilogue (row-sum reduction, O^T / l, partial LSE).
//   warp 8     producer: page-table walk and TMA loads.
//   warp 9     MMA issue and TMEM allocation (one thread issues; the rest of
//              the warp waits at the final barrier).
//   warp 10    (E4M3 cache only) V page producer.
//   warp 11    (E4M3 cache only) largest V scale of each piece.
// bf16 cache: the producer loads 16 KB operand chunks (a 64-dim slice of a
// 2-page K tile, or a 128-dim slice of one V page) straight into a ring of
// shared-memory slots in the layouts the MMAs read; the MMA thread zeroes the
// unused rows of a partial last V page (0 * NaN would poison P.V).
// E4M3 cache ("Step-3 is Large yet Affordable", section 7: 8-bit KV): both
// products are 8-bit MMAs (kind::f8f6f4) on the raw code pages as TMA stages
// them. Q enters S^T as two E4M3 terms (one power-of-two scale per piece, so
// q = t1 + t2 holds every bf16 value down to 2^-10.8 of the largest |q|); P
// enters P.V as two E4M3 terms of P * v_scale, relative to the piece's
// largest V scale. The K scale, the Q scale and the softmax scale multiply
// the logits in fp32 in the softmax warps (the row sums use the unscaled P).
// Every mbarrier wait is bounded (wait budget); on expiry the kernel records
// MFA_DEVERR_TIMEOUT, the roles stop issuing work and the CTA drains and exits.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mfa_device.cuh"

namespace mfa {
namespace {

// kMtp: two query tokens per sequence share each pass over the cache (bf16).
template <bool kFp8, bool kMtp = false>
struct Cfg;
template <>
struct Cfg<false, false> {
  static constexpr int kThreads = 320;   // two softmax warpgroups, producer, MMA
  static constexpr int kSlots = 8;       // 16 KB operand chunks
  static constexpr int kKStages = 0;     // raw code pages: K ring
  static constexpr int kVStages = 0;     // raw code pages: V ring
  static constexpr int kStages = 0;
  static constexpr int kQBufs = 2;
  static constexpr bool kCrossPiece = true;  // one tile stream across sequence pieces
  static constexpr int kScaleSlots = 0;  // per-tile scale blocks
  static constexpr int kAbFormat = 1;    // bf16 operands
  static constexpr int kSCols = 64;      // TMEM columns of one S^T buffer: 64 heads
  static constexpr int kOBufs = 2;       // O^T buffers (pieces alternate)
  static constexpr int kGroups = 2;      // softmax warpgroups (each owns 64 / kGroups heads)
  static constexpr int kSoftmaxThreads = 128 * kGroups;
  static constexpr int kProducerWarp = 4 * kGroups, kMmaWarp = kProducerWarp + 1;
  static constexpr int kQ = 1;           // query tokens per sequence
  static constexpr int kPBufs = 1;       // P buffers (one: its 16 KB buy the eighth ring slot)
  static constexpr int kCols = 64;       // softmax columns: [token][head]
  static constexpr int kHpt = 32;        // columns per softmax thread
  static constexpr int kOHalfCols = 64;  // O^T columns per 128-dim half
};
// Two query tokens per sequence (MTP): S^T and P are [token][head] = 128
// columns, warpgroup g owns query token g; one O^T of 2 x 128 columns.
template <>
struct Cfg<false, true> {
  static constexpr int kThreads = 320;
  static constexpr int kSlots = 7;       // 16 KB operand chunks
  static constexpr int kKStages = 0;
  static constexpr int kVStages = 0;
  static constexpr int kStages = 0;
  static constexpr int kQBufs = 1;
  static constexpr bool kCrossPiece = true;
  static constexpr int kScaleSlots = 0;
  static constexpr int kAbFormat = 1;
  static constexpr int kSCols = 128;
  static constexpr int kOBufs = 1;
  static constexpr int kGroups = 2;
  static constexpr int kSoftmaxThreads = 128 * kGroups;
  static constexpr int kProducerWarp = 4 * kGroups, kMmaWarp = kProducerWarp + 1;
  static constexpr int kQ = 2;
  static constexpr int kPBufs = 1;       // Q and P are twice as large: one P buffer keeps 7 ring slots
  static constexpr int kCols = 128;
  static constexpr int kHpt = 64;
  static constexpr int kOHalfCols = 128;
};
// E4M3: the producer stages the K tiles and scales, a second producer warp
// the V pages, and one warp finds each piece's largest V scale; both products
// run as 8-bit MMAs on the raw staged pages, so no code is converted on chip.
template <>
struct Cfg<true, false> {
  static constexpr int kThreads = 384;    // two softmax warpgroups, then 4 single-warp roles
  static constexpr int kSlots = 0;        // K and V are read raw by 8-bit MMAs: no operand ring
  static constexpr int kKStages = 2;      // raw K tiles (both pages of a tile, 32 KB): A of S^T
  static constexpr int kVStages = 4;      // raw V pages (16 KB): A of P.V
  static constexpr int kStages = kKStages + kVStages;
  static constexpr int kQBufs = 1;        // bf16 Q, split in place into two E4M3 terms
  static constexpr bool kCrossPiece = false;  // per-piece order (a single Q buffer)
  static constexpr int kScaleSlots = 4;
  static constexpr int kSCols = 128;      // S^T against both Q terms: [term][head]
  static constexpr int kOBufs = 1;        // O^T is [half][term][head] = 256 columns
  static constexpr int kGroups = 2;       // softmax warpgroups: heads 0-31 and 32-63
  static constexpr int kSoftmaxThreads = 128 * kGroups;
  static constexpr int kProducerWarp = 4 * kGroups, kMmaWarp = kProducerWarp + 1;
  static constexpr int kVProducerWarp = kProducerWarp + 2, kVRefWarp = kProducerWarp + 3;
  static constexpr int kQ = 1;
  static constexpr int kPBufs = 2;
  static constexpr int kCols = 64;        // per-head statistics (the two terms are summed)
  static constexpr int kHpt = 64 / kGroups;
  static constexpr int kOHalfCols = 128;  // [term][head]
};

// Token groups (multi-token decode) run on the two-token kernel and on the E4M3 kernel; the
// single-token bf16 kernel always serves one group, so its index arithmetic folds away.
template <bool kFp8, bool kMtp>
__device__ __forceinline__ int q_groups_of(const DecodeParams& p) {
  return (kFp8 || kMtp) ? p.q_groups : 1;
}

constexpr int kSlotBytes = 16384;
constexpr int kStageBytes = 16384;        // one E4M3 V page: 64 rows x 256 B (two 128 B-wide swizzled boxes)
constexpr int kKTileBytes = 32768;        // one E4M3 K tile: box h (dims [128h, 128h+128)) of 128 rows at 16 KB * h
constexpr int kQTermBytes = 8192;         // one term of one 128-dim box: [64 heads x 128 B], 128-byte swizzle
constexpr int kQBytes = 32768;            // Q of one token: 4 dim blocks of [64 heads x 128 B]
constexpr int kPBytes = 16384;            // P^T of one token: [128 tokens x 64 heads], 16-bit
constexpr int kScaleBytes = 1024;         // per tile: 128 K scales, then 128 V scales
constexpr int kTmemCols = 512;            // S^T x2 + O^T (bf16: 2 x 64 + 2 x 128; E4M3: 2 x 128 + 256)
template <bool kFp8, bool kMtp = false>
__host__ __device__ constexpr int tmem_o() { return 2 * Cfg<kFp8, kMtp>::kSCols; }  // first O^T column; bf16 buffer o at +128 * o
constexpr int kMaxBars = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// log2 units: P stays below 2^threshold between rescales. E4M3 keeps P within
// 2^3 so that P's bulk sits in the normal range of the 8-bit P operand.
template <bool kFp8>
__host__ __device__ constexpr float rescale_threshold() { return kFp8 ? 3.0f : 8.0f; }
// E4M3: the P operand is x = P * v_scale / vref * 2^5 <= 2^3 * 1 * 2^5 = 256 < 448
// (vref = the piece's largest V scale), split into two E4M3 terms x1 + x2,
// stored side by side per token: [x1 of heads 0-63 | x2 of heads 0-63].
constexpr float kPScale = 32.0f;

template <bool kFp8, bool kMtp = false>
struct Bars {  // indices into the barrier array
  using C = Cfg<kFp8, kMtp>;
  static constexpr int Full = 0;                     // [kSlots] operand chunk ready
  static constexpr int Empty = Full + C::kSlots;     // [kSlots] operand chunk consumed
  static constexpr int QFull = Empty + C::kSlots;    // [2] Q landed
  static constexpr int QEmpty = QFull + 2;           // [2] every S MMA of the piece done
  static constexpr int QReady = QEmpty + 2;          // [2] Q split into E4M3 terms (E4M3 only)
  static constexpr int SFull = QReady + 2;           // [2]
  static constexpr int SEmpty = SFull + 2;           // [2]
  static constexpr int PFull = SEmpty + 2;           // [kPBufs <= 2]
  static constexpr int PEmpty = PFull + 2;           // [kPBufs <= 2]
  static constexpr int OFree = PEmpty + 2;           // [2] one completion per epilogue of a piece using O^T buffer i
  static constexpr int Drain = OFree + 2;
  static constexpr int StFull = Drain + 1;           // [kStages] raw K tile / V page landed
  static constexpr int StEmpty = StFull + C::kStages;   // [kStages] the MMAs reading it are done
  static constexpr int ScFull = StEmpty + C::kStages;   // [kScaleSlots]
  static constexpr int ScEmpty = ScFull + C::kScaleSlots;
  static constexpr int VRefFull = ScEmpty + C::kScaleSlots;  // [2] E4M3: a piece's largest V scale is known
  static constexpr int VRefEmpty = VRefFull + 2;          // [2] E4M3: the softmax has read it
  static constexpr int Count = VRefEmpty + 2;
  static_assert(Count <= kMaxBars, "barrier array too small");
};

template <bool kFp8, bool kMtp>
__host__ __device__ constexpr uint32_t idesc_s() {  // A = K tile (K-major), B = Q (K-major), N = [token][head]
  return idesc_f16(128, Cfg<kFp8, kMtp>::kSCols, Cfg<kFp8, kMtp>::kAbFormat, 0, 0);
}
template <bool kFp8, bool kMtp>
__host__ __device__ constexpr uint32_t idesc_o() {  // A = V^T (dim-major), B = P^T (head-major), N = [token][head]
  return idesc_f16(128, 64 * Cfg<kFp8, kMtp>::kQ, Cfg<kFp8, kMtp>::kAbFormat, 1, 1);
}
// kind::f8f6f4, A and B E4M3 (format 0), both K-major, fp32 accumulate, M=128 N=128
__host__ __device__ constexpr uint32_t idesc_s_e4m3() { return (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24); }
// 4-bit cache: the A operand (the K tile, or the V page) is E2M1 (format 5) against E4M3 B
constexpr uint32_t kIdescAE2M1 = 5u << 7;
// kind::f8f6f4, A and B E4M3 (format 0), both dim/head-major, fp32 accumulate, M=128 N=128
__host__ __device__ constexpr uint32_t idesc_o_e4m3() {
  return (1u << 4) | (1u << 15) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

struct SmemLayout {
  uint32_t ring, stage, q, p, scales;  // byte offsets from the 1024-aligned base
  uint32_t len, prefix, red, bars, misc;
  uint32_t total;
};

template <bool kFp8, bool kMtp = false>
__host__ __device__ constexpr SmemLayout smem_layout(int B) {
  using C = Cfg<kFp8, kMtp>;
  SmemLayout L{};
  L.ring = 0;
  L.stage = L.ring + C::kSlots * kSlotBytes;  // E4M3: K tiles, then V pages
  L.q = L.stage + C::kKStages * kKTileBytes + C::kVStages * kStageBytes;
  L.p = L.q + C::kQBufs * C::kQ * kQBytes;  // E4M3: the Q terms overwrite the bf16 Q (same 32 KB)
  L.scales = L.p + C::kPBufs * C::kQ * kPBytes;
  L.len = L.scales + C::kScaleSlots * kScaleBytes;
  L.prefix = L.len + 4 * B;
  // float red[4][kCols], mref[kCols], alpha[kCols], inv_l[2][kCols], scratch[kCols], vref[2]
  L.red = (L.prefix + 4 * (B + 1) + 15) & ~15u;
  L.bars = (L.red + 9 * C::kCols * 4 + 8 + 7) & ~7u;    // mbarriers
  L.misc = L.bars + 8 * kMaxBars;                 // tmem base, abort flag
  L.total = L.misc + 16;
  return L;
}
constexpr uint32_t kMaxDynamicSmem = 227u * 1024u;  // per-block opt-in limit of sm_103a
static_assert(smem_layout<false>(kMaxBatch).total + 1024 <= kMaxDynamicSmem, "bf16 layout exceeds shared memory");
static_assert(smem_layout<true>(kMaxBatch).total + 1024 <= kMaxDynamicSmem, "E4M3 layout exceeds shared memory");
static_assert(smem_layout<false, true>(kMaxBatch).total + 1024 <= kMaxDynamicSmem, "MTP layout exceeds shared memory");

struct Ctx {
  uint32_t base;      // shared address of the aligned dynamic smem base
  uint32_t bar0;      // shared address of barrier 0
  volatile int* abort;
  uint32_t* err;
  uint64_t budget;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  __device__ bool wait(int i, uint32_t parity) const { return mbar_wait(bar(i), parity, budget, abort, err); }
};

// Named barriers of the softmax warps: 1 + g for warpgroup g (128 threads),
// kAllSoftmaxBarrier for all of them.
constexpr int kAllSoftmaxBarrier = 8;
__device__ __forceinline__ void barrier_group(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }
// The group barrier, returning the OR of `pred` over the group's threads.
__device__ __forceinline__ bool barrier_group_or(int g, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(1 + g)
      : "memory");
  return r != 0;
}
template <int kThreadsAll>
__device__ __forceinline__ void barrier_softmax_all() {
  asm volatile("bar.sync %0, %1;" ::"n"(kAllSoftmaxBarrier), "n"(kThreadsAll) : "memory");
}
// 2^x with the multi-function unit's approximation (relative error below
// 2^-22; subnormal results flush to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Segment iteration shared by all roles: sequence b, pages [pg0, pg1) of it.
struct Seg {
  int b, pg0, pg1, len;
};
__device__ __forceinline__ bool seg_first(const int* s_cost, int B, long long lo, long long hi, Seg& s) {
  if (lo >= hi) return false;
  s.b = seq_of_cost(s_cost, B, lo) - 1;
  return true;
}
__device__ __forceinline__ bool seg_next(const int* s_cost, const int* s_len, int B, int piece_cost, long long lo,
                                         long long hi, Seg& s) {
  for (int b = s.b + 1; b < B && s_cost[b] < hi; ++b) {
    const int np = pages_of_len(s_len[b]);
    const long long first = (long long)s_cost[b] + piece_cost;  // cost position of page 0
    const long long a = lo > first ? lo - first : 0;
    const long long e = hi - first < np ? hi - first : np;
    if (np == 0 || a >= e) continue;
    s.b = b;
    s.pg0 = (int)a;
    s.pg1 = (int)e;
    s.len = s_len[b];
    return true;
  }
  return false;
}
__device__ __forceinline__ int tiles_of(const Seg& s) { return (s.pg1 - s.pg0 + 1) / 2; }
__device__ __forceinline__ int pages_in_tile(const Seg& s, int t) { return (s.pg0 + 2 * t + 1 < s.pg1) ? 2 : 1; }

// ---------------------------------------------------------------- producer
// Page ids of one sequence piece for the producer warp: a window of 64 ids
// [base, base + 64) held as two registers per lane (lane i: ids base + i and
// base + 32 + i), filled by coalesced warp loads and handed out by shuffle.
// Requests go forward, except that V pages trail the K pages of the next tile
// by two, so the window slides by 32 only when a request reaches base + 64.
struct PageIds {
  const int32_t* row;  // page_table row of the sequence
  int pg1, base;       // valid pages end at pg1
  int lo_ids, hi_ids;
  __device__ int fetch(int pg, const DecodeParams& p) const {
    int id = 0;
    if (pg < pg1) {
      id = __ldg(row + pg);
      if (id < 0 || id >= p.num_pages) {
        raise_error(p.err, MFA_DEVERR_PAGE);
        id = 0;
      }
    }
    return id;
  }
  __device__ void start(int pg0, const DecodeParams& p, int lane) {
    base = pg0;
    lo_ids = fetch(base + lane, p);
    hi_ids = fetch(base + 32 + lane, p);
  }
  // all lanes call with the same pg, base <= pg
  __device__ int get(int pg, const DecodeParams& p, int lane) {
    while (pg >= base + 64) {
      base += 32;
      lo_ids = hi_ids;
      hi_ids = fetch(base + 32 + lane, p);
    }
    const int idx = pg - base;
    return idx < 32 ? __shfl_sync(0xffffffffu, lo_ids, idx) : __shfl_sync(0xffffffffu, hi_ids, idx - 32);
  }
};

// ---------------------------------------------------------------- LSU async copies
// 16 bytes from global to shared memory through the LSU (both addresses 16-byte aligned), and an arrival on
// an mbarrier once every such copy this thread issued has landed (the barrier's count includes it).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Block gather: cache rows of the virtual blocks of one sequence piece (the
// selected blocks in the caller's order, then the block of the last token).
// Lane j < 16 looks up block j of each 16-block tile in three steps -- the
// block id, then its page id, then the row -- each a tile apart, so that the
// two dependent loads of a tile are in flight while earlier tiles are issued.
// A block id outside [0, cur) or a bad page id is recorded as a page error and
// read as block 0 / page 0.
struct BlockRows {
  const int32_t* bidx;  // block_idx row of the sequence
  const int32_t* prow;  // page_table row
  int nb, cur, nvb;     // selected blocks, block of the last token, virtual blocks
  int vb0;              // first virtual block of the piece
  __device__ void start(const Seg& s, const DecodeParams& p) {
    const int len = clamp_len(__ldg(p.seq_lens + s.b), p.max_pages * kPageSize, nullptr);
    nb = selected_blocks(len, p.n_blocks, s.b, p.max_blocks, nullptr);  // errors: recorded by the prefix
    cur = (len - 1) >> 3;
    nvb = len > 0 ? nb + 1 : 0;
    vb0 = 8 * s.pg0;
    bidx = p.block_idx + (size_t)s.b * p.max_blocks;
    prow = p.page_table + (size_t)s.b * p.max_pages;
  }
  __device__ bool has(int t, int lane) const { return lane < 16 && vb0 + 16 * t + lane < nvb; }
  // step 1 for tile t: the block id (a load for a selected block)
  __device__ int block_id(int t, int lane) const {
    const int i = vb0 + 16 * t + lane;
    return has(t, lane) ? (i < nb ? __ldg(bidx + i) : cur) : 0;
  }
  // step 2: the block's first position (returned in pos, -1 without a block) and a load of its page id
  __device__ int page_id(int t, int lane, int r, int& pos, const DecodeParams& p) const {
    if (!has(t, lane)) {
      pos = -1;
      return 0;
    }
    if (vb0 + 16 * t + lane < nb && (r < 0 || r >= cur)) {
      raise_error(p.err, MFA_DEVERR_PAGE);
      r = 0;
    }
    pos = 8 * r;
    return __ldg(prow + (pos >> 6));
  }
  // step 3: the cache row (page id * 64 + row in the page), -1 without a block
  __device__ int row(int id, int pos, const DecodeParams& p) const {
    if (pos < 0) return -1;
    if (id < 0 || id >= p.num_pages) {
      raise_error(p.err, MFA_DEVERR_PAGE);
      id = 0;
    }
    return id * kPageSize + (pos & (kPageSize - 1));
  }
};

// The whole producer warp runs this loop (uniform control flow); lane 0
// issues the copies. Per piece: Q, then the chunks of K(0), then for each
// tile t >= 1 those of K(t) and V(t-1), then V(T-1) -- the order in which the
// MMA warp consumes them (bf16). E4M3: Q, then per tile the raw K tile and
// its scale block (the V pages come from the V producer warp).
template <bool kFp8, bool kMtp, bool kGather8 = false>
__device__ void producer_role(const DecodeParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                              const CUtensorMap* qmap, const Ctx& cx, const int* s_cost, const int* s_len,
                              long long lo, long long hi) {
  using C = Cfg<kFp8, kMtp>;
  using Bb = Bars<kFp8, kMtp>;
  const int lane = threadIdx.x & 31;
  // the CTAs of one range (token groups) read the same pages: keep them in L2 for the others
  const int qg = q_groups_of<kFp8, kMtp>(p);
  const uint64_t pol_stream = qg > 1 ? policy_evict_normal() : policy_evict_first();
  const uint64_t pol_keep = policy_evict_last();
  const int q_tok0 = (int)(blockIdx.x % qg) * C::kQ;  // first query token of this CTA's group
  const SmemLayout L = smem_layout<kFp8, kMtp>(p.B);
  uint32_t cc = 0, seg_i = 0, sc_cnt = 0;  // chunks (bf16) or staged K tiles (E4M3); pieces; tiles
  Seg s;
  bool ok = seg_first(s_cost, p.B, lo, hi, s);
  constexpr int kRing = kFp8 ? C::kKStages : C::kSlots;  // E4M3: the K stage ring (V pages: the V producer warp)
  constexpr int kRingFull = kFp8 ? Bb::StFull : Bb::Full;
  constexpr int kRingEmpty = kFp8 ? Bb::StEmpty : Bb::Empty;
  auto wait_slot = [&](uint32_t& dst, uint32_t& bar) -> bool {
    const uint32_t slot = cc % kRing, n = cc / kRing;
    const bool r = cx.wait(kRingEmpty + slot, (n & 1) ^ 1);
    __syncwarp();
    dst = cx.base + (kFp8 ? L.stage + slot * kKTileBytes : L.ring + slot * kSlotBytes);
    bar = cx.bar(kRingFull + slot);
    return r;
  };
  // bf16: K dim block d of a tile of pages pa (and pb >= 0)
  auto issue_k = [&](int d, int pa, int pb) -> bool {
    uint32_t dst, bar;
    if (!wait_slot(dst, bar)) return false;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, pb >= 0 ? 16384u : 8192u);
      tma_load_2d(dst, kmap, d * 64, pa * kPageSize, bar, pol_stream);
      if (pb >= 0) tma_load_2d(dst + 8192, kmap, d * 64, pb * kPageSize, bar, pol_stream);
    }
    ++cc;
    return true;
  };
  // bf16: V dims [hf*128, hf*128 + 128) of page pv
  auto issue_v = [&](int hf, int pv) -> bool {
    uint32_t dst, bar;
    if (!wait_slot(dst, bar)) return false;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, 16384u);
      tma_load_2d(dst, vmap, hf * 128, pv * kPageSize, bar, pol_stream);
      tma_load_2d(dst + 8192, vmap, hf * 128 + 64, pv * kPageSize, bar, pol_stream);
    }
    ++cc;
    return true;
  };
  // E4M3: the raw K pages of a tile, as two K-major A operands of 128 rows
  // (box h = dims [128h, 128h + 128): page pa's rows at 16 KB * h, pb's after them)
  auto stage_k_tile = [&](int pa, int pb) -> bool {
    uint32_t dst, bar;
    if (!wait_slot(dst, bar)) return false;
    if (lane == 0) {
      // a 4-bit page counts its packed bytes, half those of E4M3 (the gaps TMA leaves are not transferred)
      mbar_arrive_expect_tx(bar, (pb >= 0 ? 32768u : 16384u) >> p.kv_fp4);
      tma_load_2d(dst, kmap, 0, pa * kPageSize, bar, pol_stream);
      tma_load_2d(dst + 16384, kmap, 128, pa * kPageSize, bar, pol_stream);
      if (pb >= 0) {
        tma_load_2d(dst + 8192, kmap, 0, pb * kPageSize, bar, pol_stream);
        tma_load_2d(dst + 24576, kmap, 128, pb * kPageSize, bar, pol_stream);
      }
    }
    ++cc;
    return true;
  };
  // E4M3: the K and V scales of the tile's pages
  auto stage_scales = [&](int pa, int pb) -> bool {
    constexpr uint32_t kRingSc = C::kScaleSlots > 0 ? C::kScaleSlots : 1;
    const uint32_t slot = sc_cnt % kRingSc, n = sc_cnt / kRingSc;
    const bool r = cx.wait(Bb::ScEmpty + slot, (n & 1) ^ 1);
    __syncwarp();
    if (!r) return false;
    if (lane == 0) {
      const uint32_t dst = cx.base + L.scales + slot * kScaleBytes, bar = cx.bar(Bb::ScFull + slot);
      const uint32_t per_page = kPageSize * sizeof(float);
      mbar_arrive_expect_tx(bar, (pb >= 0 ? 4u : 2u) * per_page);
      bulk_load(dst, p.k_scale + (size_t)pa * kPageSize, per_page, bar);
      bulk_load(dst + 512, p.v_scale + (size_t)pa * kPageSize, per_page, bar);
      if (pb >= 0) {
        bulk_load(dst + per_page, p.k_scale + (size_t)pb * kPageSize, per_page, bar);
        bulk_load(dst + 512 + per_page, p.v_scale + (size_t)pb * kPageSize, per_page, bar);
      }
    }
    ++sc_cnt;
    return true;
  };
  // bf16: V dims of both halves of the pages of a tile
  auto issue_v_tile = [&](int pa, int pb) -> bool {
    return issue_v(0, pa) && issue_v(1, pa) && (pb < 0 || (issue_v(0, pb) && issue_v(1, pb)));
  };
  // Block gather (bf16, one query token): a tile is 16 blocks of 8 rows; lane j < 16 holds the cache
  // row of block j of the tile (-1 past the end) and copies it itself. The TMA unit spends about the
  // same time on a copy whatever its size, so every copy takes a whole block's row range, and the
  // chunks are pairs of adjacent ring slots (32 KB; the last slot of the ring is skipped so that pairs
  // never wrap): a K pair holds dim blocks 2h, 2h + 1 of the tile, block j at 2 KB * j as two swizzle
  // atoms [8 rows x 128 B] (dim block 2h first); a V pair holds one page, block j at 4 KB * j as its
  // four dim blocks. Only the pair's first slot's barriers are used.
  auto wait_pair = [&](uint32_t& dst, uint32_t& bar) -> bool {
    if (cc % kRing == kRing - 1) ++cc;  // pairs start at even slots
    const bool r = wait_slot(dst, bar);
    if (r) cc += 2;
    return r;
  };
  auto issue_k_pair = [&](int h, int row) -> bool {
    uint32_t dst, bar;
    if (!wait_pair(dst, bar)) return false;
    const bool mine = lane < 16 && row >= 0;
    const uint32_t n = __popc(__ballot_sync(0xffffffffu, mine));
    if (lane == 0) mbar_arrive_expect_tx(bar, n * 2048u);
    __syncwarp();
    if (mine) tma_load_3d(dst + lane * 2048, kmap, 0, row, 2 * h, bar, pol_stream);
    return true;
  };
  // page i (blocks 8i .. 8i + 7) of the tile; a block past the end is read from above the top of the
  // cache, which fills it with zeros (0 * NaN of a stale row would poison P.V)
  auto issue_v_pair = [&](int i, int row) -> bool {
    uint32_t dst, bar;
    if (!wait_pair(dst, bar)) return false;
    if (lane == 0) mbar_arrive_expect_tx(bar, 8u * 4096u);
    __syncwarp();
    if (lane >= 8 * i && lane < 8 * i + 8)
      tma_load_3d(dst + (uint32_t)(lane - 8 * i) * 4096u, vmap, 0, row >= 0 ? row : -8, 0, bar, pol_stream);
    return true;
  };
  auto issue_v_blocks_tile = [&](int row, bool two_pages) -> bool {
    return issue_v_pair(0, row) && (!two_pages || issue_v_pair(1, row));
  };
  uint32_t vc = 0;  // E4M3 block gather: V stages issued by this warp
  // E4M3 block gather. A K tile is staged as [block j][128-dim half h][8 rows x 128 B] (block j at 2 KB * j,
  // one 3-D copy of 2 KB per block: both halves of its 8 rows), the S^T MMA taking 2 KB between 8-row
  // groups; the tile's scale block receives each block's 8 K and 8 V scales (32 B each) at 32 B * j.
  // Lane j < 16 holds the cache row of block j of the tile (-1 past the end).
  auto stage_k_blocks = [&](int row) -> bool {
    uint32_t dst, bar;
    if (!wait_slot(dst, bar)) return false;
    const bool mine = lane < 16 && row >= 0;
    const uint32_t n = __popc(__ballot_sync(0xffffffffu, mine));
    if (lane == 0) mbar_arrive_expect_tx(bar, n * 2048u);
    __syncwarp();
    if (mine) tma_load_3d(dst + lane * 2048, kmap, 0, row, 0, bar, pol_stream);
    ++cc;
    return true;
  };
  // the 8 K and 8 V scales of each of the tile's 16 blocks by LSU copies (cp.async, 16 bytes each), not by
  // the TMA unit: these 32-byte rows are half of this mode's copies a tile, and the TMA unit takes about as
  // long per copy whatever its size. Lane i < 16 brings block i's K scales, lane 16 + i its V scales; every
  // lane's arrival (on completion of its copies) counts on the scale barrier (32 arrivals in this mode).
  auto stage_block_scales = [&](int row) -> bool {
    constexpr uint32_t kRingSc = C::kScaleSlots > 0 ? C::kScaleSlots : 1;
    const uint32_t slot = sc_cnt % kRingSc, n = sc_cnt / kRingSc;
    const bool r = cx.wait(Bb::ScEmpty + slot, (n & 1) ^ 1);
    __syncwarp();
    if (!r) return false;
    const int blk = lane & 15;
    const int brow = __shfl_sync(0xffffffffu, row, blk);  // block blk's cache row (-1: no block)
    const uint32_t dst = cx.base + L.scales + slot * kScaleBytes + (lane < 16 ? 0u : 512u) + (uint32_t)blk * 32u;
    if (brow >= 0) {
      const float* src = (lane < 16 ? p.k_scale : p.v_scale) + brow;
      cp_async_16(dst, src);
      cp_async_16(dst + 16, src + 4);
    }
    cp_async_mbar_arrive_noinc(cx.bar(Bb::ScFull + slot));
    ++sc_cnt;
    return true;
  };
  // virtual page i (blocks 8i .. 8i + 7 of the tile) of V as [block][half][8 rows x 128 B]; a block past the
  // end is read from above the top of the cache, which fills it with zeros (0 * NaN would poison P.V)
  auto stage_v_blocks = [&](int i, int row) -> bool {
    const uint32_t slot = C::kKStages + vc % (C::kVStages > 0 ? C::kVStages : 1);
    const uint32_t n = vc / (C::kVStages > 0 ? C::kVStages : 1);
    const bool r = cx.wait(Bb::StEmpty + slot, (n & 1) ^ 1);
    __syncwarp();
    if (!r) return false;
    const uint32_t dst = cx.base + L.stage + C::kKStages * kKTileBytes +
                         (vc % (C::kVStages > 0 ? C::kVStages : 1)) * kStageBytes;
    const uint32_t bar = cx.bar(Bb::StFull + slot);
    if (lane == 0) mbar_arrive_expect_tx(bar, 8u * 2048u);
    __syncwarp();
    if (lane >= 8 * i && lane < 8 * i + 8)
      tma_load_3d(dst + (uint32_t)(lane - 8 * i) * 2048u, vmap, 0, row >= 0 ? row : -8, 0, bar, pol_stream);
    ++vc;
    return true;
  };
  const bool gather = !kFp8 && !kMtp && p.block_idx != nullptr;
  constexpr bool gather8 = kGather8;  // E4M3 block gather (its own instantiation): this warp stages V as well
  static_assert(!kGather8 || (kFp8 && !kMtp), "block gather instantiation of the E4M3 kernel only");
  int pend_row = -1;  // gather: this lane's block row of the tile whose V is still to be issued
  bool pend_two = false, pend_valid = false;
  int pend_a = -1, pend_b = -1;  // pages of the tile whose V is still to be issued (tile stream)
  uint32_t last_q_parity = 0, last_qb = 0;
  bool issued_q = false;
  while (ok && seg_next(s_cost, s_len, p.B, p.piece_cost, lo, hi, s)) {
    if (*cx.abort) break;
    PageIds ids;
    ids.row = p.page_table + (size_t)s.b * p.max_pages;
    ids.pg1 = s.pg1;
    if (!gather && !kGather8) ids.start(s.pg0, p, lane);
    BlockRows blk;
    if (gather || kGather8) blk.start(s, p);
    // Q of this sequence; its buffer is free once every S MMA of the piece that
    // last used it is done (with two buffers the loads of this piece need not
    // wait for the previous piece to finish)
    const uint32_t qb = seg_i % C::kQBufs, qn = seg_i / C::kQBufs;
    const bool qfree = cx.wait(Bb::QEmpty + qb, (qn & 1) ^ 1);
    __syncwarp();
    if (!qfree) break;
    if (lane == 0) {
      // dim block d of token t at (d * kQ + t) * 8 KB: per block, the tokens'
      // 64-head rows stack into one 64 * kQ-row K-major operand
      const uint32_t q_dst = cx.base + L.q + qb * C::kQ * kQBytes;
      mbar_arrive_expect_tx(cx.bar(Bb::QFull + qb), (uint32_t)(C::kQ * kQBytes));
      for (int d = 0; d < 4; ++d)
        for (int t = 0; t < C::kQ; ++t)
          tma_load_2d(q_dst + (d * C::kQ + t) * 8192, qmap, d * 64, (s.b * p.n_query + q_tok0 + t) * kHeads,
                      cx.bar(Bb::QFull + qb), pol_keep);  // a row past the last token reads zeros
    }
    issued_q = true;
    last_q_parity = qn & 1;
    last_qb = qb;
    ++seg_i;
    const int T = tiles_of(s);
    bool good = true;
    if (C::kCrossPiece && gather) {
      // the tile stream below, with blocks: while tile t is issued, the page id of tile t + 1 and the
      // block id of tile t + 2 are in flight
      int pos0, pos1;
      const int r0 = blk.block_id(0, lane), r1 = blk.block_id(1, lane);
      const int id0 = blk.page_id(0, lane, r0, pos0, p);
      int id1 = blk.page_id(1, lane, r1, pos1, p);
      int r2 = blk.block_id(2, lane);
      int row = blk.row(id0, pos0, p);
      for (int t = 0; good && t < T; ++t) {
        for (int h = 0; good && h < 2; ++h) good = issue_k_pair(h, row);
        if (good && pend_valid) good = issue_v_blocks_tile(pend_row, pend_two);
        pend_row = row;
        pend_two = pages_in_tile(s, t) == 2;
        pend_valid = true;
        row = blk.row(id1, pos1, p);
        id1 = blk.page_id(t + 2, lane, r2, pos1, p);
        r2 = blk.block_id(t + 3, lane);
      }
    } else if constexpr (C::kCrossPiece) {
      // K(g), then V(g - 1) of the previous tile, which may belong to the
      // previous piece: the next piece's first K tile is not queued behind the
      // last V tile of the previous one
      for (int t = 0; good && t < T; ++t) {
        const int pga = s.pg0 + 2 * t;
        const int pa = ids.get(pga, p, lane);
        const int pb = (pages_in_tile(s, t) == 2) ? ids.get(pga + 1, p, lane) : -1;
        for (int d = 0; good && d < 4; ++d) good = issue_k(d, pa, pb);
        if (good && pend_a >= 0) good = issue_v_tile(pend_a, pend_b);
        pend_a = pa;
        pend_b = pb;
      }
    } else if constexpr (kGather8) {
      // K(t) and its scales, then V(t - 1), in the MMA warp's per-piece order; the block rows of tile t + 1
      // and the block ids of tile t + 2 are in flight meanwhile
      int pos0, pos1;
      const int r0 = blk.block_id(0, lane), r1 = blk.block_id(1, lane);
      const int id0 = blk.page_id(0, lane, r0, pos0, p);
      int id1 = blk.page_id(1, lane, r1, pos1, p);
      int r2 = blk.block_id(2, lane);
      int row = blk.row(id0, pos0, p), prev_row = -1;
      for (int t = 0; good && t <= T; ++t) {
        if (t < T) good = stage_k_blocks(row) && stage_block_scales(row);
        if (good && t > 0) {
          const int np = pages_in_tile(s, t - 1);
          for (int i = 0; good && i < np; ++i) good = stage_v_blocks(i, prev_row);
        }
        prev_row = row;
        row = blk.row(id1, pos1, p);
        id1 = blk.page_id(t + 2, lane, r2, pos1, p);
        r2 = blk.block_id(t + 3, lane);
      }
    } else {
    for (int t = 0; good && t <= T; ++t) {
      if (t < T) {
        const int pga = s.pg0 + 2 * t;
        const int pa = ids.get(pga, p, lane);
        const int pb = (pages_in_tile(s, t) == 2) ? ids.get(pga + 1, p, lane) : -1;
        if constexpr (kFp8) {
          good = stage_k_tile(pa, pb) && stage_scales(pa, pb);
        } else {
          for (int d = 0; good && d < 4; ++d) good = issue_k(d, pa, pb);
        }
      }
      if (!kFp8 && good && t > 0) {
        const int pgv = s.pg0 + 2 * (t - 1);
        const int np = pages_in_tile(s, t - 1);
        for (int i = 0; good && i < np; ++i) {
          const int pv = ids.get(pgv + i, p, lane);
          good = issue_v(0, pv) && issue_v(1, pv);
        }
      }
    }
    }
    if (!good) {
      pend_a = -1;
      pend_valid = false;
      break;
    }
  }
  if (C::kCrossPiece && pend_a >= 0) (void)issue_v_tile(pend_a, pend_b);
  if (C::kCrossPiece && pend_valid) (void)issue_v_blocks_tile(pend_row, pend_two);
  // drain: every copy this warp issued must land before the CTA exits
  if (lane == 0) {
    for (uint32_t k = (cc > (uint32_t)kRing ? cc - kRing : 0); k < cc; ++k) {
      // block gather: only the first slot of a pair carries its copies (the last slot is never used)
      if (gather && (((k % kRing) & 1) || k % kRing == kRing - 1)) continue;
      (void)mbar_wait(cx.bar(kRingFull + k % kRing), (k / kRing) & 1, cx.budget, nullptr, p.err);
    }
    if constexpr (kFp8) {
      for (uint32_t k = (sc_cnt > (uint32_t)C::kScaleSlots ? sc_cnt - C::kScaleSlots : 0); k < sc_cnt; ++k)
        (void)mbar_wait(cx.bar(Bb::ScFull + k % C::kScaleSlots), (k / C::kScaleSlots) & 1, cx.budget, nullptr,
                        p.err);
      if constexpr (kGather8) {  // the V stages this warp issued
        for (uint32_t k = (vc > (uint32_t)C::kVStages ? vc - C::kVStages : 0); k < vc; ++k)
          (void)mbar_wait(cx.bar(Bb::StFull + C::kKStages + k % C::kVStages), (k / C::kVStages) & 1, cx.budget,
                          nullptr, p.err);
      }
    }
    if (issued_q) (void)mbar_wait(cx.bar(Bb::QFull + last_qb), last_q_parity, cx.budget, nullptr, p.err);
  }
  __syncwarp();
}

// E4M3: the V pages of every tile, in order, into the V stage ring (its own
// warp, so K pages are never queued behind V pages waiting for P.V). A slot
// is freed by the commit of the P.V MMAs that read it.
__device__ void producer_v_role(const DecodeParams& p, const CUtensorMap* vmap, const Ctx& cx, const int* s_cost,
                                const int* s_len, long long lo, long long hi) {
  using C = Cfg<true>;
  using Bb = Bars<true>;
  const int lane = threadIdx.x & 31;
  const uint64_t pol_stream = p.q_groups > 1 ? policy_evict_normal() : policy_evict_first();
  const SmemLayout L = smem_layout<true>(p.B);
  uint32_t vc = 0;  // V pages staged
  Seg s;
  bool ok = seg_first(s_cost, p.B, lo, hi, s);
  bool good = true;
  while (good && ok && seg_next(s_cost, s_len, p.B, p.piece_cost, lo, hi, s)) {
    if (*cx.abort) break;
    PageIds ids;
    ids.row = p.page_table + (size_t)s.b * p.max_pages;
    ids.pg1 = s.pg1;
    ids.start(s.pg0, p, lane);
    for (int pg = s.pg0; good && pg < s.pg1; ++pg) {
      const int id = ids.get(pg, p, lane);
      const uint32_t slot = C::kKStages + vc % C::kVStages, n = vc / C::kVStages;
      good = cx.wait(Bb::StEmpty + slot, (n & 1) ^ 1);
      __syncwarp();
      if (good && lane == 0) {
        const uint32_t dst = cx.base + L.stage + C::kKStages * kKTileBytes + (vc % C::kVStages) * kStageBytes;
        const uint32_t bar = cx.bar(Bb::StFull + slot);
        mbar_arrive_expect_tx(bar, (uint32_t)kStageBytes >> p.kv_fp4);
        tma_load_2d(dst, vmap, 0, id * kPageSize, bar, pol_stream);
        tma_load_2d(dst + 8192, vmap, 128, id * kPageSize, bar, pol_stream);
      }
      if (good) ++vc;
    }
  }
  // drain: every copy this warp issued must land before the CTA exits
  if (lane == 0) {
    for (uint32_t k = (vc > (uint32_t)C::kVStages ? vc - C::kVStages : 0); k < vc; ++k)
      (void)mbar_wait(cx.bar(Bb::StFull + C::kKStages + k % C::kVStages), (k / C::kVStages) & 1, cx.budget, nullptr,
                      p.err);
  }
  __syncwarp();
}

// E4M3: the largest V scale of each sequence piece (vref), published for the
// softmax warps before they form the piece's first P (two slots, so this warp
// works up to two pieces ahead).
template <bool kGather8>
__device__ void vref_role(const DecodeParams& p, const Ctx& cx, const int* s_cost, const int* s_len, long long lo,
                          long long hi, float* s_vref) {
  using Bb = Bars<true>;
  const int lane = threadIdx.x & 31;
  uint32_t piece = 0;
  Seg s;
  bool ok = seg_first(s_cost, p.B, lo, hi, s);
  while (ok && seg_next(s_cost, s_len, p.B, p.piece_cost, lo, hi, s)) {
    if (*cx.abort) break;
    const uint32_t slot = piece & 1, n = piece >> 1;
    // lane i takes page g + i of each group of 32: its 64 scales in 16 vector loads
    const int32_t* row = p.page_table + (size_t)s.b * p.max_pages;
    float mx = 0.0f;
    if constexpr (kGather8) {
      // block gather: the piece's virtual blocks [8 pg0, 8 pg1) -- the selected blocks, then the block of the
      // last token -- four a lane per round (block id, page id, then its 8 scales); a bad block or page id
      // (reported by the producer) is read as block 0 / page 0, as the producer reads it
      const int len = clamp_len(__ldg(p.seq_lens + s.b), p.max_pages * kPageSize, nullptr);
      const int nb = selected_blocks(len, p.n_blocks, s.b, p.max_blocks, nullptr);
      const int cur = (len - 1) >> 3, nvb = len > 0 ? nb + 1 : 0;
      const int vb_hi = min(8 * s.pg1, nvb);
      const int32_t* bidx = p.block_idx + (size_t)s.b * p.max_blocks;
      for (int vb0 = 8 * s.pg0; vb0 < vb_hi; vb0 += 128) {
        int r[4], id[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int vb = vb0 + 32 * u + lane;
          r[u] = vb < vb_hi ? (vb < nb ? __ldg(bidx + vb) : cur) : -1;
          if (vb < nb && (r[u] < 0 || r[u] >= cur)) r[u] = 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          id[u] = r[u] >= 0 ? __ldg(row + ((8 * r[u]) >> 6)) : 0;
          if (id[u] < 0 || id[u] >= p.num_pages) id[u] = 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (r[u] < 0) continue;
          const int vb = vb0 + 32 * u + lane;
          const int cnt = vb < nb ? 8 : len - 8 * cur;  // rows of the block that hold tokens
          const float4* sc = reinterpret_cast<const float4*>(p.v_scale + (size_t)id[u] * kPageSize + ((8 * r[u]) & 63));
          const float4 a = __ldg(sc), b4 = __ldg(sc + 1);
          const float v8[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (k < cnt) mx = fmaxf(mx, v8[k]);
        }
      }
    }
    for (int g = s.pg0; !kGather8 && g < s.pg1; g += 32) {
      const int pg = g + lane;
      if (pg < s.pg1) {
        const int id = __ldg(row + pg);
        if (id >= 0 && id < p.num_pages) {  // a bad id is reported by the producer warps
          const int rows = min(kPageSize, s.len - pg * kPageSize);  // scales of unused rows are never read
          const float4* sc = reinterpret_cast<const float4*>(p.v_scale + (size_t)id * kPageSize);
          float4 v[16];
#pragma unroll
          for (int r4 = 0; r4 < 16; ++r4) v[r4] = (4 * r4 < rows) ? __ldg(sc + r4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int r4 = 0; r4 < 16; ++r4) {
            if (4 * r4 + 0 < rows) mx = fmaxf(mx, v[r4].x);
            if (4 * r4 + 1 < rows) mx = fmaxf(mx, v[r4].y);
            if (4 * r4 + 2 < rows) mx = fmaxf(mx, v[r4].z);
            if (4 * r4 + 3 < rows) mx = fmaxf(mx, v[r4].w);
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (!cx.wait(Bb::VRefEmpty + slot, (n & 1) ^ 1)) break;
    __syncwarp();
    if (lane == 0) {
      s_vref[slot] = mx > 0.0f ? mx : 1.0f;
      mbar_arrive(cx.bar(Bb::VRefFull + slot));
    }
    __syncwarp();
    ++piece;
  }
}

// ---------------------------------------------------------------- shared-memory vectors
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------- MMA issue
template <bool kFp8, bool kMtp, bool kGather8 = false>
__device__ void mma_role(const DecodeParams& p, const Ctx& cx, const int* s_cost, const int* s_len, long long lo,
                         long long hi, uint32_t tmem) {
  using C = Cfg<kFp8, kMtp>;
  using Bb = Bars<kFp8, kMtp>;
  const SmemLayout L = smem_layout<kFp8, kMtp>(p.B);
  uint32_t cc = 0, seg_i = 0, s_cnt = 0, p_cnt = 0;
  uint32_t vc = 0;  // E4M3: V pages consumed from the V stage ring
  Seg s;
  bool ok = seg_first(s_cost, p.B, lo, hi, s);
  bool alive = true;
  Seg pend_s{};        // tile stream: the tile whose P.V is still to be issued
  int pend_t = -1;
  uint32_t pend_piece = 0;

  // One thread runs this role (the rest of its warp waits at the CTA's final
  // barrier): it polls the barriers, zeroes the rows past a partial last V
  // page, issues every MMA and the commits that track them. A warp whose
  // lanes diverge around each issue block pays for the reconvergence.
  auto wait_all = [&](int bar, uint32_t parity) -> bool { return cx.wait(bar, parity); };
  const uint32_t idesc_a_fmt = p.kv_fp4 ? kIdescAE2M1 : 0u;  // E4M3 kernel on a 4-bit cache
  // block gather: operand chunks are pairs of adjacent ring slots, in the producer's sequence
  const bool gather = !kFp8 && !kMtp && p.block_idx != nullptr;
  constexpr bool gather8 = kGather8;  // E4M3 block gather: [block][half] staging
  auto next_pair = [&](uint32_t& slot, uint32_t& ph) {
    if (cc % C::kSlots == C::kSlots - 1) ++cc;
    slot = cc % C::kSlots;
    ph = (cc / C::kSlots) & 1;
    cc += 2;
  };
  auto do_s = [&](uint32_t qb) -> bool {
    const uint32_t buf = s_cnt & 1, n = s_cnt >> 1;
    if (!wait_all(Bb::SEmpty + buf, (n & 1) ^ 1)) return false;
    const uint32_t d_tmem = tmem + buf * C::kSCols;
    if constexpr (kFp8) {
      // 8-bit S^T: A = the raw K tile (tokens x dims, K-major), B = both Q
      // terms stacked (128 rows [term][head] x dims, K-major): N = 128, so S^T
      // holds K.t1^T in columns 0-63 and K.t2^T in 64-127; K = 32 dims per MMA
      const uint32_t kslot = cc % C::kKStages;
      if (!wait_all(Bb::StFull + kslot, (cc / C::kKStages) & 1)) return false;
      {
        tc_fence_after();
        const uint32_t ka = cx.base + L.stage + kslot * kKTileBytes;
        const uint32_t qa = cx.base + L.q + qb * C::kQ * kQBytes;
        if constexpr (gather8) {  // block gather: [block][half][8 rows]: half h at 1 KB * h, 8-row groups 2 KB apart
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f8(d_tmem, smem_desc(ka + h * 1024 + ks * 32, 16, 2048, 2),
                        smem_desc(qa + h * 16384 + ks * 32, 16, 1024, 2), idesc_s_e4m3() | idesc_a_fmt, (h | ks) != 0);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f8(d_tmem, smem_desc(ka + h * 16384 + ks * 32, 16, 1024, 2),
                        smem_desc(qa + h * 16384 + ks * 32, 16, 1024, 2), idesc_s_e4m3() | idesc_a_fmt, (h | ks) != 0);
        }
        tc_commit(cx.bar(Bb::StEmpty + kslot));
        tc_commit(cx.bar(Bb::SFull + buf));
      }
      ++cc;
      ++s_cnt;
      return true;
    } else if (gather) {
      // K pair h: dim blocks 2h + e at + 1 KB * e, 8-row groups 2 KB apart
      for (int h = 0; h < 2; ++h) {
        uint32_t slot, ph;
        next_pair(slot, ph);
        if (!wait_all(Bb::Full + slot, ph)) return false;
        tc_fence_after();
        const uint32_t a0 = cx.base + L.ring + slot * kSlotBytes;
        for (int e = 0; e < 2; ++e) {
          const int d = 2 * h + e;
          const uint32_t b0 = cx.base + L.q + qb * C::kQ * kQBytes + d * C::kQ * 8192;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(d_tmem, smem_desc_sw128(a0 + e * 1024 + kk * 32, 16, 2048), smem_desc_sw128(b0 + kk * 32, 16, 1024),
                   idesc_s<kFp8, kMtp>(), (d | kk) != 0);
        }
        tc_commit(cx.bar(Bb::Empty + slot));
      }
      tc_commit(cx.bar(Bb::SFull + buf));
      ++s_cnt;
      return true;
    } else {
      for (int d = 0; d < 4; ++d) {
        const uint32_t slot = cc % C::kSlots, ph = (cc / C::kSlots) & 1;
        if (!wait_all(Bb::Full + slot, ph)) return false;
        {
          tc_fence_after();
          const uint32_t a0 = cx.base + L.ring + slot * kSlotBytes;
          const uint32_t b0 = cx.base + L.q + qb * C::kQ * kQBytes + d * C::kQ * 8192;  // 64 kQ rows
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(d_tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), smem_desc_sw128(b0 + kk * 32, 16, 1024),
                   idesc_s<kFp8, kMtp>(), (d | kk) != 0);
          tc_commit(cx.bar(Bb::Empty + slot));
        }
        ++cc;
      }
      tc_commit(cx.bar(Bb::SFull + buf));
      ++s_cnt;
      return true;
    }
  };
  // P.V of tile t of piece `piece` (sg)
  auto do_pv = [&](const Seg& sg, int t, uint32_t piece) -> bool {
    const uint32_t buf = p_cnt % C::kPBufs, n = p_cnt / C::kPBufs;
    const bool first_of_seg = t == 0;
    // pieces cycle through the O^T buffers; the first P.V of piece j
    // overwrites the buffer of piece j - kOBufs, whose epilogue must be done
    const uint32_t obuf = piece % C::kOBufs;
    if (first_of_seg && !wait_all(Bb::OFree + obuf, ((piece / C::kOBufs) & 1) ^ 1)) return false;
    if (!wait_all(Bb::PFull + buf, n & 1)) return false;
    const int pga = sg.pg0 + 2 * t;
    const int np = pages_in_tile(sg, t);
    if constexpr (kFp8) {
      // 8-bit P.V: A = the raw staged V page (dims x tokens, 128-byte swizzle,
      // one 128-dim box per half), B = both P terms side by side (tokens x
      // 128 [term][head], 128-byte swizzle): N = 128, so O^T half hf holds
      // V^T.x1 in columns 0-63 and V^T.x2 in 64-127; K = 32 tokens per MMA
      // both pages of the tile are waited for (and a partial last page zeroed
      // past its rows) first, then all the tile's P.V MMAs go out as one batch
      uint32_t vs[2];
      for (int i = 0; i < np; ++i) {
        const int nv = min(kPageSize, sg.len - (pga + i) * kPageSize);  // valid rows of this page
        const uint32_t vslot = C::kKStages + (vc + i) % C::kVStages;
        if (!wait_all(Bb::StFull + vslot, ((vc + i) / C::kVStages) & 1)) return false;
        vs[i] = cx.base + L.stage + C::kKStages * kKTileBytes + ((vc + i) % C::kVStages) * kStageBytes;
        if constexpr (gather8) {
          // blocks past the end arrived as zeros; the rows past the last token inside the last block hold
          // other tokens' codes (possibly 0x7F, NaN): zero them ([block][half][8 rows x 128 B] layout)
          const int nz = min(kPageSize, (nv + 7) & ~7);
          if (nv < nz) {
            for (int r = nv; r < nz; ++r)
              for (int hf = 0; hf < 2; ++hf)
                for (int off = 0; off < 128; off += 16)
                  st_shared_v4(vs[i] + (r >> 3) * 2048 + hf * 1024 + (r & 7) * 128 + off, make_uint4(0u, 0u, 0u, 0u));
            fence_proxy_async_smem();
          }
        } else if (nv < kPageSize && !p.kv_fp4) {  // E2M1 has no NaN code: a 4-bit page needs no zeroing
          // rows [nv, 64) of both boxes (whole 128 B rows): code 0x7F is NaN and 0 * NaN would poison P.V
          const int nbytes = (kPageSize - nv) * 128;
          for (int off = 0; off < nbytes; off += 16) {
            st_shared_v4(vs[i] + nv * 128 + off, make_uint4(0u, 0u, 0u, 0u));
            st_shared_v4(vs[i] + 8192 + nv * 128 + off, make_uint4(0u, 0u, 0u, 0u));
          }
          fence_proxy_async_smem();
        }
      }
      {
        tc_fence_after();
        for (int i = 0; i < np; ++i) {
          const uint32_t bp = cx.base + L.p + buf * C::kQ * kPBytes + i * 8192;  // token rows 64i..
          if constexpr (gather8) {  // block gather: [block][half][8 rows], 8-token groups 2 KB apart
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
              for (int ks = 0; ks < 2; ++ks)
                tc_mma_f8(tmem + tmem_o<kFp8, kMtp>() + hf * 128, smem_desc(vs[i] + hf * 1024 + ks * 8192, 16, 2048, 2),
                          smem_desc(bp + ks * 4096, 16, 1024, 2), idesc_o_e4m3() | idesc_a_fmt,
                          !(first_of_seg && i == 0 && ks == 0));
          } else {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
              for (int ks = 0; ks < 2; ++ks)
                tc_mma_f8(tmem + tmem_o<kFp8, kMtp>() + hf * 128, smem_desc(vs[i] + hf * 8192 + ks * 4096, 16, 1024, 2),
                          smem_desc(bp + ks * 4096, 16, 1024, 2), idesc_o_e4m3() | idesc_a_fmt,
                          !(first_of_seg && i == 0 && ks == 0));
          }
          // the V page's stage is free once these MMAs are done
          tc_commit(cx.bar(Bb::StEmpty + C::kKStages + (vc + i) % C::kVStages));
        }
      }
      vc += np;
    } else if (gather) {
      // V pair of page i: block j at 4 KB * j, dim block c at + 1 KB * c (64-dim halves 1 KB apart,
      // 8-token groups 4 KB apart); blocks past the end arrive as zeros, so only the rows past the last
      // token of a partial block need zeroing
      for (int i = 0; i < np; ++i) {
        const int nv = min(kPageSize, sg.len - (pga + i) * kPageSize);
        uint32_t slot, ph;
        next_pair(slot, ph);
        if (!wait_all(Bb::Full + slot, ph)) return false;
        const uint32_t a0 = cx.base + L.ring + slot * kSlotBytes;
        const int nz = min(kPageSize, (nv + 7) & ~7);
        if (nv < nz) {
          for (int r = nv; r < nz; ++r)
            for (int c = 0; c < 4; ++c)
              for (int off = 0; off < 128; off += 16)
                st_shared_v4(a0 + (r >> 3) * 4096 + c * 1024 + (r & 7) * 128 + off, make_uint4(0u, 0u, 0u, 0u));
          fence_proxy_async_smem();
        }
        tc_fence_after();
        const uint32_t bp = cx.base + L.p + buf * C::kQ * kPBytes + i * 8192;
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(tmem + tmem_o<kFp8, kMtp>() + obuf * 128 + hf * C::kOHalfCols,
                   smem_desc_sw128(a0 + hf * 2048 + kk * 8192, 1024, 4096), smem_desc_sw128(bp + kk * 2048, kPBytes, 1024),
                   idesc_o<kFp8, kMtp>(), !(first_of_seg && i == 0 && kk == 0));
        }
        tc_commit(cx.bar(Bb::Empty + slot));
      }
    } else {
    for (int i = 0; i < np; ++i) {
      const int nv = min(kPageSize, sg.len - (pga + i) * kPageSize);  // valid rows of this page
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t slot = cc % C::kSlots, ph = (cc / C::kSlots) & 1;
        if (!wait_all(Bb::Full + slot, ph)) return false;
        const uint32_t a0 = cx.base + L.ring + slot * kSlotBytes;
        if (!kFp8 && nv < kPageSize) {
          // rows [nv, 64) of both 64-dim blocks (whole 128 B rows, so the
          // swizzle does not matter), 16 B per store
          const int nbytes = (kPageSize - nv) * 128;
          for (int off = 0; off < nbytes; off += 16) {
            st_shared_v4(a0 + nv * 128 + off, make_uint4(0u, 0u, 0u, 0u));
            st_shared_v4(a0 + 8192 + nv * 128 + off, make_uint4(0u, 0u, 0u, 0u));
          }
          fence_proxy_async_smem();
        }
        {
          tc_fence_after();
          // token rows 64i.. of the P buffer; query token t's [tokens x 64 heads] block at t * kPBytes
          const uint32_t bp = cx.base + L.p + buf * C::kQ * kPBytes + i * 8192;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(tmem + tmem_o<kFp8, kMtp>() + obuf * 128 + hf * C::kOHalfCols,
                   smem_desc_sw128(a0 + kk * 2048, 8192, 1024), smem_desc_sw128(bp + kk * 2048, kPBytes, 1024),
                   idesc_o<kFp8, kMtp>(),
                   !(first_of_seg && i == 0 && kk == 0));
          tc_commit(cx.bar(Bb::Empty + slot));
        }
        ++cc;
      }
    }
    }
    {
      tc_commit(cx.bar(Bb::PEmpty + buf));
    }
    ++p_cnt;
    return true;
  };

  while (alive && ok && seg_next(s_cost, s_len, p.B, p.piece_cost, lo, hi, s)) {
    const uint32_t qb = seg_i % C::kQBufs, qn = seg_i / C::kQBufs;
    if (!wait_all((kFp8 ? Bb::QReady : Bb::QFull) + qb, qn & 1)) break;
    const int T = tiles_of(s);
    if constexpr (C::kCrossPiece) {
      // S(g), then P.V(g - 1), in the producer's order
      for (int t = 0; alive && t < T; ++t) {
        alive = do_s(qb);
        if (alive && t == T - 1) tc_commit(cx.bar(Bb::QEmpty + qb));
        if (alive && pend_t >= 0) alive = do_pv(pend_s, pend_t, pend_piece);
        pend_s = s;
        pend_t = t;
        pend_piece = seg_i;
      }
    } else {
      // S^T(t) goes out before P.V(t - kLag): with kLag = 2 the K stage of tile t is released a tile
      // earlier than in strict alternation (S(t) waits only for the softmax to have read S(t - 2), which
      // it does before it forms P(t - 2)), so the next K tiles are requested sooner
      constexpr int kLag = 2;
      for (int t = 0; alive && t < T + kLag; ++t) {
        if (t < T) {
          alive = do_s(qb);
          if (alive && t == T - 1) tc_commit(cx.bar(Bb::QEmpty + qb));
        }
        if (alive && t >= kLag) alive = do_pv(s, t - kLag, seg_i);
      }
    }
    ++seg_i;
  }
  if (C::kCrossPiece && alive && pend_t >= 0) (void)do_pv(pend_s, pend_t, pend_piece);
  // drain: wait for every MMA this thread issued before TMEM is released
  {
    tc_commit(cx.bar(Bb::Drain));
    (void)mbar_wait(cx.bar(Bb::Drain), 0, cx.budget, nullptr, p.err);
  }
}

// ---------------------------------------------------------------- softmax
// Warpgroup g of the softmax warps owns heads [h0, h0 + kHpt), h0 = g * kHpt
// (kHpt = 64 / groups); its thread r (0..127) owns TMEM lane r: token r of
// the tile in S^T, dim r of each 128-dim half of O^T. The row statistics of
// different heads never meet, so each group keeps its own reference maxima,
// rescale decisions and named barrier.

// Butterfly reduce-scatter over the warp: afterwards lane l holds the result
// for columns (N / 32) * l + i, i < N / 32, in v[i] (N >= 32); with N = 16,
// lanes 2k and 2k + 1 both hold column k in v[0] (the last step is a plain
// reduction between lane pairs).
template <int N, bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N], int lane) {
  static_assert(N % 32 == 0 || N == 16, "columns");
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = (N / 2) >> step;
    const int o = 16 >> step;
    if (half >= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float keep = up ? v[i + half] : v[i];
        const float send = up ? v[i] : v[i + half];
        const float other = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = kMax ? fmaxf(keep, other) : keep + other;
      }
    } else {
      const float other = __shfl_xor_sync(0xffffffffu, v[0], o);
      v[0] = kMax ? fmaxf(v[0], other) : v[0] + other;
    }
  }
}
// Stores the reduce-scattered columns of a group's kHpt heads at dst[0 .. kHpt) (one copy each).
template <int kHpt>
__device__ __forceinline__ void store_scattered(float* dst, const float (&v)[kHpt], int lane) {
  if constexpr (kHpt >= 32) {
#pragma unroll
    for (int i = 0; i < kHpt / 32; ++i) dst[(kHpt / 32) * lane + i] = v[i];
  } else {
    if ((lane & 1) == 0) dst[lane >> 1] = v[0];
  }
}

// kHpt columns of one S^T row (taddr: the group's first column) as
// log2-domain logits minus the reference maxima: x[h] = S[h] * mult - m[h]
// (E4M3: S is the sum of the two Q terms' columns, 64 apart); m = nullptr
// gives the plain logits. Rows past the sequence read -inf (only a partial
// tile has such rows). Returns the largest x. m is 16-byte aligned, uniform.
template <bool kFp8, int kHpt>
__device__ __forceinline__ float load_logits(uint32_t taddr, bool full, bool valid, float mult, const float* m,
                                             float (&x)[kHpt]) {
  constexpr int kLd = kHpt < 32 ? kHpt : 32;  // columns per tcgen05.ld
#pragma unroll
  for (int q = 0; q < kHpt / kLd; ++q) {
    tmem_ld_cols<kLd>(taddr + q * kLd, x + q * kLd);
    if constexpr (kFp8) {
      float y[kLd];
      tmem_ld_cols<kLd>(taddr + 64 + q * kLd, y);
      tc_wait_ld();
#pragma unroll
      for (int h = 0; h < kLd; ++h) x[q * kLd + h] += y[h];
    }
  }
  if constexpr (!kFp8) tc_wait_ld();
#pragma unroll
  for (int i = 0; i < kHpt / 4; ++i) {
    const float4 r = m ? reinterpret_cast<const float4*>(m)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    x[4 * i] = fmaf(x[4 * i], mult, -r.x);
    x[4 * i + 1] = fmaf(x[4 * i + 1], mult, -r.y);
    x[4 * i + 2] = fmaf(x[4 * i + 2], mult, -r.z);
    x[4 * i + 3] = fmaf(x[4 * i + 3], mult, -r.w);
  }
  if (!full) {
#pragma unroll
    for (int h = 0; h < kHpt; ++h) x[h] = valid ? x[h] : -INFINITY;
  }
  float dm = -INFINITY;
#pragma unroll
  for (int i = 0; i < kHpt / 4; ++i)
    dm = fmaxf(dm, fmaxf(fmaxf(x[4 * i], x[4 * i + 1]), fmaxf(x[4 * i + 2], x[4 * i + 3])));
  return dm;
}

// E4M3: the bf16 Q of a piece (four 64-dim boxes of [64 heads x 128 B],
// 128-byte swizzle, as TMA loaded it) becomes, in place, two E4M3 terms
// t1 + t2 of Q * 2^e: 128-dim box b (16 KB at 16 KB * b) holds t1 of the 64
// heads, then t2 ([128 rows x 128 B], 128-byte swizzle). 2^e is the largest
// power of two with max |Q| * 2^e <= 448 (the E4M3 maximum); t1 rounds the
// scaled value, t2 the remainder, which is exact unless it falls below the
// E4M3 normal range (absolute error at most 2^-10 there, i.e. 2^-18.8 of the
// largest |Q|: elements down to 2^-10.8 of it are held exactly). Run by all
// kThreadsAll softmax threads: thread t takes head t % 64 and dims
// [D (t / 64), +D), D = 256 / (kThreadsAll / 64). scratch: one float per
// warp. Returns 2^-e. Ends with every thread's terms written and fenced for
// the tensor cores (the caller then arrives on the ready barrier).
template <int kThreadsAll>
__device__ __noinline__ float split_q_e4m3(uint32_t q_addr, float* scratch, int tid) {
  constexpr int kParts = kThreadsAll / 64, kDims = kHeadDim / kParts, kIn = kDims / 8;
  static_assert(kDims % 16 == 0, "16-dim output chunks");
  const int h = tid & 63, part = tid >> 6, d0 = part * kDims;
  uint4 v[kIn];  // input chunk j: dims [d0 + 8j, +8) in bf16 box (d0 + 8j) / 64
#pragma unroll
  for (int j = 0; j < kIn; ++j) {
    const int d = d0 + 8 * j;
    v[j] = ld_shared_v4(q_addr + (d >> 6) * 8192 + h * 128 + ((((d & 63) >> 3) ^ (h & 7)) << 4));
  }
  float mx = 0.0f;
#pragma unroll
  for (int j = 0; j < kIn; ++j) {
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) scratch[tid >> 5] = mx;
  barrier_softmax_all<kThreadsAll>();  // every thread has its Q values: the buffer may be overwritten
  float gm = 0.0f;
#pragma unroll
  for (int w = 0; w < kThreadsAll / 32; ++w) gm = fmaxf(gm, scratch[w]);
  int e = 0;
  if (gm > 0.0f && gm <= 3.0e38f) {
    const uint32_t bits = __float_as_uint(gm);
    const int E = (int)((bits >> 23) & 0xFFu) - 127;
    e = ((bits & 0x7FFFFFu) <= 0x600000u ? 8 : 7) - E;  // gm * 2^e in (224, 448]
    e = max(-126, min(126, e));
  }
  const float sq = __uint_as_float((uint32_t)(e + 127) << 23);
#pragma unroll
  for (int k = 0; k < kDims / 16; ++k) {  // output chunk: dims [d0 + 16k, +16) = input chunks 2k, 2k + 1
    uint32_t t1[4], t2[4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 in = v[2 * k + u];
      const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // two output words of four codes each
        uint32_t c1w = 0, c2w = 0;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t wd = w[2 * i + m];
          const float2 a = make_float2(__uint_as_float(wd << 16) * sq, __uint_as_float(wd & 0xFFFF0000u) * sq);
          const __nv_fp8x2_storage_t c1 = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
          const __half2_raw d1 = __nv_cvt_fp8x2_to_halfraw2(c1, __NV_E4M3);
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&d1));
          const __nv_fp8x2_storage_t c2 =
              __nv_cvt_float2_to_fp8x2(make_float2(a.x - b.x, a.y - b.y), __NV_SATFINITE, __NV_E4M3);
          c1w |= (uint32_t)c1 << (16 * m);
          c2w |= (uint32_t)c2 << (16 * m);
        }
        t1[2 * u + i] = c1w;
        t2[2 * u + i] = c2w;
      }
    }
    const int d = d0 + 16 * k;
    const uint32_t o = (d >> 7) * 16384 + h * 128 + ((((d & 127) >> 4) ^ (h & 7)) << 4);
    st_shared_v4(q_addr + o, make_uint4(t1[0], t1[1], t1[2], t1[3]));
    st_shared_v4(q_addr + kQTermBytes + o, make_uint4(t2[0], t2[1], t2[2], t2[3]));
  }
  fence_proxy_async_smem();
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// The group's O^T columns (this thread's TMEM lane, both 128-dim halves)
// times col_scale[head - h0]; E4M3: both terms' columns of each head.
template <bool kFp8, int kHpt, int kHalfCols>
__device__ __forceinline__ void scale_o_columns(uint32_t taddr_o, int h0, const float* col_scale) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
    for (int tm = 0; tm < (kFp8 ? 2 : 1); ++tm) {
      constexpr int kLd = kHpt < 32 ? kHpt : 32;
#pragma unroll
      for (int q = 0; q < kHpt / kLd; ++q) {
        const uint32_t a = taddr_o + hf * kHalfCols + tm * 64 + h0 + q * kLd;
        float o[kLd];
        tmem_ld_cols<kLd>(a, o);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < kLd; ++h) o[h] *= col_scale[q * kLd + h];
        tmem_st_cols<kLd>(a, o);
      }
    }
  }
  tc_wait_st();
}
// The E4M3 softmax calls the rescale out of line: inlined into its loop it cost that loop spilled registers.
template <int kHpt, int kHalfCols>
__device__ __noinline__ void scale_o_columns_e4m3(uint32_t taddr_o, int h0, const float* col_scale) {
  scale_o_columns<true, kHpt, kHalfCols>(taddr_o, h0, col_scale);
}

template <bool kFp8>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (kFp8) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <bool kFp8, bool kMtp>
__device__ void softmax_role(const DecodeParams& p, const Ctx& cx, const int* s_cost, const int* s_len,
                             long long lo, long long hi, uint32_t tmem, int c, uint8_t* gbase) {
  using C = Cfg<kFp8, kMtp>;
  using Bb = Bars<kFp8, kMtp>;
  constexpr int kHpt = C::kHpt;          // columns per thread
  constexpr int kCols = C::kCols;        // [query token][head] columns of the statistics
  const int g = threadIdx.x >> 7;        // head group (with two query tokens: the query token)
  const int row = threadIdx.x & 127;     // TMEM lane = token of the tile = dim of each O^T half
  const int quad = row >> 5, lane = row & 31;
  const int h0 = g * kHpt;
  const int qg = q_groups_of<kFp8, kMtp>(p);
  const int tau = (c % qg) * C::kQ + (kMtp ? g : 0);  // the query token this thread serves
  const SmemLayout L = smem_layout<kFp8, kMtp>(p.B);
  float* red = reinterpret_cast<float*>(gbase + L.red);  // [4][kCols] per-warp partial reductions
  float* mref = red + 4 * kCols;                         // [kCols] reference maxima (log2 units), uniform
  float* alpha = mref + kCols;                           // [kCols] rescale factors, uniform
  float* inv_l = alpha + kCols;                          // [2][kCols] 1/l of the piece in O^T buffer i
  float* qscratch = inv_l + 2 * kCols;                   // [8] E4M3: per-warp max |Q|
  float* s_vref = qscratch + kCols;                      // [2] E4M3: largest V scale of a piece
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const uint32_t taddr_o0 = tmem + lane_base + tmem_o<kFp8, kMtp>();
  const float c2 = p.scale * kLog2e;
  uint32_t s_cnt = 0, p_cnt = 0;
  // With n = kPBufs P buffers, P.V(g) completes phase g/n of p_empty[g % n].
  // Before P(g) is written the softmax has seen P.V(g-n) complete, and
  // P.V(g+n) cannot start before P(g+n) exists, so when it waits for P.V(g)
  // that barrier is at phase g/n or just past it: the parity wait is exact. Completion of P.V(g) implies that of
  // every earlier MMA (one issuing thread, commits track all prior MMAs).
  auto wait_pv = [&](uint32_t gi) -> bool {
    return cx.wait(Bb::PEmpty + gi % C::kPBufs, (gi / C::kPBufs) & 1);
  };
  // Pieces cycle through the O^T buffers. A piece's O^T / l is written out
  // once the next piece's first P has been handed over (its last P.V was
  // issued before that piece's first S), so the softmax warps go on to the
  // next piece without waiting for the previous one's last P.V (with one
  // buffer, E4M3, the next piece's first P.V waits for this).
  bool pend = false;
  uint32_t pend_pv = 0, pend_obuf = 0;
  size_t pend_slot = 0;
  auto write_o = [&]() -> bool {
    if (!wait_pv(pend_pv)) return false;
    tc_fence_after();
    const uint32_t ta = taddr_o0 + pend_obuf * 128;
    const float* il = inv_l + pend_obuf * kCols + h0;
    float* dst = p.part_o + (pend_slot * (C::kQ * kHeads) + h0) * kHeadDim;  // slot: [query token][head][dim]
    constexpr int kHalfCols = C::kOHalfCols;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      constexpr int kLd = kHpt < 32 ? kHpt : 32;
#pragma unroll
      for (int q = 0; q < kHpt / kLd; ++q) {
        float o[kLd];
        tmem_ld_cols<kLd>(ta + hf * kHalfCols + h0 + q * kLd, o);
        if constexpr (kFp8) {  // + the second P term's columns
          float o2[kLd];
          tmem_ld_cols<kLd>(ta + hf * kHalfCols + 64 + h0 + q * kLd, o2);
          tc_wait_ld();
#pragma unroll
          for (int h = 0; h < kLd; ++h) o[h] += o2[h];
        } else {
          tc_wait_ld();
        }
        const int dim = hf * 128 + row;
#pragma unroll
        for (int h = 0; h < kLd; ++h) dst[(q * kLd + h) * kHeadDim + dim] = o[h] * il[q * kLd + h];
      }
    }
    tc_fence_before();
    mbar_arrive(cx.bar(Bb::OFree + pend_obuf));
    pend = false;
    return true;
  };
  Seg s;
  bool ok = seg_first(s_cost, p.B, lo, hi, s);
  uint32_t piece = 0;

  while (ok && seg_next(s_cost, s_len, p.B, p.piece_cost, lo, hi, s)) {
    const uint32_t obuf = piece % C::kOBufs;
    const uint32_t taddr_o = taddr_o0 + obuf * 128;
    // E4M3: P enters the 8-bit P.V as P * v_scale * pscale (<= 256); O^T is
    // then pscale times too large, which the epilogue undoes. Q enters S^T
    // as 2^e Q, undone by qinv in the token multiplier.
    float pscale = 1.0f, qinv = 1.0f;
    if constexpr (kFp8) {
      const uint32_t vslot = piece & 1;
      if (!cx.wait(Bb::VRefFull + vslot, (piece >> 1) & 1)) return;
      pscale = kPScale / s_vref[vslot];
      mbar_arrive(cx.bar(Bb::VRefEmpty + vslot));
      // Q of the piece -> E4M3 terms (the producer loaded it once the previous
      // piece's S MMAs were done)
      if (!cx.wait(Bb::QFull, piece & 1)) return;
      qinv = split_q_e4m3<C::kSoftmaxThreads>(cx.base + L.q, qscratch, threadIdx.x);
      mbar_arrive(cx.bar(Bb::QReady));
    }
    if (row < kHpt) mref[h0 + row] = -INFINITY;
    barrier_group(g);
    float lp[kHpt];  // this thread's share of the softmax denominators
#pragma unroll
    for (int h = 0; h < kHpt; ++h) lp[h] = 0.0f;
    const int T = tiles_of(s);
    const int vis_len = min(s.len, s.len - (p.n_query - 1 - tau));
    for (int t = 0; t < T; ++t) {
      const int tok0 = (s.pg0 + 2 * t) * kPageSize;
      // valid rows of the tile: query token tau of T sees the first len - (T - 1 - tau) positions (a
      // token past the last, which only fills a group, is clamped to len; its result is not used)
      const int rows = max(0, min(pages_in_tile(s, t) * kPageSize, vis_len - tok0));
      const bool full = rows == 128, valid = row < rows;
      // E4M3: this token's K and V scales (the tile's scale block, slot = tile count)
      float kmul = c2, vmul = 1.0f;
      if constexpr (kFp8) {
        const uint32_t slot = p_cnt % C::kScaleSlots;
        if (!cx.wait(Bb::ScFull + slot, (p_cnt / C::kScaleSlots) & 1)) return;
        const float* sc = reinterpret_cast<const float*>(gbase + L.scales + slot * kScaleBytes);
        if (valid) {
          kmul = c2 * qinv * sc[row];
          vmul = sc[128 + row] * pscale;
        }
        mbar_arrive(cx.bar(Bb::ScEmpty + slot));
      }
      const uint32_t sbuf = s_cnt & 1;
      const uint32_t taddr_s = tmem + lane_base + sbuf * C::kSCols + h0;
      if (!cx.wait(Bb::SFull + sbuf, (s_cnt >> 1) & 1)) return;
      tc_fence_after();
      float x[kHpt];
      // x = logit - reference maximum (log2 units)
      const bool mine = load_logits<kFp8, kHpt>(taddr_s, full, valid, kmul, mref + h0, x) > rescale_threshold<kFp8>();
      // ---- does any logit of the group's heads exceed its reference maximum by 2^threshold?
      if (barrier_group_or(g, mine)) {
        (void)load_logits<kFp8, kHpt>(taddr_s, full, valid, kmul, nullptr, x);
        warp_reduce_scatter<kHpt, true>(x, lane);  // x is reloaded below
        store_scattered<kHpt>(red + quad * kCols + h0, x, lane);
        barrier_group(g);
        if (row < kHpt) {
          const int h = h0 + row;
          const float m_old = mref[h];
          const float m_new =
              fmaxf(m_old, fmaxf(fmaxf(red[h], red[kCols + h]), fmaxf(red[2 * kCols + h], red[3 * kCols + h])));
          alpha[h] = ex2_approx(m_old - m_new);  // 0 while m_old = -inf
          mref[h] = m_new;
        }
        barrier_group(g);
        bool rescale_o = false;
        if (t > 0) {  // the first tile of a piece has nothing to rescale
#pragma unroll
          for (int h = 0; h < kHpt; ++h) {
            lp[h] *= alpha[h0 + h];
            rescale_o |= alpha[h0 + h] != 1.0f;
          }
        }
        if (rescale_o) {
          // O^T holds the previous tiles: wait for their last P.V, then scale the group's columns
          if (!wait_pv(p_cnt - 1)) return;
          tc_fence_after();
          if constexpr (kFp8)
            scale_o_columns_e4m3<kHpt, C::kOHalfCols>(taddr_o, h0, alpha + h0);
          else
            scale_o_columns<kFp8, kHpt, C::kOHalfCols>(taddr_o, h0, alpha + h0);
        }
        (void)load_logits<kFp8, kHpt>(taddr_s, full, valid, kmul, mref + h0, x);
      }
      tc_fence_before();
      mbar_arrive(cx.bar(Bb::SEmpty + sbuf));  // S^T buffer free for the tile after next
      ++s_cnt;
      // ---- P = exp2(x - mref): row sums in fp32; this token's P^T row (times
      // the V scale) into the P buffer, 16 B chunk j at ((j ^ (row & 7)) << 4)
      // (128-byte swizzle) as soon as it is formed. bf16: chunk j = heads
      // [8j, 8j + 8); E4M3: the row is [x1 of heads 0-63 | x2 of heads 0-63],
      // chunk j = x1 and chunk 4 + j = x2 of heads [16j, 16j + 16).
      const uint32_t pbuf = p_cnt % C::kPBufs;
      if (!cx.wait(Bb::PEmpty + pbuf, ((p_cnt / C::kPBufs) & 1) ^ 1)) return;
      // with two query tokens, token g's [tokens x 64 heads] block sits at g * kPBytes
      const uint32_t prow = cx.base + L.p + pbuf * C::kQ * kPBytes + (kMtp ? g * kPBytes : 0) + row * 128;
      constexpr int kHeadsPerChunk = kFp8 ? 16 : 8;
#pragma unroll
      for (int j = 0; j < kHpt / kHeadsPerChunk; ++j) {
        const int jj = (kMtp ? 0 : h0 / kHeadsPerChunk) + j;  // chunk index within the row
        uint32_t w1[4], w2[4];
#pragma unroll
        for (int k = 0; k < kHeadsPerChunk / 2; ++k) {
          const int h = j * kHeadsPerChunk + 2 * k;
          const float p0 = ex2_approx(x[h]);
          const float p1 = ex2_approx(x[h + 1]);
          lp[h] += p0;
          lp[h + 1] += p1;
          if constexpr (kFp8) {
            // x = P * v_scale * 2^5 / vref in [0, 256], as x1 + x2 (E4M3): x2 rounds x - x1,
            // formed in f16 (x1 is exact in f16, and so is the difference)
            const __half2 xh = __floats2half2_rn(p0 * vmul, p1 * vmul);
            const __nv_fp8x2_storage_t c1 =
                __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&xh), __NV_SATFINITE, __NV_E4M3);
            const __half2_raw d1 = __nv_cvt_fp8x2_to_halfraw2(c1, __NV_E4M3);
            const __half2 rh = __hsub2(xh, *reinterpret_cast<const __half2*>(&d1));
            const __nv_fp8x2_storage_t c2 =
                __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&rh), __NV_SATFINITE, __NV_E4M3);
            if ((k & 1) == 0) {  // two heads per 16 bits, four per word
              w1[k >> 1] = (uint32_t)c1;
              w2[k >> 1] = (uint32_t)c2;
            } else {
              w1[k >> 1] |= (uint32_t)c1 << 16;
              w2[k >> 1] |= (uint32_t)c2 << 16;
            }
          } else {
            w1[k] = pack2<kFp8>(p0, p1);
          }
        }
        st_shared_v4(prow + ((jj ^ (row & 7)) << 4), make_uint4(w1[0], w1[1], w1[2], w1[3]));
        if constexpr (kFp8)
          st_shared_v4(prow + (((4 + jj) ^ (row & 7)) << 4), make_uint4(w2[0], w2[1], w2[2], w2[3]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(cx.bar(Bb::PFull + pbuf));
      ++p_cnt;
      if (t == 0 && pend && !write_o()) return;
    }
    // ---- epilogue of this sequence piece: l = sum over the 128 lanes and the
    // LSE (final once the last P is out); O^T / l follows later (write_o)
    warp_reduce_scatter<kHpt, false>(lp, lane);
    barrier_group(g);  // earlier readers of red/alpha are done
    store_scattered<kHpt>(red + quad * kCols + h0, lp, lane);
    barrier_group(g);
    const size_t slot = ((size_t)(c / qg) + s.b) * qg + c % qg;
    if (row < kHpt) {
      const int h = h0 + row;
      const float l = red[h] + red[kCols + h] + red[2 * kCols + h] + red[3 * kCols + h];
      inv_l[obuf * kCols + h] = 1.0f / (l * pscale);
      p.part_lse[slot * (C::kQ * kHeads) + h] = (mref[h] + log2f(l)) * kLn2;
    }
    barrier_group(g);
    pend = true;
    pend_pv = p_cnt - 1;
    pend_obuf = obuf;
    pend_slot = slot;
    ++piece;
  }
  if (pend) (void)write_o();
}

template <bool kFp8, bool kMtp, bool kGather8 = false>
__global__ void __launch_bounds__(Cfg<kFp8, kMtp>::kThreads)
    decode_split_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
  using C = Cfg<kFp8, kMtp>;
  using Bb = Bars<kFp8, kMtp>;
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  const uint32_t raw = smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = dyn_smem + (base - raw);
  const SmemLayout L = smem_layout<kFp8, kMtp>(p.B);
  int* s_len = reinterpret_cast<int*>(gbase + L.len);
  int* s_cost = reinterpret_cast<int*>(gbase + L.prefix);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.misc);
  int* abort_flag = reinterpret_cast<int*>(gbase + L.misc + 4);
  const int warp = threadIdx.x >> 5;
  const uint32_t bars = base + L.bars;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bars + 8 * (Bb::Full + i), 1);
      mbar_init(bars + 8 * (Bb::Empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 8 * (Bb::QFull + i), 1);
      mbar_init(bars + 8 * (Bb::QEmpty + i), 1);
      mbar_init(bars + 8 * (Bb::QReady + i), C::kSoftmaxThreads);
      mbar_init(bars + 8 * (Bb::SFull + i), 1);
      mbar_init(bars + 8 * (Bb::SEmpty + i), C::kSoftmaxThreads);
      mbar_init(bars + 8 * (Bb::PFull + i), C::kSoftmaxThreads);
      mbar_init(bars + 8 * (Bb::PEmpty + i), 1);
    }
    mbar_init(bars + 8 * (Bb::OFree + 0), C::kSoftmaxThreads);
    mbar_init(bars + 8 * (Bb::OFree + 1), C::kSoftmaxThreads);
    mbar_init(bars + 8 * Bb::Drain, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(bars + 8 * (Bb::StFull + i), 1);
      mbar_init(bars + 8 * (Bb::StEmpty + i), 1);  // released by the commit of the MMAs that read it
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 8 * (Bb::VRefFull + i), 1);
      mbar_init(bars + 8 * (Bb::VRefEmpty + i), C::kSoftmaxThreads);
    }
    for (int i = 0; i < C::kScaleSlots; ++i) {
      mbar_init(bars + 8 * (Bb::ScFull + i), kGather8 ? 32 : 1);  // block gather: one arrival per producer lane
      mbar_init(bars + 8 * (Bb::ScEmpty + i), C::kSoftmaxThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kProducerWarp && (threadIdx.x & 31) == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == C::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + L.misc),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    // the page table and Q are not written by the KV append: warm this CTA's
    // share of both in L2 while the append finishes (the first page-id and Q
    // reads are otherwise two dependent HBM round trips at start)
    prefetch_l2_share(p.page_table, (size_t)p.B * p.max_pages * sizeof(int32_t), blockIdx.x, gridDim.x);
    prefetch_l2_share(p.q, (size_t)p.B * kHeads * kHeadDim * sizeof(uint16_t), blockIdx.x, gridDim.x);
  }
  pdl_wait_prior_grid();    // the KV append (or previous step) must be complete before reading its results
  pdl_launch_dependents();  // the combine kernel may be scheduled now (its prologue reads seq_lens); it
                            // waits for this grid before it reads the partials
  build_cost_prefix(p.seq_lens, p.B, p.max_pages * kPageSize, p.err, p.piece_cost, s_len, s_cost, p.n_blocks,
                    p.max_blocks);  // ends with a barrier
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long units = s_cost[p.B];  // total cost units
  const int c = blockIdx.x;
  // token groups: CTA c works on range c / q_groups of a partition into grid / q_groups ranges
  const int qg = q_groups_of<kFp8, kMtp>(p);
  const int ranges = p.grid / qg, range = c / qg;
  const long long lo = cta_cost_lo(range, units, ranges), hi = cta_cost_lo(range + 1, units, ranges);
  Ctx cx{base, bars, abort_flag, p.err, p.wait_budget_ns};

  if (warp < 4 * C::kGroups) {
    softmax_role<kFp8, kMtp>(p, cx, s_cost, s_len, lo, hi, tmem, c, gbase);
  } else if (warp == C::kProducerWarp) {
    producer_role<kFp8, kMtp, kGather8>(p, &kmap, &vmap, &qmap, cx, s_cost, s_len, lo, hi);
  } else if (warp == C::kMmaWarp) {
    if ((threadIdx.x & 31) == 0) mma_role<kFp8, kMtp, kGather8>(p, cx, s_cost, s_len, lo, hi, tmem);
  } else if constexpr (kFp8) {
    if (warp == C::kVProducerWarp) {
      if constexpr (!kGather8) producer_v_role(p, &vmap, cx, s_cost, s_len, lo, hi);  // gather: the K producer
    }
    else if (warp == C::kVRefWarp)
      vref_role<kGather8>(p, cx, s_cost, s_len, lo, hi, reinterpret_cast<float*>(gbase + L.red) + 9 * C::kCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

template <bool kFp8, bool kMtp, bool kGather8 = false>
cudaError_t launch_tc(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      const CUtensorMap& qmap, cudaStream_t stream) {
  const size_t smem = (size_t)smem_layout<kFp8, kMtp>(p.B).total + 1024;
  static int configured[kTrackedDevices] = {};  // largest opt-in set so far, per device
  const cudaError_t e = ensure_dynamic_smem(decode_split_tc_kernel<kFp8, kMtp, kGather8>, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_split_tc_kernel<kFp8, kMtp, kGather8>, dim3(p.grid), dim3(Cfg<kFp8, kMtp>::kThreads), smem,
                    stream, p, kmap,
                    vmap, qmap);
}

}  // namespace

size_t decode_split_tc_smem_bytes(int B) { return (size_t)smem_layout<false>(B).total + 1024; }
size_t decode_split_tc_fp8_smem_bytes(int B) { return (size_t)smem_layout<true>(B).total + 1024; }
size_t decode_split_tc_mtp_smem_bytes(int B) { return (size_t)smem_layout<false, true>(B).total + 1024; }

cudaError_t launch_decode_split_tc(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   const CUtensorMap& qmap, cudaStream_t stream) {
  return launch_tc<false, false>(p, kmap, vmap, qmap, stream);
}

cudaError_t launch_decode_split_tc_fp8(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                       const CUtensorMap& qmap, cudaStream_t stream) {
  return launch_tc<true, false>(p, kmap, vmap, qmap, stream);
}

cudaError_t launch_decode_split_tc_fp8_blocks(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                              const CUtensorMap& qmap, cudaStream_t stream) {
  return launch_tc<true, false, true>(p, kmap, vmap, qmap, stream);
}

cudaError_t launch_decode_split_tc_mtp(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                       const CUtensorMap& qmap, cudaStream_t stream) {
  return launch_tc<false, true>(p, kmap, vmap, qmap, stream);
}

}  // namespace mfa
