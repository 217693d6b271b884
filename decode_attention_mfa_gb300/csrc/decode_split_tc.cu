// decode_split_tc.cu -- split-KV MFA decode for a bf16 paged cache on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators) with TMA streaming.
//
// MFA ("Step-3 is Large yet Affordable", paper summary page, section 2 /
// Table 1) gives all 64 query heads one shared K head and one shared V head
// (d = 256), so for one sequence the logits of every head against a tile of
// keys form one dense contraction. The kernel computes, per 128-token tile
// (two 64-token pages), the transposed products
//     S^T[tok, head] = K_tile[tok, :] . Q[head, :]^T       (M=128, N=64, K=256)
//     O^T[dim, head] += V_tile[:, dim]^T . P^T[tok, head]  (2 x M=128, N=64, K=128)
// so every MMA uses the full 128-lane data path (an M=64 MMA costs as much as
// an M=128 one on sm_103a), and softmax statistics are reduced across the 128
// TMEM lanes.
//
// Work split: the same stream-K page partition as the CUDA-core path (CTA c
// owns pages [c*P/G, (c+1)*P/G) of the concatenated sequences and writes one
// normalised partial result plus its natural-log LSE per sequence piece into
// slot c + b); the LSE combine kernel merges the pieces.
//
// Warp roles (192 threads, one CTA per SM):
//   warps 0-3  softmax: TMEM lane = token of the tile; online softmax in fp32
//              with a lazily updated reference maximum (only when a logit
//              exceeds it by 2^8 are P, the row sums and O^T rescaled); then
//              the epilogue (row-sum reduction, O^T / l, partial LSE).
//   warp 4     producer: page-table walk, TMA loads of Q and of K/V chunks
//              (16 KB: a 64-dim slice of a 2-page K tile, or a 128-dim slice
//              of one V page) into a ring of shared-memory slots.
//   warp 5     MMA issue (lane 0), TMEM allocation, zeroing of the unused
//              rows of a partial last V page (0 * NaN would poison P.V).
// Every mbarrier wait is bounded (wait budget); on expiry the kernel records
// MFA_DEVERR_TIMEOUT, the roles stop issuing work and the CTA drains and exits.
#include "mfa_device.cuh"

namespace mfa {
namespace {

constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kSlots = 7;                 // 16 KB ring slots
constexpr int kSlotBytes = 16384;
constexpr int kQBytes = 32768;            // Q: 4 dim blocks of [64 heads x 128 B]; two buffers
constexpr int kPBytes = 16384;            // P^T: [128 tokens x 64 heads] bf16
constexpr int kTmemCols = 256;            // S^T x2 (64 cols each) + O^T (2 x 64 cols)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f; // log2 units: P stays below 2^8

// idesc: bf16 x bf16 -> fp32, M = 128, N = 64.
constexpr uint32_t kIdescS = idesc_f16(128, 64, 1, 0, 0);  // A = K tile (K-major), B = Q (K-major)
constexpr uint32_t kIdescO = idesc_f16(128, 64, 1, 1, 1);  // A = V^T (dim-major), B = P^T (head-major)

struct SmemLayout {
  uint32_t ring, q, p;  // byte offsets from the 1024-aligned base
  uint32_t len, prefix, red, flags, bars, misc;
  uint32_t total;
};

__host__ __device__ inline SmemLayout smem_layout(int B) {
  SmemLayout L;
  L.ring = 0;
  L.q = L.ring + kSlots * kSlotBytes;
  L.p = L.q + 2 * kQBytes;
  L.len = L.p + 2 * kPBytes;
  L.prefix = L.len + 4 * B;
  L.red = (L.prefix + 4 * (B + 1) + 15) & ~15u;  // float red[4][64], mref[64], alpha[64]
  L.flags = L.red + 6 * 64 * 4;                   // int flags[2][4]
  L.bars = (L.flags + 32 + 7) & ~7u;              // mbarriers
  L.misc = L.bars + 8 * 48;                       // tmem base, abort flag
  L.total = L.misc + 16;
  return L;
}

// Barrier indices inside the barrier array.
enum : int {
  kBarFull = 0,                 // [kSlots]
  kBarEmpty = kBarFull + kSlots,  // [kSlots]
  kBarQFull = kBarEmpty + kSlots,  // [2]
  kBarQEmpty = kBarQFull + 2,       // [2]
  kBarSFull = kBarQEmpty + 2,       // [2]
  kBarSEmpty = kBarSFull + 2,   // [2]
  kBarPFull = kBarSEmpty + 2,   // [2]
  kBarPEmpty = kBarPFull + 2,   // [2]
  kBarOReady = kBarPEmpty + 2,
  kBarOFree,
  kBarDrain,
  kNumBars
};
static_assert(kNumBars <= 48, "barrier array too small");

struct Ctx {
  uint32_t base;      // shared address of the aligned dynamic smem base
  uint32_t bar0;      // shared address of barrier 0
  volatile int* abort;
  uint32_t* err;
  uint64_t budget;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  __device__ bool wait(int i, uint32_t parity) const { return mbar_wait(bar(i), parity, budget, abort, err); }
};

__device__ __forceinline__ void named_barrier_softmax() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
}

// Segment iteration shared by all roles: sequence b, pages [pg0, pg1) of it.
struct Seg {
  int b, pg0, pg1, len;
};
__device__ __forceinline__ bool seg_first(const int* s_prefix, const int* s_len, int B, long long lo, long long hi,
                                          Seg& s) {
  if (lo >= hi) return false;
  s.b = seq_of_page(s_prefix, B, lo) - 1;
  return true;
}
__device__ __forceinline__ bool seg_next(const int* s_prefix, const int* s_len, int B, long long lo, long long hi,
                                         Seg& s) {
  for (int b = s.b + 1; b < B && s_prefix[b] < hi; ++b) {
    const long long sp0 = s_prefix[b], sp1 = s_prefix[b + 1];
    if (sp1 == sp0) continue;
    s.b = b;
    s.pg0 = (int)((sp0 > lo ? sp0 : lo) - sp0);
    s.pg1 = (int)((sp1 < hi ? sp1 : hi) - sp0);
    s.len = s_len[b];
    return true;
  }
  return false;
}

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

// The whole producer warp runs this loop (uniform control flow); lane 0
// issues the copies.
__device__ void producer_role(const DecodeParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                              const CUtensorMap* qmap, const Ctx& cx, const int* s_prefix, const int* s_len,
                              long long lo, long long hi) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol_stream = policy_evict_first();
  const uint64_t pol_keep = policy_evict_last();
  const uint32_t q_base = cx.base + smem_layout(p.B).q;
  uint32_t cc = 0, seg_i = 0;
  Seg s;
  bool ok = seg_first(s_prefix, s_len, p.B, lo, hi, s);
  auto wait_slot = [&](uint32_t& dst, uint32_t& bar) -> bool {
    const uint32_t slot = cc % kSlots, n = cc / kSlots;
    const bool r = cx.wait(kBarEmpty + slot, (n & 1) ^ 1);
    __syncwarp();
    dst = cx.base + slot * kSlotBytes;
    bar = cx.bar(kBarFull + slot);
    return r;
  };
  // K dim block d of a tile of pages pa (and pb >= 0)
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
  // V dims [hf*128, hf*128 + 128) of page pv
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
  uint32_t last_q_parity = 0, last_qb = 0;
  bool issued_q = false;
  while (ok && seg_next(s_prefix, s_len, p.B, lo, hi, s)) {
    if (*cx.abort) break;
    PageIds ids;
    ids.row = p.page_table + (size_t)s.b * p.max_pages;
    ids.pg1 = s.pg1;
    ids.start(s.pg0, p, lane);
    // Q of this sequence into buffer seg_i % 2 (free once every S MMA of the
    // piece before the previous one is done, so the loads of this piece need
    // not wait for the previous piece to finish)
    const uint32_t qb = seg_i & 1;
    const bool qfree = cx.wait(kBarQEmpty + qb, ((seg_i >> 1) & 1) ^ 1);
    __syncwarp();
    if (!qfree) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(cx.bar(kBarQFull + qb), (uint32_t)kQBytes);
      for (int d = 0; d < 4; ++d)
        tma_load_2d(q_base + qb * kQBytes + d * 8192, qmap, d * 64, s.b * kHeads, cx.bar(kBarQFull + qb), pol_keep);
    }
    issued_q = true;
    last_q_parity = (seg_i >> 1) & 1;
    last_qb = qb;
    ++seg_i;
    const int T = (s.pg1 - s.pg0 + 1) / 2;
    bool good = true;
    // chunk order: K(0), then K(t), V(t-1) for t = 1..T-1, then V(T-1)
    for (int t = 0; good && t <= T; ++t) {
      if (t < T) {
        const int pga = s.pg0 + 2 * t;
        const int pa = ids.get(pga, p, lane);
        const int pb = (pga + 1 < s.pg1) ? ids.get(pga + 1, p, lane) : -1;
        for (int d = 0; good && d < 4; ++d) good = issue_k(d, pa, pb);
      }
      if (good && t > 0) {
        const int pgv = s.pg0 + 2 * (t - 1);
        const int np = (pgv + 1 < s.pg1) ? 2 : 1;
        for (int i = 0; good && i < np; ++i) {
          const int pv = ids.get(pgv + i, p, lane);
          good = issue_v(0, pv) && issue_v(1, pv);
        }
      }
    }
    if (!good) break;
  }
  // drain: every copy this warp issued must land before the CTA exits
  if (lane == 0) {
    for (uint32_t k = (cc > (uint32_t)kSlots ? cc - kSlots : 0); k < cc; ++k)
      (void)mbar_wait(cx.bar(kBarFull + k % kSlots), (k / kSlots) & 1, cx.budget, nullptr, p.err);
    if (issued_q) (void)mbar_wait(cx.bar(kBarQFull + last_qb), last_q_parity, cx.budget, nullptr, p.err);
  }
  __syncwarp();
}

// ---------------------------------------------------------------- MMA issue
__device__ void mma_role(const DecodeParams& p, const Ctx& cx, const int* s_prefix, const int* s_len, long long lo,
                         long long hi, uint32_t tmem) {
  const int lane = threadIdx.x & 31;
  const SmemLayout L = smem_layout(p.B);
  uint32_t cc = 0, seg_i = 0, s_cnt = 0, p_cnt = 0;
  Seg s;
  bool ok = seg_first(s_prefix, s_len, p.B, lo, hi, s);
  bool alive = true;

  auto wait_all = [&](int bar, uint32_t parity) -> bool {
    const bool r = cx.wait(bar, parity);  // every lane polls the same barrier
    __syncwarp();
    return r;
  };
  auto do_s = [&](int t_in_seg, uint32_t qb) -> bool {
    const uint32_t buf = s_cnt & 1, n = s_cnt >> 1;
    if (!wait_all(kBarSEmpty + buf, (n & 1) ^ 1)) return false;
    const uint32_t d_tmem = tmem + buf * 64;
    for (int d = 0; d < 4; ++d) {
      const uint32_t slot = cc % kSlots, ph = (cc / kSlots) & 1;
      if (!wait_all(kBarFull + slot, ph)) return false;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t a0 = cx.base + slot * kSlotBytes;
        const uint32_t b0 = cx.base + L.q + qb * kQBytes + d * 8192;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(d_tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), smem_desc_sw128(b0 + kk * 32, 16, 1024), kIdescS,
                 (d | kk) != 0);
        tc_commit(cx.bar(kBarEmpty + slot));
      }
      __syncwarp();
      ++cc;
    }
    if (lane == 0) tc_commit(cx.bar(kBarSFull + buf));
    __syncwarp();
    ++s_cnt;
    (void)t_in_seg;
    return true;
  };
  auto do_pv = [&](const Seg& sg, int t, bool first_of_seg) -> bool {
    const uint32_t buf = p_cnt & 1, n = p_cnt >> 1;
    if (first_of_seg && !wait_all(kBarOFree, (seg_i & 1) ^ 1)) return false;
    if (!wait_all(kBarPFull + buf, n & 1)) return false;
    const int pga = sg.pg0 + 2 * t;
    const int np = (pga + 1 < sg.pg1) ? 2 : 1;
    for (int i = 0; i < np; ++i) {
      const int nv = min(kPageSize, sg.len - (pga + i) * kPageSize);  // valid rows of this page
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t slot = cc % kSlots, ph = (cc / kSlots) & 1;
        if (!wait_all(kBarFull + slot, ph)) return false;
        const uint32_t a0 = cx.base + slot * kSlotBytes;
        if (nv < kPageSize) {
          // rows [nv, 64) of both 64-dim blocks: 128 B each, 16 B per lane and step
          const int nbytes = (kPageSize - nv) * 128;
          for (int off = lane * 16; off < 2 * nbytes; off += 32 * 16) {
            const int blk = off / nbytes, r = off % nbytes;
            const uint32_t addr = a0 + blk * 8192 + nv * 128 + r;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t bp = cx.base + L.p + buf * kPBytes + i * 8192;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(tmem + 128 + hf * 64, smem_desc_sw128(a0 + kk * 2048, 8192, 1024),
                   smem_desc_sw128(bp + kk * 2048, 8192, 1024), kIdescO, !(first_of_seg && i == 0 && kk == 0));
          tc_commit(cx.bar(kBarEmpty + slot));
        }
        __syncwarp();
        ++cc;
      }
    }
    if (lane == 0) {
      tc_commit(cx.bar(kBarPEmpty + buf));
      tc_commit(cx.bar(kBarOReady));
    }
    __syncwarp();
    ++p_cnt;
    return true;
  };

  while (alive && ok && seg_next(s_prefix, s_len, p.B, lo, hi, s)) {
    const uint32_t qb = seg_i & 1;
    if (!wait_all(kBarQFull + qb, (seg_i >> 1) & 1)) break;
    const int T = (s.pg1 - s.pg0 + 1) / 2;
    alive = do_s(0, qb);
    if (alive && T == 1 && lane == 0) tc_commit(cx.bar(kBarQEmpty + qb));
    for (int t = 1; alive && t < T; ++t) {
      alive = do_s(t, qb);
      if (alive && t == T - 1 && lane == 0) tc_commit(cx.bar(kBarQEmpty + qb));
      __syncwarp();
      if (alive) alive = do_pv(s, t - 1, t == 1);
    }
    if (alive) alive = do_pv(s, T - 1, T == 1);
    ++seg_i;
  }
  // drain: wait for every MMA this thread issued before TMEM is released
  if (lane == 0) {
    tc_commit(cx.bar(kBarDrain));
    (void)mbar_wait(cx.bar(kBarDrain), 0, cx.budget, nullptr, p.err);
  }
  __syncwarp();
}

// ---------------------------------------------------------------- softmax
// Per-thread: row t of S^T (token t of the tile), 64 head columns.
__device__ __forceinline__ void warp_reduce_scatter_max(float (&v)[64], int lane) {
  // after the 5 steps lane l holds the maxima of columns 2l and 2l+1 over the warp
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 32 >> step;
    const int o = 16 >> step;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[i + half] : v[i];
      const float send = up ? v[i] : v[i + half];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
}
__device__ __forceinline__ void warp_reduce_scatter_sum(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 32 >> step;
    const int o = 16 >> step;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[i + half] : v[i];
      const float send = up ? v[i] : v[i + half];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

__device__ __forceinline__ void load_logits(uint32_t taddr, bool valid, float c2, float (&x)[64]) {
  tmem_ld32(taddr, x);
  tmem_ld32(taddr + 32, x + 32);
  tc_wait_ld();
#pragma unroll
  for (int h = 0; h < 64; ++h) x[h] = valid ? x[h] * c2 : -INFINITY;
}

// O^T columns (this thread's TMEM lane, both 128-dim halves) times col_scale[h].
__device__ __forceinline__ void scale_o_columns(uint32_t taddr_o, const float* col_scale) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float o[32];
      tmem_ld32(taddr_o + hf * 64 + q * 32, o);
      tc_wait_ld();
#pragma unroll
      for (int h = 0; h < 32; ++h) o[h] *= col_scale[q * 32 + h];
      tmem_st32(taddr_o + hf * 64 + q * 32, o);
    }
  }
  tc_wait_st();
}

__device__ void softmax_role(const DecodeParams& p, const Ctx& cx, const int* s_prefix, const int* s_len,
                             long long lo, long long hi, uint32_t tmem, int c, uint8_t* gbase) {
  const int tid = threadIdx.x;  // 0..127: TMEM lane = token of the tile = dim of each O^T half
  const int warp = tid >> 5, lane = tid & 31;
  const SmemLayout L = smem_layout(p.B);
  float* red = reinterpret_cast<float*>(gbase + L.red);  // [4][64] per-warp partial reductions
  float* mref = red + 4 * 64;                            // [64] reference maxima (log2 units), uniform
  float* alpha = mref + 64;                              // [64] rescale factors / 1/l, uniform
  int* flags = reinterpret_cast<int*>(gbase + L.flags);  // [2][4]
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  const uint32_t taddr_o = tmem + lane_base + 128;
  const float c2 = p.scale * kLog2e;
  uint32_t s_cnt = 0, p_cnt = 0, tile_i = 0;
  // o_ready completes once per P.V; a parity wait only tells the current phase
  // from the previous one, so its completions are observed one by one, in
  // order. Waiting for P.V(g-1) before handing over P(g) keeps the barrier at
  // most one phase ahead of this count.
  uint32_t o_seen = 0;
  auto observe_pv = [&](uint32_t k) -> bool {
    while (o_seen <= k) {
      if (!cx.wait(kBarOReady, o_seen & 1)) return false;
      ++o_seen;
    }
    return true;
  };
  Seg s;
  bool ok = seg_first(s_prefix, s_len, p.B, lo, hi, s);

  while (ok && seg_next(s_prefix, s_len, p.B, lo, hi, s)) {
    if (tid < 64) mref[tid] = -INFINITY;
    named_barrier_softmax();
    float lp[64];  // this thread's share of the softmax denominators
#pragma unroll
    for (int h = 0; h < 64; ++h) lp[h] = 0.0f;
    const int T = (s.pg1 - s.pg0 + 1) / 2;
    for (int t = 0; t < T; ++t) {
      const int tok0 = (s.pg0 + 2 * t) * kPageSize;
      const int np = (s.pg0 + 2 * t + 1 < s.pg1) ? 2 : 1;
      const bool valid = tid < min(np * kPageSize, s.len - tok0);
      const uint32_t sbuf = s_cnt & 1;
      const uint32_t taddr_s = tmem + lane_base + sbuf * 64;
      if (!cx.wait(kBarSFull + sbuf, (s_cnt >> 1) & 1)) return;
      tc_fence_after();
      float x[64];
      load_logits(taddr_s, valid, c2, x);
      bool mine = false;
#pragma unroll
      for (int h = 0; h < 64; ++h) mine |= x[h] > mref[h] + kRescaleThreshold;
      // ---- does any logit of the tile exceed its reference maximum by 2^8?
      const int fl = tile_i & 1;
      const bool wany = __any_sync(0xffffffffu, mine);
      if (lane == 0) flags[fl * 4 + warp] = wany ? 1 : 0;
      named_barrier_softmax();
      if (flags[fl * 4 + 0] | flags[fl * 4 + 1] | flags[fl * 4 + 2] | flags[fl * 4 + 3]) {
        warp_reduce_scatter_max(x, lane);  // x is reloaded below
        red[warp * 64 + 2 * lane] = x[0];
        red[warp * 64 + 2 * lane + 1] = x[1];
        named_barrier_softmax();
        if (tid < 64) {
          const float m_old = mref[tid];
          const float m_new = fmaxf(m_old, fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid])));
          alpha[tid] = (m_old == -INFINITY) ? 0.0f : exp2f(m_old - m_new);
          mref[tid] = m_new;
        }
        named_barrier_softmax();
        bool rescale_o = false;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          lp[h] *= alpha[h];
          rescale_o |= alpha[h] != 1.0f;
        }
        if (t > 0 && rescale_o) {
          // O^T holds the previous tiles: wait for their last P.V, then scale its columns
          if (!observe_pv(p_cnt - 1)) return;
          tc_fence_after();
          scale_o_columns(taddr_o, alpha);
        }
        load_logits(taddr_s, valid, c2, x);
      }
      tc_fence_before();
      mbar_arrive(cx.bar(kBarSEmpty + sbuf));  // S^T buffer free for the tile after next
      ++s_cnt;
      // ---- P = exp2(x - mref): row sums in fp32, P^T row in bf16
      uint32_t packed[32];
#pragma unroll
      for (int h = 0; h < 64; h += 2) {
        const float p0 = exp2f(x[h] - mref[h]);
        const float p1 = exp2f(x[h + 1] - mref[h + 1]);
        lp[h] += p0;
        lp[h + 1] += p1;
        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
        packed[h >> 1] = *reinterpret_cast<uint32_t*>(&b2);
      }
      const uint32_t pbuf = p_cnt & 1;
      if (p_cnt > 0 && !observe_pv(p_cnt - 1)) return;
      if (!cx.wait(kBarPEmpty + pbuf, ((p_cnt >> 1) & 1) ^ 1)) return;
      const uint32_t prow = cx.base + L.p + pbuf * kPBytes + tid * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t addr = prow + ((j ^ (tid & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[4 * j]),
                     "r"(packed[4 * j + 1]), "r"(packed[4 * j + 2]), "r"(packed[4 * j + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(cx.bar(kBarPFull + pbuf));
      ++p_cnt;
      ++tile_i;
    }
    // ---- epilogue of this sequence piece: l = sum over the 128 lanes, O^T / l, LSE
    if (!observe_pv(p_cnt - 1)) return;
    tc_fence_after();
    warp_reduce_scatter_sum(lp, lane);
    named_barrier_softmax();  // earlier readers of red/alpha are done
    red[warp * 64 + 2 * lane] = lp[0];
    red[warp * 64 + 2 * lane + 1] = lp[1];
    named_barrier_softmax();
    const size_t slot = (size_t)c + s.b;
    if (tid < 64) {
      const float l = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
      alpha[tid] = 1.0f / l;
      p.part_lse[slot * kHeads + tid] = (mref[tid] + log2f(l)) * kLn2;
    }
    named_barrier_softmax();
    float* dst = p.part_o + slot * kHeads * kHeadDim;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float o[32];
        tmem_ld32(taddr_o + hf * 64 + q * 32, o);
        tc_wait_ld();
        const int dim = hf * 128 + tid;
#pragma unroll
        for (int h = 0; h < 32; ++h) dst[(q * 32 + h) * kHeadDim + dim] = o[h] * alpha[q * 32 + h];
      }
    }
    tc_fence_before();
    mbar_arrive(cx.bar(kBarOFree));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_split_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  const uint32_t raw = smem_u32(dyn_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = dyn_smem + (base - raw);
  const SmemLayout L = smem_layout(p.B);
  int* s_len = reinterpret_cast<int*>(gbase + L.len);
  int* s_prefix = reinterpret_cast<int*>(gbase + L.prefix);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.misc);
  int* abort_flag = reinterpret_cast<int*>(gbase + L.misc + 4);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(base + L.bars + 8 * (kBarFull + i), 1);
      mbar_init(base + L.bars + 8 * (kBarEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(base + L.bars + 8 * (kBarQFull + i), 1);
      mbar_init(base + L.bars + 8 * (kBarQEmpty + i), 1);
      mbar_init(base + L.bars + 8 * (kBarSFull + i), 1);
      mbar_init(base + L.bars + 8 * (kBarSEmpty + i), kSoftmaxThreads);
      mbar_init(base + L.bars + 8 * (kBarPFull + i), kSoftmaxThreads);
      mbar_init(base + L.bars + 8 * (kBarPEmpty + i), 1);
    }
    mbar_init(base + L.bars + 8 * kBarOReady, 1);
    mbar_init(base + L.bars + 8 * kBarOFree, kSoftmaxThreads);
    mbar_init(base + L.bars + 8 * kBarDrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && (threadIdx.x & 31) == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + L.misc),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  pdl_wait_prior_grid();    // the KV append (or previous step) must be complete before reading its results
  pdl_launch_dependents();  // the combine kernel may be scheduled now (its prologue reads seq_lens); it
                            // waits for this grid before it reads the partials
  build_page_prefix(p.seq_lens, p.B, p.max_pages * kPageSize, p.err, s_len, s_prefix);  // ends with a barrier
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long P = s_prefix[p.B];
  const int c = blockIdx.x;
  const long long lo = cta_page_lo(c, P, p.grid), hi = cta_page_lo(c + 1, P, p.grid);
  Ctx cx{base, base + L.bars, abort_flag, p.err, p.wait_budget_ns};

  if (warp < 4) {
    softmax_role(p, cx, s_prefix, s_len, lo, hi, tmem, c, gbase);
  } else if (warp == kProducerWarp) {
    producer_role(p, &kmap, &vmap, &qmap, cx, s_prefix, s_len, lo, hi);
  } else {
    mma_role(p, cx, s_prefix, s_len, lo, hi, tmem);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

}  // namespace

size_t decode_split_tc_smem_bytes(int B) { return (size_t)smem_layout(B).total + 1024; }

cudaError_t launch_decode_split_tc(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   const CUtensorMap& qmap, cudaStream_t stream) {
  const size_t smem = decode_split_tc_smem_bytes(p.B);
  static int configured_bytes = 0;  // largest opt-in set so far (per process; one device family)
  if ((int)smem > configured_bytes) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_bytes = (int)smem;
  }
  return launch_pdl(decode_split_tc_kernel, dim3(p.grid), dim3(kThreads), smem, stream, p, kmap, vmap, qmap);
}

}  // namespace mfa
