/*
 * mfa.h -- C ABI of libmfa: decode-time Multi-matrix Factorization Attention
 * (MFA) on one NVIDIA GB300 (sm_103a).
 *
 * What MFA decode attention is ("Step-3 is Large yet Affordable: Model-system
 * Co-design for Cost-effective Decoding", paper summary page):
 *   - section 2 / Table 1: 64 query heads share ONE key head and ONE value head,
 *     both of dimension 256;
 *   - section 8.1: the attention instance runs a custom Flash-Attention kernel
 *     over its own per-sequence KV cache (each GPU serves an independent batch);
 *   - sections 5.1 and 7: with an 8-bit KV cache this reads 512 bytes per token
 *     and does 128 FLOPs per byte, so the kernel is bound by memory bandwidth.
 * For every sequence b and head h the library computes
 *     out[b,h,:] = softmax_j( scale * q[b,h,:] . K[b,j,:] ) . V[b,j,:],  j < L_b
 *     lse[b,h]   = ln sum_j exp( scale * q[b,h,:] . K[b,j,:] )
 * (natural log of the scaled logits; L_b = 0 gives out = 0, lse = -inf).
 *
 * Conventions shared by every call:
 *   - Every pointer argument is caller-owned memory. Device pointers are
 *     marked [device]. The library never allocates, frees or synchronises
 *     inside a compute call. Work is enqueued on `stream`, a cudaStream_t
 *     passed as void* (NULL = the legacy default stream). A compute call may
 *     be captured into a CUDA graph.
 *   - The call checks its arguments on the host and returns
 *     MFA_ERR_INVALID_ARG / MFA_ERR_WORKSPACE before it enqueues anything.
 *   - Faults that only the device can see set bits in an error word in the
 *     workspace header. The kernel then skips the bad access and carries on;
 *     it never traps. These faults are a page id outside [0, num_pages), a
 *     length beyond the page table's capacity, or a pipeline wait that gave
 *     up. mfa_check_device_errors() reads and optionally clears the word.
 *   - MFA_ERR_CUDA means a CUDA runtime call or a launch failed; the
 *     message is kept per host thread and mfa_last_error() returns it.
 *   - Layouts (all row-major, contiguous):
 *       q          [batch][64][256] bf16
 *       out        [batch][64][256] bf16,  lse [batch][64] fp32
 *       k_cache, v_cache [num_pages][64][256] bf16, or E4M3 bytes for _fp8
 *       k_scale, v_scale [num_pages][64] fp32 (one scale per cached token)
 *       page_table [batch][max_pages] int32: token j of sequence b is row
 *                  j % 64 of page page_table[b][j / 64]
 *       seq_lens   [batch] int32: tokens cached per sequence (device-owned
 *                  counter: the append writes at seq_lens[b] and advances it,
 *                  and attention reads it, so the token just appended is
 *                  attended -- the "DuckLLM decode fixed-cost reduction" page,
 *                  section 7.6, decode-context kernel)
 *   - Pages hold 64 tokens. q, out and the cache base pointers must be
 *     16-byte aligned.
 *   - One device: all pointers belong to the current device of the calling
 *     thread.
 */
#ifndef MFA_H_
#define MFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MFA_HEADS 64
#define MFA_HEAD_DIM 256
#define MFA_PAGE_SIZE 64
#define MFA_MAX_BATCH 1024
#define MFA_MAX_QUERY_BATCH 256  /* batch limit of mfa_query_lowrank */
#define MFA_MAX_QUERY_RANK 16384 /* rank limit of mfa_query_lowrank */
#define MFA_MAX_QUERY_TOKENS 8   /* query tokens per sequence of the multi-token decode calls */

typedef enum {
  MFA_OK = 0,
  MFA_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size (host check) */
  MFA_ERR_UNSUPPORTED = 2,      /* device is not sm_103 */
  MFA_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
  MFA_ERR_WORKSPACE = 4,        /* workspace missing or smaller than required */
  MFA_ERR_DEVICE_PAGE = 5,      /* device saw a page id outside [0, num_pages) */
  MFA_ERR_DEVICE_CAPACITY = 6,  /* device saw a length beyond max_pages * 64 */
  MFA_ERR_DEVICE_TIMEOUT = 7    /* a pipeline wait inside a kernel gave up */
} mfa_status_t;

/* Error-word bits (the first uint32 of the workspace). */
#define MFA_DEVERR_PAGE 0x1u
#define MFA_DEVERR_CAPACITY 0x2u
#define MFA_DEVERR_TIMEOUT 0x4u

/* Static description of how a decode call splits its work.
 * Host only; needs no GPU. */
typedef struct {
  int grid_ctas;            /* CTAs of the split kernel (one per SM at most) */
  int partial_slots;        /* grid_ctas + batch - 1 split results */
  size_t workspace_bytes;   /* bytes mfa_decode_attention* needs */
} mfa_plan_t;

/* Split-KV planning (host only). The split kernel lays the sequences end to
 * end on a line of cost units: a sequence with n = ceil(L_b / 64) > 0 pages
 * takes n + k units (k units charged per piece, then one per page; k is a
 * property of the kernel variant, 1 to 3), an empty one none. The C units are cut into `grid_ctas` = G contiguous, equal
 * ranges that cross sequence boundaries: CTA c owns the pages whose units lie
 * in [floor(c*C/G), floor((c+1)*C/G)) and writes one partial result per
 * sequence b it holds pages of, into slot c + b. `max_len_hint` is the expected
 * maximum length and only sizes the grid; longer sequences are still handled.
 * `num_sms` <= 0 means the current device's SM count. Returns
 * MFA_ERR_INVALID_ARG for batch outside [1, MFA_MAX_BATCH] or a negative
 * hint. */
mfa_status_t mfa_plan_decode(int batch, int max_len_hint, int num_sms, mfa_plan_t* plan);

/* Workspace size for mfa_decode_attention* on the current device; 0 on a bad
 * argument. The same workspace also serves the append calls, which use only
 * its header. */
size_t mfa_decode_workspace_bytes(int batch, int max_len_hint);

/* Zero the first `workspace_bytes` bytes of the workspace (the error word and
 * every scratch area). Call once after allocating the workspace. [device]
 * workspace. Enqueued on `stream`. */
mfa_status_t mfa_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* KV append (bf16 cache). For every sequence b, writes n_new tokens
 * k_new[b][t][:], v_new[b][t][:] (bf16 [batch][n_new][256], [device]) at
 * positions seq_lens[b] + t, then adds n_new to seq_lens[b] on the device.
 * n_new = 1 is the decode step. The writes go in place: the cache is never
 * reallocated (the static-cache lesson of the "DuckLLM decode fixed-cost
 * reduction" page, section 7.2). A sequence whose tokens would exceed
 * max_pages * 64, or that meets a bad page id, is left unchanged and sets
 * MFA_DEVERR_CAPACITY / MFA_DEVERR_PAGE. `workspace` is any workspace sized
 * by mfa_decode_workspace_bytes (only its error word is used). */
mfa_status_t mfa_kv_append(const void* k_new, const void* v_new, int n_new,
                           void* k_cache, void* v_cache,
                           const int32_t* page_table, int32_t* seq_lens,
                           int batch, int max_pages, int num_pages,
                           void* workspace, void* stream);

/* KV append into an FP8-E4M3 cache ("Step-3 is Large yet Affordable",
 * section 7: 8-bit KV, 512 bytes per token per layer). Each new bf16 row x is
 * quantised on the device with its own fp32 scale s = absmax(x) / 448
 * (s = 1 for an all-zero row); codes are E4M3(x / s), rounded to nearest even
 * and saturated to +-448 (OCP OFP8 E4M3). s goes to k_scale / v_scale
 * [num_pages][64] at the token's slot. Everything else as mfa_kv_append. */
mfa_status_t mfa_kv_append_fp8(const void* k_new, const void* v_new, int n_new,
                               void* k_cache, void* v_cache,
                               float* k_scale, float* v_scale,
                               const int32_t* page_table, int32_t* seq_lens,
                               int batch, int max_pages, int num_pages,
                               void* workspace, void* stream);

/* MFA decode attention over a bf16 paged cache (formula at the top of this
 * file). q, out, lse, caches, page_table, seq_lens: [device], layouts above.
 * `scale` multiplies the logits (1/16 = 1/sqrt(256) for Step-3).
 * `max_len_hint`: expected maximum of seq_lens; it sizes the grid only.
 * `workspace` / `workspace_bytes`: [device] scratch of at least
 * mfa_decode_workspace_bytes(batch, max_len_hint) bytes, initialised once by
 * mfa_workspace_init. It holds the error word and the per-split partial
 * results; calls that share a workspace must not overlap on the GPU.
 * Host errors: MFA_ERR_INVALID_ARG (null or misaligned pointers, batch outside
 * [1, MFA_MAX_BATCH], max_pages < 1, num_pages < 1, hint < 0),
 * MFA_ERR_WORKSPACE. Device faults (bad page id, length beyond
 * max_pages * 64, wait timeout) set the error word; the kernel then reads
 * page 0 instead of a bad page and clamps a length to the capacity, so the
 * outputs of that sequence are meaningless. */
mfa_status_t mfa_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* page_table, const int32_t* seq_lens,
                                  void* out, float* lse, float scale,
                                  int batch, int max_pages, int num_pages, int max_len_hint,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* MFA decode attention over an FP8-E4M3 paged cache with per-token fp32
 * scales (k_scale, v_scale [num_pages][64], [device], 16-byte aligned). The
 * cached value is decode(code) * scale. Queries stay bf16. Both products run
 * on the tensor cores with 8-bit operands straight from the cache: q enters
 * as the sum of two E4M3 terms under a power-of-two scale (every element down
 * to 2^-10.8 of the largest |q| of the sequence piece is held exactly, the
 * rest within 2^-18.8 of it), and P times the V scale (relative to the
 * piece's largest V scale) as the sum of two E4M3 terms (about 2^-8
 * relative). Everything else as mfa_decode_attention. */
mfa_status_t mfa_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* page_table, const int32_t* seq_lens,
                                      void* out, float* lse, float scale,
                                      int batch, int max_pages, int num_pages, int max_len_hint,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* 4-bit KV ("Step-3 is Large yet Affordable", section 5.2: KV stored in 4
 * bits, the attention computed in 8 bits), read as OCP MX FP4 (E2M1) codes
 * with one fp32 scale per token, K and V separately:
 *   k_cache, v_cache: [device] uint8 [num_pages][64][128], 32-byte aligned:
 *     the 256 codes of a row packed two per byte, element 2k in the low nibble;
 *   k_scale, v_scale: [device] fp32 [num_pages][64].
 * mfa_kv_append_fp4 quantises each new row with s = absmax / 6 (fp32 division;
 * 1 for an all-zero row) and code = the nearest E2M1 value to x / s (fp32
 * division), ties to the even mantissa, saturating to +-6, sign kept on zero.
 * mfa_decode_attention_fp4 is the attention of mfa_decode_attention over the
 * dequantised cache (decode(code) * s). Every E2M1 value is exact in E4M3:
 * both products run as 8-bit tensor-core MMAs with the 4-bit codes as one
 * operand, Q and P as in mfa_decode_attention_fp8. Arguments, workspace,
 * lengths and errors as the _fp8 calls; MFA_ERR_INVALID_ARG also for caches
 * that are not 32-byte aligned. */
mfa_status_t mfa_kv_append_fp4(const void* k_new, const void* v_new, int n_new,
                               void* k_cache, void* v_cache,
                               float* k_scale, float* v_scale,
                               const int32_t* page_table, int32_t* seq_lens,
                               int batch, int max_pages, int num_pages,
                               void* workspace, void* stream);
mfa_status_t mfa_decode_attention_fp4(const void* q, const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* page_table, const int32_t* seq_lens,
                                      void* out, float* lse, float scale,
                                      int batch, int max_pages, int num_pages, int max_len_hint,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* MFA's low-rank query path ("Step-3 is Large yet Affordable", section 2 /
 * Table 1: the query is projected down from the model width to a low rank,
 * normalised, and projected up to 64 heads x 256; Step-3: 7168 -> 2048 ->
 * 64 x 256). Computes, for every row b,
 *     y = x[b] W_down                         (fp32 accumulation)
 *     h = bf16( y / sqrt(mean(y^2) + eps) * gamma )    (RMSNorm with gain)
 *     q[b] = bf16( h W_up )
 *   x:      [device] bf16 [batch][d_model], 16-byte aligned
 *   w_down: [device] bf16 [d_model][rank]; w_up: [device] bf16 [rank][n_out]
 *   gamma:  [device] bf16 [rank]
 *   q:      [device] bf16 [batch][n_out] (n_out = 64 * 256 = 16384 gives the
 *           [batch][64][256] query of mfa_decode_attention)
 * Both products run on the tensor cores and stream each weight once, so the
 * call is bound by memory bandwidth (96 MB of weights at the Step-3 shape).
 * The call is two kernel launches chained by programmatic dependent launch:
 * the up-projection streams W_up while the down-projection runs.
 * workspace: [device] at least mfa_query_lowrank_workspace_bytes(batch, rank,
 * n_out) bytes (a workspace sized for `batch` rows serves every call with as
 * many rows or fewer), 256-byte aligned, zeroed once by mfa_workspace_init:
 * the call needs its fp32 accumulator and arrival counters zero on entry and
 * leaves them zero (also after a device error). Calls sharing a workspace run
 * one after another on one stream.
 * Host errors: MFA_ERR_INVALID_ARG for null or misaligned pointers, batch
 * outside [1, MFA_MAX_QUERY_BATCH], d_model not a multiple of 64, rank or
 * n_out not a multiple of 128, rank above MFA_MAX_QUERY_RANK, eps < 0;
 * MFA_ERR_WORKSPACE. */
size_t mfa_query_lowrank_workspace_bytes(int batch, int rank, int n_out);
mfa_status_t mfa_query_lowrank(const void* x, const void* w_down, const void* gamma, const void* w_up, void* q,
                               int batch, int d_model, int rank, int n_out, float eps,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Multi-token (MTP) decode over a paged cache ("Step-3 is Large yet
 * Affordable", section 5.2: with multi-token prediction a decode step carries
 * extra predicted tokens that read the same KV cache, which raises the
 * attention's arithmetic intensity). Each sequence has n_query (1 to
 * MFA_MAX_QUERY_TOKENS) query tokens, its last n_query positions: the cache of
 * seq_lens[b] tokens already holds them (mfa_kv_append with n_new = n_query).
 * Query token t attends, causally, to positions j < seq_lens[b] - n_query + 1
 * + t; a token that sees no position gets out = 0 and lse = -inf.
 *   q:   [device] bf16 [batch][n_query][64][256], 16-byte aligned
 *   out: [device] bf16 [batch][n_query][64][256]; lse: fp32 [batch][n_query][64]
 * How the cache is read once for all tokens: on the bf16 cache a CTA serves two
 * tokens (their 64 heads each form one 128-column product with a tile of keys,
 * and of values); the quantised calls serve one token a CTA. With more tokens
 * than one CTA serves, the tokens form groups, and the grid holds one CTA per
 * group for every range of the work partition: the CTAs of a range stream the
 * same pages at the same time, so the cache is read from HBM about once and
 * shared through L2. mfa_decode_attention_mtp_fp8 / _fp4 take the E4M3 / E2M1
 * caches and scales of mfa_decode_attention_fp8 / _fp4.
 * workspace: at least mfa_decode_mtp_workspace_bytes(batch, n_query,
 * max_len_hint) bytes (0 for a bad argument; it covers all three cache
 * formats). Host errors: MFA_ERR_INVALID_ARG also for n_query outside
 * [1, MFA_MAX_QUERY_TOKENS]. Everything else as mfa_decode_attention. */
size_t mfa_decode_mtp_workspace_bytes(int batch, int n_query, int max_len_hint);
mfa_status_t mfa_decode_attention_mtp(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* page_table, const int32_t* seq_lens,
                                      void* out, float* lse, float scale,
                                      int batch, int n_query, int max_pages, int num_pages, int max_len_hint,
                                      void* workspace, size_t workspace_bytes, void* stream);
mfa_status_t mfa_decode_attention_mtp_fp8(const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* page_table, const int32_t* seq_lens,
                                          void* out, float* lse, float scale,
                                          int batch, int n_query, int max_pages, int num_pages, int max_len_hint,
                                          void* workspace, size_t workspace_bytes, void* stream);
mfa_status_t mfa_decode_attention_mtp_fp4(const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* page_table, const int32_t* seq_lens,
                                          void* out, float* lse, float scale,
                                          int batch, int n_query, int max_pages, int num_pages, int max_len_hint,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* Decode attention over caller-selected 8-token blocks of a bf16 paged cache
 * ("Step-5-Preview" page, sparse attention section: the query attends to the
 * original K/V rows of the selected historical blocks and of its own block
 * up to itself, with the softmax over that set; the selection -- the page's
 * indexer and top-k -- is the caller's). For sequence b of length L > 0,
 * block r covers positions 8r .. 8r + 7 and c = floor((L - 1) / 8) is the
 * block of the last token; the query attends to
 *     the blocks block_idx[b][0 .. n_blocks[b])   (each in [0, c), distinct)
 *     and positions 8c .. L - 1,
 * i.e. to J_b = {8r + i} U {8c, .., L - 1}, out = softmax(q K_J^T * scale) V_J
 * and lse as in mfa_decode_attention (L = 0: out = 0, lse = -inf).
 *   block_idx: [device] int32 [batch][max_blocks]; entries past n_blocks[b]
 *              are not read. The order is free; a block listed twice is
 *              attended twice (the caller passes a set).
 *   n_blocks:  [device] int32 [batch], in [0, min(c, max_blocks)]
 *   max_len_hint: expected maximum of 8 * n_blocks[b] + 8 (the attended
 *              tokens); it sizes the grid and the workspace
 *              (mfa_decode_workspace_bytes(batch, max_len_hint)).
 * q, caches, page_table, seq_lens, out, lse as in mfa_decode_attention.
 * Device errors: MFA_DEVERR_PAGE also for a block id outside [0, c) (read as
 * block 0), MFA_DEVERR_CAPACITY for n_blocks[b] outside its range (clamped).
 * Host errors: MFA_ERR_INVALID_ARG also for null or misaligned block lists,
 * max_blocks < 1 or above 8 * max_pages. */
mfa_status_t mfa_decode_attention_blocks(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* page_table, const int32_t* seq_lens,
                                         const int32_t* block_idx, const int32_t* n_blocks, int max_blocks,
                                         void* out, float* lse, float scale,
                                         int batch, int max_pages, int num_pages, int max_len_hint,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* Block gather over an FP8-E4M3 paged cache with per-token fp32 scales: the
 * attention of mfa_decode_attention_blocks over the dequantised cache of
 * mfa_decode_attention_fp8 (k_scale, v_scale [num_pages][64], [device],
 * 16-byte aligned). Each selected block moves as its 8 rows of codes and their
 * 8 K and 8 V scales; Q and P enter the 8-bit products as in
 * mfa_decode_attention_fp8. Arguments, errors and the workspace as
 * mfa_decode_attention_blocks. */
mfa_status_t mfa_decode_attention_blocks_fp8(const void* q, const void* k_cache, const void* v_cache,
                                             const float* k_scale, const float* v_scale,
                                             const int32_t* page_table, const int32_t* seq_lens,
                                             const int32_t* block_idx, const int32_t* n_blocks, int max_blocks,
                                             void* out, float* lse, float scale,
                                             int batch, int max_pages, int num_pages, int max_len_hint,
                                             void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free variant of mfa_decode_attention (bf16 cache). The paper
 * has no counterpart: it exists for callers that cannot give the library a
 * workspace -- a plugin or foreign-function host that passes only tensors it
 * already owns and no allocator, or a running serving loop that must not call
 * cudaMalloc (which can synchronise the whole device).
 * Inputs, outputs and their layouts are those of mfa_decode_attention. The
 * split scratch is a fixed 24 MiB device array inside the library, present on
 * every GPU that loads it until the process exits. The call itself allocates
 * nothing.
 *   - The first call on a device looks up the array's device address, with
 *     that device current. Make this first call before any stream capture.
 *   - Batches whose split results need more than 24 MiB
 *     (mfa_plan_decode().workspace_bytes > 24 MiB) return MFA_ERR_WORKSPACE
 *     with a message.
 *   - All calls share the one array, so calls that may overlap on the GPU
 *     (other streams or host threads) race and must be serialised by the
 *     caller.
 * device_error_word: optional [device] uint32 that receives the MFA_DEVERR_*
 * bits of device faults (it is not cleared by the call). With NULL, faults go
 * to a word in the shared array, which each call clears, and are not
 * reported. */
mfa_status_t mfa_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* page_table, const int32_t* seq_lens,
                                          void* out, float* lse, float scale,
                                          int batch, int max_pages, int num_pages, int max_len_hint,
                                          uint32_t* device_error_word, void* stream);

/* Synchronise `stream`, read the workspace error word and return the first
 * device fault it records (MFA_ERR_DEVICE_PAGE, _CAPACITY, _TIMEOUT) or MFA_OK.
 * `clear` != 0 resets the word afterwards. This call blocks the host. */
mfa_status_t mfa_check_device_errors(void* workspace, int clear, void* stream);

/* Budget, in nanoseconds, after which a pipeline wait inside a kernel gives up
 * and sets MFA_DEVERR_TIMEOUT (default 2e9 = 2 s). Applies to launches made
 * after the call, from any thread. */
void mfa_set_wait_budget_ns(uint64_t budget_ns);

/* Self-test of the bounded wait: launches one CTA that waits on an mbarrier
 * nothing arrives on, with the given budget; the wait must give up, set
 * MFA_DEVERR_TIMEOUT in the workspace error word and return. */
mfa_status_t mfa_selftest_wait_timeout(void* workspace, uint64_t budget_ns, void* stream);

/* Timing hook for benchmarks. With both handles non-NULL (cudaEvent_t created
 * with timing enabled), every later decode call on this host thread records
 * start_event on its stream just before the split kernel and stop_event just
 * after it, so cudaEventElapsedTime gives that kernel's device time. Under
 * stream capture the records become external event nodes of the graph.
 * (NULL, NULL) turns the hook off. */
void mfa_profile_split_events(void* start_event, void* stop_event);

/* Human-readable name of a status code (static string). */
const char* mfa_status_string(mfa_status_t status);

/* Message of the last failure seen by a call on this host thread ("" if none);
 * valid until the next call on the same thread. */
const char* mfa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MFA_H_ */
