"""Seeded synthetic inputs for MFA decode attention.

This module holds no attention arithmetic.  It draws the inputs (queries, key
and value rows, sequence lengths, page permutations) that both the CUDA path
and the CPU oracle consume, and lays token rows out in the paged cache
format.  Nothing here quantises, scales or attends.

Shapes follow the MFA head layout of "Step-3 is Large yet Affordable" (paper
summary page), section 2 / Table 1: 64 query heads sharing one K head and one
V head, head dimension 256.  Values are N(0, 1) drawn in fp32 and rounded to
bf16 (round to nearest even).  Lengths "uniform in [a, b]" are integers drawn
uniformly with both ends included.  Pages hold 64 tokens; a permuted cache
assigns a seeded random permutation of all pages to the sequences in order.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np
import torch

HEADS = 64
HEAD_DIM = 256
PAGE_SIZE = 64
SCALE = 1.0 / 16.0  # 1 / sqrt(256)

_CHUNK_TOKENS = 32768  # rows drawn per independent generator stream


@dataclass(frozen=True)
class Workload:
    """One named workload: batch size, length recipe, cache format, seed."""
    name: str
    batch: int
    lengths: tuple          # ("fixed", L) | ("list", (L0, L1, ...)) | ("uniform", lo, hi)
    kv_dtype: str           # "bf16" | "fp8" (E4M3) | "fp4" (packed E2M1)
    permute_pages: bool     # False: sequence b owns a contiguous run of pages
    append_tokens: int      # tokens appended through the KV-append call before attention
    seed: int
    description: str = ""
    queries: int = 1        # query tokens per sequence (2: multi-token decode)
    select_blocks: int = 0  # block gather: historical 8-token blocks selected per sequence (0: whole sequence)


WORKLOADS = {
    "tiny": Workload("tiny", 2, ("list", (64, 100)), "bf16", False, 0, 11,
                     "B=2, KV lengths 64 and 100, contiguous pages"),
    "ctx4k": Workload("ctx4k", 32, ("fixed", 4096), "bf16", True, 0, 22,
                      "B=32, L=4096, pages randomly permuted"),
    "ragged": Workload("ragged", 128, ("uniform", 1024, 8192), "bf16", True, 1, 33,
                       "B=128, L uniform in [1024, 8192], one appended token per sequence"),
    "fp8": Workload("fp8", 64, ("fixed", 16384), "fp8", True, 0, 44,
                    "B=64, L=16384, E4M3 cache with per-token fp32 scales"),
    "fp4": Workload("fp4", 64, ("fixed", 16384), "fp4", True, 0, 88,
                    "B=64, L=16384, 4-bit KV: packed E2M1 codes with per-token fp32 scales"),
    "mtp4k": Workload("mtp4k", 32, ("fixed", 4096), "bf16", True, 0, 66,
                      "B=32, L=4096, two query tokens per sequence (multi-token decode), pages randomly permuted",
                      queries=2),
    "mtp4k_t4": Workload("mtp4k_t4", 32, ("fixed", 4096), "bf16", True, 0, 67,
                         "B=32, L=4096, four query tokens per sequence (multi-token decode), pages randomly permuted",
                         queries=4),
    "mtp4k_fp8": Workload("mtp4k_fp8", 32, ("fixed", 4096), "fp8", True, 0, 68,
                          "B=32, L=4096, E4M3 cache with per-token fp32 scales, two query tokens per sequence "
                          "(multi-token decode), pages randomly permuted", queries=2),
    "blocks32k": Workload("blocks32k", 32, ("fixed", 32768), "bf16", True, 0, 77,
                          "B=32, L=32768, 512 selected 8-token blocks plus the last block per sequence "
                          "(4104 tokens attended, block-gather decode), pages randomly permuted",
                          select_blocks=512),
    "blocks32k_fp8": Workload("blocks32k_fp8", 32, ("fixed", 32768), "fp8", True, 0, 78,
                              "B=32, L=32768, E4M3 cache with per-token fp32 scales, 512 selected 8-token blocks plus "
                              "the last block per sequence (block-gather decode), pages randomly permuted",
                              select_blocks=512),
    "long": Workload("long", 8, ("uniform", 65536, 131072), "bf16", True, 0, 55,
                     "B=8, L uniform in [65536, 131072], pages randomly permuted"),
}


def draw_lengths(w: Workload) -> np.ndarray:
    """Initial cache lengths (before any append) as int64 [B]."""
    kind = w.lengths[0]
    if kind == "fixed":
        return np.full(w.batch, int(w.lengths[1]), dtype=np.int64)
    if kind == "list":
        vals = np.asarray(w.lengths[1], dtype=np.int64)
        assert vals.size == w.batch
        return vals.copy()
    if kind == "uniform":
        rng = np.random.default_rng([w.seed, 6])
        return rng.integers(int(w.lengths[1]), int(w.lengths[2]) + 1, size=w.batch, dtype=np.int64)
    raise ValueError(kind)


def pages_for(tokens) -> np.ndarray:
    """Pages needed to hold `tokens` tokens (elementwise ceil(tokens / 64))."""
    t = np.asarray(tokens, dtype=np.int64)
    return (t + PAGE_SIZE - 1) // PAGE_SIZE


def build_page_table(pages_per_seq, permute: bool, seed, max_pages: int | None = None,
                     spare_pages: int = 0):
    """Assign pages to sequences.

    Sequence b receives pages_per_seq[b] page ids, in order, from either the
    identity order or a seeded random permutation of all pages.  Unused table
    entries hold -1.  `spare_pages` extra pages exist in the cache but belong to
    no sequence.  Returns (page_table int32 [B, max_pages], num_pages)."""
    pps = np.asarray(pages_per_seq, dtype=np.int64)
    B = pps.size
    total = int(pps.sum()) + int(spare_pages)
    mp = int(max_pages if max_pages is not None else max(1, int(pps.max()) if B else 1))
    assert mp >= (int(pps.max()) if B else 0)
    order = (np.random.default_rng([int(x) for x in np.atleast_1d(seed)] + [7]).permutation(total)
             if permute else np.arange(total))
    table = np.full((B, mp), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(pps[b])
        table[b, :n] = order[off:off + n]
        off += n
    return table, max(total, 1)


def _draw_chunk(seed_list, rows: int, width: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(int(np.random.SeedSequence(seed_list).generate_state(1)[0]))
    return torch.randn((rows, width), generator=g, dtype=torch.float32).to(torch.bfloat16)


def draw_rows(n_rows: int, width: int, seed, stream: int) -> torch.Tensor:
    """n_rows x width bf16 values ~ N(0,1) (fp32 draw rounded to bf16), CPU tensor.

    Rows are drawn in fixed chunks, each from its own generator seeded by
    (seed, stream, chunk index), so the result does not depend on threading."""
    out = torch.empty((n_rows, width), dtype=torch.bfloat16)
    base = [int(x) for x in np.atleast_1d(seed)] + [int(stream)]
    starts = list(range(0, n_rows, _CHUNK_TOKENS))

    def work(i_s):
        i, s = i_s
        r = min(_CHUNK_TOKENS, n_rows - s)
        out[s:s + r] = _draw_chunk(base + [i], r, width)

    workers = max(1, min(len(starts), (os.cpu_count() or 1)))
    if workers == 1:
        for item in enumerate(starts):
            work(item)
    else:
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, enumerate(starts)))
    return out


def slots_of(lengths, page_table) -> np.ndarray:
    """Cache slot (page * 64 + row) of every token of every sequence, concatenated
    in sequence order: token j of sequence b sits in page page_table[b, j // 64],
    row j % 64."""
    lens = np.asarray(lengths, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    parts = []
    for b, n in enumerate(lens):
        j = np.arange(int(n), dtype=np.int64)
        parts.append(pt[b, j // PAGE_SIZE] * PAGE_SIZE + j % PAGE_SIZE)
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def scatter_rows(rows: torch.Tensor, lengths, page_table, num_pages: int, fill=float("nan")):
    """Lay concatenated token rows [sum(L), D] out as a paged cache [num_pages, 64, D].

    Slots not covered by a token are filled with `fill` (NaN by default, so a
    kernel that reads an unused slot shows it)."""
    D = rows.shape[1]
    cache = torch.full((num_pages * PAGE_SIZE, D), fill, dtype=rows.dtype)
    idx = torch.from_numpy(slots_of(lengths, page_table))
    cache[idx] = rows
    return cache.view(num_pages, PAGE_SIZE, D)


@dataclass
class Case:
    """A complete decode-attention input set on the host."""
    workload: Workload
    lengths0: np.ndarray            # cache lengths before the append, int64 [B]
    q: torch.Tensor                 # [B, 64, 256] bf16
    k_rows: torch.Tensor            # [sum(lengths0), 256] bf16, sequences concatenated
    v_rows: torch.Tensor
    k_new: torch.Tensor | None      # [B, append_tokens, 256] bf16
    v_new: torch.Tensor | None
    page_table: np.ndarray          # int32 [B, max_pages]
    num_pages: int
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.lengths0.size)

    @property
    def lengths_after_append(self) -> np.ndarray:
        return self.lengths0 + (self.workload.append_tokens if self.k_new is not None else 0)


def make_case(w: Workload, *, lengths=None, headroom_tokens: int | None = None,
              max_pages: int | None = None, spare_pages: int = 0) -> Case:
    """Draw every input of workload `w`.

    `lengths` overrides the workload's length recipe (used for small parity
    cases).  Each sequence gets pages for its initial tokens plus
    `headroom_tokens` (default: the workload's appended tokens)."""
    lens = draw_lengths(w) if lengths is None else np.asarray(lengths, dtype=np.int64)
    B = lens.size
    head = w.append_tokens if headroom_tokens is None else headroom_tokens
    pps = pages_for(lens + head)
    table, num_pages = build_page_table(pps, w.permute_pages, [w.seed], max_pages, spare_pages)
    total = int(lens.sum())
    q = draw_rows(B * HEADS, HEAD_DIM, [w.seed], 1).view(B, HEADS, HEAD_DIM)
    k_rows = draw_rows(total, HEAD_DIM, [w.seed], 2)
    v_rows = draw_rows(total, HEAD_DIM, [w.seed], 3)
    k_new = v_new = None
    if w.append_tokens:
        k_new = draw_rows(B * w.append_tokens, HEAD_DIM, [w.seed], 4).view(B, w.append_tokens, HEAD_DIM)
        v_new = draw_rows(B * w.append_tokens, HEAD_DIM, [w.seed], 5).view(B, w.append_tokens, HEAD_DIM)
    return Case(w, lens, q, k_rows, v_rows, k_new, v_new, table, num_pages)


def draw_blocks(lengths, n_select: int, seed, max_blocks: int | None = None):
    """A seeded selection of historical 8-token blocks per sequence (an input:
    the selection itself is the caller's). Sequence b of length L has
    floor((L - 1) / 8) complete blocks before the one holding its last token;
    min(n_select, that count) distinct ones are drawn uniformly, in random
    order. Returns (block_idx int32 [B, max_blocks] padded with -1, n_blocks
    int32 [B])."""
    lens = np.asarray(lengths, dtype=np.int64)
    B = lens.size
    width = max(1, n_select if max_blocks is None else max_blocks)
    rng = np.random.default_rng(np.random.SeedSequence([int(x) for x in np.atleast_1d(seed)] + [77]))
    block_idx = np.full((B, width), -1, dtype=np.int32)
    n_blocks = np.zeros(B, dtype=np.int32)
    for b in range(B):
        hist = max(0, (int(lens[b]) - 1) // 8)
        k = min(n_select, hist, width)
        if k:
            block_idx[b, :k] = rng.choice(hist, size=k, replace=False)
        n_blocks[b] = k
    return block_idx, n_blocks


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (no copy when contiguous)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def padded_rows(rows: torch.Tensor, lengths, width: int | None = None) -> torch.Tensor:
    """Concatenated rows [sum(L), D] -> [B, max L (or width), D], zero padded."""
    lens = np.asarray(lengths, dtype=np.int64)
    W = int(width if width is not None else (lens.max() if lens.size else 0))
    out = torch.zeros((lens.size, W, rows.shape[1]), dtype=rows.dtype)
    off = 0
    for b, n in enumerate(lens):
        out[b, :n] = rows[off:off + n]
        off += int(n)
    return out
