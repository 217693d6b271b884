"""Algorithmic bytes and FLOPs of one MFA decode step (roofline accounting).

Per token of context, MFA decode attention reads one K row and one V row of
HEAD_DIM elements (all 64 query heads share them) and does two 64 x 256
contractions against them (QK^T and PV), 2 FLOPs per multiply-add:

    FLOPs per token = 4 * 64 * 256 = 65,536
    KV bytes per token = 2 * 256 * bytes(element)   (+ 2 fp32 scales for E4M3)

These reproduce the pages' own accounting: "Step-3 is Large yet Affordable"
(paper summary page), Table 2 and Table 3 (Step-3 row: KV bytes and attention
FLOPs per decoded token at 8K and 32K context over 61 layers with 8-bit KV),
section 5.1 (arithmetic intensity 128 with 8-bit KV) and section 7 (512 bytes
of KV per token per layer).  tests/test_accounting.py pins them.
"""
from __future__ import annotations

import numpy as np

HEADS = 64
HEAD_DIM = 256
PAGE_SIZE = 64
STEP3_LAYERS = 61


def kv_bytes_per_token(kv_dtype: str, include_scales: bool = True, head_dim: int = HEAD_DIM) -> int:
    """Bytes of K plus V per cached token (one shared K head, one shared V head)."""
    if kv_dtype == "bf16":
        return 2 * head_dim * 2
    if kv_dtype == "fp8":
        return 2 * head_dim + (2 * 4 if include_scales else 0)
    if kv_dtype == "fp4":  # two E2M1 codes per byte
        return head_dim + (2 * 4 if include_scales else 0)
    raise ValueError(kv_dtype)


def attention_flops_per_token(heads: int = HEADS, head_dim: int = HEAD_DIM) -> int:
    """FLOPs per context token: QK^T and PV, each heads x head_dim multiply-adds."""
    return 4 * heads * head_dim


def decode_step_bytes(lengths_attended, kv_dtype: str, appended_tokens: int = 0, n_query: int = 1) -> int:
    """Algorithmic HBM bytes of one decode step over a batch.

    Counts each byte the step must move once: the KV rows attended (after the
    append; with n_query query tokens per sequence, multi-token decode, the
    rows of the longest, last token, which cover the others), the queries
    (bf16), the outputs (bf16) and per-head LSE (fp32) of every query token,
    the page-table entries and sequence lengths read, and for an append the
    new bf16 K/V rows read plus the cache rows (and scales) written.  Split-KV
    partial results are an implementation choice and are not counted."""
    lens = np.asarray(lengths_attended, dtype=np.int64)
    B = int(lens.size)
    kv = int(lens.sum()) * kv_bytes_per_token(kv_dtype)
    q = n_query * B * HEADS * HEAD_DIM * 2
    out = n_query * (B * HEADS * HEAD_DIM * 2 + B * HEADS * 4)
    table = int(((lens + PAGE_SIZE - 1) // PAGE_SIZE).sum()) * 4 + B * 4
    app = 0
    if appended_tokens:
        app = B * appended_tokens * (2 * HEAD_DIM * 2 + kv_bytes_per_token(kv_dtype)) + B * 4
    return kv + q + out + table + app


def blocks_attended(seq_lens, n_blocks) -> np.ndarray:
    """Tokens a block-gather decode attends per sequence: 8 per selected block
    plus the last block up to the last token (none for an empty sequence)."""
    L = np.asarray(seq_lens, dtype=np.int64)
    nb = np.asarray(n_blocks, dtype=np.int64)
    return np.where(L > 0, 8 * nb + L - 8 * ((L - 1) // 8), 0)


def decode_blocks_step_bytes(seq_lens, n_blocks, kv_dtype: str = "bf16") -> int:
    """Algorithmic HBM bytes of one block-gather decode step: the K/V rows of
    the attended tokens, queries, outputs and LSE, one page-table entry per
    attended block, the selected block ids, and the per-sequence length and
    block count."""
    att = blocks_attended(seq_lens, n_blocks)
    B = int(att.size)
    nb = np.asarray(n_blocks, dtype=np.int64)
    kv = int(att.sum()) * kv_bytes_per_token(kv_dtype)
    q = B * HEADS * HEAD_DIM * 2
    out = B * HEADS * HEAD_DIM * 2 + B * HEADS * 4
    blocks = int(np.where(att > 0, nb + 1, 0).sum()) * 4 + int(nb.sum()) * 4
    return kv + q + out + blocks + B * 8


def decode_step_flops(lengths_attended, n_query: int = 1) -> int:
    """FLOPs of one decode step; query token t of n_query sees L - n_query + 1 + t tokens."""
    lens = np.asarray(lengths_attended, dtype=np.int64)
    seen = sum(int(np.maximum(lens - n_query + 1 + t, 0).sum()) for t in range(n_query))
    return seen * attention_flops_per_token()
