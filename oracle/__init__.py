"""Double-precision CPU oracle for decode-time MFA attention -- TEST INFRASTRUCTURE.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it, and it shares no
code with the CUDA library: the arithmetic lives in ``mfa_oracle.c`` (plain C,
fp64, written from the definitions cited there) and this module only marshals
numpy arrays through ctypes.

Sources (see ``mfa_oracle.c`` for the full list):
  * "Step-3 is Large yet Affordable" (paper summary page), section 2 / Table 1:
    64 query heads share one key head and one value head of dimension 256.
  * Same page, sections 7 and 8.1: decode attention over the per-sequence KV
    cache, 8-bit KV at 512 bytes per token per layer.
  * OCP 8-bit floating point specification, E4M3 format.

Every function here has its pins in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mfa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmfa_oracle.so")
_lock = threading.Lock()
_lib = None

PAGE_SIZE = 64


def build(force: bool = False) -> str:
    """Compile ``mfa_oracle.c`` into ``libmfa_oracle.so`` (gcc, -O2, OpenMP if available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = f64
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = f64
        lib.oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_f32.restype = ctypes.c_uint8
        lib.oracle_e4m3_from_f32_array.argtypes = [P, i64, P]
        lib.oracle_e4m3_from_f32_array.restype = None
        lib.oracle_e4m3_to_f64_array.argtypes = [P, i64, P]
        lib.oracle_e4m3_to_f64_array.restype = None
        lib.oracle_quantize_tokens_e4m3.argtypes = [P, i64, i32, P, P]
        lib.oracle_quantize_tokens_e4m3.restype = None
        lib.oracle_e2m1_to_f64_array.argtypes = [P, i64, P]
        lib.oracle_e2m1_to_f64_array.restype = None
        lib.oracle_e2m1_from_f32_array.argtypes = [P, i64, P]
        lib.oracle_e2m1_from_f32_array.restype = None
        lib.oracle_quantize_tokens_e2m1.argtypes = [P, i64, i32, P, P]
        lib.oracle_quantize_tokens_e2m1.restype = None
        lib.oracle_mfa_decode_rows.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                               i64, f64, P, P, i64, P, P, i32]
        lib.oracle_mfa_decode_rows.restype = i32
        lib.oracle_mfa_decode.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i64,
                                          f64, P, P, i32]
        lib.oracle_mfa_decode.restype = i32
        lib.oracle_kv_append.argtypes = [P, P, i32, P, P, P, P, i32, P, P, i32, i32, i32, i32, i64]
        lib.oracle_kv_append.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------- E4M3 codec
def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> exact fp64 values (OCP OFP8 E4M3 definition)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_to_f64_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> nearest E4M3 code, ties to even, saturating to +-448."""
    xa = _c(x, np.float32)
    out = np.empty(xa.shape, dtype=np.uint8)
    _load().oracle_e4m3_from_f32_array(_ptr(xa), xa.size, _ptr(out))
    return out


def quantize_tokens_e4m3(x_bf16_bits) -> tuple[np.ndarray, np.ndarray]:
    """Per-token E4M3 quantisation of bf16 rows [..., d] (given as uint16 bit patterns).

    Returns (codes uint8 [..., d], scales float32 [...]): scale = absmax / 448 in
    fp32 (1 when the row is all zero), code = E4M3(x / scale)."""
    x = _c(x_bf16_bits, np.uint16)
    d = x.shape[-1]
    n = x.size // d
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    _load().oracle_quantize_tokens_e4m3(_ptr(x), n, d, _ptr(codes), _ptr(scales))
    return codes, scales


# ---------------------------------------------------------------- E2M1 codec (4-bit KV)
def e2m1_decode(codes) -> np.ndarray:
    """4-bit E2M1 codes (uint8 values 0..15) -> exact fp64 values (OCP MX FP4 definition)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e2m1_to_f64_array(_ptr(c), c.size, _ptr(out))
    return out


def e2m1_encode(x) -> np.ndarray:
    """fp32 values -> nearest E2M1 code (0..15), ties to the even mantissa, saturating to +-6."""
    xa = _c(x, np.float32)
    out = np.empty(xa.shape, dtype=np.uint8)
    _load().oracle_e2m1_from_f32_array(_ptr(xa), xa.size, _ptr(out))
    return out


def quantize_tokens_e2m1(x_bf16_bits) -> tuple[np.ndarray, np.ndarray]:
    """Per-token 4-bit quantisation of bf16 rows [..., d] (uint16 bit patterns, d even).

    "Step-3 is Large yet Affordable" (paper summary page), section 5.2: KV stored
    in 4 bits, attention computed in 8 bits. Returns (packed uint8 [..., d/2],
    scales float32 [...]): scale = absmax / 6 in fp32 (1 for an all-zero row),
    code = E2M1(x / scale), element 2k in the low nibble of byte k."""
    x = _c(x_bf16_bits, np.uint16)
    d = x.shape[-1]
    n = x.size // d
    packed = np.empty(x.shape[:-1] + (d // 2,), dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    _load().oracle_quantize_tokens_e2m1(_ptr(x), n, d, _ptr(packed), _ptr(scales))
    return packed, scales


def unpack_e2m1(packed) -> np.ndarray:
    """Packed bytes [..., d/2] -> codes [..., d] (element 2k from the low nibble)."""
    p = _c(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


def _kv_format(cache, head_dim) -> int:
    """0 bf16 (uint16 [..., D]), 1 E4M3 (uint8 [..., D]), 2 packed E2M1 (uint8 [..., D/2])."""
    a = np.asarray(cache)
    if a.dtype == np.uint16:
        return 0
    if a.dtype == np.uint8 and a.shape[-1] == head_dim:
        return 1
    if a.dtype == np.uint8 and 2 * a.shape[-1] == head_dim:
        return 2
    raise ValueError(f"cache of dtype {a.dtype} and row width {a.shape[-1]} matches no format for D = {head_dim}")


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values."""
    b = _c(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- attention
def mfa_decode(q_bits, k_cache, v_cache, page_table, seq_lens, scale, *, k_scale=None,
               v_scale=None, rows=None, threads=None):
    """MFA decode attention over a paged KV cache, in fp64.

    q_bits     [B, H, D] uint16 (bf16 bits)
    k_cache    [num_pages, page, D] uint16 (bf16 bits) or uint8 (E4M3 codes), or
               [num_pages, page, D/2] uint8 (packed E2M1 codes, 4-bit KV)
    v_cache    same as k_cache
    page_table [B, max_pages] int32, seq_lens [B] int32
    k_scale/v_scale [num_pages, page] float32 for an E4M3 or E2M1 cache
    rows       optional (b_idx, h_idx) int arrays: compute only those rows
    Returns (out, lse): out [B, H, D] (or [n_rows, D]) fp64, lse [B, H] (or [n_rows]).
    """
    q = _c(q_bits, np.uint16)
    B, H, D = q.shape
    fmt = _kv_format(k_cache, D)
    if _kv_format(v_cache, D) != fmt:
        raise ValueError("k_cache and v_cache differ in format")
    fp8 = fmt != 0
    kc = _c(k_cache, np.uint8 if fp8 else np.uint16)
    vc = _c(v_cache, np.uint8 if fp8 else np.uint16)
    num_pages, page_size = kc.shape[0], kc.shape[1]
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    if fp8 and (ks is None or vs is None):
        raise ValueError("an E4M3 cache needs k_scale and v_scale")
    threads = threads or default_threads()
    lib = _load()
    if rows is None:
        out = np.empty((B, H, D), dtype=np.float64)
        lse = np.empty((B, H), dtype=np.float64)
        st = lib.oracle_mfa_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), fmt,
                                   _ptr(pt), _ptr(sl), B, H, D, page_size, pt.shape[1], num_pages,
                                   float(scale), _ptr(out), _ptr(lse), int(threads))
    else:
        rb = _c(rows[0], np.int32)
        rh = _c(rows[1], np.int32)
        out = np.empty((rb.size, D), dtype=np.float64)
        lse = np.empty((rb.size,), dtype=np.float64)
        st = lib.oracle_mfa_decode_rows(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), fmt,
                                        _ptr(pt), _ptr(sl), B, H, D, page_size, pt.shape[1],
                                        num_pages, float(scale), _ptr(rb), _ptr(rh), rb.size,
                                        _ptr(out), _ptr(lse), int(threads))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (code {st})")
    return out, lse


def mfa_decode_mtp(q_bits, k_cache, v_cache, page_table, seq_lens, scale, *, k_scale=None,
                   v_scale=None, threads=None):
    """Multi-token (MTP) decode: T query tokens per sequence, in fp64.

    "Step-3 is Large yet Affordable" (paper summary page), section 5.2: with
    multi-token prediction a decode step carries extra predicted tokens, which
    read the same KV cache. The tokens are the last T positions of sequence b
    (the cache of seq_lens[b] tokens already holds them), so query token t sits
    at position L_b - T + t and attends, causally, to positions
    j < L_b - T + 1 + t. Each (b, t) is therefore the single-token decode of
    ``mfa_decode`` over the first L_b - T + 1 + t tokens of sequence b (none if
    that is <= 0: out = 0, lse = -inf).

    q_bits [B, T, H, D] uint16 (bf16 bits); the other arguments as in mfa_decode.
    Returns (out, lse): out [B, T, H, D] fp64, lse [B, T, H]."""
    q = _c(q_bits, np.uint16)
    B, T, H, D = q.shape
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32).astype(np.int64)
    lens = np.maximum(sl[:, None] - T + 1 + np.arange(T)[None, :], 0).astype(np.int32).reshape(B * T)
    out, lse = mfa_decode(q.reshape(B * T, H, D), k_cache, v_cache, np.repeat(pt, T, axis=0), lens, scale,
                          k_scale=k_scale, v_scale=v_scale, threads=threads)
    return out.reshape(B, T, H, D), lse.reshape(B, T, H)


BLOCK_SIZE = 8


def selected_positions(seq_len, blocks):
    """Positions attended by a decode query over selected 8-token blocks.

    "Step-5-Preview" page (sparse attention, selection and main attention): the
    query at position t = L - 1 attends to the union of the selected historical
    blocks r (each covering positions 8r .. 8r + 7, with r < floor(t / 8)) and
    the positions of its own block up to itself, 8 floor(t / 8) .. t; the
    softmax runs over that set of original K/V rows. Returns the positions in
    ascending order. Raises ValueError for a block outside [0, floor(t / 8))
    or a block listed twice (the selection is a set)."""
    L = int(seq_len)
    blocks = [int(r) for r in blocks]
    if L <= 0:
        if blocks:
            raise ValueError("an empty sequence has no blocks to select")
        return np.zeros(0, dtype=np.int64)
    cur = (L - 1) // BLOCK_SIZE
    if len(set(blocks)) != len(blocks):
        raise ValueError("a block is selected twice")
    for r in blocks:
        if not 0 <= r < cur:
            raise ValueError(f"block {r} is not a historical block of a length-{L} sequence")
    pos = [BLOCK_SIZE * r + i for r in sorted(blocks) for i in range(BLOCK_SIZE)]
    pos += list(range(BLOCK_SIZE * cur, L))
    return np.asarray(pos, dtype=np.int64)


def mfa_decode_blocks(q_bits, k_cache, v_cache, page_table, seq_lens, block_idx, n_blocks, scale, *,
                      k_scale=None, v_scale=None, threads=None):
    """MFA decode attention over caller-selected 8-token blocks, in fp64.

    The selection rule of ``selected_positions`` with the block list
    block_idx[b, :n_blocks[b]] of sequence b, applied to MFA's shared K/V head
    (the selection itself is an input). The selected rows are copied, in
    ascending position order, into a fresh paged cache of their own (a plain
    gather; for a quantised cache the codes and their per-token scales move
    together), and ``mfa_decode`` runs over it with the selected count as length.

    q_bits [B, H, D] uint16; caches [num_pages, 64, D] uint16 (bf16 bits) or the
    quantised formats of ``mfa_decode`` with k_scale/v_scale [num_pages, 64];
    page_table [B, max_pages], seq_lens [B], block_idx [B, max_blocks],
    n_blocks [B] int32. Returns (out [B, H, D], lse [B, H]) fp64."""
    q = _c(q_bits, np.uint16)
    B, H, D = q.shape
    fmt = _kv_format(k_cache, D)
    quantised = fmt != 0
    kc = _c(k_cache, np.uint8 if quantised else np.uint16)
    vc = _c(v_cache, np.uint8 if quantised else np.uint16)
    if quantised and (k_scale is None or v_scale is None):
        raise ValueError("a quantised cache needs k_scale and v_scale")
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    bi = np.asarray(block_idx, dtype=np.int32).reshape(B, -1)
    nb = np.asarray(n_blocks, dtype=np.int32).reshape(B)
    num_pages, page, W = kc.shape[0], kc.shape[1], kc.shape[2]
    k_rows, v_rows = kc.reshape(-1, W), vc.reshape(-1, W)
    if quantised:
        ks_rows = _c(k_scale, np.float32).reshape(-1)
        vs_rows = _c(v_scale, np.float32).reshape(-1)
    sel = []
    for b in range(B):
        if not 0 <= nb[b] <= bi.shape[1]:
            raise ValueError(f"n_blocks[{b}] = {nb[b]} outside [0, {bi.shape[1]}]")
        pos = selected_positions(sl[b], bi[b, :nb[b]])
        ids = pt[b, pos // page].astype(np.int64)
        if np.any((ids < 0) | (ids >= num_pages)):
            raise ValueError(f"sequence {b}: page id out of range")
        sel.append(ids * page + pos % page)
    lens = np.array([len(x) for x in sel], dtype=np.int32)
    pages_of = [(n + page - 1) // page for n in lens]
    max_p = max(1, max(pages_of))
    tot = max(1, sum(pages_of))
    gk = np.zeros((tot * page, W), dtype=kc.dtype)
    gv = np.zeros((tot * page, W), dtype=vc.dtype)
    gks = np.ones(tot * page, dtype=np.float32)
    gvs = np.ones(tot * page, dtype=np.float32)
    gpt = np.zeros((B, max_p), dtype=np.int32)
    nxt = 0
    for b in range(B):
        gk[nxt * page:nxt * page + lens[b]] = k_rows[sel[b]]
        gv[nxt * page:nxt * page + lens[b]] = v_rows[sel[b]]
        if quantised:
            gks[nxt * page:nxt * page + lens[b]] = ks_rows[sel[b]]
            gvs[nxt * page:nxt * page + lens[b]] = vs_rows[sel[b]]
        gpt[b, :pages_of[b]] = np.arange(nxt, nxt + pages_of[b])
        nxt += pages_of[b]
    if not quantised:
        return mfa_decode(q, gk.reshape(tot, page, W), gv.reshape(tot, page, W), gpt, lens, scale, threads=threads)
    return mfa_decode(q, gk.reshape(tot, page, W), gv.reshape(tot, page, W), gpt, lens, scale,
                      k_scale=gks.reshape(tot, page), v_scale=gvs.reshape(tot, page), threads=threads)


def query_lowrank(x_bits, w_down_bits, gamma_bits, w_up_bits, eps):
    """MFA's low-rank query path in fp64.

    "Step-3 is Large yet Affordable" (paper summary page), section 2 / Table 1:
    the query is projected down from the model width (7168) to a low rank
    (2048), normalised, then projected up to 64 heads x 256. The normalisation
    is read as RMSNorm with a learned gain: h = y / sqrt(mean(y^2) + eps) *
    gamma, with y = x W_down. matmul is the library primitive for the two
    products.

    x_bits [B, Dm], w_down_bits [Dm, R], gamma_bits [R], w_up_bits [R, N]
    (uint16, bf16 bits). Returns (q [B, N], h [B, R]) in fp64; q reshapes to
    [B, 64, 256] when N = 16384."""
    x = bf16_to_f64(_c(x_bits, np.uint16))
    wd = bf16_to_f64(_c(w_down_bits, np.uint16))
    g = bf16_to_f64(_c(gamma_bits, np.uint16))
    wu = bf16_to_f64(_c(w_up_bits, np.uint16))
    y = x @ wd
    h = y / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + float(eps)) * g[None, :]
    return h @ wu, h


def kv_append(k_new_bits, v_new_bits, k_cache, v_cache, page_table, seq_lens, *, k_scale=None,
              v_scale=None):
    """Append n_new tokens per sequence to host copies of the cache, in place.

    k_new_bits/v_new_bits: [B, n_new, D] uint16 (bf16 bits).  For an E4M3 or a
    packed E2M1 cache (uint8 k_cache/v_cache) the tokens are quantised per token;
    k_scale/v_scale are updated in place.  seq_lens is incremented in place."""
    kn = _c(k_new_bits, np.uint16)
    vn = _c(v_new_bits, np.uint16)
    B, n_new, D = kn.shape
    fmt = _kv_format(k_cache, D)
    fp8 = fmt != 0
    for a in (k_cache, v_cache, page_table, seq_lens) + ((k_scale, v_scale) if fp8 else ()):
        if not a.flags.c_contiguous:
            raise ValueError("in-place arrays must be C-contiguous")
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    st = _load().oracle_kv_append(_ptr(kn), _ptr(vn), n_new, _ptr(k_cache), _ptr(v_cache),
                                  _ptr(k_scale) if fp8 else None, _ptr(v_scale) if fp8 else None,
                                  fmt, _ptr(page_table), _ptr(seq_lens), B, D, page_size,
                                  page_table.shape[1], num_pages)
    if st != 0:
        raise ValueError(f"oracle append rejected the inputs (code {st})")
