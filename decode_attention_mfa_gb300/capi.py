"""Thin ctypes binding of libmfa (include/mfa.h), same names as the C ABI.

Arguments are marshalled only: a torch tensor becomes its data pointer, a
stream its CUDA handle.  Every computation runs in the CUDA library; there is
no CPU or PyTorch fallback, and a missing library raises at the first call.
A status other than MFA_OK raises MFAError with the library's message.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmfa.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "mfa.h")

MFA_OK = 0
STATUS_NAMES = {0: "MFA_OK", 1: "MFA_ERR_INVALID_ARG", 2: "MFA_ERR_UNSUPPORTED", 3: "MFA_ERR_CUDA",
                4: "MFA_ERR_WORKSPACE", 5: "MFA_ERR_DEVICE_PAGE", 6: "MFA_ERR_DEVICE_CAPACITY",
                7: "MFA_ERR_DEVICE_TIMEOUT"}
HEADS, HEAD_DIM, PAGE_SIZE, MAX_BATCH, MAX_QUERY_TOKENS = 64, 256, 64, 1024, 8

_lock = threading.Lock()
_lib = None


class MFAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Plan(ctypes.Structure):
    _fields_ = [("grid_ctas", ctypes.c_int), ("partial_slots", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t)]


_P, _I, _F, _Z, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
_SIGNATURES = {
    "mfa_plan_decode": ([_I, _I, _I, ctypes.POINTER(Plan)], _I),
    "mfa_decode_workspace_bytes": ([_I, _I], _Z),
    "mfa_workspace_init": ([_P, _Z, _P], _I),
    "mfa_kv_append": ([_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "mfa_kv_append_fp8": ([_P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "mfa_decode_attention": ([_P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_decode_attention_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_kv_append_fp4": ([_P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "mfa_decode_attention_fp4": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_decode_attention_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _P, _P], _I),
    "mfa_decode_mtp_workspace_bytes": ([_I, _I, _I], _Z),
    "mfa_query_lowrank_workspace_bytes": ([_I, _I, _I], _Z),
    "mfa_query_lowrank": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _Z, _P], _I),
    "mfa_decode_attention_mtp": ([_P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_decode_attention_mtp_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_decode_attention_mtp_fp4": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_decode_attention_blocks": ([_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _F, _I, _I, _I, _I, _P, _Z, _P], _I),
    "mfa_decode_attention_blocks_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _F, _I, _I, _I, _I, _P, _Z,
                                         _P], _I),
    "mfa_check_device_errors": ([_P, _I, _P], _I),
    "mfa_set_wait_budget_ns": ([_U64], None),
    "mfa_selftest_wait_timeout": ([_P, _U64, _P], _I),
    "mfa_profile_split_events": ([_P, _P], None),
    "mfa_status_string": ([_I], ctypes.c_char_p),
    "mfa_last_error": ([], ctypes.c_char_p),
}


def header_functions() -> list[str]:
    """Names of the functions include/mfa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mfa_[a-z0-9_]+)\s*\(", text)))


def load():
    """Load libmfa.so (built by decode_attention_mfa_gb300.build); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmfa.so is not built ({LIB_PATH}); run "
                               "`python -m decode_attention_mfa_gb300.build` first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != MFA_OK:
        msg = load().mfa_last_error().decode(errors="replace")
        raise MFAError(status, msg)


# ----------------------------------------------------------------- C ABI
def mfa_plan_decode(batch: int, max_len_hint: int, num_sms: int = 0) -> Plan:
    plan = Plan()
    _check(load().mfa_plan_decode(batch, max_len_hint, num_sms, ctypes.byref(plan)))
    return plan


def mfa_decode_workspace_bytes(batch: int, max_len_hint: int) -> int:
    n = load().mfa_decode_workspace_bytes(batch, max_len_hint)
    if n == 0:
        _check(load().mfa_plan_decode(batch, max_len_hint, 0, ctypes.byref(Plan())))
    return int(n)


def mfa_workspace_init(workspace, workspace_bytes: int, stream=None):
    _check(load().mfa_workspace_init(_ptr(workspace), workspace_bytes, _stream(stream)))


def mfa_kv_append(k_new, v_new, n_new, k_cache, v_cache, page_table, seq_lens, batch, max_pages,
                  num_pages, workspace, stream=None):
    _check(load().mfa_kv_append(_ptr(k_new), _ptr(v_new), n_new, _ptr(k_cache), _ptr(v_cache),
                                _ptr(page_table), _ptr(seq_lens), batch, max_pages, num_pages,
                                _ptr(workspace), _stream(stream)))


def mfa_kv_append_fp8(k_new, v_new, n_new, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                      batch, max_pages, num_pages, workspace, stream=None):
    _check(load().mfa_kv_append_fp8(_ptr(k_new), _ptr(v_new), n_new, _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scale), _ptr(v_scale), _ptr(page_table), _ptr(seq_lens),
                                    batch, max_pages, num_pages, _ptr(workspace), _stream(stream)))


def mfa_kv_append_fp4(k_new, v_new, n_new, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                      batch, max_pages, num_pages, workspace, stream=None):
    """4-bit KV append: caches uint8 [num_pages, 64, 128] (packed E2M1), scales fp32 [num_pages, 64]."""
    _check(load().mfa_kv_append_fp4(_ptr(k_new), _ptr(v_new), n_new, _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scale), _ptr(v_scale), _ptr(page_table), _ptr(seq_lens),
                                    batch, max_pages, num_pages, _ptr(workspace), _stream(stream)))


def mfa_decode_attention_fp4(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, out, lse, scale,
                             batch, max_pages, num_pages, max_len_hint, workspace, workspace_bytes,
                             stream=None):
    """Decode attention over a 4-bit (packed E2M1 + per-token scale) cache."""
    _check(load().mfa_decode_attention_fp4(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                           _ptr(v_scale), _ptr(page_table), _ptr(seq_lens), _ptr(out),
                                           _ptr(lse), float(scale), batch, max_pages, num_pages,
                                           max_len_hint, _ptr(workspace), workspace_bytes,
                                           _stream(stream)))


def mfa_decode_attention(q, k_cache, v_cache, page_table, seq_lens, out, lse, scale, batch, max_pages,
                         num_pages, max_len_hint, workspace, workspace_bytes, stream=None):
    _check(load().mfa_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                       _ptr(seq_lens), _ptr(out), _ptr(lse), float(scale), batch,
                                       max_pages, num_pages, max_len_hint, _ptr(workspace),
                                       workspace_bytes, _stream(stream)))


MAX_QUERY_BATCH = 256
MAX_QUERY_RANK = 16384


def mfa_query_lowrank_workspace_bytes(batch: int, rank: int, n_out: int) -> int:
    """Workspace bytes for query-path calls of up to `batch` rows."""
    n = load().mfa_query_lowrank_workspace_bytes(batch, rank, n_out)
    if n == 0:
        raise MFAError(1, "bad arguments for mfa_query_lowrank_workspace_bytes")
    return n


def mfa_query_lowrank(x, w_down, gamma, w_up, q, batch, d_model, rank, n_out, eps, workspace, workspace_bytes,
                      stream=None):
    """Low-rank query path: q = bf16(RMSNorm(x W_down) * gamma) W_up, bf16 in and out."""
    _check(load().mfa_query_lowrank(_ptr(x), _ptr(w_down), _ptr(gamma), _ptr(w_up), _ptr(q), batch, d_model, rank,
                                    n_out, float(eps), _ptr(workspace), workspace_bytes, _stream(stream)))


def mfa_decode_mtp_workspace_bytes(batch: int, n_query: int, max_len_hint: int) -> int:
    n = load().mfa_decode_mtp_workspace_bytes(batch, n_query, max_len_hint)
    if n == 0:
        raise MFAError(1, "bad arguments for mfa_decode_mtp_workspace_bytes")
    return n


def mfa_decode_attention_mtp(q, k_cache, v_cache, page_table, seq_lens, out, lse, scale, batch, n_query,
                             max_pages, num_pages, max_len_hint, workspace, workspace_bytes, stream=None):
    """Multi-token decode: q and out [batch, n_query, 64, 256] bf16, lse [batch, n_query, 64] fp32."""
    _check(load().mfa_decode_attention_mtp(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                           _ptr(seq_lens), _ptr(out), _ptr(lse), float(scale), batch, n_query,
                                           max_pages, num_pages, max_len_hint, _ptr(workspace),
                                           workspace_bytes, _stream(stream)))


def mfa_decode_attention_mtp_fp8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, out, lse, scale,
                                 batch, n_query, max_pages, num_pages, max_len_hint, workspace, workspace_bytes,
                                 stream=None):
    """Multi-token decode over an E4M3 cache with per-token fp32 scales."""
    _check(load().mfa_decode_attention_mtp_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                               _ptr(page_table), _ptr(seq_lens), _ptr(out), _ptr(lse), float(scale),
                                               batch, n_query, max_pages, num_pages, max_len_hint, _ptr(workspace),
                                               workspace_bytes, _stream(stream)))


def mfa_decode_attention_mtp_fp4(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, out, lse, scale,
                                 batch, n_query, max_pages, num_pages, max_len_hint, workspace, workspace_bytes,
                                 stream=None):
    """Multi-token decode over a packed E2M1 cache with per-token fp32 scales."""
    _check(load().mfa_decode_attention_mtp_fp4(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                               _ptr(page_table), _ptr(seq_lens), _ptr(out), _ptr(lse), float(scale),
                                               batch, n_query, max_pages, num_pages, max_len_hint, _ptr(workspace),
                                               workspace_bytes, _stream(stream)))


def mfa_decode_attention_blocks(q, k_cache, v_cache, page_table, seq_lens, block_idx, n_blocks, max_blocks, out,
                                lse, scale, batch, max_pages, num_pages, max_len_hint, workspace, workspace_bytes,
                                stream=None):
    """Decode over selected 8-token blocks: block_idx int32 [batch, max_blocks], n_blocks int32 [batch]."""
    _check(load().mfa_decode_attention_blocks(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                              _ptr(seq_lens), _ptr(block_idx), _ptr(n_blocks), max_blocks, _ptr(out),
                                              _ptr(lse), float(scale), batch, max_pages, num_pages, max_len_hint,
                                              _ptr(workspace), workspace_bytes, _stream(stream)))


def mfa_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, out, lse, scale,
                             batch, max_pages, num_pages, max_len_hint, workspace, workspace_bytes,
                             stream=None):
    _check(load().mfa_decode_attention_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                           _ptr(v_scale), _ptr(page_table), _ptr(seq_lens), _ptr(out),
                                           _ptr(lse), float(scale), batch, max_pages, num_pages,
                                           max_len_hint, _ptr(workspace), workspace_bytes,
                                           _stream(stream)))


def mfa_decode_attention_noalloc(q, k_cache, v_cache, page_table, seq_lens, out, lse, scale, batch, max_pages,
                                 num_pages, max_len_hint, device_error_word=None, stream=None):
    """Same as mfa_decode_attention, but the split scratch is the library's own
    static device array (no workspace argument); see include/mfa.h."""
    _check(load().mfa_decode_attention_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                               _ptr(seq_lens), _ptr(out), _ptr(lse), float(scale), batch,
                                               max_pages, num_pages, max_len_hint, _ptr(device_error_word),
                                               _stream(stream)))


def mfa_decode_attention_blocks_fp8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, block_idx,
                                    n_blocks, max_blocks, out, lse, scale, batch, max_pages, num_pages, max_len_hint,
                                    workspace, workspace_bytes, stream=None):
    """Block gather over an E4M3 cache with per-token fp32 scales."""
    _check(load().mfa_decode_attention_blocks_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                                  _ptr(v_scale), _ptr(page_table), _ptr(seq_lens), _ptr(block_idx),
                                                  _ptr(n_blocks), max_blocks, _ptr(out), _ptr(lse), float(scale),
                                                  batch, max_pages, num_pages, max_len_hint, _ptr(workspace),
                                                  workspace_bytes, _stream(stream)))


def mfa_check_device_errors(workspace, clear: bool = True, stream=None):
    _check(load().mfa_check_device_errors(_ptr(workspace), int(clear), _stream(stream)))


def mfa_set_wait_budget_ns(budget_ns: int):
    load().mfa_set_wait_budget_ns(int(budget_ns))


def mfa_selftest_wait_timeout(workspace, budget_ns: int, stream=None):
    _check(load().mfa_selftest_wait_timeout(_ptr(workspace), int(budget_ns), _stream(stream)))


def mfa_profile_split_events(start_event, stop_event):
    """torch.cuda.Event objects (or raw handles); None, None turns the hook off."""
    def handle(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    load().mfa_profile_split_events(handle(start_event), handle(stop_event))


def mfa_status_string(status: int) -> str:
    return load().mfa_status_string(status).decode()


def mfa_last_error() -> str:
    return load().mfa_last_error().decode(errors="replace")
