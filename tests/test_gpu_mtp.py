"""Multi-token (MTP) decode on the GPU against the fp64 oracle.

Two query tokens per sequence share each pass over the bf16 cache; token t
attends causally to positions j < L - 2 + 1 + t. Small cases put the causal
boundary on every tile position that matters (a token that sees nothing, the
last row of a page or of a tile, a one-row last tile), on the planned grid and
on one CTA; the 4K-context shape runs at full size. Tolerances as for
single-token decode."""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import DeviceCache, compare

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

T = 2


def mtp_case(lengths, seed, n_query=T, headroom=0):
    w = wl.Workload("mtp", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
    case = wl.make_case(w, lengths=lengths, spare_pages=1, headroom_tokens=headroom)
    q = wl.draw_rows(len(lengths) * n_query * wl.HEADS, wl.HEAD_DIM, [seed, 90], 0)
    return case, q.view(len(lengths), n_query, wl.HEADS, wl.HEAD_DIM)


def run_mtp(dev, q, n_query=T, hint=None):
    qd = q.to(dev.q.device).contiguous()
    out = torch.empty((dev.B, n_query, wl.HEADS, wl.HEAD_DIM), dtype=torch.bfloat16, device=dev.q.device)
    lse = torch.empty((dev.B, n_query, wl.HEADS), dtype=torch.float32, device=dev.q.device)
    hint = dev.max_len_hint if hint is None else hint
    ws_bytes = capi.mfa_decode_mtp_workspace_bytes(dev.B, n_query, hint)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev.q.device)
    capi.mfa_workspace_init(ws, ws_bytes)
    capi.mfa_decode_attention_mtp(qd, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, out, lse, wl.SCALE,
                                  dev.B, n_query, dev.max_pages, dev.num_pages, hint, ws, ws_bytes)
    capi.mfa_check_device_errors(ws, clear=True)
    return out, lse


def oracle_mtp(oracle_mod, dev, q):
    kc, vc, _, _, sl = dev.host_caches()
    return oracle_mod.mfa_decode_mtp(wl.bits(q), kc, vc, dev.case.page_table, sl, wl.SCALE)


@pytest.mark.parametrize("grid", ["planned", "one_cta"])
def test_mtp_small_parity(oracle_mod, grid):
    lengths = [1, 2, 3, 63, 64, 65, 127, 128, 129, 130, 1000, 4097]
    case, q = mtp_case(lengths, seed=41)
    dev = DeviceCache(case)
    out, lse = run_mtp(dev, q, hint=0 if grid == "one_cta" else None)
    out_ref, lse_ref = oracle_mtp(oracle_mod, dev, q)
    compare(out, lse, out_ref, lse_ref, f"mtp/{grid}", bf16_storage_slack=True)
    assert torch.all(out[0, 0] == 0) and torch.all(torch.isneginf(lse[0, 0]))  # L = 1: token 0 sees nothing


def test_mtp_many_splits(oracle_mod):
    """Few long sequences over a full grid: many pieces per sequence and token."""
    case, q = mtp_case([3001, 6000, 129], seed=42)
    dev = DeviceCache(case)
    out_ref, lse_ref = oracle_mtp(oracle_mod, dev, q)
    for hint in (0, 256, 1 << 20):
        out, lse = run_mtp(dev, q, hint=hint)
        compare(out, lse, out_ref, lse_ref, f"mtp/hint={hint}")


def test_mtp_with_one_query_is_single_token_decode():
    case, q = mtp_case([700, 129, 64], seed=43, n_query=1)
    dev = DeviceCache(case)
    out, lse = run_mtp(dev, q, n_query=1)
    dev.q = q[:, 0].to(dev.q.device).contiguous()
    dev.attend()
    assert torch.equal(out[:, 0], dev.out) and torch.equal(lse[:, 0], dev.lse)


def test_mtp_after_appending_the_two_tokens(oracle_mod):
    """The serving order: append the step's two tokens, then attend with both."""
    lengths = [500, 63, 1]
    case, q = mtp_case(lengths, seed=44, headroom=T)
    dev = DeviceCache(case)
    k_new = wl.draw_rows(len(lengths) * T, wl.HEAD_DIM, [44, 1], 0).view(len(lengths), T, wl.HEAD_DIM)
    v_new = wl.draw_rows(len(lengths) * T, wl.HEAD_DIM, [44, 2], 0).view(len(lengths), T, wl.HEAD_DIM)
    dev.append(k_new, v_new)
    dev.check_errors()
    out, lse = run_mtp(dev, q, hint=int(max(lengths)) + T)
    out_ref, lse_ref = oracle_mtp(oracle_mod, dev, q)
    compare(out, lse, out_ref, lse_ref, "mtp/append", bf16_storage_slack=True)


def test_mtp_rejects_unsupported_query_counts():
    case, q = mtp_case([64], seed=45)
    dev = DeviceCache(case)
    for nq in (0, 3):
        with pytest.raises(capi.MFAError) as e:
            capi.mfa_decode_attention_mtp(dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, dev.out,
                                          dev.lse, wl.SCALE, dev.B, nq, dev.max_pages, dev.num_pages, 64,
                                          dev.workspace, dev.ws_bytes)
        assert e.value.status == 1


def test_mtp_4k_context_full_size(oracle_mod):
    """B = 32 sequences of 4096 tokens (the 4K-context shape), two query tokens each."""
    case, q = mtp_case([4096] * 32, seed=46)
    dev = DeviceCache(case)
    out, lse = run_mtp(dev, q)
    out_ref, lse_ref = oracle_mtp(oracle_mod, dev, q)
    compare(out, lse, out_ref, lse_ref, "mtp/4k")


def test_mtp_maximum_batch(oracle_mod):
    """MFA_MAX_BATCH sequences with two query tokens each: the largest shared-
    memory layout of the two-token kernel and a 2048-row combine grid; short
    ragged lengths, two of them 0 and two of them 1 (token 0 sees nothing)."""
    rng = np.random.default_rng(321)
    lengths = [int(x) for x in rng.integers(0, 200, size=capi.MAX_BATCH)]
    lengths[3] = lengths[500] = 0
    lengths[7] = lengths[900] = 1
    case, q = mtp_case(lengths, seed=47)
    dev = DeviceCache(case)
    out, lse = run_mtp(dev, q)
    out_ref, lse_ref = oracle_mtp(oracle_mod, dev, q)
    compare(out, lse, out_ref, lse_ref, "mtp/max-batch", bf16_storage_slack=True)
    assert torch.all(out[3] == 0) and torch.all(torch.isneginf(lse[3]))
    assert torch.all(out[7, 0] == 0) and torch.all(torch.isneginf(lse[7, 0])) and torch.all(torch.isfinite(lse[7, 1]))
