"""Multi-token (MTP) decode on the GPU against the fp64 oracle.

T query tokens per sequence; token t attends causally to positions
j < L - T + 1 + t. On the bf16 cache a CTA serves two tokens (one pass over
the cache for both); the quantised caches serve one token a CTA; with more
tokens than a CTA serves, the tokens form groups whose CTAs stream the same
pages together. Small cases put the causal boundary on every tile position
that matters (a token that sees nothing, the last row of a page or of a tile,
a one-row last tile), on the planned grid and on one range; the 4K-context
shape runs at full size. The oracle always reads its own host copy of the
cache (its own quantiser and append). Tolerances as for single-token decode."""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import DeviceCache, compare, oracle_caches

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SMALL_LENGTHS = [1, 2, 3, 4, 5, 63, 64, 65, 127, 128, 129, 130, 1000, 4097]


def mtp_case(lengths, seed, n_query, headroom=0):
    w = wl.Workload("mtp", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
    case = wl.make_case(w, lengths=lengths, spare_pages=1, headroom_tokens=headroom)
    q = wl.draw_rows(len(lengths) * n_query * wl.HEADS, wl.HEAD_DIM, [seed, 90], 0)
    return case, q.view(len(lengths), n_query, wl.HEADS, wl.HEAD_DIM)


def run_mtp(dev, q, n_query, hint=None):
    qd = q.to(dev.q.device).contiguous()
    out = torch.empty((dev.B, n_query, wl.HEADS, wl.HEAD_DIM), dtype=torch.bfloat16, device=dev.q.device)
    lse = torch.empty((dev.B, n_query, wl.HEADS), dtype=torch.float32, device=dev.q.device)
    hint = dev.max_len_hint if hint is None else hint
    ws_bytes = capi.mfa_decode_mtp_workspace_bytes(dev.B, n_query, hint)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev.q.device)
    capi.mfa_workspace_init(ws, ws_bytes)
    if dev.kv_dtype == "bf16":
        capi.mfa_decode_attention_mtp(qd, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, out, lse,
                                      wl.SCALE, dev.B, n_query, dev.max_pages, dev.num_pages, hint, ws, ws_bytes)
    else:
        fn = capi.mfa_decode_attention_mtp_fp8 if dev.kv_dtype == "fp8" else capi.mfa_decode_attention_mtp_fp4
        fn(qd, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.page_table, dev.seq_lens, out, lse,
           wl.SCALE, dev.B, n_query, dev.max_pages, dev.num_pages, hint, ws, ws_bytes)
    capi.mfa_check_device_errors(ws, clear=True)
    return out, lse


def oracle_mtp(oracle_mod, case, q, kv="bf16", k_new=None, v_new=None):
    """The oracle on its own host copy of the cache (after its own append of k_new/v_new, if given)."""
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, kv)
    if k_new is not None:
        oracle_mod.kv_append(wl.bits(k_new), wl.bits(v_new), kc, vc, case.page_table, sl, k_scale=ks, v_scale=vs)
    return oracle_mod.mfa_decode_mtp(wl.bits(q), kc, vc, case.page_table, sl, wl.SCALE, k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("grid", ["planned", "one_range"])
@pytest.mark.parametrize("n_query", [2, 3, 4])
def test_mtp_small_parity(oracle_mod, n_query, grid):
    case, q = mtp_case(SMALL_LENGTHS, seed=41 + n_query, n_query=n_query)
    dev = DeviceCache(case)
    out, lse = run_mtp(dev, q, n_query, hint=0 if grid == "one_range" else None)
    out_ref, lse_ref = oracle_mtp(oracle_mod, case, q)
    compare(out, lse, out_ref, lse_ref, f"mtp{n_query}/{grid}", bf16_storage_slack=True)
    # L = 1: only the last token sees a position; L = 2 with T >= 3: token 0 sees nothing
    assert torch.all(out[0, :-1] == 0) and torch.all(torch.isneginf(lse[0, :-1]))
    assert torch.all(torch.isfinite(lse[0, -1]))


@pytest.mark.parametrize("n_query", [2, 3])
@pytest.mark.parametrize("kv", ["fp8", "fp4"])
def test_mtp_quantised_small_parity(oracle_mod, kv, n_query):
    """E4M3 and packed E2M1 caches: one token a CTA, n_query CTAs per range,
    against the oracle on the dequantised cache."""
    case, q = mtp_case(SMALL_LENGTHS, seed=51 + n_query, n_query=n_query)
    dev = DeviceCache(case, kv)
    out, lse = run_mtp(dev, q, n_query)
    out_ref, lse_ref = oracle_mtp(oracle_mod, case, q, kv)
    compare(out, lse, out_ref, lse_ref, f"mtp{n_query}/{kv}", bf16_storage_slack=True)


@pytest.mark.parametrize("n_query", [2, 3, 4, 8])
def test_mtp_many_splits(oracle_mod, n_query):
    """Few long sequences over a full grid: many pieces per sequence and token."""
    case, q = mtp_case([3001, 6000, 129], seed=42, n_query=n_query)
    dev = DeviceCache(case)
    out_ref, lse_ref = oracle_mtp(oracle_mod, case, q)
    for hint in (0, 256, 1 << 20):
        out, lse = run_mtp(dev, q, n_query, hint=hint)
        compare(out, lse, out_ref, lse_ref, f"mtp{n_query}/hint={hint}")


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp4"])
def test_mtp_with_one_query_is_single_token_decode(kv):
    case, q = mtp_case([700, 129, 64], seed=43, n_query=1)
    dev = DeviceCache(case, kv)
    out, lse = run_mtp(dev, q, 1)
    dev.q = q[:, 0].to(dev.q.device).contiguous()
    dev.attend()
    assert torch.equal(out[:, 0], dev.out) and torch.equal(lse[:, 0], dev.lse)


@pytest.mark.parametrize("n_query", [2, 3])
def test_mtp_after_appending_the_tokens(oracle_mod, n_query):
    """The serving order: append the step's tokens, then attend with all of them."""
    lengths = [500, 63, 1]
    case, q = mtp_case(lengths, seed=44, n_query=n_query, headroom=n_query)
    dev = DeviceCache(case)
    k_new = wl.draw_rows(len(lengths) * n_query, wl.HEAD_DIM, [44, 1], 0).view(len(lengths), n_query, wl.HEAD_DIM)
    v_new = wl.draw_rows(len(lengths) * n_query, wl.HEAD_DIM, [44, 2], 0).view(len(lengths), n_query, wl.HEAD_DIM)
    dev.append(k_new, v_new)
    dev.check_errors()
    out, lse = run_mtp(dev, q, n_query, hint=int(max(lengths)) + n_query)
    out_ref, lse_ref = oracle_mtp(oracle_mod, case, q, k_new=k_new, v_new=v_new)
    compare(out, lse, out_ref, lse_ref, f"mtp{n_query}/append", bf16_storage_slack=True)


def test_mtp_rejects_unsupported_query_counts():
    case, q = mtp_case([64], seed=45, n_query=2)
    dev = DeviceCache(case)
    for nq in (0, capi.MAX_QUERY_TOKENS + 1):
        with pytest.raises(capi.MFAError) as e:
            capi.mfa_decode_attention_mtp(dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, dev.out,
                                          dev.lse, wl.SCALE, dev.B, nq, dev.max_pages, dev.num_pages, 64,
                                          dev.workspace, dev.ws_bytes)
        assert e.value.status == 1


@pytest.mark.parametrize("kv,n_query", [("bf16", 2), ("bf16", 3), ("bf16", 4), ("fp8", 2)])
def test_mtp_4k_context_full_size(oracle_mod, kv, n_query):
    """B = 32 sequences of 4096 tokens (the 4K-context shape), n_query query tokens each."""
    case, q = mtp_case([4096] * 32, seed=46, n_query=n_query)
    dev = DeviceCache(case, kv)
    out, lse = run_mtp(dev, q, n_query)
    out_ref, lse_ref = oracle_mtp(oracle_mod, case, q, kv)
    compare(out, lse, out_ref, lse_ref, f"mtp{n_query}/{kv}/4k")


@pytest.mark.parametrize("n_query", [2, 3])
def test_mtp_maximum_batch(oracle_mod, n_query):
    """MFA_MAX_BATCH sequences with n_query query tokens each: the largest shared-
    memory layout and the largest combine grid; short ragged lengths, two of
    them 0 and two of them 1 (only the last token sees a position)."""
    rng = np.random.default_rng(321)
    lengths = [int(x) for x in rng.integers(0, 200, size=capi.MAX_BATCH)]
    lengths[3] = lengths[500] = 0
    lengths[7] = lengths[900] = 1
    case, q = mtp_case(lengths, seed=47, n_query=n_query)
    dev = DeviceCache(case)
    out, lse = run_mtp(dev, q, n_query)
    out_ref, lse_ref = oracle_mtp(oracle_mod, case, q)
    compare(out, lse, out_ref, lse_ref, f"mtp{n_query}/max-batch", bf16_storage_slack=True)
    assert torch.all(out[3] == 0) and torch.all(torch.isneginf(lse[3]))
    assert torch.all(out[7, :-1] == 0) and torch.all(torch.isneginf(lse[7, :-1]))
    assert torch.all(torch.isfinite(lse[7, -1]))
