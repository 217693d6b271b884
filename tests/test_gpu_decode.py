"""MFA decode attention on the GPU against the fp64 oracle.

Small cases span several 128-token tiles, ragged tails, one-token and empty
sequences and many-split layouts, compared element by element; the five
named workloads run at full size in the launch configuration the benchmark
times, also compared on every output. Tolerances: max-abs 1e-2, relative L2
5e-3, |dLSE| 1e-3."""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import DeviceCache, compare, oracle_caches

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SMALL = {
    "one_token": [1],
    "one_page": [64],
    "page_plus_one": [65],
    "tile_edges": [127, 128, 129],
    "mixed": [1000, 1, 300, 64],
    "single_long": [5000],
    "many_short": None,  # drawn below
}


def _case(lengths, seed, kv="bf16", permute=True):
    w = wl.Workload("parity", len(lengths), ("list", tuple(lengths)), kv, permute, 0, seed)
    return wl.make_case(w, lengths=lengths, spare_pages=1)


def _lengths(name):
    if name == "many_short":
        return [int(x) for x in np.random.default_rng(77).integers(1, 600, size=37)]
    return SMALL[name]


def _oracle(oracle_mod, case, kv):
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, kv)
    return oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, sl, wl.SCALE, k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("grid", ["planned", "one_cta"])
@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp4"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_parity(oracle_mod, kv, name, grid):
    """`planned` uses the grid the planner picks (few tiles per CTA); `one_cta`
    (length hint 0) makes one CTA walk every tile of every sequence."""
    lengths = _lengths(name)
    case = _case(lengths, seed=1 + list(SMALL).index(name), kv=kv)
    dev = DeviceCache(case, kv)
    dev.attend(max_len_hint=0 if grid == "one_cta" else None)
    dev.check_errors()
    out_ref, lse_ref = _oracle(oracle_mod, case, kv)
    compare(dev.out, dev.lse, out_ref, lse_ref, f"{kv}/{name}/{grid}")


def test_empty_sequences(oracle_mod):
    case = _case([0, 70, 0], seed=5)
    dev = DeviceCache(case, "bf16")
    dev.attend()
    dev.check_errors()
    assert torch.all(dev.out[0] == 0) and torch.all(dev.out[2] == 0)
    assert torch.all(torch.isneginf(dev.lse[0])) and torch.all(torch.isneginf(dev.lse[2]))
    out_ref, lse_ref = _oracle(oracle_mod, case, "bf16")
    compare(dev.out, dev.lse, out_ref, lse_ref, "empty")


def test_single_token_returns_v_exactly():
    case = _case([1, 1], seed=6)
    dev = DeviceCache(case, "bf16")
    dev.attend()
    v = case.v_rows.cuda()
    assert torch.equal(dev.out[0], v[0].expand(wl.HEADS, -1))
    assert torch.equal(dev.out[1], v[1].expand(wl.HEADS, -1))


def test_constant_keys_give_mean_of_v():
    case = _case([300, 1000], seed=7)
    case.k_rows[:300] = case.k_rows[0]
    case.k_rows[300:] = case.k_rows[300]
    dev = DeviceCache(case, "bf16")
    dev.attend()
    mean0 = case.v_rows[:300].double().mean(0)
    mean1 = case.v_rows[300:].double().mean(0)
    assert torch.allclose(dev.out[0].double().cpu(), mean0.expand(wl.HEADS, -1), atol=2e-3, rtol=0)
    assert torch.allclose(dev.out[1].double().cpu(), mean1.expand(wl.HEADS, -1), atol=2e-3, rtol=0)


def test_page_placement_is_bitwise_invariant():
    lengths = [700, 129, 1500]
    a = _case(lengths, seed=8, permute=False)
    b = _case(lengths, seed=8, permute=True)
    da, db = DeviceCache(a, "bf16"), DeviceCache(b, "bf16")
    da.attend()
    db.attend()
    assert torch.equal(da.out, db.out) and torch.equal(da.lse, db.lse)


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp4"])
def test_split_count_invariance(oracle_mod, kv):
    """Different grid sizes (one CTA, a few, one per SM) all match the oracle."""
    case = _case([3000, 17, 900], seed=9, kv=kv)
    dev = DeviceCache(case, kv)
    out_ref, lse_ref = _oracle(oracle_mod, case, kv)
    for hint in (0, 128, 1024, 1 << 20):
        dev.attend(max_len_hint=hint)
        dev.check_errors()
        compare(dev.out, dev.lse, out_ref, lse_ref, f"{kv}/hint={hint}")


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp4"])
def test_query_heads_of_very_different_norms(oracle_mod, kv):
    """Head h of Q scaled by 2^-(h % 13) (a 4096x spread), four heads by 8
    (peaked softmax): the E4M3 path splits Q into E4M3 terms under one
    power-of-two scale per piece, so small heads sit far below the largest."""
    case = _case([700, 129, 2000], seed=31, kv=kv)
    mult = torch.tensor([2.0 ** -(h % 13) for h in range(wl.HEADS)], dtype=torch.float32)
    mult[[3, 17, 40, 63]] = 8.0
    case.q.copy_((case.q.float() * mult[None, :, None]).to(torch.bfloat16))
    dev = DeviceCache(case, kv)
    dev.attend()
    dev.check_errors()
    out_ref, lse_ref = _oracle(oracle_mod, case, kv)
    compare(dev.out, dev.lse, out_ref, lse_ref, f"{kv}/head-norm spread")


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp4"])
def test_maximum_batch(oracle_mod, kv):
    """The largest batch the ABI accepts (MFA_MAX_BATCH sequences): the largest
    shared-memory layout of the split kernel and the widest combine grid.
    Short ragged lengths (two start empty), one appended token per sequence."""
    rng = np.random.default_rng(123)
    lengths = [int(x) for x in rng.integers(0, 260, size=capi.MAX_BATCH)]
    lengths[5] = lengths[700] = 0
    w = wl.Workload("max_batch", len(lengths), ("list", tuple(lengths)), kv, True, 1, 13)
    case = wl.make_case(w, lengths=lengths)
    dev = DeviceCache(case, kv)
    k_new = wl.draw_rows(len(lengths), wl.HEAD_DIM, [13, 1], 21).view(len(lengths), 1, wl.HEAD_DIM)
    v_new = wl.draw_rows(len(lengths), wl.HEAD_DIM, [13, 2], 22).view(len(lengths), 1, wl.HEAD_DIM)
    dev.append(k_new, v_new)
    dev.attend()
    dev.check_errors()
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, kv)
    oracle_mod.kv_append(wl.bits(k_new), wl.bits(v_new), kc, vc, case.page_table, sl, k_scale=ks, v_scale=vs)
    assert np.array_equal(dev.seq_lens.cpu().numpy(), sl)
    out_ref, lse_ref = oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, sl, wl.SCALE,
                                             k_scale=ks, v_scale=vs)
    compare(dev.out, dev.lse, out_ref, lse_ref, f"{kv}/B={len(lengths)}", bf16_storage_slack=True)


def test_bad_page_and_capacity_set_error_word():
    case = _case([200, 50], seed=10)
    dev = DeviceCache(case, "bf16")
    pt = dev.page_table.clone()
    dev.page_table[1, 0] = -3
    dev.attend()
    with pytest.raises(capi.MFAError) as ei:
        dev.check_errors()
    assert ei.value.status == 5
    dev.page_table.copy_(pt)
    dev.seq_lens[0] = dev.max_pages * wl.PAGE_SIZE + 1
    dev.attend()
    with pytest.raises(capi.MFAError) as ei:
        dev.check_errors()
    assert ei.value.status == 6


def test_decode_rejects_bad_arguments():
    case = _case([10], seed=11)
    dev = DeviceCache(case, "bf16")
    args = [dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, dev.out, dev.lse, wl.SCALE, 1,
            dev.max_pages, dev.num_pages, 10, dev.workspace, dev.ws_bytes]
    bad_ws = list(args); bad_ws[13] = 16
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_decode_attention(*bad_ws)
    assert ei.value.status == 4
    no_out = list(args); no_out[5] = None
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_decode_attention(*no_out)
    assert ei.value.status == 1
    big_b = list(args); big_b[8] = 2000
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_decode_attention(*big_b)
    assert ei.value.status == 1


@pytest.mark.parametrize("name", ["tiny", "ctx4k", "ragged", "fp8", "fp4", "long"])
def test_named_workload_full_size(oracle_mod, name):
    """Every output of each named workload, as the benchmark launches it."""
    w = wl.WORKLOADS[name]
    case = wl.make_case(w)
    dev = DeviceCache(case, w.kv_dtype)
    if case.k_new is not None:
        dev.append(case.k_new, case.v_new)
    dev.attend()
    dev.check_errors()
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, w.kv_dtype)
    if case.k_new is not None:
        oracle_mod.kv_append(wl.bits(case.k_new), wl.bits(case.v_new), kc, vc, case.page_table, sl,
                             k_scale=ks, v_scale=vs)
    assert np.array_equal(dev.seq_lens.cpu().numpy(), sl)
    out_ref, lse_ref = oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, sl, wl.SCALE,
                                             k_scale=ks, v_scale=vs)
    err = compare(dev.out, dev.lse, out_ref, lse_ref, name)
    print(f"{name}: {err}")
