"""Block-gather decode on the GPU against the fp64 oracle.

The query attends to the caller's selected historical 8-token blocks and to
its own block up to its last token ("Step-5-Preview" page, sparse attention;
MFA's shared K/V head). Small cases put the selection and the last block on
every tile position that matters, on the planned grid and on one CTA;
selecting every block must give the dense kernel's output bit for bit; the
Step-5 budget (512 blocks = 4096 tokens + the current block) runs on long
sequences; malformed selections raise the device error word. The E4M3 cache
(codes and per-token scales gathered by block) runs the same cases against the
oracle on its own quantised copy of the cache. Tolerances as for single-token
decode."""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import DeviceCache, compare, oracle_caches

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def block_case(lengths, seed):
    w = wl.Workload("blocks", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
    return wl.make_case(w, lengths=lengths, spare_pages=1)


def run_blocks(dev, block_idx, n_blocks, hint=None):
    bi = torch.from_numpy(np.ascontiguousarray(block_idx, dtype=np.int32)).to(dev.q.device)
    nb = torch.from_numpy(np.ascontiguousarray(n_blocks, dtype=np.int32)).to(dev.q.device)
    if hint is None:
        hint = int(8 * np.max(n_blocks) + 8) if len(n_blocks) else 0
    ws_bytes = capi.mfa_decode_workspace_bytes(dev.B, hint)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev.q.device)
    capi.mfa_workspace_init(ws, ws_bytes)
    out = torch.empty_like(dev.out)
    lse = torch.empty_like(dev.lse)
    capi.mfa_decode_attention_blocks(dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, bi, nb,
                                     bi.shape[1], out, lse, wl.SCALE, dev.B, dev.max_pages, dev.num_pages, hint, ws,
                                     ws_bytes)
    return out, lse, ws


def oracle_blocks(oracle_mod, dev, block_idx, n_blocks):
    kc, vc, _, _, sl = dev.host_caches()
    return oracle_mod.mfa_decode_blocks(wl.bits(dev.case.q), kc, vc, dev.case.page_table, sl, block_idx, n_blocks,
                                        wl.SCALE)


@pytest.mark.parametrize("grid", ["planned", "one_cta"])
def test_blocks_small_parity(oracle_mod, grid):
    lengths = [0, 1, 8, 9, 16, 17, 63, 64, 65, 129, 200, 1000, 4097]
    case = block_case(lengths, seed=51)
    dev = DeviceCache(case)
    bi, nb = wl.draw_blocks(lengths, 40, [51])
    out, lse, ws = run_blocks(dev, bi, nb, hint=0 if grid == "one_cta" else None)
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks(oracle_mod, dev, bi, nb)
    compare(out, lse, out_ref, lse_ref, f"blocks/{grid}", bf16_storage_slack=True)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_blocks_ragged_counts_and_positions(oracle_mod):
    """Selections of every size up to a few tiles, in random order, some blocks in the last page."""
    rng = np.random.default_rng(52)
    lengths = [int(x) for x in rng.integers(100, 3000, size=24)]
    case = block_case(lengths, seed=52)
    dev = DeviceCache(case)
    bi = np.full((24, 64), -1, dtype=np.int32)
    nb = np.zeros(24, dtype=np.int32)
    for b, L in enumerate(lengths):
        hist = (L - 1) // 8
        k = min(hist, int(rng.integers(0, 64)))
        sel = rng.choice(hist, size=k, replace=False)
        if k and hist - 1 not in sel:
            sel[0] = hist - 1  # the block just before the current one
        bi[b, :k] = sel
        nb[b] = k
    out, lse, ws = run_blocks(dev, bi, nb)
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks(oracle_mod, dev, bi, nb)
    compare(out, lse, out_ref, lse_ref, "blocks/ragged", bf16_storage_slack=True)


def test_every_block_is_the_dense_kernel():
    lengths = [1, 8, 65, 700, 4096, 5001]
    case = block_case(lengths, seed=53)
    dev = DeviceCache(case)
    hist = [(L - 1) // 8 for L in lengths]
    bi = np.full((len(lengths), max(hist)), -1, dtype=np.int32)
    for b, n in enumerate(hist):
        bi[b, :n] = np.arange(n)
    hint = max(lengths)
    out, lse, ws = run_blocks(dev, bi, np.array(hist, np.int32), hint=hint)
    capi.mfa_check_device_errors(ws, clear=True)
    dev.attend(max_len_hint=hint)
    dev.check_errors()
    assert torch.equal(out, dev.out) and torch.equal(lse, dev.lse)


def test_step5_budget_on_long_sequences(oracle_mod):
    """512 selected blocks (4096 tokens) plus the current block of 16K-32K-token sequences."""
    lengths = [16384, 32768, 20001, 30000]
    case = block_case(lengths, seed=54)
    dev = DeviceCache(case)
    bi, nb = wl.draw_blocks(lengths, 512, [54])
    out, lse, ws = run_blocks(dev, bi, nb)
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks(oracle_mod, dev, bi, nb)
    compare(out, lse, out_ref, lse_ref, "blocks/step5")


def test_blocks_maximum_batch(oracle_mod):
    rng = np.random.default_rng(55)
    lengths = [int(x) for x in rng.integers(0, 300, size=capi.MAX_BATCH)]
    case = block_case(lengths, seed=55)
    dev = DeviceCache(case)
    bi, nb = wl.draw_blocks(lengths, 12, [55])
    out, lse, ws = run_blocks(dev, bi, nb)
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks(oracle_mod, dev, bi, nb)
    compare(out, lse, out_ref, lse_ref, "blocks/max-batch", bf16_storage_slack=True)


def test_bad_selection_sets_the_error_word():
    lengths = [100, 100]  # historical blocks 0..11; block 12 holds the last token
    case = block_case(lengths, seed=56)
    dev = DeviceCache(case)
    for bad, code in ((np.array([[3, 12], [0, 1]], np.int32), 5),
                      (np.array([[3, -1], [0, 1]], np.int32), 5)):
        _, _, ws = run_blocks(dev, bad, np.array([2, 2], np.int32))
        with pytest.raises(capi.MFAError) as e:
            capi.mfa_check_device_errors(ws, clear=True)
        assert e.value.status == code
    _, _, ws = run_blocks(dev, np.zeros((2, 16), np.int32), np.array([13, 2], np.int32), hint=200)
    with pytest.raises(capi.MFAError) as e:
        capi.mfa_check_device_errors(ws, clear=True)
    assert e.value.status == 6


def test_blocks_host_argument_checks():
    case = block_case([64], seed=57)
    dev = DeviceCache(case)
    bi = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    nb = torch.zeros(1, dtype=torch.int32, device="cuda")
    for args in ((None, nb, 4), (bi, None, 4), (bi, nb, 0), (bi, nb, 8 * dev.max_pages + 1)):
        with pytest.raises(capi.MFAError) as e:
            capi.mfa_decode_attention_blocks(dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens,
                                             *args, dev.out, dev.lse, wl.SCALE, 1, dev.max_pages, dev.num_pages, 64,
                                             dev.workspace, dev.ws_bytes)
        assert e.value.status == 1


def test_blocks32k_workload_full_size(oracle_mod):
    """The benchmark's block-gather workload as the benchmark launches it: B=32 sequences of 32768
    tokens, 512 selected blocks each (4104 tokens attended), every output against the oracle."""
    w = wl.WORKLOADS["blocks32k"]
    case = wl.make_case(w, headroom_tokens=0)
    dev = DeviceCache(case)
    bi, nb = wl.draw_blocks(case.lengths0, w.select_blocks, [w.seed])
    out, lse, ws = run_blocks(dev, bi, nb)   # length hint = the largest attended count, as in bench.py
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks(oracle_mod, dev, bi, nb)
    compare(out, lse, out_ref, lse_ref, "blocks32k")


def run_blocks_fp8(dev, block_idx, n_blocks, hint=None):
    bi = torch.from_numpy(np.ascontiguousarray(block_idx, dtype=np.int32)).to(dev.q.device)
    nb = torch.from_numpy(np.ascontiguousarray(n_blocks, dtype=np.int32)).to(dev.q.device)
    if hint is None:
        hint = int(8 * np.max(n_blocks) + 8) if len(n_blocks) else 0
    ws_bytes = capi.mfa_decode_workspace_bytes(dev.B, hint)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev.q.device)
    capi.mfa_workspace_init(ws, ws_bytes)
    out = torch.empty_like(dev.out)
    lse = torch.empty_like(dev.lse)
    capi.mfa_decode_attention_blocks_fp8(dev.q, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale, dev.page_table,
                                         dev.seq_lens, bi, nb, bi.shape[1], out, lse, wl.SCALE, dev.B, dev.max_pages,
                                         dev.num_pages, hint, ws, ws_bytes)
    return out, lse, ws


def oracle_blocks_fp8(oracle_mod, case, block_idx, n_blocks):
    """The oracle on its own E4M3 copy of the cache (its quantiser; unused slots poisoned)."""
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, "fp8")
    return oracle_mod.mfa_decode_blocks(wl.bits(case.q), kc, vc, case.page_table, sl, block_idx, n_blocks, wl.SCALE,
                                        k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("grid", ["planned", "one_cta"])
def test_blocks_fp8_small_parity(oracle_mod, grid):
    lengths = [0, 1, 8, 9, 16, 17, 63, 64, 65, 129, 200, 1000, 4097]
    case = block_case(lengths, seed=61)
    dev = DeviceCache(case, "fp8")  # NaN-poisoned codes and scales, filled by the device append
    bi, nb = wl.draw_blocks(lengths, 40, [61])
    out, lse, ws = run_blocks_fp8(dev, bi, nb, hint=0 if grid == "one_cta" else None)
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks_fp8(oracle_mod, case, bi, nb)
    compare(out, lse, out_ref, lse_ref, f"blocks-fp8/{grid}", bf16_storage_slack=True)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_blocks_fp8_every_block_is_the_dense_kernel():
    lengths = [1, 8, 65, 700, 4096, 5001]
    case = block_case(lengths, seed=62)
    dev = DeviceCache(case, "fp8")
    hist = [(L - 1) // 8 for L in lengths]
    bi = np.full((len(lengths), max(hist)), -1, dtype=np.int32)
    for b, n in enumerate(hist):
        bi[b, :n] = np.arange(n)
    hint = max(lengths)
    out, lse, ws = run_blocks_fp8(dev, bi, np.array(hist, np.int32), hint=hint)
    capi.mfa_check_device_errors(ws, clear=True)
    dev.attend(max_len_hint=hint)
    dev.check_errors()
    assert torch.equal(out, dev.out) and torch.equal(lse, dev.lse)


def test_blocks_fp8_step5_budget_on_long_sequences(oracle_mod):
    """512 selected blocks (4096 tokens) plus the current block of 16K-32K-token sequences, E4M3 cache."""
    lengths = [16384, 32768, 20001, 30000]
    case = block_case(lengths, seed=63)
    dev = DeviceCache(case, "fp8")
    bi, nb = wl.draw_blocks(lengths, 512, [63])
    out, lse, ws = run_blocks_fp8(dev, bi, nb)
    capi.mfa_check_device_errors(ws, clear=True)
    out_ref, lse_ref = oracle_blocks_fp8(oracle_mod, case, bi, nb)
    compare(out, lse, out_ref, lse_ref, "blocks-fp8/step5")
