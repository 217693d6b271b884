"""The allocation-free decode entry point (mfa_decode_attention_noalloc).

It serves callers that cannot pass the library a workspace, such as a plugin
or foreign-function host that gives it only tensors it already owns, or a
running serving loop that must not call cudaMalloc. Its split results live in
the library's own fixed device array instead. The test calls it through the
C ABI twice in a row, on two different batches, and checks each output
against the regular entry point (which uses a caller workspace) and against
the fp64 oracle, within the tolerances of the other parity tests. A third call
passes no error word, so the word kept inside the fixed array (cleared by the
call itself) is the one in use. It also checks that a batch too large for the
fixed array is refused with MFA_ERR_WORKSPACE. This file is collected last so
that a stop-at-first-failure run has run everything else first.
"""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import LSE_ABS, MAX_ABS, REL_L2, DeviceCache, compare, oracle_caches

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _within_tolerance(out, lse, ref_out, ref_lse):
    o, r = out.double(), ref_out.double()
    max_abs = (o - r).abs().max().item()
    rel_l2 = ((o - r).norm() / r.norm()).item()
    finite = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), finite)
    dlse = (lse[finite] - ref_lse[finite]).abs().max().item()
    assert max_abs <= MAX_ABS and rel_l2 <= REL_L2 and dlse <= LSE_ABS, (max_abs, rel_l2, dlse)


def test_noalloc_matches_workspace_entry_point_on_two_calls(oracle_mod):
    cases = [([700, 1, 2049, 64], 61), ([4096] * 8, 62)]
    devs, refs, outs, oracle_refs = [], [], [], []
    for lengths, seed in cases:
        w = wl.Workload("noalloc", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
        case = wl.make_case(w, lengths=lengths)
        kc, vc, _, _, sl = oracle_caches(oracle_mod, case, "bf16")
        oracle_refs.append(oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, sl, wl.SCALE))
        dev = DeviceCache(case, "bf16")
        dev.attend()                                   # regular entry point, caller workspace
        dev.check_errors()
        refs.append((dev.out.clone(), dev.lse.clone()))
        outs.append((torch.full_like(dev.out, float("nan")), torch.full_like(dev.lse, float("nan"))))
        devs.append(dev)
    err_words = torch.zeros(len(cases), dtype=torch.int32, device="cuda")
    for i, dev in enumerate(devs):                      # two calls in a row, sharing the static scratch
        capi.mfa_decode_attention_noalloc(dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens,
                                          outs[i][0], outs[i][1], wl.SCALE, dev.B, dev.max_pages,
                                          dev.num_pages, dev.max_len_hint, err_words.data_ptr() + 4 * i)
    torch.cuda.synchronize()
    assert err_words.tolist() == [0, 0]
    for (out, lse), (ref_out, ref_lse), (o_out, o_lse) in zip(outs, refs, oracle_refs):
        _within_tolerance(out, lse, ref_out, ref_lse)
        compare(out, lse, o_out, o_lse, "noalloc vs oracle")
    # a third call without an error word: faults would go to the word inside the fixed array, which the call
    # clears first; the output must match as before
    dev = devs[0]
    out3, lse3 = torch.full_like(dev.out, float("nan")), torch.full_like(dev.lse, float("nan"))
    capi.mfa_decode_attention_noalloc(dev.q, dev.k_cache, dev.v_cache, dev.page_table, dev.seq_lens, out3, lse3,
                                      wl.SCALE, dev.B, dev.max_pages, dev.num_pages, dev.max_len_hint, None)
    torch.cuda.synchronize()
    _within_tolerance(out3, lse3, *refs[0])
    compare(out3, lse3, *oracle_refs[0], "noalloc (no error word) vs oracle")


def test_noalloc_refuses_a_batch_larger_than_its_scratch():
    plan = capi.mfa_plan_decode(1024, 1 << 16)
    assert plan.workspace_bytes > 24 << 20
    t = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_decode_attention_noalloc(t, t, t, t, t, t, t, wl.SCALE, 1024, 1, 1, 1 << 16)
    assert ei.value.status == 4  # MFA_ERR_WORKSPACE
    assert "scratch" in str(ei.value)
