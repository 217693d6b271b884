"""The low-rank query path on the GPU against the fp64 oracle.

Synthetic bf16 weights with the Step-3 shapes (7168 -> 2048 -> 64 x 256) and
a small shape; batch sizes that exercise the padding of the batch to 16 rows
and the 256-row maximum. The GPU rounds h to bf16 before the up-projection
and q to bf16 on output; the bounds are those of the attention outputs, with
the bf16 storage slack for |q| of a few units: max-abs 1e-2 + 2^-8 |ref|,
relative L2 5e-3."""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

STEP3 = (7168, 2048, 64 * 256)


def weights(d_model, rank, n_out, seed):
    g = torch.Generator().manual_seed(seed)
    w_down = (torch.randn(d_model, rank, generator=g) / d_model ** 0.5).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn(rank, generator=g)).to(torch.bfloat16)
    w_up = (torch.randn(rank, n_out, generator=g) / rank ** 0.5).to(torch.bfloat16)
    return w_down, gamma, w_up


def run_query(x, w_down, gamma, w_up, eps, ws=None, calls=1):
    B, d_model = x.shape
    rank, n_out = w_up.shape
    dev = torch.device("cuda")
    xd, wd, gd, wu = (t.to(dev).contiguous() for t in (x, w_down, gamma, w_up))
    q = torch.empty((B, n_out), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws_bytes = capi.mfa_query_lowrank_workspace_bytes(B, rank, n_out)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        capi.mfa_workspace_init(ws, ws_bytes)
    ws_bytes = ws.numel()  # the whole workspace: its layout follows from its size
    for _ in range(calls):
        capi.mfa_query_lowrank(xd, wd, gd, wu, q, B, d_model, rank, n_out, eps, ws, ws_bytes)
    capi.mfa_check_device_errors(ws, clear=True)
    return q


def check(q_gpu, q_ref, label):
    o = q_gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), label
    excess = np.abs(o - q_ref) - 2.0 ** -8 * np.abs(q_ref)
    assert float(np.max(excess)) <= 1e-2, f"{label}: max-abs excess {np.max(excess):.3e}"
    rel = float(np.linalg.norm(o - q_ref) / np.linalg.norm(q_ref))
    assert rel <= 5e-3, f"{label}: rel-L2 {rel:.3e}"
    return rel


@pytest.mark.parametrize("B", [1, 17, 32, 256])
def test_query_lowrank_step3_shape(oracle_mod, B):
    w_down, gamma, w_up = weights(*STEP3, seed=3)
    x = wl.draw_rows(B, STEP3[0], [71, B], 0)
    q = run_query(x, w_down, gamma, w_up, 1e-6)
    q_ref, _ = oracle_mod.query_lowrank(wl.bits(x), wl.bits(w_down), wl.bits(gamma), wl.bits(w_up), 1e-6)
    check(q, q_ref, f"step3/B={B}")


def test_query_lowrank_small_shape_and_eps(oracle_mod):
    w_down, gamma, w_up = weights(256, 128, 384, seed=4)
    x = wl.draw_rows(5, 256, [72], 0) * 0.01  # small rows: eps matters
    q = run_query(x, w_down, gamma, w_up, 1e-2)
    q_ref, _ = oracle_mod.query_lowrank(wl.bits(x), wl.bits(w_down), wl.bits(gamma), wl.bits(w_up), 1e-2)
    check(q, q_ref, "small")


def test_query_feeds_decode_attention(oracle_mod):
    """q from the query path, reshaped to [B][64][256], is a valid decode query."""
    w_down, gamma, w_up = weights(*STEP3, seed=5)
    x = wl.draw_rows(4, STEP3[0], [73], 0)
    q = run_query(x, w_down, gamma, w_up, 1e-6)
    assert q.view(4, 64, 256).is_contiguous()


def test_query_leaves_its_scratch_zero(oracle_mod):
    """The fp32 accumulator and the arrival counters are zero after every call,
    so single calls on one workspace (different inputs, different batch sizes,
    larger and smaller than before) each agree with the oracle."""
    w_down, gamma, w_up = weights(*STEP3, seed=7)
    _, rank, n_out = STEP3
    cap = capi.MAX_QUERY_BATCH
    ws_bytes = capi.mfa_query_lowrank_workspace_bytes(cap, rank, n_out)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)
    capi.mfa_workspace_init(ws, ws_bytes)
    # the regions that must be zero between calls: the header's counter bytes 128-255, then y [cap * rank] fp32
    zero_end = 256 + cap * rank * 4
    for i, B in enumerate((32, 7, 32, 256, 1)):
        x = wl.draw_rows(B, STEP3[0], [75, i], 0)
        q = run_query(x, w_down, gamma, w_up, 1e-6, ws=ws)  # one call: its result needs zero scratch on entry
        q_ref, _ = oracle_mod.query_lowrank(wl.bits(x), wl.bits(w_down), wl.bits(gamma), wl.bits(w_up), 1e-6)
        check(q, q_ref, f"repeat/B={B}")
        assert torch.count_nonzero(ws[128:zero_end]) == 0, f"B={B}: counters or accumulator not zero"


def test_query_rejects_bad_shapes():
    w_down, gamma, w_up = weights(256, 128, 384, seed=6)
    x = wl.draw_rows(2, 256, [74], 0).cuda()
    q = torch.empty((2, 384), dtype=torch.bfloat16, device="cuda")
    ws_bytes = capi.mfa_query_lowrank_workspace_bytes(2, 128, 384)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for args in ((2, 250, 128, 384), (2, 256, 100, 384), (2, 256, 128, 300), (0, 256, 128, 384), (300, 256, 128, 384),
                 (2, 256, capi.MAX_QUERY_RANK + 128, 384)):
        with pytest.raises(capi.MFAError) as e:
            capi.mfa_query_lowrank(x, w_down.cuda(), gamma.cuda(), w_up.cuda(), q, *args, 1e-6, ws, ws_bytes)
        assert e.value.status == 1
