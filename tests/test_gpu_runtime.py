"""Runtime behaviour on the GPU: CUDA-graph capture and replay of a decode step
(the replay must see the advancing device-owned length, the state-hygiene
lesson of the "DuckLLM decode fixed-cost reduction" page, section 7.5), and
the bounded pipeline wait giving up with an error status instead of hanging."""
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import DeviceCache, compare, oracle_caches

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_graph_replay_matches_eager(oracle_mod, kv):
    lengths = [130, 64, 999]
    steps = 4
    w = wl.Workload("graph", 3, ("list", tuple(lengths)), kv, True, 1, 21)
    case = wl.make_case(w, lengths=lengths, headroom_tokens=steps)
    dev = DeviceCache(case, kv)
    eager = DeviceCache(case, kv)
    new_k = wl.draw_rows(3 * steps, wl.HEAD_DIM, [21], 8).view(steps, 3, 1, -1)
    new_v = wl.draw_rows(3 * steps, wl.HEAD_DIM, [21], 9).view(steps, 3, 1, -1)
    new_q = wl.draw_rows(steps * 3 * wl.HEADS, wl.HEAD_DIM, [21], 10).view(steps, 3, wl.HEADS, -1)
    k_buf = torch.empty((3, 1, wl.HEAD_DIM), dtype=torch.bfloat16, device="cuda")
    v_buf = torch.empty_like(k_buf)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    dev.attend()  # first call outside capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        dev.append(k_buf, v_buf)
        dev.attend()
    torch.cuda.synchronize()
    assert dev.seq_lens.cpu().tolist() == lengths  # capture does not execute
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, kv)
    for t in range(steps):
        k_buf.copy_(new_k[t]); v_buf.copy_(new_v[t]); dev.q.copy_(new_q[t])
        graph.replay()
        eager.q.copy_(new_q[t])
        eager.append(new_k[t], new_v[t])
        eager.attend()
        torch.cuda.synchronize()
        assert dev.seq_lens.cpu().tolist() == [n + t + 1 for n in lengths]
        assert torch.equal(dev.out, eager.out) and torch.equal(dev.lse, eager.lse)
        oracle_mod.kv_append(wl.bits(new_k[t]), wl.bits(new_v[t]), kc, vc, case.page_table, sl,
                             k_scale=ks, v_scale=vs)
    dev.check_errors()
    out_ref, lse_ref = oracle_mod.mfa_decode(wl.bits(new_q[steps - 1]), kc, vc, case.page_table, sl, wl.SCALE,
                                             k_scale=ks, v_scale=vs)
    compare(dev.out, dev.lse, out_ref, lse_ref, f"graph/{kv}")


def test_bounded_wait_gives_up_and_context_survives(oracle_mod):
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    capi.mfa_workspace_init(ws, ws.numel())
    capi.mfa_selftest_wait_timeout(ws, 50_000_000)  # 50 ms budget on a barrier nobody arrives on
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_check_device_errors(ws, clear=True)
    assert ei.value.status == 7  # MFA_ERR_DEVICE_TIMEOUT
    capi.mfa_check_device_errors(ws, clear=True)  # cleared
    case = wl.make_case(wl.WORKLOADS["tiny"])
    dev = DeviceCache(case, "bf16")
    dev.attend()
    dev.check_errors()
    kc, vc, _, _, sl = oracle_caches(oracle_mod, case, "bf16")
    out_ref, lse_ref = oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, sl, wl.SCALE)
    compare(dev.out, dev.lse, out_ref, lse_ref, "after-timeout")
