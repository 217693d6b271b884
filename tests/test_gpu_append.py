"""KV append on the GPU: bit-exact against the oracle's append (bf16 copy and
per-token E4M3 quantisation), counter advance, capacity and page faults."""
import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import capi
from decode_attention_mfa_gb300 import workloads as wl
from gpu_util import POISON, DeviceCache, oracle_caches, used_slots_equal

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _case(lengths, seed, headroom, kv="bf16"):
    w = wl.Workload("append", len(lengths), ("list", tuple(lengths)), kv, True, 0, seed)
    return wl.make_case(w, lengths=lengths, headroom_tokens=headroom, spare_pages=2)


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp4"])
@pytest.mark.parametrize("n_new", [1, 70])
def test_append_bit_exact(oracle_mod, kv, n_new):
    lengths = [0, 1, 63, 64, 200]
    case = _case(lengths, seed=100 + n_new, headroom=n_new, kv=kv)
    dev = DeviceCache(case, kv)
    kn = wl.draw_rows(len(lengths) * n_new, wl.HEAD_DIM, [7, n_new], 4).view(len(lengths), n_new, -1)
    vn = wl.draw_rows(len(lengths) * n_new, wl.HEAD_DIM, [7, n_new], 5).view(len(lengths), n_new, -1)
    dev.append(kn, vn)
    dev.check_errors()
    kc, vc, ks, vs, sl = oracle_caches(oracle_mod, case, kv)
    oracle_mod.kv_append(wl.bits(kn), wl.bits(vn), kc, vc, case.page_table, sl, k_scale=ks, v_scale=vs)
    gk, gv, gks, gvs, gsl = dev.host_caches()
    assert np.array_equal(gsl, sl)
    assert np.array_equal(gsl, np.asarray(lengths) + n_new)
    assert used_slots_equal(gk, kc, sl, case.page_table)
    assert used_slots_equal(gv, vc, sl, case.page_table)
    if kv != "bf16":
        assert used_slots_equal(gks[..., None], ks[..., None], sl, case.page_table)
        assert used_slots_equal(gvs[..., None], vs[..., None], sl, case.page_table)
    # slots past the new lengths are untouched (still poisoned)
    all_slots = np.arange(case.num_pages * wl.PAGE_SIZE)
    unused = np.setdiff1d(all_slots, wl.slots_of(sl, case.page_table))
    flat = gk.reshape(case.num_pages * wl.PAGE_SIZE, -1)[unused]
    if kv == "bf16":
        assert np.all((flat & 0x7FFF) > 0x7F80)  # NaN bit patterns
    else:
        assert np.all(flat == POISON[kv])


def test_fp8_quantiser_special_rows(oracle_mod):
    """All-zero rows, rows with tiny entries (negative zero codes), saturating
    magnitudes and exactly representable values quantise exactly like the oracle."""
    rows = wl.draw_rows(6, wl.HEAD_DIM, [5], 9).float()
    rows[0] = 0.0
    rows[1] = rows[1] * 1e-4
    rows[1, 0] = 3.0                      # most entries round to +-0 at scale 3/448
    rows[2] = torch.linspace(-448.0, 448.0, wl.HEAD_DIM)
    rows[3] = rows[3] * 1e30
    rows[4, :] = 2.0 ** -7
    rows[5] = -rows[5].abs()
    rows = rows.to(torch.bfloat16)
    case = _case([0], seed=3, headroom=6, kv="fp8")
    dev = DeviceCache(case, "fp8")
    dev.append(rows.view(1, 6, -1), rows.view(1, 6, -1))
    dev.check_errors()
    codes, scales = oracle_mod.quantize_tokens_e4m3(wl.bits(rows))
    gk, _, gks, _, gsl = dev.host_caches()
    assert gsl[0] == 6
    slots = wl.slots_of([6], case.page_table)
    assert np.array_equal(gk.reshape(-1, wl.HEAD_DIM)[slots], codes)
    assert np.array_equal(gks.reshape(-1)[slots].view(np.uint32), scales.view(np.uint32))
    assert np.any(codes[1] == 0x80)  # the sign survives on zero codes


def test_append_capacity_fault_leaves_sequence_unchanged():
    case = _case([60, 10], seed=8, headroom=0)
    dev = DeviceCache(case, "bf16")
    before = dev.k_cache.clone()
    cap = dev.max_pages * wl.PAGE_SIZE
    n_new = cap - 60 + 1   # one token too many for sequence 0
    kn = wl.draw_rows(2 * n_new, wl.HEAD_DIM, [8], 4).view(2, n_new, -1)
    dev.append(kn, kn)
    with pytest.raises(capi.MFAError) as ei:
        dev.check_errors()
    assert ei.value.status == 6  # MFA_ERR_DEVICE_CAPACITY
    sl = dev.seq_lens.cpu().tolist()
    assert sl == [60, 10 + n_new]
    page0 = int(case.page_table[0, 0])
    assert torch.equal(dev.k_cache[page0].view(torch.int16), before[page0].view(torch.int16))


def test_append_bad_page_fault():
    case = _case([64, 3], seed=9, headroom=1)
    dev = DeviceCache(case, "bf16")
    dev.page_table[0, 1] = case.num_pages + 5   # the page the next token of sequence 0 lands in
    kn = wl.draw_rows(2, wl.HEAD_DIM, [9], 4).view(2, 1, -1)
    dev.append(kn, kn)
    with pytest.raises(capi.MFAError) as ei:
        dev.check_errors()
    assert ei.value.status == 5  # MFA_ERR_DEVICE_PAGE
    assert dev.seq_lens.cpu().tolist() == [64, 4]


def test_append_rejects_bad_arguments():
    t = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_kv_append(None, t, 1, t, t, t, t, 1, 1, 1, ws)
    assert ei.value.status == 1
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_kv_append(t, t, 1, t, t, t, t, 0, 1, 1, ws)
    assert ei.value.status == 1
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_kv_append(t.data_ptr() + 2, t, 1, t, t, t, t, 1, 1, 1, ws)
    assert ei.value.status == 1
    with pytest.raises(capi.MFAError) as ei:
        capi.mfa_kv_append(t, t, 1, t, t, t, t, 1, 1, 1, None)
    assert ei.value.status == 4


def test_fp4_quantiser_special_rows(oracle_mod):
    """All-zero rows, rows whose scaled values sit exactly on the E2M1 midpoints
    (ties go to the even mantissa), tiny entries (negative zero codes) and
    huge magnitudes quantise exactly like the oracle, packed low nibble first."""
    rows = wl.draw_rows(6, wl.HEAD_DIM, [6], 9).float()
    rows[0] = 0.0
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])  # absmax 6: scale 1
    rows[1] = ties.repeat(wl.HEAD_DIM // 8) * torch.where(torch.arange(wl.HEAD_DIM) % 16 < 8, 1.0, -1.0)
    rows[2] = rows[2] * 1e-4
    rows[2, 0] = 3.0                      # most entries round to +-0 at scale 0.5
    rows[3] = rows[3] * 1e30
    rows[5] = -rows[5].abs()
    rows = rows.to(torch.bfloat16)
    case = _case([0], seed=4, headroom=6, kv="fp4")
    dev = DeviceCache(case, "fp4")
    dev.append(rows.view(1, 6, -1), rows.view(1, 6, -1))
    dev.check_errors()
    packed, scales = oracle_mod.quantize_tokens_e2m1(wl.bits(rows))
    gk, _, gks, _, gsl = dev.host_caches()
    assert gsl[0] == 6
    slots = wl.slots_of([6], case.page_table)
    assert np.array_equal(gk.reshape(-1, wl.HEAD_DIM // 2)[slots], packed)
    assert np.array_equal(gks.reshape(-1)[slots].view(np.uint32), scales.view(np.uint32))
    codes = oracle_mod.unpack_e2m1(packed)
    assert scales[1] == 1.0 and np.array_equal(oracle_mod.e2m1_decode(codes[1, :8]), [0, 1, 1, 2, 2, 4, 4, 6])
    assert np.any(codes[2] == 8)  # the sign survives on zero codes
