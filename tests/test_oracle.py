"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a brute-force
evaluation in extended precision without max subtraction, closed forms (L=1,
constant keys), invariances (KV permutation, page permutation), the shared-KV
reduction to 64 independent single-head attentions computed with library
routines, the OCP E4M3 table and torch's float8_e4m3fn conversion, and a
statistical closed form for N(0,1) data.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from decode_attention_mfa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
H, D, PAGE = wl.HEADS, wl.HEAD_DIM, wl.PAGE_SIZE


def small_case(lengths, seed=5, permute=True, spare_pages=0, headroom=0):
    w = wl.Workload("pin", len(lengths), ("list", tuple(lengths)), "bf16", permute, 0, seed)
    return wl.make_case(w, lengths=lengths, headroom_tokens=headroom, spare_pages=spare_pages)


def paged_bf16(case):
    kc = wl.scatter_rows(case.k_rows, case.lengths0, case.page_table, case.num_pages)
    vc = wl.scatter_rows(case.v_rows, case.lengths0, case.page_table, case.num_pages)
    return wl.bits(kc), wl.bits(vc)


def dense_f64(rows_bits, lengths):
    """Concatenated bf16 rows -> list of per-sequence fp64 [L, D] arrays."""
    from oracle import bf16_to_f64
    vals = bf16_to_f64(rows_bits)
    out, off = [], 0
    for n in lengths:
        out.append(vals[off:off + int(n)])
        off += int(n)
    return out


# ------------------------------------------------------------------ attention
def test_brute_force_extended_precision(oracle_mod):
    """Direct formula in long double, no max subtraction, on tiny inputs."""
    lengths = [1, 2, 3, 64, 100]
    case = small_case(lengths)
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                     case.lengths0.astype(np.int32), wl.SCALE)
    q = oracle_mod.bf16_to_f64(wl.bits(case.q)).astype(np.longdouble)
    Ks = dense_f64(wl.bits(case.k_rows), lengths)
    Vs = dense_f64(wl.bits(case.v_rows), lengths)
    for b, n in enumerate(lengths):
        K = Ks[b].astype(np.longdouble)
        V = Vs[b].astype(np.longdouble)
        s = np.longdouble(wl.SCALE) * np.einsum("hd,jd->hj", q[b], K)
        e = np.exp(s)
        z = e.sum(axis=1)
        ref = np.einsum("hj,jd->hd", e, V) / z[:, None]
        ref_lse = np.log(z)
        np.testing.assert_allclose(out[b], ref.astype(np.float64), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[b], ref_lse.astype(np.float64), rtol=0, atol=1e-12)


def test_single_token_returns_v(oracle_mod):
    """L=1: the softmax weight is exactly 1, so out = v and lse = s_0."""
    case = small_case([1, 1, 1], seed=9)
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                     case.lengths0.astype(np.int32), wl.SCALE)
    v = oracle_mod.bf16_to_f64(wl.bits(case.v_rows))
    k = oracle_mod.bf16_to_f64(wl.bits(case.k_rows))
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))
    for b in range(3):
        assert np.array_equal(out[b], np.broadcast_to(v[b], (H, D)))
        s0 = wl.SCALE * (q[b] @ k[b])
        np.testing.assert_allclose(lse[b], s0, rtol=0, atol=1e-12)


def test_constant_keys_give_mean_of_v(oracle_mod):
    """All keys equal: every weight is 1/L, out = mean(v), lse = s + ln L."""
    lengths = [5, 64, 130]
    case = small_case(lengths, seed=3)
    off = 0
    for n in lengths:
        case.k_rows[off:off + n] = case.k_rows[off]
        off += n
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                     case.lengths0.astype(np.int32), wl.SCALE)
    Vs = dense_f64(wl.bits(case.v_rows), lengths)
    Ks = dense_f64(wl.bits(case.k_rows), lengths)
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))
    for b, n in enumerate(lengths):
        np.testing.assert_allclose(out[b], np.broadcast_to(Vs[b].mean(axis=0), (H, D)),
                                   rtol=1e-12, atol=1e-14)
        s = wl.SCALE * (q[b] @ Ks[b][0])
        np.testing.assert_allclose(lse[b], s + math.log(n), rtol=0, atol=1e-12)


def test_kv_permutation_invariance(oracle_mod):
    """Permuting the KV positions of a sequence leaves out and lse unchanged."""
    lengths = [77, 200]
    case = small_case(lengths, seed=21)
    kb, vb = paged_bf16(case)
    out1, lse1 = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                       case.lengths0.astype(np.int32), wl.SCALE)
    rng = np.random.default_rng(0)
    perm = np.concatenate([rng.permutation(lengths[0]), lengths[0] + rng.permutation(lengths[1])])
    case.k_rows = case.k_rows[torch.from_numpy(perm)]
    case.v_rows = case.v_rows[torch.from_numpy(perm)]
    kb, vb = paged_bf16(case)
    out2, lse2 = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                       case.lengths0.astype(np.int32), wl.SCALE)
    np.testing.assert_allclose(out1, out2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse1, lse2, rtol=0, atol=1e-12)


def test_page_permutation_is_bitwise_invariant(oracle_mod):
    """Where the pages sit in the cache does not change the result at all."""
    lengths = [64, 65, 1, 190]
    a = small_case(lengths, seed=4, permute=False)
    b = small_case(lengths, seed=4, permute=True, spare_pages=3)
    assert not np.array_equal(a.page_table, b.page_table[:, :a.page_table.shape[1]])
    ra = oracle_mod.mfa_decode(wl.bits(a.q), *paged_bf16(a), a.page_table,
                               a.lengths0.astype(np.int32), wl.SCALE)
    rb = oracle_mod.mfa_decode(wl.bits(b.q), *paged_bf16(b), b.page_table,
                               b.lengths0.astype(np.int32), wl.SCALE)
    assert np.array_equal(ra[0], rb[0]) and np.array_equal(ra[1], rb[1])


def test_shared_kv_equals_independent_heads(oracle_mod):
    """MFA row h == single-head attention of q_h over the same K, V, computed
    with numpy matmul and scipy's softmax/logsumexp (64 independent attentions
    with the shared KV replicated)."""
    special = pytest.importorskip("scipy.special")
    lengths = [129, 300]
    case = small_case(lengths, seed=8)
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                     case.lengths0.astype(np.int32), wl.SCALE)
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))
    Ks = dense_f64(wl.bits(case.k_rows), lengths)
    Vs = dense_f64(wl.bits(case.v_rows), lengths)
    for b in range(len(lengths)):
        for h in range(H):
            s = wl.SCALE * (Ks[b] @ q[b, h])
            ref = special.softmax(s) @ Vs[b]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-10, atol=1e-13)
            np.testing.assert_allclose(lse[b, h], special.logsumexp(s), rtol=0, atol=1e-12)


def test_unused_slots_never_leak(oracle_mod):
    """NaN in the unused rows of the last page (and in spare pages) changes nothing."""
    lengths = [10, 70]
    case = small_case(lengths, seed=12, spare_pages=2)
    kc = wl.scatter_rows(case.k_rows, lengths, case.page_table, case.num_pages, fill=0.0)
    vc = wl.scatter_rows(case.v_rows, lengths, case.page_table, case.num_pages, fill=0.0)
    r0 = oracle_mod.mfa_decode(wl.bits(case.q), wl.bits(kc), wl.bits(vc), case.page_table,
                               case.lengths0.astype(np.int32), wl.SCALE)
    r1 = oracle_mod.mfa_decode(wl.bits(case.q), *paged_bf16(case), case.page_table,
                               case.lengths0.astype(np.int32), wl.SCALE)
    assert np.all(np.isfinite(r1[0])) and np.array_equal(r0[0], r1[0])
    assert np.array_equal(r0[1], r1[1])


def test_large_logits_dominant_token(oracle_mod):
    """Logits 2048 apart: the largest one takes all the weight (the others are
    exp(-2048) = 0 in fp64), so out = v of that token and lse = its logit.
    Evaluating without subtracting the running maximum would overflow here."""
    L = 70
    case = small_case([L], seed=13)
    case.q.zero_()
    case.q[0, :, 0] = 256.0
    case.k_rows[:, 0] = -64.0
    case.k_rows[37, 0] = 64.0
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                     case.lengths0.astype(np.int32), wl.SCALE)
    v = oracle_mod.bf16_to_f64(wl.bits(case.v_rows))
    assert np.array_equal(out[0], np.broadcast_to(v[37], (H, D)))
    assert np.all(lse[0] == 256.0 * 64.0 * wl.SCALE)


def test_empty_sequence(oracle_mod):
    case = small_case([0, 3], seed=2, headroom=1)
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                     case.lengths0.astype(np.int32), wl.SCALE)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


def test_rows_entry_matches_full(oracle_mod):
    case = small_case([33, 140], seed=6)
    kb, vb = paged_bf16(case)
    sl = case.lengths0.astype(np.int32)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table, sl, wl.SCALE)
    rb = np.array([1, 0, 1], dtype=np.int32)
    rh = np.array([63, 0, 17], dtype=np.int32)
    o2, l2 = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table, sl, wl.SCALE,
                                   rows=(rb, rh))
    assert np.array_equal(o2, out[rb, rh]) and np.array_equal(l2, lse[rb, rh])


def test_bad_page_and_length_are_rejected(oracle_mod):
    case = small_case([70], seed=1)
    kb, vb = paged_bf16(case)
    bad = case.page_table.copy()
    bad[0, 1] = case.num_pages  # out of range
    with pytest.raises(ValueError):
        oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, bad, case.lengths0.astype(np.int32), wl.SCALE)
    with pytest.raises(ValueError):
        oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                              np.array([10_000], dtype=np.int32), wl.SCALE)


def test_statistical_closed_form(oracle_mod):
    """For N(0,1) keys, E[exp(s_j)] = exp(|q|^2 / 512) (s_j ~ N(0, |q|^2/256)),
    so lse ~= ln L + |q_h|^2 / 512 with a relative spread of about 1.3/sqrt(L)."""
    L = 4096
    case = small_case([L], seed=17)
    kb, vb = paged_bf16(case)
    _, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table,
                                   case.lengths0.astype(np.int32), wl.SCALE)
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))[0]
    expect = math.log(L) + (q * q).sum(axis=1) / 512.0
    assert np.max(np.abs(lse[0] - expect)) < 0.15
    assert abs(np.mean(lse[0] - expect)) < 0.03


# ------------------------------------------------------------------ E4M3 codec
def test_e4m3_ocp_points(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "e4m3_ocp_points.json")))
    for p in g["points"]:
        assert oracle_mod.e4m3_decode(np.array([p["code"]]))[0] == p["value"]
        assert int(oracle_mod.e4m3_encode(np.array([p["value"]]))[0]) == p["code"]
    assert np.all(np.isnan(oracle_mod.e4m3_decode(np.array(g["nan_codes"]))))


def test_e4m3_decode_matches_torch_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_encode_roundtrip_and_torch(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (127, 255)], dtype=np.uint8)
    vals = oracle_mod.e4m3_decode(codes).astype(np.float32)
    back = oracle_mod.e4m3_encode(vals)
    assert np.array_equal(back, codes)
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.standard_normal(400_000).astype(np.float32) * np.float32(100),
        rng.standard_normal(300_000).astype(np.float32),
        rng.standard_normal(200_000).astype(np.float32) * np.float32(0.01),
        (rng.standard_normal(100_000) * 1e-3).astype(np.float32),
    ])
    mine = oracle_mod.e4m3_encode(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_e4m3_ties_to_even_and_saturation(oracle_mod):
    enc = lambda v: int(oracle_mod.e4m3_encode(np.array([v], dtype=np.float32))[0])
    assert enc(1.0625) == 0x38          # midway 1.0 / 1.125 -> even mantissa (1.0)
    assert enc(1.1875) == 0x3A          # midway 1.125 / 1.25 -> 1.25
    assert enc(2.0 ** -10) == 0x00      # midway 0 / 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02  # midway 2^-9 / 2^-8 -> 2^-8
    assert enc(464.0) == 0x7E and enc(1e30) == 0x7E and enc(float("inf")) == 0x7E
    assert enc(-1e30) == 0xFE
    assert enc(-1e-30) == 0x80          # sign kept on a zero result


def test_quantize_tokens(oracle_mod):
    rows = wl.draw_rows(512, D, [3], 9)
    rows[5] = 0
    codes, scales = oracle_mod.quantize_tokens_e4m3(wl.bits(rows))
    x = rows.float().numpy()
    amax = np.abs(x).max(axis=1)
    expect_scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(scales, expect_scale)
    assert np.all(codes[5] == 0) and scales[5] == 1.0
    # the absmax element becomes +-448
    i = np.abs(x).argmax(axis=1)
    top = np.delete(codes[np.arange(512), i], 5)
    assert np.all((top & 0x7F) == 0x7E)
    # dequantisation error: at most half a mantissa step (2^-4 relative) in the normal range
    deq = oracle_mod.e4m3_decode(codes) * scales[:, None].astype(np.float64)
    y = x.astype(np.float64) / scales[:, None]
    normal = np.abs(y) >= 2.0 ** -6
    rel = np.abs(deq - x) / np.abs(x).clip(1e-30)
    assert np.all(rel[normal] <= 2.0 ** -4 + 1e-12)
    sub = ~normal
    assert np.all(np.abs(deq - x)[sub] <= (2.0 ** -10) * np.broadcast_to(scales[:, None], x.shape)[sub] + 1e-30)


def test_fp8_attention_equals_definition_on_dequantised_values(oracle_mod):
    special = pytest.importorskip("scipy.special")
    lengths = [100, 64]
    case = small_case(lengths, seed=31)
    kcodes, kscale = oracle_mod.quantize_tokens_e4m3(wl.bits(case.k_rows))
    vcodes, vscale = oracle_mod.quantize_tokens_e4m3(wl.bits(case.v_rows))
    slots = wl.slots_of(lengths, case.page_table)
    n = case.num_pages * PAGE
    kc = np.zeros((n, D), np.uint8); kc[slots] = kcodes
    vc = np.zeros((n, D), np.uint8); vc[slots] = vcodes
    ks = np.zeros(n, np.float32); ks[slots] = kscale
    vs = np.zeros(n, np.float32); vs[slots] = vscale
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kc.reshape(-1, PAGE, D), vc.reshape(-1, PAGE, D),
                                     case.page_table, case.lengths0.astype(np.int32), wl.SCALE,
                                     k_scale=ks.reshape(-1, PAGE), v_scale=vs.reshape(-1, PAGE))
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))
    kd = torch.from_numpy(kcodes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * kscale[:, None]
    vd = torch.from_numpy(vcodes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * vscale[:, None]
    off = 0
    for b, L in enumerate(lengths):
        s = wl.SCALE * (q[b] @ kd[off:off + L].T)
        np.testing.assert_allclose(out[b], special.softmax(s, axis=1) @ vd[off:off + L],
                                   rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(lse[b], special.logsumexp(s, axis=1), rtol=0, atol=1e-12)
        off += L


# ------------------------------------------------------------------ append
def test_append_then_attend_includes_new_token(oracle_mod):
    """After appending, attention covers the old tokens plus the new one (the
    decode-context lesson: the attended length is cached length + 1)."""
    special = pytest.importorskip("scipy.special")
    lengths = [63, 64, 1]
    case = small_case(lengths, seed=40, headroom=1)
    kb, vb = paged_bf16(case)
    kb, vb = kb.copy(), vb.copy()
    sl = case.lengths0.astype(np.int32).copy()
    kn = wl.draw_rows(3, D, [40], 4).view(3, 1, D)
    vn = wl.draw_rows(3, D, [40], 5).view(3, 1, D)
    oracle_mod.kv_append(wl.bits(kn), wl.bits(vn), kb, vb, case.page_table, sl)
    assert list(sl) == [64, 65, 2]
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table, sl, wl.SCALE)
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))
    Ks = dense_f64(wl.bits(case.k_rows), lengths)
    Vs = dense_f64(wl.bits(case.v_rows), lengths)
    for b in range(3):
        K = np.vstack([Ks[b], oracle_mod.bf16_to_f64(wl.bits(kn[b]))])
        V = np.vstack([Vs[b], oracle_mod.bf16_to_f64(wl.bits(vn[b]))])
        s = wl.SCALE * (q[b] @ K.T)
        np.testing.assert_allclose(out[b], special.softmax(s, axis=1) @ V, rtol=1e-10, atol=1e-13)


def test_append_fp8_and_capacity(oracle_mod):
    lengths = [0, 5]
    case = small_case(lengths, seed=41, headroom=64)
    n = case.num_pages
    kc = np.zeros((n, PAGE, D), np.uint8); vc = np.zeros((n, PAGE, D), np.uint8)
    ks = np.zeros((n, PAGE), np.float32); vs = np.zeros((n, PAGE), np.float32)
    sl = np.array([0, 5], np.int32)
    kn = wl.draw_rows(2 * 3, D, [41], 4).view(2, 3, D)
    vn = wl.draw_rows(2 * 3, D, [41], 5).view(2, 3, D)
    oracle_mod.kv_append(wl.bits(kn), wl.bits(vn), kc, vc, case.page_table, sl, k_scale=ks, v_scale=vs)
    assert list(sl) == [3, 8]
    codes, scales = oracle_mod.quantize_tokens_e4m3(wl.bits(kn[1]))
    for t in range(3):
        pos = 5 + t
        page = case.page_table[1, pos // PAGE]
        assert np.array_equal(kc[page, pos % PAGE], codes[t]) and ks[page, pos % PAGE] == scales[t]
    big = wl.draw_rows(2 * 200, D, [41], 6).view(2, 200, D)
    with pytest.raises(ValueError):
        oracle_mod.kv_append(wl.bits(big), wl.bits(big), kc, vc, case.page_table, sl,
                             k_scale=ks, v_scale=vs)
