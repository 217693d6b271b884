"""Pins of the oracle's 4-bit KV ("Step-3 is Large yet Affordable", section
5.2: KV stored in 4 bits, attention computed in 8 bits), read as OCP MX FP4
(E2M1) codes with one fp32 scale per token.

The codec is pinned to the format's value table (tests/golden) and to
properties any correct round-to-nearest-even encoder has; the quantiser to its
scale rule, its packing and its error bound; the attention over a 4-bit cache
to an independent softmax over the dequantised values; the append to the
quantiser."""
import json
import os

import numpy as np
import pytest

from decode_attention_mfa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAGE, D = wl.PAGE_SIZE, wl.HEAD_DIM


def test_e2m1_value_table(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "e2m1_ocp_values.json")))
    got = oracle_mod.e2m1_decode(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(got, np.array(g["values"]))
    assert np.array_equal(np.signbit(got), np.signbit(np.array(g["values"])))


def test_e2m1_encode_roundtrip_monotone_and_saturating(oracle_mod):
    vals = oracle_mod.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(oracle_mod.e2m1_encode(vals.astype(np.float32)), np.arange(16))
    x = np.linspace(-8, 8, 20001).astype(np.float32)
    dec = oracle_mod.e2m1_decode(oracle_mod.e2m1_encode(x))
    assert np.all(np.diff(dec) >= 0)                       # monotone
    assert np.all(np.abs(dec) <= 6.0)                      # saturating
    assert np.all(dec[x >= 6] == 6.0) and np.all(dec[x <= -6] == -6.0)


def test_e2m1_nearest_with_half_spacing_bound(oracle_mod):
    rng = np.random.default_rng(5)
    x = rng.uniform(-6, 6, 200000).astype(np.float32)
    dec = oracle_mod.e2m1_decode(oracle_mod.e2m1_encode(x))
    a = np.abs(x.astype(np.float64))
    spacing = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))  # 0.5 below 2, 1 in [2, 4), 2 in [4, 6]
    assert np.all(np.abs(dec - x) <= spacing / 2 + 1e-12)
    assert np.all(np.sign(dec[dec != 0]) == np.sign(x[dec != 0]))


def test_e2m1_ties_go_to_even_mantissa(oracle_mod):
    # midpoints between neighbours: the neighbour with mantissa bit 0 wins
    mid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0])
    np.testing.assert_array_equal(oracle_mod.e2m1_decode(oracle_mod.e2m1_encode(mid)), want)
    np.testing.assert_array_equal(oracle_mod.e2m1_decode(oracle_mod.e2m1_encode(-mid)), -want)
    assert oracle_mod.e2m1_encode(np.array([-0.1], np.float32))[0] == 8  # sign kept on zero


def test_quantize_tokens_e2m1(oracle_mod):
    rows = wl.draw_rows(300, D, [9], 0)
    x = oracle_mod.bf16_to_f64(wl.bits(rows))
    x[7] = 0.0  # an all-zero row
    bits = wl.bits(rows).copy()
    bits[7] = 0
    packed, scales = oracle_mod.quantize_tokens_e2m1(bits)
    assert packed.shape == (300, D // 2) and scales.shape == (300,)
    codes = oracle_mod.unpack_e2m1(packed)
    np.testing.assert_array_equal(codes[:, 0::2], packed & 15)  # element 2k in the low nibble
    amax = np.abs(x).max(axis=1)
    expect = np.where(amax > 0, (amax.astype(np.float32) / np.float32(6.0)), 1.0).astype(np.float32)
    np.testing.assert_array_equal(scales, expect)
    deq = oracle_mod.e2m1_decode(codes) * scales[:, None].astype(np.float64)
    big = np.argmax(np.abs(x), axis=1)
    live = amax > 0
    np.testing.assert_array_equal(np.abs(deq[np.arange(300), big])[live], 6.0 * scales[live].astype(np.float64))
    # within half a spacing of the scaled grid (x / s is an fp32 division: allow its rounding)
    a = np.abs(x) / scales[:, None]
    spacing = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0)) * scales[:, None]
    assert np.all(np.abs(deq - x) <= spacing / 2 * (1 + 1e-6) + 1e-30)
    assert np.all(codes[7] == 0) and scales[7] == 1.0


def fp4_cache(oracle_mod, case):
    kp, ks_ = oracle_mod.quantize_tokens_e2m1(wl.bits(case.k_rows))
    vp, vs_ = oracle_mod.quantize_tokens_e2m1(wl.bits(case.v_rows))
    slots = wl.slots_of(case.lengths0, case.page_table)
    n = case.num_pages * PAGE
    kc = np.zeros((n, D // 2), np.uint8); kc[slots] = kp
    vc = np.zeros((n, D // 2), np.uint8); vc[slots] = vp
    ks = np.ones(n, np.float32); ks[slots] = ks_
    vs = np.ones(n, np.float32); vs[slots] = vs_
    return (kc.reshape(-1, PAGE, D // 2), vc.reshape(-1, PAGE, D // 2), ks.reshape(-1, PAGE), vs.reshape(-1, PAGE),
            kp, ks_, vp, vs_)


def test_fp4_attention_equals_definition_on_dequantised_values(oracle_mod):
    special = pytest.importorskip("scipy.special")
    lengths = [100, 64, 1]
    w = wl.Workload("fp4-pin", 3, ("list", tuple(lengths)), "bf16", True, 0, 32)
    case = wl.make_case(w, lengths=lengths)
    kc, vc, ks, vs, kp, ks_, vp, vs_ = fp4_cache(oracle_mod, case)
    out, lse = oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, case.lengths0.astype(np.int32),
                                     wl.SCALE, k_scale=ks, v_scale=vs)
    q = oracle_mod.bf16_to_f64(wl.bits(case.q))
    kd = oracle_mod.e2m1_decode(oracle_mod.unpack_e2m1(kp)) * ks_[:, None].astype(np.float64)
    vd = oracle_mod.e2m1_decode(oracle_mod.unpack_e2m1(vp)) * vs_[:, None].astype(np.float64)
    off = 0
    for b, L in enumerate(lengths):
        s = wl.SCALE * (q[b] @ kd[off:off + L].T)
        np.testing.assert_allclose(out[b], special.softmax(s, axis=1) @ vd[off:off + L], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(lse[b], special.logsumexp(s, axis=1), rtol=0, atol=1e-12)
        off += L


def test_fp4_append_quantises_into_the_slot(oracle_mod):
    lengths = [5, 64]
    w = wl.Workload("fp4-app", 2, ("list", tuple(lengths)), "bf16", True, 0, 33)
    case = wl.make_case(w, lengths=lengths, headroom_tokens=3)
    kc, vc, ks, vs, *_ = fp4_cache(oracle_mod, case)
    sl = case.lengths0.astype(np.int32).copy()
    kn = wl.draw_rows(2 * 3, D, [33, 1], 0).view(2, 3, D)
    vn = wl.draw_rows(2 * 3, D, [33, 2], 0).view(2, 3, D)
    oracle_mod.kv_append(wl.bits(kn), wl.bits(vn), kc, vc, case.page_table, sl, k_scale=ks, v_scale=vs)
    assert list(sl) == [8, 67]
    for b, L in enumerate(lengths):
        for t in range(3):
            pos = L + t
            page, row = case.page_table[b][pos // PAGE], pos % PAGE
            kp, ksc = oracle_mod.quantize_tokens_e2m1(wl.bits(kn[b, t:t + 1]))
            vp, vsc = oracle_mod.quantize_tokens_e2m1(wl.bits(vn[b, t:t + 1]))
            assert np.array_equal(kc[page, row], kp[0]) and ks[page, row] == ksc[0]
            assert np.array_equal(vc[page, row], vp[0]) and vs[page, row] == vsc[0]
