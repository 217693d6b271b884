"""Pins of the oracle's multi-token (MTP) decode ("Step-3 is Large yet
Affordable", section 5.2: extra predicted tokens read the same KV cache).

The T query tokens of sequence b are its last T positions; token t attends,
causally, to positions j < L_b - T + 1 + t. The pins check that reading
against an explicit masked softmax in extended precision, the T = 1 reduction
to single-token decode, and causality (a later position never changes an
earlier token's output)."""
import numpy as np
import pytest

from decode_attention_mfa_gb300 import workloads as wl

H, D = wl.HEADS, wl.HEAD_DIM


def mtp_case(lengths, T, seed=7):
    w = wl.Workload("mtp-pin", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
    case = wl.make_case(w, lengths=lengths)
    q = wl.draw_rows(len(lengths) * T * H, D, [seed, 90], 0).view(len(lengths), T, H, D)
    return case, q


def paged_bf16(case):
    kc = wl.scatter_rows(case.k_rows, case.lengths0, case.page_table, case.num_pages)
    vc = wl.scatter_rows(case.v_rows, case.lengths0, case.page_table, case.num_pages)
    return wl.bits(kc), wl.bits(vc)


def dense_rows(oracle_mod, rows_bits, lengths):
    vals = oracle_mod.bf16_to_f64(rows_bits)
    out, off = [], 0
    for n in lengths:
        out.append(vals[off:off + int(n)])
        off += int(n)
    return out


@pytest.mark.parametrize("T", [2, 3, 4, 8])
def test_mtp_matches_masked_softmax_in_extended_precision(oracle_mod, T):
    """Explicit causal mask over the dense K/V rows, long double, no max subtraction."""
    lengths = [3, 5, 70, 129]
    case, q = mtp_case(lengths, T)
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode_mtp(wl.bits(q), kb, vb, case.page_table, case.lengths0.astype(np.int32),
                                         wl.SCALE)
    assert out.shape == (len(lengths), T, H, D) and lse.shape == (len(lengths), T, H)
    qf = oracle_mod.bf16_to_f64(wl.bits(q)).astype(np.longdouble)
    Ks = dense_rows(oracle_mod, wl.bits(case.k_rows), lengths)
    Vs = dense_rows(oracle_mod, wl.bits(case.v_rows), lengths)
    for b, L in enumerate(lengths):
        K, V = Ks[b].astype(np.longdouble), Vs[b].astype(np.longdouble)
        s = np.longdouble(wl.SCALE) * np.einsum("thd,jd->thj", qf[b], K)  # [T, H, L]
        mask = np.arange(L)[None, :] <= (L - T + np.arange(T))[:, None]   # [T, L]: j <= position of token t
        e = np.where(mask[:, None, :], np.exp(s), 0.0)
        z = e.sum(axis=2)
        seen = z > 0  # a token whose mask is empty (L < T) sees nothing: out = 0, lse = -inf
        with np.errstate(invalid="ignore", divide="ignore"):
            ref = np.einsum("thj,jd->thd", e, V) / z[..., None]
            ref_lse = np.log(z)
        np.testing.assert_allclose(out[b][seen], ref[seen].astype(np.float64), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[b][seen], ref_lse[seen].astype(np.float64), rtol=0, atol=1e-12)
        assert np.all(out[b][~seen] == 0) and np.all(np.isneginf(lse[b][~seen]))


def test_mtp_with_one_token_is_single_token_decode(oracle_mod):
    lengths = [1, 64, 65, 300]
    case, q = mtp_case(lengths, 1, seed=8)
    kb, vb = paged_bf16(case)
    sl = case.lengths0.astype(np.int32)
    out, lse = oracle_mod.mfa_decode_mtp(wl.bits(q), kb, vb, case.page_table, sl, wl.SCALE)
    ref, ref_lse = oracle_mod.mfa_decode(wl.bits(q[:, 0]), kb, vb, case.page_table, sl, wl.SCALE)
    assert np.array_equal(out[:, 0], ref) and np.array_equal(lse[:, 0], ref_lse)


def test_mtp_is_causal(oracle_mod):
    """Changing the K/V row of the last position changes only the last token."""
    T, lengths = 3, [130, 7]
    case, q = mtp_case(lengths, T, seed=9)
    kb, vb = paged_bf16(case)
    sl = case.lengths0.astype(np.int32)
    out, lse = oracle_mod.mfa_decode_mtp(wl.bits(q), kb, vb, case.page_table, sl, wl.SCALE)
    kb2, vb2 = kb.copy(), vb.copy()
    for b, L in enumerate(lengths):
        page, row = case.page_table[b][(L - 1) // 64], (L - 1) % 64
        kb2[page, row] ^= np.uint16(0x0040)  # flip a mantissa bit of every element
        vb2[page, row] ^= np.uint16(0x0040)
    out2, lse2 = oracle_mod.mfa_decode_mtp(wl.bits(q), kb2, vb2, case.page_table, sl, wl.SCALE)
    assert np.array_equal(out2[:, :T - 1], out[:, :T - 1]) and np.array_equal(lse2[:, :T - 1], lse[:, :T - 1])
    assert not np.array_equal(out2[:, T - 1], out[:, T - 1])


def test_mtp_sequence_shorter_than_the_tokens(oracle_mod):
    """L_b < T: the earliest tokens see no position (out = 0, lse = -inf)."""
    T, lengths = 3, [1, 0]
    case, q = mtp_case(lengths, T, seed=10)
    kb, vb = paged_bf16(case)
    out, lse = oracle_mod.mfa_decode_mtp(wl.bits(q), kb, vb, case.page_table, case.lengths0.astype(np.int32),
                                         wl.SCALE)
    assert np.all(out[0, :2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.all(np.isfinite(lse[0, 2]))
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    v0 = oracle_mod.bf16_to_f64(wl.bits(case.v_rows[:1]))[0]
    np.testing.assert_array_equal(out[0, 2], np.broadcast_to(v0, (H, D)))


def test_mtp_on_an_e4m3_cache_is_the_masked_softmax_of_the_dequantised_rows(oracle_mod):
    """Quantised cache: the same causal masked softmax, in long double, over
    decode(code) * scale of every row (codes and scales from the oracle's own
    per-token quantiser, whose codec is pinned against the OCP table)."""
    T, lengths = 3, [2, 66, 129]
    case, q = mtp_case(lengths, T, seed=11)
    kcodes, kscale = oracle_mod.quantize_tokens_e4m3(wl.bits(case.k_rows))
    vcodes, vscale = oracle_mod.quantize_tokens_e4m3(wl.bits(case.v_rows))
    n = case.num_pages * wl.PAGE_SIZE
    slots = wl.slots_of(case.lengths0, case.page_table)
    kc = np.zeros((n, D), np.uint8); vc = np.zeros((n, D), np.uint8)
    ks = np.ones(n, np.float32); vs = np.ones(n, np.float32)
    kc[slots], vc[slots], ks[slots], vs[slots] = kcodes, vcodes, kscale, vscale
    sl = case.lengths0.astype(np.int32)
    out, lse = oracle_mod.mfa_decode_mtp(wl.bits(q), kc.reshape(-1, 64, D), vc.reshape(-1, 64, D), case.page_table,
                                         sl, wl.SCALE, k_scale=ks.reshape(-1, 64), v_scale=vs.reshape(-1, 64))
    kd = oracle_mod.e4m3_decode(kcodes).astype(np.longdouble) * kscale.astype(np.longdouble)[:, None]
    vd = oracle_mod.e4m3_decode(vcodes).astype(np.longdouble) * vscale.astype(np.longdouble)[:, None]
    qf = oracle_mod.bf16_to_f64(wl.bits(q)).astype(np.longdouble)
    off = 0
    for b, L in enumerate(lengths):
        K, V = kd[off:off + L], vd[off:off + L]
        off += L
        s = np.longdouble(wl.SCALE) * np.einsum("thd,jd->thj", qf[b], K)
        mask = np.arange(L)[None, :] <= (L - T + np.arange(T))[:, None]
        e = np.where(mask[:, None, :], np.exp(s), 0.0)
        z = e.sum(axis=2)
        with np.errstate(invalid="ignore", divide="ignore"):
            ref = np.einsum("thj,jd->thd", e, V) / z[..., None]
            ref_lse = np.log(z)
        seen = z > 0
        np.testing.assert_allclose(out[b][seen], ref[seen].astype(np.float64), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[b][seen], ref_lse[seen].astype(np.float64), rtol=0, atol=1e-12)
        assert np.all(out[b][~seen] == 0) and np.all(np.isneginf(lse[b][~seen]))
