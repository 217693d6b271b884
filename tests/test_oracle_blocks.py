"""Pins of the oracle's block-gather decode ("Step-5-Preview" page, sparse
attention: the query attends to the original K/V rows of the selected
historical 8-token blocks and of its own block up to itself; the softmax
runs over that set).

The pins: selecting every historical block is dense decode (bit for bit);
the order of the selection does not matter; an explicit position mask in
extended precision; the current block alone (one position: the value row
itself); rows outside the selection do not matter; malformed selections are
rejected."""
import numpy as np
import pytest

from decode_attention_mfa_gb300 import workloads as wl

H, D = wl.HEADS, wl.HEAD_DIM


def block_case(lengths, seed=11):
    w = wl.Workload("blocks-pin", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
    case = wl.make_case(w, lengths=lengths)
    kb = wl.bits(wl.scatter_rows(case.k_rows, case.lengths0, case.page_table, case.num_pages))
    vb = wl.bits(wl.scatter_rows(case.v_rows, case.lengths0, case.page_table, case.num_pages))
    return case, kb, vb


def run(oracle_mod, case, kb, vb, block_idx, n_blocks):
    return oracle_mod.mfa_decode_blocks(wl.bits(case.q), kb, vb, case.page_table, case.lengths0.astype(np.int32),
                                        block_idx, n_blocks, wl.SCALE)


def test_every_block_is_dense_decode(oracle_mod):
    lengths = [1, 8, 9, 64, 65, 200, 513]
    case, kb, vb = block_case(lengths)
    hist = [(L - 1) // 8 for L in lengths]
    bi = np.full((len(lengths), max(hist)), -1, dtype=np.int32)
    for b, n in enumerate(hist):
        bi[b, :n] = np.arange(n)
    out, lse = run(oracle_mod, case, kb, vb, bi, np.array(hist, dtype=np.int32))
    ref, ref_lse = oracle_mod.mfa_decode(wl.bits(case.q), kb, vb, case.page_table, case.lengths0.astype(np.int32),
                                         wl.SCALE)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_selection_order_does_not_matter(oracle_mod):
    lengths = [300, 1000]
    case, kb, vb = block_case(lengths, seed=12)
    bi, nb = wl.draw_blocks(lengths, 20, [12])
    out, lse = run(oracle_mod, case, kb, vb, bi, nb)
    bi2 = bi.copy()
    for b in range(len(lengths)):
        bi2[b, :nb[b]] = bi2[b, :nb[b]][::-1]
    out2, lse2 = run(oracle_mod, case, kb, vb, bi2, nb)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_matches_masked_softmax_in_extended_precision(oracle_mod):
    """A position mask over the whole sequence, long double, no max subtraction."""
    lengths = [77, 260]
    case, kb, vb = block_case(lengths, seed=13)
    bi, nb = wl.draw_blocks(lengths, 5, [13])
    out, lse = run(oracle_mod, case, kb, vb, bi, nb)
    qf = oracle_mod.bf16_to_f64(wl.bits(case.q)).astype(np.longdouble)
    off = 0
    for b, L in enumerate(lengths):
        K = oracle_mod.bf16_to_f64(wl.bits(case.k_rows[off:off + L])).astype(np.longdouble)
        V = oracle_mod.bf16_to_f64(wl.bits(case.v_rows[off:off + L])).astype(np.longdouble)
        off += L
        j = np.arange(L)
        chosen = set(int(r) for r in bi[b, :nb[b]])
        mask = np.array([(x // 8) in chosen or x >= 8 * ((L - 1) // 8) for x in j])
        s = np.longdouble(wl.SCALE) * (qf[b] @ K.T)  # [H, L]
        e = np.where(mask[None, :], np.exp(s), 0.0)
        z = e.sum(axis=1)
        np.testing.assert_allclose(out[b], (e @ V / z[:, None]).astype(np.float64), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[b], np.log(z).astype(np.float64), rtol=0, atol=1e-12)


def test_current_block_alone(oracle_mod):
    """No selected block and a length of 8c + 1: one position, the last one."""
    lengths = [1, 17, 129]
    case, kb, vb = block_case(lengths, seed=14)
    out, lse = run(oracle_mod, case, kb, vb, np.full((3, 1), -1, np.int32), np.zeros(3, np.int32))
    off = 0
    for b, L in enumerate(lengths):
        off += L
        v_last = oracle_mod.bf16_to_f64(wl.bits(case.v_rows[off - 1:off]))[0]
        k_last = oracle_mod.bf16_to_f64(wl.bits(case.k_rows[off - 1:off]))[0].astype(np.longdouble)
        np.testing.assert_array_equal(out[b], np.broadcast_to(v_last, (H, D)))
        qf = oracle_mod.bf16_to_f64(wl.bits(case.q[b])).astype(np.longdouble)
        np.testing.assert_allclose(lse[b], (np.longdouble(wl.SCALE) * (qf @ k_last)).astype(np.float64),
                                   rtol=1e-12, atol=1e-12)


def test_rows_outside_the_selection_do_not_matter(oracle_mod):
    lengths = [400]
    case, kb, vb = block_case(lengths, seed=15)
    bi = np.array([[3, 10, 40]], dtype=np.int32)
    nb = np.array([3], dtype=np.int32)
    out, lse = run(oracle_mod, case, kb, vb, bi, nb)
    kb2, vb2 = kb.copy(), vb.copy()
    for pos in (8 * 4 + 2, 8 * 20, 8 * 48 + 7):  # blocks 4, 20, 48: not selected and not current
        page, row = case.page_table[0][pos // 64], pos % 64
        kb2[page, row] ^= np.uint16(0x0040)
        vb2[page, row] ^= np.uint16(0x0040)
    out2, lse2 = run(oracle_mod, case, kb2, vb2, bi, nb)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    pos = 8 * 10 + 5  # a selected row changes the result
    page, row = case.page_table[0][pos // 64], pos % 64
    vb2[page, row] ^= np.uint16(0x0040)
    out3, _ = run(oracle_mod, case, kb2, vb2, bi, nb)
    assert not np.array_equal(out3, out)


@pytest.mark.parametrize("blocks", [[5], [-1], [2, 2]])
def test_malformed_selection_is_rejected(oracle_mod, blocks):
    lengths = [41]  # blocks 0..4 are historical; block 5 holds the last token
    case, kb, vb = block_case(lengths, seed=16)
    with pytest.raises(ValueError):
        run(oracle_mod, case, kb, vb, np.array([blocks], dtype=np.int32), np.array([len(blocks)], np.int32))


def test_draw_blocks_is_a_valid_selection():
    lengths = [0, 1, 9, 70, 5000]
    bi, nb = wl.draw_blocks(lengths, 16, [3])
    for b, L in enumerate(lengths):
        hist = max(0, (L - 1) // 8)
        assert nb[b] == min(16, hist)
        sel = bi[b, :nb[b]]
        assert len(set(sel.tolist())) == nb[b] and np.all((sel >= 0) & (sel < hist))
        assert np.all(bi[b, nb[b]:] == -1)


def quantised_case(oracle_mod, lengths, kv, seed):
    """Codes and per-token scales of the oracle's own quantiser, laid out in pages (unused slots hold the
    format's poison and NaN scales)."""
    w = wl.Workload("blocks-pin-q", len(lengths), ("list", tuple(lengths)), "bf16", True, 0, seed)
    case = wl.make_case(w, lengths=lengths)
    quant = oracle_mod.quantize_tokens_e2m1 if kv == "fp4" else oracle_mod.quantize_tokens_e4m3
    width = D // 2 if kv == "fp4" else D
    kcodes, kscale = quant(wl.bits(case.k_rows))
    vcodes, vscale = quant(wl.bits(case.v_rows))
    n = case.num_pages * wl.PAGE_SIZE
    slots = wl.slots_of(case.lengths0, case.page_table)
    poison = 0x77 if kv == "fp4" else 0x7F
    kc = np.full((n, width), poison, np.uint8); vc = np.full((n, width), poison, np.uint8)
    ks = np.full(n, np.nan, np.float32); vs = np.full(n, np.nan, np.float32)
    kc[slots], vc[slots], ks[slots], vs[slots] = kcodes, vcodes, kscale, vscale
    shape = (case.num_pages, wl.PAGE_SIZE)
    return case, kc.reshape(shape + (width,)), vc.reshape(shape + (width,)), ks.reshape(shape), vs.reshape(shape)


@pytest.mark.parametrize("kv", ["fp8", "fp4"])
def test_every_block_on_a_quantised_cache_is_dense_decode(oracle_mod, kv):
    """E4M3 / E2M1 cache: the codes and their scales are gathered together, so
    selecting every block is the dense quantised decode, bit for bit."""
    lengths = [1, 9, 65, 200, 513]
    case, kc, vc, ks, vs = quantised_case(oracle_mod, lengths, kv, seed=21)
    hist = [(L - 1) // 8 for L in lengths]
    bi = np.full((len(lengths), max(hist)), -1, dtype=np.int32)
    for b, n in enumerate(hist):
        bi[b, :n] = np.arange(n)
    sl = case.lengths0.astype(np.int32)
    out, lse = oracle_mod.mfa_decode_blocks(wl.bits(case.q), kc, vc, case.page_table, sl, bi,
                                            np.array(hist, dtype=np.int32), wl.SCALE, k_scale=ks, v_scale=vs)
    ref, ref_lse = oracle_mod.mfa_decode(wl.bits(case.q), kc, vc, case.page_table, sl, wl.SCALE, k_scale=ks,
                                         v_scale=vs)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_quantised_selection_ignores_other_rows(oracle_mod):
    """E4M3: poisoning every code and scale outside the selection (NaN codes, NaN scales) changes nothing,
    and the result is the masked softmax of the dequantised selected rows in extended precision."""
    lengths = [300, 777]
    case, kc, vc, ks, vs = quantised_case(oracle_mod, lengths, "fp8", seed=22)
    bi, nb = wl.draw_blocks(lengths, 12, [22])
    sl = case.lengths0.astype(np.int32)
    out, lse = oracle_mod.mfa_decode_blocks(wl.bits(case.q), kc, vc, case.page_table, sl, bi, nb, wl.SCALE,
                                            k_scale=ks, v_scale=vs)
    kc2, vc2, ks2, vs2 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    qf = oracle_mod.bf16_to_f64(wl.bits(case.q)).astype(np.longdouble)
    for b, L in enumerate(lengths):
        pos = oracle_mod.selected_positions(L, bi[b, :nb[b]])
        keep = np.zeros(L, bool); keep[pos] = True
        for j in np.nonzero(~keep)[0]:
            page, row = case.page_table[b][j // 64], j % 64
            kc2[page, row] = 0x7F; vc2[page, row] = 0x7F; ks2[page, row] = np.nan; vs2[page, row] = np.nan
        # extended-precision reference over the selected rows
        pg, rw = case.page_table[b][pos // 64], pos % 64
        K = oracle_mod.e4m3_decode(kc[pg, rw]).astype(np.longdouble) * ks[pg, rw].astype(np.longdouble)[:, None]
        V = oracle_mod.e4m3_decode(vc[pg, rw]).astype(np.longdouble) * vs[pg, rw].astype(np.longdouble)[:, None]
        e = np.exp(np.longdouble(wl.SCALE) * (qf[b] @ K.T))
        z = e.sum(axis=1)
        np.testing.assert_allclose(out[b], ((e @ V) / z[:, None]).astype(np.float64), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[b], np.log(z).astype(np.float64), rtol=0, atol=1e-12)
    out2, lse2 = oracle_mod.mfa_decode_blocks(wl.bits(case.q), kc2, vc2, case.page_table, sl, bi, nb, wl.SCALE,
                                              k_scale=ks2, v_scale=vs2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
