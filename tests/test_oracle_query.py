"""Pins of the oracle's low-rank query path ("Step-3 is Large yet Affordable",
section 2 / Table 1: down-projection to rank 2048, normalisation,
up-projection to 64 x 256), read as RMSNorm with a learned gain."""
import numpy as np
import torch

from decode_attention_mfa_gb300 import workloads as wl


def bits(a):
    return wl.bits(torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def rand_bits(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return bits(g.standard_normal(shape) * scale)


def test_query_lowrank_matches_explicit_loops(oracle_mod):
    """Tiny shapes, every sum written out as a Python loop."""
    B, Dm, R, N = 3, 6, 4, 5
    xb, wdb, gb, wub = rand_bits((B, Dm), 1), rand_bits((Dm, R), 2), rand_bits((R,), 3), rand_bits((R, N), 4)
    eps = 1e-6
    q, h = oracle_mod.query_lowrank(xb, wdb, gb, wub, eps)
    x, wd, g, wu = (oracle_mod.bf16_to_f64(a) for a in (xb, wdb, gb, wub))
    for b in range(B):
        y = [sum(x[b, i] * wd[i, r] for i in range(Dm)) for r in range(R)]
        ms = sum(v * v for v in y) / R
        hh = [y[r] / np.sqrt(ms + eps) * g[r] for r in range(R)]
        for n in range(N):
            ref = sum(hh[r] * wu[r, n] for r in range(R))
            assert abs(q[b, n] - ref) <= 1e-12 * (1 + abs(ref))
        np.testing.assert_allclose(h[b], hh, rtol=1e-13, atol=1e-15)


def test_normalisation_is_rms_without_centering(oracle_mod):
    """eps = 0, gain 1: h has root-mean-square 1, and a constant y stays
    constant (a mean-subtracting norm would map it to 0)."""
    B, Dm, R, N = 2, 8, 16, 3
    wd = np.zeros((Dm, R), np.float32)
    wd[0, :] = 1.0  # y = x[:, 0] in every column
    xb = bits(np.array([[3.0] + [0.0] * 7, [-0.5] + [1.0] * 7]))
    q, h = oracle_mod.query_lowrank(xb, bits(wd), bits(np.ones(R)), rand_bits((R, N), 5), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(h * h, axis=1)), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(h[0], np.ones(R))
    np.testing.assert_array_equal(h[1], -np.ones(R))


def test_query_is_invariant_to_scaling_the_input(oracle_mod):
    """With eps = 0 the normalisation removes any scale of x exactly (powers of two)."""
    xb, wdb, gb, wub = rand_bits((4, 64), 6), rand_bits((64, 32), 7), rand_bits((32,), 8), rand_bits((32, 16), 9)
    q1, _ = oracle_mod.query_lowrank(xb, wdb, gb, wub, 0.0)
    x4 = bits(oracle_mod.bf16_to_f64(xb) * 4.0)
    q4, _ = oracle_mod.query_lowrank(x4, wdb, gb, wub, 0.0)
    np.testing.assert_allclose(q4, q1, rtol=1e-12, atol=1e-12)


def test_zero_gain_gives_zero_query(oracle_mod):
    q, _ = oracle_mod.query_lowrank(rand_bits((2, 8), 10), rand_bits((8, 4), 11), bits(np.zeros(4)),
                                    rand_bits((4, 6), 12), 1e-6)
    assert np.all(q == 0)
