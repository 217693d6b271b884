"""C-ABI library checks that need no GPU: the library loads, exports every
function include/mfa.h declares, plans splits, names its status codes, and
the split partition it implements is a valid one (checked on the formulas)."""
import ctypes

import numpy as np
import pytest

from decode_attention_mfa_gb300 import build as mfa_build
from decode_attention_mfa_gb300 import capi


@pytest.fixture(scope="module")
def lib():
    mfa_build.build()
    return capi.load()


def test_exports_every_declared_symbol(lib):
    names = capi.header_functions()
    assert len(names) >= 12
    raw = ctypes.CDLL(capi.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in include/mfa.h but not exported"
    assert set(names) == set(capi._SIGNATURES), "binding and header disagree"


def test_mtp_query_count_is_checked_before_any_device_work(lib):
    """n_query outside [1, MFA_MAX_QUERY_TOKENS]: MFA_ERR_INVALID_ARG from the
    host checks of all three cache formats; the workspace size query answers 0."""
    for nq in (0, capi.MAX_QUERY_TOKENS + 1, -1):
        assert lib.mfa_decode_attention_mtp(None, None, None, None, None, None, None, 0.0625, 1, nq, 1, 1, 0,
                                            None, 0, None) == 1
        for fn in (lib.mfa_decode_attention_mtp_fp8, lib.mfa_decode_attention_mtp_fp4):
            assert fn(None, None, None, None, None, None, None, None, None, 0.0625, 1, nq, 1, 1, 0, None, 0,
                      None) == 1
        assert lib.mfa_decode_mtp_workspace_bytes(4, nq, 1024) == 0


def test_block_lists_are_checked_before_any_device_work(lib):
    """Block gather: null or misaligned block lists and max_blocks outside
    [1, 8 * max_pages] are refused by the host checks."""
    arr = (ctypes.c_int32 * 8)()
    p = ctypes.addressof(arr)
    cases = [(None, p, 4), (p, None, 4), (p + 2, p, 4), (p, p, 0), (p, p, 8 * 3 + 1)]
    for bi, nb, mb in cases:
        assert lib.mfa_decode_attention_blocks(None, None, None, None, None, bi, nb, mb, None, None, 0.0625, 1, 3, 3,
                                               64, None, 0, None) == 1


def test_four_bit_caches_must_be_32_byte_aligned(lib):
    """4-bit KV: TMA reads the packed codes only from 32-byte aligned rows;
    a misaligned cache is refused before any device work."""
    buf = (ctypes.c_uint8 * 128)()
    base = (ctypes.addressof(buf) + 31) & ~31
    for kc, vc in ((base + 16, base), (base, base + 16)):
        assert lib.mfa_decode_attention_fp4(None, kc, vc, None, None, None, None, None, None, 0.0625, 1, 1, 1, 64,
                                            None, 0, None) == 1
        assert lib.mfa_kv_append_fp4(None, None, 1, kc, vc, None, None, None, None, 1, 1, 1, None, None) == 1


def test_query_workspace_size_rules(lib):
    """The query path's workspace grows with the batch it holds and is refused
    (0) outside the limits; a workspace sized for more rows serves fewer."""
    R, N = 2048, 16384
    sizes = [lib.mfa_query_lowrank_workspace_bytes(b, R, N) for b in (1, 16, 32, 256)]
    assert all(x > 0 for x in sizes) and sizes == sorted(sizes)
    for b, r, n in ((0, R, N), (257, R, N), (4, 100, N), (4, R, 100), (4, capi.MAX_QUERY_RANK + 128, N)):
        assert lib.mfa_query_lowrank_workspace_bytes(b, r, n) == 0


def test_status_strings(lib):
    for code, name in capi.STATUS_NAMES.items():
        assert capi.mfa_status_string(code) == name


def test_plan_without_gpu(lib):
    p = capi.mfa_plan_decode(32, 4096, 152)
    assert p.grid_ctas == 152 and p.partial_slots == 152 + 31
    assert p.workspace_bytes == 256 + p.partial_slots * (64 * 256 * 4 + 64 * 4)
    assert capi.mfa_plan_decode(2, 100, 152).grid_ctas == 2
    one = capi.mfa_plan_decode(1, 0, 152)
    assert one.grid_ctas == 1 and one.partial_slots == 1
    for bad in ((0, 10), (2000, 10), (4, -1)):
        with pytest.raises(capi.MFAError):
            capi.mfa_plan_decode(bad[0], bad[1], 152)


def _cta_lo(c, C, G):
    return c * C // G


def _cta_of_cost(x, C, G):
    return ((x + 1) * G - 1) // C


@pytest.mark.parametrize("seed", range(24))
def test_partition_slots_are_unique_and_combine_finds_them(seed):
    """Split scheme used by the split and combine kernels: a sequence with
    n > 0 pages costs n + piece_cost units, its page k sits at unit
    cost_prefix[b] + piece_cost + k, and CTA c owns units [c*C//G,
    (c+1)*C//G); its piece of sequence b goes to slot c + b. Every page is
    owned by exactly one CTA, slots never collide and stay below G + B - 1,
    and the combine's CTA interval for b is exactly the CTAs that own pages
    of b."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 60))
    pages = rng.integers(0, 40, size=B) * (rng.random(B) < 0.9)
    if seed % 4 == 0:
        pages[:] = rng.integers(1, 3)  # many short sequences, more CTAs than pages
    G = int(rng.integers(1, 160))
    piece_cost = int(rng.integers(0, 4))
    cost = np.where(pages > 0, pages + piece_cost, 0)
    C = int(cost.sum())
    if C == 0:
        return
    prefix = np.concatenate([[0], np.cumsum(cost)])
    owners, slots, covered = {}, set(), np.zeros(B, dtype=np.int64)
    for c in range(G):
        lo, hi = _cta_lo(c, C, G), _cta_lo(c + 1, C, G)
        for b in range(B):
            first = prefix[b] + piece_cost
            pg0, pg1 = max(lo - first, 0), min(hi - first, pages[b])
            if pages[b] > 0 and pg0 < pg1:
                covered[b] += pg1 - pg0
                s = c + b
                assert s not in slots and s < G + B - 1
                slots.add(s)
                owners.setdefault(b, []).append(c)
    assert (covered == pages).all()
    for b in range(B):
        if pages[b] == 0:
            assert b not in owners
            continue
        first = prefix[b] + piece_cost
        cf, cl = _cta_of_cost(first, C, G), _cta_of_cost(first + pages[b] - 1, C, G)
        found = [c for c in range(cf, cl + 1) if _cta_lo(c, C, G) < _cta_lo(c + 1, C, G)]
        assert found == owners[b]


@pytest.mark.parametrize("seed", range(16))
def test_token_group_slots_are_unique_and_combine_finds_them(seed):
    """Multi-token decode with token groups: T query tokens, q_per_cta of them
    a CTA, so g = ceil(T / q_per_cta) groups; the grid holds g CTAs for each of
    R ranges (CTA c: range c // g, group c % g). The piece of sequence b that
    range i holds, for group r, is written to slot (i + b) * g + r, each slot
    holding q_per_cta tokens. Every (sequence, token, page) is covered by
    exactly one CTA, slots never collide and stay below (R + B - 1) * g, and
    the combine's address for (b, token, range) is the slot that range wrote."""
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 40))
    T = int(rng.integers(1, capi.MAX_QUERY_TOKENS + 1))
    q_per_cta = int(rng.integers(1, 3)) if T > 1 else 1
    g = -(-T // q_per_cta)
    pages = rng.integers(0, 30, size=B) * (rng.random(B) < 0.9)
    R = int(rng.integers(1, 152 // g + 1))
    piece_cost = 1
    cost = np.where(pages > 0, pages + piece_cost, 0)
    C = int(cost.sum())
    if C == 0:
        return
    prefix = np.concatenate([[0], np.cumsum(cost)])
    written = {}  # (slot, token in slot) -> (b, token, pages covered)
    covered = np.zeros((B, T), dtype=np.int64)
    for c in range(R * g):
        i, r = c // g, c % g
        lo, hi = _cta_lo(i, C, R), _cta_lo(i + 1, C, R)
        for b in range(B):
            first = prefix[b] + piece_cost
            pg0, pg1 = max(lo - first, 0), min(hi - first, pages[b])
            if pages[b] == 0 or pg0 >= pg1:
                continue
            slot = (i + b) * g + r
            assert slot < (R + B - 1) * g
            for t in range(q_per_cta):
                tau = r * q_per_cta + t
                assert (slot, t) not in written
                written[(slot, t)] = (b, tau)
                if tau < T:
                    covered[b, tau] += pg1 - pg0
    assert (covered == pages[:, None]).all()
    for b in range(B):
        if pages[b] == 0:
            continue
        first = prefix[b] + piece_cost
        cf, cl = _cta_of_cost(first, C, R), _cta_of_cost(first + pages[b] - 1, C, R)
        for tau in range(T):
            r, t = tau // q_per_cta, tau % q_per_cta
            for i in range(cf, cl + 1):
                if _cta_lo(i, C, R) < _cta_lo(i + 1, C, R):
                    assert written[((i + b) * g + r, t)] == (b, tau)
