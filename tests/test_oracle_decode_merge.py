"""Pins for the oracle's split-KV decode partials and the (m, l, O) merge
(CPU only)."""

import itertools
import math
import random

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def rand(shape, seed, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * mult).numpy()


# ---------------------------------------------------------------------------
# merge
# ---------------------------------------------------------------------------

def test_merge_pair_closed_form():
    a = (math.log(2.0), 1.0, np.array([1.0, 2.0]))
    b = (0.0, 1.0, np.array([4.0, -2.0]))
    m, l, O = oracle.merge_pair(a, b)
    assert m == math.log(2.0)
    assert l == pytest.approx(1.5, rel=1e-15)
    np.testing.assert_allclose(O, [1.0 + 2.0, 2.0 - 1.0], rtol=1e-15)


def test_merge_equal_maxima_adds():
    a = (0.3, 2.0, np.array([1.0]))
    b = (0.3, 5.0, np.array([7.0]))
    m, l, O = oracle.merge_pair(a, b)
    assert (m, l, O[0]) == (0.3, 7.0, 8.0)


def test_empty_partial_is_the_identity():
    a = (0.7, 3.0, np.array([1.5, -2.0]))
    e = (-math.inf, 0.0, np.zeros(2))
    for x, y in ((a, e), (e, a)):
        m, l, O = oracle.merge_pair(x, y)
        assert m == a[0] and l == a[1]
        np.testing.assert_array_equal(O, a[2])
    m, l, O = oracle.merge_pair(e, e)
    assert m == -math.inf and l == 0.0 and np.all(O == 0)


def _random_partials(n, D, seed):
    rng = np.random.default_rng(seed)
    return [(float(rng.normal() * 5), float(rng.uniform(1, 50)), rng.normal(size=D))
            for _ in range(n)]


def _tree_merge(parts, rng):
    parts = list(parts)
    while len(parts) > 1:
        i = rng.randrange(len(parts) - 1)
        parts[i:i + 2] = [oracle.merge_pair(parts[i], parts[i + 1])]
    return parts[0]


@pytest.mark.parametrize("seed", range(6))
def test_merge_associative_and_commutative(seed):
    parts = _random_partials(9, 5, seed)
    rng = random.Random(seed)
    ref = oracle.merge(np.array([[p[0] for p in parts]]), np.array([[p[1] for p in parts]]),
                       np.array([[p[2] for p in parts]]), finalize=False)
    for _ in range(5):
        shuffled = parts[:]
        rng.shuffle(shuffled)
        m, l, O = _tree_merge(shuffled, rng)
        assert m == ref[0][0]
        assert l == pytest.approx(ref[1][0], rel=1e-14)
        np.testing.assert_allclose(O, ref[2][0], rtol=1e-13, atol=1e-13)


def test_merge_finalize_and_empty_group():
    pm = np.array([[0.0, -math.inf], [-math.inf, -math.inf]])
    pl = np.array([[2.0, 0.0], [0.0, 0.0]])
    po = np.array([[[4.0], [0.0]], [[0.0], [0.0]]])
    On, m, l, lse = oracle.merge(pm, pl, po, finalize=True)
    assert On[0, 0] == 2.0 and lse[0] == pytest.approx(math.log(2.0))
    assert On[1, 0] == 0.0 and m[1] == -math.inf and l[1] == 0.0 and lse[1] == -math.inf


def test_merging_two_halves_of_a_row_equals_the_row():
    # The identity the whole method rests on: softmax state of a row equals
    # the merge of the states of its two halves.
    x = rand((40,), 50, 4.0)
    v = rand((40, 3), 51)
    def state(xs, vs):
        m = xs.max()
        w = np.exp(xs - m)
        return m, w.sum(), w @ vs
    m, l, O = oracle.merge_pair(state(x[:13], v[:13]), state(x[13:], v[13:]))
    mf, lf, Of = state(x, v)
    assert m == mf and l == pytest.approx(lf, rel=1e-14)
    np.testing.assert_allclose(O, Of, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# split bounds and decode partials
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L,S", [(1, 16), (15, 16), (16, 16), (17, 16), (1000, 16), (32768, 16), (7, 3)])
def test_split_bounds_cover_disjointly(L, S):
    covered = []
    chunk = -(-L // S)
    for j in range(S):
        lo, hi = oracle.split_bounds(L, S, j)
        assert 0 <= lo <= hi <= L
        assert hi - lo <= chunk
        covered.extend(range(lo, hi))
    assert covered == list(range(L))


def test_decode_partials_brute_force():
    B, H, Lmax, D, S = 2, 2, 11, 3, 4
    q, k, v = rand((B, H, D), 60), rand((B, H, Lmax, D), 61), rand((B, H, Lmax, D), 62)
    kv_len = np.array([11, 2])
    s = 0.8
    pm, pl, po = oracle.decode_partials(q, k, v, kv_len, S, s)
    for b, h, j in itertools.product(range(B), range(H), range(S)):
        L = kv_len[b]
        chunk = -(-L // S)
        keys = [t for t in range(L) if t // chunk == j]
        if not keys:
            assert pm[b, h, j] == -math.inf and pl[b, h, j] == 0.0
            assert np.all(po[b, h, j] == 0.0)
            continue
        sc = {t: s * sum(q[b, h, d] * k[b, h, t, d] for d in range(D)) for t in keys}
        mm = max(sc.values())
        assert pm[b, h, j] == pytest.approx(mm, rel=1e-14)
        assert pl[b, h, j] == pytest.approx(sum(math.exp(x - mm) for x in sc.values()), rel=1e-13)
        for e in range(D):
            want = sum(math.exp(sc[t] - mm) * v[b, h, t, e] for t in keys)
            assert po[b, h, j, e] == pytest.approx(want, rel=1e-12, abs=1e-13)


def test_decode_matches_torch_sdpa_and_merged_partials():
    B, H, Lmax, D, S = 3, 4, 70, 16, 16
    q, k, v = rand((B, H, D), 70), rand((B, H, Lmax, D), 71), rand((B, H, Lmax, D), 72)
    kv_len = np.array([70, 5, 33])  # 5 < 16 splits: most splits empty
    s = 1.0 / math.sqrt(D)
    O, lse = oracle.decode(q, k, v, kv_len, s)
    for b in range(B):
        L = kv_len[b]
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(q[b][:, None, :]), torch.from_numpy(k[b, :, :L]),
            torch.from_numpy(v[b, :, :L]), scale=s)[:, 0].numpy()
        np.testing.assert_allclose(O[b], ref, rtol=1e-12, atol=1e-13)
    pm, pl, po = oracle.decode_partials(q, k, v, kv_len, S, s)
    On, m, l, lse_m = oracle.merge(pm.reshape(B * H, S), pl.reshape(B * H, S),
                                   po.reshape(B * H, S, D), finalize=True)
    np.testing.assert_allclose(On.reshape(B, H, D), O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_m.reshape(B, H), lse, rtol=1e-13)
    assert np.sum(np.isinf(pm[1])) == H * (S - 5)


def test_decode_single_key_returns_that_value():
    q, k, v = rand((1, 2, 4), 80), rand((1, 2, 9, 4), 81), rand((1, 2, 9, 4), 82)
    O, lse = oracle.decode(q, k, v, np.array([1]), 0.5)
    np.testing.assert_array_equal(O[0], v[0, :, 0])
    np.testing.assert_allclose(lse[0], 0.5 * np.einsum("hd,hd->h", q[0], k[0, :, 0]), rtol=1e-15)
