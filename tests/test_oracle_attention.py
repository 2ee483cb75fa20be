"""Pins for the oracle's materialised attention and its step-by-step
recurrence, plus mutation tests (CPU only).

The mutation tests plant each failure the roadmapper page lists ("Things
that break", "Initialise honestly") in a copy of the oracle's online routine
and check that the same checks that pass the oracle reject the copy.
"""

import itertools
import math

import numpy as np
import scipy.special
import pytest
import torch
import torch.nn.functional as F

import oracle

LOG2E = 1.0 / math.log(2.0)


def rand(shape, seed, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * mult).numpy()


# ---------------------------------------------------------------------------
# Closed forms and brute force
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    B, H, S, D = 1, 2, 9, 4
    q = np.zeros((B, H, S, D))
    k = rand((B, H, S, D), 1)
    v = rand((B, H, S, D), 2)
    O, lse = oracle.attention(q, k, v, scale=0.3, causal=causal)
    for i in range(S):
        n = i + 1 if causal else S
        np.testing.assert_allclose(O[:, :, i], v[:, :, :n].mean(axis=2), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), rtol=1e-14)


def test_causal_first_row_is_first_value():
    q, k, v = rand((2, 3, 7, 5), 3), rand((2, 3, 7, 5), 4), rand((2, 3, 7, 5), 5)
    O, lse = oracle.attention(q, k, v, scale=0.7, causal=True)
    np.testing.assert_array_equal(O[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.7 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), rtol=1e-14)


def test_all_ones_values():
    q, k = rand((1, 1, 6, 3), 6, 4.0), rand((1, 1, 6, 3), 7, 4.0)
    v = np.ones((1, 1, 6, 3))
    for causal in (False, True):
        O, _ = oracle.attention(q, k, v, scale=1.0, causal=causal)
        np.testing.assert_allclose(O, 1.0, rtol=1e-14)


def test_brute_force_tiny():
    B, H, Sq, Sk, D, Dv = 2, 2, 3, 5, 4, 3
    q, k, v = rand((B, H, Sq, D), 8), rand((B, H, Sk, D), 9), rand((B, H, Sk, Dv), 10)
    s = 0.6
    O, lse = oracle.attention(q, k, v, scale=s)
    for b, h, i in itertools.product(range(B), range(H), range(Sq)):
        scores = [s * sum(q[b, h, i, d] * k[b, h, j, d] for d in range(D)) for j in range(Sk)]
        total = sum(math.exp(x) for x in scores)
        assert lse[b, h, i] == pytest.approx(math.log(total), rel=1e-13)
        for e in range(Dv):
            want = sum(math.exp(scores[j]) * v[b, h, j, e] for j in range(Sk)) / total
            assert O[b, h, i, e] == pytest.approx(want, rel=1e-12, abs=1e-14)


@pytest.mark.parametrize("causal,Sq,Sk", [(False, 17, 29), (False, 32, 32), (True, 40, 40)])
def test_matches_torch_sdpa_float64(causal, Sq, Sk):
    B, H, D = 2, 3, 16
    q = torch.from_numpy(rand((B, H, Sq, D), 11))
    k = torch.from_numpy(rand((B, H, Sk, D), 12))
    v = torch.from_numpy(rand((B, H, Sk, D), 13))
    s = 1.0 / math.sqrt(D)
    O, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), scale=s, causal=causal)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=s).numpy()
    np.testing.assert_allclose(O, ref, rtol=1e-12, atol=1e-13)
    scores = torch.einsum("bhqd,bhkd->bhqk", q, k) * s
    if causal:
        scores = scores.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(1), -math.inf)
    # scipy's logsumexp, not torch's: torch.logsumexp on float64 CPU tensors
    # returned results 1.6e-10 off (relative) in a few percent of fresh
    # processes on this host, with its input scores exact to 1e-15
    np.testing.assert_allclose(lse, scipy.special.logsumexp(scores.numpy(), axis=-1), rtol=1e-13)


def test_row_subset_matches_full():
    q, k, v = rand((2, 2, 12, 8), 14), rand((2, 2, 12, 8), 15), rand((2, 2, 12, 8), 16)
    O, lse = oracle.attention(q, k, v, scale=0.4, causal=True)
    rows = [(0, 1, 0), (1, 0, 11), (1, 1, 5)]
    Os, ls = oracle.attention(q, k, v, scale=0.4, causal=True, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(Os[n], O[b, h, i], rtol=1e-14, atol=1e-15)
        assert ls[n] == pytest.approx(lse[b, h, i], rel=1e-14)


# ---------------------------------------------------------------------------
# The step-by-step recurrence, and mutants of it
# ---------------------------------------------------------------------------

def online_cases():
    """(q, K, V, scale, block, mask) cases that together separate a correct
    recurrence from each planted failure."""
    D = 8
    cases = []
    # 1. a single tile
    cases.append((rand((D,), 20), rand((16, D), 21), rand((16, D), 22), 0.5, 16, None))
    # 2. several tiles whose maximum rises tile after tile
    q = np.ones(D)
    K = np.repeat(np.linspace(-1.0, 1.0, 6)[:, None], D, axis=1)
    K = np.repeat(K, 4, axis=0) + rand((24, D), 23) * 0.01
    cases.append((q, K, rand((24, D), 24), 1.0, 4, None))
    # 3. scores that fall by more than 709 from one tile to the next
    K = np.concatenate([np.full((4, D), 120.0), np.zeros((4, D)), rand((4, D), 25)])
    cases.append((np.ones(D), K, rand((12, D), 26), 1.0, 4, None))
    # 4. a fully masked first tile (what a causal diagonal-first order gives)
    mask = np.array([False] * 4 + [True] * 8)
    cases.append((rand((D,), 27), rand((12, D), 28), rand((12, D), 29), 0.7, 4, mask))
    # 5. random, ragged tail
    cases.append((rand((D,), 30), rand((37, D), 31, 3.0), rand((37, D), 32), 0.35, 8, None))
    return cases


def reference_row(q, K, V, scale, mask):
    s = scale * (K @ q)
    if mask is not None:
        s = np.where(mask, s, -math.inf)
    _, m, l = oracle.softmax_rows(s[None, :])
    w = np.exp(s - m[0]) / l[0]
    return w @ V, m[0] + math.log(l[0])


def routine_passes(fn):
    """True when ``fn`` (an online (m, l, O) routine) agrees with the
    materialised definition on every case."""
    for q, K, V, scale, block, mask in online_cases():
        with np.errstate(all="ignore"):
            m, l, O = fn(q, K, V, scale, block, mask)
            if not (np.isfinite(l) and l > 0 and np.all(np.isfinite(O))):
                return False
            o_ref, lse_ref = reference_row(q, K, V, scale, mask)
            if not np.allclose(O / l, o_ref, rtol=1e-11, atol=1e-12):
                return False
            if not math.isclose(m + math.log(l), lse_ref, rel_tol=1e-12, abs_tol=1e-12):
                return False
    return True


def test_oracle_recurrence_passes_the_checks():
    assert routine_passes(oracle.online_attention_row)


@pytest.mark.parametrize("block", [1, 3, 5, 16, 64])
def test_recurrence_is_block_size_invariant(block):
    q, K, V = rand((8,), 40), rand((50, 8), 41, 2.0), rand((50, 8), 42)
    m, l, O = oracle.online_attention_row(q, K, V, 0.5, block)
    o_ref, lse_ref = reference_row(q, K, V, 0.5, None)
    np.testing.assert_allclose(O / l, o_ref, rtol=1e-12, atol=1e-13)
    assert m + math.log(l) == pytest.approx(lse_ref, rel=1e-13)


def _generic(q, K, V, scale, block, mask, *, rescale_o=True, mixed_base=False,
             carry_max=True, guard=True):
    """A copy of the recurrence with switches that plant the page's bugs."""
    n = K.shape[0]
    if mask is None:
        mask = np.ones(n, dtype=bool)
    m, l, O = -math.inf, 0.0, np.zeros(V.shape[1])
    for start in range(0, n, block):
        idx = list(range(start, min(n, start + block)))
        S = [scale * float(np.dot(q, K[j])) if mask[j] else -math.inf for j in idx]
        if mixed_base:
            S = [x * LOG2E for x in S]  # log2(e) folded into the scores ...
        m_new = max(m, max(S)) if carry_max else max(S)
        if guard and m_new == -math.inf:
            continue
        if mixed_base:
            c = math.exp(m - m_new) if m != -math.inf else 0.0  # ... but alpha in base e
            P = [2.0 ** (x - m_new) for x in S]
        else:
            with np.errstate(all="ignore"):
                c = float(np.exp(np.float64(m) - np.float64(m_new)))
                P = [float(np.exp(np.float64(x) - np.float64(m_new))) for x in S]
        l = l * c + sum(P)
        contrib = sum(p * V[j] for p, j in zip(P, idx))
        O = (O * c if rescale_o else O) + contrib
        m = m_new
    if mixed_base:
        m = m / LOG2E
    return m, l, O


def test_generic_copy_without_bugs_passes():
    assert routine_passes(_generic)


def test_mutant_rescale_l_but_not_o_is_caught():
    mutant = lambda *a: _generic(*a, rescale_o=False)
    # right on a single tile, so a short test passes ...
    q, K, V, scale, block, mask = online_cases()[0]
    m, l, O = mutant(q, K, V, scale, block, mask)
    np.testing.assert_allclose(O / l, reference_row(q, K, V, scale, mask)[0], rtol=1e-12)
    # ... and caught once the maximum rises across tiles
    assert not routine_passes(mutant)


def test_mutant_mixed_bases_is_caught():
    assert not routine_passes(lambda *a: _generic(*a, mixed_base=True))


def test_mutant_max_recomputed_per_block_is_caught():
    assert not routine_passes(lambda *a: _generic(*a, carry_max=False))


def test_mutant_without_empty_tile_guard_is_caught():
    assert not routine_passes(lambda *a: _generic(*a, guard=False))
