"""Pins for the oracle's step-by-step online normaliser (CPU only).

The curionode page prints readouts for one worked example (64 logits in
blocks of 8); ``tests/golden/curionode_one_pass_exactly.json`` holds them with
their citation. The page's seed is not given, so the seed-specific numbers
are checked as the relations they illustrate, and a constructed input
reproduces the printed counts exactly.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from pass_attention_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
EPS = np.finfo(np.float64).eps
BOUND = 64 * EPS  # float64 rounding bound for a 64-term normaliser


@pytest.fixture(scope="module")
def golden():
    with open(os.path.join(HERE, "golden", "curionode_one_pass_exactly.json")) as f:
        return json.load(f)


def strict_block_records(x, block):
    """Count blocks after the first whose maximum is a new strict record,
    computed independently of the oracle with numpy's running maximum."""
    x = np.asarray(x, dtype=np.float64)
    bmax = np.array([x[i:i + block].max() for i in range(0, len(x), block)])
    prev = np.maximum.accumulate(bmax)[:-1]
    return int(np.sum(bmax[1:] > prev))


def two_pass_l(x, scale=1.0):
    _, m, l = oracle.softmax_rows(np.asarray(x, dtype=np.float64)[None, :], scale=scale)
    return m[0], l[0]


def page_logits():
    w = workloads.ROW64
    return workloads.logits(w.rows, w.cols, w.mult, w.seed).numpy()[0].astype(np.float64)


def test_worked_example_counts_and_error(golden):
    p = golden["printed"]
    x = page_logits()
    assert len(x) == golden["n_logits"]
    m, l, updates, rescales = oracle.online_normaliser(x, golden["block"])
    assert updates == p["block_updates"] == 8
    assert rescales == strict_block_records(x, golden["block"])
    m2, l2 = two_pass_l(x)
    assert m == m2
    rel = abs(l / l2 - 1.0)
    assert rel <= BOUND
    assert p["normaliser_rel_error_vs_two_pass"] <= BOUND  # the page's figure obeys it too


def test_worked_example_scaled_up(golden):
    p = golden["printed"]
    x = page_logits()
    s = p["scale_up"]
    naive = oracle.naive_normaliser(x, scale=s)
    assert int(math.isfinite(naive)) == p["naive_sum_finite_at_scale_up"] == 0
    m, l, _, _ = oracle.online_normaliser(x, golden["block"], scale=s)
    m2, l2 = two_pass_l(x, scale=s)
    assert math.isfinite(l) and math.isfinite(m)
    assert abs(l / l2 - 1.0) <= BOUND
    assert p["online_rel_error_at_scale_up"] <= BOUND


def test_worked_example_blocks_of_one(golden):
    x = page_logits()
    m8, l8, _, _ = oracle.online_normaliser(x, 8)
    m1, l1, updates, rescales = oracle.online_normaliser(x, 1)
    assert updates == 64
    assert rescales == strict_block_records(x, 1)  # once per new maximum
    assert m1 == m8 and abs(l1 / l8 - 1.0) <= BOUND  # "the result is the same"


def test_constructed_input_reproduces_printed_counts(golden):
    # Two new maxima after the first element, in distinct blocks of 8: the
    # page's "rescales 2 times" for blocks of 8 and blocks of one.
    p = golden["printed"]
    rng = np.random.default_rng(0)
    x = -np.abs(rng.standard_normal(64)) - 1.0  # everything below 0 ...
    x[0] = 0.0       # first element is the first maximum
    x[20] = 0.5      # a record in block 2
    x[45] = 1.5      # a record in block 5
    _, _, upd8, r8 = oracle.online_normaliser(x, 8)
    _, _, upd1, r1 = oracle.online_normaliser(x, 1)
    assert upd8 == p["block_updates"]
    assert r8 == p["rescalings"] == 2
    assert r1 == p["block_one_rescalings"] == 2


@pytest.mark.parametrize("block", [1, 2, 3, 7, 8, 64])
def test_block_size_invariance_and_record_count(block):
    rng = np.random.default_rng(100 + block)
    x = rng.standard_normal(64)
    m, l, updates, rescales = oracle.online_normaliser(x, block)
    m2, l2 = two_pass_l(x)
    assert updates == -(-64 // block)
    assert rescales == strict_block_records(x, block)
    assert m == m2
    assert abs(l / l2 - 1.0) <= BOUND


def test_increasing_row_closed_form():
    # x_i = i*d: every element is a new record; l = sum_k exp(-k d), k=0..n-1.
    n, d = 40, 0.3
    x = np.arange(n) * d
    m, l, updates, rescales = oracle.online_normaliser(x, 1)
    assert rescales == n - 1
    assert m == x[-1]
    closed = (1 - math.exp(-n * d)) / (1 - math.exp(-d))
    assert l == pytest.approx(closed, rel=BOUND)


def test_constant_row_never_rescales():
    m, l, _, rescales = oracle.online_normaliser([0.25] * 50, 4)
    assert rescales == 0 and m == 0.25 and l == pytest.approx(50.0, rel=BOUND)


def test_masked_first_blocks_are_guarded():
    # An all -inf first block would form -inf - -inf = NaN without the guard
    # (roadmapper "Online softmax", "Initialise honestly").
    x = [-math.inf] * 8 + [0.0, 1.0, 2.0] + [-math.inf] * 5
    m, l, updates, rescales = oracle.online_normaliser(x, 8)
    assert m == 2.0 and l == pytest.approx(1 + math.exp(-1) + math.exp(-2), rel=BOUND)
    assert rescales == 0
    m, l, _, _ = oracle.online_normaliser([-math.inf] * 5, 2)
    assert m == -math.inf and l == 0.0
