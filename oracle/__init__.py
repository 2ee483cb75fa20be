"""fp64 CPU oracle for the online-softmax hot path.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` use it. It shares no code with
``pass_attention_gb300`` and imports nothing from it.

The online recurrence reaches the plain two-pass safe-softmax result exactly
in exact arithmetic (roadmapper "Online softmax", section "Why the values are
preserved"; curionode "The Online Softmax", introduction: at the end the
running sum is exactly the safe normaliser).  So the reference functions here
are the plain definitions, written out in float64, with no online recurrence:

* :func:`softmax_rows`        -- safe softmax of each row, three plain passes.
* :func:`attention`           -- softmax(scale * Q K^T) V with the full score
                                 row materialised, plus log-sum-exp.
* :func:`decode_partials`     -- the per-chunk (m, l, O) of one query against
                                 each split of its keys, by the definition.
* :func:`decode`              -- single-query attention over kv_len keys.
* :func:`merge`               -- the n-ary merge of (m, l, O) partials.

For the tests that pin the pages' worked example and failure modes, it also
carries small pure-Python routines that follow the pages' recurrence step by
step: :func:`naive_normaliser`, :func:`online_normaliser`,
:func:`online_attention_row` and :func:`merge_pair`.

Units.  ``m`` is the row maximum of ``scale * x`` in natural units, ``l`` is
the sum of ``exp(scale * x - m)`` (the normaliser taken relative to the true
maximum, as the curionode page's workshop compares it), and
``lse = m + ln(l)``.

Readings of points the pages leave open (each also listed in the design
notes):

* An empty or fully masked row has ``m = -inf``, ``l = 0``, ``O = 0`` and
  ``lse = -inf``; its normalised output is 0, not NaN (roadmapper "Online
  softmax", "Initialise honestly", names the NaN but not the guard).
* A causal mask lets query ``i`` see keys ``0..i`` (``Sq == Sk``).
* Split ``j`` of a sequence of ``L`` keys cut into ``S`` splits covers keys
  ``[j*ceil(L/S), min(L, (j+1)*ceil(L/S)))``; a split past the end is empty.
* A "rescaling" is a block whose maximum strictly exceeds a finite running
  maximum (curionode "The Online Softmax", "One pass, exactly").

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, library routines (torch float64) or the
pages' printed worked example; none is "parity unpinned".
"""

from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

NEG_INF = -math.inf

__all__ = [
    "softmax_rows",
    "attention",
    "decode_partials",
    "decode",
    "merge",
    "merge_pair",
    "naive_normaliser",
    "online_normaliser",
    "online_attention_row",
    "split_bounds",
]


# ---------------------------------------------------------------------------
# Safe softmax, by definition
# ---------------------------------------------------------------------------

def _softmax_lastdim(z: np.ndarray):
    """Safe softmax along the last axis of float64 scores ``z``.

    Three plain passes (curionode "The Online Softmax", introduction): the
    maximum ``m``, the sum ``l`` of ``exp(z - m)``, then ``exp(z - m) / l``.
    Entries equal to -inf carry zero weight. A slice that is entirely -inf
    gives ``m = -inf, l = 0`` and zero weights.
    """
    m = z.max(axis=-1)
    finite = np.isfinite(m)
    shift = np.where(finite, m, 0.0)
    e = np.exp(z - shift[..., None])  # exp(-inf) = 0 for masked entries
    l = e.sum(axis=-1)
    safe_l = np.where(l > 0.0, l, 1.0)
    y = np.where(finite[..., None], e / safe_l[..., None], 0.0)
    l = np.where(finite, l, 0.0)
    return y, m, l


def softmax_rows(x, scale: float = 1.0):
    """Row-wise safe softmax of ``scale * x`` in float64.

    x: array-like [rows, cols] (any real dtype; converted exactly to float64).
    Returns ``(y, m, l)``: y [rows, cols], m [rows] = max_j scale*x[r, j],
    l [rows] = sum_j exp(scale*x[r, j] - m[r]).

    The product ``scale * x`` of two float32 numbers is exact in float64, so
    ``m`` rounded to float32 is the maximum of the float32 products.
    """
    z = np.asarray(x, dtype=np.float64) * float(scale)
    if z.ndim != 2:
        raise ValueError("softmax_rows expects a 2-D array")
    return _softmax_lastdim(z)


def naive_normaliser(x, scale: float = 1.0) -> float:
    """sum_j exp(scale * x_j) with no shift, in float64.

    The unsafe form the curionode page contrasts with the safe one: it
    overflows once an exponent passes about 709 (its "Workshop" section).
    """
    with np.errstate(over="ignore"):
        return float(np.exp(np.asarray(x, dtype=np.float64) * float(scale)).sum())


# ---------------------------------------------------------------------------
# The pages' recurrence, step by step (tests only, small inputs)
# ---------------------------------------------------------------------------

def online_normaliser(x: Sequence[float], block: int, scale: float = 1.0):
    """One pass over ``x`` in blocks of ``block``, carrying (m, l).

    Per block (curionode "The Online Softmax", introduction; roadmapper
    "Online softmax", "The recurrence"): the new maximum is the larger of the
    running maximum and the block maximum; the running sum is multiplied by
    exp(m_old - m_new) and the block's exp(x - m_new) are added.

    Starts from m = -inf, l = 0 ("Initialise honestly"). A block whose new
    maximum is still -inf (all entries masked) leaves the state unchanged
    instead of forming -inf - -inf.

    Returns ``(m, l, updates, rescales)``: ``updates`` counts the blocks
    folded in, ``rescales`` the blocks whose maximum strictly exceeds a
    finite running maximum.
    """
    if block < 1:
        raise ValueError("block must be >= 1")
    vals = [float(scale) * float(v) for v in x]
    m = NEG_INF
    l = 0.0
    updates = 0
    rescales = 0
    for start in range(0, len(vals), block):
        blk = vals[start:start + block]
        m_new = max(m, max(blk))
        updates += 1
        if m_new == NEG_INF:
            continue
        if m != NEG_INF and m_new > m:
            rescales += 1
        c = math.exp(m - m_new)  # exp(-inf) = 0 on the first non-empty block
        l = l * c + sum(math.exp(v - m_new) for v in blk)
        m = m_new
    return m, l, updates, rescales


def online_attention_row(q: Sequence[float], K, V, scale: float, block: int,
                         mask=None):
    """(m, l, O) recurrence for one query row over key blocks, in float64.

    Per tile of scores S (metalworking "Online Softmax", the five-line
    recurrence; roadmapper "Online softmax", "The recurrence"):
    m_new = max(m, max S); c = exp(m - m_new); P = exp(S - m_new);
    l = l*c + sum P; O = O*c + P V; m = m_new. After the last tile the
    caller divides O by l.

    ``mask`` (optional, bool per key, True = visible) sets hidden keys'
    scores to -inf; a tile whose keys are all hidden so far leaves the state
    unchanged (the guard "Initialise honestly" calls for).
    Returns ``(m, l, O_unnormalised)``.
    """
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    n = K.shape[0]
    if mask is None:
        mask = np.ones(n, dtype=bool)
    m = NEG_INF
    l = 0.0
    O = np.zeros(V.shape[1], dtype=np.float64)
    for start in range(0, n, block):
        idx = range(start, min(n, start + block))
        S = [float(scale) * float(np.dot(q, K[j])) if mask[j] else NEG_INF
             for j in idx]
        m_new = max(m, max(S))
        if m_new == NEG_INF:
            continue  # fully masked tile so far: nothing to add, no NaN
        c = math.exp(m - m_new)
        P = [math.exp(s - m_new) for s in S]
        l = l * c + sum(P)
        O = O * c + sum(p * V[j] for p, j in zip(P, idx))
        m = m_new
    return m, l, O


# ---------------------------------------------------------------------------
# Attention, materialised
# ---------------------------------------------------------------------------

def _as64(t) -> np.ndarray:
    return np.asarray(t, dtype=np.float64)


def attention(q, k, v, scale: float, causal: bool = False,
              rows: Iterable[tuple[int, int, int]] | None = None):
    """softmax(scale * Q K^T [+ causal mask]) V with full score rows, float64.

    q [B, H, Sq, D], k [B, H, Sk, D], v [B, H, Sk, Dv]: the (bf16) inputs as
    exact float64 values. The score row S_i = scale * q_i K^T is formed in
    full (what the tiled method avoids storing: curionode "The Online
    Softmax", introduction), masked entries are set to -inf, then the safe
    softmax of each row weights the rows of V.

    Causal: query i sees keys 0..i (requires Sq == Sk).

    Returns ``(O, lse)``; O [B, H, Sq, Dv], lse [B, H, Sq] = m + ln(l).
    With ``rows`` given (an iterable of (b, h, i)), only those rows are
    computed and the results are O [n, Dv], lse [n] in the order given.
    """
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if causal and Sq != Sk:
        raise ValueError("causal attention is defined here for Sq == Sk")

    if rows is not None:
        rows = [tuple(int(x) for x in r) for r in rows]
        O = np.zeros((len(rows), v.shape[3]), dtype=np.float64)
        lse = np.zeros(len(rows), dtype=np.float64)
        groups: dict = {}
        for n, (b, h, i) in enumerate(rows):
            groups.setdefault((b, h), []).append((n, i))
        for (b, h), items in groups.items():
            idx = np.array([n for n, _ in items])
            qi = np.array([i for _, i in items])
            S = float(scale) * (q[b, h, qi] @ k[b, h].T)  # score rows of these queries
            if causal:
                S[np.arange(Sk)[None, :] > qi[:, None]] = NEG_INF
            W, m, l = _softmax_lastdim(S)
            O[idx] = W @ v[b, h]
            with np.errstate(divide="ignore"):
                lse[idx] = np.where(l > 0.0, m + np.log(np.where(l > 0.0, l, 1.0)), NEG_INF)
        return O, lse

    O = np.zeros((B, H, Sq, v.shape[3]), dtype=np.float64)
    lse = np.zeros((B, H, Sq), dtype=np.float64)
    if causal:
        mask = np.triu(np.ones((Sq, Sk), dtype=bool), k=1)  # j > i is hidden
    for b in range(B):
        for h in range(H):
            S = float(scale) * (q[b, h] @ k[b, h].T)
            if causal:
                S[mask] = NEG_INF
            W, m, l = _softmax_lastdim(S)
            O[b, h] = W @ v[b, h]
            with np.errstate(divide="ignore"):
                lse[b, h] = np.where(l > 0.0, m + np.log(l), NEG_INF)
    return O, lse


# ---------------------------------------------------------------------------
# Split-KV decode and the merge
# ---------------------------------------------------------------------------

def split_bounds(L: int, num_splits: int, j: int) -> tuple[int, int]:
    """Key range [lo, hi) of split j when L keys are cut into num_splits
    chunks of ceil(L / num_splits); a split past the end is empty."""
    chunk = -(-int(L) // int(num_splits))
    lo = min(int(L), j * chunk)
    hi = min(int(L), (j + 1) * chunk)
    return lo, hi


def decode_partials(q, k, v, kv_len, num_splits: int, scale: float):
    """Per-split partial results of single-query attention, by definition.

    q [B, H, D], k [B, H, Lmax, D], v [B, H, Lmax, Dv], kv_len [B] (1..Lmax).
    For split j of batch b the keys are those of :func:`split_bounds`; its
    partial is m = max of the scores s_t = scale * q.k_t over the split,
    l = sum exp(s_t - m), O = sum exp(s_t - m) v_t (not divided by l). An
    empty split is (-inf, 0, 0). These are the partial softmaxes that
    split-KV decode kernels compute and later merge (metalworking "Online
    Softmax", closing note).

    Returns part_m [B, H, S], part_l [B, H, S], part_o [B, H, S, Dv].
    """
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    kv_len = np.asarray(kv_len).astype(np.int64)
    B, H, D = q.shape
    Dv = v.shape[3]
    S = int(num_splits)
    part_m = np.full((B, H, S), NEG_INF, dtype=np.float64)
    part_l = np.zeros((B, H, S), dtype=np.float64)
    part_o = np.zeros((B, H, S, Dv), dtype=np.float64)
    for b in range(B):
        L = int(kv_len[b])
        scores = float(scale) * np.einsum("hd,hld->hl", q[b], k[b, :, :L])
        for j in range(S):
            lo, hi = split_bounds(L, S, j)
            if hi <= lo:
                continue
            s = scores[:, lo:hi]
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            part_m[b, :, j] = m
            part_l[b, :, j] = e.sum(axis=1)
            part_o[b, :, j] = np.einsum("hl,hld->hd", e, v[b, :, lo:hi])
    return part_m, part_l, part_o


def decode(q, k, v, kv_len, scale: float):
    """Single-query attention of q [B, H, D] over the first kv_len[b] keys.

    The definition with the whole score row: returns O [B, H, Dv] and
    lse [B, H].
    """
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    kv_len = np.asarray(kv_len).astype(np.int64)
    B, H, D = q.shape
    O = np.zeros((B, H, v.shape[3]), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    for b in range(B):
        L = int(kv_len[b])
        s = float(scale) * np.einsum("hd,hld->hl", q[b], k[b, :, :L])
        w, m, l = _softmax_lastdim(s)
        O[b] = np.einsum("hl,hld->hd", w, v[b, :, :L])
        lse[b] = m + np.log(l)
    return O, lse


def merge(part_m, part_l, part_o, finalize: bool = True):
    """Merge partial softmax results over the last partial axis, in float64.

    part_m, part_l [G, S]; part_o [G, S, D]. The merged state is the n-ary
    form of the pairwise identity (curionode "The Online Softmax", "One pass,
    exactly": the rescaling identity for pairs is associative):
    m = max_s m_s, l = sum_s l_s exp(m_s - m), O = sum_s O_s exp(m_s - m).
    A group whose partials are all empty gives (-inf, 0, 0).

    finalize=False returns (m, l, O); finalize=True returns
    (O / l, m, l, lse) with O / l = 0 and lse = -inf for an empty group.
    """
    pm = _as64(part_m)
    pl = _as64(part_l)
    po = _as64(part_o)
    m = pm.max(axis=-1)
    finite = np.isfinite(m)
    shift = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(pm), np.exp(pm - shift[..., None]), 0.0)
    l = (w * pl).sum(axis=-1)
    O = (w[..., None] * po).sum(axis=-2)
    l = np.where(finite, l, 0.0)
    O = np.where(finite[..., None], O, 0.0)
    if not finalize:
        return m, l, O
    safe_l = np.where(l > 0.0, l, 1.0)
    On = np.where((l > 0.0)[..., None], O / safe_l[..., None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0.0, m + np.log(safe_l), NEG_INF)
    return On, m, l, lse


def merge_pair(a, b):
    """The pairwise merge of two partial states (m, l, O), float64.

    m = max(m1, m2); each side is rescaled by exp(m_k - m) before the sums
    and outputs are added. Two empty sides give (-inf, 0, 0).
    """
    m1, l1, O1 = a
    m2, l2, O2 = b
    m = max(m1, m2)
    if m == NEG_INF:
        return NEG_INF, 0.0, np.zeros_like(np.asarray(O1, dtype=np.float64))
    c1 = math.exp(m1 - m)
    c2 = math.exp(m2 - m)
    return m, l1 * c1 + l2 * c2, np.asarray(O1, np.float64) * c1 + np.asarray(O2, np.float64) * c2
