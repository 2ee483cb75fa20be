"""Tolerances and comparisons shared by the GPU parity tests.

Floating-point bars:
- fp32 softmax: |y - y_ref| <= 1e-5 |y_ref| + 2^-126 per element (relative
  1e-5; below the smallest normal fp32 a relative bound cannot be
  represented, so the bar there is the smallest normal); m bit-exact against
  the oracle's maximum rounded to fp32; l within 1e-5 relative, taken
  relative to that same fp32 m.
- 16-bit softmax rows (y stored in bf16 / fp16): m and l as for fp32 (they
  stay fp32); y within the type's unit roundoff u (2^-8 bf16, 2^-11 fp16)
  plus the fp32 bar, relative, with an absolute floor: for fp16 half its
  smallest subnormal spacing (2^-25); for bf16 the fp32 bar's 2^-126, since
  the weights are formed in fp32 and flush below its smallest normal.
- bf16-in / fp32-accumulate attention and decode: |err| <= 2e-2 + 2e-2 |ref|
  on O and on lse (and on partial m, lse and O / l).
"""

import numpy as np

FLT_MIN = 2.0 ** -126


def f32(scale):
    """The scale as the library receives it: the ABI's scale argument is a
    C float, so the definition is evaluated with that fp32 value."""
    return float(np.float32(scale))
SOFTMAX_RTOL = 1e-5
ATTN_ATOL = 2e-2
ATTN_RTOL = 2e-2


def check_softmax(y, m, l, y_ref, m_ref, l_ref, what=""):
    y = np.asarray(y, dtype=np.float64)
    m = np.asarray(m, dtype=np.float32)
    l = np.asarray(l, dtype=np.float64)
    m32 = np.asarray(m_ref).astype(np.float32)
    bad = np.nonzero(m.view(np.uint32) != m32.view(np.uint32))[0]
    assert bad.size == 0, f"{what} m not bit-exact at rows {bad[:8]}: {m[bad[:4]]} vs {m32[bad[:4]]}"
    finite = np.isfinite(m_ref)
    with np.errstate(invalid="ignore", over="ignore"):
        l_at = np.where(finite, l_ref * np.exp(m_ref - m32.astype(np.float64)), 0.0)
    err_l = np.abs(l - l_at)
    assert np.all(err_l <= SOFTMAX_RTOL * np.abs(l_at)), \
        f"{what} l rel err {np.max(err_l / np.maximum(l_at, 1e-300)):.3e}"
    err = np.abs(y - y_ref)
    lim = SOFTMAX_RTOL * np.abs(y_ref) + FLT_MIN
    ok = err <= lim
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what} y mismatch at {idx.tolist()}: "
                             f"{[(y[tuple(i)], y_ref[tuple(i)]) for i in idx]}")
    return float(np.max(err / (np.abs(y_ref) + FLT_MIN)))


Y16_BARS = {"bf16": (2.0 ** -8, FLT_MIN), "f16": (2.0 ** -11, 2.0 ** -25)}


def check_softmax16(y, m, l, y_ref, m_ref, l_ref, kind, what=""):
    """y: the kernel's 16-bit output widened to float64."""
    check_softmax(np.zeros_like(y_ref), m, l, np.zeros_like(y_ref), m_ref, l_ref, what=what)
    u, floor = Y16_BARS[kind]
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    lim = (u + SOFTMAX_RTOL) * np.abs(y_ref) + floor
    ok = err <= lim
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what} y mismatch at {idx.tolist()}: "
                             f"{[(y[tuple(i)], y_ref[tuple(i)]) for i in idx]}")
    return float(np.max(err / (np.abs(y_ref) + floor)))


def check_attn(x, ref, what=""):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_ninf = np.isneginf(x) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_ninf, 0.0, np.abs(x - ref))
    lim = ATTN_ATOL + ATTN_RTOL * np.abs(np.where(both_ninf, 0.0, ref))
    ok = err <= lim
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what} mismatch at {idx.tolist()}: "
                             f"{[(x[tuple(i)], ref[tuple(i)]) for i in idx]} (max err {np.nanmax(err):.3e})")
    return float(np.max(err)) if err.size else 0.0


# ---------------------------------------------------------------------------
# Secondary bars for attention, decode and the partial states
#
# The spec bar above (2e-2 + 2e-2 |ref|) stays the pass/fail of record,
# but at full size it is too wide to see a lost KV tile or split: lse ~ 9
# allows +-0.2, while dropping one of attn_4k's 32 KV tiles moves lse by
# ln(31/32) = -0.032. The bars below come from the arithmetic of the kernels
# (bf16 inputs, exact products, fp32 sums) and are one to two orders of
# magnitude tighter. Each is a worst-case bound, not a fitted tolerance:
#
# * Scores. s_j = scale * q.k_j sums D exact bf16 products in fp32, in any
#   order; with u = 2^-24 and a factor 2 for any rounding mode the error is
#   at most  e_s = scale * 2 D u * ||q||_2 * max_j ||k_j||_2  (Cauchy-Schwarz
#   on sum |q_d k_jd|).  A maximum m moves by at most e_s.
# * lse = ln sum_j exp(s_j) moves by at most max_j |ds_j| <= e_s; the fp32
#   sum of the weights, the ex2 / log2 approximations and the final roundings
#   add well under 1e-5 at these magnitudes. Bar: 1e-4 + 2 e_s.
# * O = sum_j p_j v_j / l (per row, 2-norm over the head dims):
#     - O rounded to bf16:               2^-9 ||O||        (bar 2^-8 ||O||)
#     - each p_j rounded to bf16 for the P V product: |sum_j eps_j p_j v_jd| / l
#       <= 2^-9 sum_j p_j |v_jd| / l = 2^-9 A_d, A = softmax-weighted |V|
#     - the fp32 sum over n keys of the P V product:  2 n u A_d
#     - the score error moves every weight by a factor exp(+-2 e_s):
#       2 e_s (A_d + |O_d|)
#   A is the oracle's own attention with |V| in place of V.
# ---------------------------------------------------------------------------

U32 = 2.0 ** -24
LSE_FLOOR = 1e-4


def score_error_bound(q, k, scale):
    """e_s per query row: q [..., Sq, D], k [..., Sk, D] (float64 values of
    the bf16 inputs). Returns [..., Sq]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    D = q.shape[-1]
    qn = np.linalg.norm(q, axis=-1)
    kn = np.linalg.norm(k, axis=-1).max(axis=-1)
    return float(scale) * 2.0 * D * U32 * qn * kn[..., None]


def lse_bar(e_s):
    return LSE_FLOOR + 2.0 * np.asarray(e_s, dtype=np.float64)


def o_bar(ref, a_abs, e_s, n_keys):
    """Per-row bound on ||O - O_ref||_2 (last axis = head dims)."""
    ref = np.asarray(ref, dtype=np.float64)
    a_abs = np.asarray(a_abs, dtype=np.float64)
    e_s = np.asarray(e_s, dtype=np.float64)
    no = np.linalg.norm(ref, axis=-1)
    na = np.linalg.norm(a_abs, axis=-1)
    return (2.0 ** -8) * no + ((2.0 ** -9) + 2.0 * np.asarray(n_keys, dtype=np.float64) * U32) * na \
        + 2.0 * e_s * (na + no) + 1e-6


def check_lse_tight(x, ref, bar, what=""):
    """|x - ref| <= bar elementwise (both -inf counts as equal). Returns the
    largest err / bar."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bar = np.broadcast_to(np.asarray(bar, dtype=np.float64), ref.shape)
    both = np.isneginf(x) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both, 0.0, np.abs(x - ref))
    ratio = np.where(both, 0.0, err / bar)
    bad = ~(ratio <= 1.0)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what} beyond the tight bar at {idx.tolist()}: "
                             f"{[(x[tuple(i)], ref[tuple(i)], bar[tuple(i)]) for i in idx]}")
    return float(ratio.max()) if ratio.size else 0.0


def check_o_tight(x, ref, bar, what=""):
    """Per row: ||x - ref||_2 <= bar. Returns the largest ratio."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.linalg.norm(x - ref, axis=-1)
    bar = np.broadcast_to(np.asarray(bar, dtype=np.float64), err.shape)
    ratio = err / bar
    bad = ~(ratio <= 1.0)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what} O beyond the tight bar at rows {idx.tolist()}: "
                             f"{[(err[tuple(i)], bar[tuple(i)]) for i in idx]}")
    return float(ratio.max()) if ratio.size else 0.0


def report(what, **ratios):
    """One line with the largest error of each quantity as a fraction of its
    bar (shown with pytest -s or on failure)."""
    print(f"[parity] {what}: " + ", ".join(f"{k} {v:.3g}" for k, v in ratios.items()))
