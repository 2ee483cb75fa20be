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
