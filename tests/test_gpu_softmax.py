"""os_softmax_rows against the oracle, element by element (GPU)."""

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, f32

pytestmark = pytest.mark.gpu


def run(x, scale):
    y, m, l = oss.softmax_rows(x, scale)
    torch.cuda.synchronize()
    return y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()


def test_worked_example_row64():
    w = workloads.ROW64
    x = workloads.logits(w.rows, w.cols, w.mult, w.seed, device="cuda")
    y, m, l = run(x, w.scale)
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(w.scale)), what="row64")


SHAPES = [(1, 1), (3, 3), (5, 7), (37, 1000), (64, 1024), (9, 1025), (16, 4096), (8, 8195),
          (4, 16384), (3, 16385), (2, 40003)]


@pytest.mark.parametrize("rows,cols", SHAPES)
# 0.1 and 10 make the low part of scale*log2(e) negative, the case in which
# a masked or padding entry must not turn the FMA exponent into NaN
@pytest.mark.parametrize("scale", [1.0, 0.125, 3.0, 0.1, 10.0])
def test_shapes_and_scales_aligned(rows, cols, scale):
    # leading dimension rounded up to 4 floats: the 16-byte (register-resident
    # up to 16384 columns) path, with a ragged tail when cols % 4 != 0
    ld = (cols + 3) // 4 * 4
    x = workloads.logits(rows, ld, 10.0, seed=rows * 7919 + cols, device="cuda")[:, :cols]
    y = torch.empty((rows, ld), device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows(x, scale, y=y)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(scale)), what=f"{rows}x{cols}")


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 3), (5, 7), (9, 1025), (8, 8195), (2, 40003)])
def test_shapes_unaligned(rows, cols):
    # dense rows whose length is not a multiple of 4, and a base offset by one
    # float: the scalar streaming path
    x = workloads.logits(rows, cols, 10.0, seed=rows + cols, device="cuda")
    y, m, l = run(x, 0.3)
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(0.3)), what=f"unaligned {rows}x{cols}")
    buf = workloads.logits(1, rows * cols + 1, 10.0, seed=3, device="cuda")
    x1 = buf[0, 1:].view(rows, cols)
    y, m, l = run(x1, 1.0)
    check_softmax(y, m, l, *oracle.softmax_rows(x1.cpu().numpy(), f32(1.0)), what="offset base")


@pytest.mark.parametrize("cols,pad", [(1000, 8), (8192, 4), (20000, 12)])
def test_leading_dimension(cols, pad):
    big = workloads.logits(6, cols + pad, 10.0, seed=cols, device="cuda")
    x = big[:, :cols]
    yb = torch.full((6, cols + pad), 7.0, device="cuda")
    y, m, l = oss.softmax_rows(x, 1.0, y=yb[:, :cols])
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(1.0)), what="ld")
    assert torch.all(yb[:, cols:] == 7.0)  # padding untouched


@pytest.mark.parametrize("cols", [64, 8192, 20000])
@pytest.mark.parametrize("scale", [1.0, 0.1])
def test_masked_entries_and_empty_rows(cols, scale):
    x = workloads.logits(8, cols, 10.0, seed=cols + 1, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.3] = -float("inf")
    x[2] = -float("inf")                  # an entirely masked row
    x[5, : cols // 2] = -float("inf")     # masked first half (first blocks empty)
    y, m, l = run(x, scale)
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(scale)), what="masked")
    assert m[2] == -np.inf and l[2] == 0.0 and np.all(y[2] == 0.0)
    assert not np.any(np.isnan(y))


def test_extreme_logits_stay_finite():
    # logits spread by thousands: an unshifted exp overflows, the online form does not
    x = workloads.logits(4, 4096, 1000.0, seed=9, device="cuda")
    y, m, l = run(x, 1.0)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(l))
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(1.0)), what="x1000")


@pytest.mark.slow
def test_full_size_softmax_32k_every_row():
    w = workloads.SOFTMAX_32K
    x = workloads.logits(w.rows, w.cols, w.mult, w.seed, device="cuda")
    y, m, l = oss.softmax_rows(x, w.scale)
    torch.cuda.synchronize()
    worst = 0.0
    step = 2048
    for r0 in range(0, w.rows, step):
        xs = x[r0:r0 + step].cpu().numpy()
        ref = oracle.softmax_rows(xs, f32(w.scale))
        worst = max(worst, check_softmax(y[r0:r0 + step].cpu().numpy(), m[r0:r0 + step].cpu().numpy(),
                                         l[r0:r0 + step].cpu().numpy(), *ref, what=f"rows {r0}+"))
    print(f"softmax_32k worst relative error {worst:.3e}")


@pytest.mark.parametrize("rows,cols,chunk", [(1000, 4096, 300), (37, 1000, None), (5, 7, 2)])
def test_from_host_pipelined_matches_device_call(rows, cols, chunk):
    # os_softmax_rows_from_host copies and computes in row blocks on three
    # streams; every row sees the same kernel, so the results are identical
    x = workloads.logits(rows, cols, 10.0, seed=rows + cols, device="cuda")
    y_ref, m_ref, l_ref = oss.softmax_rows(x, 0.5)
    torch.cuda.synchronize()
    yh, mh, lh = oss.softmax_rows_from_host(x.cpu().pin_memory(), 0.5, chunk_rows=chunk)
    assert torch.equal(yh, y_ref.cpu()) and torch.equal(mh, m_ref.cpu()) and torch.equal(lh, l_ref.cpu())


def test_from_host_c_call_without_m_and_l_after_prior_work():
    # the C call with no m and l, in blocks that do not divide the rows; the
    # device staging buffer is overwritten on the stream just before the call,
    # so an upload that did not wait for that work would leave NaN behind
    import ctypes
    rows, cols = 301, 2500
    x = workloads.logits(rows, cols, 10.0, seed=17, device="cuda")
    y_ref, _, _ = oss.softmax_rows(x, 0.7)
    torch.cuda.synchronize()
    xh = x.cpu().pin_memory()
    yh = torch.empty((rows, cols), dtype=torch.float32, pin_memory=True)
    x_dev = torch.empty_like(x)
    y_dev = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    x_dev.fill_(float("nan"))
    st = oss.load().os_softmax_rows_from_host(
        xh.data_ptr(), yh.data_ptr(), None, None, x_dev.data_ptr(), y_dev.data_ptr(), None, None,
        rows, cols, ctypes.c_float(0.7), 64, stream.cuda_stream)
    assert st == 0, oss.load().os_status_string(st)
    stream.synchronize()
    assert oss.check_device_error() == 0
    assert torch.equal(yh, y_ref.cpu())
    assert torch.equal(x_dev, x) and torch.equal(y_dev, y_ref)
