"""Rows beyond a cluster's shared memory (over 1.6 MB) with a workspace:
the cooperative kernel that takes a few rows at a time over the whole GPU,
merges the slices' (max, sum) states at a grid barrier and reads each slice
a second time from L2 (GPU).

The cases cover groups that do not divide the rows, rows off the 16-byte
grid, masked entries and whole masked rows, 16-bit rows, agreement with the
call without a workspace (which streams the rows twice from HBM), and the
64 x 2^22 fp32 matrix the bench measures, on sampled rows."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, check_softmax16, f32

pytestmark = pytest.mark.gpu


def no_workspace(x, scale):
    """os_softmax_rows without a workspace (the twice-streaming kernel)."""
    rows, cols = x.shape
    y = torch.empty_like(x)
    m = torch.empty(rows, device=x.device)
    l = torch.empty(rows, device=x.device)
    st = oss.load().os_softmax_rows(x.data_ptr(), y.data_ptr(), m.data_ptr(), l.data_ptr(), rows,
                                    cols, x.stride(0), y.stride(0), ctypes.c_float(scale),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    return y, m, l


@pytest.mark.parametrize("rows,cols", [
    (9, 1 << 21),      # 8 MB rows: eight to a group, the second group has one live row
    (1, 3_000_001),    # one row, ragged last chunk
    (40, 500_000),     # 2 MB rows, several groups
    (3, 409_601),      # just beyond the cluster path
])
@pytest.mark.parametrize("mask", [False, True])
def test_wide_fp32(rows, cols, mask):
    assert oss.softmax_rows_workspace_bytes(rows, cols) > 0
    x = workloads.logits(rows, cols, 10.0, seed=rows * 31 + cols + mask, device="cuda")
    if mask:
        g = torch.Generator(device="cuda").manual_seed(cols)
        x[torch.rand(x.shape, generator=g, device="cuda") < 0.2] = -float("inf")
        x[0, : cols - 7] = -float("inf")     # only the last slice of row 0 has live entries
        if rows > 2:
            x[2] = -float("inf")             # a whole masked row
    y, m, l = oss.softmax_rows(x, 0.7)
    assert oss.check_device_error() == 0
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(0.7)), what=f"wide {rows}x{cols}")
    # the same outputs as the call without a workspace, within the bar
    y2, m2, l2 = no_workspace(x, 0.7)
    torch.cuda.synchronize()
    assert torch.equal(m, m2)
    fin = torch.isfinite(m)
    assert torch.allclose(l[fin], l2[fin], rtol=2e-5, atol=0)


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("rows,cols", [(5, 1 << 21), (2, 819_201)])
def test_wide_16bit(kind, rows, cols):
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    assert oss.softmax_rows_workspace_bytes(rows, cols, dtype) > 0
    x = workloads.logits(rows, cols, 10.0, seed=cols + rows, device="cuda").to(dtype)
    g = torch.Generator(device="cuda").manual_seed(rows)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.1] = -float("inf")
    y, m, l = oss.softmax_rows_16bit(x, 0.9)
    assert oss.check_device_error() == 0
    xr = x.float().cpu().numpy().astype(np.float64)
    check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                    *oracle.softmax_rows(xr, f32(0.9)), kind=kind, what=f"wide {kind} {rows}x{cols}")


@pytest.mark.parametrize("rows,cols,ld,offset", [(3, 1_000_003, 1_000_005, 1), (2, 700_001, 700_001, 3)])
def test_wide_rows_off_the_grid(rows, cols, ld, offset):
    # x and y at the same offset from the 16-byte grid: element-wise accesses
    buf = workloads.logits(1, rows * ld + offset, 10.0, seed=cols, device="cuda")
    x = buf[0, offset:].view(rows, ld)[:, :cols]
    ybuf = torch.full((rows * ld + offset,), 7.0, device="cuda")
    y = ybuf[offset:].view(rows, ld)[:, :cols]
    y, m, l = oss.softmax_rows(x, 1.3, y=y)
    assert oss.check_device_error() == 0
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(1.3)), what=f"wide off-grid {rows}x{cols}")
    # nothing outside the rows was written
    yb = ybuf[offset:].view(rows, ld)
    assert bool((yb[:, cols:] == 7.0).all()) and float(ybuf[:offset].sum()) == 7.0 * offset


def test_wide_repeat_identical():
    # slice states are merged in slice order: results repeat bit for bit
    x = workloads.logits(5, 1 << 21, 10.0, seed=9, device="cuda")
    y1, m1, l1 = oss.softmax_rows(x, 1.0)
    y2, m2, l2 = oss.softmax_rows(x, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(m1, m2) and torch.equal(l1, l2)


@pytest.mark.slow
def test_wide_64_rows_of_4m_sampled():
    # the 64 x 2^22 fp32 matrix (1 GiB): every row's m and l, and the full y
    # of a seeded sample of rows, against the oracle
    rows, cols = 64, 1 << 22
    x = workloads.logits(rows, cols, 10.0, seed=64, device="cuda")
    y, m, l = oss.softmax_rows(x, 1.0)
    assert oss.check_device_error() == 0
    rng = np.random.default_rng(64)
    sample = sorted(set(int(r) for r in rng.integers(0, rows, 6)) | {0, rows - 1})
    for r in sample:
        ry, rm, rl = oracle.softmax_rows(x[r:r + 1].cpu().numpy(), 1.0)
        check_softmax(y[r:r + 1].cpu().numpy(), m[r:r + 1].cpu().numpy(), l[r:r + 1].cpu().numpy(),
                      ry, rm, rl, what=f"64x4M row {r}")
    mx = x.max(dim=1).values.cpu().numpy()
    np.testing.assert_array_equal(m.cpu().numpy(), mx.astype(np.float32))
