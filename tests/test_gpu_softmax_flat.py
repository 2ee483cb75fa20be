"""Short rows of dense matrices, staged through shared memory, against the
oracle (GPU).

Rows whose x rows lie back to back (leading dimension = row length), at
most 512 bytes long or at most 1 KB and off the 16-byte grid, are taken in
tiles of whole rows: the tile's 16-byte granules are bulk-copied into shared
memory and each row is read from there in 16-byte chunks on the grid of its
own offset, by a group of 1 to 32 threads. y is written in chunks when its
rows have x's offsets and element by element otherwise, so y may sit at any
offset and leading dimension. The lengths span every group size; the bases
put x's first and last granules at every offset; the row counts leave a
ragged last tile and give some CTAs several tiles, so that every buffer is
refilled; tiny matrices fit in one or two granules. (Aligned rows longer than
512 bytes go to the grouped kernel, and are checked here all the same.)"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, check_softmax16, f32

pytestmark = pytest.mark.gpu

F32_COLS = [1, 2, 3, 5, 8, 31, 33, 64, 65, 100, 101, 127, 128, 129, 200, 255, 256]
H16_COLS = [1, 3, 7, 8, 9, 63, 64, 65, 100, 101, 128, 129, 200, 255, 256, 257, 300, 301, 511, 512]


def rows_for(cols):
    return max(3, min(150001, 3_000_000 // cols))


def dense_at(rows, cols, dtype, offset, seed):
    """A [rows, cols] view with leading dimension cols, `offset` elements into
    its buffer (moves the base off the 16-byte grid), and the buffer."""
    n = rows * cols + offset + 7
    buf = workloads.logits(1, n, 10.0, seed, device="cuda").to(dtype)[0]
    return buf[offset:offset + rows * cols].view(rows, cols), buf


def masked(x, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.25] = -float("inf")
    x[3::7] = -float("inf")   # whole rows
    return x


def run(x, scale, y):
    if x.dtype == torch.float32:
        return oss.softmax_rows(x, scale, y=y)
    return oss.softmax_rows_16bit(x, scale, y=y)


def check(x, y, m, l, scale, what):
    torch.cuda.synchronize()
    assert oss.check_device_error() == 0
    if x.dtype == torch.float32:
        check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                      *oracle.softmax_rows(x.cpu().numpy(), f32(scale)), what=what)
    else:
        kind = "bf16" if x.dtype == torch.bfloat16 else "f16"
        xr = x.float().cpu().numpy().astype(np.float64)
        check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                        *oracle.softmax_rows(xr, f32(scale)), kind=kind, what=what)


@pytest.mark.parametrize("cols", F32_COLS)
@pytest.mark.parametrize("x_off", [0, 1, 3])
def test_fp32_dense_short_rows(cols, x_off):
    rows = rows_for(cols)
    x, _ = dense_at(rows, cols, torch.float32, x_off, seed=cols * 4 + x_off)
    if x_off == 3:
        x = masked(x, cols)
    y, m, l = run(x, 0.7, None)
    check(x, y, m, l, 0.7, f"fp32 {rows}x{cols} x+{x_off}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols", H16_COLS)
@pytest.mark.parametrize("x_off", [0, 1, 5])
def test_16bit_dense_short_rows(kind, cols, x_off):
    rows = rows_for(cols)
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    x, _ = dense_at(rows, cols, dtype, x_off, seed=cols * 8 + x_off)
    if x_off == 5:
        x = masked(x, cols + 1)
    y, m, l = run(x, 0.7, None)
    check(x, y, m, l, 0.7, f"{kind} {rows}x{cols} x+{x_off}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cols", [3, 100, 129, 256])
def test_y_at_any_layout(dtype, cols):
    # y off the grid, out of step with x and with its own leading dimension;
    # the padding around y's rows is never written
    rows = 5003
    x, _ = dense_at(rows, cols, dtype, 2, seed=cols)
    ld = cols + 5
    ybuf = torch.full((rows * ld + 3,), 7.0, dtype=dtype, device="cuda")
    y = ybuf[1:1 + rows * ld].view(rows, ld)[:, :cols]
    y, m, l = run(x, 1.1, y)
    check(x, y, m, l, 1.1, f"{dtype} {rows}x{cols} y ld {ld}")
    yb = ybuf[1:1 + rows * ld].view(rows, ld)
    assert torch.all(yb[:, cols:] == 7.0) and ybuf[0] == 7.0 and torch.all(ybuf[1 + rows * ld:] == 7.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 3), (2, 3), (3, 2), (1, 7), (2, 5), (4, 4),
                                       (1, 256), (2, 129), (9, 17)])
@pytest.mark.parametrize("x_off", [0, 1, 3, 7])
def test_tiny_matrices(dtype, rows, cols, x_off):
    # a matrix within one or two granules: no bulk copy, or one granule of it
    if dtype == torch.float32 and cols > 256:
        pytest.skip("longer than the staged rows")
    x, _ = dense_at(rows, cols, dtype, x_off, seed=rows * 100 + cols + x_off)
    y, m, l = run(x, 0.9, None)
    check(x, y, m, l, 0.9, f"{dtype} {rows}x{cols} x+{x_off}")


def test_fewer_rows_than_ctas():
    # tiles of a row or two, so every CTA of one wave has a tile
    for rows in (1, 37, 600, 1217):
        x, _ = dense_at(rows, 300, torch.bfloat16, 1, seed=rows)
        y, m, l = run(x, 1.0, None)
        check(x, y, m, l, 1.0, f"bf16 {rows}x300")


def test_null_m_and_l():
    rows, cols = 20011, 77
    x, _ = dense_at(rows, cols, torch.float32, 1, seed=9)
    y = torch.empty_like(x)
    lib = oss.load()
    st = lib.os_softmax_rows(x.data_ptr(), y.data_ptr(), None, None, rows, cols, cols, cols,
                             ctypes.c_float(1.0), None)
    assert st == 0
    _, m, l = oss.softmax_rows(x, 1.0)
    y2 = torch.empty_like(x)
    oss.softmax_rows(x, 1.0, y=y2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    xb = x.to(torch.bfloat16)
    yb = torch.empty_like(xb)
    st = lib.os_softmax_rows_16bit(xb.data_ptr(), yb.data_ptr(), None, None, rows, cols, cols, cols,
                                   ctypes.c_float(1.0), 1, None)
    assert st == 0
    yb2, _, _ = oss.softmax_rows_16bit(xb, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(yb, yb2)


def test_repeat_identical():
    # a fixed reduction order: results repeat bit for bit
    x, _ = dense_at(100003, 100, torch.bfloat16, 1, seed=4)
    a = oss.softmax_rows_16bit(x, 1.0)
    b = oss.softmax_rows_16bit(x, 1.0)
    torch.cuda.synchronize()
    assert all(torch.equal(p, q) for p, q in zip(a, b))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("cols", [3, 7, 33, 100, 101, 255, 300])
@pytest.mark.parametrize("off", [1, 3, 5])
def test_y_like_x_tiles_leave_by_bulk_copies(dtype, cols, off):
    # x and y at the same offset from the 16-byte grid, rows back to back, row
    # lengths off the grid: tiles of y leave through shared memory by bulk
    # copies, and the granules where two tiles meet are shared by two CTAs
    # (each stores its own elements); the canaries around y stay intact
    esz = torch.tensor([], dtype=dtype).element_size()
    if dtype == torch.float32 and cols * esz > 1024:
        pytest.skip("longer than the staged rows")
    rows = max(7, min(120001, 2_000_000 // cols))
    x, _ = dense_at(rows, cols, dtype, off, seed=cols * 3 + off)
    ybuf = torch.full((rows * cols + off + 16,), 7.0, dtype=dtype, device="cuda")
    y = ybuf[off:off + rows * cols].view(rows, cols)
    if off == 5:
        x = masked(x, cols)
    y, m, l = run(x, 0.8, y)
    check(x, y, m, l, 0.8, f"{dtype} {rows}x{cols} y like x +{off}")
    assert bool((ybuf[:off] == 7.0).all()) and bool((ybuf[off + rows * cols:] == 7.0).all())


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols", [128, 256])
@pytest.mark.parametrize("rows", [1, 2, 55, 56, 57, 111, 112, 113, 5000])
def test_16bit_rows_on_the_grid_in_eight_chunk_groups(kind, cols, rows):
    # 16-bit rows of 128 or 256 elements on the 16-byte grid take groups of 2
    # or 4 threads of eight chunks and tiles of 28 KB (112 or 56 rows): row
    # counts around a tile, masked entries and whole masked rows
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    x, _ = dense_at(rows, cols, dtype, 0, seed=rows * 3 + cols)
    assert x.data_ptr() % 16 == 0
    if rows > 3:
        x = masked(x, rows + cols)
    y, m, l = run(x, 1.1, None)
    check(x, y, m, l, 1.1, f"{kind} {rows}x{cols} eight-chunk groups")
