"""Row softmax on rows short enough that several rows share a CTA (GPU).

os_softmax_rows (fp32 rows of up to 2048 elements) and os_softmax_rows_16bit
(rows of up to 16384 elements) give each row a group of 8, 16, 32, 64, 128 or
256 threads and let the groups of a CTA run through their rows independently,
some prefetching the next row; groups narrower than a warp walk their rows
with their warp. The lengths below sit on both sides of every
change of group size; the row counts make every group take several rows and
leave the last CTAs with groups that have no row at all. Masked entries, and
fully masked rows at a stride that is not a multiple of any group count, land
in every position within a group."""

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, check_softmax16, f32

pytestmark = pytest.mark.gpu

F32_COLS = [1, 3, 31, 32, 33, 64, 65, 128, 129, 255, 256, 257, 500, 512, 513, 1000, 1024, 1025,
            2047, 2048, 2049]
H16_COLS = [1, 7, 64, 65, 127, 128, 129, 255, 256, 257, 512, 513, 1000, 1024, 1025, 2048, 2049,
            4096, 4097, 8192, 8193, 16384]


def rows_for(cols, elems=3_000_000, most=30011):
    return max(7, min(most, elems // cols))


def masked(x, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.3] = -float("inf")
    x[::7] = -float("inf")   # whole rows: every 7th
    return x


@pytest.mark.parametrize("cols", F32_COLS)
@pytest.mark.parametrize("mask", [False, True])
def test_fp32_rows_per_group(cols, mask):
    rows = rows_for(cols)
    ld = (cols + 3) // 4 * 4
    x = workloads.logits(rows, ld, 10.0, seed=cols * 3 + mask, device="cuda")[:, :cols]
    if mask:
        x = masked(x, cols)
    y = torch.empty((rows, ld), device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows(x, 0.7, y=y)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(0.7)), what=f"fp32 {rows}x{cols}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols", H16_COLS)
@pytest.mark.parametrize("mask", [False, True])
def test_16bit_rows_per_group(kind, cols, mask):
    rows = rows_for(cols)
    ld = (cols + 7) // 8 * 8
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    x = workloads.logits(rows, ld, 10.0, seed=cols * 5 + mask, device="cuda").to(dtype)[:, :cols]
    if mask:
        x = masked(x, cols + 1)
    y = torch.empty((rows, ld), dtype=dtype, device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows_16bit(x, 0.7, y=y)
    torch.cuda.synchronize()
    xr = x.float().cpu().numpy().astype(np.float64)
    check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                    *oracle.softmax_rows(xr, f32(0.7)), kind=kind, what=f"{kind} {rows}x{cols}")


@pytest.mark.parametrize("rows", [1, 2, 5, 9, 33])
@pytest.mark.parametrize("cols", [20, 60, 100, 700, 1500])
def test_fewer_rows_than_groups(rows, cols):
    # one CTA, most of whose groups have no row; for the shortest rows the
    # groups are narrower than a warp, and a warp's groups past the last
    # row run as empty rows
    x = workloads.logits(rows, cols, 10.0, seed=rows * 31 + cols, device="cuda")
    y, m, l = oss.softmax_rows(x, 1.0)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), 1.0), what=f"{rows}x{cols}")
    xb = x.to(torch.bfloat16)
    yb, mb, lb = oss.softmax_rows_16bit(xb, 1.0)
    torch.cuda.synchronize()
    check_softmax16(yb.float().cpu().numpy(), mb.cpu().numpy(), lb.cpu().numpy(),
                    *oracle.softmax_rows(xb.float().cpu().numpy().astype(np.float64), 1.0),
                    kind="bf16", what=f"bf16 {rows}x{cols}")


@pytest.mark.parametrize("cols", [1, 5, 17, 31, 32, 33, 63, 64])
def test_fp32_narrow_groups_many_rows(cols):
    # groups of 8 and 16 threads, four and two to a warp; more rows than one
    # wave of the persistent grid holds, so every warp walks several rows and
    # the last ones end part-way through a warp
    rows = 100003
    ld = (cols + 3) // 4 * 4
    x = masked(workloads.logits(rows, ld, 10.0, seed=cols + 7, device="cuda")[:, :cols], cols)
    y = torch.empty((rows, ld), device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows(x, 1.3, y=y)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(1.3)), what=f"fp32 {rows}x{cols}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols", [1, 9, 63, 64, 65, 100, 127, 128])
def test_16bit_narrow_groups_many_rows(kind, cols):
    rows = 100003
    ld = (cols + 7) // 8 * 8
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    x = workloads.logits(rows, ld, 10.0, seed=cols + 9, device="cuda").to(dtype)[:, :cols]
    x = masked(x, cols + 2)
    y = torch.empty((rows, ld), dtype=dtype, device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows_16bit(x, 1.3, y=y)
    torch.cuda.synchronize()
    xr = x.float().cpu().numpy().astype(np.float64)
    check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                    *oracle.softmax_rows(xr, f32(1.3)), kind=kind, what=f"{kind} {rows}x{cols}")
