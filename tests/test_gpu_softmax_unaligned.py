"""Rows that do not start on a 16-byte boundary, against the oracle (GPU).

When x's and y's rows start at the same offset from a 16-byte boundary (an
odd leading dimension, or both bases moved by the same number of elements),
the kernels cut each row into 16-byte chunks on the grid: the whole chunks
move as 16-byte accesses (bulk copies for rows held in a cluster's shared
memory), the partial first and last chunks element by element. With an odd
leading dimension the offset changes from row to row. Rows whose x and y
offsets differ are streamed. The lengths span every kernel and group size."""

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, check_softmax16, f32

pytestmark = pytest.mark.gpu

F32_COLS = [1, 3, 5, 31, 33, 63, 127, 129, 255, 513, 1001, 2047, 2049, 4095, 8191, 8193, 16383,
            16385, 50257, 100003]
H16_COLS = [1, 7, 9, 63, 65, 127, 129, 1001, 2049, 4095, 8193, 16383, 16385, 50257, 131071]


def rows_for(cols):
    return max(3, min(2000, 3_000_000 // cols))


def layouts(rows, cols, dtype, seed):
    """(x, y) pairs in step: dense with an odd leading dimension, and both
    bases moved by one element with a leading dimension of cols + 1."""
    out = []
    x = workloads.logits(rows, cols, 10.0, seed, device="cuda").to(dtype)
    out.append(("dense", x, torch.empty_like(x)))
    ld = cols + 1
    bx = workloads.logits(1, rows * ld + 1, 10.0, seed + 1, device="cuda").to(dtype)[0]
    by = torch.empty(rows * ld + 1, dtype=dtype, device="cuda")
    out.append(("offset", bx[1:].view(rows, ld)[:, :cols], by[1:].view(rows, ld)[:, :cols]))
    return out


def masked(x, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.2] = -float("inf")
    x[1::4] = -float("inf")
    return x


@pytest.mark.parametrize("cols", F32_COLS)
def test_fp32_rows_off_the_grid(cols):
    rows = rows_for(cols)
    for name, x, y in layouts(rows, cols, torch.float32, cols):
        for mask in (False, True):
            if mask:
                x = masked(x, cols + 3)
            y, m, l = oss.softmax_rows(x, 0.8, y=y)
            torch.cuda.synchronize()
            assert oss.check_device_error() == 0
            check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                          *oracle.softmax_rows(x.cpu().numpy(), f32(0.8)),
                          what=f"fp32 {name} {rows}x{cols} mask={mask}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols", H16_COLS)
def test_16bit_rows_off_the_grid(kind, cols):
    rows = rows_for(cols)
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    for name, x, y in layouts(rows, cols, dtype, cols * 3):
        for mask in (False, True):
            if mask:
                x = masked(x, cols + 5)
            y, m, l = oss.softmax_rows_16bit(x, 0.8, y=y)
            torch.cuda.synchronize()
            assert oss.check_device_error() == 0
            xr = x.float().cpu().numpy().astype(np.float64)
            check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                            *oracle.softmax_rows(xr, f32(0.8)), kind=kind,
                            what=f"{kind} {name} {rows}x{cols} mask={mask}")


@pytest.mark.parametrize("cols", [1001, 50257])
def test_offsets_out_of_step_are_streamed(cols):
    # x moved by one element, y not: the chunks cannot line up for both
    rows = rows_for(cols)
    bx = workloads.logits(1, rows * cols + 1, 10.0, seed=cols, device="cuda")[0]
    x = bx[1:].view(rows, cols)
    y, m, l = oss.softmax_rows(x, 0.8)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(0.8)), what=f"out of step {cols}")


def test_output_padding_untouched():
    # the partial chunks write only the row's own elements
    rows, cols, ld = 37, 1001, 1003
    big = workloads.logits(rows, ld, 10.0, seed=2, device="cuda")
    yb = torch.full((rows, ld), 7.0, device="cuda")
    oss.softmax_rows(big[:, 1:cols + 1], 1.0, y=yb[:, 1:cols + 1])
    torch.cuda.synchronize()
    assert torch.all(yb[:, 0] == 7.0) and torch.all(yb[:, cols + 1:] == 7.0)
    bb = big.to(torch.bfloat16)
    yh = torch.full((rows, ld), 7.0, dtype=torch.bfloat16, device="cuda")
    oss.softmax_rows_16bit(bb[:, 1:cols + 1], 1.0, y=yh[:, 1:cols + 1])
    torch.cuda.synchronize()
    assert torch.all(yh[:, 0] == 7.0) and torch.all(yh[:, cols + 1:] == 7.0)
