"""Rows longer than 16384 elements against the oracle (GPU).

Aligned rows of up to 8 x 2048 chunks of 16 bytes (131072 16-bit elements,
65536 fp32; fp32 rows of more than 80 KB) are held in the registers of a
thread-block cluster: CTA r of a cluster of C CTAs holds slice r, the CTAs
send their (max, sum) states to each other by asynchronous stores into
distributed shared memory, and each writes its slice once. Other rows of up
to 8 x 200 KB are held in the shared memory of a cluster, merged through a
cluster barrier; a row of at most 48 KB takes one CTA with two slice buffers
(the next row's copies overlap the current row). Longer rows fall back to the
streaming kernel. The lengths below take every cluster size of both paths,
5 to 8 chunks a thread in the register path, one CTA with two buffers, one
with one buffer, ragged last slices and slices that are empty; most row counts
exceed the clusters resident at once, so each cluster walks several rows,
and some are fewer than the clusters."""

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, check_softmax16, f32

pytestmark = pytest.mark.gpu

# (cols, rows); the row's size and the fewest 200 KB slices that hold it
F32_CASES = [
    (16385, 301),    # 64 KB, one CTA, ragged tail
    (20000, 401),    # 80 KB; more rows than resident CTAs
    (20481, 150),    # registers: 3 CTAs of 7 chunks a thread
    (24576, 150),    # registers: 3 CTAs of 8
    (25601, 160),    # 100 KB, one element past a 16-byte chunk (registers: 4 of 7)
    (32768, 160),    # 128 KB (registers: 4 of 8)
    (40000, 100),    # registers: 5 CTAs
    (57345, 50),     # registers: 8 CTAs, the last one short
    (65536, 130),    # 256 KB (registers: 8 CTAs)
    (65536, 3),      # fewer rows than clusters
    (65537, 40),     # one element past the register path: shared memory
    (100003, 41),    # 391 KB, ragged
    (204800, 21),    # 800 KB: four or more
    (204801, 21),    # one element more: five or more
    (409600, 9),     # 1.6 MB: eight, the longest held row
    (409601, 9),     # beyond: the streaming kernel
]
H16_CASES = [
    (16385, 301),    # 32 KB: one CTA, two buffers
    (18432, 301),    # 36 KB: the longest that stays in one CTA's two buffers
    (18440, 301),    # registers: 2 CTAs of 5 chunks a thread
    (20000, 401),    # registers: 2 CTAs of 5
    (24000, 301),    # registers: 2 CTAs of 6
    (32768, 200),    # registers: 2 CTAs of 8
    (51201, 160),    # registers: 4 CTAs of 7, ragged
    (100000, 40),    # registers: 7 CTAs of 7
    (131072, 64),    # 256 KB: registers, 8 CTAs of 8
    (131072, 3),     # fewer rows than clusters
    (131073, 30),    # one element past the register path: shared memory
    (409600, 12), (409601, 12),
    (819200, 6),     # 1.6 MB: eight
    (819201, 6),     # beyond: the streaming kernel
]


def masked(x, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.2] = -float("inf")
    x[1::5] = -float("inf")   # whole rows
    cols = x.shape[1]
    x[2, : cols // 2] = -float("inf")   # first half masked: leading slices empty
    return x


@pytest.mark.parametrize("cols,rows", F32_CASES)
@pytest.mark.parametrize("mask", [False, True])
def test_fp32_long_rows(cols, rows, mask):
    ld = (cols + 3) // 4 * 4
    x = workloads.logits(rows, ld, 10.0, seed=cols + mask, device="cuda")[:, :cols]
    if mask:
        x = masked(x, cols)
    y = torch.empty((rows, ld), device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows(x, 0.9, y=y)
    torch.cuda.synchronize()
    assert oss.check_device_error() == 0
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(0.9)), what=f"fp32 {rows}x{cols}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols,rows", H16_CASES)
@pytest.mark.parametrize("mask", [False, True])
def test_16bit_long_rows(kind, cols, rows, mask):
    ld = (cols + 7) // 8 * 8
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    x = workloads.logits(rows, ld, 10.0, seed=cols * 3 + mask, device="cuda").to(dtype)[:, :cols]
    if mask:
        x = masked(x, cols + 1)
    y = torch.empty((rows, ld), dtype=dtype, device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows_16bit(x, 0.9, y=y)
    torch.cuda.synchronize()
    assert oss.check_device_error() == 0
    xr = x.float().cpu().numpy().astype(np.float64)
    check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                    *oracle.softmax_rows(xr, f32(0.9)), kind=kind, what=f"{kind} {rows}x{cols}")


def test_long_rows_repeat_identical():
    # the cluster merge runs in a fixed order: results repeat bit for bit
    x = workloads.logits(50, 100000, 10.0, seed=5, device="cuda")
    y1, m1, l1 = oss.softmax_rows(x, 1.0)
    y2, m2, l2 = oss.softmax_rows(x, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(m1, m2) and torch.equal(l1, l2)


@pytest.mark.parametrize("rows,cols,ld,offset", [
    (2, 40003, 40003, 0),      # unaligned rows, too few to fill the GPU: a cluster per row
    (3, 300001, 300002, 1),    # unaligned base and leading dimension
    (1, 2000000, 2000000, 0),  # aligned but beyond a cluster's shared memory (8 MB)
    (5, 600000, 600000, 0),
])
@pytest.mark.parametrize("mask", [False, True])
def test_fp32_streamed_rows_split_across_a_cluster(rows, cols, ld, offset, mask):
    # rows that take the streaming kernel, with fewer rows than the GPU holds
    # CTAs: each row is cut into slices streamed by the CTAs of a cluster,
    # whose states merge through distributed shared memory
    buf = workloads.logits(1, rows * ld + offset, 10.0, seed=cols + offset + mask, device="cuda")
    x = buf[0, offset:].view(rows, ld)[:, :cols]
    if mask:
        g = torch.Generator(device="cuda").manual_seed(cols)
        x[torch.rand(x.shape, generator=g, device="cuda") < 0.2] = -float("inf")
        x[0, : cols - 10] = -float("inf")  # only the last slice has live entries
    ybuf = torch.empty(rows * ld + offset, device="cuda")
    y = ybuf[offset:].view(rows, ld)[:, :cols]
    y, m, l = oss.softmax_rows(x, 0.6, y=y)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(0.6)), what=f"fp32 {rows}x{cols}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("rows,cols,ld,offset", [
    (2, 40003, 40003, 0), (3, 300001, 300003, 1), (1, 4000000, 4000000, 0),
])
def test_16bit_streamed_rows_split_across_a_cluster(kind, rows, cols, ld, offset):
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    buf = workloads.logits(1, rows * ld + offset, 10.0, seed=cols * 7 + offset, device="cuda").to(dtype)
    x = buf[0, offset:].view(rows, ld)[:, :cols]
    g = torch.Generator(device="cuda").manual_seed(cols + 1)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.2] = -float("inf")
    ybuf = torch.empty(rows * ld + offset, dtype=dtype, device="cuda")
    y = ybuf[offset:].view(rows, ld)[:, :cols]
    y, m, l = oss.softmax_rows_16bit(x, 0.6, y=y)
    torch.cuda.synchronize()
    xr = x.float().cpu().numpy().astype(np.float64)
    check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                    *oracle.softmax_rows(xr, f32(0.6)), kind=kind, what=f"{kind} {rows}x{cols}")
