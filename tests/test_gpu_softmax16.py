"""os_softmax_rows_16bit (bf16 and fp16 rows) against the oracle, element by
element (GPU). The oracle sees the exact values of the 16-bit inputs."""

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax16, f32

pytestmark = pytest.mark.gpu

KINDS = {"bf16": torch.bfloat16, "f16": torch.float16}


def make(rows, ld, mult, seed, kind):
    return workloads.logits(rows, ld, mult, seed, device="cuda").to(KINDS[kind])


def check(x, y, m, l, scale, kind, what):
    torch.cuda.synchronize()
    xr = x.float().cpu().numpy().astype(np.float64)
    return check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                           *oracle.softmax_rows(xr, f32(scale)), kind=kind, what=what)


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (5, 8), (37, 1000), (9, 2049),
                                       (16, 8192), (4, 16384), (3, 16385), (2, 40007)])
@pytest.mark.parametrize("scale", [1.0, 0.1])
def test_shapes_aligned(kind, rows, cols, scale):
    # leading dimension rounded up to 8 elements: the 16-byte path (register
    # resident up to 16384 columns), with a ragged tail when cols % 8 != 0
    ld = (cols + 7) // 8 * 8
    x = make(rows, ld, 10.0, rows * 131 + cols, kind)[:, :cols]
    y = torch.empty((rows, ld), dtype=x.dtype, device="cuda")[:, :cols]
    y, m, l = oss.softmax_rows_16bit(x, scale, y=y)
    check(x, y, m, l, scale, kind, f"{kind} {rows}x{cols}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("rows,cols", [(1, 3), (7, 999), (2, 20001)])
def test_unaligned(kind, rows, cols):
    buf = make(1, rows * cols + 1, 10.0, 17, kind)
    x = buf[0, 1:].view(rows, cols)          # base offset by one element
    y, m, l = oss.softmax_rows_16bit(x, 0.3)
    check(x, y, m, l, 0.3, kind, f"unaligned {kind}")


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("cols", [64, 8192, 20000])
def test_masked_and_empty_rows(kind, cols):
    x = make(8, cols, 10.0, cols + 2, kind)
    g = torch.Generator(device="cuda").manual_seed(8)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.3] = -float("inf")
    x[2] = -float("inf")
    x[5, : cols // 2] = -float("inf")
    y, m, l = oss.softmax_rows_16bit(x, 0.1)
    check(x, y, m, l, 0.1, kind, "masked")
    yn = y.float().cpu().numpy()
    assert m[2].item() == -np.inf and l[2].item() == 0.0 and np.all(yn[2] == 0.0)
    assert not np.any(np.isnan(yn))


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_wide_logits(kind):
    # bf16 carries the fp32 exponent range: logits in the thousands; fp16
    # tops out at 65504, so 3000 there as well
    x = make(4, 4096, 3000.0 if kind == "f16" else 1000.0, 19, kind)
    y, m, l = oss.softmax_rows_16bit(x, 1.0)
    assert torch.all(torch.isfinite(y)) and torch.all(torch.isfinite(l))
    check(x, y, m, l, 1.0, kind, "wide")


def test_sampled_rows_full_size_bf16():
    w = workloads.SOFTMAX_32K
    x = make(w.rows, w.cols, w.mult, w.seed, "bf16")
    y, m, l = oss.softmax_rows_16bit(x, w.scale)
    torch.cuda.synchronize()
    rows = np.random.default_rng(7).choice(w.rows, 256, replace=False)
    rows = np.sort(np.concatenate([rows, [0, w.rows - 1]]))
    idx = torch.as_tensor(rows, device="cuda")
    check(x[idx], y[idx], m[idx], l[idx], w.scale, "bf16", "softmax_32k bf16 sampled")
