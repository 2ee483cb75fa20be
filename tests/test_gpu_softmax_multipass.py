"""os_softmax_rows_multipass (the 2- and 3-pass comparators) against the
oracle, element by element (GPU)."""

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_softmax, f32

pytestmark = pytest.mark.gpu


def run(x, passes, scale):
    y, m, l = oss.softmax_rows_multipass(x, passes, scale)
    torch.cuda.synchronize()
    return y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()


@pytest.mark.parametrize("passes", [2, 3])
@pytest.mark.parametrize("rows,cols", [(1, 1), (5, 7), (37, 1000), (9, 1025), (3, 16385),
                                       (2, 40003)])
@pytest.mark.parametrize("scale", [1.0, 0.1])
def test_shapes_aligned(passes, rows, cols, scale):
    ld = (cols + 3) // 4 * 4
    x = workloads.logits(rows, ld, 10.0, seed=rows * 31 + cols, device="cuda")[:, :cols]
    y, m, l = run(x, passes, scale)
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(scale)),
                  what=f"{passes}-pass {rows}x{cols}")


@pytest.mark.parametrize("passes", [2, 3])
def test_unaligned_rows(passes):
    x = workloads.logits(7, 999, 10.0, seed=11, device="cuda")
    y, m, l = run(x, passes, 0.3)
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(0.3)), what="unaligned")


@pytest.mark.parametrize("passes", [2, 3])
def test_masked_and_empty_rows(passes):
    x = workloads.logits(6, 3000, 10.0, seed=12, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(6)
    x[torch.rand(x.shape, generator=g, device="cuda") < 0.4] = -float("inf")
    x[1] = -float("inf")
    x[4, :2000] = -float("inf")
    y, m, l = run(x, passes, 0.1)
    check_softmax(y, m, l, *oracle.softmax_rows(x.cpu().numpy(), f32(0.1)), what="masked")
    assert m[1] == -np.inf and l[1] == 0.0 and np.all(y[1] == 0.0)
    assert not np.any(np.isnan(y))


@pytest.mark.parametrize("passes", [2, 3])
def test_agrees_with_one_pass(passes):
    # all three forms compute the same definition; they differ in how often
    # the row is read and in the order of the sums, so l and y agree to the
    # softmax parity bar (1e-5 relative), m exactly
    x = workloads.logits(64, 8192, 10.0, seed=13, device="cuda")
    y1, m1, l1 = oss.softmax_rows(x, 1.0)
    yk, mk, lk = oss.softmax_rows_multipass(x, passes, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(m1, mk)
    torch.testing.assert_close(lk, l1, rtol=1e-5, atol=0)
    torch.testing.assert_close(yk, y1, rtol=1e-5, atol=2.0 ** -126)
