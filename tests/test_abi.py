"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/oss.h declares, and rejects invalid arguments before touching the
device. No call here reaches a kernel launch."""

import ctypes
import os
import re

import pytest

import pass_attention_gb300 as oss
from pass_attention_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "oss.h")

INVALID, MISALIGNED, UNSUPPORTED = 1, 2, 3
A = 4096  # a 16-byte-aligned stand-in address; never dereferenced by these calls


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return oss.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"OSS_API\s+[\w\s\*]+?\b(os_\w+)\s*\(", text)


def test_header_declares_the_binding_signatures():
    names = declared_functions()
    assert sorted(names) == sorted(oss.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.os_abi_version() == 1
    for code, name in oss.STATUS_NAMES.items():
        assert lib.os_status_string(code).decode() == name
    assert lib.os_status_string(99).decode() == "OS_ERR_UNKNOWN"


def test_softmax_rows_rejects_bad_arguments(lib):
    f = lib.os_softmax_rows
    assert f(None, A, None, None, 4, 8, 8, 8, 1.0, None) == INVALID
    assert f(A, None, None, None, 4, 8, 8, 8, 1.0, None) == INVALID
    assert f(A, A, None, None, 0, 8, 8, 8, 1.0, None) == INVALID
    assert f(A, A, None, None, 4, 0, 8, 8, 1.0, None) == INVALID
    assert f(A, A, None, None, 4, 8, 7, 8, 1.0, None) == INVALID   # ld_x < cols
    assert f(A, A, None, None, 4, 8, 8, 8, 0.0, None) == INVALID   # scale must be > 0
    assert f(A, A, None, None, 4, 8, 8, 8, -1.0, None) == INVALID
    assert f(A, A, None, None, 4, 8, 8, 8, float("nan"), None) == INVALID
    assert f(A, A, None, None, 4, 8, 8, 8, float("inf"), None) == INVALID
    assert f(A + 2, A, None, None, 4, 8, 8, 8, 1.0, None) == MISALIGNED   # not float-aligned
    assert f(A, A + 1, None, None, 4, 8, 8, 8, 1.0, None) == MISALIGNED
    assert f(A, A, A + 2, None, 4, 8, 8, 8, 1.0, None) == MISALIGNED   # m not float-aligned
    assert f(A, A, None, A + 1, 4, 8, 8, 8, 1.0, None) == MISALIGNED   # l


def test_softmax_rows_from_host_rejects_bad_arguments(lib):
    f = lib.os_softmax_rows_from_host
    ok = dict(xh=A, yh=A, mh=A, lh=A, xd=A, yd=A, md=A, ld=A)

    def call(rows=4, cols=8, scale=1.0, chunk=0, **kw):
        a = dict(ok, **kw)
        return f(a["xh"], a["yh"], a["mh"], a["lh"], a["xd"], a["yd"], a["md"], a["ld"], rows, cols,
                 ctypes.c_float(scale), chunk, None)
    assert call(xh=None) == INVALID
    assert call(yh=None) == INVALID
    assert call(xd=None) == INVALID
    assert call(yd=None) == INVALID
    assert call(md=None) == INVALID            # host m without its device buffer
    assert call(ld=None) == INVALID            # host l without its device buffer
    assert call(rows=0) == INVALID
    assert call(cols=0) == INVALID
    assert call(chunk=-1) == INVALID
    assert call(scale=0.0) == INVALID
    assert call(scale=float("nan")) == INVALID
    assert call(xd=A + 2) == MISALIGNED
    assert call(ld=A + 1) == MISALIGNED


def test_softmax_rows_multipass_rejects_bad_arguments(lib):
    f = lib.os_softmax_rows_multipass
    for passes in (2, 3):
        assert f(None, A, A, A, 4, 8, 8, 8, 1.0, passes, None) == INVALID
        assert f(A, A, None, A, 4, 8, 8, 8, 1.0, passes, None) == INVALID   # m carries state
        assert f(A, A, A, None, 4, 8, 8, 8, 1.0, passes, None) == INVALID   # so does l
        assert f(A, A, A, A, 4, 8, 7, 8, 1.0, passes, None) == INVALID
        assert f(A, A, A, A, 4, 8, 8, 8, 0.0, passes, None) == INVALID
        assert f(A, A, A, A + 2, 4, 8, 8, 8, 1.0, passes, None) == MISALIGNED
    for passes in (0, 1, 4, -2):
        assert f(A, A, A, A, 4, 8, 8, 8, 1.0, passes, None) == INVALID


def test_softmax_rows_16bit_rejects_bad_arguments(lib):
    f = lib.os_softmax_rows_16bit
    for dt in (1, 2):
        assert f(None, A, None, None, 4, 8, 8, 8, 1.0, dt, None) == INVALID
        assert f(A, None, None, None, 4, 8, 8, 8, 1.0, dt, None) == INVALID
        assert f(A, A, None, None, 4, 8, 7, 8, 1.0, dt, None) == INVALID
        assert f(A, A, None, None, 4, 8, 8, 8, -1.0, dt, None) == INVALID
        assert f(A + 1, A, None, None, 4, 8, 8, 8, 1.0, dt, None) == MISALIGNED
        assert f(A, A, A + 2, None, 4, 8, 8, 8, 1.0, dt, None) == MISALIGNED
    for dt in (0, 3, -1):
        assert f(A, A, None, None, 4, 8, 8, 8, 1.0, dt, None) == INVALID


def test_attention_fwd_rejects_bad_arguments(lib):
    f = lib.os_attention_fwd
    ok = (1, 2, 64, 64, 128, 0.1, 0, None)
    assert f(None, A, A, A, None, *ok) == INVALID
    assert f(A, A, A, None, None, *ok) == INVALID
    assert f(A, A, A, A, None, 0, 2, 64, 64, 128, 0.1, 0, None) == INVALID
    assert f(A, A, A, A, None, 1, 2, 0, 64, 128, 0.1, 0, None) == INVALID
    assert f(A, A, A, A, None, 1, 2, 64, 64, 128, 0.0, 0, None) == INVALID
    assert f(A + 2, A, A, A, None, *ok) == MISALIGNED
    assert f(A, A, A, A, None, 1, 2, 64, 64, 64, 0.1, 0, None) == UNSUPPORTED   # D != 128
    assert f(A, A, A, A, None, 1, 2, 64, 32, 128, 0.1, 1, None) == UNSUPPORTED  # causal, Sq != Sk


def test_attention_partial_rejects_bad_arguments(lib):
    f = lib.os_attention_fwd_partial
    ok = (1, 2, 64, 64, 128, 0.1, 0)
    assert f(A, A, A, *ok, None, A, A, 2, 0, None) == INVALID
    assert f(A, A, A, *ok, A, A, A, 2, 2, None) == INVALID    # index past the stride
    assert f(A, A, A, *ok, A, A, A, 0, 0, None) == INVALID
    assert f(A, A, A, *ok, A, A, A + 4, 2, 0, None) == MISALIGNED
    assert f(A, A, A, 1, 2, 64, 32, 128, 0.1, 1, A, A, A, 2, 0, None) == UNSUPPORTED


def test_decode_rejects_bad_arguments(lib):
    f = lib.os_attention_decode_splitkv
    assert f(A, A, A, None, 2, 2, 64, 128, 4, 0.1, A, A, A, None) == INVALID
    assert f(A, A, A, A, 2, 2, 64, 128, 0, 0.1, A, A, A, None) == INVALID
    assert f(A, A, A, A, 2, 2, 64, 128, 4, -0.1, A, A, A, None) == INVALID
    assert f(A, A, A, A, 2, 2, 64, 128, 4, 0.1, A, A, A + 4, None) == MISALIGNED
    assert f(A, A, A, A, 2, 2, 64, 96, 4, 0.1, A, A, A, None) == UNSUPPORTED
    assert f(A, A, A, A, 2, 2, 64, 128, 65, 0.1, A, A, A, None) == UNSUPPORTED


def test_merge_rejects_bad_arguments(lib):
    f = lib.os_merge_partials
    assert f(None, A, A, 4, 16, 128, 1, A, None, None, None, None) == INVALID
    assert f(A, A, A, 4, 16, 128, 1, None, None, None, None, None) == INVALID
    assert f(A, A, A, 0, 16, 128, 1, A, None, None, None, None) == INVALID
    assert f(A, A, A + 8, 4, 16, 128, 1, A, None, None, None, None) == MISALIGNED
    assert f(A, A, A, 4, 65, 128, 1, A, None, None, None, None) == UNSUPPORTED
    assert f(A, A, A, 4, 16, 130, 1, A, None, None, None, None) == UNSUPPORTED


def test_fault_hook_validates_and_disarms(lib):
    f = lib.os_debug_inject_fault
    assert f(3, 0, 0) == INVALID
    assert f(-1, 0, 0) == INVALID
    assert f(1, -1, 0) == INVALID
    assert f(1, 0, -5) == INVALID
    assert f(2, 0, -5) == INVALID
    assert f(2, 0, 1000) == 0  # armed for the next row softmax of this thread
    assert f(0, 0, 0) == 0  # disarm; touches no device


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        oss.softmax_rows(torch.zeros(2, 4))
    with pytest.raises(ValueError):
        oss.attention_fwd(*(torch.zeros(1, 1, 4, 128, dtype=torch.bfloat16) for _ in range(3)))


def test_every_device_call_refuses_host_tensors(lib):
    # the binding has no CPU path: host tensors are refused before any call
    # into the library, for every entry point that takes device tensors
    import torch
    bf16 = torch.bfloat16
    x = torch.zeros(4, 64)
    q = torch.zeros(1, 2, 64, 128, dtype=bf16)
    qd = torch.zeros(1, 2, 128, dtype=bf16)
    kd = torch.zeros(1, 2, 32, 128, dtype=bf16)
    pm = torch.zeros(1, 2, 64, 2)
    po = torch.zeros(1, 2, 64, 2, 128)
    calls = [
        lambda: oss.softmax_rows(x),
        lambda: oss.softmax_rows_16bit(x.to(bf16)),
        lambda: oss.softmax_rows_16bit(x.to(torch.float16)),
        lambda: oss.softmax_rows_multipass(x, 2),
        lambda: oss.softmax_rows_multipass(x, 3),
        lambda: oss.attention_fwd(q, q, q),
        lambda: oss.attention_fwd(q, q, q, causal=True),
        lambda: oss.attention_fwd_partial(q, q, q, pm, pm, po, 0),
        lambda: oss.attention_decode_splitkv(qd, kd, kd, torch.ones(1, dtype=torch.int32), 4),
        lambda: oss.merge_partials(pm, pm, po),
        lambda: oss.merge_partials(pm, pm, po, finalize=False),
    ]
    for i, call in enumerate(calls):
        with pytest.raises((ValueError, TypeError)):
            call()
            pytest.fail(f"call {i} accepted host tensors")
    # a wrong element type is refused as well
    with pytest.raises(TypeError):
        oss.softmax_rows_16bit(x)


def test_binding_refuses_host_outputs(lib):
    # the output check itself (device tensors are not available here): a
    # host tensor, a wrong shape or type is refused before any library call
    import torch
    dev = torch.device("cuda", 0)
    with pytest.raises(ValueError):
        oss._out(torch.zeros(3), "m", torch.float32, (3,), dev)
    with pytest.raises(TypeError):
        oss._out(None, "m", torch.float32, (3,), dev)


def test_partial_rejects_too_many_heads(lib):
    f = lib.os_attention_fwd_partial
    # B * H beyond the kernel's grid bound, as os_attention_fwd
    assert f(A, A, A, 65535, 65, 64, 64, 128, 0.1, 0, A, A, A, 1, 0, None) == UNSUPPORTED
    assert lib.os_attention_fwd(A, A, A, A, None, 65535, 65, 64, 64, 128, 0.1, 0, None) == UNSUPPORTED


def test_rescale_policy_selector(lib):
    f = lib.os_attention_set_rescale_policy
    assert lib.os_attention_rescale_policy() == 0          # threshold by default
    for bad in (-1, 3, 100):
        assert f(bad) == INVALID
        assert lib.os_attention_rescale_policy() == 0      # a refused value changes nothing
    for p in (1, 2, 0):
        assert f(p) == 0 and lib.os_attention_rescale_policy() == p
    oss.set_rescale_policy("on_rise")
    assert oss.rescale_policy() == "on_rise"
    oss.set_rescale_policy("threshold")
