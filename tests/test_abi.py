"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every entry point include/ffpa.h declares, and
reject every malformed call on the host, before any CUDA call, with the
documented status code.  Descriptors here carry fake (but aligned) device
addresses: validation never dereferences them.
"""
import ctypes
import os
import re

import pytest

from head_dim_attention_gb300 import _lib
from head_dim_attention_gb300._lib import FfpaTensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, ALIGN = 0, 1, 2, 3


def header_symbols():
    text = open(os.path.join(ROOT, "include", "ffpa.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(ffpa_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert set(syms) == set(_lib.EXPORTS)
    for s in syms:
        assert hasattr(lib, s), s


def test_version_and_status_strings(lib):
    assert lib.ffpa_version() >= 100
    for code in range(6):
        assert lib.ffpa_status_string(code)
    assert lib.ffpa_status_string(99) == b"unknown status"


ADDR = 1 << 20  # fake, 16-byte aligned


def t4(shape, dtype=_lib.FFPA_BF16, addr=ADDR, stride=None):
    d = FfpaTensor()
    d.data = addr
    d.dtype = dtype
    d.reserved = 0
    if stride is None:
        stride = [shape[1] * shape[2] * shape[3], shape[2] * shape[3], shape[3], 1]
    for i in range(4):
        d.shape[i] = shape[i]
        d.stride[i] = stride[i]
    return d


def fwd(lib, q, k, v, out, bias=None, lse=None, causal=0, scale=0.05):
    r = lambda x: None if x is None else ctypes.byref(x)
    return lib.ffpa_fwd(r(q), r(k), r(v), r(bias), causal, scale, r(out), r(lse), None)


def good(B=1, Hq=4, Hkv=2, Nq=100, Nkv=200, D=512):
    return t4([B, Hq, Nq, D]), t4([B, Hkv, Nkv, D]), t4([B, Hkv, Nkv, D]), t4([B, Hq, Nq, D])


@pytest.mark.parametrize("case,expect", [
    ("null_q", INVALID), ("null_data", INVALID), ("gqa_indivisible", INVALID), ("nq_zero", INVALID),
    ("kv_shape_mismatch", INVALID), ("out_shape", INVALID), ("scale_zero", INVALID), ("scale_nan", INVALID),
    ("causal_2", INVALID), ("d_not_64", UNSUPPORTED), ("d_too_big", UNSUPPORTED), ("f32_inputs", UNSUPPORTED),
    ("dtype_mix", INVALID), ("inner_stride", UNSUPPORTED), ("misaligned_ptr", ALIGN), ("row_stride_odd", ALIGN),
    ("bias_f16", UNSUPPORTED), ("bias_shape", INVALID), ("lse_shape", INVALID), ("lse_dtype", UNSUPPORTED),
    ("reserved", INVALID),
])
def test_fwd_rejects(lib, case, expect):
    q, k, v, out = good()
    bias = lse = None
    causal, scale = 0, 0.05
    if case == "null_q":
        q = None
    elif case == "null_data":
        k.data = None
    elif case == "gqa_indivisible":
        q, out = t4([1, 3, 100, 512]), t4([1, 3, 100, 512])
    elif case == "nq_zero":
        q, out = t4([1, 4, 0, 512], stride=[0, 0, 512, 1]), t4([1, 4, 0, 512], stride=[0, 0, 512, 1])
    elif case == "kv_shape_mismatch":
        v = t4([1, 2, 201, 512])
    elif case == "out_shape":
        out = t4([1, 4, 101, 512])
    elif case == "scale_zero":
        scale = 0.0
    elif case == "scale_nan":
        scale = float("nan")
    elif case == "causal_2":
        causal = 2
    elif case == "d_not_64":
        q, k, v, out = good(D=96)
    elif case == "d_too_big":
        q, k, v, out = good(D=1088)
    elif case == "f32_inputs":
        q, k, v, out = (t4(list(x.shape), dtype=_lib.FFPA_F32) for x in (q, k, v, out))
    elif case == "dtype_mix":
        k.dtype = _lib.FFPA_F16
    elif case == "inner_stride":
        q.stride[3] = 2
    elif case == "misaligned_ptr":
        v.data = ADDR + 8
    elif case == "row_stride_odd":
        k.stride[2] = 516
    elif case == "bias_f16":
        bias = t4([1, 1, 1, 200], dtype=_lib.FFPA_F16)
    elif case == "bias_shape":
        bias = t4([1, 1, 1, 199], dtype=_lib.FFPA_F32)
    elif case == "lse_shape":
        lse = t4([1, 4, 99, 1], dtype=_lib.FFPA_F32)
    elif case == "lse_dtype":
        lse = t4([1, 4, 100, 1], dtype=_lib.FFPA_BF16)
    elif case == "reserved":
        q.reserved = 7
    assert fwd(lib, q, k, v, out, bias, lse, causal, scale) == expect


def test_bwd_rejects(lib):
    q, k, v, out = good()
    lse = t4([1, 4, 100, 1], dtype=_lib.FFPA_F32)
    dout, dq, dk, dv = t4([1, 4, 100, 512]), t4([1, 4, 100, 512]), t4([1, 2, 200, 512]), t4([1, 2, 200, 512])
    r = ctypes.byref
    call = lambda **over: lib.ffpa_bwd(
        r(over.get("q", q)), r(k), r(v), None, 0, 0.05, r(out),
        None if over.get("lse", lse) is None else r(over.get("lse", lse)), r(dout), r(dq),
        r(over.get("dk", dk)), r(dv), None)
    assert call(lse=None) == INVALID          # lse is required by the backward
    assert call(dk=t4([1, 4, 200, 512])) == INVALID
    assert call(q=t4([1, 4, 100, 320])) == INVALID


@pytest.mark.parametrize("p,D,expect", [(1.0, 512, INVALID), (-0.1, 512, INVALID), (float("nan"), 512, INVALID),
                                         (1.5, 512, INVALID), (0.1, 256, UNSUPPORTED), (0.1, 64, UNSUPPORTED)])
def test_dropout_rejects(lib, p, D, expect):
    # dropout: 0 <= p < 1, and only the D = 320 .. 1024 kernels draw keep masks
    q, k, v, out = good(D=D)
    lse = t4([1, 4, 100, 1], dtype=_lib.FFPA_F32)
    r = ctypes.byref
    assert lib.ffpa_fwd_dropout(r(q), r(k), r(v), None, 0, 0.05, p, 7, 0, r(out), r(lse), None) == expect
    dout, dq, dk, dv = t4([1, 4, 100, D]), t4([1, 4, 100, D]), t4([1, 2, 200, D]), t4([1, 2, 200, D])
    assert lib.ffpa_bwd_dropout(r(q), r(k), r(v), None, 0, 0.05, p, 7, 0, r(out), r(lse), r(dout), r(dq), r(dk),
                                r(dv), None) == expect


def test_binding_rejects_host_tensors():
    # the binding passes data pointers as device addresses: host tensors never reach the library
    import torch
    with pytest.raises(ValueError):
        _lib.describe(torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16))
    assert _lib.describe(None) is None


def test_binding_checks_devices():
    # every tensor of a call on one CUDA device, and that device the current one
    import types

    import torch
    on = lambda kind, index=None: types.SimpleNamespace(device=torch.device(kind, index))  # noqa: E731
    _lib.check_devices((on("cuda", 0), on("cuda", 0), None), 0)
    _lib.check_devices((on("cuda", 1), on("cuda", 1)), 1)
    with pytest.raises(ValueError, match="one CUDA device"):
        _lib.check_devices((on("cuda", 0), on("cuda", 1)), 0)
    with pytest.raises(ValueError, match="current device"):
        _lib.check_devices((on("cuda", 1), on("cuda", 1)), 0)
    with pytest.raises(ValueError, match="CUDA tensors"):
        _lib.check_devices((on("cpu"),), 0)
