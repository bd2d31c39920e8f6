"""ctypes binding of libffpa.so: argument marshalling only.

Each Python function here has the name of the C entry point it calls and does
nothing but fill ``ffpa_tensor_t`` descriptors from torch tensors (pointer,
dtype, sizes, strides) and pass the current CUDA stream.  Every step of the
computation runs in the library's kernels.  If the library cannot be built or
loaded, loading raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

FFPA_F16, FFPA_BF16, FFPA_F32 = 0, 1, 2
STATUS = {0: "FFPA_OK", 1: "FFPA_ERR_INVALID_ARG", 2: "FFPA_ERR_UNSUPPORTED", 3: "FFPA_ERR_ALIGNMENT",
          4: "FFPA_ERR_CUDA", 5: "FFPA_ERR_TIMEOUT", 6: "FFPA_ERR_SCRATCH_LIMIT"}
EXPORTS = ("ffpa_fwd", "ffpa_bwd", "ffpa_fwd_dropout", "ffpa_bwd_dropout", "ffpa_fwd_decode_noalloc", "ffpa_status_string", "ffpa_check_status",
           "ffpa_set_timing_events", "ffpa_selftest_wait_timeout", "ffpa_version")


class FfpaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class FfpaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


_LIB = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libffpa.so (building it first if it is missing or stale)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    lib_path = path or _build.build()
    if not os.path.exists(lib_path):
        raise FileNotFoundError(lib_path)
    lib = ctypes.CDLL(lib_path)
    P = ctypes.POINTER(FfpaTensor)
    lib.ffpa_fwd.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.ffpa_fwd.restype = ctypes.c_int
    lib.ffpa_bwd.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_float, P, P, P, P, P, P, ctypes.c_void_p]
    lib.ffpa_bwd.restype = ctypes.c_int
    D, U64, U32 = ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32
    lib.ffpa_fwd_dropout.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_float, D, U64, U32, P, P, ctypes.c_void_p]
    lib.ffpa_fwd_dropout.restype = ctypes.c_int
    lib.ffpa_bwd_dropout.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_float, D, U64, U32, P, P, P, P, P, P,
                                     ctypes.c_void_p]
    lib.ffpa_bwd_dropout.restype = ctypes.c_int
    lib.ffpa_fwd_decode_noalloc.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.ffpa_fwd_decode_noalloc.restype = ctypes.c_int
    lib.ffpa_status_string.argtypes = [ctypes.c_int]
    lib.ffpa_status_string.restype = ctypes.c_char_p
    lib.ffpa_check_status.argtypes = [ctypes.c_void_p]
    lib.ffpa_check_status.restype = ctypes.c_int
    lib.ffpa_set_timing_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    lib.ffpa_set_timing_events.restype = ctypes.c_int
    lib.ffpa_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
    lib.ffpa_selftest_wait_timeout.restype = ctypes.c_int
    lib.ffpa_version.argtypes = []
    lib.ffpa_version.restype = ctypes.c_int
    if path is None:
        _LIB = lib
    return lib


def _dtype_code(t) -> int:
    import torch
    return {torch.float16: FFPA_F16, torch.bfloat16: FFPA_BF16, torch.float32: FFPA_F32}.get(t.dtype, -1)


def describe(t, as_lse: bool = False):
    """ffpa_tensor_t for a torch tensor (4-D; an lse [B,H,N] gets a trailing size-1 dim)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("ffpa tensors must be CUDA tensors (the library takes device pointers)")
    d = FfpaTensor()
    d.data = t.data_ptr()
    d.dtype = _dtype_code(t)
    d.reserved = 0
    shape, stride = list(t.shape), list(t.stride())
    if as_lse and len(shape) == 3:
        shape, stride = shape + [1], stride + [1]
    if len(shape) != 4:
        raise ValueError("ffpa tensors are 4-D")
    for i in range(4):
        d.shape[i] = shape[i]
        d.stride[i] = stride[i]
    return d


def check_devices(tensors, current: int) -> None:
    """All tensors of one call on one CUDA device, and that device the current
    one: the library encodes its TMA maps, reads its status word and launches
    on the current device, so a tensor elsewhere would be addressed from the
    wrong GPU."""
    devs = {(t.device.type, t.device.index) for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"ffpa tensors must all be on one CUDA device, got {sorted(map(str, devs))}")
    kind, index = devs.pop()
    if kind != "cuda":
        raise ValueError("ffpa tensors must be CUDA tensors (the library takes device pointers)")
    if index != current:
        raise ValueError(f"ffpa tensors are on cuda:{index} but the current device is cuda:{current}; "
                         f"call torch.cuda.set_device({index}) or use torch.cuda.device({index}) first")


def _current_device() -> int:
    import torch
    return torch.cuda.current_device()


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _raise(code: int):
    if code != 0:
        raise FfpaError(code, load().ffpa_status_string(code).decode())


def ffpa_fwd(q, k, v, bias, causal, scale, out, lse, stream=None) -> None:
    """Call ffpa_fwd on torch tensors (device memory); raises FfpaError on a non-zero status."""
    lib = load()
    check_devices((q, k, v, bias, out, lse), _current_device())
    ds = [describe(q), describe(k), describe(v), describe(bias), describe(out), describe(lse, as_lse=True)]
    rc = lib.ffpa_fwd(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), _ref(ds[3]), int(causal), float(scale),
                      _ref(ds[4]), _ref(ds[5]), _stream(stream))
    _raise(rc)


def ffpa_fwd_dropout(q, k, v, bias, causal, scale, dropout_p, seed, offset, out, lse, stream=None) -> None:
    """Call ffpa_fwd_dropout (the forward with dropout on P); raises FfpaError on a non-zero status."""
    lib = load()
    check_devices((q, k, v, bias, out, lse), _current_device())
    ds = [describe(q), describe(k), describe(v), describe(bias), describe(out), describe(lse, as_lse=True)]
    rc = lib.ffpa_fwd_dropout(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), _ref(ds[3]), int(causal), float(scale),
                              float(dropout_p), int(seed), int(offset), _ref(ds[4]), _ref(ds[5]), _stream(stream))
    _raise(rc)


def ffpa_bwd_dropout(q, k, v, bias, causal, scale, dropout_p, seed, offset, out, lse, dout, dq, dk, dv,
                     stream=None) -> None:
    """Call ffpa_bwd_dropout (the backward of ffpa_fwd_dropout with the same p, seed and offset)."""
    lib = load()
    check_devices((q, k, v, bias, out, lse, dout, dq, dk, dv), _current_device())
    ds = [describe(x) for x in (q, k, v, bias, out)] + [describe(lse, as_lse=True)] + \
        [describe(x) for x in (dout, dq, dk, dv)]
    rc = lib.ffpa_bwd_dropout(*[_ref(x) for x in ds[:4]], int(causal), float(scale), float(dropout_p), int(seed),
                              int(offset), *[_ref(x) for x in ds[4:]], _stream(stream))
    _raise(rc)


def ffpa_fwd_decode_noalloc(q, k, v, bias, causal, scale, out, lse, stream=None) -> None:
    """Call ffpa_fwd_decode_noalloc (decode forward, Nq <= 16, no device allocation)."""
    lib = load()
    check_devices((q, k, v, bias, out, lse), _current_device())
    ds = [describe(q), describe(k), describe(v), describe(bias), describe(out), describe(lse, as_lse=True)]
    rc = lib.ffpa_fwd_decode_noalloc(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), _ref(ds[3]), int(causal),
                                     float(scale), _ref(ds[4]), _ref(ds[5]), _stream(stream))
    _raise(rc)


def ffpa_bwd(q, k, v, bias, causal, scale, out, lse, dout, dq, dk, dv, stream=None) -> None:
    """Call ffpa_bwd on torch tensors (device memory); raises FfpaError on a non-zero status."""
    lib = load()
    check_devices((q, k, v, bias, out, lse, dout, dq, dk, dv), _current_device())
    ds = [describe(x) for x in (q, k, v, bias, out)] + [describe(lse, as_lse=True)] + \
        [describe(x) for x in (dout, dq, dk, dv)]
    rc = lib.ffpa_bwd(*[_ref(x) for x in ds[:4]], int(causal), float(scale), *[_ref(x) for x in ds[4:]],
                      _stream(stream))
    _raise(rc)


def ffpa_check_status(stream=None) -> int:
    return load().ffpa_check_status(_stream(stream))


def ffpa_status_string(code: int) -> str:
    return load().ffpa_status_string(code).decode()


def ffpa_set_timing_events(events) -> None:
    """Register torch.cuda.Event objects (enable_timing=True) the library records between its launches."""
    handles = [int(e.cuda_event) for e in (events or [])]
    if any(h == 0 for h in handles):
        raise ValueError("record each torch.cuda.Event once before registering it (torch creates events lazily)")
    arr = (ctypes.c_void_p * max(1, len(handles)))(*handles)
    _raise(load().ffpa_set_timing_events(arr if handles else None, len(handles)))


def ffpa_selftest_wait_timeout(stream=None) -> None:
    """Launch the timeout self-check (a wait that nothing completes); see include/ffpa.h."""
    _raise(load().ffpa_selftest_wait_timeout(_stream(stream)))


def ffpa_version() -> int:
    return load().ffpa_version()
