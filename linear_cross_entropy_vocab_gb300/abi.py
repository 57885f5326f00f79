"""ctypes binding of libflce.so (include/flce.h), one Python function per C
entry point, same names. Argument marshalling only: pointers are passed as
integers (``tensor.data_ptr()``), the stream as ``cudaStream_t`` integer.

The library must have been built (``linear_cross_entropy_vocab_gb300.build``
or ``__graft_entry__.build()``); loading fails loudly otherwise. There is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import native_build as _build

FLCE_OK = 0
FLCE_ERR_INVALID_ARG = 1
FLCE_ERR_UNSUPPORTED = 2
FLCE_ERR_WORKSPACE = 3
FLCE_ERR_CUDA = 4
FLCE_ERR_DEVICE_TIMEOUT = 5

FLCE_F32 = 0
FLCE_BF16 = 1
FLCE_F16 = 2

FLCE_RED_NONE = 0
FLCE_RED_SUM = 1
FLCE_RED_MEAN = 2

FLCE_SKIP_IGNORED_ROWS = 1

FLCE_DEVERR_TARGET_RANGE = 1
FLCE_DEVERR_TIMEOUT = 2

REDUCTIONS = {"none": FLCE_RED_NONE, "sum": FLCE_RED_SUM, "mean": FLCE_RED_MEAN}

FLCE_KL_NONE = 0
FLCE_KL_SUM = 1
FLCE_KL_BATCHMEAN = 2
FLCE_KL_MEAN = 3

KL_REDUCTIONS = {"none": FLCE_KL_NONE, "sum": FLCE_KL_SUM, "batchmean": FLCE_KL_BATCHMEAN,
                 "mean": FLCE_KL_MEAN}

# Every symbol include/flce.h declares.
EXPORTS = (
    "flce_forward_workspace_size",
    "flce_forward",
    "flce_forward_noalloc",
    "flce_backward_workspace_size",
    "flce_backward",
    "flce_kl_forward_workspace_size",
    "flce_kl_forward",
    "flce_kl_backward_workspace_size",
    "flce_kl_backward",
    "flce_selftest_wait_timeout",
    "flce_status_string",
    "flce_last_error",
    "flce_device_supported",
    "flce_profile_enable",
    "flce_profile_collect",
)

FLCE_PROFILE_MAX_RECORDS = 8192
FLCE_PROFILE_NAME_LEN = 40


class flce_problem(ctypes.Structure):  # noqa: N801  (C name)
    _fields_ = [
        ("n", ctypes.c_int64),
        ("h", ctypes.c_int64),
        ("v", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("has_bias", ctypes.c_int32),
        ("ignore_index", ctypes.c_int64),
        ("logit_scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("reduction", ctypes.c_int32),
        ("grad_weight_dtype", ctypes.c_int32),
        ("vocab_chunk", ctypes.c_int64),
        ("flags", ctypes.c_int32),
        ("label_smoothing", ctypes.c_float),
        ("z_loss", ctypes.c_float),
        ("reserved", ctypes.c_int32),
    ]


class flce_kl_problem(ctypes.Structure):  # noqa: N801  (C name)
    _fields_ = [
        ("n", ctypes.c_int64),
        ("h", ctypes.c_int64),
        ("v", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("has_bias", ctypes.c_int32),
        ("ignore_index", ctypes.c_int64),
        ("temperature", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("reduction", ctypes.c_int32),
        ("grad_weight_dtype", ctypes.c_int32),
        ("vocab_chunk", ctypes.c_int64),
        ("flags", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class flce_kernel_time(ctypes.Structure):  # noqa: N801  (C name)
    _fields_ = [
        ("name", ctypes.c_char * FLCE_PROFILE_NAME_LEN),
        ("launches", ctypes.c_int32),
        ("total_ms", ctypes.c_double),
    ]


class FlceError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_PROB = ctypes.POINTER(flce_problem)
_KLPROB = ctypes.POINTER(flce_kl_problem)


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libflce.so (built in-tree). Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -m linear_cross_entropy_vocab_gb300.native_build)")
        lib = ctypes.CDLL(path)
        lib.flce_forward_workspace_size.argtypes = [_PROB]
        lib.flce_forward_workspace_size.restype = ctypes.c_size_t
        lib.flce_backward_workspace_size.argtypes = [_PROB]
        lib.flce_backward_workspace_size.restype = ctypes.c_size_t
        lib.flce_forward.argtypes = [_PROB] + [_P] * 15
        lib.flce_forward.argtypes[-2] = ctypes.c_size_t
        lib.flce_forward.restype = ctypes.c_int
        lib.flce_forward_noalloc.argtypes = [_PROB] + [_P] * 13
        lib.flce_forward_noalloc.restype = ctypes.c_int
        lib.flce_backward.argtypes = [_PROB] + [_P] * 14
        lib.flce_backward.argtypes[-2] = ctypes.c_size_t
        lib.flce_backward.restype = ctypes.c_int
        lib.flce_kl_forward_workspace_size.argtypes = [_KLPROB]
        lib.flce_kl_forward_workspace_size.restype = ctypes.c_size_t
        lib.flce_kl_backward_workspace_size.argtypes = [_KLPROB]
        lib.flce_kl_backward_workspace_size.restype = ctypes.c_size_t
        lib.flce_kl_forward.argtypes = [_KLPROB] + [_P] * 14
        lib.flce_kl_forward.argtypes[-2] = ctypes.c_size_t
        lib.flce_kl_forward.restype = ctypes.c_int
        lib.flce_kl_backward.argtypes = [_KLPROB] + [_P] * 16
        lib.flce_kl_backward.argtypes[-2] = ctypes.c_size_t
        lib.flce_kl_backward.restype = ctypes.c_int
        lib.flce_selftest_wait_timeout.argtypes = [_P, _P, ctypes.c_double, _P]
        lib.flce_selftest_wait_timeout.restype = ctypes.c_int
        lib.flce_status_string.argtypes = [ctypes.c_int]
        lib.flce_status_string.restype = ctypes.c_char_p
        lib.flce_last_error.argtypes = []
        lib.flce_last_error.restype = ctypes.c_char_p
        lib.flce_device_supported.argtypes = []
        lib.flce_device_supported.restype = ctypes.c_int
        lib.flce_profile_enable.argtypes = [ctypes.c_int]
        lib.flce_profile_enable.restype = ctypes.c_int
        lib.flce_profile_collect.argtypes = [ctypes.POINTER(flce_kernel_time), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int32)]
        lib.flce_profile_collect.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, call: str):
    if status != FLCE_OK:
        lib = load()
        name = lib.flce_status_string(status).decode()
        detail = lib.flce_last_error().decode()
        raise FlceError(status, f"{call}: {name}: {detail}")


def make_problem(n, h, v, dtype, has_bias, ignore_index=-100, logit_scale=1.0,
                 softcap=None, reduction="mean", grad_weight_dtype=None,
                 vocab_chunk=0, skip_ignored=False, label_smoothing=0.0,
                 z_loss=0.0) -> flce_problem:
    p = flce_problem()
    p.n, p.h, p.v = int(n), int(h), int(v)
    p.dtype = int(dtype)
    p.has_bias = 1 if has_bias else 0
    p.ignore_index = int(ignore_index)
    p.logit_scale = float(logit_scale)
    p.softcap = float(softcap) if softcap is not None else 0.0
    p.reduction = REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction)
    p.grad_weight_dtype = int(dtype if grad_weight_dtype is None else grad_weight_dtype)
    p.vocab_chunk = int(vocab_chunk)
    p.flags = FLCE_SKIP_IGNORED_ROWS if skip_ignored else 0
    p.label_smoothing = float(label_smoothing)
    p.z_loss = float(z_loss)
    p.reserved = 0
    return p


def flce_forward_workspace_size(p: flce_problem) -> int:
    return load().flce_forward_workspace_size(ctypes.byref(p))


def flce_backward_workspace_size(p: flce_problem) -> int:
    return load().flce_backward_workspace_size(ctypes.byref(p))


def flce_forward(p, hidden, weight, bias, targets, loss_rows, lse_rows, correct_rows,
                 entropy_rows, loss_out, metrics_out, n_valid, err_word, workspace,
                 workspace_bytes, stream, check=True) -> int:
    st = load().flce_forward(ctypes.byref(p), hidden, weight, bias, targets, loss_rows,
                             lse_rows, correct_rows, entropy_rows, loss_out, metrics_out,
                             n_valid, err_word, workspace, workspace_bytes, stream)
    if check:
        _check(st, "flce_forward")
    return st


def flce_forward_noalloc(p, hidden, weight, bias, targets, loss_rows, lse_rows, correct_rows,
                         entropy_rows, loss_out, metrics_out, n_valid, err_word, stream,
                         check=True) -> int:
    """flce_forward without a workspace: for callers that cannot allocate
    device memory; the scratch is a fixed 16 MiB array inside the library."""
    st = load().flce_forward_noalloc(ctypes.byref(p), hidden, weight, bias, targets, loss_rows,
                                     lse_rows, correct_rows, entropy_rows, loss_out,
                                     metrics_out, n_valid, err_word, stream)
    if check:
        _check(st, "flce_forward_noalloc")
    return st


def flce_backward(p, hidden, weight, bias, targets, lse_rows, n_valid, grad_out,
                  grad_hidden, grad_weight, grad_bias, err_word, workspace,
                  workspace_bytes, stream, check=True) -> int:
    st = load().flce_backward(ctypes.byref(p), hidden, weight, bias, targets, lse_rows,
                              n_valid, grad_out, grad_hidden, grad_weight, grad_bias,
                              err_word, workspace, workspace_bytes, stream)
    if check:
        _check(st, "flce_backward")
    return st


def make_kl_problem(n, h, v, dtype, has_bias, ignore_index=-100, temperature=1.0, eps=1e-10,
                    reduction="batchmean", grad_weight_dtype=None, vocab_chunk=0,
                    skip_ignored=False) -> flce_kl_problem:
    p = flce_kl_problem()
    p.n, p.h, p.v = int(n), int(h), int(v)
    p.dtype = int(dtype)
    p.has_bias = 1 if has_bias else 0
    p.ignore_index = int(ignore_index)
    p.temperature = float(temperature)
    p.eps = float(eps)
    p.reduction = KL_REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction)
    p.grad_weight_dtype = int(dtype if grad_weight_dtype is None else grad_weight_dtype)
    p.vocab_chunk = int(vocab_chunk)
    p.flags = FLCE_SKIP_IGNORED_ROWS if skip_ignored else 0
    p.reserved = 0
    return p


def flce_kl_forward_workspace_size(p: flce_kl_problem) -> int:
    return load().flce_kl_forward_workspace_size(ctypes.byref(p))


def flce_kl_backward_workspace_size(p: flce_kl_problem) -> int:
    return load().flce_kl_backward_workspace_size(ctypes.byref(p))


def flce_kl_forward(p, hidden, weight, bias, target_probs, labels, loss_rows, lse_rows,
                    qsum_rows, loss_out, n_counted, err_word, workspace, workspace_bytes,
                    stream, check=True) -> int:
    st = load().flce_kl_forward(ctypes.byref(p), hidden, weight, bias, target_probs, labels,
                                loss_rows, lse_rows, qsum_rows, loss_out, n_counted, err_word,
                                workspace, workspace_bytes, stream)
    if check:
        _check(st, "flce_kl_forward")
    return st


def flce_kl_backward(p, hidden, weight, bias, target_probs, labels, lse_rows, qsum_rows,
                     n_counted, grad_out, grad_hidden, grad_weight, grad_bias, err_word,
                     workspace, workspace_bytes, stream, check=True) -> int:
    st = load().flce_kl_backward(ctypes.byref(p), hidden, weight, bias, target_probs, labels,
                                 lse_rows, qsum_rows, n_counted, grad_out, grad_hidden,
                                 grad_weight, grad_bias, err_word, workspace, workspace_bytes,
                                 stream)
    if check:
        _check(st, "flce_kl_backward")
    return st


def flce_selftest_wait_timeout(err_word, result, budget_s, stream, check=True) -> int:
    """Run the bounded-wait self-test (see include/flce.h)."""
    st = load().flce_selftest_wait_timeout(err_word, result, float(budget_s), stream)
    if check:
        _check(st, "flce_selftest_wait_timeout")
    return st


def flce_status_string(status: int) -> str:
    return load().flce_status_string(int(status)).decode()


def flce_last_error() -> str:
    return load().flce_last_error().decode()


def flce_device_supported() -> bool:
    return bool(load().flce_device_supported())


def flce_profile_enable(enable: bool) -> None:
    _check(load().flce_profile_enable(1 if enable else 0), "flce_profile_enable")


def flce_profile_collect(max_entries: int = 16):
    """Returns ({kernel role: (launches, total_ms)}, dropped launches)."""
    arr = (flce_kernel_time * max_entries)()
    dropped = ctypes.c_int32(0)
    n = load().flce_profile_collect(arr, max_entries, ctypes.byref(dropped))
    if n < 0:
        raise FlceError(FLCE_ERR_CUDA, "flce_profile_collect: CUDA error")
    return ({arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n)},
            dropped.value)
