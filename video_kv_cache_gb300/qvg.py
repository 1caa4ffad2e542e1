"""ctypes binding of libqvg's C ABI (include/qvg.h), with the same names.

This module only marshals arguments: every step of the compression path runs in the CUDA
kernels of libqvg.so.  There is no fallback; if the library is missing or does not load,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqvg.so")

QVG_OK = 0
QVG_ERR_INVALID_ARG = 1
QVG_ERR_UNSUPPORTED = 2
QVG_ERR_WORKSPACE = 3
QVG_ERR_CUDA = 4
QVG_ERR_DEVICE = 5
QVG_ERR_SCRATCH_LIMIT = 6
QVG_STATIC_SCRATCH_BYTES = 64 << 20

QVG_DEV_NONFINITE = 0x1
QVG_DEV_TIMEOUT = 0x2
QVG_DEV_BAD_INDEX = 0x4

QVG_F16, QVG_BF16, QVG_F32 = 0, 1, 2
QVG_QSCHEME_SYMMETRIC, QVG_QSCHEME_MIDRISE = 0, 1
QVG_STEP_PLANES, QVG_STEP_GEMM, QVG_STEP_REFINE = 1, 2, 4
QVG_CENTROIDS_F32, QVG_CENTROIDS_F16, QVG_CENTROIDS_BF16 = 0, 1, 2


class qvg_quant_params(ctypes.Structure):
    _fields_ = [
        ("n_tensors", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("N", ctypes.c_int64),
        ("C", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("iters", ctypes.c_int32),
        ("in_dtype", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("tensor_id_base", ctypes.c_int64),
        ("x_stride", ctypes.c_int64),
        ("token_offset", ctypes.c_int64),
        ("token_capacity", ctypes.c_int64),
        ("table_index", ctypes.c_int32),
        ("n_tables", ctypes.c_int32),
        ("warm_stride", ctypes.c_int64),
        ("qscheme", ctypes.c_int32),
        ("centroid_format", ctypes.c_int32),
    ]


class qvg_buffers(ctypes.Structure):
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("pi", ctypes.c_void_p),
        ("centroids", ctypes.c_void_p),
    ]


class qvg_dequant_params(ctypes.Structure):
    _fields_ = [
        ("n_tensors", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("N", ctypes.c_int64),
        ("C", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("chunk_len", ctypes.c_int64),
        ("token_capacity", ctypes.c_int64),
        ("n_tables", ctypes.c_int32),
        ("out_stride", ctypes.c_int64),
        ("qscheme", ctypes.c_int32),
    ]


class qvg_attention_params(ctypes.Structure):
    _fields_ = [
        ("n_heads", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("M", ctypes.c_int32),
        ("N", ctypes.c_int64),
        ("C", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("qscheme", ctypes.c_int32),
        ("chunk_len", ctypes.c_int64),
        ("token_capacity", ctypes.c_int64),
        ("n_tables", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("k_first", ctypes.c_int64),
        ("v_first", ctypes.c_int64),
        ("tensor_step", ctypes.c_int64),
    ]


# Every symbol include/qvg.h declares, with its ctypes signature.
SIGNATURES = {
    "qvg_quantize_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(qvg_quant_params)]),
    "qvg_quantize": (ctypes.c_int, [ctypes.POINTER(qvg_quant_params), ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.POINTER(qvg_buffers),
                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                     ctypes.c_void_p]),
    "qvg_quantize_static": (ctypes.c_int, [ctypes.POINTER(qvg_quant_params), ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.POINTER(qvg_buffers),
                                            ctypes.c_void_p, ctypes.c_void_p]),
    "qvg_reassign": (ctypes.c_int, [ctypes.POINTER(qvg_quant_params), ctypes.c_void_p,
                                    ctypes.POINTER(qvg_buffers), ctypes.c_void_p,
                                    ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "qvg_reassign_steps": (ctypes.c_int, [ctypes.POINTER(qvg_quant_params), ctypes.c_void_p,
                                          ctypes.POINTER(qvg_buffers), ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p,
                                          ctypes.c_void_p]),
    "qvg_selftest_assign_timeout": (ctypes.c_int, [ctypes.POINTER(qvg_quant_params),
                                                   ctypes.c_void_p, ctypes.POINTER(qvg_buffers),
                                                   ctypes.c_void_p, ctypes.c_size_t,
                                                   ctypes.c_void_p, ctypes.c_void_p]),
    "qvg_dequantize": (ctypes.c_int, [ctypes.POINTER(qvg_dequant_params),
                                      ctypes.POINTER(qvg_buffers), ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "qvg_attention_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(qvg_attention_params)]),
    "qvg_attention": (ctypes.c_int, [ctypes.POINTER(qvg_attention_params), ctypes.c_void_p,
                                     ctypes.POINTER(qvg_buffers), ctypes.POINTER(qvg_buffers),
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.c_void_p, ctypes.c_void_p]),
    "qvg_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qvg_version": (ctypes.c_uint32, []),
}

_lock = threading.Lock()
_lib = None


class QVGError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (status %d)" % (what, qvg_status_string(code)
                                                        if _lib is not None else "?", code))


def load(path: str | None = None):
    """Load libqvg.so (once).  Raises if it is missing: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libqvg.so not found at %s; build it with "
                               "video_kv_cache_gb300.build.build()" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ref(obj):
    return ctypes.byref(obj) if obj is not None else None


def qvg_quantize_workspace_bytes(params: qvg_quant_params) -> int:
    return int(load().qvg_quantize_workspace_bytes(_ref(params)))


def qvg_quantize(params: qvg_quant_params, X: int, warm_centroids: int | None,
                 out: qvg_buffers, workspace: int, workspace_bytes: int,
                 dev_status: int | None, stream: int | None) -> int:
    return int(load().qvg_quantize(_ref(params), X, warm_centroids, _ref(out),
                                   workspace, workspace_bytes, dev_status, stream))


def qvg_quantize_static(params: qvg_quant_params, X: int, warm_centroids: int | None,
                        out: qvg_buffers, dev_status: int | None, stream: int | None) -> int:
    return int(load().qvg_quantize_static(_ref(params), X, warm_centroids, _ref(out),
                                          dev_status, stream))


def qvg_reassign(params: qvg_quant_params, X: int, out: qvg_buffers, workspace: int,
                 workspace_bytes: int, dev_status: int | None, stream: int | None) -> int:
    return int(load().qvg_reassign(_ref(params), X, _ref(out), workspace, workspace_bytes,
                                   dev_status, stream))


def qvg_reassign_steps(params: qvg_quant_params, X: int, out: qvg_buffers, workspace: int,
                       workspace_bytes: int, steps: int, dev_status: int | None,
                       stream: int | None) -> int:
    return int(load().qvg_reassign_steps(_ref(params), X, _ref(out), workspace, workspace_bytes,
                                         steps, dev_status, stream))


def qvg_selftest_assign_timeout(params: qvg_quant_params, X: int, out: qvg_buffers,
                                workspace: int, workspace_bytes: int, dev_status: int | None,
                                stream: int | None) -> int:
    return int(load().qvg_selftest_assign_timeout(_ref(params), X, _ref(out), workspace,
                                                  workspace_bytes, dev_status, stream))


def qvg_dequantize(params: qvg_dequant_params, inp: qvg_buffers, X_hat: int,
                   dev_status: int | None, stream: int | None) -> int:
    return int(load().qvg_dequantize(_ref(params), _ref(inp), X_hat,
                                     dev_status, stream))


def qvg_attention_workspace_bytes(params: qvg_attention_params) -> int:
    return int(load().qvg_attention_workspace_bytes(_ref(params)))


def qvg_attention(params: qvg_attention_params, Q: int, k_cache: qvg_buffers,
                  v_cache: qvg_buffers, O: int, workspace: int | None, workspace_bytes: int,
                  dev_status: int | None, stream: int | None) -> int:
    return int(load().qvg_attention(_ref(params), Q, _ref(k_cache), _ref(v_cache), O,
                                    workspace, workspace_bytes, dev_status, stream))


def qvg_status_string(code: int) -> str:
    return load().qvg_status_string(code).decode()


def qvg_version() -> int:
    return int(load().qvg_version())
