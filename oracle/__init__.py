"""Oracle for the Quant VideoGen KV-cache compression path.

TEST INFRASTRUCTURE ONLY.  A plain, slow fp64 CPU statement of what the method computes,
written in C (``qvg_oracle.c``) and wrapped here with ctypes.  Only ``tests/``, the
package smoke check and the benchmark's CPU-baseline leg may import it; the product
library never does, and this module imports nothing from the product package.

The method steps and the readings taken where the pages are silent are documented at the
top of ``qvg_oracle.c``.  Every array crossing this wrapper is a numpy array in C order.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qvg_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liborc.so")
_lock = threading.Lock()
_lib = None

_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")


def compile_source(src: str, so: str) -> str:
    """Compile a C source of the oracle into the shared library `so` (ISO C11, no FP
    contraction, the flags every build of the oracle uses)."""
    tmp = so + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-O2", "-ffp-contract=off",
           "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, so)
    return so


def build(force: bool = False) -> str:
    """Compile the oracle and return the .so path."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    return compile_source(_SRC, _SO)


def _load():
    """The oracle library.  QVG_ORACLE_LIB, if set, names a prebuilt copy to load instead:
    the planted-mistake tests use it to run the pins against a mutated oracle."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(os.environ.get("QVG_ORACLE_LIB") or build())
        c = ctypes
        lib.orc_e4m3_decode.restype = c.c_double
        lib.orc_e4m3_decode.argtypes = [c.c_uint8]
        lib.orc_e4m3_encode.restype = c.c_uint8
        lib.orc_e4m3_encode.argtypes = [c.c_double]
        lib.orc_e4m3_encode_n.restype = None
        lib.orc_e4m3_encode_n.argtypes = [_f64p, c.c_int64, _u8p]
        lib.orc_e4m3_decode_n.restype = None
        lib.orc_e4m3_decode_n.argtypes = [_u8p, c.c_int64, _f64p]
        lib.orc_init_indices.restype = c.c_int
        lib.orc_init_indices.argtypes = [c.c_uint64, c.c_int64, c.c_int, c.c_int64, c.c_int, _i64p]
        lib.orc_assign.restype = None
        lib.orc_assign.argtypes = [_f64p, c.c_int64, c.c_int, _f32p, c.c_int, _i32p, _f64p]
        lib.orc_update.restype = None
        lib.orc_update.argtypes = [_f64p, c.c_int64, c.c_int, _i32p, c.c_int, _f32p, _i64p]
        lib.orc_objective.restype = c.c_double
        lib.orc_objective.argtypes = [_f64p, c.c_int64, c.c_int, _i32p, _f32p]
        lib.orc_subtract.restype = None
        lib.orc_subtract.argtypes = [_f64p, c.c_int64, c.c_int, _i32p, _f32p]
        lib.orc_lloyd.restype = None
        lib.orc_lloyd.argtypes = [_f64p, c.c_int64, c.c_int, c.c_int, c.c_int, _f32p, _i32p]
        lib.orc_encode.restype = None
        lib.orc_encode.argtypes = [_f64p, c.c_int64, c.c_int, c.c_int, c.c_int, c.c_int, _u8p,
                                   _u8p]
        lib.orc_decode_codes.restype = None
        lib.orc_decode_codes.argtypes = [_u8p, _u8p, c.c_int64, c.c_int, c.c_int, c.c_int,
                                         c.c_int, _f64p]
        lib.orc_dequantize.restype = None
        lib.orc_dequantize.argtypes = [_u8p, _u8p, _u8p, _f32p, c.c_int64, c.c_int, c.c_int,
                                       c.c_int, c.c_int, c.c_int, c.c_int, _f64p]
        lib.orc_quantize.restype = c.c_int
        lib.orc_quantize.argtypes = [c.c_int64, c.c_int64, c.c_int, c.c_int, c.c_int, c.c_int,
                                     c.c_int, c.c_int, c.c_uint64, c.c_int64, _f64p,
                                     c.c_void_p, _u8p, _u8p, _u8p, _f32p, _f64p, c.c_int,
                                     c.c_int, c.c_int]
        lib.orc_store_n.restype = None
        lib.orc_store_n.argtypes = [_f64p, c.c_int64, c.c_int, _f32p]
        lib.orc_num_cores.restype = c.c_int
        lib.orc_num_cores.argtypes = []
        _lib = lib
        return lib


# ---------------------------------------------------------------------------------------
# Input decoding (exact): fp16 and bf16 values are exactly representable in fp64.
# ---------------------------------------------------------------------------------------

def decode_input(x) -> np.ndarray:
    """fp16 / bf16 / fp32 array (numpy or CPU torch tensor) -> float64, exactly."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                bits = x.view(torch.int16).numpy().astype(np.uint16).astype(np.uint32) << 16
                return bits.view(np.float32).astype(np.float64)
            return x.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x).astype(np.float64)


# ---------------------------------------------------------------------------------------
# Thin wrappers, one per oracle step.
# ---------------------------------------------------------------------------------------

def num_cores() -> int:
    return int(_load().orc_num_cores())


def e4m3_decode(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.zeros(b.shape, dtype=np.float64)
    _load().orc_e4m3_decode_n(b.reshape(-1), b.size, out.reshape(-1))
    return out


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_n(x.reshape(-1), x.size, out.reshape(-1))
    return out


def init_indices(seed: int, tensor_id: int, stage: int, N: int, C: int) -> np.ndarray:
    idx = np.zeros(C, dtype=np.int64)
    rc = _load().orc_init_indices(seed & (2**64 - 1), tensor_id, stage, N, C, idx)
    if rc != 0:
        raise ValueError("orc_init_indices failed (%d)" % rc)
    return idx


def _rows(R):
    R = np.ascontiguousarray(R, dtype=np.float64)
    assert R.ndim == 2
    return R, R.shape[0], R.shape[1]


def assign(R, cent):
    """(pi int32 [N], squared distance to the chosen centroid [N])."""
    R, N, d = _rows(R)
    cent = np.ascontiguousarray(cent, dtype=np.float32)
    pi = np.zeros(N, dtype=np.int32)
    dist = np.zeros(N, dtype=np.float64)
    _load().orc_assign(R, N, d, cent, cent.shape[0], pi, dist)
    return pi, dist


def update(R, pi, cent):
    """(new fp32 centroids, cluster counts).  Empty clusters keep ``cent``'s rows."""
    R, N, d = _rows(R)
    out = np.array(cent, dtype=np.float32, copy=True, order="C")
    counts = np.zeros(out.shape[0], dtype=np.int64)
    _load().orc_update(R, N, d, np.ascontiguousarray(pi, dtype=np.int32), out.shape[0], out,
                       counts)
    return out, counts


def objective(R, pi, cent) -> float:
    R, N, d = _rows(R)
    return float(_load().orc_objective(R, N, d, np.ascontiguousarray(pi, dtype=np.int32),
                                       np.ascontiguousarray(cent, dtype=np.float32)))


def subtract(R, pi, cent) -> np.ndarray:
    R, N, d = _rows(R)
    R = R.copy()
    _load().orc_subtract(R, N, d, np.ascontiguousarray(pi, dtype=np.int32),
                         np.ascontiguousarray(cent, dtype=np.float32))
    return R


def lloyd(R, cent, iters: int):
    """`iters` rounds of (assign, update) from ``cent``; returns (centroids, last pi)."""
    R, N, d = _rows(R)
    out = np.array(cent, dtype=np.float32, copy=True, order="C")
    pi = np.zeros(N, dtype=np.int32)
    _load().orc_lloyd(R, N, d, out.shape[0], iters, out, pi)
    return out, pi


def store_centroids(x, centroid_format: int) -> np.ndarray:
    """The stored value of each x in a centroid storage format: 0 fp32, 1 IEEE binary16,
    2 bfloat16 (round to nearest even once, from fp64)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.float32)
    _load().orc_store_n(x.reshape(-1), x.size, centroid_format, out.reshape(-1))
    return out


def encode(R, bits: int, group: int, scheme: int = 0):
    """Q(R): (codes uint8 [N][d*bits/8], E4M3 scale bytes uint8 [N][d/group]).
    scheme 0: symmetric restricted grid; 1: mid-rise (levels at half-integers)."""
    R, N, d = _rows(R)
    codes = np.zeros((N, d * bits // 8), dtype=np.uint8)
    scales = np.zeros((N, d // group), dtype=np.uint8)
    _load().orc_encode(R, N, d, bits, group, scheme, codes, scales)
    return codes, scales


def decode_codes(codes, scales, bits: int, group: int, scheme: int = 0) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N = codes.shape[0]
    d = codes.shape[1] * 8 // bits
    out = np.zeros((N, d), dtype=np.float64)
    _load().orc_decode_codes(codes, scales, N, d, bits, group, scheme, out)
    return out


def dequantize(codes, scales, pi, cent, bits: int, group: int, scheme: int = 0) -> np.ndarray:
    """One tensor: codes [N][d*b/8], scales [N][d/B], pi [T][N] uint8, cent [T][C][d]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N = codes.shape[0]
    d = codes.shape[1] * 8 // bits
    pi = np.ascontiguousarray(pi, dtype=np.uint8).reshape(-1, N)
    T = pi.shape[0]
    cent = np.ascontiguousarray(cent, dtype=np.float32)
    C = cent.shape[1] if T > 0 else 1
    if T == 0:
        cent = np.zeros((1, 1, d), dtype=np.float32)
        pi = np.zeros((1, N), dtype=np.uint8)
    out = np.zeros((N, d), dtype=np.float64)
    _load().orc_dequantize(codes, scales, pi, cent, N, d, C, T, bits, group, scheme, out)
    return out


def quantize(X, C: int, T: int, bits: int, group: int, iters: int, seed: int,
             tensor_id_base: int = 0, warm=None, nthreads: int = 0, scheme: int = 0,
             centroid_format: int = 0) -> dict:
    """The whole quantize path over a batch X [H][N][d] (float64, already decoded).

    Returns codes [H][N][d*b/8], scales [H][N][d/B], pi [H][T][N] (uint8),
    centroids [H][T][C][d] (fp32) and J [H][T] (each stage's Lloyd objective).
    """
    X = np.ascontiguousarray(X, dtype=np.float64)
    H, N, d = X.shape
    Ce = max(C, 1)
    codes = np.zeros((H, N, d * bits // 8), dtype=np.uint8)
    scales = np.zeros((H, N, d // group), dtype=np.uint8)
    pi = np.zeros((H, max(T, 1), N), dtype=np.uint8)
    cent = np.zeros((H, max(T, 1), Ce, d), dtype=np.float32)
    J = np.zeros((H, max(T, 1)), dtype=np.float64)
    warm_arr = None
    warm_ptr = None
    if warm is not None:
        warm_arr = np.ascontiguousarray(warm, dtype=np.float32)
        assert warm_arr.shape == (H, T, C, d)
        warm_ptr = warm_arr.ctypes.data
    rc = _load().orc_quantize(H, N, d, Ce, T, bits, group, iters, seed & (2**64 - 1),
                              tensor_id_base, X, warm_ptr, codes, scales, pi, cent, J,
                              nthreads, scheme, centroid_format)
    if rc != 0:
        raise ValueError("orc_quantize rejected the arguments (%d)" % rc)
    return {"codes": codes, "scales": scales, "pi": pi[:, :T], "centroids": cent[:, :T],
            "J": J[:, :T]}


def residual(X, pi, cent, upto: int) -> np.ndarray:
    """R^(upto) of one tensor: X [N][d] minus stages 1..upto's assigned centroids (fp64)."""
    R, _, _ = _rows(X)
    R = R.copy()
    for t in range(upto):
        R = subtract(R, np.asarray(pi[t], dtype=np.int32), cent[t])
    return R
