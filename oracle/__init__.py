"""FP64 oracle for the dense projection GEMM family -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The CUDA library never does, and this package
imports nothing from it: the two share only the seeded input tensors.

The arithmetic lives in ``oracle.c`` (plain C, FP64, natural summation order);
this module compiles it with gcc when needed and marshals numpy arrays to it.

Operations (row-major operands; see oracle.c for the definitions and the pages
they follow):

  forward          Y  = X  W^T     X[T,K], W[N,K]   -> Y[T,N]
  input gradient   dX = dY W       dY[T,N], W[N,K]  -> dX[T,K]
  weight gradient  dW = dY^T X     dY[T,N], X[T,K]  -> dW[N,K]

Each comes in three input flavours: bf16 bit patterns (uint16), FP32 (the
router's plain FP64 reference), and BF16x3 (the router's three-term restatement
on pre-split hi/lo halves).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_GCC_FLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc; a second or two)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_GCC_FLAGS, _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I = ctypes.c_int64
    for name in ("oracle_fwd_bf16", "oracle_dgrad_bf16", "oracle_wgrad_bf16",
                 "oracle_fwd_f32", "oracle_dgrad_f32", "oracle_wgrad_f32"):
        getattr(lib, name).argtypes = [P, P, P, I, I, I]
        getattr(lib, name).restype = None
    for name in ("oracle_fwd_x3", "oracle_dgrad_x3", "oracle_wgrad_x3"):
        getattr(lib, name).argtypes = [P, P, P, P, P, I, I, I]
        getattr(lib, name).restype = None
    for name in ("oracle_fwd_bf16_at", "oracle_dgrad_bf16_at", "oracle_wgrad_bf16_at",
                 "oracle_fwd_f32_at", "oracle_dgrad_f32_at", "oracle_wgrad_f32_at"):
        getattr(lib, name).argtypes = [P, P, I, I, I, P, P, I, P]
        getattr(lib, name).restype = None
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_split_bf16x3.argtypes = [P, P, P, I]
    lib.oracle_split_bf16x3.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def num_threads() -> int:
    """Threads the oracle's parallel loops use (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- marshalling

def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _bits(a) -> np.ndarray:
    """Accept a uint16 bit array, or a torch bf16 CPU tensor, and return uint16 bits."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return a.contiguous().view(torch.int16).numpy().view(np.uint16)
    return _c(a, np.uint16)


def _f32(a) -> np.ndarray:
    if hasattr(a, "numpy") and not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return _c(a, np.float32)


def _index(a) -> np.ndarray:
    return _c(np.asarray(a).reshape(-1), np.int64)


# ------------------------------------------------------------- scalar helpers

def f32_to_bf16(x) -> np.ndarray:
    """Round FP32 values to bf16 bit patterns (nearest, ties to even)."""
    lib = _load()
    x = _f32(x)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, np.uint16)
    for i, v in enumerate(flat):
        out[i] = lib.oracle_f32_to_bf16_rne(ctypes.c_float(v))
    return out.reshape(x.shape)


def bf16_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    b = _bits(bits)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def split_bf16x3(x):
    """BF16x3 split of FP32 values: (hi, lo) bf16 bit arrays, hi = RNE(x), lo = RNE(x - hi)."""
    x = _f32(x)
    hi = np.empty(x.shape, np.uint16)
    lo = np.empty(x.shape, np.uint16)
    _load().oracle_split_bf16x3(_ptr(x), _ptr(hi), _ptr(lo), x.size)
    return hi, lo


# ----------------------------------------------------------- full operations

def _full(name, a, b, shape_out, T, N, K, conv):
    a = conv(a)
    b = conv(b)
    out = np.empty(shape_out, np.float64)
    getattr(_load(), name)(_ptr(a), _ptr(b), _ptr(out), T, N, K)
    return out


def fwd_bf16(X, W) -> np.ndarray:
    """Y[T,N] = X[T,K] W[N,K]^T on bf16 operands, FP64 result."""
    X, W = _bits(X), _bits(W)
    T, K = X.shape
    N = W.shape[0]
    assert W.shape[1] == K
    return _full("oracle_fwd_bf16", X, W, (T, N), T, N, K, _bits)


def dgrad_bf16(dY, W) -> np.ndarray:
    """dX[T,K] = dY[T,N] W[N,K] on bf16 operands, FP64 result."""
    dY, W = _bits(dY), _bits(W)
    T, N = dY.shape
    K = W.shape[1]
    assert W.shape[0] == N
    return _full("oracle_dgrad_bf16", dY, W, (T, K), T, N, K, _bits)


def wgrad_bf16(dY, X) -> np.ndarray:
    """dW[N,K] = dY[T,N]^T X[T,K] on bf16 operands, FP64 result."""
    dY, X = _bits(dY), _bits(X)
    T, N = dY.shape
    K = X.shape[1]
    assert X.shape[0] == T
    return _full("oracle_wgrad_bf16", dY, X, (N, K), T, N, K, _bits)


def fwd_f32(X, W) -> np.ndarray:
    """Plain FP64 forward of FP32 operands (the router's budget reference)."""
    X, W = _f32(X), _f32(W)
    T, K = X.shape
    N = W.shape[0]
    return _full("oracle_fwd_f32", X, W, (T, N), T, N, K, _f32)


def dgrad_f32(dY, W) -> np.ndarray:
    dY, W = _f32(dY), _f32(W)
    T, N = dY.shape
    K = W.shape[1]
    return _full("oracle_dgrad_f32", dY, W, (T, K), T, N, K, _f32)


def wgrad_f32(dY, X) -> np.ndarray:
    dY, X = _f32(dY), _f32(X)
    T, N = dY.shape
    K = X.shape[1]
    return _full("oracle_wgrad_f32", dY, X, (N, K), T, N, K, _f32)


def _x3(name, a, b, shape_out, T, N, K):
    ah, al = split_bf16x3(a)
    bh, bl = split_bf16x3(b)
    out = np.empty(shape_out, np.float64)
    getattr(_load(), name)(_ptr(ah), _ptr(al), _ptr(bh), _ptr(bl), _ptr(out), T, N, K)
    return out


def fwd_bf16x3(X, W) -> np.ndarray:
    """Router forward through BF16x3: sum_k hi*hi + hi*lo + lo*hi, in FP64."""
    X, W = _f32(X), _f32(W)
    T, K = X.shape
    N = W.shape[0]
    return _x3("oracle_fwd_x3", X, W, (T, N), T, N, K)


def dgrad_bf16x3(dY, W) -> np.ndarray:
    dY, W = _f32(dY), _f32(W)
    T, N = dY.shape
    K = W.shape[1]
    return _x3("oracle_dgrad_x3", dY, W, (T, K), T, N, K)


def wgrad_bf16x3(dY, X) -> np.ndarray:
    dY, X = _f32(dY), _f32(X)
    T, N = dY.shape
    K = X.shape[1]
    return _x3("oracle_wgrad_x3", dY, X, (N, K), T, N, K)


# -------------------------------------------------------- sampled operations

def _at(name, a, b, T, N, K, rows, cols, conv):
    a, b = conv(a), conv(b)
    r, c = _index(rows), _index(cols)
    assert r.shape == c.shape
    out = np.empty(r.shape, np.float64)
    getattr(_load(), name)(_ptr(a), _ptr(b), T, N, K, _ptr(r), _ptr(c), r.size, _ptr(out))
    return out


def fwd_bf16_at(X, W, rows, cols) -> np.ndarray:
    """Y[rows[i], cols[i]] of the bf16 forward, one ordered FP64 sum each."""
    X, W = _bits(X), _bits(W)
    return _at("oracle_fwd_bf16_at", X, W, X.shape[0], W.shape[0], X.shape[1], rows, cols, _bits)


def dgrad_bf16_at(dY, W, rows, cols) -> np.ndarray:
    dY, W = _bits(dY), _bits(W)
    return _at("oracle_dgrad_bf16_at", dY, W, dY.shape[0], dY.shape[1], W.shape[1], rows, cols, _bits)


def wgrad_bf16_at(dY, X, rows, cols) -> np.ndarray:
    dY, X = _bits(dY), _bits(X)
    return _at("oracle_wgrad_bf16_at", dY, X, dY.shape[0], dY.shape[1], X.shape[1], rows, cols, _bits)


def fwd_f32_at(X, W, rows, cols) -> np.ndarray:
    X, W = _f32(X), _f32(W)
    return _at("oracle_fwd_f32_at", X, W, X.shape[0], W.shape[0], X.shape[1], rows, cols, _f32)


def dgrad_f32_at(dY, W, rows, cols) -> np.ndarray:
    dY, W = _f32(dY), _f32(W)
    return _at("oracle_dgrad_f32_at", dY, W, dY.shape[0], dY.shape[1], W.shape[1], rows, cols, _f32)


def wgrad_f32_at(dY, X, rows, cols) -> np.ndarray:
    dY, X = _f32(dY), _f32(X)
    return _at("oracle_wgrad_f32_at", dY, X, dY.shape[0], dY.shape[1], X.shape[1], rows, cols, _f32)
