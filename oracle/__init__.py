"""ctypes wrapper of the plain-C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  The oracle is the slow CPU definition of INT8
mixed-precision linear layers that the CUDA path is checked against.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import
it; the product package never does, and the two share no code.

Arrays are numpy: bf16 tensors travel as their raw uint16 bit patterns, codes
as int8, scales as float32, accumulators as int32.  This module only marshals
arguments; every step of the arithmetic is in oracle.c.
"""
import contextlib
import ctypes
import os

import numpy as np

from . import build as _build

RNE, SR = 0, 1
AxBT, AxB, ATxB = 0, 1, 2
STREAM_FWD_X, STREAM_FWD_W, STREAM_GI_DY, STREAM_GI_W, STREAM_GW_DY, STREAM_GW_X = range(6)

_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_u32 = ctypes.c_uint32
_int = ctypes.c_int


def _load(path):
    L = ctypes.CDLL(path)
    L.orc_philox4x32_10.argtypes = [_p, _p, _p]
    L.orc_philox4x32_10.restype = None
    L.orc_quantize.argtypes = [_p, _i64, _i64, _i64, _int, _int, _u64, _u64, _u32, _p, _p]
    L.orc_mm_s32.argtypes = [_p, _p, _i64, _i64, _i64, _int, _p, _int]
    L.orc_rescale_bf16.argtypes = [_p, _p, _p, _i64, _i64, _p]
    L.orc_scaled_mm.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _int]
    L.orc_linear_fwd.argtypes = [_p, _p, _i64, _i64, _i64, _int, _u64, _u64, _p, _int]
    L.orc_linear_bwd.argtypes = [_p, _p, _p, _i64, _i64, _i64, _int, _u64, _u64, _p, _p, _int]
    L.orc_matmul_bf16.argtypes = [_p, _p, _i64, _i64, _i64, _int, _p, _int]
    L.orc_linear_fwd_cfg.argtypes = [_p, _p, _i64, _i64, _i64, _int, _int, _u64, _u64, _p, _int]
    L.orc_linear_bwd_cfg.argtypes = [_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _u64, _u64,
                                     _p, _p, _int]
    L.orc_rescale_f32.argtypes = [_p, _p, _p, _i64, _i64, _p]
    L.orc_scaled_mm_f32.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _int]
    L.orc_grad_weight_sharded.argtypes = [_p, _p, _i64, _i64, _i64, _int, _int, _u64, _p, _p, _int]
    L.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
    for name in ("orc_quantize", "orc_mm_s32", "orc_rescale_bf16", "orc_scaled_mm",
                 "orc_linear_fwd", "orc_linear_bwd", "orc_matmul_bf16", "orc_linear_fwd_cfg",
                 "orc_linear_bwd_cfg", "orc_rescale_f32", "orc_scaled_mm_f32",
                 "orc_grad_weight_sharded"):
        getattr(L, name).restype = _int
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Temporarily route every call through another build of the oracle
    (used by the tests that plant mistakes in a copy of oracle.c)."""
    global _lib
    saved = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = saved


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def default_threads():
    return max(1, os.cpu_count() or 1)


def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def bf16_rne(f):
    """fp32 value -> bf16 bit pattern, round half to even."""
    return int(lib().orc_f32_to_bf16_rne(float(np.float32(f))))


def quantize(x, axis, mode=RNE, seed=0, offset=0, stream_id=0, cols=None):
    """x: uint16 [rows, ld] bf16 bits.  Returns (codes int8, scale float32);
    axis 0 codes are [rows, cols], axis 1 codes are [cols, rows]."""
    x = _c(x, np.uint16)
    rows, ld = x.shape
    cols = ld if cols is None else cols
    groups, glen = (rows, cols) if axis == 0 else (cols, rows)
    q = np.zeros((groups, glen), dtype=np.int8)
    s = np.zeros(groups, dtype=np.float32)
    _check(lib().orc_quantize(_ptr(x), rows, cols, ld, axis, mode, seed, offset, stream_id,
                              _ptr(q), _ptr(s)), "quantize")
    return q, s


def mm_s32(A, B, M, N, K, layout=AxBT, nthreads=None):
    A = _c(A, np.int8)
    B = _c(B, np.int8)
    acc = np.zeros((M, N), dtype=np.int32)
    _check(lib().orc_mm_s32(_ptr(A), _ptr(B), M, N, K, layout, _ptr(acc),
                            nthreads or default_threads()), "mm_s32")
    return acc


def rescale_bf16(acc, sA, sB):
    acc = _c(acc, np.int32)
    M, N = acc.shape
    out = np.zeros((M, N), dtype=np.uint16)
    _check(lib().orc_rescale_bf16(_ptr(acc), _ptr(_c(sA, np.float32)), _ptr(_c(sB, np.float32)),
                                  M, N, _ptr(out)), "rescale")
    return out


def scaled_mm(A, sA, B, sB, M, N, K, layout=AxBT, nthreads=None):
    out = np.zeros((M, N), dtype=np.uint16)
    _check(lib().orc_scaled_mm(_ptr(_c(A, np.int8)), _ptr(_c(sA, np.float32)),
                               _ptr(_c(B, np.int8)), _ptr(_c(sB, np.float32)),
                               M, N, K, layout, _ptr(out), nthreads or default_threads()),
           "scaled_mm")
    return out


def linear_fwd(X, W, mode=RNE, seed=0, offset=0, nthreads=None):
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    T, K = X.shape
    N = W.shape[0]
    Y = np.zeros((T, N), dtype=np.uint16)
    _check(lib().orc_linear_fwd(_ptr(X), _ptr(W), T, N, K, mode, seed, offset, _ptr(Y),
                                nthreads or default_threads()), "linear_fwd")
    return Y


def linear_bwd(dY, X, W, mode=RNE, seed=0, offset=0, nthreads=None, want_dx=True, want_dw=True):
    dY = _c(dY, np.uint16)
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    T, K = X.shape
    N = W.shape[0]
    dX = np.zeros((T, K), dtype=np.uint16) if want_dx else None
    dW = np.zeros((N, K), dtype=np.uint16) if want_dw else None
    _check(lib().orc_linear_bwd(_ptr(dY), _ptr(X), _ptr(W), T, N, K, mode, seed, offset,
                                _ptr(dX), _ptr(dW), nthreads or default_threads()), "linear_bwd")
    return dX, dW


def rescale_f32(acc, sA, sB):
    acc = _c(acc, np.int32)
    M, N = acc.shape
    out = np.zeros((M, N), dtype=np.float32)
    _check(lib().orc_rescale_f32(_ptr(acc), _ptr(_c(sA, np.float32)), _ptr(_c(sB, np.float32)),
                                 M, N, _ptr(out)), "rescale_f32")
    return out


def scaled_mm_f32(A, sA, B, sB, M, N, K, layout=AxBT, nthreads=None):
    """The scaled matmul's fp32 value before the bf16 rounding."""
    out = np.zeros((M, N), dtype=np.float32)
    _check(lib().orc_scaled_mm_f32(_ptr(_c(A, np.int8)), _ptr(_c(sA, np.float32)),
                                   _ptr(_c(B, np.int8)), _ptr(_c(sB, np.float32)),
                                   M, N, K, layout, _ptr(out), nthreads or default_threads()),
           "scaled_mm_f32")
    return out


def grad_weight_sharded(dY, X, nshards, offsets, mode=RNE, seed=0, nthreads=None):
    """dW [N,K] of token-sharded data parallelism: per-shard fp32 partials
    summed in shard order, rounded once to bf16 (bits)."""
    dY = _c(dY, np.uint16)
    X = _c(X, np.uint16)
    T, N = dY.shape
    K = X.shape[1]
    offs = _c(np.asarray(offsets, dtype=np.uint64), np.uint64)
    assert len(offs) == nshards
    out = np.zeros((N, K), dtype=np.uint16)
    _check(lib().orc_grad_weight_sharded(_ptr(dY), _ptr(X), T, N, K, nshards, mode, seed,
                                         _ptr(offs), _ptr(out), nthreads or default_threads()),
           "grad_weight_sharded")
    return out


def matmul_bf16(A, B, M, N, K, layout=AxBT, nthreads=None):
    """BF16 pass: bf16_RNE(fp32_RN(sum in fp64)), operands as bf16 bits."""
    out = np.zeros((M, N), dtype=np.uint16)
    _check(lib().orc_matmul_bf16(_ptr(_c(A, np.uint16)), _ptr(_c(B, np.uint16)), M, N, K, layout,
                                 _ptr(out), nthreads or default_threads()), "matmul_bf16")
    return out


def linear_fwd_cfg(X, W, int8_fwd=1, mode=RNE, seed=0, offset=0, nthreads=None):
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    T, K = X.shape
    N = W.shape[0]
    Y = np.zeros((T, N), dtype=np.uint16)
    _check(lib().orc_linear_fwd_cfg(_ptr(X), _ptr(W), T, N, K, int8_fwd, mode, seed, offset,
                                    _ptr(Y), nthreads or default_threads()), "linear_fwd_cfg")
    return Y


def linear_bwd_cfg(dY, X, W, int8_grad_in=1, int8_grad_w=1, mode=RNE, seed=0, offset=0,
                   nthreads=None):
    dY = _c(dY, np.uint16)
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    T, K = X.shape
    N = W.shape[0]
    dX = np.zeros((T, K), dtype=np.uint16)
    dW = np.zeros((N, K), dtype=np.uint16)
    _check(lib().orc_linear_bwd_cfg(_ptr(dY), _ptr(X), _ptr(W), T, N, K, int8_grad_in, int8_grad_w,
                                    mode, seed, offset, _ptr(dX), _ptr(dW),
                                    nthreads or default_threads()), "linear_bwd_cfg")
    return dX, dW
