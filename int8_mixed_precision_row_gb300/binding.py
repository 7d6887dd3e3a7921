"""Thin ctypes binding of libint8mp.so (include/int8mp.h).

Names follow the C entry points.  This module only marshals arguments:
torch supplies device memory and the current CUDA stream, and every step of
the computation runs in the library's CUDA kernels.  There is no fallback:
if the library is missing or the device is not sm_103, calls raise.
"""
import ctypes
import os

import torch

from . import build as _build

# ---- constants mirrored from include/int8mp.h -----------------------------
INT8MP_OK = 0
INT8MP_ERR_INVALID_ARG = 1
INT8MP_ERR_ALIGNMENT = 2
INT8MP_ERR_UNSUPPORTED_DEVICE = 3
INT8MP_ERR_CUDA = 4
INT8MP_ERR_TIMEOUT = 5
INT8MP_ERR_WORKSPACE = 6
INT8MP_ERR_BOUNDS = 7

INT8MP_RNE, INT8MP_SR = 0, 1
INT8MP_AxBT, INT8MP_AxB, INT8MP_ATxB = 0, 1, 2
INT8MP_GROUP_ROWS, INT8MP_GROUP_COLS_T, INT8MP_GROUP_COLS = 0, 1, 2
INT8MP_CODES_S8, INT8MP_CODES_F16 = 0, 1
(INT8MP_STREAM_FWD_X, INT8MP_STREAM_FWD_W, INT8MP_STREAM_GI_DY, INT8MP_STREAM_GI_W,
 INT8MP_STREAM_GW_DY, INT8MP_STREAM_GW_X) = range(6)
INT8MP_MAX_K = 133143
INT8MP_MAX_ROWS_JOBS = 2

# every symbol the public headers declare
EXPORTED = (
    "int8mp_quantize_rowwise", "int8mp_scaled_mm", "int8mp_mm_s32",
    "int8mp_linear_workspace_size", "int8mp_linear_fwd", "int8mp_linear_bwd",
    "int8mp_poll_device_status", "int8mp_status_string", "int8mp_version",
    "int8mp_debug_mm_s32_drop_first_load", "int8mp_linear_fwd_noalloc",
    "int8mp_debug_check_division", "int8mp_quantize_rows_colmax", "int8mp_quantize_cols_absmax",
    "int8mp_linear_fwd_save", "int8mp_linear_bwd_saved", "int8mp_mm_workspace_size",
    "int8mp_scaled_mm_ws", "int8mp_mm_s32_ws", "int8mp_quantize_rows_batch",
    "int8mp_scaled_mm_f32", "int8mp_round_bf16", "int8mp_debug_scaled_mm_quant_b",
    "int8mp_quantize_cols_batch",
)
INT8MP_NOALLOC_SCRATCH_BYTES = 32 << 20


class Int8mpError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {int8mp_status_string(status)} (status {status})")


class int8mp_rows_job(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("ld", ctypes.c_int64),
                ("offset", ctypes.c_uint64), ("stream_id", ctypes.c_uint32),
                ("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("colmax", ctypes.c_void_p)]


class int8mp_linear_cfg(ctypes.Structure):
    _fields_ = [("int8_fwd", ctypes.c_int), ("int8_grad_in", ctypes.c_int),
                ("int8_grad_w", ctypes.c_int), ("mode", ctypes.c_int),
                ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


def linear_cfg(mode=INT8MP_RNE, seed=0, offset=0, int8_fwd=1, int8_grad_in=1, int8_grad_w=1):
    """int8_* = 1: that pass in INT8; 0: in BF16 (plain bf16 product)."""
    return int8mp_linear_cfg(int(int8_fwd), int(int8_grad_in), int(int8_grad_w), int(mode),
                             int(seed), int(offset))


_lib = None
_P, _I64, _U64, _U32, _INT, _SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                   ctypes.c_uint32, ctypes.c_int, ctypes.c_size_t)


def library_path():
    return _build.LIB


class use_library:
    """Context manager: route the binding's calls to another build of the
    library (e.g. the bounds-checked one from build.build(check=True)) while
    inside, then back."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = None
        return load(self.path)

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def load(path=None):
    """Load libint8mp.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libint8mp.so is not built ({path}); run int8_mixed_precision_row_gb300."
                           "build.build() or __graft_entry__.build()")
    L = ctypes.CDLL(path)
    L.int8mp_quantize_rowwise.argtypes = [_P, _I64, _I64, _I64, _INT, _INT, _U64, _U64, _U32, _P,
                                          _INT, _P, _P]
    L.int8mp_scaled_mm.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _INT, _P, _I64, _P]
    L.int8mp_mm_s32.argtypes = [_P, _P, _I64, _I64, _I64, _INT, _INT, _P, _I64, _P]
    L.int8mp_linear_workspace_size.argtypes = [_I64, _I64, _I64, ctypes.POINTER(int8mp_linear_cfg)]
    L.int8mp_linear_workspace_size.restype = _SZ
    L.int8mp_linear_fwd.argtypes = [_P, _P, _P, _I64, _I64, _I64, ctypes.POINTER(int8mp_linear_cfg),
                                    _P, _SZ, _P]
    L.int8mp_linear_bwd.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64,
                                    ctypes.POINTER(int8mp_linear_cfg), _P, _SZ, _P]
    L.int8mp_poll_device_status.argtypes = [_P]
    L.int8mp_status_string.argtypes = [_INT]
    L.int8mp_status_string.restype = ctypes.c_char_p
    L.int8mp_version.argtypes = []
    L.int8mp_debug_mm_s32_drop_first_load.argtypes = [_P, _P, _I64, _I64, _I64, _P, _I64, _INT, _P]
    L.int8mp_linear_fwd_noalloc.argtypes = [_P, _P, _P, _I64, _I64, _I64,
                                            ctypes.POINTER(int8mp_linear_cfg), _P]
    L.int8mp_debug_check_division.argtypes = [_P, _P]
    L.int8mp_quantize_rows_colmax.argtypes = [_P, _I64, _I64, _I64, _INT, _U64, _U64, _U32, _P,
                                              _INT, _P, _P, _P]
    L.int8mp_quantize_cols_absmax.argtypes = [_P, _I64, _I64, _I64, _P, _INT, _U64, _U64, _U32, _P,
                                              _INT, _P, _P]
    L.int8mp_linear_fwd_save.argtypes = [_P, _P, _P, _I64, _I64, _I64,
                                         ctypes.POINTER(int8mp_linear_cfg), _P, _P, _SZ, _P]
    L.int8mp_linear_bwd_saved.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64,
                                          ctypes.POINTER(int8mp_linear_cfg), _P, _P, _SZ, _P]
    L.int8mp_quantize_rows_batch.argtypes = [ctypes.POINTER(int8mp_rows_job), _INT, _I64, _INT, _U64,
                                             _INT, _P]
    L.int8mp_quantize_cols_batch.argtypes = [ctypes.POINTER(int8mp_rows_job), _INT, _I64, _INT, _U64,
                                             _INT, _P]
    L.int8mp_mm_workspace_size.argtypes = []
    L.int8mp_mm_workspace_size.restype = _SZ
    L.int8mp_scaled_mm_ws.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _INT, _P, _I64, _P,
                                      _SZ, _P]
    L.int8mp_mm_s32_ws.argtypes = [_P, _P, _I64, _I64, _I64, _INT, _INT, _P, _I64, _P, _SZ, _P]
    L.int8mp_scaled_mm_f32.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _INT, _INT, _P, _I64, _P,
                                       _SZ, _P]
    L.int8mp_round_bf16.argtypes = [_P, _P, _I64, _P]
    L.int8mp_debug_scaled_mm_quant_b.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P]
    for name in ("int8mp_quantize_cols_batch", "int8mp_scaled_mm_ws", "int8mp_mm_s32_ws", "int8mp_scaled_mm_f32",
                 "int8mp_round_bf16", "int8mp_debug_scaled_mm_quant_b",
                 "int8mp_quantize_rowwise", "int8mp_scaled_mm", "int8mp_mm_s32",
                 "int8mp_linear_fwd", "int8mp_linear_bwd", "int8mp_poll_device_status",
                 "int8mp_version", "int8mp_debug_mm_s32_drop_first_load",
                 "int8mp_linear_fwd_noalloc", "int8mp_debug_check_division",
                 "int8mp_quantize_rows_colmax", "int8mp_quantize_cols_absmax",
                 "int8mp_linear_fwd_save", "int8mp_linear_bwd_saved"):
        getattr(L, name).restype = _INT
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != INT8MP_OK:
        raise Int8mpError(status, what)


def _code_dtype(codes):
    return torch.int8 if codes == INT8MP_CODES_S8 else torch.float16


def int8mp_status_string(status):
    return load().int8mp_status_string(int(status)).decode()


def int8mp_version():
    return load().int8mp_version()


def int8mp_quantize_rowwise(x, axis=0, mode=INT8MP_RNE, seed=0, offset=0, stream_id=0,
                            codes=INT8MP_CODES_S8, cols=None, q=None, scale=None, stream=None):
    """x: bf16 CUDA tensor [rows, ld] (row stride ld).  Returns (codes, scale);
    axis 0 (row groups) and 2 (column groups) codes are [rows, cols], axis 1
    (column groups) codes are [cols, rows]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda
    rows = x.shape[0]
    ld = x.stride(0) if rows > 0 else x.shape[1]
    cols = x.shape[1] if cols is None else cols
    shape = (cols, rows) if axis == INT8MP_GROUP_COLS_T else (rows, cols)
    if q is None:
        q = torch.empty(shape, dtype=_code_dtype(codes), device=x.device)
    if scale is None:
        scale = torch.empty((rows if axis == INT8MP_GROUP_ROWS else cols,), dtype=torch.float32,
                            device=x.device)
    _check(load().int8mp_quantize_rowwise(_ptr(x), rows, cols, ld, int(axis), int(mode), int(seed),
                                          int(offset), int(stream_id), _ptr(q), int(codes),
                                          _ptr(scale), _stream(stream)), "int8mp_quantize_rowwise")
    return q, scale


def _check_out(out, M, N, dtype):
    """The matmul writes rows of N elements at stride out.stride(0)."""
    if out.shape != (M, N) or out.dtype != dtype or (N > 1 and out.stride(1) != 1):
        raise ValueError(f"out must be {dtype} [{M}, {N}] with contiguous rows, got "
                         f"{out.dtype} {tuple(out.shape)} strides {out.stride()}")


def _mm_sizes(A, B, layout):
    if layout == INT8MP_AxBT:
        return A.shape[0], B.shape[0], A.shape[1]
    if layout == INT8MP_AxB:
        return A.shape[0], B.shape[1], A.shape[1]
    return A.shape[1], B.shape[1], A.shape[0]


def int8mp_quantize_rows_colmax(x, colmax, mode=INT8MP_RNE, seed=0, offset=0, stream_id=0,
                                codes=INT8MP_CODES_S8, q=None, scale=None, stream=None):
    """Row groups of x [rows, cols] (codes [rows, cols], scale [rows]) and,
    in the same pass, colmax [cols] (fp32, caller-initialized) max-merged
    with each column's absmax."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda
    rows, cols = x.shape
    ld = x.stride(0) if rows > 0 else cols
    if q is None:
        q = torch.empty((rows, cols), dtype=_code_dtype(codes), device=x.device)
    if scale is None:
        scale = torch.empty((rows,), dtype=torch.float32, device=x.device)
    _check(load().int8mp_quantize_rows_colmax(_ptr(x), rows, cols, ld, int(mode), int(seed),
                                              int(offset), int(stream_id), _ptr(q), int(codes),
                                              _ptr(scale), _ptr(colmax), _stream(stream)),
           "int8mp_quantize_rows_colmax")
    return q, scale


def int8mp_quantize_rows_batch(xs, mode=INT8MP_RNE, seed=0, offsets=None, stream_ids=None,
                               codes=INT8MP_CODES_S8, qs=None, scales=None, colmaxes=None,
                               stream=None):
    """Row groups of up to two bf16 matrices with the same number of columns
    in one launch; as one int8mp_quantize_rows_colmax call per matrix when
    colmaxes is given, else as int8mp_quantize_rowwise(axis=0).  Returns the
    list of (codes, scale) pairs."""
    n = len(xs)
    cols = xs[0].shape[1]
    offsets = offsets or [0] * n
    stream_ids = stream_ids or [0] * n
    qs = qs or [None] * n
    scales = scales or [None] * n
    colmaxes = colmaxes or [None] * n
    arr = (int8mp_rows_job * max(n, 1))()
    out = []
    for i, x in enumerate(xs):
        assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda and x.shape[1] == cols
        rows = x.shape[0]
        q = qs[i] if qs[i] is not None else torch.empty((rows, cols), dtype=_code_dtype(codes),
                                                        device=x.device)
        sc = scales[i] if scales[i] is not None else torch.empty((rows,), dtype=torch.float32,
                                                                 device=x.device)
        arr[i] = int8mp_rows_job(x.data_ptr(), rows, x.stride(0) if rows > 0 else cols,
                                 int(offsets[i]), int(stream_ids[i]), q.data_ptr(), sc.data_ptr(),
                                 colmaxes[i].data_ptr() if colmaxes[i] is not None else None)
        out.append((q, sc))
    _check(load().int8mp_quantize_rows_batch(arr, n, cols, int(mode), int(seed), int(codes),
                                             _stream(stream)), "int8mp_quantize_rows_batch")
    return out


def int8mp_quantize_cols_batch(xs, mode=INT8MP_RNE, seed=0, offsets=None, stream_ids=None,
                               codes=INT8MP_CODES_S8, qs=None, scales=None, stream=None):
    """Column groups (codes in x's layout) of up to two bf16 matrices with the
    same number of columns, as one int8mp_quantize_rowwise(axis=
    INT8MP_GROUP_COLS) call per matrix.  Returns the list of (codes, scale)."""
    n = len(xs)
    cols = xs[0].shape[1]
    offsets = offsets or [0] * n
    stream_ids = stream_ids or [0] * n
    qs = qs or [None] * n
    scales = scales or [None] * n
    arr = (int8mp_rows_job * max(n, 1))()
    out = []
    for i, x in enumerate(xs):
        assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda and x.shape[1] == cols
        rows = x.shape[0]
        q = qs[i] if qs[i] is not None else torch.empty((rows, cols), dtype=_code_dtype(codes),
                                                        device=x.device)
        sc = scales[i] if scales[i] is not None else torch.empty((cols,), dtype=torch.float32,
                                                                 device=x.device)
        arr[i] = int8mp_rows_job(x.data_ptr(), rows, x.stride(0) if rows > 0 else cols,
                                 int(offsets[i]), int(stream_ids[i]), q.data_ptr(), sc.data_ptr(),
                                 None)
        out.append((q, sc))
    _check(load().int8mp_quantize_cols_batch(arr, n, cols, int(mode), int(seed), int(codes),
                                             _stream(stream)), "int8mp_quantize_cols_batch")
    return out


def int8mp_quantize_cols_absmax(x, colmax, mode=INT8MP_RNE, seed=0, offset=0, stream_id=0,
                                codes=INT8MP_CODES_S8, q=None, scale=None, stream=None):
    """Column groups of x [rows, cols] with each column's absmax given:
    codes [rows, cols], scale [cols]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda
    rows, cols = x.shape
    ld = x.stride(0) if rows > 0 else cols
    if q is None:
        q = torch.empty((rows, cols), dtype=_code_dtype(codes), device=x.device)
    if scale is None:
        scale = torch.empty((cols,), dtype=torch.float32, device=x.device)
    _check(load().int8mp_quantize_cols_absmax(_ptr(x), rows, cols, ld, _ptr(colmax), int(mode),
                                              int(seed), int(offset), int(stream_id), _ptr(q),
                                              int(codes), _ptr(scale), _stream(stream)),
           "int8mp_quantize_cols_absmax")
    return q, scale


def int8mp_mm_workspace_size():
    return int(load().int8mp_mm_workspace_size())


def _mm_ws(workspace, device):
    """workspace: None (plain schedule), True (allocate one) or a uint8 tensor."""
    if workspace is None or workspace is False:
        return None, 0
    if workspace is True:
        workspace = torch.empty(int8mp_mm_workspace_size(), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def _mm_codes(A, B, codes):
    """The code container: given, or that of the operands' dtype (int8 ->
    INT8MP_CODES_S8, float16 -> INT8MP_CODES_F16)."""
    if codes is None:
        codes = INT8MP_CODES_S8 if A.dtype == torch.int8 else INT8MP_CODES_F16
    want = _code_dtype(codes)
    if A.dtype != want or B.dtype != want:
        raise ValueError(f"codes {codes} need {want} operands, got {A.dtype} and {B.dtype}")
    return codes


def int8mp_scaled_mm(A, sA, B, sB, layout=INT8MP_AxBT, codes=None, out=None,
                     stream=None, workspace=None):
    """Codes A, B (int8, or f16 containers) stored per layout -- A@B.T: A
    [M,K], B [N,K]; A@B: A [M,K], B [K,N]; A.T@B: A [K,M], B [K,N] -- sA [M],
    sB [N] -> bf16 [M,N]."""
    codes = _mm_codes(A, B, codes)
    M, N, K = _mm_sizes(A, B, layout)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M, N, torch.bfloat16)
    ldo = out.stride(0) if M > 0 else N
    ws, nbytes = _mm_ws(workspace, A.device)
    if ws is None:
        _check(load().int8mp_scaled_mm(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K, int(layout),
                                       int(codes), _ptr(out), ldo, _stream(stream)),
               "int8mp_scaled_mm")
    else:
        _check(load().int8mp_scaled_mm_ws(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K,
                                          int(layout), int(codes), _ptr(out), ldo, _ptr(ws), nbytes,
                                          _stream(stream)), "int8mp_scaled_mm_ws")
    return out


def int8mp_mm_s32(A, B, layout=INT8MP_AxBT, codes=None, out=None, stream=None,
                  workspace=None):
    """The exact int32 product of codes A, B (int8 or f16 containers)."""
    codes = _mm_codes(A, B, codes)
    M, N, K = _mm_sizes(A, B, layout)
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=A.device)
    _check_out(out, M, N, torch.int32)
    ldo = out.stride(0) if M > 0 else N
    ws, nbytes = _mm_ws(workspace, A.device)
    if ws is None:
        _check(load().int8mp_mm_s32(_ptr(A), _ptr(B), M, N, K, int(layout), int(codes), _ptr(out),
                                    ldo, _stream(stream)), "int8mp_mm_s32")
    else:
        _check(load().int8mp_mm_s32_ws(_ptr(A), _ptr(B), M, N, K, int(layout), int(codes),
                                       _ptr(out), ldo, _ptr(ws), nbytes, _stream(stream)),
               "int8mp_mm_s32_ws")
    return out


def int8mp_scaled_mm_f32(A, sA, B, sB, layout=INT8MP_AxBT, codes=None, out=None, stream=None,
                         workspace=None):
    """The scaled matmul of codes A, B (layouts as int8mp_scaled_mm) with an
    fp32 result [M, N] that is not rounded to bf16 (a token shard's partial
    grad-weight)."""
    codes = _mm_codes(A, B, codes)
    M, N, K = _mm_sizes(A, B, layout)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check_out(out, M, N, torch.float32)
    ldo = out.stride(0) if M > 0 else N
    ws, nbytes = _mm_ws(workspace, A.device)
    _check(load().int8mp_scaled_mm_f32(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K, int(layout),
                                       int(codes), _ptr(out), ldo, _ptr(ws), nbytes,
                                       _stream(stream)), "int8mp_scaled_mm_f32")
    return out


def int8mp_round_bf16(x, y=None, stream=None):
    """bf16 round-to-nearest-even of a contiguous fp32 CUDA tensor."""
    assert x.dtype == torch.float32 and x.is_cuda and x.is_contiguous()
    if y is None:
        y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    assert y.dtype == torch.bfloat16 and y.is_contiguous() and y.numel() == x.numel()
    _check(load().int8mp_round_bf16(_ptr(x), _ptr(y), x.numel(), _stream(stream)),
           "int8mp_round_bf16")
    return y


def int8mp_linear_workspace_size(T, N, K, cfg=None):
    cfg = cfg or linear_cfg()
    return int(load().int8mp_linear_workspace_size(T, N, K, ctypes.byref(cfg)))


def _workspace(T, N, K, cfg, workspace, device):
    need = int8mp_linear_workspace_size(T, N, K, cfg)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def int8mp_linear_fwd(X, W, cfg=None, Y=None, workspace=None, stream=None):
    """Y [T,N] = X [T,K] . W [N,K]^T in INT8 mixed precision."""
    cfg = cfg or linear_cfg()
    T, K = X.shape
    N = W.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.bfloat16, device=X.device)
    ws, nbytes = _workspace(T, N, K, cfg, workspace, X.device)
    _check(load().int8mp_linear_fwd(_ptr(X), _ptr(W), _ptr(Y), T, N, K, ctypes.byref(cfg), _ptr(ws),
                                    nbytes, _stream(stream)), "int8mp_linear_fwd")
    return Y


def int8mp_linear_bwd(dY, X, W, cfg=None, dX=None, dW=None, want_dx=True, want_dw=True,
                      workspace=None, stream=None):
    """dX [T,K] = dY . W and dW [N,K] = dY^T . X in INT8 mixed precision."""
    cfg = cfg or linear_cfg()
    T, K = X.shape
    N = W.shape[0]
    if want_dx and dX is None:
        dX = torch.empty((T, K), dtype=torch.bfloat16, device=X.device)
    if want_dw and dW is None:
        dW = torch.empty((N, K), dtype=torch.bfloat16, device=X.device)
    ws, nbytes = _workspace(T, N, K, cfg, workspace, X.device)
    _check(load().int8mp_linear_bwd(_ptr(dY), _ptr(X), _ptr(W), _ptr(dX if want_dx else None),
                                    _ptr(dW if want_dw else None), T, N, K, ctypes.byref(cfg),
                                    _ptr(ws), nbytes, _stream(stream)), "int8mp_linear_bwd")
    return (dX if want_dx else None), (dW if want_dw else None)


def int8mp_linear_fwd_save(X, W, absmax, cfg=None, Y=None, workspace=None, stream=None):
    """int8mp_linear_fwd that also fills absmax (fp32 [2K]) with the column
    absmax of X and of W for int8mp_linear_bwd_saved."""
    cfg = cfg or linear_cfg()
    T, K = X.shape
    N = W.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.bfloat16, device=X.device)
    ws, nbytes = _workspace(T, N, K, cfg, workspace, X.device)
    _check(load().int8mp_linear_fwd_save(_ptr(X), _ptr(W), _ptr(Y), T, N, K, ctypes.byref(cfg),
                                         _ptr(absmax), _ptr(ws), nbytes, _stream(stream)),
           "int8mp_linear_fwd_save")
    return Y


def int8mp_linear_bwd_saved(dY, X, W, absmax, cfg=None, dX=None, dW=None, want_dx=True,
                            want_dw=True, workspace=None, stream=None):
    """int8mp_linear_bwd given the absmax saved by int8mp_linear_fwd_save."""
    cfg = cfg or linear_cfg()
    T, K = X.shape
    N = W.shape[0]
    if want_dx and dX is None:
        dX = torch.empty((T, K), dtype=torch.bfloat16, device=X.device)
    if want_dw and dW is None:
        dW = torch.empty((N, K), dtype=torch.bfloat16, device=X.device)
    ws, nbytes = _workspace(T, N, K, cfg, workspace, X.device)
    _check(load().int8mp_linear_bwd_saved(_ptr(dY), _ptr(X), _ptr(W), _ptr(dX if want_dx else None),
                                          _ptr(dW if want_dw else None), T, N, K,
                                          ctypes.byref(cfg), _ptr(absmax), _ptr(ws), nbytes,
                                          _stream(stream)), "int8mp_linear_bwd_saved")
    return (dX if want_dx else None), (dW if want_dw else None)


def int8mp_poll_device_status(stream=None):
    return load().int8mp_poll_device_status(_stream(stream))


def int8mp_debug_check_division():
    """(code_mismatches, pairs, fast_pairs, quotient_differences,
    (absmax_bits, x_bits)) of the exhaustive division check."""
    res = (ctypes.c_uint64 * 4)()
    first = (ctypes.c_uint32 * 2)()
    _check(load().int8mp_debug_check_division(res, first), "int8mp_debug_check_division")
    return res[0], res[1], res[2], res[3], (first[0], first[1])


def int8mp_debug_mm_s32_drop_first_load(A, B, out, wait_limit_ms=200, stream=None):
    M, K = A.shape
    N = B.shape[0]
    return load().int8mp_debug_mm_s32_drop_first_load(_ptr(A), _ptr(B), M, N, K, _ptr(out),
                                                      out.stride(0), int(wait_limit_ms),
                                                      _stream(stream))


def int8mp_debug_scaled_mm_quant_b(A, sA, B, sB, out=None, stream=None):
    """Test only: A (f16 codes [M,K]) @ B.T with B bf16 [N,K] quantized in
    the GEMM's prologue from its row scales sB -> bf16 [M,N]."""
    M, K = A.shape
    N = B.shape[0]
    assert A.dtype == torch.float16 and B.dtype == torch.bfloat16
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M, N, torch.bfloat16)
    _check(load().int8mp_debug_scaled_mm_quant_b(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K,
                                                 _ptr(out), out.stride(0) if M > 0 else N,
                                                 _stream(stream)),
           "int8mp_debug_scaled_mm_quant_b")
    return out


def int8mp_linear_fwd_noalloc(X, W, cfg=None, Y=None, stream=None):
    """Y [T,N] = X [T,K] . W [N,K]^T like int8mp_linear_fwd, with the
    workspace in the library's fixed per-device scratch array instead of a
    caller-provided buffer (for callers that cannot allocate device memory).
    Y is allocated here only when the caller passes none."""
    cfg = cfg or linear_cfg()
    T, K = X.shape
    N = W.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.bfloat16, device=X.device)
    _check(load().int8mp_linear_fwd_noalloc(_ptr(X), _ptr(W), _ptr(Y), T, N, K, ctypes.byref(cfg),
                                            _stream(stream)), "int8mp_linear_fwd_noalloc")
    return Y
