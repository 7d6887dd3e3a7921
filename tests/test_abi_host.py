"""C-ABI checks that need no GPU: the library loads, exports every symbol the
public headers declare, and rejects bad arguments on the host before it
touches a device."""
import ctypes
import os
import re

import pytest

import int8_mixed_precision_row_gb300 as m
from int8_mixed_precision_row_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return m.load()


def _declared_symbols():
    names = set()
    for h in ("int8mp.h", "int8mp_debug.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(int8mp_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert declared == set(m.EXPORTED), declared ^ set(m.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert m.int8mp_version() >= 100
    for st in range(8):
        assert m.int8mp_status_string(st) != "unknown status"
    assert m.int8mp_status_string(99) == "unknown status"


def test_checked_build_compiles_and_exports_everything():
    path = mbuild.build(check=True)
    assert path != mbuild.LIB and os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(lib, name), name


P = ctypes.c_void_p


def _q(lib, x, rows, cols, ld, axis, mode=0, codes=0, q=16, scale=16):
    return lib.int8mp_quantize_rowwise(P(x), rows, cols, ld, axis, mode, 0, 0, 0, P(q), codes,
                                       P(scale), None)


def test_quantize_host_validation(lib):
    assert _q(lib, 16, 8, 8, 8, axis=3) == m.INT8MP_ERR_INVALID_ARG
    assert _q(lib, 16, 8, 8, 8, axis=0, mode=3) == m.INT8MP_ERR_INVALID_ARG
    assert _q(lib, 16, 8, 8, 8, axis=0, codes=5) == m.INT8MP_ERR_INVALID_ARG
    assert _q(lib, 16, 8, 16, 8, axis=0) == m.INT8MP_ERR_INVALID_ARG      # ld < cols
    assert _q(lib, 0, 8, 8, 8, axis=0) == m.INT8MP_ERR_INVALID_ARG        # null x
    assert _q(lib, 16, 0, 8, 8, axis=0, q=0, scale=0) == m.INT8MP_OK      # empty: nothing to do
    assert _q(lib, 16, 8, 12, 16, axis=0) == m.INT8MP_ERR_ALIGNMENT       # cols % 8
    assert _q(lib, 24, 8, 8, 8, axis=0) == m.INT8MP_ERR_ALIGNMENT         # x not 16-byte aligned
    assert _q(lib, 16, 12, 8, 8, axis=1) == m.INT8MP_ERR_ALIGNMENT        # axis 1 needs rows % 8


def test_absmax_entry_points_host_validation(lib):
    rc = lib.int8mp_quantize_rows_colmax(P(16), 8, 8, 8, 0, 0, 0, 0, P(16), 1, P(16), None, None)
    assert rc == m.INT8MP_ERR_INVALID_ARG                                 # colmax missing
    rc = lib.int8mp_quantize_rows_colmax(P(16), 8, 8, 8, 0, 0, 0, 0, P(16), 1, P(16), P(18), None)
    assert rc == m.INT8MP_ERR_ALIGNMENT                                   # colmax misaligned
    rc = lib.int8mp_quantize_cols_absmax(P(16), 8, 8, 8, None, 0, 0, 0, 0, P(16), 1, P(16), None)
    assert rc == m.INT8MP_ERR_INVALID_ARG
    rc = lib.int8mp_quantize_cols_absmax(P(16), 8, 12, 16, P(16), 0, 0, 0, 0, P(16), 1, P(16), None)
    assert rc == m.INT8MP_ERR_ALIGNMENT                                   # cols % 8
    assert lib.int8mp_quantize_cols_absmax(P(16), 0, 8, 8, None, 0, 0, 0, 0, None, 1, None,
                                           None) == m.INT8MP_OK          # empty
    cfg = m.linear_cfg()
    ref = ctypes.byref(cfg)
    assert lib.int8mp_linear_fwd_save(P(16), P(16), P(16), 32, 32, 32, ref, None, P(256), 1 << 20,
                                      None) == m.INT8MP_ERR_INVALID_ARG
    assert lib.int8mp_linear_bwd_saved(P(16), P(16), P(16), P(16), P(16), 32, 32, 32, ref, None,
                                       P(256), 1 << 20, None) == m.INT8MP_ERR_INVALID_ARG
    assert lib.int8mp_linear_bwd_saved(P(16), P(16), P(16), P(16), P(16), 32, 32, 32, ref, P(18),
                                       P(256), 1 << 20, None) == m.INT8MP_ERR_ALIGNMENT


def test_cols_batch_host_validation(lib):
    J = m.int8mp_rows_job

    def run(*jobs, n=None, cols=8, mode=0, codes=1):
        arr = (J * max(len(jobs), 1))(*jobs)
        return lib.int8mp_quantize_cols_batch(arr if jobs else None, len(jobs) if n is None else n,
                                              cols, mode, 0, codes, None)
    plain = J(16, 8, 8, 0, 0, 16, 16, None)
    assert run() == m.INT8MP_ERR_INVALID_ARG                               # no jobs
    assert run(plain, n=0) == m.INT8MP_ERR_INVALID_ARG                     # njobs 0
    assert run(plain, plain, plain) == m.INT8MP_ERR_INVALID_ARG            # more than two
    assert run(J(16, 8, 8, 0, 1, 16, 16, 16)) == m.INT8MP_ERR_INVALID_ARG  # colmax given
    assert run(plain, mode=3) == m.INT8MP_ERR_INVALID_ARG
    assert run(plain, codes=4) == m.INT8MP_ERR_INVALID_ARG
    assert run(J(24, 8, 8, 0, 0, 16, 16, None)) == m.INT8MP_ERR_ALIGNMENT  # x misaligned
    assert run(J(16, 8, 8, 0, 0, 24, 16, None)) == m.INT8MP_ERR_ALIGNMENT  # q misaligned
    assert run(plain, cols=12) == m.INT8MP_ERR_INVALID_ARG                 # ld < cols
    assert run(J(16, 8, 16, 0, 0, 16, 16, None), cols=12) == m.INT8MP_ERR_ALIGNMENT  # cols % 8
    assert run(J(16, 0, 8, 0, 0, 16, 16, None)) == m.INT8MP_OK             # empty: nothing launched


def test_rows_batch_host_validation(lib):
    J = m.int8mp_rows_job

    def run(*jobs, n=None, cols=8, mode=0, codes=1):
        arr = (J * max(len(jobs), 1))(*jobs)
        return lib.int8mp_quantize_rows_batch(arr if jobs else None, len(jobs) if n is None else n,
                                              cols, mode, 0, codes, None)
    plain = J(16, 8, 8, 0, 0, 16, 16, None)
    kept = J(16, 8, 8, 0, 1, 16, 16, 16)
    assert run() == m.INT8MP_ERR_INVALID_ARG                               # no jobs
    assert run(plain, n=0) == m.INT8MP_ERR_INVALID_ARG                     # njobs 0
    assert run(plain, plain, plain) == m.INT8MP_ERR_INVALID_ARG            # more than two
    assert run(plain, kept) == m.INT8MP_ERR_INVALID_ARG                    # colmax for one only
    assert run(plain, mode=3) == m.INT8MP_ERR_INVALID_ARG
    assert run(plain, codes=4) == m.INT8MP_ERR_INVALID_ARG
    assert run(J(24, 8, 8, 0, 0, 16, 16, None)) == m.INT8MP_ERR_ALIGNMENT  # x misaligned
    assert run(plain, cols=12) == m.INT8MP_ERR_INVALID_ARG                 # ld < cols
    assert run(J(16, 8, 16, 0, 0, 16, 16, None), cols=12) == m.INT8MP_ERR_ALIGNMENT  # cols % 8
    assert run(J(16, 8, 8, 0, 1, 16, 16, 18)) == m.INT8MP_ERR_ALIGNMENT   # colmax misaligned
    assert run(J(16, 0, 8, 0, 0, None, None, None)) == m.INT8MP_OK         # empty: nothing to do


def _mm(lib, M, N, K, layout=0, codes=1, A=16, B=16, out=16, ldo=None):
    return lib.int8mp_mm_s32(P(A), P(B), M, N, K, layout, codes, P(out), N if ldo is None else ldo,
                             None)


def test_matmul_host_validation(lib):
    assert _mm(lib, 8, 8, 16, layout=3) == m.INT8MP_ERR_INVALID_ARG       # no such layout
    assert _mm(lib, 8, 8, 16, codes=2) == m.INT8MP_ERR_INVALID_ARG        # no such code container
    assert _mm(lib, 8, 24, 16, layout=1, codes=0) == m.INT8MP_ERR_ALIGNMENT   # int8 [K,N] rows: N % 16
    assert _mm(lib, 24, 16, 16, layout=2, codes=0) == m.INT8MP_ERR_ALIGNMENT  # int8 [K,M] rows: M % 16
    assert _mm(lib, 12, 8, 16, layout=2) == m.INT8MP_ERR_ALIGNMENT        # A.T@B: rows of A^T, M % 8
    assert _mm(lib, 8, 12, 16, layout=1) == m.INT8MP_ERR_ALIGNMENT        # A@B: rows of B, N % 8
    assert _mm(lib, 8, 8, m.INT8MP_MAX_K + 1) == m.INT8MP_ERR_INVALID_ARG
    assert _mm(lib, 8, 8, 24) == m.INT8MP_ERR_ALIGNMENT                   # K % 16
    assert _mm(lib, 8, 12, 16) == m.INT8MP_ERR_ALIGNMENT                  # N % 8
    assert _mm(lib, 8, 8, 16, A=8) == m.INT8MP_ERR_ALIGNMENT
    assert _mm(lib, 8, 8, 16, out=0) == m.INT8MP_ERR_INVALID_ARG
    assert _mm(lib, 0, 8, 16, A=0, B=0, out=0) == m.INT8MP_OK             # empty


def test_matmul_workspace_host_validation(lib):
    need = m.int8mp_mm_workspace_size()
    assert need >= 76 * 256 * 256 * 4                                     # an int32 tile per SM pair
    f = lib.int8mp_mm_s32_ws
    assert f(P(16), P(16), 8, 8, 16, 0, 1, P(16), 8, P(128), need, None) == m.INT8MP_ERR_ALIGNMENT
    assert f(P(16), P(16), 8, 8, 16, 0, 1, P(256), 8, P(256), need - 1, None) == \
        m.INT8MP_ERR_WORKSPACE
    g = lib.int8mp_scaled_mm_ws
    assert g(P(16), P(16), P(16), P(16), 8, 8, 16, 0, 1, P(16), 8, P(256), 16, None) == \
        m.INT8MP_ERR_WORKSPACE
    assert g(P(16), P(16), P(16), P(16), 8, 8, 16, 0, 2, P(16), 8, P(256), need, None) == \
        m.INT8MP_ERR_INVALID_ARG                                          # no such code container


def test_linear_host_validation(lib):
    cfg = m.linear_cfg()
    ref = ctypes.byref(cfg)
    f = lib.int8mp_linear_fwd
    assert f(P(16), P(16), P(16), 32, 32, 32, None, P(256), 1 << 20, None) == m.INT8MP_ERR_INVALID_ARG
    assert f(P(16), P(16), P(16), 32, 32, 24, ref, P(256), 1 << 20, None) == m.INT8MP_ERR_ALIGNMENT
    assert f(P(16), P(16), P(16), 32, 32, 32, ref, P(256), 16, None) == m.INT8MP_ERR_WORKSPACE
    bad = m.int8mp_linear_cfg(2, 1, 1, 0, 0, 0)   # a pass switch is 0 (BF16) or 1 (INT8)
    assert f(P(16), P(16), P(16), 32, 32, 32, ctypes.byref(bad), P(256), 1 << 20, None) == \
        m.INT8MP_ERR_INVALID_ARG
    assert lib.int8mp_linear_fwd_noalloc(P(16), P(16), P(16), 32, 32, 32, None,
                                         None) == m.INT8MP_ERR_INVALID_ARG   # no cfg
    need = m.int8mp_linear_workspace_size(32, 48, 64, cfg)
    assert need >= 2 * (32 * 64 + 48 * 64) + m.int8mp_mm_workspace_size() and need % 256 == 0
    assert m.int8mp_linear_workspace_size(32, 48, 24, cfg) == 0


def test_product_path_has_no_oracle_or_fallback():
    pkg = os.path.join(ROOT, "int8_mixed_precision_row_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "liboracle" not in text and "oracle.h" not in text, fn
