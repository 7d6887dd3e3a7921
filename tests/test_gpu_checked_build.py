"""The bounds-checked build (-DINT8MP_CHECK): every global index the kernels
compute is checked against its buffer before the access.  Run the paths of
the library through it -- row and column quantization in every variant, the
column maxima, two matrices' rows (and column groups) in one launch, the GEMM in three layouts
with and without the split last wave (f16 containers and int8 codes), the
linear layer in INT8 and in BF16 -- on ragged sizes: no
check may fail, and every result must equal the ordinary build's bit for
bit."""
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
from int8_mixed_precision_row_gb300 import build, synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def checked_lib():
    build.build()
    m.load()
    return build.build(check=True)


def _codes_and_gemms():
    out = []
    for rows, cols in ((77, 136), (1032, 64), (300, 5632), (9, 24576), (3, 53248)):
        x = synth.bf16_normal((rows, cols), rows + cols, outlier_frac=0.01, outlier_scale=20.0).to(DEV)
        for mode in (m.INT8MP_RNE, m.INT8MP_SR):
            for codes in (m.INT8MP_CODES_S8, m.INT8MP_CODES_F16):
                kw = dict(mode=mode, seed=3, offset=5, codes=codes)
                out += list(m.int8mp_quantize_rowwise(x, axis=0, **kw))
                out += list(m.int8mp_quantize_rowwise(x, axis=m.INT8MP_GROUP_COLS, **kw))
                if rows % 8 == 0:
                    out += list(m.int8mp_quantize_rowwise(x, axis=m.INT8MP_GROUP_COLS_T, **kw))
                cm = torch.zeros(cols, dtype=torch.float32, device=DEV)
                out += list(m.int8mp_quantize_rows_colmax(x, cm, **kw)) + [cm]
                out += list(m.int8mp_quantize_cols_absmax(x, cm, **kw))
                x2 = synth.bf16_normal((rows // 2 + 1, cols), rows + 7).to(DEV)
                cms = [torch.zeros(cols, dtype=torch.float32, device=DEV) for _ in range(2)]
                bkw = dict(mode=mode, seed=3, offsets=[5, 9], stream_ids=[0, 1], codes=codes)
                for pair in m.int8mp_quantize_rows_batch([x, x2], **bkw):
                    out += list(pair)
                for pair in m.int8mp_quantize_rows_batch([x, x2], colmaxes=cms, **bkw):
                    out += list(pair)
                for pair in m.int8mp_quantize_cols_batch([x, x2], **bkw):
                    out += list(pair)
                out += cms
    g = torch.Generator().manual_seed(9)
    for M, N, K, lay in ((200, 264, 144, m.INT8MP_AxBT), (2560, 2048, 4096, m.INT8MP_AxB),
                         (2312, 1800, 8256, m.INT8MP_ATxB), (1000, 776, 2096, m.INT8MP_AxB)):
        a_shape = (K, M) if lay == m.INT8MP_ATxB else (M, K)
        b_shape = (N, K) if lay == m.INT8MP_AxBT else (K, N)
        a = torch.randint(-127, 128, a_shape, generator=g).to(torch.float16).to(DEV)
        b = torch.randint(-127, 128, b_shape, generator=g).to(torch.float16).to(DEV)
        sa = torch.rand(M, generator=g).to(DEV)
        sb = torch.rand(N, generator=g).to(DEV)
        out.append(m.int8mp_mm_s32(a, b, layout=lay))
        out.append(m.int8mp_mm_s32(a, b, layout=lay, workspace=True))
        out.append(m.int8mp_scaled_mm(a, sa, b, sb, layout=lay, workspace=True))
        if (lay == m.INT8MP_AxBT or N % 16 == 0) and (lay != m.INT8MP_ATxB or M % 16 == 0):
            # int8 operands (widened in the CTA-pair kernel)
            a8, b8 = a.to(torch.int8), b.to(torch.int8)
            out.append(m.int8mp_mm_s32(a8, b8, layout=lay, workspace=True))
            out.append(m.int8mp_scaled_mm(a8, sa, b8, sb, layout=lay))
    T, N, K = 1040, 2048, 2048
    X = synth.bf16_normal((T, K), 1).to(DEV)
    W = synth.bf16_normal((N, K), 2, std=0.02).to(DEV)
    dY = synth.bf16_normal((T, N), 3, std=1e-3).to(DEV)
    cfg = m.linear_cfg(mode=m.INT8MP_SR, seed=4)
    absmax = torch.empty(2 * K, dtype=torch.float32, device=DEV)
    out.append(m.int8mp_linear_fwd_save(X, W, absmax, cfg))
    out += list(m.int8mp_linear_bwd_saved(dY, X, W, absmax, cfg))
    out += list(m.int8mp_linear_bwd(dY, X, W, cfg))
    bf16 = m.linear_cfg(int8_fwd=0, int8_grad_in=0, int8_grad_w=0)  # the BF16 passes
    out.append(m.int8mp_linear_fwd(X, W, bf16))
    out += list(m.int8mp_linear_bwd(dY, X, W, bf16))
    torch.cuda.synchronize()
    return out


def test_checked_build_finds_no_out_of_bounds_access(checked_lib):
    plain = _codes_and_gemms()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    with m.use_library(checked_lib):
        checked = _codes_and_gemms()
        status = m.int8mp_poll_device_status()
    assert status == m.INT8MP_OK, m.int8mp_status_string(status)
    assert len(plain) == len(checked)
    for i, (a, b) in enumerate(zip(plain, checked)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), i
