"""The GEMM with its B operand quantized in the prologue (test-only entry
int8mp_debug_scaled_mm_quant_b): the alternative to the separate row pass
that "Integrate INT8 mixed-precision from torchao 0.7" (limitations) points
at, kept so that the library's choice can be measured.  Its codes must be
the row quantizer's, so its products equal int8mp_scaled_mm on the
quantizer's codes bit for bit -- including rows whose scale takes the IEEE
division path (all-zero, subnormal and huge rows) -- and the oracle's.
"""
import numpy as np
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
import oracle
from helpers import bf16_bits
from int8_mixed_precision_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


@pytest.mark.parametrize("shape", [(256, 256, 512), (1040, 264, 1040), (4096, 2048, 2048),
                                   (200, 520, 8192)])
def test_prologue_quantized_b_equals_the_separate_pass(shape):
    M, N, K = shape
    A = synth.bf16_normal((M, K), 71, outlier_frac=0.01, outlier_scale=20.0)
    B = synth.bf16_normal((N, K), 72, std=0.02, outlier_frac=0.005, outlier_scale=30.0)
    B[0] = 0.0                                   # zero scale
    B[1] = B[1] * 1e-38                          # subnormal scale: IEEE division
    B[2] = B[2] * 1e30                           # scale above 2^10: IEEE division
    Ad, Bd = A.to(DEV), B.to(DEV)
    qa, sa = m.int8mp_quantize_rowwise(Ad, axis=m.INT8MP_GROUP_ROWS, codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(Bd, axis=m.INT8MP_GROUP_ROWS, codes=m.INT8MP_CODES_F16)
    got = m.int8mp_debug_scaled_mm_quant_b(qa, sa, Bd, sb)
    ref = m.int8mp_scaled_mm(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    rows = np.unique(np.linspace(0, M - 1, 5).astype(np.int64))
    qar, sar = oracle.quantize(bf16_bits(A), 0)
    qbr, sbr = oracle.quantize(bf16_bits(B), 0)
    expect = oracle.scaled_mm(qar[rows], sar[rows], qbr, sbr, len(rows), N, K)
    np.testing.assert_array_equal(bf16_bits(got[torch.from_numpy(rows).to(DEV)].cpu()), expect)
