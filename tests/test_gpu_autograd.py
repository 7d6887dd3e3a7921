"""The autograd wrapper: same bits as the direct C-ABI calls, gradients of
the right shape, and close to the bf16 matmul it approximates."""
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
from int8_mixed_precision_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


@pytest.mark.parametrize("stochastic", [False, True])
def test_module_matches_direct_calls(stochastic):
    torch.manual_seed(0)
    lin = m.Int8MixedPrecisionLinear(256, 192, device=DEV, stochastic=stochastic, seed=5)
    x = synth.bf16_normal((2, 64, 256), 1).to(DEV).requires_grad_(True)
    dy = synth.bf16_normal((2, 64, 192), 2, std=1e-3).to(DEV)
    y = lin(x)
    y.backward(dy)
    mode = m.INT8MP_SR if stochastic else m.INT8MP_RNE
    cfg = m.linear_cfg(mode=mode, seed=5, offset=0)
    x2 = x.detach().reshape(-1, 256)
    y_ref = m.int8mp_linear_fwd(x2, lin.weight.detach(), cfg)
    dx_ref, dw_ref = m.int8mp_linear_bwd(dy.reshape(-1, 192), x2, lin.weight.detach(), cfg)
    assert torch.equal(y.detach().reshape(-1, 192).view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(x.grad.reshape(-1, 256).view(torch.int16), dx_ref.view(torch.int16))
    assert torch.equal(lin.weight.grad.view(torch.int16), dw_ref.view(torch.int16))
    if stochastic:
        assert lin.offset == m.Int8MixedPrecisionLinear.OFFSET_STEP


def test_module_close_to_bf16_matmul():
    torch.manual_seed(0)
    lin = m.Int8MixedPrecisionLinear(512, 256, device=DEV)
    x = synth.bf16_normal((128, 512), 3).to(DEV).requires_grad_(True)
    y = lin(x)
    ref = (x.detach().double() @ lin.weight.detach().double().T)
    err = (y.double() - ref).norm() / ref.norm()
    assert 1e-3 < err < 3e-2
    y.sum().backward()
    assert x.grad.shape == x.shape and lin.weight.grad.shape == lin.weight.shape


def test_weight_only_gradient():
    lin = m.Int8MixedPrecisionLinear(128, 64, device=DEV)
    x = synth.bf16_normal((32, 128), 4).to(DEV)  # no input gradient wanted
    lin(x).float().sum().backward()
    assert lin.weight.grad is not None
