"""A Llama2-1B-shaped decoder layer's linears through the autograd module.

"Integrate INT8 mixed-precision from torchao 0.7", discussion (module swap,
the INT8 linear's autograd function) and torchao issue 1887
(`quantize_(model, int8_mixed_precision_training(), filter_fn)`): every
linear of the model is replaced by one whose forward, grad-input and
grad-weight matmuls run in INT8.

Int8MixedPrecisionDecoderLinears (q, k, v, o, gate, up, down with SwiGLU;
attention core and norms out of scope) runs forward and backward through
torch.autograd on the GPU.  The same composition is rebuilt on the CPU from
the oracle's linear passes alone -- no GPU value enters it -- with the
elementwise glue in float64 torch CPU ops.  Every linear's output, the
layer's output, the input gradient and all seven weight gradients must match
bit for bit, with nearest-even and with stochastic rounding.
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
HIDDEN, INTER = 2048, 5632
T = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


def _bits(t):
    return bf16_bits(t.detach().cpu())


def _from_bits(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def _weights():
    shapes = {"q": (HIDDEN, HIDDEN), "k": (HIDDEN, HIDDEN), "v": (HIDDEN, HIDDEN),
              "o": (HIDDEN, HIDDEN), "gate": (INTER, HIDDEN), "up": (INTER, HIDDEN),
              "down": (HIDDEN, INTER)}
    return {n: synth.bf16_normal(shapes[n], 20 + i, std=0.02)
            for i, n in enumerate(m.Int8MixedPrecisionDecoderLinears.NAMES)}


def _oracle_layer(x, dy, W, mode, seed):
    """The decoder layer's forward and backward composed from oracle passes
    (glue in float64 on the CPU).  Returns (linear outputs, y, dx, dW)."""
    G, bf = torch.float64, torch.bfloat16
    idx = {n: i for i, n in enumerate(m.Int8MixedPrecisionDecoderLinears.NAMES)}
    kw = lambda n: dict(mode=mode, seed=seed + idx[n], offset=0)

    def fwd(n, inp):
        return _from_bits(oracle.linear_fwd(_bits(inp), _bits(W[n]), **kw(n)))

    def bwd(n, d_out, inp):
        dX, dW = oracle.linear_bwd(_bits(d_out), _bits(inp), _bits(W[n]), **kw(n))
        return _from_bits(dX), _from_bits(dW)

    outs = {}
    xg = x.to(G)
    xb = xg.to(bf)
    outs["q"], outs["k"], outs["v"] = fwd("q", xb), fwd("k", xb), fwd("v", xb)
    qg, kg, vg = outs["q"].to(G), outs["k"].to(G), outs["v"].to(G)
    a = (vg + qg * kg).to(bf)
    outs["o"] = fwd("o", a)
    h = xg + outs["o"].to(G)
    hb = h.to(bf)
    outs["gate"], outs["up"] = fwd("gate", hb), fwd("up", hb)
    g, u = outs["gate"].to(G), outs["up"].to(G)
    s = torch.sigmoid(g)
    z = (g * s * u).to(bf)
    outs["down"] = fwd("down", z)
    y = (h + outs["down"].to(G)).to(bf)

    dW = {}
    dyg = dy.to(G)
    dz, dW["down"] = bwd("down", dy, z)
    dzg = dz.to(G)
    du = (dzg * (g * s)).to(bf)
    dgs = dzg * u                                  # d(g * s)
    dg = (dgs * s + dgs * g * s * (1.0 - s)).to(bf)
    dh_g, dW["gate"] = bwd("gate", dg, hb)
    dh_u, dW["up"] = bwd("up", du, hb)
    dh = dyg + dh_g.to(G) + dh_u.to(G)             # sums of bf16 values: exact
    da, dW["o"] = bwd("o", dh.to(bf), a)
    dag = da.to(G)
    dq, dk, dv = (dag * kg).to(bf), (dag * qg).to(bf), dag.to(bf)
    dx_q, dW["q"] = bwd("q", dq, xb)
    dx_k, dW["k"] = bwd("k", dk, xb)
    dx_v, dW["v"] = bwd("v", dv, xb)
    dx = (dh + dx_q.to(G) + dx_k.to(G) + dx_v.to(G)).to(bf)
    return outs, y, dx, dW


@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
def test_decoder_layer_matches_oracle_composition(mode):
    seed = 40
    W = _weights()
    x = synth.bf16_normal((T, HIDDEN), 10)
    dy = synth.bf16_normal((T, HIDDEN), 30, std=1e-3)
    layer = m.Int8MixedPrecisionDecoderLinears(HIDDEN, INTER, device=DEV,
                                               stochastic=mode == m.INT8MP_SR, seed=seed,
                                               glue_dtype=torch.float64)
    seen = {}
    for name, lin in layer.linears():
        with torch.no_grad():
            lin.weight.copy_(W[name].to(DEV))
        lin.register_forward_hook(lambda mod, inp, out, name=name: seen.__setitem__(name, out))
    xd = x.to(DEV).requires_grad_(True)
    y = layer(xd)
    y.backward(dy.to(DEV))
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK

    outs, y_ref, dx_ref, dW_ref = _oracle_layer(x, dy, W, mode, seed)
    for name in m.Int8MixedPrecisionDecoderLinears.NAMES:
        np.testing.assert_array_equal(_bits(seen[name]), _bits(outs[name]), err_msg=f"{name} output")
    np.testing.assert_array_equal(_bits(y), _bits(y_ref), err_msg="layer output")
    np.testing.assert_array_equal(_bits(xd.grad), _bits(dx_ref), err_msg="input gradient")
    for name, lin in layer.linears():
        np.testing.assert_array_equal(_bits(lin.weight.grad), _bits(dW_ref[name]),
                                      err_msg=f"{name} weight gradient")
