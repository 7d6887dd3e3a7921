"""The kernels of token-sharded data parallelism on one GPU.

Every run here has one GPU, so the ranks are emulated in turn on it: each
shard's partial grad-weight comes from dp.grad_weight_partial (column
quantization of its rows, int8mp_scaled_mm_f32), the partials are added on
the device in rank order (what the all-reduce does; exact in any order for
two ranks), and int8mp_round_bf16 rounds the sum.  Each partial must equal
the oracle's shard partial bit for bit, and the result the oracle's sharded
grad-weight.  The all-reduce itself runs with two gloo ranks in
test_dp_gloo.py.
"""
import numpy as np
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
import oracle
from helpers import bf16_bits
from int8_mixed_precision_row_gb300 import dp, synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


CASES = [(2, 2048, 5632, 2048, m.INT8MP_RNE), (2, 1024, 2048, 5632, m.INT8MP_SR),
         (4, 4096, 1040, 264, m.INT8MP_RNE)]


@pytest.mark.parametrize("world,T,N,K,mode", CASES)
def test_sharded_grad_weight_kernels(world, T, N, K, mode):
    dY = synth.bf16_normal((T, N), 51, std=1e-3)
    X = synth.bf16_normal((T, K), 52, outlier_frac=0.005, outlier_scale=30.0)
    dYd, Xd = dY.to(DEV), X.to(DEV)
    ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=DEV)
    total = None
    offsets = []
    for r in range(world):
        t0, t1 = dp.shard_rows(T, world, r)
        offsets.append(dp.shard_offset(3, r))
        cfg = m.linear_cfg(mode=mode, seed=17, offset=offsets[-1])
        part = dp.grad_weight_partial(dYd[t0:t1], Xd[t0:t1], cfg, workspace=ws)
        torch.cuda.synchronize()
        g, x = bf16_bits(dY[t0:t1]), bf16_bits(X[t0:t1])
        kw = dict(mode=mode, seed=17, offset=offsets[-1])
        qg, sg = oracle.quantize(g, 1, stream_id=oracle.STREAM_GW_DY, **kw)
        qx, sx = oracle.quantize(x, 1, stream_id=oracle.STREAM_GW_X, **kw)
        ref = oracle.scaled_mm_f32(qg, sg, qx, sx, N, K, t1 - t0)
        np.testing.assert_array_equal(part.cpu().numpy().view(np.int32), ref.view(np.int32),
                                      err_msg=f"partial of shard {r}")
        total = part if total is None else total + part      # the all-reduce, in rank order
    dW = m.int8mp_round_bf16(total)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    ref = oracle.grad_weight_sharded(bf16_bits(dY), bf16_bits(X), world, offsets, mode=mode,
                                     seed=17)
    np.testing.assert_array_equal(bf16_bits(dW.cpu()), ref)


def test_round_bf16_matches_the_oracle_rounding():
    g = torch.Generator().manual_seed(8)
    x = torch.randn(1000003, generator=g) * 10.0 ** torch.randint(-30, 30, (1000003,), generator=g)
    x[:6] = torch.tensor([0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.0e38, 1e-40])
    y = m.int8mp_round_bf16(x.to(DEV))
    torch.cuda.synchronize()
    got = bf16_bits(y.cpu())
    idx = np.random.default_rng(0).choice(x.numel(), 5000, replace=False)
    idx = np.concatenate([np.arange(6), idx])
    ref = np.array([oracle.bf16_rne(float(x[i])) for i in idx], dtype=np.uint16)
    np.testing.assert_array_equal(got[idx], ref)
