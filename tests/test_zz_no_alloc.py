"""int8mp_linear_fwd_noalloc: the forward pass for callers that cannot
allocate device memory (their host program owns all device memory through
its own pool, or they may not call cudaMalloc/cudaFree at run time because
those calls can synchronize the device).  It takes its workspace from the
library's fixed per-device scratch array.

The test calls it through the C ABI twice in a row and requires the same
bits as int8mp_linear_fwd, which the parity tests hold to the oracle.  The
file sorts last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
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


def _inputs(T, N, K, seed):
    X = synth.bf16_normal((T, K), seed, outlier_frac=0.005, outlier_scale=30.0).to(DEV)
    W = synth.bf16_normal((N, K), seed + 1, std=0.02).to(DEV)
    return X, W


def test_noalloc_forward_matches_workspace_forward_on_two_calls_in_a_row():
    cases = [((256, 256, 512), m.linear_cfg()),                                   # first call on the device
             ((1040, 64, 1056), m.linear_cfg(mode=m.INT8MP_SR, seed=11, offset=5)),  # second: other sizes, SR
             # a long contraction: the CTA-pair matmul, whose last wave the
             # workspace forward splits but the scratch array must not
             ((384, 256, 8192), m.linear_cfg()),
             ((256, 256, 512), m.linear_cfg(mode=m.INT8MP_SR, seed=3))]
    for (T, N, K), cfg in cases:
        X, W = _inputs(T, N, K, seed=T + K)
        ref = m.int8mp_linear_fwd(X, W, cfg)
        got = m.int8mp_linear_fwd_noalloc(X, W, cfg)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (T, N, K)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 4096 x 4096 operands need 2 * 2 * 4096 * 4096 bytes of codes: 64 MiB
    X = torch.zeros((4096, 4096), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((4096, 4096), dtype=torch.bfloat16, device=DEV)
    Y = torch.full((4096, 4096), 3.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(m.Int8mpError) as err:
        m.int8mp_linear_fwd_noalloc(X, W, Y=Y)
    assert err.value.status == m.INT8MP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(Y == 3.0)  # nothing was launched
