"""Token-sharded data parallelism with two gloo ranks on the CPU.

Each rank takes its block of token rows (dp.shard_rows), its stochastic
rounding offset (dp.shard_offset), forms its fp32 partial grad-weight from
the oracle (this machine has no GPU; the library's kernels for the same
steps are checked on one GPU in test_gpu_sharded.py), and the ranks sum the
partials with dp.reduce_partials (a gloo all-reduce).  The reduced sum must be
the two partials added exactly, and its bf16 rounding the oracle's sharded
grad-weight (the sum of per-shard oracle results, rounded once).
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    from int8_mixed_precision_row_gb300 import synth
    T, N, K = 64, 24, 40
    dY = synth.bf16_normal((T, N), 31, std=1e-3)
    X = synth.bf16_normal((T, K), 32, outlier_frac=0.05, outlier_scale=20.0)
    return dY, X


def _worker(rank, world, port, mode, async_op, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch
    import torch.distributed as dist
    import oracle
    from helpers import bf16_bits
    from int8_mixed_precision_row_gb300 import dp
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    dY, X = _inputs()
    T, N = dY.shape
    K = X.shape[1]
    t0, t1 = dp.shard_rows(T, world, rank)
    off = dp.shard_offset(5, rank)
    g, x = bf16_bits(dY[t0:t1]), bf16_bits(X[t0:t1])
    qg, sg = oracle.quantize(g, 1, mode=mode, seed=9, offset=off, stream_id=oracle.STREAM_GW_DY)
    qx, sx = oracle.quantize(x, 1, mode=mode, seed=9, offset=off, stream_id=oracle.STREAM_GW_X)
    mine = oracle.scaled_mm_f32(qg, sg, qx, sx, N, K, t1 - t0)
    part = torch.from_numpy(mine.copy())
    if async_op:  # started, then waited for (the bench step overlaps it with later linears)
        dp.reduce_partials(part, async_op=True).wait()
    else:
        dp.reduce_partials(part)
    out[rank] = (mine, part.numpy().copy())
    dist.destroy_process_group()


@pytest.mark.parametrize("async_op", [False, True])
@pytest.mark.parametrize("mode", [0, 1])
def test_two_rank_grad_weight_is_the_sum_of_shard_oracles(mode, async_op):
    import oracle
    from helpers import bf16_bits
    from int8_mixed_precision_row_gb300 import dp
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, mode, async_op, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (p0, s0), (p1, s1) = out[0], out[1]
    np.testing.assert_array_equal(s0, s1)                      # every rank holds the sum
    np.testing.assert_array_equal(s0, p0 + p1)                 # fp32, exact order for two ranks
    dY, X = _inputs()
    ref = oracle.grad_weight_sharded(bf16_bits(dY), bf16_bits(X), 2,
                                     [dp.shard_offset(5, 0), dp.shard_offset(5, 1)], mode=mode,
                                     seed=9)
    rounded = np.array([[oracle.bf16_rne(v) for v in row] for row in s0], dtype=np.uint16)
    np.testing.assert_array_equal(rounded, ref)


def test_shard_rows_and_offsets():
    from int8_mixed_precision_row_gb300 import dp
    assert [dp.shard_rows(64, 2, r) for r in range(2)] == [(0, 32), (32, 64)]
    assert [dp.shard_rows(32768, 4, r)[0] for r in range(4)] == [0, 8192, 16384, 24576]
    with pytest.raises(ValueError):
        dp.shard_rows(48, 2, 0)                                 # 24 rows: not a multiple of 16
    assert dp.shard_offset(7, 3) == 7 + 3 * (1 << 40)
