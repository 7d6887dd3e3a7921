"""Token-sharded data parallelism of the INT8 linear layer.

"Integrate INT8 mixed-precision from torchao 0.7", discussion: the method
trains with FSDP2 across two A100s; torchao issue 1887: in ZeRO-3 style
training the weight gradients are reduce-scattered across the ranks.  The
method shards naturally over tokens: the forward and grad-input matmuls
contract over K and N and are independent per token, so each rank runs them
on its own rows; the grad-weight matmul contracts over T, so each rank forms
the part of dW its own tokens give, and the ranks sum those parts.

Reading (the pages give no arithmetic for the exchange): rank r quantizes
its rows of dY and X along T with its own column scales (the grad-weight
operands of its shard, exactly as a single device would for those rows),
forms the fp32 partial P_r = (fp32(acc) * s_dY) * s_X without rounding it
(int8mp_scaled_mm_f32), the ranks add their partials in fp32 (one
all-reduce), and the sum is rounded to bf16 once (int8mp_round_bf16):
dW = bf16_RNE(P_0 + ... + P_{n-1}).  With two ranks the fp32 sum has one
order; with more, the all-reduce's order decides the last fp32 bits.
Stochastic rounding on rank r draws from counters offset + r * 2^40, so the
ranks' streams are disjoint.

This module only arranges the calls: every quantization, matmul and rounding
runs in the library's kernels, and the sum is a torch.distributed
all-reduce.
"""
from . import binding as b

SHARD_OFFSET_STRIDE = 1 << 40


def shard_rows(T, world, rank):
    """[t0, t1) of rank `rank`'s tokens: world equal blocks of consecutive
    rows, each a multiple of 16 (the library's size rule)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if T % (16 * world):
        raise ValueError(f"T = {T} does not split into {world} shards of a multiple of 16 rows")
    t = T // world
    return rank * t, (rank + 1) * t


def shard_offset(offset, rank):
    """Stochastic-rounding counter offset of rank `rank`."""
    return int(offset) + int(rank) * SHARD_OFFSET_STRIDE


def grad_weight_partial(dY, X, cfg, colmax_dy=None, colmax_x=None, workspace=None, stream=None):
    """fp32 [N, K] part of dW = dY^T X given by this rank's rows dY [T_r, N]
    and X [T_r, K]: both quantized along T by columns (codes left in place;
    from the given column absmax when the row passes recorded it), then the
    A.T @ B matmul with an unrounded fp32 result."""
    kw = dict(mode=cfg.mode, seed=cfg.seed, offset=cfg.offset, codes=b.INT8MP_CODES_F16,
              stream=stream)
    if colmax_dy is None:
        qg, sg = b.int8mp_quantize_rowwise(dY, axis=b.INT8MP_GROUP_COLS,
                                           stream_id=b.INT8MP_STREAM_GW_DY, **kw)
    else:
        qg, sg = b.int8mp_quantize_cols_absmax(dY, colmax_dy, stream_id=b.INT8MP_STREAM_GW_DY, **kw)
    if colmax_x is None:
        qx, sx = b.int8mp_quantize_rowwise(X, axis=b.INT8MP_GROUP_COLS,
                                           stream_id=b.INT8MP_STREAM_GW_X, **kw)
    else:
        qx, sx = b.int8mp_quantize_cols_absmax(X, colmax_x, stream_id=b.INT8MP_STREAM_GW_X, **kw)
    return b.int8mp_scaled_mm_f32(qg, sg, qx, sx, layout=b.INT8MP_ATxB, workspace=workspace,
                                  stream=stream)


def reduce_partials(partial, group=None, async_op=False):
    """The ranks' fp32 partials summed in place on every rank (one
    all-reduce of the [N, K] buffer).  async_op: start it and return its
    handle (the sum is in place once handle.wait() returns; on the GPU, work
    queued after wait() on the current stream sees it), so that it runs
    while later work is computed."""
    import torch.distributed as dist
    work = dist.all_reduce(partial, op=dist.ReduceOp.SUM, group=group, async_op=async_op)
    return work if async_op else partial


def grad_weight_data_parallel(dY, X, cfg, group=None, dW=None, workspace=None, stream=None):
    """bf16 dW [N, K] of the whole job from this rank's rows: partial,
    all-reduce, one rounding."""
    p = grad_weight_partial(dY, X, cfg, workspace=workspace, stream=stream)
    reduce_partials(p, group)
    return b.int8mp_round_bf16(p, dW, stream=stream)
