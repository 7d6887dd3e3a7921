"""torch.autograd wiring of the INT8 mixed-precision linear layer.

"Integrate INT8 mixed-precision from torchao 0.7": the linear layer's
forward and backward matmuls run in INT8 while the weight and the saved
activation stay bf16 (memory does not change).  Int8MixedPrecisionLinear
is a bias-free drop-in for nn.Linear with a bf16 weight [out, in]; both
passes call the library (int8mp_linear_fwd / int8mp_linear_bwd) and do
nothing else.  The forward pass keeps one thing for the backward pass
besides X and W: their column absmax (2 x in_features floats, recorded while
the forward pass reads them), so that the backward pass's column
quantizations of X and W need no extra pass over them
(int8mp_linear_fwd_save / int8mp_linear_bwd_saved; results are those of the
plain passes bit for bit).  Requirements of the library apply to the
flattened input: the token count, in_features and out_features must be
multiples of 16.
"""
import torch

from . import binding as b


class Int8MixedPrecisionLinearFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, mode, seed, offset):
        K = x.shape[-1]
        N = weight.shape[0]
        x2 = x.reshape(-1, K)
        if not x2.is_contiguous():
            x2 = x2.contiguous()
        cfg = b.linear_cfg(mode=mode, seed=seed, offset=offset)
        absmax = torch.empty((2 * K,), dtype=torch.float32, device=x.device)
        y = b.int8mp_linear_fwd_save(x2, weight, absmax, cfg)
        ctx.save_for_backward(x2, weight, absmax)
        ctx.cfg = (mode, seed, offset)
        ctx.in_shape = x.shape
        return y.reshape(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, dy):
        x2, weight, absmax = ctx.saved_tensors
        N = weight.shape[0]
        dy2 = dy.reshape(-1, N)
        if not dy2.is_contiguous():
            dy2 = dy2.contiguous()
        mode, seed, offset = ctx.cfg
        cfg = b.linear_cfg(mode=mode, seed=seed, offset=offset)
        dx, dw = b.int8mp_linear_bwd_saved(dy2, x2, weight, absmax, cfg,
                                           want_dx=ctx.needs_input_grad[0],
                                           want_dw=ctx.needs_input_grad[1])
        if dx is not None:
            dx = dx.reshape(ctx.in_shape)
        return dx, dw, None, None, None


class Int8MixedPrecisionLinear(torch.nn.Module):
    """y = x @ weight.T with every matmul of forward and backward in INT8.

    stochastic: stochastic rounding for all six quantizations of a step
    (Philox4x32-10 keyed by `seed`); every call advances the element offset
    by 2^32 so that successive calls draw new numbers.  Nearest-even
    rounding otherwise.
    """

    OFFSET_STEP = 1 << 32

    def __init__(self, in_features, out_features, device=None, stochastic=False, seed=0):
        super().__init__()
        self.in_features = in_features
        self.out_features = out_features
        self.weight = torch.nn.Parameter(
            torch.empty((out_features, in_features), dtype=torch.bfloat16, device=device))
        torch.nn.init.normal_(self.weight, std=0.02)
        self.mode = b.INT8MP_SR if stochastic else b.INT8MP_RNE
        self.seed = int(seed)
        self.offset = 0

    def forward(self, x):
        offset = self.offset
        if self.mode == b.INT8MP_SR:
            self.offset += self.OFFSET_STEP
        return Int8MixedPrecisionLinearFunction.apply(x, self.weight, self.mode, self.seed, offset)

    def extra_repr(self):
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"{'stochastic' if self.mode == b.INT8MP_SR else 'nearest-even'} rounding")
