"""The linear layers of a Llama decoder layer in INT8 mixed precision.

"Integrate INT8 mixed-precision from torchao 0.7", discussion: the method
swaps the model's linear layers (module swap) for ones whose three matmuls
run in INT8, and leaves everything else in BF16.  torchao issue 1887 applies
it to a model with `quantize_(model, int8_mixed_precision_training(),
filter_fn)`.  The "Quantized model training" README times it on Llama2-1B
(LM head excluded).

Int8MixedPrecisionDecoderLinears holds the seven linears of one decoder
layer -- q, k, v, o (hidden x hidden) and gate, up (intermediate x hidden),
down (hidden x intermediate) -- each an Int8MixedPrecisionLinear, joined
the way a Llama decoder layer joins them:

    q, k, v = Lq(x), Lk(x), Lv(x)
    a       = attn(q, k, v)          (stand-in, see below)
    h       = x + Lo(a)
    z       = silu(Lg(h)) * Lu(h)     (SwiGLU)
    y       = h + Ld(z)

The attention core (softmax over the sequence) and the RMSNorms are not part
of the method and are left out: `attn` is the per-token, per-channel
stand-in a = v + q * k, which keeps q and k in the gradient path.  Every
elementwise step and every fan-out (x into q/k/v and the residual, h into
gate/up and the residual) is computed in `glue_dtype` and rounded to bf16
where a linear reads it; with float64 the gradients that autograd sums at a
fan-out are sums of bf16 values and so exact in any order, which makes the
whole layer reproducible by an independent CPU composition bit for bit.
"""
import torch

from .autograd import Int8MixedPrecisionLinear


class Int8MixedPrecisionDecoderLinears(torch.nn.Module):
    NAMES = ("q", "k", "v", "o", "gate", "up", "down")

    def __init__(self, hidden, intermediate, device=None, stochastic=False, seed=0,
                 glue_dtype=torch.float32):
        super().__init__()
        self.hidden = hidden
        self.intermediate = intermediate
        self.glue_dtype = glue_dtype
        shapes = {"q": (hidden, hidden), "k": (hidden, hidden), "v": (hidden, hidden),
                  "o": (hidden, hidden), "gate": (hidden, intermediate),
                  "up": (hidden, intermediate), "down": (intermediate, hidden)}
        for i, name in enumerate(self.NAMES):
            fin, fout = shapes[name]
            # each linear draws its own stochastic-rounding numbers (seed + i)
            setattr(self, name, Int8MixedPrecisionLinear(fin, fout, device=device,
                                                         stochastic=stochastic, seed=seed + i))

    def linears(self):
        return [(name, getattr(self, name)) for name in self.NAMES]

    def forward(self, x):
        G, bf = self.glue_dtype, torch.bfloat16
        xg = x.to(G)
        q = self.q(xg.to(bf))
        k = self.k(xg.to(bf))
        v = self.v(xg.to(bf))
        a = (v.to(G) + q.to(G) * k.to(G)).to(bf)
        h = xg + self.o(a).to(G)
        g = self.gate(h.to(bf)).to(G)
        u = self.up(h.to(bf)).to(G)
        z = (g * torch.sigmoid(g) * u).to(bf)
        return (h + self.down(z).to(G)).to(bf)

    def extra_repr(self):
        return f"hidden={self.hidden}, intermediate={self.intermediate}, glue={self.glue_dtype}"

