"""Seeded synthetic bf16 inputs shaped like the pages' workloads.

Shared by the tests (oracle and CUDA sides read the same bf16 bits) and the
benchmark.  Holds no arithmetic of the method: it only draws numbers.

Recipe: a CPU torch.Generator seeded with `seed` draws fp32 N(0, 1) values,
which are multiplied by `std`; optionally a Bernoulli(p) mask drawn from a
second generator seeded 1000 + seed multiplies the selected entries by
`outlier_scale`; the result is cast to bf16 (round to nearest even).
"""
import torch


def bf16_normal(shape, seed, std=1.0, outlier_frac=0.0, outlier_scale=1.0):
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outlier_frac > 0.0:
        gm = torch.Generator().manual_seed(1000 + int(seed))
        mask = torch.rand(tuple(shape), generator=gm) < outlier_frac
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def single_matmul_inputs():
    """X [256,512] and W [256,512], N(0,1), both from one generator seeded 0,
    X drawn first."""
    g = torch.Generator().manual_seed(0)
    X = torch.randn((256, 512), generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = torch.randn((256, 512), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return X, W


def square_inputs(S, layout):
    """A and B of the square sweep, N(0,1) with 1% of entries x20, stored as
    the layout needs: A@B.T -> A [S,S] (M,K), B [S,S] (N,K); A@B -> B is
    (K,N); A.T@B -> A is (K,M), B is (K,N).  Square, so only the meaning of
    the axes changes.  A from seed 0, B from seed 1."""
    A = bf16_normal((S, S), 0, outlier_frac=0.01, outlier_scale=20.0)
    B = bf16_normal((S, S), 1, outlier_frac=0.01, outlier_scale=20.0)
    return A, B


# (name, N = out_features, K = in_features, activation that feeds it)
LLAMA2_1B = {
    "name": "llama2-1b", "T": 16 * 2048, "hidden": 2048, "inter": 5632,
    "linears": [("q", 2048, 2048, "attn"), ("k", 2048, 2048, "attn"), ("v", 2048, 2048, "attn"),
                ("o", 2048, 2048, "o"), ("gate", 5632, 2048, "mlp"), ("up", 5632, 2048, "mlp"),
                ("down", 2048, 5632, "down")],
    "x_outliers": (0.0, 1.0),
}
LLAMA3_8B = {
    "name": "llama3-8b", "T": 16384, "hidden": 4096, "inter": 14336,
    "linears": [("q", 4096, 4096, "attn"), ("k", 1024, 4096, "attn"), ("v", 1024, 4096, "attn"),
                ("o", 4096, 4096, "o"), ("gate", 14336, 4096, "mlp"), ("up", 14336, 4096, "mlp"),
                ("down", 4096, 14336, "down")],
    "x_outliers": (0.005, 30.0),
}
ACT_SEEDS = {"attn": 10, "o": 11, "mlp": 12, "down": 13}


def layer_shapes(spec):
    return [(name, N, K) for name, N, K, _ in spec["linears"]]


def linear_inputs(spec, name, T=None):
    """(X [T,K], W [N,K], dY [T,N]) of one linear of the layer, drawn exactly
    as layer_inputs draws it."""
    T = spec["T"] if T is None else T
    frac, scale = spec["x_outliers"]
    for i, (lname, N, K, act) in enumerate(spec["linears"]):
        if lname == name:
            X = bf16_normal((T, K), ACT_SEEDS[act], outlier_frac=frac, outlier_scale=scale)
            W = bf16_normal((N, K), 20 + i, std=0.02)
            dY = bf16_normal((T, N), 30 + i, std=1e-3)
            return X, W, dY
    raise KeyError(name)


def layer_inputs(spec, T=None):
    """Activations (shared where the decoder layer shares them), weights and
    output gradients of one decoder layer's linears:
      activations N(0,1) (+ the spec's outliers), seeds 10..13
      weights     N(0, 0.02), seed 20 + i
      grad_out    N(0, 1e-3), seed 30 + i
    Returns dict name -> (X [T,K], W [N,K], dY [T,N])."""
    T = spec["T"] if T is None else T
    frac, scale = spec["x_outliers"]
    acts = {}
    out = {}
    for i, (name, N, K, act) in enumerate(spec["linears"]):
        if act not in acts:
            acts[act] = bf16_normal((T, K), ACT_SEEDS[act], outlier_frac=frac, outlier_scale=scale)
        W = bf16_normal((N, K), 20 + i, std=0.02)
        dY = bf16_normal((T, N), 30 + i, std=1e-3)
        out[name] = (acts[act], W, dY)
    return out
