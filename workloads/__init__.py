"""Seeded synthetic inputs for the MXFP8 MoE hot path.

This module is shared by the CUDA path, the CPU oracle, the tests and the
bench.  It draws random numbers and rounds them to the storage dtype of each
input (bf16 by round-to-nearest-even through torch), and nothing else: it holds
none of the method's arithmetic (no quantization, routing, permutation, GEMM or
SwiGLU).

Workloads (shapes and distributions of the MoE training step that the
"1.5x faster MoE training on Blackwell with MXFP8 kernels built from scratch"
article and the pytorch/ao "mxfp8 moe training" PR stack describe; the pages
print no shapes, so every size below is a stated synthetic choice):

* ``tiny_layer``      T=512, H=256, E=4, F=512, top-1 ids uniform, gate 1.
* ``quantize``        bf16 [16384, 7168] N(0,1), 1% of entries x100, two exact
                      zeros in every 32-element row block.
* ``permute``         T=32768, H=5120, E=16, k=4, Zipf(1.1) expert choice over
                      14 live experts (two experts empty).
* ``grouped_gemm``    E=8, 32768 routed rows in Zipf-skewed groups that are
                      multiples of 128 (one empty), K=7168, N=2048.
* ``full_layer``      T=16384, H=5120, E=16, F=8192, top-1 router with softmax
                      gate on N(0,1) logits.

Every generator takes a ``seed`` and a torch ``device``; the same seed and
device give the same tensors.  Tensors come back as torch tensors (bf16 data
as ``torch.bfloat16``, ids as int32, logits/gates as float32).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "LayerDims",
    "TINY_LAYER",
    "FULL_LAYER",
    "QUANTIZE_SHAPE",
    "PERMUTE_DIMS",
    "GEMM_DIMS",
    "generator",
    "randn_bf16",
    "quantize_input",
    "zipf_topk_ids",
    "uniform_ids",
    "gemm_group_sizes",
    "layer_inputs",
    "gemm_inputs",
    "permute_inputs",
    "bf16_bits",
]


@dataclass(frozen=True)
class LayerDims:
    T: int   # tokens
    H: int   # hidden size
    E: int   # experts
    F: int   # FFN width of one expert (SwiGLU: W1, W3 are H x F, W2 is F x H)
    k: int   # experts per token


TINY_LAYER = LayerDims(T=512, H=256, E=4, F=512, k=1)
FULL_LAYER = LayerDims(T=16384, H=5120, E=16, F=8192, k=1)
QUANTIZE_SHAPE = (16384, 7168)
PERMUTE_DIMS = dict(T=32768, H=5120, E=16, k=4)
GEMM_DIMS = dict(E=8, M=32768, K=7168, N=2048)


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, then rounded to bf16 (RNE)."""
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """The raw uint16 bit patterns of a bf16 tensor, as a numpy array."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def quantize_input(rows: int, cols: int, seed: int = 0, device="cpu",
                   outlier_p: float = 0.01, outlier_mul: float = 100.0,
                   zeros_per_block: int = 2) -> torch.Tensor:
    """bf16 [rows, cols]: N(0,1); a Bernoulli(outlier_p) mask of entries is
    multiplied by ``outlier_mul``; in every 32-element row block
    ``zeros_per_block`` distinct seeded positions are set to +0.0."""
    assert cols % 32 == 0
    g = generator(seed, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    mask = torch.rand((rows, cols), generator=g, device=device) < outlier_p
    x = torch.where(mask, x * outlier_mul, x)
    if zeros_per_block:
        nb = rows * (cols // 32)
        # distinct positions per block: the first `zeros_per_block` entries of a
        # random permutation of 0..31, via argsort of uniform keys
        keys = torch.rand((nb, 32), generator=g, device=device)
        pos = keys.argsort(dim=1)[:, :zeros_per_block]
        xb = x.view(nb, 32)
        xb.scatter_(1, pos, 0.0)
    return x.to(torch.bfloat16)


def uniform_ids(T: int, E: int, k: int, g: torch.Generator, device) -> torch.Tensor:
    """k distinct expert ids per token, uniform over E (k=1: plain uniform)."""
    if k == 1:
        return torch.randint(0, E, (T, 1), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    keys = torch.rand((T, E), generator=g, device=device)
    return keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def zipf_topk_ids(T: int, E: int, k: int, live: int, alpha: float,
                  g: torch.Generator, device) -> torch.Tensor:
    """k distinct experts per token, drawn without replacement from a Zipf(alpha)
    distribution over ``live`` experts (rank r has p_r ~ r^-alpha); a seeded
    permutation maps ranks to expert ids, and the E - live experts left over
    get p = 0 (they stay empty).  Sampling without replacement uses the
    Gumbel-top-k construction on log p."""
    assert k <= live <= E
    ranks = torch.arange(1, live + 1, dtype=torch.float64)
    p = ranks.pow(-alpha)
    p = p / p.sum()
    perm = torch.randperm(E, generator=g, device=device).cpu()
    logp = torch.full((E,), -math.inf, dtype=torch.float64)
    logp[perm[:live]] = p.log()
    u = torch.rand((T, E), generator=g, device=device, dtype=torch.float64)
    gumbel = -torch.log(-torch.log(u.clamp_min(1e-300)))
    score = logp.to(device).unsqueeze(0) + gumbel
    return score.topk(k, dim=1).indices.to(torch.int32).contiguous()


def gemm_group_sizes(E: int = 8, M: int = 32768, alpha: float = 1.1, unit: int = 128,
                     seed: int = 0) -> list[int]:
    """Zipf-skewed group sizes in units of ``unit`` rows with one empty group.
    Rank r of the E-1 live ranks gets floor((M/unit) * p_r) * unit rows with
    p_r ~ r^-alpha, the remainder goes to rank 1, and a seeded permutation maps
    ranks to expert ids (the last rank is the empty expert)."""
    live = E - 1
    w = [r ** -alpha for r in range(1, live + 1)]
    s = sum(w)
    units = M // unit
    sizes = [math.floor(units * wi / s) * unit for wi in w]
    sizes[0] += M - sum(sizes)
    sizes.append(0)
    g = torch.Generator().manual_seed(int(seed))
    perm = torch.randperm(E, generator=g).tolist()
    out = [0] * E
    for rank, e in enumerate(perm):
        out[e] = sizes[rank]
    return out


def layer_inputs(d: LayerDims, seed: int = 0, device="cpu", router: str = "uniform"):
    """Inputs of one MoE SwiGLU layer step.

    router="uniform": ids uniform over experts (k distinct), gate = 1.
    router="logits":  logits [T, E] ~ N(0,1) fp32 are returned and ids/gate are
                      left for the router to compute.
    Weights: W1, W3 [E, H, F] and W2 [E, F, H], N(0, 0.02^2) bf16; x, dOut
    [T, H] N(0,1) bf16."""
    g = generator(seed, device)
    out = {}
    if router == "uniform":
        out["ids"] = uniform_ids(d.T, d.E, d.k, g, device)
        out["gate"] = torch.ones((d.T, d.k), dtype=torch.float32, device=device)
        out["logits"] = None
    elif router == "logits":
        out["logits"] = torch.randn((d.T, d.E), generator=g, device=device, dtype=torch.float32)
        out["ids"] = None
        out["gate"] = None
    else:
        raise ValueError(router)
    out["x"] = randn_bf16((d.T, d.H), 1.0, g, device)
    out["W1"] = randn_bf16((d.E, d.H, d.F), 0.02, g, device)
    out["W3"] = randn_bf16((d.E, d.H, d.F), 0.02, g, device)
    out["W2"] = randn_bf16((d.E, d.F, d.H), 0.02, g, device)
    out["dOut"] = randn_bf16((d.T, d.H), 1.0, g, device)
    return out


def gemm_inputs(E: int, M: int, K: int, N: int, sizes: list[int], seed: int = 0, device="cpu"):
    """Grouped-GEMM operands: A [M, K] N(0,1), W [E, K, N] N(0, 0.02^2),
    dC [M, N] N(0,1), all bf16; ``sizes`` rows per expert (sum = M)."""
    assert sum(sizes) == M and len(sizes) == E
    g = generator(seed, device)
    return {
        "A": randn_bf16((M, K), 1.0, g, device),
        "W": randn_bf16((E, K, N), 0.02, g, device),
        "dC": randn_bf16((M, N), 1.0, g, device),
        "sizes": list(sizes),
    }


def permute_inputs(T: int, H: int, E: int, k: int, seed: int = 0, device="cpu",
                   live: int | None = None, alpha: float = 1.1):
    """Token permute inputs: x [T, H] N(0,1) bf16, Zipf top-k ids, gates U(0,1)
    (fp32, used by the unpermute combine) and y rows for the combine."""
    g = generator(seed, device)
    live = E - 2 if live is None else live
    ids = zipf_topk_ids(T, E, k, live, alpha, g, device)
    x = randn_bf16((T, H), 1.0, g, device)
    gate = torch.rand((T, k), generator=g, device=device, dtype=torch.float32)
    return {"x": x, "ids": ids, "gate": gate}
