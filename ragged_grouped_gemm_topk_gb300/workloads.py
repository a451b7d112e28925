"""Seeded synthetic MoE-layer workloads.

This module only draws inputs: shapes, value distributions and seeds.  It holds
none of the layer's arithmetic (no routing, permutation, quantisation, GEMM or
combine), so the CUDA path and the CPU oracle can both be fed from it without
sharing any of the method.

The five layer shapes follow the models the NVIDIA blog "Accelerating Dropless
MoE Training in JAX with NVIDIA Transformer Engine" names (DeepSeek, Qwen,
Mixtral; first section): a tiny fp32 layer, a Mixtral-shaped layer, a
Qwen3-235B-shaped layer and two DeepSeek-V3-shaped layers.  The pages train on
real data; here every tensor is synthetic and seeded.

A sixth entry, the MXFP8 training step, is the DeepSeek-V3-shaped training
layer again with every GEMM on MXFP8 operands: it reuses that layer's seed, so
both see the same routing, activations, weights and upstream gradient.  A
seventh, the NVFP4 layer, is the DeepSeek-V3-shaped MXFP8 layer's forward with
NVFP4 operands, on that layer's seed and inputs.

Recipe (per workload, seed ``s`` = its position in ``WORKLOADS``, shared by the
MXFP8 training step with the bf16 one):

* router logits ``z + b`` with ``z ~ N(0,1)`` of shape [T, E] and a
  per-expert bias ``b`` (zero, Gaussian, or the log of a Zipf pmf over a seeded
  permutation of expert ranks, which gives the skewed, data-dependent expert
  loads of the blog's "ragged tensor" figure).  Logits are always fp32.
* activations ``x ~ N(0,1)`` (the tiny layer scales by 1/sqrt(d)), expert
  weights ``W1 ~ N(0,1)/sqrt(d)`` with shape [E, 2f, d] (gate rows then up
  rows, each row contiguous over d) and ``W2 ~ N(0,1)/sqrt(f)`` with shape
  [E, d, f]; the upstream gradient ``dy ~ N(0,1)`` of shape [T, d].
* small tensors come from ``numpy.random.default_rng(s)``; large tensors from a
  ``torch.Generator`` on the target device seeded ``1000*s + id``.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    d: int          # model dim
    E: int          # routed experts
    k: int          # experts per token
    f: int          # expert FFN hidden dim (SwiGLU: W1 has 2f rows)
    dtype: str      # "f32", "bf16", "mxfp8" or "nvfp4" (bf16 storage, block-scaled GEMM operands)
    bias: str       # "none", "gauss" or "zipf"
    bias_param: float
    seed: int
    backward: bool = False
    renormalize: bool = True

    @property
    def M(self) -> int:
        """Permuted rows: exactly T*k (dropless, nothing dropped or padded)."""
        return self.T * self.k

    @property
    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs of the two grouped GEMMs: 2*M*d*2f + 2*M*f*d."""
        return 6.0 * self.M * self.d * self.f

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, T: int | None = None, E: int | None = None, k: int | None = None,
               d: int | None = None, f: int | None = None, name: str | None = None) -> "Workload":
        """A smaller copy with the same distributions (for parity at oracle-friendly sizes)."""
        return dataclasses.replace(
            self, T=T or self.T, E=E or self.E, k=k or self.k, d=d or self.d, f=f or self.f,
            name=name or (self.name + "-scaled"))


WORKLOADS = [
    Workload("tiny-fp32", 256, 256, 8, 2, 512, "f32", "none", 0.0, 0),
    Workload("mixtral-bf16", 4096, 4096, 8, 2, 14336, "bf16", "gauss", 0.5, 1),
    Workload("qwen3-235b-bf16", 8192, 4096, 128, 8, 1536, "bf16", "zipf", 1.1, 2),
    Workload("dsv3-mxfp8", 8192, 7168, 256, 8, 2048, "mxfp8", "zipf", 1.3, 3),
    Workload("dsv3-bf16-train", 16384, 7168, 256, 8, 2048, "bf16", "zipf", 1.5, 4, backward=True),
    Workload("dsv3-mxfp8-train", 16384, 7168, 256, 8, 2048, "mxfp8", "zipf", 1.5, 4, backward=True),
    Workload("dsv3-nvfp4", 8192, 7168, 256, 8, 2048, "nvfp4", "zipf", 1.3, 3),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def expert_bias(w: Workload) -> np.ndarray:
    """Per-expert logit bias b[E] (float64), drawn from the workload's seed."""
    rng = np.random.default_rng(w.seed)
    if w.bias == "none":
        return np.zeros(w.E)
    if w.bias == "gauss":
        return rng.normal(0.0, w.bias_param, size=w.E)
    if w.bias == "zipf":
        ranks = rng.permutation(w.E) + 1                 # expert e has popularity rank ranks[e]
        pmf = ranks.astype(np.float64) ** (-w.bias_param)
        pmf /= pmf.sum()
        return np.log(pmf)
    raise ValueError(w.bias)


def make_logits(w: Workload) -> np.ndarray:
    """Router logits [T, E] float32: N(0,1) noise plus the expert bias."""
    b = expert_bias(w)
    rng = np.random.default_rng([w.seed, 1])
    z = rng.standard_normal((w.T, w.E))
    return (z + b[None, :]).astype(np.float32)


def _gen(w: Workload, device, tid: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 * w.seed + tid)
    return g


def _randn(shape, scale, dtype, device, gen):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    return t.to(dtype)


def make_x(w: Workload, device="cpu") -> torch.Tensor:
    scale = 1.0 / math.sqrt(w.d) if w.name == "tiny-fp32" else 1.0
    return _randn((w.T, w.d), scale, w.torch_dtype, device, _gen(w, device, 1))


def make_w1(w: Workload, device="cpu") -> torch.Tensor:
    """[E, 2f, d]: rows 0..f-1 are the gate projection, rows f..2f-1 the up projection."""
    return _randn((w.E, 2 * w.f, w.d), 1.0 / math.sqrt(w.d), w.torch_dtype, device, _gen(w, device, 2))


def make_w2(w: Workload, device="cpu") -> torch.Tensor:
    """[E, d, f]: the down projection, each output row contiguous over f."""
    return _randn((w.E, w.d, w.f), 1.0 / math.sqrt(w.f), w.torch_dtype, device, _gen(w, device, 3))


def make_dy(w: Workload, device="cpu") -> torch.Tensor:
    return _randn((w.T, w.d), 1.0, w.torch_dtype, device, _gen(w, device, 4))


def make_matrix(rows: int, cols: int, seed: int, dtype=torch.bfloat16, device="cpu",
                scale: float = 1.0) -> torch.Tensor:
    """A generic seeded N(0, scale^2) matrix (stand-alone quantiser / GEMM cases)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return _randn((rows, cols), scale, dtype, device, g)
