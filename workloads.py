"""Seeded synthetic inputs for the ZeRO-1 step: the five workloads.

This module holds none of the method's arithmetic.  It only draws inputs:
per-rank bf16 gradients and the initial fp32 master weights, with the shapes
and value distributions of each workload.  Both the CUDA path and the CPU
oracle consume the same drawn tensors (the tests copy device draws to the
host for the oracle).

Seeds: rank r's gradient at step t (1-based) comes from a torch generator
seeded with ``seed_base + 1000 * t + r``; the master weights from
``seed_base + 999_983``.  Draws are made on the target device in chunks of at
most 2**26 entries so that multi-billion-entry buffers need no large fp32
temporaries; the chunking is part of the recipe (same chunks, same values).

Workloads (parameters N, ranks W):
  tiny        N = 4096, W = 4, grads ~ N(0, 0.01^2), 10 steps, clip 1.0
  gpt2_small  the GPT-2-small parameter list flattened in order
              (50257x768 token embedding, 1024x768 positions, 12 x {768x2304
              qkv, 768x768 proj, 768x3072, 3072x768, 4 LayerNorm vectors of
              768}) = 124,355,328 parameters, W = 8, grads ~ N(0, 1e-3^2),
              20 steps
  ragged_1p3b N = 1,300,000,005 (not a multiple of W = 8), grads ~
              N(0, 1e-3^2) with 1% of entries (Bernoulli per rank and step)
              multiplied by 100 before the bf16 cast, 10 steps
  state_7b    N = 7,000,000,000, W = 2, grads ~ N(0, 1e-3^2), 5 steps
  stress_w64  N = 350,000,000, W = 64, grads ~ N(r * 1e-5, 1e-3^2) for rank
              r, clip 0.5, 5 steps
All: master ~ N(0, 0.02^2), m = v = 0, lr 1e-3, betas (0.9, 0.95), eps 1e-8,
weight decay 0.1.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

CHUNK = 1 << 26
MASTER_SEED = 999_983


def gpt2_small_shapes() -> list[tuple[int, ...]]:
    shapes: list[tuple[int, ...]] = [(50257, 768), (1024, 768)]
    for _ in range(12):
        shapes += [(768, 2304), (768, 768), (768, 3072), (3072, 768), (768,), (768,), (768,), (768,)]
    return shapes


def _numel(shape) -> int:
    out = 1
    for d in shape:
        out *= d
    return out


GPT2_SMALL_N = sum(_numel(s) for s in gpt2_small_shapes())


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    world: int
    sigma: float
    steps: int
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    rank_mean_step: float = 0.0
    master_sigma: float = 0.02
    seed_base: int = 0
    tensors: tuple = field(default=(), compare=False)

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, max_norm=self.max_norm)

    def with_n(self, n: int, name: str | None = None) -> "Workload":
        """The same recipe at another size (parity cases, bounded samples)."""
        return replace(self, n=n, name=name or f"{self.name}@{n}", tensors=())

    def bytes_per_step(self) -> int:
        """Algorithmic HBM bytes of one step: 2W (read grads) + 2W (write
        replicas) + 24 (read and write fp32 master, m, v) per parameter."""
        return (4 * self.world + 24) * self.n


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 4096, 4, 0.01, 10),
        Workload("gpt2_small", GPT2_SMALL_N, 8, 1e-3, 20, tensors=tuple(gpt2_small_shapes())),
        Workload("ragged_1p3b", 1_300_000_005, 8, 1e-3, 10, outlier_frac=0.01, outlier_scale=100.0),
        Workload("state_7b", 7_000_000_000, 2, 1e-3, 5),
        Workload("stress_w64", 350_000_000, 64, 1e-3, 5, max_norm=0.5, rank_mean_step=1e-5),
    ]
}


@dataclass(frozen=True)
class AllReduceWorkload:
    """An all-reduce of W emulated ranks' buffers of n elements each."""
    name: str
    n: int
    world: int
    dtype: torch.dtype
    average: bool


# The lecture's benchmark (1e8 fp32 elements, world size 4, sum) and the DDP
# gradient all-reduce of the GPT-2-small list (bf16, W = 8, mean).
ALLREDUCE_WORKLOADS = {
    w.name: w for w in [
        AllReduceWorkload("lecture_fp32_w4", 100_000_000, 4, torch.float32, False),
        AllReduceWorkload("ddp_gpt2_small_bf16_w8", GPT2_SMALL_N, 8, torch.bfloat16, True),
    ]
}


def allreduce_inputs(w: AllReduceWorkload, device) -> list[torch.Tensor]:
    """Rank r's buffer ~ N(0, 1) from seed 5000 + r, cast to the element type."""
    out = []
    for r in range(w.world):
        g = _gen(5000 + r, device)
        t = torch.empty(w.n, dtype=w.dtype, device=device)
        for lo in range(0, w.n, CHUNK):
            hi = min(lo + CHUNK, w.n)
            t[lo:hi].copy_(torch.randn(hi - lo, generator=g, device=device))
        out.append(t)
    return out


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def fill_grad(out: torch.Tensor, w: Workload, step: int, rank: int) -> torch.Tensor:
    """Draw rank `rank`'s bf16 gradient for step `step` into `out` (1-D bf16)."""
    assert out.dtype == torch.bfloat16 and out.dim() == 1
    g = _gen(w.seed_base + 1000 * step + rank, out.device)
    mean = rank * w.rank_mean_step
    for lo in range(0, out.numel(), CHUNK):
        hi = min(lo + CHUNK, out.numel())
        x = torch.randn(hi - lo, generator=g, device=out.device, dtype=torch.float32)
        x.mul_(w.sigma)
        if mean:
            x.add_(mean)
        if w.outlier_frac > 0:
            hit = torch.rand(hi - lo, generator=g, device=out.device) < w.outlier_frac
            x[hit] *= w.outlier_scale
        out[lo:hi].copy_(x)
        del x
    return out


def grads(w: Workload, step: int, device, out: list[torch.Tensor] | None = None) -> list[torch.Tensor]:
    """All W ranks' gradients for one step (allocated unless `out` is given)."""
    if out is None:
        out = [torch.empty(w.n, dtype=torch.bfloat16, device=device) for _ in range(w.world)]
    for r, t in enumerate(out):
        fill_grad(t, w, step, r)
    return out


def master(w: Workload, device, out: torch.Tensor | None = None) -> torch.Tensor:
    """Initial fp32 master weights ~ N(0, master_sigma^2)."""
    if out is None:
        out = torch.empty(w.n, dtype=torch.float32, device=device)
    g = _gen(w.seed_base + MASTER_SEED, out.device)
    for lo in range(0, out.numel(), CHUNK):
        hi = min(lo + CHUNK, out.numel())
        out[lo:hi].normal_(0.0, w.master_sigma, generator=g)
    return out
