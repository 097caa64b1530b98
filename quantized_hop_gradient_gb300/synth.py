"""Seeded synthetic gradients for the DynamiQ all-reduce workloads.

This module holds no step of the method: it only draws the inputs (bf16
gradients of N simulated workers) that both the CUDA path and the oracle are
fed.  Draws use torch's generator on the requested device, so one seed gives
one buffer per device type; every comparison feeds the SAME buffer to both
sides.

The pages evaluate on real LLM fine-tuning gradients (BERT-large, Gemma 1B,
LLaMA 1B; scribe notes "Evaluation").  These synthetic workloads stand in for
them with the parameter counts of those models and heavy-tailed, layer-scaled
value distributions:

* per-super-group or per-layer scales are shared by all workers (the workers
  see the same distribution), entries are independent per worker;
* "N(0, v)" means variance v;
* layer blocks are the J super-groups split into L equal contiguous runs;
* Student-t(nu) is Z / sqrt(chi2_nu / nu) with chi2_nu a sum of nu squared
  normals;
* the coordinate count is padded with zeros to a multiple of 256.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

SG = 256


@dataclass(frozen=True)
class Workload:
    name: str
    n_ranks: int
    topology: str            # "ring" or "butterfly"
    n: int                   # coordinates per worker before padding
    budget: float = 5.0
    correlated: bool = True
    dist: str = "layer_gauss"
    layers: int = 1
    sigma: float = 1.0       # std of the log-scale
    nu: int = 3
    bucket: int = 0          # coords per bucket (0: one all-reduce over everything)
    budgets: tuple = field(default=())

    @property
    def n_pad(self) -> int:
        return (self.n + SG - 1) // SG * SG

    @property
    def n_sg(self) -> int:
        return self.n_pad // SG

    def scaled(self, n: int, **kw) -> "Workload":
        """Same distribution with ``n`` coordinates per worker (for tests)."""
        return replace(self, n=n, bucket=0, **kw)


WORKLOADS = {
    # 4 workers, ring, 1 Mi coords: per-super-group lognormal(0,1) scale,
    # N(0, scale^2) entries, 0.1% outliers at 20x scale.
    "ring4_1m": Workload("ring4_1m", 4, "ring", 1_048_576, dist="sg_lognormal_outliers"),
    # BERT-large-sized gradient, 8 workers, ring, 24 layers, log-scale std 1.5.
    "bert_large_ring8": Workload("bert_large_ring8", 8, "ring", 335_141_888,
                                 dist="layer_gauss", layers=24, sigma=1.5),
    # LLaMA-1B-sized gradient, 8 workers, butterfly, Student-t(3) x layer scale.
    "llama1b_butterfly8": Workload("llama1b_butterfly8", 8, "butterfly", 1_235_814_400,
                                   dist="layer_student", layers=16, sigma=1.0, nu=3),
    # Gemma-1B-sized gradient, 16 workers, ring, two-component super-group
    # mixture with a non-zero super-group mean; budget sweep 4/5/6.
    "gemma1b_ring16": Workload("gemma1b_ring16", 16, "ring", 999_885_952, dist="mixture",
                               budgets=(4.0, 5.0, 6.0)),
    # Llama-3-8B-sized gradient, 8 workers, ring, streamed as 25 MB buckets.
    "llama3_8b_ring8_buckets": Workload("llama3_8b_ring8_buckets", 8, "ring", 8_030_261_248,
                                        dist="layer_student", layers=32, sigma=1.0, nu=4,
                                        bucket=13_107_200),
}


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _rand(shape, gen, device):
    return torch.rand(shape, generator=gen, device=device, dtype=torch.float32)


def _sg_scales(w: Workload, gen, device, J: int, sg0: int = 0, J_total: int = 0):
    """Per-super-group scale (shared by all workers) and optional mean."""
    J_total = J_total or J
    mean = None
    if w.dist == "sg_lognormal_outliers":
        scale = torch.exp(w.sigma * _randn(J, gen, device))
    elif w.dist in ("layer_gauss", "layer_student"):
        layer_scale = torch.exp(w.sigma * _randn(w.layers, gen, device))
        j = torch.arange(sg0, sg0 + J, device=device, dtype=torch.int64)
        layer = torch.clamp(j * w.layers // J_total, max=w.layers - 1)
        scale = layer_scale[layer]
    elif w.dist == "mixture":
        wide = _rand(J, gen, device) < 0.2
        scale = torch.where(wide, torch.full((J,), 0.1, device=device),
                            torch.full((J,), 0.01, device=device))
        mean = math.sqrt(1e-3) * _randn(J, gen, device)
    else:
        raise ValueError(f"unknown distribution {w.dist}")
    return scale, mean


def _entries(w: Workload, gen, device, scale, mean, n_sg: int):
    """One worker's fp32 entries for n_sg super-groups."""
    n = n_sg * SG
    z = _randn(n, gen, device)
    if w.dist == "layer_student":
        chi2 = torch.zeros(n, device=device)
        for _ in range(w.nu):
            chi2 += _randn(n, gen, device) ** 2
        z = z / torch.sqrt(chi2 / w.nu)
    x = z.view(n_sg, SG) * scale.view(n_sg, 1)
    if w.dist == "sg_lognormal_outliers":
        hit = _rand(n, gen, device).view(n_sg, SG) < 1e-3
        big = _randn(n, gen, device).view(n_sg, SG) * (20.0 * scale.view(n_sg, 1))
        x = torch.where(hit, big, x)
    if mean is not None:
        x = x + mean.view(n_sg, 1)
    return x.reshape(-1)


def generate(w: Workload, device="cpu", seed: int = 0, ranks=None, slice_sg: int = 1 << 18,
             sg0: int = 0, n_sg: int = 0, n_valid: int = 0, J_total: int = 0):
    """bf16 gradients (one 1-D tensor of n_pad coords per worker in ``ranks``).

    Draws the shared scales, then each worker's entries in slices of
    ``slice_sg`` super-groups (bounded temporary memory).  The coordinates
    past ``w.n`` are zero.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    J = n_sg or w.n_sg
    n_valid = n_valid or w.n
    scale, mean = _sg_scales(w, gen, device, J, sg0, J_total)
    ranks = range(w.n_ranks) if ranks is None else ranks
    out = []
    for r in range(w.n_ranks):
        keep = r in ranks
        g = torch.empty(J * SG, dtype=torch.bfloat16, device=device) if keep else None
        for a in range(0, J, slice_sg):
            b = min(J, a + slice_sg)
            x = _entries(w, gen, device, scale[a:b], None if mean is None else mean[a:b], b - a)
            if keep:
                g[a * SG:b * SG] = x.to(torch.bfloat16)
        if keep:
            if n_valid < J * SG:
                g[n_valid:] = 0
            out.append(g)
    return out


def bucket_count(w: Workload) -> int:
    return (w.n + w.bucket - 1) // w.bucket


def generate_bucket(w: Workload, k: int, device="cpu", seed: int = 0):
    """Gradients of bucket k of a streamed workload (drawn on the fly)."""
    lo = k * w.bucket
    hi = min(w.n, lo + w.bucket)
    n_sg = (hi - lo + SG - 1) // SG
    J_total = (w.n + SG - 1) // SG
    return generate(w, device, seed=seed * 1_000_003 + k, sg0=lo // SG, n_sg=n_sg,
                    n_valid=hi - lo, J_total=J_total)


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
