"""Accuracy studies of the GPU path: ablations, rank scaling and the MXFP8
comparison, measured as vNMSE on the synthetic workloads.

vNMSE = ||out - s||^2 / ||s||^2 with s the exact sum of the workers' bf16
gradients (the pages' compression-error measure; scribe notes
"Evaluation").  Every all-reduce runs through the C ABI (DynamiQAllReduce,
MXFP8AllReduce); torch only draws the inputs and reduces the error in fp64.

    python -m quantized_hop_gradient_gb300.study ablations [--coords N] [--rounds R]
    python -m quantized_hop_gradient_gb300.study scaling   [--coords N] [--rounds R]
    python -m quantized_hop_gradient_gb300.study all --json out.json

Ablations [scribe notes "Key idea and contribution": the techniques; review
minor comment 1: variable vs uniform bitwidth]: the method as published
(budget 5), uniform levels (eps = inf), independent rounding, fp32 group
scales, variable vs fixed 4-bit allocation at 4 bits, and MXFP8.
Scaling [review: evaluation up to 64 workers; "If this is right": the
butterfly's O(n^2) against the ring's O(n^3) error bounds]: N = 4 .. 64,
ring and butterfly, DynamiQ at budget 5 and MXFP8.
"""
from __future__ import annotations

import argparse
import json
import math
import time

import torch

from . import synth
from .allreduce import DynamiQAllReduce, MXFP8AllReduce


def exact_sum(grads) -> torch.Tensor:
    """fp64 sum of bf16 gradients (bf16 -> fp64 is exact; the sum is exact
    while a coordinate's addends span fewer than 2^45 in magnitude)."""
    s = torch.zeros(grads[0].numel(), dtype=torch.float64, device=grads[0].device)
    for g in grads:
        s += g.double()
    return s


def vnmse(out: torch.Tensor, s: torch.Tensor) -> float:
    d = out.double() - s
    den = float(torch.dot(s, s))
    num = float(torch.dot(d, d))
    return num / den if den > 0 else num


def _dynamiq(grads, N, butterfly, rounds, **kw):
    J = grads[0].numel() // synth.SG
    ar = DynamiQAllReduce(N, J, butterfly=butterfly, seed=0, **kw)
    outs = ar.new_outputs()
    s = exact_sum(grads)
    for r in range(2):                          # warm-up (workspace, tables, clocks); not timed
        ar(grads, round=rounds + r, outs=outs)
    torch.cuda.synchronize()
    t0 = time.perf_counter()                    # wall clock: includes the plan's host sync
    for r in range(rounds):
        ar(grads, round=r, outs=outs)
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / rounds
    vs = []
    for r in range(rounds):
        ar(grads, round=r, outs=outs)
        vs.append(vnmse(outs[0], s))
    return sum(vs) / len(vs), sec, ar.info


def _mxfp8(grads, N, butterfly):
    mx = MXFP8AllReduce(N, grads[0].numel(), butterfly=butterfly)
    outs = mx(grads)
    return vnmse(outs[0], exact_sum(grads))


def _grads(name: str, coords: int, N: int = 0, seed: int = 0):
    w = synth.WORKLOADS[name]
    if coords:
        w = w.scaled(coords)
    if N:
        w = w.__class__(**{**w.__dict__, "n_ranks": N})
    return w, synth.generate(w, "cuda", seed=seed)


ABLATION_WORKLOADS = [("ring4_1m", False), ("bert_large_ring8", False), ("llama1b_butterfly8", True),
                      ("gemma1b_ring16", False)]


def ablations(coords: int = 1 << 24, rounds: int = 3):
    rows = []
    for name, butterfly in ABLATION_WORKLOADS:
        w, grads = _grads(name, min(coords, synth.WORKLOADS[name].n) if coords else 0)
        N = w.n_ranks
        res = {"workload": name, "n_ranks": N, "topology": "butterfly" if butterfly else "ring",
               "coords_per_worker": w.n_pad}
        for label, kw in [("dynamiq_b5", dict(budget=5.0)),
                          ("uniform_levels_b5", dict(budget=5.0, eps=math.inf)),
                          ("independent_rounding_b5", dict(budget=5.0, correlated=False)),
                          ("fp32_scales_b5", dict(budget=5.0, scale_fp32=True)),
                          ("dynamiq_b4", dict(budget=4.0)),
                          ("fixed4", dict(budget=4.0, fixed_bits=4))]:
            v, _, _ = _dynamiq(grads, N, butterfly, rounds, **kw)
            res[label] = v
        res["mxfp8"] = _mxfp8(grads, N, butterfly)
        res["mxfp8_over_dynamiq_b5"] = res["mxfp8"] / res["dynamiq_b5"]
        rows.append(res)
        del grads
        torch.cuda.empty_cache()
    return rows


def scaling(coords: int = 1 << 22, rounds: int = 3, ranks=(4, 8, 16, 32, 64), name: str = "llama1b_butterfly8"):
    rows = []
    for N in ranks:
        w, grads = _grads(name, coords, N=N, seed=N)
        for butterfly in (False, True):
            v, sec, _ = _dynamiq(grads, N, butterfly, rounds, budget=5.0)
            rows.append({"workload": name, "n_ranks": N, "topology": "butterfly" if butterfly else "ring",
                         "coords_per_worker": w.n_pad, "dynamiq_b5": v, "mxfp8": _mxfp8(grads, N, butterfly),
                         "ms_per_allreduce": sec * 1e3})
        del grads
        torch.cuda.empty_cache()
    return rows


def _table(rows, keys):
    out = [" | ".join(keys)]
    for r in rows:
        out.append(" | ".join(f"{r[k]:.3e}" if isinstance(r[k], float) else str(r[k]) for k in keys))
    return "\n".join(out)


def main(argv=None):
    p = argparse.ArgumentParser(description="vNMSE studies of the GPU path")
    p.add_argument("study", choices=["ablations", "scaling", "all"])
    p.add_argument("--coords", type=int, default=0, help="coordinates per worker (0: the study's default)")
    p.add_argument("--rounds", type=int, default=3)
    p.add_argument("--json", default="")
    a = p.parse_args(argv)
    res = {}
    if a.study in ("ablations", "all"):
        res["ablations"] = ablations(a.coords or (1 << 24), a.rounds)
        print(_table(res["ablations"], ["workload", "n_ranks", "topology", "dynamiq_b5", "uniform_levels_b5",
                                        "independent_rounding_b5", "fp32_scales_b5", "dynamiq_b4", "fixed4",
                                        "mxfp8", "mxfp8_over_dynamiq_b5"]))
    if a.study in ("scaling", "all"):
        res["scaling"] = scaling(a.coords or (1 << 22), a.rounds)
        print(_table(res["scaling"], ["workload", "n_ranks", "topology", "dynamiq_b5", "mxfp8", "ms_per_allreduce"]))
    if a.json:
        with open(a.json, "w") as f:
            json.dump(res, f, indent=1)


if __name__ == "__main__":
    main()
