#!/usr/bin/env python3
"""Benchmark of the DynamiQ hot path on one GB300: one step = one full
simulated all-reduce round of N workers (statistics, metadata all-reduce,
allocation, reordering, compress, N-1 decompress-accumulate-recompress hops
or the butterfly steps, and every rank's final decode) over synthetic bf16
gradients already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

Prints one JSON line (rank 0).  Under torchrun each GPU runs an independent
replica of the whole simulation (the path does not shard across GPUs: all N
simulated workers live in one GPU's memory), timed between barriers, and the
slowest rank's time is reported ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DAR Gcoords/s/hop and % of HBM peak; simulated all-reduce ms per GB of grad"
UNIT = "ms/GB"
DEFAULT_WORKLOAD = "gemma1b_ring16"
SG = 256


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["dq", "reference"], default="dq")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--coords", type=int, default=0,
                   help="coordinates per worker (0: the workload's own size; smaller for profiling)")
    p.add_argument("--e2e-steps", type=int, default=0, help="steps of the end-to-end timing (0: auto)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    p.add_argument("--exchange", choices=["auto", "fused", "multi", "pipelined"], default="auto",
                   help="ring exchange as one cooperative launch (fused), one launch per step (multi) or pipelined "
                        "over parts of the super-groups (pipelined); auto: the faster path for the size "
                        "(allreduce.exchange_mode: fused up to 2^17 super-groups per worker, pipelined above, rings "
                        "of up to 64 ranks; the butterfly runs step by step)")
    p.add_argument("--parts", type=int, default=0,
                   help="parts of the pipelined exchange (0: allreduce.pipeline_parts)")
    p.add_argument("--lean", action="store_true",
                   help="the timed rounds only: no end-to-end, MXFP8, budget-sweep or accuracy legs and no extra "
                        "workloads (for profiler captures, whose launch lists stay short)")
    p.add_argument("--extras", default="",
                   help="comma-separated workloads measured after the headline one ('none': skip; default: "
                        + ",".join(EXTRA_WORKLOADS) + ")")
    p.add_argument("--bucket-pool", type=int, default=16,
                   help="streamed workloads: distinct buckets kept resident and cycled through a full pass")
    return p.parse_args(argv)


# --------------------------------------------------------------------------- distributed helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as td
    if world > 1 and not td.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        td.init_process_group(backend=backend)
    return td


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as td
        if device is not None and td.get_backend() == "nccl":
            td.barrier(device_ids=[device.index])
        else:
            td.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (works with nccl and gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as td
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if td.get_backend() == "nccl" else "cpu")
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        try:
            fd, self.path = tempfile.mkstemp(prefix="dq_clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    @staticmethod
    def _epoch(ts: str):
        import datetime
        try:
            return datetime.datetime.strptime(ts.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, t0: float = None, t1: float = None):
        """Summary of the samples taken between wall-clock times t0 and t1."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    t = self._epoch(parts[0])
                    if t0 is not None and t is not None and not (t0 - 0.05 <= t <= t1 + 0.05):
                        continue
                    rows.append(parts[1:])
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# The device code of each profiled kernel: its own file plus the shared
# definitions (the launch parameters and tables come from the host files, so
# those count too where they shape the kernel's work).
KERNEL_SOURCES = {
    "hop_kernel": ["dq_common.cuh", "dq_hop.cu"],
    "decode_kernel": ["dq_common.cuh", "dq_hop.cu"],
    "fused_ring_kernel": ["dq_common.cuh", "dq_hop.cu"],
    "wave_ring_kernel": ["dq_common.cuh", "dq_hop.cu"],
    "stream_ring_kernel": ["dq_common.cuh", "dq_hop.cu"],
    "stats_kernel": ["dq_common.cuh", "dq_codec.cu"],
    "mx_hop_kernel": ["dq_common.cuh", "dq_mx.cu"],
}


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank lines (string literals in
    these files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str) -> str:
    """sha256 prefix of the code (comments and blank lines dropped) of the
    files that define `kernel` (its name before any template arguments)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_hop_gradient_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel.split("<")[0]]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:12]


def ncu_counters(kernel: str, workload: str):
    """(DRAM bytes per launch, warp-instructions per super-group) from the
    committed ncu summary, if it was taken on the current kernel sources
    (else (None, None))."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None, None
    want = kernel_source_hash(kernel)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                    and parts[3] == want:
                return float(parts[2]), (float(parts[4]) if len(parts) > 4 else None)
    return None, None


# --------------------------------------------------------------------------- algorithmic bytes
def step_roofline(kernels, per_step_key, ms_step, peak):
    """The whole step against the HBM roofline: the algorithmic bytes of every
    kernel launched in one step (each kernel's bytes per launch times its
    launches per step) over the step's time."""
    by = sum(k["alg_bytes_per_launch"] * k[per_step_key] for k in kernels.values())
    gbs = by / (ms_step * 1e-3) / 1e9
    return {"alg_bytes": by, "achieved": gbs, "frac": gbs / peak,
            "note": "every kernel of one step: its algorithmic bytes per launch times its launches per step, over "
                    "the step's time"}


def stream_message_bytes(dq, info, N):
    lo = dq.dq_chunk_cuts(info.n2, info.n4, info.n8, N)
    e2, e4 = info.n2, info.n2 + info.n4
    return sum(dq.dq_message_bytes(dq.rng(lo[c], lo[c + 1], e2, e4)) for c in range(N))


def launch_bytes(kind: int, sgs: int, msg_per_sg: float, fp32_addend: bool = False, n_ranks: int = 1,
                 send_frac: float = 1.0) -> float:
    """Algorithmic HBM bytes of one launch over `sgs` super-groups: every
    input byte read once and every output byte written once, nothing else.
    compress: bf16 gradient 512 B/SG + message out + mean and perm 8 B/SG;
    DAR: message in + addend (512 B/SG bf16 with mean and perm 8 B/SG, or
    1 KiB/SG fp32 with perm 4 B/SG) + the send fraction's message out + the
    kept fraction's fp32 rows (1 KiB/SG; a butterfly step sends half and keeps
    half, a ring hop sends everything);
    decode: fp32 output 1 KiB per super-group written, message in + 8 B per
    super-group read (once for up to 16 outputs);
    stats: bf16 gradient 512 B/SG + mean and squared norm 8 B/SG;
    allocate + reorder span: N x 8 B/SG of statistics read, M, F, mu written
    (12 B/SG), then two more select passes and the bitwidth pass over F
    (12 B/SG), the bitwidths written and read back (2 B/SG) and the
    permutation written (4 B/SG); fused ring exchange: the compress, N-1 DARs
    and a decode that reads each message once and writes N outputs;
    pipelined ring exchange: the same bytes per round, each launch counted
    by its share of the round's super-groups (its logged hop and decode
    super-groups add up to J (N + 1) per round); bucket stream: likewise per
    bucket (a bucket's J super-groups are logged by each of the N + 1
    launches it takes part in)."""
    if kind == 0:
        return sgs * (512 + send_frac * msg_per_sg + 8 + (1.0 - send_frac) * 1024)
    if kind == 1:
        add = 1024 + 4 if fp32_addend else 512 + 8
        return sgs * (msg_per_sg + add + send_frac * msg_per_sg + (1.0 - send_frac) * 1024)
    if kind == 2:   # sgs = super-groups written; each launch reads a message once for up to 16 outputs
        return sgs * 1024 + sgs / min(n_ranks, 16) * (msg_per_sg + 8)
    if kind == 3:
        return sgs * (512 + 8)
    if kind in (7, 8, 9):   # fused, pipelined or bucket-stream ring: J (N + 1) super-groups per bucket
        J = sgs / (n_ranks + 1)
        return J * ((512 + msg_per_sg + 8) + (n_ranks - 1) * (2 * msg_per_sg + 512 + 8) +
                    (msg_per_sg + 8 + 1024 * n_ranks))
    return sgs * (8 * n_ranks + 12 + 12 + 2 + 4)


def hop_roles(butterfly: bool, n_ranks: int):
    """(name, fp32 addend, send fraction) of the hop launches of one round,
    in launch order (one launch per step: every rank's hop of that step).
    Ring: the compress, then N-1 DARs with bf16 addends that send
    everything.  Butterfly (L = log2 N): the compress of the half each rank
    sends; step 1 decodes, adds the bf16 gradient and splits (half sent,
    half kept in fp32); steps 2 .. L-1 add the fp32 kept half and split;
    step L is the owner's single quantization of its chunk."""
    if not butterfly:
        return [("compress", False, 1.0)] + [("dar", False, 1.0)] * (n_ranks - 1)
    L = max(1, n_ranks.bit_length() - 1)
    roles = [("compress", False, 1.0)]
    for s in range(1, L + 1):
        if s == L:
            roles.append(("dar_f32_final", True, 1.0) if L >= 2 else ("dar_bf16_final", False, 1.0))
        elif s == 1:
            roles.append(("dar_bf16_split", False, 0.5))
        else:
            roles.append(("dar_f32_split", True, 0.5))
    return roles


# --------------------------------------------------------------------------- oracle on the host
def oracle_allreduce_seconds(w, gu, round_=0):
    import oracle
    cfg = oracle.Config(w.n_ranks, w.budget, correlated=w.correlated, seed=0, round=round_)
    t = time.perf_counter()
    oracle.allreduce(cfg, gu, butterfly=w.topology == "butterfly")
    return time.perf_counter() - t


def oracle_threads() -> int:
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def calibrated_sample(w, host_slices, target_s: float):
    """Coordinates per worker for a run of about target_s seconds."""
    probe = min(w.n_pad, 1 << 18)
    t = oracle_allreduce_seconds(w, [h[:probe] for h in host_slices(probe)])
    n = int(probe * target_s / max(t, 1e-3))
    n = max(probe, min(w.n_pad, n)) // SG * SG
    return n


def cpu_baseline(w, grads_dev, target_s: float):
    """The oracle, as it stands, on the first coordinates of every worker of
    the same workload (its own all-reduce over that sample)."""
    from quantized_hop_gradient_gb300 import synth

    def slices(n):
        return [synth.as_u16(g[:n]) for g in grads_dev]

    n = calibrated_sample(w, slices, target_s)
    gu = slices(n)
    secs = oracle_allreduce_seconds(w, gu)
    gb = n * 2 / 1e9
    return {"value": secs * 1e3 / gb, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"first {n} of {w.n_pad} coordinates of each of the {w.n_ranks} workers "
                      f"({n // SG} super-groups): statistics, allocation, reordering, the "
                      f"{w.topology} all-reduce and one decode, {secs:.1f} s"}


# --------------------------------------------------------------------------- the GPU arm
# Workloads measured after the headline one, each with its own DAR roofline
# fraction (a compact line: per-kernel times, DAR, vNMSE; no end-to-end or
# CPU leg).  Skipped under torchrun (N > 1 replicas) and with --extras none.
EXTRA_WORKLOADS = ("bert_large_ring8", "llama1b_butterfly8")
KERNEL_NAMES = {"compress": "hop_kernel<false,false> (compress)", "dar": "hop_kernel<true,false> (DAR, bf16 addend)",
                "dar_bf16_split": "hop_kernel<true,false> (DAR, bf16 addend, split)",
                "dar_f32_split": "hop_kernel<true,true> (DAR, fp32 addend, split)",
                "dar_f32_final": "hop_kernel<true,true> (DAR, fp32 addend)",
                "dar_bf16_final": "hop_kernel<true,false> (DAR, bf16 addend)",
                "decode": "decode_kernel", "stats": "stats_kernel", "fused_ring": "fused_ring_kernel",
                "pipelined": "wave_ring_kernel (pipelined ring exchange: hop steps of later parts and the final "
                             "decode of an earlier part in each launch)",
                "stream": "stream_ring_kernel (bucket stream: ring steps of N buckets and the final decode of one "
                          "bucket in each launch)"}
# the key under which profiles/dram_traffic.txt lists a kernel role
TRAFFIC_KEY = {"dar": "hop_kernel<true,false>", "dar_bf16_split": "hop_kernel<true,false>:split",
               "dar_bf16_final": "hop_kernel<true,false>:final", "dar_f32_split": "hop_kernel<true,true>:split",
               "dar_f32_final": "hop_kernel<true,true>:final", "compress": "hop_kernel<false,false>",
               "decode": "decode_kernel", "stats": "stats_kernel", "fused_ring": "fused_ring_kernel",
               "pipelined": "wave_ring_kernel", "stream": "stream_ring_kernel"}


def kernel_table(log, steps: int, ms_step: float, msg_per_sg: float, N: int, butterfly: bool):
    """Per-role launch statistics of `steps` logged rounds: launches, average
    launch time (CUDA events on the launching stream), share of the step,
    algorithmic bytes and the GB/s and Gcoords/s they imply.  Hop launches
    are named by their role in the round (hop_roles)."""
    roles = hop_roles(butterfly, N)
    other = {2: "decode", 3: "stats", 4: "allocate_reorder", 7: "fused_ring", 8: "pipelined"}
    per = {}
    hop_i = 0
    for kind, sgs, t in log.launches():
        if kind == 3:                   # a round's planning starts: hop launches count from 0 again
            hop_i = 0
        if kind in (0, 1):
            name, f32, frac = roles[min(hop_i, len(roles) - 1)] if butterfly else \
                (("compress", False, 1.0) if kind == 0 else ("dar", False, 1.0))
            hop_i += 1
            by = launch_bytes(kind, sgs, msg_per_sg, fp32_addend=f32, n_ranks=N, send_frac=frac)
        else:
            name = other.get(kind, f"kind{kind}")
            by = launch_bytes(kind, sgs, msg_per_sg, n_ranks=N)
        d = per.setdefault(name, {"launches": 0, "ms": 0.0, "sgs": 0, "bytes": 0.0})
        d["launches"] += 1
        d["ms"] += t
        d["sgs"] += sgs
        d["bytes"] += by
    out = {}
    for name, d in per.items():
        avg_ms = d["ms"] / d["launches"]
        out[name] = {"launches_per_step": d["launches"] / steps, "avg_launch_ms": avg_ms,
                     "share_of_step": d["ms"] / steps / ms_step,
                     "alg_bytes_per_launch": d["bytes"] / d["launches"],
                     "achieved_gbs": d["bytes"] / d["launches"] / (avg_ms * 1e-3) / 1e9,
                     "gcoords_per_s": d["sgs"] / d["launches"] * SG / (avg_ms * 1e-3) / 1e9}
    return out


def dar_summary(kernels, peak, workload):
    """The DAR hop(s) of a round against the HBM roofline: per role, Gcoords/s
    per hop, GB/s and the fraction of the measured copy bandwidth."""
    out = {}
    for name, k in kernels.items():
        if name.startswith("dar"):
            traffic, inst = ncu_counters(TRAFFIC_KEY[name], workload)
            out[name] = {"kernel": KERNEL_NAMES[name], "gcoords_per_s_per_hop": k["gcoords_per_s"],
                         "achieved_gbs": k["achieved_gbs"], "hbm_frac": k["achieved_gbs"] / peak,
                         "avg_launch_ms": k["avg_launch_ms"], "launches_per_step": k["launches_per_step"],
                         "alg_bytes_per_launch": k["alg_bytes_per_launch"], "traffic": traffic,
                         "warp_instructions_per_super_group": inst}
    return out


def measure_round(args, w, dev, world, K, W, full: bool, local: int = 0):
    """Times K simulated all-reduce rounds of workload w (after W warm-up
    rounds) and returns the per-kernel breakdown; with `full` also the
    end-to-end timing, the MXFP8 comparison and the budget sweep."""
    import torch

    from quantized_hop_gradient_gb300 import dq, study, synth
    from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce, exchange_mode, pipeline_parts

    N, J = w.n_ranks, w.n_sg
    butterfly = w.topology == "butterfly"
    grads = synth.generate(w, dev, seed=0)
    ar = DynamiQAllReduce(N, J, budget=w.budget, correlated=w.correlated, butterfly=butterfly, seed=0)
    outs = ar.new_outputs()
    ring64 = not butterfly and N <= dq.MAX_FUSED_RANKS
    # (fused, parts) of the exchange
    mode = {"auto": exchange_mode(N, butterfly, J), "fused": (True, None), "multi": (False, None),
            "pipelined": (False, pipeline_parts(N, J))}[args.exchange]
    if mode[1] and args.parts > 0:
        mode = (False, args.parts)
    if mode != (False, None) and not ring64:
        raise SystemExit("the fused and pipelined exchanges cover rings of up to 64 ranks")
    STEPWISE = (False, None)

    def step(i, log=None, mode=mode, ar=ar):
        ar.plan(grads, round=i, log=log)
        ar.exchange(grads, outs, round=i, log=log, fused=mode[0], parts=mode[1])

    def measure(fused_, steps, first, sample_clocks=False, ar_=ar):
        """Times `steps` rounds (CUDA events on the launching stream, a
        barrier and a synchronize on both sides) and records every launch."""
        log = dq.LaunchLog(steps * (6 * N + 12))
        log.c.count = 0
        torch.cuda.synchronize()
        barrier(world, dev)
        torch.cuda.synchronize()
        n0 = dq.dq_launch_count()
        clocks = ClockSampler(local).start() if sample_clocks else None
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e0.record()
        for i in range(steps):
            step(first + i, log, fused_, ar_)
        e1.record()
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world, dev)
        if fused_[0]:
            ar_.check_status()
        clk = clocks.stop(t0, t1) if clocks else None
        return e0.elapsed_time(e1) / steps, log, dq.dq_launch_count() - n0, clk

    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    ms, log, n_launch, clk = measure(mode, K, W, sample_clocks=full)
    peak, peak_kind = measured_peaks()
    msg_per_sg = stream_message_bytes(dq, ar.info, N) / J
    kernels = kernel_table(log, K, ms, msg_per_sg, N, butterfly)
    kernels_multi = ms_multi = None
    if mode != STEPWISE:
        # the per-step kernels of the multi-launch exchange, for the hop breakdown
        step(W + K, None, STEPWISE)
        KM = max(3, min(K, 10))
        ms_multi, log_m, _, _ = measure(STEPWISE, KM, W + K + 1)
        kernels_multi = kernel_table(log_m, KM, ms_multi, msg_per_sg, N, butterfly)
    dominant = max((k for k in kernels if k != "allocate_reorder"), key=lambda k: kernels[k]["share_of_step"])
    dk = kernels[dominant]
    traffic, _ = ncu_counters(TRAFFIC_KEY[dominant], w.name)
    roofline = {"bound": "hbm", "kernel": KERNEL_NAMES[dominant], "achieved": dk["achieved_gbs"], "peak": peak,
                "unit": "GB/s", "frac": dk["achieved_gbs"] / peak, "peak_source": peak_kind,
                "traffic": traffic, "alg_bytes_per_launch": dk["alg_bytes_per_launch"],
                "step": step_roofline(kernels, "launches_per_step", ms, peak)}
    gb = J * SG * 2 / 1e9
    res = {"workload": w.name, "ms_per_step": ms, "ms_per_gb": ms / gb, "grad_gb_per_worker": gb,
           "simulated_workers": N, "topology": w.topology, "coords_per_worker": w.n, "super_groups": J,
           "budget_bits": w.budget, "correlated_rounding": w.correlated,
           "allocation": {"T": ar.info.T, "n2": ar.info.n2, "n4": ar.info.n4, "n8": ar.info.n8},
           "exchange": ("fused (one cooperative launch per round)" if mode[0] else
                        f"pipelined over {mode[1]} parts ({N + mode[1]} launches per round)" if mode[1] else
                        "one launch per step"),
           "dar": dar_summary(kernels_multi or kernels, peak, w.name), "kernels": kernels,
           "kernels_multi_launch": kernels_multi, "ms_per_step_multi_launch": ms_multi, "roofline": roofline,
           "gpu_launches": n_launch, "clocks": clk, "steps": K, "warmup": W}

    if args.lean:
        return res, grads
    # accuracy of the last timed round's configuration (round K + W + ...: a fresh round, same inputs)
    s_exact = study.exact_sum(grads)
    step(10_000)
    torch.cuda.synchronize()
    acc = {"vnmse": study.vnmse(outs[0], s_exact),
           "wire_bytes_per_coord": msg_per_sg / SG, "rounds_measured": 1}
    if butterfly:
        # correlated rounding shares one uniform among the senders of a
        # butterfly stage; independent rounding draws its own per sender
        ind = DynamiQAllReduce(N, J, budget=w.budget, correlated=False, butterfly=True, seed=0)
        v_c, v_i = [], []
        for r in range(2):
            ar(grads, round=20_000 + r, outs=outs)
            v_c.append(study.vnmse(outs[0], s_exact))
            ind(grads, round=20_000 + r, outs=outs)
            v_i.append(study.vnmse(outs[0], s_exact))
        acc.update({"vnmse_correlated": sum(v_c) / 2, "vnmse_independent": sum(v_i) / 2,
                    "independent_over_correlated": sum(v_i) / sum(v_c), "rounds_compared": 2})
        del ind
    else:
        acc["correlated_rounding_note"] = ("a ring stage has one quantizer, so correlated rounding changes the "
                                           "random stream but not the expected error")
    res["accuracy"] = acc

    if full:
        res["e2e"] = e2e_timing(args, w, ar, grads, outs, mode, dev, world)
        res["accuracy"], res["mxfp8"] = compare_mxfp8(w, grads, outs, ar, dev, N, J, butterfly, peak, acc, s_exact)
        res["budget_sweep"] = budget_sweep(w, grads, outs, dev, N, J, butterfly, peak, s_exact, mode)
    del s_exact
    return res, grads


def budget_sweep(w, grads, outs, dev, N, J, butterfly, peak, s_exact, mode):
    """The workload's other budgets (same gradients): ms per round (exchange
    `mode` = (fused, parts)), the DAR hop (one launch per step) and vNMSE at
    each."""
    import torch

    from quantized_hop_gradient_gb300 import dq, study
    from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce

    out = {}
    for B in w.budgets:
        if B == w.budget:
            continue
        ar = DynamiQAllReduce(N, J, budget=B, correlated=w.correlated, butterfly=butterfly, seed=0)
        KB = 5

        def rounds(mode_, first, log=None):
            for i in range(2):
                ar(grads, round=i, outs=outs, fused=mode_[0], parts=mode_[1])
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(KB):
                ar.plan(grads, round=first + i, log=log)
                ar.exchange(grads, outs, round=first + i, log=log, fused=mode_[0], parts=mode_[1])
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / KB

        ms = rounds(mode, 100)
        log = dq.LaunchLog(KB * (6 * N + 12))
        log.c.count = 0
        ms_steps = rounds((False, None), 200, log)
        msg = stream_message_bytes(dq, ar.info, N) / J
        kt = kernel_table(log, KB, ms_steps, msg, N, butterfly)
        out[str(B)] = {"ms_per_step": ms, "ms_per_gb": ms / (J * SG * 2 / 1e9),
                       "wire_bytes_per_coord": msg / SG, "vnmse": study.vnmse(outs[0], s_exact),
                       "allocation": {"T": ar.info.T, "n2": ar.info.n2, "n4": ar.info.n4, "n8": ar.info.n8},
                       "dar": dar_summary(kt, peak, w.name)}
        del ar
    return out


def e2e_timing(args, w, ar, grads, outs, mode, dev, world):
    """End to end: the gradients start in pinned host memory and rank 0's fp32
    result ends there; every copy is inside the timed region.  Round i+1's
    upload (copy stream) runs while round i computes, into the other of two
    device gradient buffers; each rank's statistics wait only for that rank's
    upload; the result download runs on a third stream."""
    import torch

    N, J = w.n_ranks, w.n_sg
    KE = args.e2e_steps or max(3, min(args.steps, 10))
    # one pinned host copy per simulated worker; under torchrun (one process
    # per GPU, all on one node) the simulated workers of a process share one
    # pinned copy, so the node's pinned memory stays one gradient per GPU (the
    # bytes copied per step are the same)
    shared = world > 1
    hosts = pinned_host_copies([grads[0]]) * N if shared else pinned_host_copies(grads)
    out_host = torch.empty(J * SG, dtype=torch.float32, pin_memory=True)
    gbuf = [grads, [torch.empty_like(g) for g in grads]]
    main = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(N)] for _ in range(2)]
    ev_free = [torch.cuda.Event(), torch.cuda.Event()]
    ev_dec, ev_out = torch.cuda.Event(), torch.cuda.Event()

    def upload(i):
        b = i & 1
        cin.wait_event(ev_free[b])
        with torch.cuda.stream(cin):
            for r in range(N):
                gbuf[b][r].copy_(hosts[r], non_blocking=True)
                ev_in[b][r].record(cin)

    def compute(i):
        b = i & 1
        ar.plan(gbuf[b], round=i, ready=ev_in[b])
        main.wait_event(ev_out)
        ar.exchange(gbuf[b], outs, round=i, fused=mode[0], parts=mode[1])
        ev_free[b].record(main)
        ev_dec.record(main)
        cout.wait_event(ev_dec)
        with torch.cuda.stream(cout):
            out_host.copy_(outs[0], non_blocking=True)
            ev_out.record(cout)

    def e2e_run(first, steps):
        upload(first)
        for i in range(first, first + steps):
            if i + 1 < first + steps:
                upload(i + 1)
            compute(i)
        main.wait_event(ev_out)

    # the host link's rate on this machine now: plain uploads of the same buffers
    # (the first one warms the path; the second is timed)
    link = []
    for _ in range(2):
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(cin)
        with torch.cuda.stream(cin):
            for r in range(N):
                gbuf[1][r].copy_(hosts[r], non_blocking=True)
        l1.record(cin)
        cin.synchronize()
        link.append(l0.elapsed_time(l1))
    link_gbs = N * J * SG * 2 / (link[-1] * 1e-3) / 1e9
    e2e_run(0, 2)
    torch.cuda.synchronize()
    barrier(world, dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(main)
    cin.wait_event(f0)
    e2e_run(2, KE)
    f1.record(main)
    torch.cuda.synchronize()
    barrier(world, dev)
    ms_e2e = max_over_ranks(f0.elapsed_time(f1) / KE, world, dev)
    gb = J * SG * 2 / 1e9
    h2d = N * J * SG * 2
    res = {"value": ms_e2e / (world * gb), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": J * SG * 4, "ms_per_step": ms_e2e, "steps": KE,
           "h2d_gbs": h2d / (ms_e2e * 1e-3) / 1e9,
           "host_buffers": "one pinned buffer shared by the simulated workers of each process" if shared
           else "the simulated workers' gradients as slices of one pinned allocation",
           "link_gbs": link_gbs, "link_floor_ms": h2d / (link_gbs * 1e9) * 1e3,
           "link_note": "link_gbs: a plain upload of the same pinned buffers timed just before; link_floor_ms: "
                        "the upload of every rank's gradient at that rate, which bounds the end-to-end step (the "
                        "link's rate varies from box to box and over time on some)"}
    del gbuf[1], hosts
    return res


def pinned_host_copies(ts):
    """Pinned host copies of device tensors ts (same dtype), as slices of ONE
    pinned allocation.  Measured on these boxes: host-to-device copies from
    16 separately pinned 2 GB buffers ran at 43-191 GB/s, varying from round
    to round, against a steady 211.6 GB/s from slices of one 32 GB
    allocation (whatever the destinations)."""
    import torch
    total = sum(t.numel() for t in ts)
    h = torch.empty(total, dtype=ts[0].dtype, pin_memory=True)
    out, o = [], 0
    for t in ts:
        v = h[o:o + t.numel()]
        v.copy_(t)
        out.append(v)
        o += t.numel()
    return out


def run_gpu(args, rank, world, local):
    import torch

    from quantized_hop_gradient_gb300 import dq, synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    dq.lib(build=True)
    w = synth.WORKLOADS[args.workload]
    if args.coords:
        w = w.scaled(args.coords)
    if w.bucket:
        return run_gpu_bucketed(args, rank, world, local, w, dev)
    K, W = args.steps, max(args.warmup, 0)
    main, grads = measure_round(args, w, dev, world, K, W, full=True, local=local)
    ms_max = max_over_ranks(main["ms_per_step"], world, dev)
    gb = main["grad_gb_per_worker"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.lean:
        cpu = cpu_baseline(w, grads, args.cpu_seconds)
    del grads
    torch.cuda.empty_cache()

    extras = {}
    names = [] if (world > 1 or args.extras == "none" or args.coords or args.lean) else \
        [x for x in (args.extras.split(",") if args.extras else EXTRA_WORKLOADS) if x and x != w.name]
    for name in names:
        xw = synth.WORKLOADS[name]
        KX, WX = max(3, min(K, 10)), 3
        r, g = measure_round(args, xw, dev, world, KX, WX, full=False, local=local)
        del g
        torch.cuda.empty_cache()
        extras[name] = {k: r[k] for k in ("ms_per_step", "ms_per_gb", "simulated_workers", "topology",
                                          "coords_per_worker", "budget_bits", "correlated_rounding", "allocation",
                                          "exchange", "dar", "roofline", "accuracy", "steps", "warmup")}
        extras[name]["kernels"] = {k: {kk: v[kk] for kk in ("avg_launch_ms", "share_of_step", "achieved_gbs")}
                                   for k, v in r["kernels"].items()}

    dar = main["dar"].get("dar") or next(iter(main["dar"].values()), {})
    line = {
        "metric": METRIC, "value": ms_max / (world * gb), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_max, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 codec, 2/4/8-bit codes", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "simulated_workers": w.n_ranks, "topology": w.topology,
                   "coords_per_worker": w.n, "super_groups": w.n_sg, "budget_bits": w.budget,
                   "correlated_rounding": w.correlated, "grad_gb_per_worker": gb,
                   "parallelism": f"replicas x{world} (all simulated workers on each GPU)",
                   "l2": "inputs larger than L2 (no flush needed)", "allocation": main["allocation"]},
        "dar": {"gcoords_per_s_per_hop": dar.get("gcoords_per_s_per_hop"), "achieved_gbs": dar.get("achieved_gbs"),
                "hbm_frac": dar.get("hbm_frac"), "avg_launch_ms": dar.get("avg_launch_ms"),
                "roles": main["dar"]},
        "exchange": main["exchange"],
        "kernels": main["kernels"],
        "kernels_multi_launch": main["kernels_multi_launch"],
        "ms_per_step_multi_launch": main["ms_per_step_multi_launch"],
        "roofline": main["roofline"],
        "e2e": main.get("e2e"),
        "gpu_launches": main["gpu_launches"],
        "clocks": main["clocks"],
        "accuracy": main.get("accuracy"),
        "mxfp8": main.get("mxfp8"),
        "budget_sweep": main.get("budget_sweep"),
        "extra_workloads": extras or None,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def compare_mxfp8(w, grads, outs, ar, dev, N, J, butterfly, peak, acc, s_exact):
    """After the timed region: the vNMSE of a DynamiQ round and of the MXFP8
    baseline on the same gradients, and the MXFP8 all-reduce's time on the
    same GPU (its hops read 1 + 1/32 B of message, 2 B of bf16 gradient and
    write 1 + 1/32 B per coordinate)."""
    import torch

    from quantized_hop_gradient_gb300 import dq, study
    from quantized_hop_gradient_gb300.allreduce import MXFP8AllReduce

    v_dq = acc["vnmse"]
    mx = MXFP8AllReduce(N, J * SG, butterfly=butterfly, device=dev)
    for _ in range(2):
        mx(grads, outs)
    KM = 5
    log = dq.LaunchLog(KM * (2 * N + 8))
    log.c.count = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(KM):
        mx(grads, outs, log=log)
    e1.record()
    torch.cuda.synchronize()
    ms_mx = e0.elapsed_time(e1) / KM
    v_mx = study.vnmse(outs[0], s_exact)
    hops = [(sgs, t) for k, sgs, t in log.launches() if k == dq.DQ_LAUNCH_MX_HOP]
    per_round = len(hops) // KM
    dar = [h for i, h in enumerate(hops) if i % per_round != 0] if not butterfly else []
    mx_line = {"ms_per_step": ms_mx, "ms_per_gb": ms_mx / (J * SG * 2 / 1e9),
               "wire_bytes_per_coord": (1 + 1 / 32)}
    if dar:
        coords = sum(sgs for sgs, _ in dar) * SG / len(dar)
        t = sum(tt for _, tt in dar) / len(dar) * 1e-3
        gbs = coords * (2 + 2 * (1 + 1 / 32)) / t / 1e9
        mx_line.update({"dar_avg_launch_ms": t * 1e3, "dar_gcoords_per_s": coords / t / 1e9, "dar_gbs": gbs,
                        "dar_hbm_frac": gbs / peak})
    del mx
    torch.cuda.empty_cache()
    acc = dict(acc)
    acc.update({"vnmse_mxfp8": v_mx, "mxfp8_over_dynamiq": v_mx / v_dq if v_dq > 0 else None})
    return acc, mx_line


# --------------------------------------------------------------------------- streamed workloads
def run_gpu_bucketed(args, rank, world, local, w, dev):
    """A streamed workload (DDP buckets): one step is a full pass over the
    model's buckets, each bucket a DynamiQ round.  Rings of up to 8 ranks
    run the bucket stream whose exchange is pipelined across buckets
    (stream.BucketStream: each launch carries N buckets' ring steps and one
    bucket's decode; planning a few buckets ahead on a second stream); the
    per-bucket stream (one cooperative exchange launch per bucket, the next
    bucket's planning on a second stream) is timed beside it.  The gradient
    data cycle through a pool of resident buckets drawn from across the model
    (the whole model does not fit in HBM with every worker's copy)."""
    import torch

    from quantized_hop_gradient_gb300 import dq, synth
    from quantized_hop_gradient_gb300.allreduce import use_fused
    from quantized_hop_gradient_gb300.stream import BucketedAllReduce, BucketStream

    N = w.n_ranks
    nb = synth.bucket_count(w)
    P = max(2, min(args.bucket_pool, nb))
    picks = sorted({round(i * (nb - 2) / (P - 2)) for i in range(P - 1)}) + [nb - 1]
    pool = [synth.generate_bucket(w, k, dev, seed=0) for k in picks]
    full, last = pool[:-1], pool[-1]
    pool_of = [i % len(full) for i in range(nb - 1)] + [len(pool) - 1]   # bucket k -> pool entry
    seq = [pool[i] for i in pool_of]
    outs_pool = [[torch.empty(g.numel(), dtype=torch.float32, device=dev) for g in b] for b in pool]
    seq_out = [outs_pool[i] for i in pool_of]
    bucket_sg = w.bucket // SG
    kw = dict(budget=w.budget, correlated=w.correlated, butterfly=w.topology == "butterfly", seed=0)
    # the pipelined bucket stream where it applies (rings of up to 8 ranks);
    # the per-bucket stream with its own choice of exchange ("auto": the
    # cooperative one-launch exchange for rings of up to 64 ranks and 2^17
    # super-groups) is timed beside it for comparison
    piped = w.topology == "ring" and N <= dq.MAX_STREAM_RANKS
    per_bucket = BucketedAllReduce(N, bucket_sg, overlap=True, fused="auto", **kw)
    ov = BucketStream(N, bucket_sg, budget=w.budget, correlated=w.correlated, seed=0) if piped else per_bucket
    alt = per_bucket if piped else None
    sq = BucketedAllReduce(N, bucket_sg, overlap=False, fused=False, **kw)
    K, W = args.steps, max(args.warmup, 0)

    def timed(ar, steps, first, log=None):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(world, dev)
        e0.record()
        for i in range(steps):
            ar.run(seq, seq_out, round0=(first + i) * nb, log=log)
        e1.record()
        torch.cuda.synchronize()
        barrier(world, dev)
        return e0.elapsed_time(e1) / steps

    clocks = ClockSampler(local).start()
    for i in range(W):
        ov.run(seq, seq_out, round0=i * nb)
    n0 = dq.dq_launch_count()
    t0 = time.time()
    ms = timed(ov, K, W)
    t1 = time.time()
    n_launch = dq.dq_launch_count() - n0
    clk = clocks.stop(t0, t1)
    if getattr(ov, "fused", False):
        for s_ in ov.sets:
            s_.check_status()
    # one more pass with every launch recorded: per-kernel times and the roofline
    log = dq.LaunchLog(nb * 20)
    log.c.count = 0
    ms_logged = timed(ov, 1, W + K, log=log)
    infos_msg = []
    per = {}
    kind_name = {0: "compress", 1: "dar", 2: "decode", 3: "stats", 4: "allocate_reorder", 7: "fused_ring",
                 9: "stream"}
    ref_set = per_bucket.sets[0]
    for kind, sgs, t in log.launches():
        d = per.setdefault(kind_name.get(kind, str(kind)), {"launches": 0, "ms": 0.0, "sgs": 0})
        d["launches"] += 1
        d["ms"] += t
        d["sgs"] += sgs
    # message bytes per super-group of a typical bucket (the first pool entry)
    info0 = ref_set.plan(pool[0], round=0)
    torch.cuda.synchronize()
    msg_per_sg = stream_message_bytes(dq, info0, N) / bucket_sg
    kernels = {}
    for name, d in per.items():
        kind = [k for k, v in kind_name.items() if v == name][0]
        avg = d["ms"] / d["launches"]
        by = launch_bytes(kind, d["sgs"] / d["launches"], msg_per_sg, n_ranks=N)
        kernels[name] = {"launches_per_step": d["launches"], "avg_launch_ms": avg,
                         "share_of_step_serial": d["ms"] / ms_logged, "alg_bytes_per_launch": by,
                         "achieved_gbs": by / (avg * 1e-3) / 1e9,
                         "gcoords_per_s": d["sgs"] / d["launches"] * SG / (avg * 1e-3) / 1e9}
    peak, peak_kind = measured_peaks()
    dominant = max((k for k in kernels if k != "allocate_reorder"), key=lambda k: kernels[k]["share_of_step_serial"])
    dk = kernels[dominant]
    traffic, _ = ncu_counters(TRAFFIC_KEY.get(dominant, dominant), w.name)
    roofline = {"bound": "hbm", "kernel": KERNEL_NAMES.get(dominant, dominant), "achieved": dk["achieved_gbs"],
                "peak": peak, "unit": "GB/s", "frac": dk["achieved_gbs"] / peak, "peak_source": peak_kind,
                "traffic": traffic, "alg_bytes_per_launch": dk["alg_bytes_per_launch"],
                "note": "planning kernels run on a second stream under the exchange's launches, so the "
                        "launch shares add up to more than the step",
                "step": step_roofline(kernels, "launches_per_step", ms, peak)}

    ms_seq = ms_alt = None
    if not args.lean:
        sq.run(seq, seq_out, round0=(W + K + 2) * nb)      # warm-up pass (workspace allocation)
        ms_seq = timed(sq, 1, W + K + 3)
    if alt is not None and not args.lean:
        alt.run(seq, seq_out, round0=(W + K + 4) * nb)
        ms_alt = timed(alt, 2, W + K + 5)
        if alt.fused:
            for s_ in alt.sets:
                s_.check_status()
    ms_max = max_over_ranks(ms, world, dev)
    gb = w.n * 2 / 1e9

    e2e = None if args.lean else bucketed_e2e(args, w, ov, pool, pool_of, outs_pool, nb, dev, world, gb)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.lean:
        cpu = bucketed_cpu_baseline(w, nb, gb)
    line = {
        "metric": METRIC, "value": ms_max / (world * gb), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 codec, 2/4/8-bit codes", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "simulated_workers": N, "topology": w.topology, "coords_per_worker": w.n,
                   "bucket_coords": w.bucket, "buckets": nb, "resident_bucket_pool": len(pool),
                   "budget_bits": w.budget, "correlated_rounding": w.correlated, "grad_gb_per_worker": gb,
                   "parallelism": f"replicas x{world} (all simulated workers on each GPU)",
                   "l2": "each pass streams 8 x 16 GB of gradients through the pool; one bucket's working set "
                         "(about 0.6 GB) exceeds L2"},
        "per_bucket_ms": ms_max / nb,
        "exchange": ("pipelined across buckets (N + 1 buckets per launch; planning "
                     f"{ov.lookahead} buckets ahead on a second stream with {ov.plan_sms} SMs left to it)"
                     if piped else ("one cooperative launch per bucket" if ov.fused else "one launch per step")),
        "per_bucket_stream": {"ms_per_pass": ms_alt if piped else ms,
                              "exchange": "one cooperative launch per bucket" if per_bucket.fused
                              else "one launch per step",
                              "note": "the next bucket's planning on a second stream"},
        "one_stream": {"ms_per_pass": ms_seq, "note": "per-bucket rounds, one launch per step, no overlap"},
        "kernels": kernels, "ms_per_step_logged": ms_logged, "roofline": roofline,
        "gpu_launches": n_launch, "clocks": clk, "cpu_baseline": cpu, "e2e": e2e,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def bucketed_e2e(args, w, ar, pool, pool_of, outs_pool, nb, dev, world, gb):
    """End to end over a full pass: every bucket's N gradients are uploaded
    from pinned host memory (a host copy of the resident pool) into one of the
    stream's device staging sets on a copy stream, later buckets' uploads and
    planning overlapping earlier buckets' exchange; rank 0's fp32 result of
    every bucket is downloaded on a third stream.  All copies are inside the
    timed region.  The bucket stream enqueues the copies itself
    (dq_allreduce_stream_io); the per-bucket stream through its hooks."""
    import torch

    N = w.n_ranks
    flat = pinned_host_copies([g for b in pool for g in b])
    hosts = [flat[i * N:(i + 1) * N] for i in range(len(pool))]
    out_host = [torch.empty(o[0].numel(), dtype=torch.float32, pin_memory=True) for o in outs_pool]
    # a bucket's gradients are read until its last ring step: the pipelined
    # stream keeps `depth` buckets in flight, the per-bucket stream two
    S = getattr(ar, "depth", 2)
    stage = [[torch.empty(g.numel(), dtype=g.dtype, device=dev) for g in pool[0]] for _ in range(S)]
    stage_last = [[torch.empty(g.numel(), dtype=g.dtype, device=dev) for g in pool[-1]] for _ in range(S)]
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(N)] for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(len(outs_pool))]
    ev_exch = [torch.cuda.Event() for _ in range(nb)]
    P = len(outs_pool)
    last = nb - 1
    bufs = [stage_last[k % S] if k == last else stage[k % S] for k in range(nb)]
    outs = [outs_pool[pool_of[k]] for k in range(nb)]

    def before_plan(k, side):
        cin.wait_stream(side)                       # the staging set's previous bucket has finished
        with torch.cuda.stream(cin):
            for r in range(N):
                bufs[k][r].copy_(hosts[pool_of[k]][r], non_blocking=True)
                ev_in[k][r].record(cin)

    def before_exchange(k, main):
        main.wait_event(ev_out[pool_of[k]])         # this output buffer's last download has finished

    def after_exchange(k, main):
        ev_exch[k].record(main)
        cout.wait_event(ev_exch[k])
        with torch.cuda.stream(cout):
            out_host[pool_of[k]].copy_(outs[k][0], non_blocking=True)
            ev_out[pool_of[k]].record(cout)

    # the bucket stream stages natively: the library enqueues every upload and
    # download itself (dq_allreduce_stream_io), no Python per bucket
    native = hasattr(ar, "copy_streams")
    if native:
        src = [hosts[pool_of[k]] for k in range(nb)]
        dst = [out_host[pool_of[k]] for k in range(nb)]

    def one_pass(first):
        if native:
            ar.run(bufs, outs, round0=first * nb, src_host=src, dst_host=dst, copy_in=cin, copy_out=cout)
            return
        ar.run(bufs, outs, round0=first * nb, ready=ev_in, before_plan=before_plan,
               before_exchange=before_exchange, after_exchange=after_exchange)
        torch.cuda.current_stream().wait_stream(cout)

    # the host link's rate on this machine now: plain uploads of the pool's host
    # copies into the staging sets (the first round warms the path)
    link = []
    for _ in range(2):
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(cin)
        with torch.cuda.stream(cin):
            for i in range(len(pool)):
                into = stage_last[0] if i == len(pool) - 1 else stage[i % S]
                for r in range(N):
                    into[r].copy_(hosts[i][r], non_blocking=True)
        l1.record(cin)
        cin.synchronize()
        link.append(l0.elapsed_time(l1))
    link_gbs = sum(g.numel() * 2 for b in pool for g in b) / (link[-1] * 1e-3) / 1e9
    one_pass(1_000)
    torch.cuda.synchronize()
    barrier(world, dev)
    KE = args.e2e_steps or 2
    main = torch.cuda.current_stream()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(main)
    cin.wait_event(f0)
    for i in range(KE):
        one_pass(1_001 + i)
    f1.record(main)
    torch.cuda.synchronize()
    barrier(world, dev)
    ms = max_over_ranks(f0.elapsed_time(f1) / KE, world, dev)
    h2d = sum(sum(g.numel() * 2 for g in pool[pool_of[k]]) for k in range(nb))
    d2h = sum(outs_pool[pool_of[k]][0].numel() * 4 for k in range(nb))
    del hosts, out_host, stage, stage_last
    return {"value": ms / (world * gb), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": KE, "h2d_gbs": h2d / (ms * 1e-3) / 1e9,
            "link_gbs": link_gbs, "link_floor_ms": h2d / (link_gbs * 1e9) * 1e3,
            "link_note": "link_gbs: a plain upload of the pool's pinned buffers timed just before; "
                         "link_floor_ms: the upload of every bucket at that rate, which bounds the pass (the link's "
                         "rate varies from box to box and over time on some)",
            "staging": "copies enqueued by the library (dq_allreduce_stream_io)" if native
                       else "copies enqueued by Python hooks per bucket"}


def bucketed_cpu_baseline(w, nb: int, gb: float):
    """The oracle, as it stands, on three buckets of the streamed workload
    (the first, the middle one and the last), its time extrapolated to all
    buckets by coordinates."""
    from quantized_hop_gradient_gb300 import synth
    ks = sorted({0, nb // 2, nb - 1})
    secs = 0.0
    coords = 0
    for k in ks:
        gu = [synth.as_u16(g) for g in synth.generate_bucket(w, k, "cpu", seed=0)]
        secs += oracle_allreduce_seconds(w, gu, round_=k)
        coords += gu[0].size
    total = secs * (w.n_pad / coords)
    return {"value": total * 1e3 / gb, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"buckets {', '.join(str(k) for k in ks)} of {nb} ({coords} coordinates per worker, "
                      f"{secs:.1f} s), extrapolated to the {w.n_pad} coordinates of a full pass"}


# --------------------------------------------------------------------------- the reference arm (oracle)
def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is the oracle's
    whole all-reduce over a bounded sample of the same workload."""
    if rank != 0:
        return
    from quantized_hop_gradient_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.coords:
        w = w.scaled(args.coords)
    K, W = args.steps, max(args.warmup, 0)
    per_step = max(0.5, min(8.0, 150.0 / max(1, K + W)))
    full = None

    def slices(n):
        nonlocal full
        if full is None or full[0].size < n:
            full = [synth.as_u16(g) for g in synth.generate(w.scaled(max(n, 1 << 18)), "cpu", seed=0)]
        return [f[:n] for f in full]

    n = calibrated_sample(w, slices, per_step)
    gu = slices(n)
    for i in range(W):
        oracle_allreduce_seconds(w, gu, round_=i)
    t = time.perf_counter()
    for i in range(K):
        oracle_allreduce_seconds(w, gu, round_=W + i)
    secs = (time.perf_counter() - t) / K
    gb = n * 2 / 1e9
    value = secs * 1e3 / gb
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": secs * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, fp32 codec, 2/4/8-bit codes", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "simulated_workers": w.n_ranks, "topology": w.topology,
                   "coords_per_worker": w.n, "budget_bits": w.budget, "correlated_rounding": w.correlated},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                         "sample": f"first {n} of {w.n_pad} coordinates of each of the {w.n_ranks} workers "
                                   f"per step, whole oracle all-reduce"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world, local)
    if world > 1:
        import torch.distributed as td
        td.destroy_process_group()


if __name__ == "__main__":
    main()
