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
DEFAULT_WORKLOAD = "bert_large_ring8"
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
    p.add_argument("--exchange", choices=["auto", "fused", "multi"], default="auto",
                   help="ring exchange as one cooperative launch (fused) or one launch per step (multi); "
                        "auto: fused where it is the faster path (allreduce.use_fused: rings of up to 64 ranks, up to 2^17 "
                        "super-groups per worker)")
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
def stream_message_bytes(dq, info, N):
    lo = dq.dq_chunk_cuts(info.n2, info.n4, info.n8, N)
    e2, e4 = info.n2, info.n2 + info.n4
    return sum(dq.dq_message_bytes(dq.rng(lo[c], lo[c + 1], e2, e4)) for c in range(N))


def launch_bytes(kind: int, sgs: int, msg_per_sg: float, fp32_addend: bool = False, n_ranks: int = 1) -> float:
    """Algorithmic HBM bytes of one launch over `sgs` super-groups: every
    input byte read once and every output byte written once, nothing else.
    compress: bf16 gradient 512 B/SG + message out + mean and perm 8 B/SG;
    DAR: message in + addend (512 B/SG bf16, 1 KiB fp32) + message out + 8 B/SG;
    decode: fp32 output 1 KiB per super-group written, message in + 8 B per
    super-group read (once for up to 16 outputs);
    stats: bf16 gradient 512 B/SG + mean and squared norm 8 B/SG;
    allocate + reorder span: N x 8 B/SG of statistics read, M, F, mu written
    (12 B/SG), then about five passes over F (20 B/SG) and the bitwidths and
    permutation (about 7 B/SG); fused ring exchange: the compress, N-1 DARs
    and a decode that reads each message once and writes N outputs."""
    if kind == 0:
        return sgs * (512 + msg_per_sg + 8)
    if kind == 1:
        return sgs * (2 * msg_per_sg + (1024 if fp32_addend else 512) + 8)
    if kind == 2:   # sgs = super-groups written; each launch reads a message once for up to 16 outputs
        return sgs * 1024 + sgs / min(n_ranks, 16) * (msg_per_sg + 8)
    if kind == 3:
        return sgs * (512 + 8)
    if kind == 7:   # fused ring: sgs = J (N + 1); compress, N - 1 DARs, one decode read, N outputs
        J = sgs / (n_ranks + 1)
        return J * ((512 + msg_per_sg + 8) + (n_ranks - 1) * (2 * msg_per_sg + 512 + 8) +
                    (msg_per_sg + 8 + 1024 * n_ranks))
    return sgs * (8 * n_ranks + 12 + 20 + 7)


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
def run_gpu(args, rank, world, local):
    import torch

    from quantized_hop_gradient_gb300 import dq, synth
    from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce, use_fused

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
    N, J = w.n_ranks, w.n_sg
    butterfly = w.topology == "butterfly"
    grads = synth.generate(w, dev, seed=0)
    ar = DynamiQAllReduce(N, J, budget=w.budget, correlated=w.correlated, butterfly=butterfly, seed=0)
    outs = ar.new_outputs()
    K, W = args.steps, max(args.warmup, 0)
    fusable = not butterfly and N <= dq.MAX_FUSED_RANKS
    fused = use_fused(N, butterfly, J) if args.exchange == "auto" else (args.exchange == "fused")
    if fused and not fusable:
        raise SystemExit("the fused exchange covers rings of up to 64 ranks")

    def step(i, log=None, fused=fused):
        ar.plan(grads, round=i, log=log)
        ar.exchange(grads, outs, round=i, log=log, fused=fused)

    def measure(fused_, steps, first, sample_clocks=False):
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
            step(first + i, log, fused_)
        e1.record()
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world, dev)
        if fused_:
            ar.check_status()
        clk = clocks.stop(t0, t1) if clocks else None
        return e0.elapsed_time(e1) / steps, log, dq.dq_launch_count() - n0, clk

    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    ms, log, n_launch, clk = measure(fused, K, W, sample_clocks=True)
    ms_max = max_over_ranks(ms, world, dev)

    # per-launch times of the recorded kernels
    msg_total = stream_message_bytes(dq, ar.info, N)
    msg_per_sg = msg_total / J
    names = {0: "compress", 1: "dar", 2: "decode", 3: "stats", 4: "allocate_reorder", 7: "fused_ring"}

    def per_kernel(log_, steps, ms_step):
        per_kind = {}
        for kind, sgs, t in log_.launches():
            d = per_kind.setdefault(kind, {"launches": 0, "ms": 0.0, "sgs": 0, "bytes": 0.0})
            d["launches"] += 1
            d["ms"] += t
            d["sgs"] += sgs
            d["bytes"] += launch_bytes(kind, sgs, msg_per_sg, fp32_addend=False, n_ranks=N)
        out = {}
        for kind, d in per_kind.items():
            avg_ms = d["ms"] / d["launches"]
            gbs = d["bytes"] / d["launches"] / (avg_ms * 1e-3) / 1e9
            out[names[kind]] = {"launches_per_step": d["launches"] / steps, "avg_launch_ms": avg_ms,
                                "share_of_step": d["ms"] / steps / ms_step,
                                "alg_bytes_per_launch": d["bytes"] / d["launches"], "achieved_gbs": gbs,
                                "gcoords_per_s": d["sgs"] / d["launches"] * SG / (avg_ms * 1e-3) / 1e9}
        return out

    peak, peak_kind = measured_peaks()
    kernels = per_kernel(log, K, ms)
    kernels_multi = None
    ms_multi = None
    if fused:
        # the per-step kernels of the multi-launch exchange, for the hop breakdown
        step(W + K, None, False)
        KM = max(3, min(K, 10))
        ms_multi, log_m, _, _ = measure(False, KM, W + K + 1)
        kernels_multi = per_kernel(log_m, KM, ms_multi)
    dominant = max((k for k in kernels if k != "allocate_reorder"), key=lambda k: kernels[k]["share_of_step"])
    dk = kernels[dominant]
    kname = {"compress": "hop_kernel<false,false>", "dar": "hop_kernel<true,false>", "decode": "decode_kernel",
             "stats": "stats_kernel", "fused_ring": "fused_ring_kernel"}
    traffic, _ = ncu_counters(kname[dominant], w.name)
    roofline = {"bound": "hbm", "kernel": kname[dominant], "achieved": dk["achieved_gbs"], "peak": peak,
                "unit": "GB/s", "frac": dk["achieved_gbs"] / peak, "peak_source": peak_kind,
                "traffic": traffic, "alg_bytes_per_launch": dk["alg_bytes_per_launch"]}
    dar = (kernels_multi or kernels).get("dar", {})
    # The DAR hop is bound by instruction issue, not HBM: its issue roofline
    # (warp-instructions per super-group from the committed ncu capture,
    # times super-groups per launch, over the measured launch time) against
    # 4 issue slots per SM per cycle at the maximum SM clock.
    dar_issue = None
    _, inst_per_sg = ncu_counters("hop_kernel<true,false>", w.name)
    if dar and inst_per_sg:
        sm_mhz = 2070.0
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                sm_mhz = float(json.load(f).get("sm_max_mhz", sm_mhz))
        except Exception:
            pass
        issue_peak = 4 * torch.cuda.get_device_properties(dev).multi_processor_count * sm_mhz * 1e6
        sgs = dar["gcoords_per_s"] * 1e9 / SG * dar["avg_launch_ms"] * 1e-3
        achieved = inst_per_sg * sgs / (dar["avg_launch_ms"] * 1e-3)
        dar_issue = {"bound": "alu", "achieved": achieved / 1e12, "peak": issue_peak / 1e12,
                     "unit": "T warp-instructions/s", "frac": achieved / issue_peak,
                     "warp_instructions_per_super_group": inst_per_sg}
    gb = J * SG * 2 / 1e9

    # End to end: the gradients start in pinned host memory and rank 0's fp32
    # result ends there; every copy is inside the timed region.  Round i+1's
    # upload (copy stream) runs while round i computes, into the other of two
    # device gradient buffers; each rank's statistics wait only for that
    # rank's upload; the result download runs on a third stream.
    KE = args.e2e_steps or max(3, min(K, 10))
    hosts = [torch.empty(g.numel(), dtype=torch.bfloat16, pin_memory=True) for g in grads]
    for h, g in zip(hosts, grads):
        h.copy_(g)
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
        ar.exchange(gbuf[b], outs, round=i, fused=fused)
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

    accuracy, mxfp8 = compare_mxfp8(args, w, grads, outs, ar, dev, N, J, butterfly, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, grads, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": ms_max / (world * gb), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_max, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 codec, 2/4/8-bit codes", "data": "synthetic (seeded; see DESIGN.md)",
        "config": {"workload": w.name, "simulated_workers": N, "topology": w.topology,
                   "coords_per_worker": w.n, "super_groups": J, "budget_bits": w.budget,
                   "correlated_rounding": w.correlated, "grad_gb_per_worker": gb,
                   "parallelism": f"replicas x{world} (all simulated workers on each GPU)",
                   "l2": "inputs larger than L2 (no flush needed)",
                   "allocation": {"T": ar.info.T, "n2": ar.info.n2, "n4": ar.info.n4, "n8": ar.info.n8}},
        "dar": {"gcoords_per_s_per_hop": dar.get("gcoords_per_s"), "achieved_gbs": dar.get("achieved_gbs"),
                "hbm_frac": (dar["achieved_gbs"] / peak) if dar else None, "avg_launch_ms": dar.get("avg_launch_ms"),
                "issue_roofline": dar_issue},
        "exchange": "fused (one cooperative launch per round)" if fused else "one launch per step",
        "kernels": kernels,
        "kernels_multi_launch": kernels_multi,
        "ms_per_step_multi_launch": ms_multi,
        "roofline": roofline,
        "e2e": {"value": ms_e2e / (world * gb), "unit": UNIT, "h2d_bytes_per_step": N * J * SG * 2,
                "d2h_bytes_per_step": J * SG * 4, "ms_per_step": ms_e2e},
        "gpu_launches": n_launch,
        "clocks": clk,
        "accuracy": accuracy,
        "mxfp8": mxfp8,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def compare_mxfp8(args, w, grads, outs, ar, dev, N, J, butterfly, peak):
    """After the timed region: the vNMSE of the last DynamiQ round and of
    the MXFP8 baseline on the same gradients, and the MXFP8 all-reduce's
    time on the same GPU (its hops read 1 + 1/32 B of message, 2 B of bf16
    gradient and write 1 + 1/32 B per coordinate)."""
    import torch

    from quantized_hop_gradient_gb300 import dq, study
    from quantized_hop_gradient_gb300.allreduce import MXFP8AllReduce

    s = study.exact_sum(grads)
    v_dq = study.vnmse(outs[0], s)
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
    v_mx = study.vnmse(outs[0], s)
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
    msg = stream_message_bytes(dq, ar.info, N) / (J * SG)
    return ({"vnmse": v_dq, "vnmse_mxfp8": v_mx, "mxfp8_over_dynamiq": v_mx / v_dq if v_dq > 0 else None,
             "wire_bytes_per_coord": msg, "rounds_measured": 1}, mx_line)


# --------------------------------------------------------------------------- streamed workloads
def run_gpu_bucketed(args, rank, world, local, w, dev):
    """A streamed workload (DDP buckets): one step is a full pass over the
    model's buckets, each bucket a DynamiQ round; bucket k+1's planning runs
    on a second stream under bucket k's hops.  The gradient data cycle
    through a pool of resident buckets drawn from across the model (the
    whole model does not fit in HBM with every worker's copy)."""
    import torch

    from quantized_hop_gradient_gb300 import dq, synth
    from quantized_hop_gradient_gb300.stream import BucketedAllReduce

    N = w.n_ranks
    nb = synth.bucket_count(w)
    P = max(2, min(args.bucket_pool, nb))
    picks = sorted({round(i * (nb - 2) / (P - 2)) for i in range(P - 1)}) + [nb - 1]
    pool = [synth.generate_bucket(w, k, dev, seed=0) for k in picks]
    full, last = pool[:-1], pool[-1]
    seq = [full[i % len(full)] for i in range(nb - 1)] + [last]
    outs_pool = [[torch.empty(g.numel(), dtype=torch.float32, device=dev) for g in b] for b in pool]
    seq_out = [outs_pool[i % len(full)] for i in range(nb - 1)] + [outs_pool[-1]]
    bucket_sg = w.bucket // SG
    kw = dict(budget=w.budget, correlated=w.correlated, butterfly=w.topology == "butterfly", seed=0)
    # the overlapped stream picks its exchange itself ("auto": the cooperative
    # one-launch exchange for rings of up to 64 ranks and 2^17 super-groups);
    # the other exchange is timed beside it for comparison
    from quantized_hop_gradient_gb300.allreduce import use_fused
    fusable = use_fused(N, w.topology == "butterfly", bucket_sg)
    ov = BucketedAllReduce(N, bucket_sg, overlap=True, fused="auto", **kw)
    alt = BucketedAllReduce(N, bucket_sg, overlap=True, fused=not ov.fused, **kw) \
        if (fusable or ov.fused) else None
    sq = BucketedAllReduce(N, bucket_sg, overlap=False, fused=False, **kw)
    K, W = args.steps, max(args.warmup, 0)

    def timed(ar, steps, first):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(world, dev)
        e0.record()
        for i in range(steps):
            ar.run(seq, seq_out, round0=(first + i) * nb)
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
    if ov.fused:
        for s_ in ov.sets:
            s_.check_status()
    sq.run(seq, seq_out, round0=(W + K) * nb)          # warm-up pass (workspace allocation)
    ms_seq = timed(sq, 1, W + K + 1)
    ms_alt = None
    if alt is not None:
        alt.run(seq, seq_out, round0=(W + K + 2) * nb)
        ms_alt = timed(alt, 2, W + K + 3)
        if alt.fused:
            for s_ in alt.sets:
                s_.check_status()
    ms_fused = ms if ov.fused else ms_alt
    ms_ml = ms_alt if ov.fused else ms
    ms_max = max_over_ranks(ms, world, dev)
    gb = w.n * 2 / 1e9
    line = {
        "metric": METRIC, "value": ms_max / (world * gb), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 codec, 2/4/8-bit codes", "data": "synthetic (seeded; see DESIGN.md)",
        "config": {"workload": w.name, "simulated_workers": N, "topology": w.topology, "coords_per_worker": w.n,
                   "bucket_coords": w.bucket, "buckets": nb, "resident_bucket_pool": len(pool),
                   "budget_bits": w.budget, "correlated_rounding": w.correlated, "grad_gb_per_worker": gb,
                   "parallelism": f"replicas x{world} (all simulated workers on each GPU)",
                   "l2": "inputs larger than L2 (no flush needed)"},
        "per_bucket_ms": ms_max / nb,
        "two_streams": {"ms_per_pass_overlapped": ms, "ms_per_pass_one_stream": ms_seq,
                        "saved_frac": 1.0 - ms / ms_seq},
        "fused_exchange": {"used": ov.fused, "ms_per_pass_fused": ms_fused, "ms_per_pass_multi_launch": ms_ml},
        "gpu_launches": n_launch, "clocks": clk, "cpu_baseline": None, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


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
