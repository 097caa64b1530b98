"""N simulated ranks on one GPU: one DynamiQ all-reduce round per call.

Holds the device buffers of the planning and exchange phases and calls the
two schedule entry points of libdq (``dq_plan``, ``dq_exchange``).  The
workers' gradients are device tensors; a "hop" is a message buffer handed
from one simulated rank to the next inside the exchange workspace.
"""
from __future__ import annotations

import math

import torch

from . import dq

SG = dq.SG

# Largest per-worker size (super-groups) at which the fused ring exchange is
# the faster one on a GB300 (BERT-large distribution, exchange alone, ms):
# at 2^16 super-groups 0.164 / 0.315 / 0.617 for rings of 4 / 8 / 16 against
# 0.228 / 0.436 / 0.866 pipelined (one part) and 0.174 / 0.344 / 0.690 step
# by step; at 1.25 * 2^16 the fused exchange jumps to 0.278 / 0.543 / 1.074
# (its messages no longer stay in L2) and the one-part pipeline leads with
# 0.241 / 0.468 / 0.931.
FUSED_MAX_SG = 1 << 16


def use_fused(n_ranks: int, butterfly: bool, n_sg: int) -> bool:
    """Whether the ring exchange should run as one cooperative launch."""
    return (not butterfly) and n_ranks <= dq.MAX_FUSED_RANKS and n_sg <= FUSED_MAX_SG


def pipeline_parts(n_ranks: int, n_sg: int) -> int:
    """Parts of the pipelined ring exchange.  More parts shorten the first
    N launches, which carry hop steps only (no part has finished its ring
    yet), to (N + 1) / 2P of the hop work; each part adds a launch.  The
    best count measured on a GB300 (exchange alone) grows like N times the
    square root of the work units (32 super-groups each): N = 8: 16,385
    units 4 (4 to 8 within 0.5%), 32,769 units 12, 40,911 (BERT-large)
    8 to 10 (16: 2.3% slower), 65,537 units 16; N = 16: 32,769 units 24,
    65,537 units 32, 122,057 (Gemma-1B) 32 to 40.  Up to 16,384 units one
    part is best (8,193 units: 1.013 ms at one part, 1.026 at four, N = 8).
    At most 2N parts."""
    units = -(-n_sg // dq.UNIT)
    if units <= 16384:
        return 1
    return max(1, min(2 * n_ranks, round(n_ranks * math.sqrt(units) / 144), dq.MAX_WAVE_PARTS))


def exchange_mode(n_ranks: int, butterfly: bool, n_sg: int):
    """(fused, parts) of the ring exchange that is fastest at this size: one
    cooperative launch up to FUSED_MAX_SG super-groups per worker, the
    pipelined exchange above (rings of up to 64 ranks); the butterfly runs
    step by step: (False, None)."""
    if butterfly or n_ranks > dq.MAX_FUSED_RANKS:
        return False, None
    if n_sg <= FUSED_MAX_SG:
        return True, None
    return False, pipeline_parts(n_ranks, n_sg)


class DynamiQAllReduce:
    def __init__(self, n_ranks: int, n_sg: int, *, budget: float = 5.0, eps: float = 1.0,
                 correlated: bool = True, butterfly: bool = False, seed: int = 0,
                 out_dtype: torch.dtype = torch.float32, device="cuda", fixed_bits: int = 0,
                 scale_fp32: bool = False):
        """``fixed_bits`` (2/4/8) and ``scale_fp32`` are ablation switches:
        uniform bitwidth instead of the allocation, fp32 group scales instead
        of the UINT8 second level."""
        self.n_ranks, self.n_sg = n_ranks, n_sg
        self.budget, self.eps, self.correlated, self.butterfly = budget, eps, correlated, butterfly
        self.seed = seed
        self.fixed_bits, self.scale_fp32 = fixed_bits, scale_fp32
        self.out_dtype = out_dtype
        self.device = torch.device(device)
        dq.lib()
        self.mu = torch.empty(n_sg, dtype=torch.float32, device=self.device)
        self.perm = torch.empty(n_sg, dtype=torch.int32, device=self.device)
        nb = dq.dq_plan_workspace_bytes(n_ranks, n_sg)
        self.plan_ws = torch.empty(nb, dtype=torch.uint8, device=self.device)
        self.ws = torch.empty(0, dtype=torch.uint8, device=self.device)
        self.info = None
        self.final = None
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def config(self, round: int = 0):
        return dq.config(self.n_ranks, self.budget, self.eps, self.correlated, self.seed, round,
                         self.fixed_bits, self.scale_fp32)

    def plan(self, grads, round: int = 0, stream=None, log=None, ready=None, n_sg=None):
        """Statistics, allocation and reordering.  ``ready``: optional
        per-rank events the statistics of each rank wait on.  ``n_sg``: a
        smaller super-group count than the buffers were sized for."""
        cfg = self.config(round)
        self.cur_sg = n_sg or self.n_sg
        if self.cur_sg > self.n_sg:
            raise ValueError("more super-groups than the buffers hold")
        self.info = dq.dq_plan(cfg, grads, self.cur_sg, self.mu, self.perm, self.plan_ws, self.plan_ws.numel(),
                               log, stream, ready)
        return self.info

    def reserve(self, nbytes: int):
        if self.ws.numel() < nbytes:
            self.ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)

    def exchange(self, grads, outs, round: int = 0, stream=None, log=None, fused="auto", parts=None):
        """``fused``: True runs the ring exchange as one cooperative launch
        (ring, at most 64 ranks); its device status is in ``self.status``
        (check with ``check_status`` after synchronising).  ``parts``: run
        the ring exchange pipelined over that many parts of the super-groups
        (``dq_exchange_pipelined``) instead.  ``fused="auto"`` with no
        ``parts`` picks the faster path for the size (``exchange_mode``)."""
        cfg = self.config(round)
        n_sg = getattr(self, "cur_sg", self.n_sg)
        bf16 = self.out_dtype == torch.bfloat16
        if fused == "auto" and parts is None:
            fused, parts = exchange_mode(self.n_ranks, self.butterfly, n_sg)
        if parts is not None:
            if self.butterfly:
                raise ValueError("the pipelined exchange is the ring's")
            need = dq.dq_exchange_pipelined_workspace_bytes(cfg, n_sg, self.info)
            if need == 0:
                raise dq.DQError(dq.DQ_ERR_INVALID_ARG, "dq_exchange_pipelined_workspace_bytes")
            self.reserve(need)
            self.final = dq.dq_exchange_pipelined(cfg, grads, n_sg, self.mu, self.perm, self.info, self.ws,
                                                  self.ws.numel(), outs, parts, bf16, log, stream)
            return outs
        if fused:
            if self.butterfly:
                raise ValueError("the fused exchange is the ring's")
            need = dq.dq_exchange_fused_workspace_bytes(cfg, n_sg, self.info)
            if need == 0:
                raise dq.DQError(dq.DQ_ERR_INVALID_ARG, "dq_exchange_fused_workspace_bytes")
            self.reserve(need)
            self.final = dq.dq_exchange_fused(cfg, grads, n_sg, self.mu, self.perm, self.info, self.ws,
                                              self.ws.numel(), outs, self.status, bf16, log, stream)
            return outs
        need = dq.dq_exchange_workspace_bytes(cfg, self.butterfly, n_sg, self.info)
        if need == 0:
            raise dq.DQError(dq.DQ_ERR_INVALID_ARG, "dq_exchange_workspace_bytes")
        self.reserve(need)
        self.final = dq.dq_exchange(cfg, self.butterfly, grads, n_sg, self.mu, self.perm, self.info,
                                    self.ws, self.ws.numel(), outs, bf16, log, stream)
        return outs

    def check_status(self):
        """Raises if the last fused exchange reported a device error."""
        s = dq.dq_get_device_status(self.status)
        if s != dq.DQ_DEVICE_OK:
            raise RuntimeError(f"fused exchange: device status {s} (barrier timeout)")

    def new_outputs(self):
        return [torch.empty(self.n_sg * SG, dtype=self.out_dtype, device=self.device)
                for _ in range(self.n_ranks)]

    def __call__(self, grads, round: int = 0, outs=None, stream=None, fused="auto", parts=None):
        if len(grads) != self.n_ranks:
            raise ValueError("one gradient per rank")
        if outs is None:
            outs = self.new_outputs()
        self.plan(grads, round, stream)
        return self.exchange(grads, outs, round, stream, fused=fused, parts=parts)

    def chunk_lo(self):
        i = self.info
        return dq.dq_chunk_cuts(i.n2, i.n4, i.n8, self.n_ranks)

    def final_message(self, c: int) -> torch.Tensor:
        """Copy of the final message of chunk c (device bytes -> host uint8)."""
        lo = self.chunk_lo()
        i = self.info
        r = dq.rng(lo[c], lo[c + 1], i.n2, i.n2 + i.n4)
        nb = dq.dq_message_bytes(r, self.scale_fp32)
        off = self.final[c] - self.ws.data_ptr()
        return self.ws[off:off + nb].cpu()


class MXFP8AllReduce:
    """The MXFP8 comparison baseline over the same N-rank schedules: every
    hop decodes, adds in fp32 and re-encodes 32-element E4M3 blocks with an
    E8M0 scale (OCP MX v1.0).  Outputs are fp32 sums."""

    def __init__(self, n_ranks: int, n_coords: int, *, butterfly: bool = False, device="cuda"):
        if n_coords % dq.MX_BLOCK:
            raise ValueError("the coordinate count must be a multiple of 32")
        self.n_ranks, self.n_blk, self.butterfly = n_ranks, n_coords // dq.MX_BLOCK, butterfly
        self.device = torch.device(device)
        dq.lib()
        nb = dq.dq_mx_exchange_workspace_bytes(n_ranks, butterfly, self.n_blk)
        if nb == 0:
            raise dq.DQError(dq.DQ_ERR_INVALID_ARG, "dq_mx_exchange_workspace_bytes")
        self.ws = torch.empty(nb, dtype=torch.uint8, device=self.device)
        self.final = None

    def chunk_lo(self):
        return [c * self.n_blk // self.n_ranks for c in range(self.n_ranks + 1)]

    def new_outputs(self):
        return [torch.empty(self.n_blk * dq.MX_BLOCK, dtype=torch.float32, device=self.device)
                for _ in range(self.n_ranks)]

    def __call__(self, grads, outs=None, stream=None, log=None):
        if len(grads) != self.n_ranks:
            raise ValueError("one gradient per rank")
        if outs is None:
            outs = self.new_outputs()
        self.final = dq.dq_mx_exchange(self.n_ranks, self.butterfly, grads, self.n_blk, self.ws,
                                       self.ws.numel(), outs, log, stream)
        return outs

    def final_message(self, c: int) -> torch.Tensor:
        lo = self.chunk_lo()
        nb = dq.dq_mx_message_bytes(lo[c + 1] - lo[c])
        off = self.final[c] - self.ws.data_ptr()
        return self.ws[off:off + nb].cpu()
