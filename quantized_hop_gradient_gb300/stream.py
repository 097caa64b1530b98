"""Bucketed (DDP-style) all-reduce of a large gradient on one GPU.

The gradient of every simulated worker is cut into buckets of a fixed number
of super-groups, as DDP cuts it into communication buckets; each bucket is
one DynamiQ round with its own statistics, allocation, reordering, hops and
decode.  Bucket k+1's planning runs on a second CUDA stream while bucket k's
hops and decode run on the first; two buffer sets alternate between buckets,
ordered by events.
"""
from __future__ import annotations

import torch

from .allreduce import DynamiQAllReduce, use_fused


class BucketedAllReduce:
    def __init__(self, n_ranks: int, bucket_sg: int, *, overlap: bool = True, fused="auto", **kw):
        """``fused``: each bucket's ring exchange as one cooperative launch
        (dq_exchange_fused): True, False, or "auto", which follows
        ``use_fused``.  The one-launch exchange wins with or without the
        overlap: 25 MB buckets of an 8-rank ring took 0.322 ms each against
        0.373 with per-step launches, the next bucket's planning on the
        second stream in both."""
        self.n_ranks, self.bucket_sg, self.overlap = n_ranks, bucket_sg, overlap
        if fused == "auto":
            fused = use_fused(n_ranks, kw.get("butterfly", False), bucket_sg)
        self.fused = bool(fused)
        self.sets = [DynamiQAllReduce(n_ranks, bucket_sg, **kw) for _ in range(2)]
        self.plan_stream = torch.cuda.Stream() if overlap else None
        self.ev_plan = [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_done = [torch.cuda.Event(), torch.cuda.Event()]

    def run(self, buckets, outs, round0: int = 0, log=None, ready=None, before_plan=None, before_exchange=None,
            after_exchange=None):
        """buckets[k][r]: rank r's bf16 gradient of bucket k (device, a multiple
        of 256 coordinates, at most bucket_sg super-groups); outs[k][r]: where
        rank r's fp32 (or bf16) result of bucket k goes.  Returns the plan
        infos of the buckets.

        Optional: ``log`` (a dq.LaunchLog) records every launch; ``ready[k]``
        is a list of per-rank events that bucket k's statistics wait on (e.g.
        its upload); the hooks are called with (k, stream) just before bucket
        k's planning is enqueued (on the planning stream, after it waited for
        the buffer set's previous bucket), before its exchange and after it
        (on the exchange stream), so a caller can enqueue copies in order."""
        main = torch.cuda.current_stream()
        side = self.plan_stream if self.overlap else main
        infos = []

        def plan(k):
            s = k & 1
            n_sg = buckets[k][0].numel() // 256
            side.wait_event(self.ev_done[s])           # the set's previous bucket has finished
            if before_plan is not None:
                before_plan(k, side)
            with torch.cuda.stream(side):
                infos.append(self.sets[s].plan(buckets[k], round=round0 + k, n_sg=n_sg, log=log,
                                               ready=None if ready is None else ready[k]))
                self.ev_plan[s].record(side)

        plan(0)
        for k in range(len(buckets)):
            s = k & 1
            main.wait_event(self.ev_plan[s])
            if before_exchange is not None:
                before_exchange(k, main)
            self.sets[s].exchange(buckets[k], outs[k], round=round0 + k, fused=self.fused, log=log)
            self.ev_done[s].record(main)
            if after_exchange is not None:
                after_exchange(k, main)
            if k + 1 < len(buckets):
                plan(k + 1)
        return infos
