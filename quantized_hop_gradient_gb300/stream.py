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


class BucketStream:
    """The bucket stream with the ring exchange pipelined across buckets
    (``dq_exchange_stream_step``): launch t runs ring step t - b of every
    bucket b in flight and the final decode of bucket t - N, so the N + 1
    buckets in flight fill the GPU where one 25 MB bucket's step cannot.
    Each bucket is planned by ``dq_plan_async`` on a second, higher-priority
    stream, one bucket ahead; its 2/4/8 counts stay on the device, so the
    host never waits for a plan.  ``depth`` buffer sets (plan outputs and
    messages) rotate over the buckets; a set is reused once its previous
    bucket's decode has finished.  Rings of up to 8 ranks."""

    def __init__(self, n_ranks: int, bucket_sg: int, *, budget: float = 5.0, eps: float = 1.0,
                 correlated: bool = True, seed: int = 0, out_dtype=torch.float32, device="cuda",
                 fixed_bits: int = 0, scale_fp32: bool = False, depth: int = 0, lookahead: int = 3,
                 plan_sms: int = -1):
        from . import dq
        if n_ranks > dq.MAX_STREAM_RANKS:
            raise ValueError("the bucket stream covers rings of up to 8 ranks")
        self.dq = dq
        self.n_ranks, self.bucket_sg = n_ranks, bucket_sg
        self.budget, self.eps, self.correlated, self.seed = budget, eps, correlated, seed
        self.fixed_bits, self.scale_fp32 = fixed_bits, scale_fp32
        self.out_is_bf16 = out_dtype == torch.bfloat16
        # N + 1 buckets in the exchange at once and `lookahead` planned ahead.
        # The planning (its statistics read every rank's bucket) runs beside
        # the exchange on SMs the exchange's launches leave free.  Measured
        # on the Llama-3-8B stream of 8 ranks (613 buckets of 25 MB, ms per
        # pass), lookahead 3: with 8 to 28 of 152 SMs left free, 125.1 to
        # 127.3; with 32, 137.8; with 40, 143.7.  Lookahead 2 and 4 measure
        # the same as 3.  The ratio of planning to exchange work does not
        # depend on N.
        if plan_sms < 0:
            sms = torch.cuda.get_device_properties(torch.device(device)).multi_processor_count
            plan_sms = round(sms * 16 / 152)
        self.lookahead, self.plan_sms = lookahead, plan_sms
        self.depth = depth or n_ranks + lookahead + 1
        if self.depth < n_ranks + lookahead + 1:
            raise ValueError("depth must be at least N + lookahead + 1")
        dev = torch.device(device)
        dq.lib()
        cfg = self.config(0)
        plan_bytes = dq.dq_plan_workspace_bytes(n_ranks, bucket_sg)
        msg_bytes = dq.dq_bucket_msgs_bytes(cfg, bucket_sg)
        if plan_bytes == 0 or msg_bytes == 0:
            raise dq.DQError(dq.DQ_ERR_INVALID_ARG, "bucket stream workspace")
        self.sets = [{"mu": torch.empty(bucket_sg, dtype=torch.float32, device=dev),
                      "perm": torch.empty(bucket_sg, dtype=torch.int32, device=dev),
                      "plan_ws": torch.empty(plan_bytes, dtype=torch.uint8, device=dev),
                      "msgs": torch.empty(msg_bytes, dtype=torch.uint8, device=dev)} for _ in range(self.depth)]
        self.plan_stream = torch.cuda.Stream(device=dev, priority=-1)
        self.ev_plan = [torch.cuda.Event() for _ in range(self.depth)]
        self.ev_free = [torch.cuda.Event() for _ in range(self.depth)]
        self.counters = torch.zeros(1024, dtype=torch.int32, device=dev)
        self.nonfinite = [None] * self.depth
        # set by the library when some bucket of the last pass had non-finite statistics
        self.pass_nonfinite = torch.zeros(1, dtype=torch.int32, device=dev)

    def config(self, round: int = 0):
        return self.dq.config(self.n_ranks, self.budget, self.eps, self.correlated, self.seed, round,
                              self.fixed_bits, self.scale_fp32)

    def check(self):
        """Raises dq.NonFinite if some bucket of the last pass driven by the
        library had non-finite statistics (a NaN or infinite gradient, or
        squares beyond fp32); synchronises the current stream.  The passes
        with hooks plan bucket by bucket and are not covered."""
        if self.dq.dq_get_device_status(self.pass_nonfinite) != 0:
            raise self.dq.NonFinite(self.dq.DQ_ERR_NONFINITE, "bucket stream: non-finite gradient statistics")

    def copy_streams(self):
        """The (upload, download) streams of the library's host staging."""
        if getattr(self, "_copy_streams", None) is None:
            self._copy_streams = (torch.cuda.Stream(device=self.counters.device),
                                  torch.cuda.Stream(device=self.counters.device))
        return self._copy_streams

    def run(self, buckets, outs, round0: int = 0, log=None, ready=None, before_plan=None, before_exchange=None,
            after_exchange=None, src_host=None, dst_host=None, copy_in=None, copy_out=None):
        """As ``BucketedAllReduce.run``: buckets[k][r] is rank r's bf16
        gradient of bucket k (a multiple of 256 coordinates, at most
        bucket_sg super-groups), outs[k][r] its result; bucket k is round
        round0 + k.  The hooks are called with (k, stream): before bucket k's
        planning is enqueued (on the planning stream, once the buffer set's
        previous bucket has finished: its staging may be reused), before its
        first launch and after its decode (on the exchange stream).  A
        bucket's gradients are read until its last ring step, so a caller
        that stages them needs ``depth`` staging sets (set k % depth).

        Host staging without hooks: ``src_host[k][r]`` (pinned host tensors)
        are copied into buckets[k][r] before bucket k's planning, and rank
        0's result of bucket k into ``dst_host[k]`` (a pinned host tensor)
        after its decode, all by the library (dq_allreduce_stream_io) on the
        copy streams ``copy_in`` and ``copy_out`` (None: streams of its
        own); staging sets must be at least N + lookahead apart."""
        import ctypes as C
        dq = self.dq
        N, nb, D = self.n_ranks, len(buckets), self.depth
        if self.counters.numel() < nb + N:
            self.counters = torch.zeros(nb + N, dtype=torch.int32, device=self.counters.device)
        main = torch.cuda.current_stream()
        side = self.plan_stream
        if ready is None and before_plan is None and before_exchange is None and after_exchange is None:
            # nothing to interleave: the library drives the whole pass
            keep = []
            arr = (dq.dq_bucket * nb)()
            for k in range(nb):
                gp = (C.c_void_p * N)(*[g.data_ptr() for g in buckets[k]])
                op = (C.c_void_p * N)(*[o.data_ptr() for o in outs[k]])
                keep += [gp, op]
                arr[k] = dq.dq_bucket(buckets[k][0].numel() // 256, C.cast(gp, C.c_void_p), C.cast(op, C.c_void_p),
                                      round0 + k)
            sets = (dq.dq_stream_set * D)(*[dq.dq_stream_set(s["mu"].data_ptr(), s["perm"].data_ptr(),
                                                                 s["plan_ws"].data_ptr(), s["plan_ws"].numel(),
                                                                 s["msgs"].data_ptr(), s["msgs"].numel())
                                            for s in self.sets])
            if src_host is None and dst_host is None:
                dq.dq_allreduce_stream(self.config(0), arr, sets, self.counters, self.out_is_bf16, side, main, log,
                                       lookahead=self.lookahead, plan_sms=self.plan_sms,
                                       nonfinite=self.pass_nonfinite)
                return
            io = (dq.dq_bucket_io * nb)()
            for k in range(nb):
                # the library copies whole buffers: sizes must match the device sides
                if src_host is not None and any(h.device.type != "cpu" or h.numel() != g.numel() or
                                                h.element_size() != 2 for h, g in zip(src_host[k], buckets[k])):
                    raise ValueError(f"src_host[{k}]: host bf16 buffers of the device gradients' sizes "
                                     f"({[(h.device.type, h.numel(), h.element_size()) for h in src_host[k]]} "
                                     f"against {[g.numel() for g in buckets[k]]})")
                if dst_host is not None and (dst_host[k].device.type != "cpu" or
                                             dst_host[k].numel() != outs[k][0].numel() or
                                             dst_host[k].element_size() != outs[k][0].element_size()):
                    raise ValueError(f"dst_host[{k}]: a host buffer of rank 0's output size and type "
                                     f"({dst_host[k].device}, {dst_host[k].numel()} x {dst_host[k].element_size()} "
                                     f"bytes against {outs[k][0].numel()} x {outs[k][0].element_size()})")
                sp = None
                if src_host is not None:
                    sp = (C.c_void_p * N)(*[h.data_ptr() for h in src_host[k]])
                    keep.append(sp)
                io[k] = dq.dq_bucket_io(C.cast(sp, C.c_void_p) if sp is not None else None,
                                        dst_host[k].data_ptr() if dst_host is not None else None)
            if copy_in is None:
                copy_in = self.copy_streams()[0]
            if copy_out is None:
                copy_out = self.copy_streams()[1]
            dq.dq_allreduce_stream_io(self.config(0), arr, io, sets, self.counters, self.out_is_bf16, copy_in,
                                      copy_out, side, main, log, lookahead=self.lookahead, plan_sms=self.plan_sms,
                                      nonfinite=self.pass_nonfinite)
            return
        if src_host is not None or dst_host is not None:
            raise ValueError("host staging by the library cannot be combined with hooks or ready events")
        self.counters[: nb + N].zero_()
        live = {}

        def plan(k):
            si = k % D
            side.wait_event(self.ev_free[si])            # the set's previous bucket has been decoded
            if before_plan is not None:
                before_plan(k, side)
            s = self.sets[si]
            n_sg = buckets[k][0].numel() // 256
            if n_sg > self.bucket_sg:
                raise ValueError("a bucket larger than bucket_sg")
            counts, nonfinite = dq.dq_plan_async(self.config(round0 + k), buckets[k], n_sg, s["mu"], s["perm"],
                                                 s["plan_ws"], s["plan_ws"].numel(), log=log, stream=side,
                                                 ready=None if ready is None else ready[k])
            self.ev_plan[si].record(side)
            self.nonfinite[si] = nonfinite
            gp = (C.c_void_p * N)(*[g.data_ptr() for g in buckets[k]])
            op = (C.c_void_p * N)(*[o.data_ptr() for o in outs[k]])
            live[k] = (si, n_sg, counts, gp, op)

        cfg = self.config(0)
        plan(0)
        for t in range(nb + N):
            if t + 1 < nb:
                plan(t + 1)
            if t < nb:
                main.wait_event(self.ev_plan[live[t][0]])
                if before_exchange is not None:
                    before_exchange(t, main)
            steps = []
            for b in range(max(0, t - N), min(t, nb - 1) + 1):
                si, n_sg, counts, gp, op = live[b]
                s = self.sets[si]
                steps.append(dq.dq_bucket_step(n_sg, counts, C.cast(gp, C.c_void_p), C.cast(op, C.c_void_p),
                                               s["mu"].data_ptr(), s["perm"].data_ptr(), s["msgs"].data_ptr(),
                                               s["msgs"].numel(), round0 + b, t - b))
            arr = (dq.dq_bucket_step * len(steps))(*steps)
            dq.dq_exchange_stream_step(cfg, arr, self.counters[t:], self.out_is_bf16, log, main)
            if t >= N:
                b = t - N
                self.ev_free[live[b][0]].record(main)
                if after_exchange is not None:
                    after_exchange(b, main)
                del live[b]
