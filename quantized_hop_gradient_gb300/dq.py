"""Thin Python binding of libdq (argument marshalling only).

Every function here has the name of a C entry point of ``include/dq.h`` and
only converts arguments: torch tensors become device pointers, the current
torch stream becomes the cudaStream_t, status codes become exceptions.  All
computation runs in libdq's CUDA kernels; there is no fallback: loading fails
loudly if the library is missing.
"""
from __future__ import annotations

import ctypes as C
import math
import os
import threading
from dataclasses import dataclass

import torch

from . import build as _build

SG = 256
DQ_OK, DQ_ERR_INVALID_ARG, DQ_ERR_ALIGNMENT, DQ_ERR_BUDGET_INFEASIBLE, DQ_ERR_CUDA, DQ_ERR_NONFINITE = range(6)

_lock = threading.Lock()
_lib = None


class DQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class BudgetInfeasible(DQError):
    pass


class NonFinite(DQError):
    """dq_plan found a NaN or infinite super-group statistic."""


class dq_config(C.Structure):
    _fields_ = [("n_ranks", C.c_int32), ("budget_bits", C.c_float), ("eps", C.c_double),
                ("correlated", C.c_int32), ("seed", C.c_uint64), ("round", C.c_uint64),
                ("fixed_bits", C.c_int32), ("scale_fp32", C.c_int32)]


class dq_stage(C.Structure):
    _fields_ = [("rank", C.c_int32), ("hop", C.c_int32), ("slot", C.c_int32), ("n_slots", C.c_int32)]


class dq_range(C.Structure):
    _fields_ = [("lo", C.c_int64), ("hi", C.c_int64), ("end2", C.c_int64), ("end4", C.c_int64)]


class dq_launch_log(C.Structure):
    _fields_ = [("events", C.c_void_p), ("kinds", C.c_void_p), ("sgs", C.c_void_p),
                ("capacity", C.c_int32), ("count", C.c_int32)]


DQ_LAUNCH_COMPRESS, DQ_LAUNCH_DAR, DQ_LAUNCH_DECODE, DQ_LAUNCH_STATS, DQ_LAUNCH_ALLOCATE_REORDER = 0, 1, 2, 3, 4
DQ_LAUNCH_MX_HOP, DQ_LAUNCH_MX_DECODE, DQ_LAUNCH_FUSED_RING, DQ_LAUNCH_PIPELINED = 5, 6, 7, 8
DQ_LAUNCH_STREAM = 9
MAX_STREAM_RANKS = 8   # dq_exchange_stream_step: rings of up to 8 ranks
DQ_DEVICE_OK, DQ_DEVICE_BARRIER_TIMEOUT = 0, 1
MAX_FUSED_RANKS = 64
MAX_WAVE_PARTS = 256   # dq_exchange_pipelined cuts n_parts to this
UNIT = 32              # super-groups per work unit of the kernels


class dq_plan_info(C.Structure):
    _fields_ = [("T", C.c_float), ("n2", C.c_int64), ("n4", C.c_int64), ("n8", C.c_int64)]


class dq_bucket(C.Structure):
    _fields_ = [("n_sg", C.c_int64), ("grads_host", C.c_void_p), ("outs_host", C.c_void_p), ("round", C.c_uint64)]


class dq_stream_set(C.Structure):
    _fields_ = [("mu", C.c_void_p), ("perm", C.c_void_p), ("plan_ws", C.c_void_p), ("plan_ws_bytes", C.c_size_t),
                ("msgs", C.c_void_p), ("msgs_bytes", C.c_size_t)]


class dq_bucket_io(C.Structure):
    _fields_ = [("src_host", C.c_void_p), ("dst_host", C.c_void_p)]


class dq_bucket_step(C.Structure):
    _fields_ = [("n_sg", C.c_int64), ("counts_dev", C.c_void_p), ("grads_host", C.c_void_p),
                ("outs_host", C.c_void_p), ("mu", C.c_void_p), ("perm", C.c_void_p), ("msgs", C.c_void_p),
                ("msgs_bytes", C.c_size_t), ("round", C.c_uint64), ("step", C.c_int32)]


_SIGS = {
    "dq_version": ([], C.c_char_p),
    "dq_launch_count": ([], C.c_uint64),
    "dq_status_string": ([C.c_int], C.c_char_p),
    "dq_message_bytes": ([dq_range, C.c_int32], C.c_size_t),
    "dq_level_table": ([C.c_int32, C.c_double, C.c_void_p], C.c_int),
    "dq_stats": ([C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_stats_reduce": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_int64, C.c_void_p, C.c_void_p,
                         C.c_void_p, C.c_void_p], C.c_int),
    "dq_workspace_bytes": ([C.c_int64], C.c_size_t),
    "dq_allocate": ([C.c_void_p, C.c_int64, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p,
                     C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "dq_reorder": ([C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "dq_reorder_static": ([C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p], C.c_int),
    "dq_get_device_status": ([C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_chunk_cuts": ([C.c_int64, C.c_int64, C.c_int64, C.c_int32, C.c_void_p], C.c_int),
    "dq_compress": ([C.POINTER(dq_config), dq_range, dq_stage, C.c_void_p, C.c_void_p,
                     C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_dar": ([C.POINTER(dq_config), dq_range, dq_stage, C.c_void_p, C.c_void_p,
                C.c_int32, C.c_void_p, C.c_void_p, dq_range, C.c_void_p, dq_range, C.c_void_p,
                C.c_void_p], C.c_int),
    "dq_decode": ([C.POINTER(dq_config), dq_range, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                   C.c_int32, C.c_void_p], C.c_int),
    "dq_plan_workspace_bytes": ([C.c_int32, C.c_int64], C.c_size_t),
    "dq_plan": ([C.POINTER(dq_config), C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                 C.c_size_t, C.POINTER(dq_plan_info), C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_exchange_workspace_bytes": ([C.POINTER(dq_config), C.c_int32, C.c_int64,
                                     C.POINTER(dq_plan_info)], C.c_size_t),
    "dq_exchange": ([C.POINTER(dq_config), C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                     C.POINTER(dq_plan_info), C.c_void_p, C.c_size_t, C.c_void_p, C.c_int32,
                     C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_exchange_fused_workspace_bytes": ([C.POINTER(dq_config), C.c_int64, C.POINTER(dq_plan_info)],
                                           C.c_size_t),
    "dq_exchange_fused": ([C.POINTER(dq_config), C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                           C.POINTER(dq_plan_info), C.c_void_p, C.c_size_t, C.c_void_p, C.c_int32, C.c_void_p,
                           C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_exchange_pipelined_workspace_bytes": ([C.POINTER(dq_config), C.c_int64, C.POINTER(dq_plan_info)],
                                               C.c_size_t),
    "dq_exchange_pipelined": ([C.POINTER(dq_config), C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                               C.POINTER(dq_plan_info), C.c_void_p, C.c_size_t, C.c_void_p, C.c_int32, C.c_int32,
                               C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_plan_async": ([C.POINTER(dq_config), C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                       C.c_size_t, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_bucket_msgs_bytes": ([C.POINTER(dq_config), C.c_int64], C.c_size_t),
    "dq_allreduce_stream": ([C.POINTER(dq_config), C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int32,
                             C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p],
                            C.c_int),
    "dq_allreduce_stream_io": ([C.POINTER(dq_config), C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_int32,
                                C.c_int32, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_exchange_stream_step": ([C.POINTER(dq_config), C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                 C.c_void_p], C.c_int),
    "dq_barrier_selftest": ([C.c_int32, C.c_int32, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "dq_mx_message_bytes": ([C.c_int64], C.c_size_t),
    "dq_mx_quantize": ([C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p], C.c_int),
    "dq_mx_dequantize": ([C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p], C.c_int),
    "dq_mx_exchange_workspace_bytes": ([C.c_int32, C.c_int32, C.c_int64], C.c_size_t),
    "dq_mx_exchange": ([C.c_int32, C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_size_t, C.c_void_p,
                        C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
}


def library_path() -> str:
    return _build.LIB


def lib(build: bool = False):
    """Loads libdq (building it first when ``build``).  Raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            if not os.path.exists(path):
                raise ImportError(f"libdq is not built ({path}); run quantized_hop_gradient_gb300.build")
            L = C.CDLL(path)
            for name, (args, res) in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def status_string(s: int) -> str:
    return lib().dq_status_string(s).decode()


def _check(status: int, what: str):
    if status == DQ_ERR_BUDGET_INFEASIBLE:
        raise BudgetInfeasible(status, what)
    if status == DQ_ERR_NONFINITE:
        raise NonFinite(status, what)
    if status != DQ_OK:
        raise DQError(status, what)


def _ptr(t) -> int:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def config(n_ranks: int, budget_bits: float = 5.0, eps: float = 1.0, correlated: bool = True,
           seed: int = 0, round: int = 0, fixed_bits: int = 0, scale_fp32: bool = False) -> dq_config:
    return dq_config(n_ranks, budget_bits, eps, int(correlated), seed, round, int(fixed_bits), int(scale_fp32))


def rng(lo: int, hi: int, end2: int, end4: int) -> dq_range:
    return dq_range(lo, hi, end2, end4)


def stage(rank: int, hop: int, slot: int = 0, n_slots: int = 1) -> dq_stage:
    return dq_stage(rank, hop, slot, n_slots)


# ------------------------------------------------------------------ entry points (same names as dq.h)
def dq_version() -> str:
    return lib().dq_version().decode()


def dq_launch_count() -> int:
    return lib().dq_launch_count()


def dq_message_bytes(r: dq_range, scale_fp32: bool = False) -> int:
    return lib().dq_message_bytes(r, int(scale_fp32))


def dq_level_table(bits: int, eps: float = 1.0):
    import numpy as np
    q = np.zeros(1 << bits, np.float32)
    _check(lib().dq_level_table(bits, eps, q.ctypes.data), "dq_level_table")
    return q


def dq_stats(g, n_sg, mean, sq, stream=None):
    _check(lib().dq_stats(_ptr(g), n_sg, _ptr(mean), _ptr(sq), _stream(stream)), "dq_stats")


def dq_stats_reduce(mean_all, sq_all, n_ranks, n_sg, M, F, mu, stream=None):
    _check(lib().dq_stats_reduce(_ptr(mean_all), _ptr(sq_all), n_ranks, n_sg, _ptr(M), _ptr(F), _ptr(mu),
                                 _stream(stream)), "dq_stats_reduce")


def dq_workspace_bytes(n_sg: int) -> int:
    return lib().dq_workspace_bytes(n_sg)


def dq_allocate(F, n_sg, budget, b, T_dev, counts_dev, ws, ws_bytes, stream=None):
    _check(lib().dq_allocate(_ptr(F), n_sg, budget, _ptr(b), _ptr(T_dev), _ptr(counts_dev), _ptr(ws),
                             ws_bytes, _stream(stream)), "dq_allocate")


def dq_reorder(b, n_sg, perm, ws, ws_bytes, stream=None):
    _check(lib().dq_reorder(_ptr(b), n_sg, _ptr(perm), _ptr(ws), ws_bytes, _stream(stream)), "dq_reorder")


REORDER_STATIC_MAX_SG = 8388608


def dq_reorder_static(b, n_sg, perm, stream=None):
    """dq_reorder without a workspace (scratch inside the library); for
    callers that cannot allocate device memory."""
    _check(lib().dq_reorder_static(_ptr(b), n_sg, _ptr(perm), _stream(stream)), "dq_reorder_static")


def dq_chunk_cuts(n2, n4, n8, n_chunks):
    out = (C.c_int64 * (n_chunks + 1))()
    _check(lib().dq_chunk_cuts(n2, n4, n8, n_chunks, C.addressof(out)), "dq_chunk_cuts")
    return list(out)


def dq_compress(cfg, r, st, g, mu, perm, msg_out, stream=None):
    _check(lib().dq_compress(C.byref(cfg), r, st, _ptr(g), _ptr(mu), _ptr(perm), _ptr(msg_out),
                             _stream(stream)), "dq_compress")


def dq_dar(cfg, r_in, st, msg_in, addend, addend_is_fp32, mu, perm, send, msg_out, keep, keep_out,
           stream=None):
    _check(lib().dq_dar(C.byref(cfg), r_in, st, _ptr(msg_in), _ptr(addend), int(addend_is_fp32),
                        _ptr(mu), _ptr(perm), send, _ptr(msg_out), keep, _ptr(keep_out), _stream(stream)),
           "dq_dar")


def dq_decode(cfg, r, msg, mu, perm, out, out_is_bf16=False, stream=None):
    _check(lib().dq_decode(C.byref(cfg), r, _ptr(msg), _ptr(mu), _ptr(perm), _ptr(out), int(out_is_bf16),
                           _stream(stream)), "dq_decode")


def dq_plan_workspace_bytes(n_ranks, n_sg) -> int:
    return lib().dq_plan_workspace_bytes(n_ranks, n_sg)


def dq_plan(cfg, grads, n_sg, mu, perm, ws, ws_bytes, log=None, stream=None, ready=None) -> dq_plan_info:
    """``ready``: optional list of torch.cuda.Event, one per rank (or None)."""
    ptrs = (C.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    ev = None
    if ready is not None:
        ev = (C.c_void_p * len(grads))(*[(e.cuda_event if e is not None else None) for e in ready])
    info = dq_plan_info()
    _check(lib().dq_plan(C.byref(cfg), C.cast(ptrs, C.c_void_p), n_sg, _ptr(mu), _ptr(perm), _ptr(ws),
                         ws_bytes, C.byref(info), C.cast(ev, C.c_void_p) if ev is not None else None,
                         C.byref(log.c) if log is not None else None, _stream(stream)), "dq_plan")
    return info


def dq_plan_async(cfg, grads, n_sg, mu, perm, ws, ws_bytes, log=None, stream=None, ready=None):
    """dq_plan without the readback or the sync.  Returns the device
    addresses (ints) of the plan's three int64 counts and of its non-finite
    flag."""
    ptrs = (C.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    ev = None
    if ready is not None:
        ev = (C.c_void_p * len(grads))(*[(e.cuda_event if e is not None else None) for e in ready])
    counts, nonfinite = C.c_void_p(), C.c_void_p()
    _check(lib().dq_plan_async(C.byref(cfg), C.cast(ptrs, C.c_void_p), n_sg, _ptr(mu), _ptr(perm), _ptr(ws),
                               ws_bytes, C.byref(counts), C.byref(nonfinite),
                               C.cast(ev, C.c_void_p) if ev is not None else None,
                               C.byref(log.c) if log is not None else None, _stream(stream)), "dq_plan_async")
    return counts.value, nonfinite.value


def dq_bucket_msgs_bytes(cfg, n_sg) -> int:
    return lib().dq_bucket_msgs_bytes(C.byref(cfg), n_sg)


def dq_allreduce_stream(cfg, buckets, sets, counters, out_is_bf16=False, plan_stream=None, stream=None,
                        log: "LaunchLog" = None, lookahead: int = 1, plan_sms: int = 0, nonfinite=None):
    """A whole bucket stream in one call.  ``buckets``: a ctypes array of
    dq_bucket; ``sets``: a ctypes array of dq_stream_set; ``counters``: a
    device int32 tensor of at least len(buckets) + N words; ``nonfinite``:
    None or a device int32 that becomes 1 if some bucket's statistics are
    not finite."""
    _check(lib().dq_allreduce_stream(C.byref(cfg), C.cast(buckets, C.c_void_p), len(buckets),
                                     C.cast(sets, C.c_void_p), len(sets), int(lookahead), int(plan_sms),
                                     _ptr(counters), int(out_is_bf16),
                                     _ptr(nonfinite) if nonfinite is not None else None,
                                     _stream(plan_stream) if plan_stream is not None else None, _stream(stream),
                                     C.byref(log.c) if log is not None else None), "dq_allreduce_stream")


def dq_allreduce_stream_io(cfg, buckets, io, sets, counters, out_is_bf16=False, copy_in_stream=None,
                           copy_out_stream=None, plan_stream=None, stream=None, log: "LaunchLog" = None,
                           lookahead: int = 1, plan_sms: int = 0, nonfinite=None):
    """dq_allreduce_stream with each bucket's upload and download done by the
    library.  ``io``: a ctypes array of dq_bucket_io, one per bucket."""
    if len(io) != len(buckets):
        raise ValueError("one dq_bucket_io per bucket")
    opt = lambda st: _stream(st) if st is not None else None
    _check(lib().dq_allreduce_stream_io(C.byref(cfg), C.cast(buckets, C.c_void_p), C.cast(io, C.c_void_p),
                                        len(buckets), C.cast(sets, C.c_void_p), len(sets), int(lookahead),
                                        int(plan_sms), _ptr(counters), int(out_is_bf16),
                                        _ptr(nonfinite) if nonfinite is not None else None, opt(copy_in_stream),
                                        opt(copy_out_stream), opt(plan_stream), _stream(stream),
                                        C.byref(log.c) if log is not None else None), "dq_allreduce_stream_io")


def dq_exchange_stream_step(cfg, steps, counter, out_is_bf16=False, log: "LaunchLog" = None, stream=None):
    """One launch of the bucket stream.  ``steps``: a ctypes array of
    dq_bucket_step; ``counter``: a device uint32 (tensor or address), zero at
    the launch."""
    _check(lib().dq_exchange_stream_step(C.byref(cfg), C.cast(steps, C.c_void_p), len(steps), _ptr(counter),
                                         int(out_is_bf16), C.byref(log.c) if log is not None else None,
                                         _stream(stream)), "dq_exchange_stream_step")


def dq_exchange_workspace_bytes(cfg, butterfly, n_sg, info) -> int:
    return lib().dq_exchange_workspace_bytes(C.byref(cfg), int(butterfly), n_sg, C.byref(info))


class LaunchLog:
    """Host side of a dq_launch_log: caller-created CUDA events (from torch)."""

    def __init__(self, capacity: int, stream=None):
        import numpy as np
        st = torch.cuda.current_stream() if stream is None else stream
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:          # torch creates the CUDA event on first record
            e.record(st)
        self._ev = (C.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self.kinds = np.zeros(capacity, np.int32)
        self.sgs = np.zeros(capacity, np.int64)
        self.c = dq_launch_log(C.cast(self._ev, C.c_void_p), self.kinds.ctypes.data, self.sgs.ctypes.data,
                               capacity, 0)

    def launches(self):
        """[(kind, super-groups, milliseconds)] of the recorded launches (after a sync)."""
        return [(int(self.kinds[i]), int(self.sgs[i]), self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i in range(self.c.count)]


def dq_exchange(cfg, butterfly, grads, n_sg, mu, perm, info, ws, ws_bytes, outs, out_is_bf16=False,
                log: LaunchLog = None, stream=None):
    """Returns the N device addresses of the final chunk messages (inside ws)."""
    n = len(grads)
    gp = (C.c_void_p * n)(*[_ptr(g) for g in grads])
    op = (C.c_void_p * n)(*[_ptr(o) for o in outs])
    fin = (C.c_void_p * n)()
    _check(lib().dq_exchange(C.byref(cfg), int(butterfly), C.cast(gp, C.c_void_p), n_sg, _ptr(mu), _ptr(perm),
                             C.byref(info), _ptr(ws), ws_bytes, C.cast(op, C.c_void_p), int(out_is_bf16),
                             C.cast(fin, C.c_void_p), C.byref(log.c) if log is not None else None,
                             _stream(stream)), "dq_exchange")
    return [fin[i] for i in range(n)]


# ------------------------------------------------------------------ MXFP8 comparison baseline
MX_BLOCK = 32


def dq_mx_message_bytes(n_blk: int) -> int:
    return lib().dq_mx_message_bytes(n_blk)


def dq_mx_quantize(x, n_blk, msg, stream=None):
    _check(lib().dq_mx_quantize(_ptr(x), n_blk, _ptr(msg), _stream(stream)), "dq_mx_quantize")


def dq_mx_dequantize(msg, n_blk, out, stream=None):
    _check(lib().dq_mx_dequantize(_ptr(msg), n_blk, _ptr(out), _stream(stream)), "dq_mx_dequantize")


def dq_mx_exchange_workspace_bytes(n_ranks, butterfly, n_blk) -> int:
    return lib().dq_mx_exchange_workspace_bytes(n_ranks, int(butterfly), n_blk)


def dq_mx_exchange(n_ranks, butterfly, grads, n_blk, ws, ws_bytes, outs, log: LaunchLog = None, stream=None):
    """Returns the N device addresses of the final chunk messages (inside ws)."""
    gp = (C.c_void_p * n_ranks)(*[_ptr(g) for g in grads])
    op = (C.c_void_p * n_ranks)(*[_ptr(o) for o in outs])
    fin = (C.c_void_p * n_ranks)()
    _check(lib().dq_mx_exchange(n_ranks, int(butterfly), C.cast(gp, C.c_void_p), n_blk, _ptr(ws), ws_bytes,
                                C.cast(op, C.c_void_p), C.cast(fin, C.c_void_p),
                                C.byref(log.c) if log is not None else None, _stream(stream)), "dq_mx_exchange")
    return [fin[i] for i in range(n_ranks)]


# ------------------------------------------------------------------ fused ring exchange
def dq_exchange_fused_workspace_bytes(cfg, n_sg, info) -> int:
    return lib().dq_exchange_fused_workspace_bytes(C.byref(cfg), n_sg, C.byref(info))


def dq_exchange_fused(cfg, grads, n_sg, mu, perm, info, ws, ws_bytes, outs, status, out_is_bf16=False,
                      log: LaunchLog = None, stream=None):
    """The ring exchange in one cooperative launch.  ``status``: a device
    int32 tensor that ends as DQ_DEVICE_OK (or DQ_DEVICE_BARRIER_TIMEOUT).
    Returns the N device addresses of the final chunk messages."""
    n = len(grads)
    gp = (C.c_void_p * n)(*[_ptr(g) for g in grads])
    op = (C.c_void_p * n)(*[_ptr(o) for o in outs])
    fin = (C.c_void_p * n)()
    _check(lib().dq_exchange_fused(C.byref(cfg), C.cast(gp, C.c_void_p), n_sg, _ptr(mu), _ptr(perm),
                                   C.byref(info), _ptr(ws), ws_bytes, C.cast(op, C.c_void_p), int(out_is_bf16),
                                   _ptr(status), C.cast(fin, C.c_void_p),
                                   C.byref(log.c) if log is not None else None, _stream(stream)),
           "dq_exchange_fused")
    return [fin[i] for i in range(n)]


def dq_exchange_pipelined_workspace_bytes(cfg, n_sg, info) -> int:
    return lib().dq_exchange_pipelined_workspace_bytes(C.byref(cfg), n_sg, C.byref(info))


def dq_exchange_pipelined(cfg, grads, n_sg, mu, perm, info, ws, ws_bytes, outs, n_parts, out_is_bf16=False,
                          log: LaunchLog = None, stream=None):
    """The ring exchange pipelined over ``n_parts`` parts of the
    super-groups (N + n_parts launches).  Returns the N device addresses of
    the final chunk messages."""
    n = len(grads)
    gp = (C.c_void_p * n)(*[_ptr(g) for g in grads])
    op = (C.c_void_p * n)(*[_ptr(o) for o in outs])
    fin = (C.c_void_p * n)()
    _check(lib().dq_exchange_pipelined(C.byref(cfg), C.cast(gp, C.c_void_p), n_sg, _ptr(mu), _ptr(perm),
                                       C.byref(info), _ptr(ws), ws_bytes, C.cast(op, C.c_void_p),
                                       int(out_is_bf16), int(n_parts), C.cast(fin, C.c_void_p),
                                       C.byref(log.c) if log is not None else None, _stream(stream)),
           "dq_exchange_pipelined")
    return [fin[i] for i in range(n)]


def dq_get_device_status(status_dev, stream=None) -> int:
    """The device status word ``status_dev`` (an int32 device tensor) read
    into host memory; synchronises ``stream``."""
    out = C.c_int32(-1)
    _check(lib().dq_get_device_status(_ptr(status_dev), C.addressof(out), _stream(stream)), "dq_get_device_status")
    return out.value


def dq_barrier_selftest(n_blocks, missing, timeout_cycles, scratch, status, stream=None):
    _check(lib().dq_barrier_selftest(n_blocks, missing, timeout_cycles, _ptr(scratch), _ptr(status),
                                     _stream(stream)), "dq_barrier_selftest")
