"""The C ABI without a GPU: the library builds and loads, exports every
entry point that include/dq.h declares, its host-side pure functions agree
with the oracle, and bad arguments are rejected before any CUDA call."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import oracle
from quantized_hop_gradient_gb300 import build, dq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dq.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return dq.lib()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dq_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_entry_point(L):
    names = declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert sorted(dq.exported_symbols()) == names   # the binding covers the ABI


def test_version_and_status_strings(L):
    assert "sm_103a" in dq.dq_version()
    assert dq.status_string(dq.DQ_ERR_BUDGET_INFEASIBLE).startswith("budget")
    assert "non-finite" in dq.status_string(dq.DQ_ERR_NONFINITE)


@pytest.mark.parametrize("eps", [1.0, 0.25, 0.5, 3.7, 4.0, math.inf])
def test_level_tables_bitwise_equal_to_oracle(L, eps):
    for bits in (2, 4, 8):
        a = dq.dq_level_table(bits, eps)
        b = oracle.level_table(bits, eps)
        assert np.array_equal(a.view(np.int32), b.view(np.int32))


def test_chunk_cuts_equal_oracle(L):
    rs = np.random.default_rng(0)
    for N in (1, 2, 3, 4, 8, 16, 64):
        for J in (1, 2, 7, 100, 4096):
            b = rs.choice([2, 4, 8], J, p=[0.3, 0.5, 0.2]).astype(np.uint8)
            perm = oracle.reorder(b)
            counts = [int((b == k).sum()) for k in (2, 4, 8)]
            assert dq.dq_chunk_cuts(*counts, N) == oracle.chunk_cuts(b, perm, N).tolist()


def test_message_bytes_equal_oracle(L):
    rs = np.random.default_rng(1)
    for _ in range(200):
        J = int(rs.integers(1, 5000))
        end2 = int(rs.integers(0, J + 1))
        end4 = int(rs.integers(end2, J + 1))
        lo = int(rs.integers(0, J + 1))
        hi = int(rs.integers(lo, J + 1))
        assert dq.dq_message_bytes(dq.rng(lo, hi, end2, end4)) == oracle.range_message_bytes(lo, hi, end2, end4 - end2)
        assert (dq.dq_message_bytes(dq.rng(lo, hi, end2, end4), True)
                == oracle.range_message_bytes(lo, hi, end2, end4 - end2, True))


def test_mx_message_bytes_equal_oracle(L):
    for n in (0, 1, 15, 16, 17, 1000, 4_194_304):
        assert dq.dq_mx_message_bytes(n) == oracle.mx_message_bytes(n)
    assert dq.dq_mx_message_bytes(-1) == 0
    # the workspace holds two messages per rank (plus fp32 halves and final chunks for the butterfly)
    assert dq.dq_mx_exchange_workspace_bytes(4, False, 1000) >= 8 * dq.dq_mx_message_bytes(250)
    assert dq.dq_mx_exchange_workspace_bytes(3, True, 1000) == 0      # butterfly needs 2^k ranks
    assert dq.dq_mx_exchange_workspace_bytes(4, True, 1000) > dq.dq_mx_exchange_workspace_bytes(4, False, 1000)


def test_bad_arguments_rejected_on_the_host(L):
    P = 4096  # a fake, aligned address: validation fails before it could be used
    st = 0
    assert L.dq_allocate(P, 10, 1.5, P, P, P, P, 1 << 20, st) == dq.DQ_ERR_BUDGET_INFEASIBLE
    assert L.dq_allocate(P, 0, 5.0, P, P, P, P, 1 << 20, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allocate(P, 10, 5.0, P, P, P, P, 16, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allocate(P, 1 << 27, 5.0, P, P, P, P, 1 << 30, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allocate(None, 10, 5.0, P, P, P, P, 1 << 20, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_stats(P + 8, 4, P, P, st) == dq.DQ_ERR_ALIGNMENT
    cfg = dq.config(4)
    r = dq.rng(0, 8, 4, 6)
    assert L.dq_compress(cfg, r, dq.stage(4, 0), P, P, P, P, st) == dq.DQ_ERR_INVALID_ARG     # rank >= N
    assert L.dq_compress(cfg, r, dq.stage(0, 0, 2, 2), P, P, P, P, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_compress(cfg, r, dq.stage(0, 0), P + 4, P, P, P, st) == dq.DQ_ERR_ALIGNMENT
    assert L.dq_compress(dq.config(4, eps=0.0), r, dq.stage(0, 0), P, P, P, P, st) == dq.DQ_ERR_INVALID_ARG
    # send + keep must split `in`
    bad = L.dq_dar(cfg, r, dq.stage(0, 1), P, P, 0, P, P, dq.rng(0, 4, 4, 6), P, dq.rng(5, 8, 4, 6), P, st)
    assert bad == dq.DQ_ERR_INVALID_ARG
    info = dq.dq_plan_info(0.0, 1, 1, 1)
    assert dq.dq_exchange_workspace_bytes(dq.config(3), True, 3, info) == 0   # butterfly needs 2^k ranks
    assert dq.dq_exchange_workspace_bytes(dq.config(3), False, 3, info) > 0
    assert dq.dq_message_bytes(dq.rng(5, 4, 0, 0)) == 0
    assert dq.dq_message_bytes(dq.rng(0, 4, 0, 0), 2) == 0
    # ablation switches: only 0/2/4/8 bits and 0/1 scale modes
    for bad_cfg in (dq.config(4, fixed_bits=3), dq.config(4, fixed_bits=16), dq.config(4, scale_fp32=2)):
        assert L.dq_compress(bad_cfg, r, dq.stage(0, 0), P, P, P, P, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_mx_quantize(P, -1, P, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_mx_quantize(P + 4, 8, P, st) == dq.DQ_ERR_ALIGNMENT
    assert L.dq_mx_dequantize(P, 8, None, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_mx_exchange(3, 1, P, 10, P, 1 << 20, P, None, None, st) == dq.DQ_ERR_INVALID_ARG
    # fused exchange: ring of at most 64 ranks, a status word is required
    assert dq.dq_exchange_fused_workspace_bytes(dq.config(65), 3, info) == 0
    assert dq.dq_exchange_fused_workspace_bytes(dq.config(3), 3, info) > dq.dq_exchange_workspace_bytes(
        dq.config(3), False, 3, info)
    assert L.dq_exchange_fused(dq.config(3), P, 3, P, P, info, P, 1 << 30, P, 0, None, None, None,
                               st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_barrier_selftest(0, 0, 1000, P, P, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_barrier_selftest(4, 0, 0, P, P, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_barrier_selftest(4, 0, 1000, P + 2, P, st) == dq.DQ_ERR_ALIGNMENT
    host = (ctypes.c_int32 * 1)()
    assert L.dq_get_device_status(None, ctypes.addressof(host), st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_get_device_status(P, None, st) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_get_device_status(P + 2, ctypes.addressof(host), st) == dq.DQ_ERR_ALIGNMENT


def test_bucket_stream_arguments_rejected_on_the_host(L):
    """The whole-pass bucket stream drivers refuse bad arguments before they
    touch the GPU: no buckets, a ring above 8 ranks, a lookahead below 1,
    too few buffer sets, and (for the staged driver) no staging list."""
    P = 4096
    st = 0
    ptrs = (ctypes.c_void_p * 4)(*([P] * 4))
    b = (dq.dq_bucket * 2)(*[dq.dq_bucket(100, ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(ptrs, ctypes.c_void_p), k)
                             for k in range(2)])
    sets = (dq.dq_stream_set * 8)(*[dq.dq_stream_set(P, P, P, 1 << 20, P, 1 << 20) for _ in range(8)])
    io = (dq.dq_bucket_io * 2)(*[dq.dq_bucket_io(ctypes.cast(ptrs, ctypes.c_void_p), P) for _ in range(2)])
    cfg4, cfg9 = dq.config(4), dq.config(9)
    # dq_allreduce_stream(cfg, buckets, n, sets, n_sets, lookahead, plan_sms, counters, bf16, nonfinite,
    #                     plan_stream, stream, log)
    assert L.dq_allreduce_stream(cfg4, b, 0, sets, 8, 3, 0, P, 0, P, None, st, None) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allreduce_stream(cfg9, b, 2, sets, 8, 3, 0, P, 0, P, None, st, None) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allreduce_stream(cfg4, b, 2, sets, 8, 0, 0, P, 0, P, None, st, None) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allreduce_stream(cfg4, b, 2, sets, 7, 3, 0, P, 0, None, None, st, None) == dq.DQ_ERR_INVALID_ARG
    # dq_allreduce_stream_io(cfg, buckets, io, n, sets, n_sets, lookahead, plan_sms, counters, bf16, nonfinite,
    #                        copy_in, copy_out, plan_stream, stream, log)
    assert L.dq_allreduce_stream_io(cfg4, b, None, 2, sets, 8, 3, 0, P, 0, P, None, None, None, st,
                                    None) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allreduce_stream_io(cfg4, b, io, 2, sets, 7, 3, 0, P, 0, None, None, None, None, st,
                                    None) == dq.DQ_ERR_INVALID_ARG
    assert L.dq_allreduce_stream_io(cfg9, b, io, 2, sets, 8, 3, 0, P, 0, P, None, None, None, st,
                                    None) == dq.DQ_ERR_INVALID_ARG
