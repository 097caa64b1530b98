"""The fused ring exchange (one cooperative launch for all hops and the
decode) against the oracle and against the multi-launch exchange, and the
failure path of its grid barrier: a wait that nothing will satisfy runs out,
reports DQ_DEVICE_BARRIER_TIMEOUT and leaves the context usable.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import build, dq, synth
from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    dq.lib()


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def bits32(a):
    return np.ascontiguousarray(a, np.float32).view(np.int32)


def grads_for(name, n, N, seed=0):
    w = synth.WORKLOADS[name].scaled(n)
    w = w.__class__(**{**w.__dict__, "n_ranks": N})
    return [synth.as_u16(g) for g in synth.generate(w, "cpu", seed=seed)]


def _run(gr, N, fused, **kw):
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J, seed=1, **kw)
    gd = [dev_u16(g) for g in gr]
    outs = ar.new_outputs()
    ar.plan(gd, round=2)
    ar.exchange(gd, outs, round=2, fused=fused)
    torch.cuda.synchronize()
    if fused:
        ar.check_status()
    lo = ar.chunk_lo()
    msgs = [ar.final_message(c).numpy() for c in range(N)]
    return ar, [o.cpu() for o in outs], msgs, lo


@pytest.mark.parametrize("N", [1, 2, 3, 8, 16, 33, 64])
def test_fused_equals_oracle_and_multi_launch(N):
    gr = grads_for("bert_large_ring8", 256 * 700 + 13, N, seed=N)
    ar, outs, msgs, lo = _run(gr, N, True, budget=5.0, correlated=True)
    _, outs2, msgs2, _ = _run(gr, N, False, budget=5.0, correlated=True)
    for a, b in zip(outs, outs2):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    for a, b in zip(msgs, msgs2):
        assert np.array_equal(a, b)
    cfg = oracle.Config(N, 5.0, correlated=True, seed=1, round=2)
    p, exp = oracle.allreduce(cfg, gr)
    for o in outs:
        assert np.array_equal(bits32(o.numpy()), bits32(exp))


@pytest.mark.parametrize("kw", [dict(eps=0.3), dict(eps=math.inf, correlated=False), dict(scale_fp32=True),
                                dict(fixed_bits=8, budget=8.0), dict(out_dtype=torch.bfloat16)])
def test_fused_modes(kw):
    N = 8
    gr = grads_for("llama1b_butterfly8", 256 * 500 + 3, N, seed=7)
    _, outs, msgs, _ = _run(gr, N, True, **kw)
    _, outs2, msgs2, _ = _run(gr, N, False, **kw)
    for a, b in zip(outs, outs2):
        assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                           b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))
    for a, b in zip(msgs, msgs2):
        assert np.array_equal(a, b)


def test_fused_is_one_launch():
    N = 8
    gr = grads_for("ring4_1m", 256 * 300, N)
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J)
    gd = [dev_u16(g) for g in gr]
    outs = ar.new_outputs()
    ar.plan(gd)
    torch.cuda.synchronize()
    log = dq.LaunchLog(8)
    n0 = dq.dq_launch_count()
    ar.exchange(gd, outs, fused=True, log=log)
    torch.cuda.synchronize()
    # the exchange is one cooperative launch; a one-thread kernel before it
    # zeroes its barrier counter and status word (in stream order, without
    # a memset that a copy engine could hold behind other streams' copies)
    assert dq.dq_launch_count() - n0 == 2
    assert [k for k, _, _ in log.launches()] == [dq.DQ_LAUNCH_FUSED_RING]
    ar.check_status()


def test_fused_rejects_what_it_does_not_cover():
    ar = DynamiQAllReduce(65, 64)
    ar.info = dq.dq_plan_info(0.0, 0, 64, 0)
    assert dq.dq_exchange_fused_workspace_bytes(ar.config(), 64, ar.info) == 0   # more than 64 ranks
    with pytest.raises(dq.DQError):
        ar.exchange([torch.zeros(64 * 256, dtype=torch.bfloat16, device=DEV)] * 65, ar.new_outputs(), fused=True)


def test_barrier_timeout_reports_status_and_context_survives():
    scratch = torch.zeros(4, dtype=torch.int32, device=DEV)
    status = torch.full((1,), 77, dtype=torch.int32, device=DEV)
    n = min(8, torch.cuda.get_device_properties(0).multi_processor_count)
    # every CTA arrives: the barrier passes
    dq.dq_barrier_selftest(n, 0, 2_000_000, scratch, status)
    torch.cuda.synchronize()
    assert int(status.item()) == dq.DQ_DEVICE_OK
    # one arrival never comes: each bounded wait runs out (2e6 cycles, about
    # a millisecond), the status says so and the kernel returns
    dq.dq_barrier_selftest(n, 1, 2_000_000, scratch, status)
    torch.cuda.synchronize()
    assert int(status.item()) == dq.DQ_DEVICE_BARRIER_TIMEOUT
    assert int(scratch[0].item()) == n
    # the same two states read through the C ABI's status call (it
    # synchronises the stream itself)
    dq.dq_barrier_selftest(n, 0, 2_000_000, scratch, status)
    assert dq.dq_get_device_status(status) == dq.DQ_DEVICE_OK
    dq.dq_barrier_selftest(n, 1, 2_000_000, scratch, status)
    assert dq.dq_get_device_status(status) == dq.DQ_DEVICE_BARRIER_TIMEOUT
    # the context is still usable: a fused exchange right after is correct
    test_fused_is_one_launch()


def test_plan_reports_nonfinite_gradients():
    """A NaN, an infinity, or values whose squares overflow fp32 make the
    plan fail with DQ_ERR_NONFINITE; a clean plan afterwards succeeds."""
    N, J = 4, 300
    gr = grads_for("ring4_1m", 256 * J, N, seed=3)
    ar = DynamiQAllReduce(N, J)
    for bad in (float("nan"), float("inf"), -float("inf"), 3.0e38):
        gd = [dev_u16(g) for g in gr]
        gd[2][256 * 123 + 7] = bad
        with pytest.raises(dq.NonFinite):
            ar.plan(gd)
    ar.plan([dev_u16(g) for g in gr])
    assert ar.info.n2 + ar.info.n4 + ar.info.n8 == J


def test_multi_launch_exchange_structure():
    """Ring of 8 through dq_exchange: one compress launch, seven DAR launches
    and one decode launch that reads each chunk once and writes all eight
    outputs (its log entry counts J super-groups per output)."""
    N = 8
    gr = grads_for("ring4_1m", 256 * 400, N, seed=2)
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J)
    gd = [dev_u16(g) for g in gr]
    outs = ar.new_outputs()
    ar.plan(gd)
    torch.cuda.synchronize()
    log = dq.LaunchLog(32)
    ar.exchange(gd, outs, log=log, fused=False)
    torch.cuda.synchronize()
    got = log.launches()
    assert [k for k, _, _ in got] == [dq.DQ_LAUNCH_COMPRESS] + [dq.DQ_LAUNCH_DAR] * 7 + [dq.DQ_LAUNCH_DECODE]
    assert got[-1][1] == J * N
