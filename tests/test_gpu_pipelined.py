"""The ring exchange pipelined over parts of the super-groups
(dq_exchange_pipelined) against the oracle and against the per-step
exchange: final messages and outputs bit for bit, for part counts from one
to more than the work units (cut to that count), ragged sizes, every
ablation mode and bf16 outputs."""
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


def bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def grads_for(name, n, N, seed=0):
    w = synth.WORKLOADS[name].scaled(n)
    w = w.__class__(**{**w.__dict__, "n_ranks": N})
    return [synth.as_u16(g) for g in synth.generate(w, "cpu", seed=seed)]


def _run(gr, N, parts, log=None, **kw):
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J, seed=1, **kw)
    gd = [dev_u16(g) for g in gr]
    outs = ar.new_outputs()
    ar.plan(gd, round=2)
    ar.exchange(gd, outs, round=2, fused=False, parts=parts, log=log)
    torch.cuda.synchronize()
    msgs = [ar.final_message(c).numpy() for c in range(N)]
    return ar, [o.cpu() for o in outs], msgs


@pytest.mark.parametrize("N,parts", [(1, 1), (1, 3), (2, 2), (3, 5), (8, 1), (8, 8), (8, 19), (16, 16),
                                     (16, 33), (5, 100000)])
def test_pipelined_equals_oracle_and_per_step(N, parts):
    gr = grads_for("bert_large_ring8", 256 * 1500 + 77, N, seed=N + parts)
    _, outs, msgs = _run(gr, N, parts, budget=5.0, correlated=True)
    _, outs2, msgs2 = _run(gr, N, None, budget=5.0, correlated=True)
    for a, b in zip(msgs, msgs2):
        assert np.array_equal(a, b)
    for a, b in zip(outs, outs2):
        assert torch.equal(bits(a), bits(b))
    cfg = oracle.Config(N, 5.0, correlated=True, seed=1, round=2)
    _, exp = oracle.allreduce(cfg, gr)
    for o in outs:
        assert np.array_equal(o.numpy().view(np.int32), np.ascontiguousarray(exp, np.float32).view(np.int32))


@pytest.mark.parametrize("N,parts", [(32, 1), (32, 7), (64, 3), (64, 40)])
def test_pipelined_many_ranks_equals_oracle(N, parts):
    """Rings of 32 and 64 ranks (up to the exchange's limit): N x N message
    buffers, decodes into more than 16 outputs per launch (2N row copies per
    pair of super-groups), and more parts than a chunk has units."""
    gr = grads_for("gemma1b_ring16", 256 * 400 + 13, N, seed=N * 7 + parts)
    _, outs, _ = _run(gr, N, parts, budget=5.0, correlated=True)
    cfg = oracle.Config(N, 5.0, correlated=True, seed=1, round=2)
    _, exp = oracle.allreduce(cfg, gr)
    want = np.ascontiguousarray(exp, np.float32).view(np.int32)
    for r in (0, 1, N // 2, N - 1):
        assert np.array_equal(outs[r].numpy().view(np.int32), want), r


@pytest.mark.parametrize("kw", [dict(eps=0.3), dict(eps=math.inf, correlated=False), dict(scale_fp32=True),
                                dict(fixed_bits=2, budget=2.0), dict(fixed_bits=8, budget=8.0),
                                dict(out_dtype=torch.bfloat16)])
def test_pipelined_modes(kw):
    N = 8
    gr = grads_for("llama1b_butterfly8", 256 * 900 + 5, N, seed=3)
    _, outs, msgs = _run(gr, N, 6, **kw)
    _, outs2, msgs2 = _run(gr, N, None, **kw)
    for a, b in zip(msgs, msgs2):
        assert np.array_equal(a, b)
    for a, b in zip(outs, outs2):
        assert torch.equal(bits(a), bits(b))


def test_pipelined_launch_count_and_log():
    """N + parts launches, each logged as DQ_LAUNCH_PIPELINED; the logged
    super-groups add up to N steps of every super-group plus the decode."""
    N, parts = 4, 7
    gr = grads_for("bert_large_ring8", 256 * 2000 + 1, N, seed=5)
    J = gr[0].size // 256
    log = dq.LaunchLog(64)
    before = dq.lib().dq_launch_count()
    _run(gr, N, parts, log=log)
    kinds = [k for k, _, _ in log.launches()]
    # dq_plan's launches come first; the exchange's are the pipelined ones
    piped = [(k, s) for k, s, _ in log.launches() if k == dq.DQ_LAUNCH_PIPELINED]
    assert len(piped) == N + parts
    assert sum(s for _, s in piped) == J * (N + 1)
    assert kinds[-(N + parts):] == [dq.DQ_LAUNCH_PIPELINED] * (N + parts)
    assert dq.lib().dq_launch_count() - before >= N + parts + 1   # + the counters' zeroing


def test_pipelined_rejects_bad_arguments():
    N = 4
    gr = grads_for("bert_large_ring8", 256 * 300, N, seed=1)
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J, seed=1)
    gd = [dev_u16(g) for g in gr]
    outs = ar.new_outputs()
    ar.plan(gd, round=0)
    cfg = ar.config(0)
    need = dq.dq_exchange_pipelined_workspace_bytes(cfg, J, ar.info)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    with pytest.raises(dq.DQError):
        dq.dq_exchange_pipelined(cfg, gd, J, ar.mu, ar.perm, ar.info, ws, need - 1, outs, 2)
    with pytest.raises(dq.DQError):
        dq.dq_exchange_pipelined(cfg, gd, J, ar.mu, ar.perm, ar.info, ws, need, outs, 0)
