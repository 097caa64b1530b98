"""Parity at full workload sizes, in the launch configuration bench.py times.

The GPU runs the whole all-reduce exactly as the benchmark does (gradients
drawn on the device, DynamiQAllReduce).  The oracle recomputes the plan for
the whole gradient (statistics, allocation, reordering: compared in full,
bit for bit) and then follows a sample of super-groups one by one through
the topology (random ones plus the first and last of every chunk and of
every bitwidth stream); their outputs and final message bytes must match
bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import build, dq, synth
from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce

pytestmark = pytest.mark.gpu


def _sample(J, chunk_lo, n2, n4, rs, k=1500):
    pts = set(rs.integers(0, J, k).tolist())
    for c in chunk_lo:
        for d in (-2, -1, 0, 1):
            if 0 <= c + d < J:
                pts.add(int(c + d))
    for e in (n2, n2 + n4):
        for d in (-2, -1, 0, 1):
            if 0 <= e + d < J:
                pts.add(int(e + d))
    return np.array(sorted(pts), dtype=np.int64)


def _full_size(name, butterfly, budget=None):
    build.build()
    w = synth.WORKLOADS[name]
    if budget is not None:
        w = w.scaled(w.n, budget=budget)
    N, J = w.n_ranks, w.n_sg
    grads = synth.generate(w, "cuda", seed=0)
    ar = DynamiQAllReduce(N, J, budget=w.budget, correlated=w.correlated, butterfly=butterfly, seed=0)
    outs = ar(grads, round=3)
    torch.cuda.synchronize()
    gu = [synth.as_u16(g) for g in grads]
    del grads
    cfg = oracle.Config(N, w.budget, correlated=w.correlated, seed=0, round=3)
    p = oracle.plan(cfg, gu)
    info = ar.info
    assert [info.n2, info.n4, info.n8] == p.counts.tolist()
    assert np.float32(info.T).view(np.int32) == np.float32(p.T).view(np.int32)
    assert np.array_equal(ar.perm.cpu().numpy(), p.perm)
    assert np.array_equal(ar.mu.cpu().numpy().view(np.int32), (p.M / np.float32(N)).view(np.int32))
    lo = ar.chunk_lo()
    assert lo == p.chunk_lo.tolist()
    sel = _sample(J, lo, info.n2, info.n4, np.random.default_rng(7))
    rows, fin = oracle.allreduce_sg(cfg, butterfly, gu, p.M, p.perm, int(info.n2), int(info.n4), p.chunk_lo, sel)
    old = torch.from_numpy(p.perm[sel].astype(np.int64)).cuda()
    idx = (old[:, None] * 256 + torch.arange(256, device="cuda")[None, :]).reshape(-1)
    for r in (0, N - 1):
        got = outs[r][idx].cpu().numpy().reshape(-1, 256)
        assert np.array_equal(got.view(np.int32), rows.view(np.int32)), f"rank {r}: outputs differ"
    # E bytes and UINT8 scales of the sampled super-groups in the final chunk messages
    for c in range(N):
        a, b = lo[c], lo[c + 1]
        inside = sel[(sel >= a) & (sel < b)]
        if inside.size == 0:
            continue
        m = ar.final_message(c).numpy()
        cnt = b - a
        off_u = -(-cnt // 16) * 16
        for j in inside:
            s = int(j - a)
            f = fin[np.searchsorted(sel, j)]
            assert m[s] == f[0]
            assert np.array_equal(m[off_u + 16 * s: off_u + 16 * s + 16], f[1:17])


def test_bert_large_ring8_full_size_sampled():
    _full_size("bert_large_ring8", butterfly=False)


def test_llama1b_butterfly8_full_size_sampled():
    _full_size("llama1b_butterfly8", butterfly=True)


def test_gemma1b_ring16_full_size_sampled():
    """Gemma-1B-sized gradient, 16 workers, ring (the pipelined exchange
    over 32 parts that the bench times at this size), budget 5."""
    _full_size("gemma1b_ring16", butterfly=False)


@pytest.mark.parametrize("B", [4.0, 6.0])
def test_gemma1b_ring16_budget_sweep_full_size_sampled(B):
    """The other budgets of the Gemma-1B workload's sweep, at full size."""
    _full_size("gemma1b_ring16", butterfly=False, budget=B)


def test_llama3_8b_buckets_full_size():
    """The streamed Llama-3-8B workload at full bucket size: 25 MB buckets of
    13,107,200 coordinates, 8 ranks.  The first bucket, one from the middle
    and the short last bucket (of 613) are reduced as one pass of the bucket
    stream in the bench's configuration (BucketStream: lookahead 3, the
    default share of SMs left to the planning stream), and as one stream of
    per-bucket rounds (the cooperative one-launch exchange, and per-step
    launches); every result is compared with the oracle in full."""
    from quantized_hop_gradient_gb300.allreduce import use_fused
    from quantized_hop_gradient_gb300.stream import BucketedAllReduce, BucketStream
    build.build()
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    N = w.n_ranks
    nb = synth.bucket_count(w)
    picks = [0, nb // 2, nb - 1]
    buckets = [synth.generate_bucket(w, k, "cuda", seed=0) for k in picks]
    assert buckets[-1][0].numel() < w.bucket and buckets[0][0].numel() == w.bucket
    exps = []
    for i, b in enumerate(buckets):
        gu = [synth.as_u16(g) for g in b]
        cfg = oracle.Config(N, w.budget, correlated=w.correlated, seed=0, round=100 + i)
        exps.append(oracle.allreduce(cfg, gu)[1])
    for mode in ("stream", False, "auto"):
        outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
        if mode == "stream":
            ar = BucketStream(N, w.bucket // 256, budget=w.budget, correlated=w.correlated, seed=0)
            assert ar.lookahead == 3
        else:
            ar = BucketedAllReduce(N, w.bucket // 256, overlap=True, fused=mode, budget=w.budget,
                                   correlated=w.correlated, seed=0)
            assert ar.fused == (mode == "auto")   # "auto" takes the one-launch exchange at this size
            assert all(use_fused(N, False, s.n_sg) for s in ar.sets)   # the size allows the one-launch exchange
        ar.run(buckets, outs, round0=100)
        torch.cuda.synchronize()
        if mode == "auto":
            for s in ar.sets:
                s.check_status()
        for i in range(len(buckets)):
            for r in (0, N - 1):
                got = outs[i][r].cpu().numpy()
                assert np.array_equal(got.view(np.int32), exps[i].view(np.int32)), (mode, picks[i], r)
