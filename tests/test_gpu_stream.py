"""The bucketed (DDP-style) all-reduce: every bucket's result equals the
oracle's all-reduce of that bucket (bit for bit), with and without the
two-stream overlap, including a short last bucket."""
import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import build, synth
from quantized_hop_gradient_gb300.stream import BucketedAllReduce

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("butterfly", [False, True])
@pytest.mark.parametrize("overlap", [True, False])
def test_buckets_match_oracle(butterfly, overlap):
    build.build()
    N, bucket_sg = 4, 37
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (5 * bucket_sg + 11), "bucket": 256 * bucket_sg})
    buckets = [synth.generate_bucket(w, k, "cuda", seed=1) for k in range(synth.bucket_count(w))]
    assert buckets[-1][0].numel() == 256 * 11
    outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
    ar = BucketedAllReduce(N, bucket_sg, overlap=overlap, budget=5.0, correlated=True, butterfly=butterfly)
    ar.run(buckets, outs, round0=10)
    torch.cuda.synchronize()
    for k, b in enumerate(buckets):
        gu = [synth.as_u16(g) for g in b]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=10 + k), gu, butterfly=butterfly)
        for r in range(N):
            got = outs[k][r].cpu().numpy()
            assert np.array_equal(got.view(np.int32), exp.view(np.int32)), (k, r)


@pytest.mark.parametrize("fused", [False, True])
def test_buckets_uploaded_through_hooks_match_oracle(fused):
    """The streamed pass as the end-to-end benchmark drives it: every
    bucket's gradients come from pinned host memory into two alternating
    device staging sets on a copy stream (enqueued by the planning hook,
    waited on through per-rank ready events), and rank 0's result goes back
    to the host on a third stream after each exchange.  The results equal
    the oracle's, bit for bit."""
    build.build()
    N, bucket_sg = 4, 37
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (5 * bucket_sg + 11), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cpu", seed=2) for k in range(nb)]
    hosts = [[g.pin_memory() for g in b] for b in buckets]
    stage = [[torch.empty(256 * bucket_sg, dtype=torch.bfloat16, device="cuda") for _ in range(N)] for _ in range(2)]
    bufs = [[s[:g.numel()] for s, g in zip(stage[k & 1], buckets[k])] for k in range(nb)]
    outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
    res = [torch.empty(g[0].numel(), dtype=torch.float32, pin_memory=True) for g in buckets]
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [[torch.cuda.Event() for _ in range(N)] for _ in range(nb)]
    done = [torch.cuda.Event() for _ in range(nb)]

    def before_plan(k, side):
        cin.wait_stream(side)                  # the staging set's previous bucket has finished
        with torch.cuda.stream(cin):
            for r in range(N):
                bufs[k][r].copy_(hosts[k][r], non_blocking=True)
                ready[k][r].record(cin)

    def after_exchange(k, main):
        done[k].record(main)
        cout.wait_event(done[k])
        with torch.cuda.stream(cout):
            res[k].copy_(outs[k][0], non_blocking=True)

    ar = BucketedAllReduce(N, bucket_sg, overlap=True, fused=fused, budget=5.0, correlated=True)
    ar.run(bufs, outs, round0=20, ready=ready, before_plan=before_plan, after_exchange=after_exchange)
    torch.cuda.synchronize()
    for k in range(nb):
        gu = [synth.as_u16(g) for g in buckets[k]]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=20 + k), gu)
        assert np.array_equal(res[k].numpy().view(np.int32), exp.view(np.int32)), k
        for r in range(N):
            assert np.array_equal(outs[k][r].cpu().numpy().view(np.int32), exp.view(np.int32)), (k, r)
