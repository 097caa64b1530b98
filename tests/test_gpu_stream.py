"""The bucketed (DDP-style) all-reduce: every bucket's result equals the
oracle's all-reduce of that bucket (bit for bit), with and without the
two-stream overlap, including a short last bucket; and the same for the
bucket stream whose ring exchange is pipelined across buckets
(dq_exchange_stream_step), with more buckets than buffer sets."""
import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import build, synth
from quantized_hop_gradient_gb300.stream import BucketedAllReduce, BucketStream

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


@pytest.mark.parametrize("lookahead,plan_sms", [(3, -1), (1, 0), (2, 16)])
@pytest.mark.parametrize("N,n_full", [(1, 3), (2, 5), (4, 9), (8, 13)])
def test_bucket_stream_matches_oracle(N, n_full, lookahead, plan_sms):
    """Every bucket of the cross-bucket pipelined stream equals the oracle's
    all-reduce of that bucket, bit for bit: outputs of every rank, with a
    short last bucket and more buckets than the stream's buffer sets."""
    build.build()
    bucket_sg = 37
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (n_full * bucket_sg + 11), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cuda", seed=3) for k in range(nb)]
    outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
    bs = BucketStream(N, bucket_sg, budget=5.0, correlated=True, lookahead=lookahead, plan_sms=plan_sms)
    assert nb > bs.depth or N < 8
    bs.run(buckets, outs, round0=30)
    torch.cuda.synchronize()
    for k, b in enumerate(buckets):
        gu = [synth.as_u16(g) for g in b]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=30 + k), gu)
        for r in range(N):
            assert np.array_equal(outs[k][r].cpu().numpy().view(np.int32), exp.view(np.int32)), (k, r)


@pytest.mark.parametrize("kw", [dict(eps=0.3), dict(scale_fp32=True), dict(fixed_bits=4, budget=4.0),
                                dict(out_dtype=torch.bfloat16)])
def test_bucket_stream_modes_match_per_bucket_rounds(kw):
    """The stream in every mode equals one DynamiQ round per bucket through
    the per-step exchange (itself pinned to the oracle), bit for bit."""
    build.build()
    N, bucket_sg = 4, 53
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (6 * bucket_sg + 5), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cuda", seed=4) for k in range(nb)]
    dt = kw.get("out_dtype", torch.float32)
    outs = [[torch.empty(g.numel(), dtype=dt, device="cuda") for g in b] for b in buckets]
    BucketStream(N, bucket_sg, seed=2, **kw).run(buckets, outs, round0=7)
    torch.cuda.synchronize()
    from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce
    for k, b in enumerate(buckets):
        J = b[0].numel() // 256
        ar = DynamiQAllReduce(N, J, seed=2, **kw)
        exp = ar(b, round=7 + k, fused=False)
        torch.cuda.synchronize()
        for r in range(N):
            bits = torch.int16 if dt == torch.bfloat16 else torch.int32
            assert torch.equal(outs[k][r].view(bits), exp[r].view(bits)), (k, r)


def test_bucket_stream_uploaded_through_hooks_matches_oracle():
    """The stream as the end-to-end benchmark drives it: every bucket's
    gradients come from pinned host memory into one of `depth` staging sets
    on a copy stream, enqueued by the planning hook and waited on through
    per-rank ready events; rank 0's result goes back to the host after each
    bucket's decode.  Results equal the oracle's."""
    build.build()
    N, bucket_sg = 4, 29
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (11 * bucket_sg + 7), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cpu", seed=6) for k in range(nb)]
    hosts = [[g.pin_memory() for g in b] for b in buckets]
    bs = BucketStream(N, bucket_sg, budget=5.0, correlated=True)
    stage = [[torch.empty(256 * bucket_sg, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
             for _ in range(bs.depth)]
    bufs = [[s[:g.numel()] for s, g in zip(stage[k % bs.depth], buckets[k])] for k in range(nb)]
    outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
    res = [torch.empty(g[0].numel(), dtype=torch.float32, pin_memory=True) for g in buckets]
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [[torch.cuda.Event() for _ in range(N)] for _ in range(nb)]
    done = [torch.cuda.Event() for _ in range(nb)]

    def before_plan(k, side):
        cin.wait_stream(side)
        with torch.cuda.stream(cin):
            for r in range(N):
                bufs[k][r].copy_(hosts[k][r], non_blocking=True)
                ready[k][r].record(cin)

    def after_exchange(k, main):
        done[k].record(main)
        cout.wait_event(done[k])
        with torch.cuda.stream(cout):
            res[k].copy_(outs[k][0], non_blocking=True)

    bs.run(bufs, outs, round0=40, ready=ready, before_plan=before_plan, after_exchange=after_exchange)
    torch.cuda.synchronize()
    for k in range(nb):
        gu = [synth.as_u16(g) for g in buckets[k]]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=40 + k), gu)
        assert np.array_equal(res[k].numpy().view(np.int32), exp.view(np.int32)), k


def test_bucket_stream_large_buckets_match_oracle():
    """Buckets above 16,384 super-groups (planned by the multi-kernel
    allocation and reorder, not the single-block one): every bucket equals
    the oracle's all-reduce of it, bit for bit."""
    build.build()
    N, bucket_sg = 2, 20000
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (2 * bucket_sg + 999), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cuda", seed=8) for k in range(nb)]
    outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
    BucketStream(N, bucket_sg, budget=5.0, correlated=True).run(buckets, outs, round0=50)
    torch.cuda.synchronize()
    for k, b in enumerate(buckets):
        gu = [synth.as_u16(g) for g in b]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=50 + k), gu)
        for r in range(N):
            assert np.array_equal(outs[k][r].cpu().numpy().view(np.int32), exp.view(np.int32)), (k, r)


@pytest.mark.parametrize("N,lookahead,n_out,dt", [(4, 3, 3, torch.float32), (8, 1, 2, torch.float32),
                                                   (2, 2, 1, torch.bfloat16)])
def test_bucket_stream_library_staging_matches_oracle(N, lookahead, n_out, dt):
    """The stream with its host staging done by the library
    (dq_allreduce_stream_io): every bucket's gradients are copied from pinned
    host memory into device staging sets cycled at the smallest allowed
    distance (N + lookahead buckets), and rank 0's result of every bucket is
    copied to its own pinned host buffer while only n_out device output sets
    are cycled (a decode waits for the download that still reads its
    buffer).  The host results equal the oracle's, bit for bit (bf16: the
    fp32 result rounded to nearest-even)."""
    build.build()
    bucket_sg = 31
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (14 * bucket_sg + 9), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cpu", seed=9) for k in range(nb)]
    hosts = [[g.pin_memory() for g in b] for b in buckets]
    bs = BucketStream(N, bucket_sg, budget=5.0, correlated=True, lookahead=lookahead, out_dtype=dt)
    S = N + lookahead
    stage = [[torch.empty(256 * bucket_sg, dtype=torch.bfloat16, device="cuda") for _ in range(N)] for _ in range(S)]
    bufs = [[s[:g.numel()] for s, g in zip(stage[k % S], buckets[k])] for k in range(nb)]
    oset = [[torch.empty(256 * bucket_sg, dtype=dt, device="cuda") for _ in range(N)] for _ in range(n_out)]
    outs = [[o[:g.numel()] for o, g in zip(oset[k % n_out], buckets[k])] for k in range(nb)]
    res = [torch.full((g[0].numel(),), -1.0, dtype=dt).pin_memory() for g in buckets]
    bs.run(bufs, outs, round0=60, src_host=hosts, dst_host=res)
    torch.cuda.current_stream().synchronize()   # the call joins its copy streams to this one
    for k in range(nb):
        gu = [synth.as_u16(g) for g in buckets[k]]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=60 + k), gu)
        if dt == torch.bfloat16:
            got = res[k].view(torch.int16).numpy()
            want = torch.from_numpy(exp).to(torch.bfloat16).view(torch.int16).numpy()
        else:
            got, want = res[k].numpy().view(np.int32), exp.view(np.int32)
        assert np.array_equal(got, want), k


def test_bucket_stream_library_staging_rejects_close_reuse():
    """Staging sets closer than N + lookahead buckets apart cannot be
    refilled in time: the call is refused before anything is enqueued."""
    from quantized_hop_gradient_gb300 import dq
    build.build()
    N, lookahead, bucket_sg = 4, 3, 17
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * 10 * bucket_sg, "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cpu", seed=10) for k in range(nb)]
    hosts = [[g.pin_memory() for g in b] for b in buckets]
    S = N + lookahead - 1
    stage = [[torch.empty(256 * bucket_sg, dtype=torch.bfloat16, device="cuda") for _ in range(N)] for _ in range(S)]
    bufs = [stage[k % S] for k in range(nb)]
    outs = [[torch.empty(256 * bucket_sg, device="cuda") for _ in range(N)] for _ in range(nb)]
    bs = BucketStream(N, bucket_sg, lookahead=lookahead)
    with pytest.raises(dq.DQError):
        bs.run(bufs, outs, src_host=hosts)


@pytest.mark.parametrize("last_sg", [1, 3, 7])
def test_bucket_stream_last_bucket_smaller_than_ring(last_sg):
    """A last bucket with fewer super-groups than the ring has ranks (8):
    some chunks are empty, which the device-side chunk geometry must cut the
    same way as the host's; every bucket equals the oracle's all-reduce."""
    build.build()
    N, bucket_sg = 8, 23
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (4 * bucket_sg + last_sg), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    buckets = [synth.generate_bucket(w, k, "cuda", seed=11 + last_sg) for k in range(nb)]
    assert buckets[-1][0].numel() == 256 * last_sg
    outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in buckets]
    BucketStream(N, bucket_sg, budget=5.0, correlated=True).run(buckets, outs, round0=70)
    torch.cuda.synchronize()
    for k, b in enumerate(buckets):
        gu = [synth.as_u16(g) for g in b]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=70 + k), gu)
        for r in range(N):
            assert np.array_equal(outs[k][r].cpu().numpy().view(np.int32), exp.view(np.int32)), (k, r)


@pytest.mark.parametrize("bucket_sg,staged", [(29, False), (20000, False), (29, True)])
def test_bucket_stream_reports_nonfinite(bucket_sg, staged):
    """A NaN in one rank's gradient of one bucket makes the pass's flag read
    non-finite (BucketStream.check raises dq.NonFinite), on both planning
    paths (single-block up to 16,384 super-groups, the launch chain above)
    and with the library's host staging; the other buckets still equal the
    oracle's, and a clean pass afterwards checks clean."""
    from quantized_hop_gradient_gb300 import dq
    build.build()
    N = 2
    w = synth.WORKLOADS["llama3_8b_ring8_buckets"]
    w = w.__class__(**{**w.__dict__, "n_ranks": N, "n": 256 * (5 * bucket_sg + 3), "bucket": 256 * bucket_sg})
    nb = synth.bucket_count(w)
    clean = [synth.generate_bucket(w, k, "cpu", seed=12) for k in range(nb)]
    bad = [[g.clone() for g in b] for b in clean]
    bad[2][1][256 * (bucket_sg // 2) + 5] = float("nan")
    bs = BucketStream(N, bucket_sg, budget=5.0, correlated=True)

    def run(src):
        outs = [[torch.empty(g.numel(), dtype=torch.float32, device="cuda") for g in b] for b in src]
        if staged:
            S = bs.depth
            stage = [[torch.empty(256 * bucket_sg, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
                     for _ in range(S)]
            bufs = [[t[:g.numel()] for t, g in zip(stage[k % S], src[k])] for k in range(nb)]
            hosts = [[g.pin_memory() for g in b] for b in src]
            res = [torch.empty(b[0].numel(), dtype=torch.float32).pin_memory() for b in src]
            bs.run(bufs, outs, round0=80, src_host=hosts, dst_host=res)
            torch.cuda.current_stream().synchronize()
            return [r.numpy() for r in res]
        bs.run([[g.cuda() for g in b] for b in src], outs, round0=80)
        torch.cuda.synchronize()
        return [o[0].cpu().numpy() for o in outs]

    got = run(bad)
    with pytest.raises(dq.NonFinite):
        bs.check()
    for k in range(nb):
        if k == 2:
            continue
        gu = [synth.as_u16(g) for g in clean[k]]
        _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, round=80 + k), gu)
        assert np.array_equal(got[k].view(np.int32), exp.view(np.int32)), k
    run(clean)
    bs.check()
