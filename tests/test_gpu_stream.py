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
