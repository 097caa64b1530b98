"""Degenerate gradients through every exchange path, bit for bit against the
oracle: all-zero gradients, a rank of zeros beside random ones, zero,
single-spike and constant super-groups, identical gradients on every rank,
bf16 subnormals (whose squares vanish in fp32) and values near 1e15.  The
method's special cases live here: super-groups whose group maxima are all
zero (u = 0, E = 0, decoded as the mean alone), F_j = 0 at the allocation's
lowest key, x = 0 exactly after the mean is subtracted, and the exponent
clamp of the UINT8 scale hierarchy at both ends."""
import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import build, synth
from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _grads(kind: str, N: int, J: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    n = J * 256
    if kind == "all_zero":
        xs = [torch.zeros(n) for _ in range(N)]
    elif kind == "one_rank_zero":
        xs = [torch.randn(n, generator=g) for _ in range(N)]
        xs[1].zero_()
    elif kind == "mixed_supergroups":
        xs = []
        for r in range(N):
            x = torch.randn(n, generator=g).view(J, 256)
            x[0::5] = 0.0                                # zero super-groups
            x[1::5] = 0.0
            x[1::5, 17] = 3.0 * (r + 1)                  # one spike
            x[2::5] = 0.25 * (r + 1)                     # constant within the super-group
            x[3::5, :16] = 0.0                           # a zero group beside non-zero ones
            xs.append(x.reshape(-1))
    elif kind == "identical":
        x = torch.randn(n, generator=g)
        xs = [x.clone() for _ in range(N)]
    elif kind == "tiny":
        # bf16 subnormals and the smallest normals: squares underflow to zero
        xs = [torch.randn(n, generator=g) * 1e-39 for _ in range(N)]
        xs[0].view(J, 256)[::3] = 0.0
    elif kind == "huge":
        xs = [torch.randn(n, generator=g) * 1e15 for _ in range(N)]
    else:
        raise ValueError(kind)
    return [x.to(torch.bfloat16) for x in xs]


KINDS = ["all_zero", "one_rank_zero", "mixed_supergroups", "identical", "tiny", "huge"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("path", ["fused", "step", "pipelined", "butterfly"])
def test_degenerate_gradients_match_oracle(kind, path):
    build.build()
    N, J = 4, 1537
    gb = _grads(kind, N, J, seed=KINDS.index(kind))
    gu = [synth.as_u16(x) for x in gb]
    butterfly = path == "butterfly"
    ar = DynamiQAllReduce(N, J, budget=5.0, correlated=True, butterfly=butterfly, seed=5)
    gd = [x.to(DEV) for x in gb]
    ar.plan(gd, round=2)
    outs = ar.new_outputs()
    if path == "fused":
        ar.exchange(gd, outs, round=2, fused=True)
    elif path == "pipelined":
        ar.exchange(gd, outs, round=2, fused=False, parts=3)
    else:
        ar.exchange(gd, outs, round=2, fused=False)
    torch.cuda.synchronize()
    if path == "fused":
        ar.check_status()
    _, exp = oracle.allreduce(oracle.Config(N, 5.0, correlated=True, seed=5, round=2), gu, butterfly=butterfly)
    for r in range(N):
        got = outs[r].cpu().numpy()
        assert np.array_equal(got.view(np.int32), exp.view(np.int32)), (kind, path, r)
    if kind == "all_zero":
        assert not np.any(exp.view(np.int32))   # every output exactly +0
