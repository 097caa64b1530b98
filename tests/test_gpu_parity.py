"""Parity of the CUDA path (through the C ABI) with the oracle, on the GPU.

Bar: codes, scales, bitwidth maps, permutations, thresholds and counts
bit-exact; decoded fp32 values bit-exact as well (both sides perform the
same correctly rounded fp32 steps), which is stricter than the 1e-6
relative bound the decode is held to; vNMSE equal.
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
    """numpy uint16 bf16 patterns -> device bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def host(t):
    return t.detach().cpu().numpy()


def bits32(a):
    return np.ascontiguousarray(a, np.float32).view(np.int32)


def grads_for(name, n, N=None, seed=0):
    w = synth.WORKLOADS[name].scaled(n)
    if N is not None:
        w = w.__class__(**{**w.__dict__, "n_ranks": N})
    return w, [synth.as_u16(g) for g in synth.generate(w, "cpu", seed=seed)]


# --------------------------------------------------------------------------- statistics
@pytest.mark.parametrize("J", [1, 3, 37, 4096, 20001])
def test_stats_bit_exact(J):
    _, gr = grads_for("ring4_1m", J * 256, seed=J)
    for g in gr[:2]:
        m = torch.empty(J, device=DEV)
        q = torch.empty(J, device=DEV)
        dq.dq_stats(dev_u16(g), J, m, q)
        em, eq = oracle.stats(g)
        assert np.array_equal(bits32(host(m)), bits32(em))
        assert np.array_equal(bits32(host(q)), bits32(eq))


def test_stats_reduce_bit_exact():
    rs = np.random.default_rng(0)
    for N, J in [(1, 5), (4, 4096), (16, 777)]:
        means = (rs.standard_normal((N, J)) * 10.0 ** rs.integers(-8, 8, (N, J))).astype(np.float32)
        sqs = np.abs(rs.standard_normal((N, J)) * 10.0 ** rs.integers(-8, 8, (N, J))).astype(np.float32)
        M = torch.empty(J, device=DEV)
        F = torch.empty(J, device=DEV)
        mu = torch.empty(J, device=DEV)
        dq.dq_stats_reduce(torch.from_numpy(means).to(DEV), torch.from_numpy(sqs).to(DEV), N, J, M, F, mu)
        eM, eF = oracle.stats_reduce(means, sqs)
        assert np.array_equal(bits32(host(M)), bits32(eM))
        assert np.array_equal(bits32(host(F)), bits32(eF))
        assert np.array_equal(bits32(host(mu)), bits32(eM / np.float32(N)))   # fl(M / N)


# --------------------------------------------------------------------------- allocation and reorder
def _F_cases(rs):
    yield np.exp(rs.normal(0, 3, 4096))
    yield rs.choice([0.0, 1.0, 30.117647, 30.12, 1e6], 5000)
    yield np.full(17, 2.5)
    yield np.array([7.0])
    yield np.zeros(64)
    yield rs.exponential(1.0, 100_000) * 1e-35
    yield np.exp(rs.normal(0, 8, 250_000))


def test_allocate_bit_exact():
    rs = np.random.default_rng(1)
    for F in _F_cases(rs):
        F = F.astype(np.float32)
        J = F.size
        Fd = torch.from_numpy(F).to(DEV)
        ws = torch.empty(dq.dq_workspace_bytes(J), dtype=torch.uint8, device=DEV)
        for B in (2.0, 2.01, 3.3, 4.0, 5.0, 6.0, 7.99, 8.0, 12.0):
            b = torch.empty(J, dtype=torch.uint8, device=DEV)
            T = torch.empty(1, device=DEV)
            counts = torch.empty(3, dtype=torch.int64, device=DEV)
            dq.dq_allocate(Fd, J, B, b, T, counts, ws, ws.numel())
            eb, eT, ec = oracle.allocate(F, B)
            assert bits32(host(T))[0] == bits32(np.array([eT]))[0], (J, B)
            assert np.array_equal(host(b), eb)
            assert np.array_equal(host(counts), ec)
    with pytest.raises(dq.BudgetInfeasible):
        dq.dq_allocate(Fd, J, 1.9, b, T, counts, ws, ws.numel())


@pytest.mark.parametrize("J", [1, 5, 2047, 2048, 2049, 100_003])
def test_reorder_bit_exact(J):
    rs = np.random.default_rng(J)
    b = rs.choice([2, 4, 8], J, p=[0.25, 0.5, 0.25]).astype(np.uint8)
    perm = torch.empty(J, dtype=torch.int32, device=DEV)
    ws = torch.empty(dq.dq_workspace_bytes(J), dtype=torch.uint8, device=DEV)
    dq.dq_reorder(torch.from_numpy(b).to(DEV), J, perm, ws, ws.numel())
    assert np.array_equal(host(perm), oracle.reorder(b))


# --------------------------------------------------------------------------- compress / DAR / decode
def _plan(gr, N, B=5.0):
    cfg = oracle.Config(N, B)
    return oracle.plan(cfg, gr)


def _ranges(p, N):
    lo = p.chunk_lo
    N2, N4 = int(p.counts[0]), int(p.counts[1])
    J = p.b.size
    cuts = sorted({0, J, N2, N2 + N4, max(0, N2 - 3), min(J, N2 + 5), (N2 + N4) // 2})
    out = [(int(lo[c]), int(lo[c + 1])) for c in range(N)]
    out += [(cuts[i], cuts[j]) for i in range(len(cuts)) for j in range(i + 1, len(cuts))][:12]
    return out, N2, N4


@pytest.mark.parametrize("eps", [1.0, math.inf, 0.3])
@pytest.mark.parametrize("correlated", [False, True])
def test_compress_dar_decode_bit_exact(eps, correlated):
    N = 4
    _, gr = grads_for("ring4_1m", 256 * 3000, N=N, seed=5)
    p = _plan(gr, N)
    M = torch.from_numpy(p.M / np.float32(N)).to(DEV)   # mu = fl(M / N)
    perm = torch.from_numpy(p.perm).to(DEV)
    gd = [dev_u16(g) for g in gr]
    cfg_o = oracle.Config(N, 5.0, eps=eps, correlated=correlated, seed=11, round=3)
    cfg = dq.config(N, 5.0, eps=eps, correlated=correlated, seed=11, round=3)
    ranges, N2, N4 = _ranges(p, N)
    E4 = N2 + N4
    for (a, b) in ranges:
        if b <= a:
            continue
        r = dq.rng(a, b, N2, E4)
        nb = dq.dq_message_bytes(r)
        # compress
        st = (1, 0, 1, 2)
        msg = torch.zeros(nb, dtype=torch.uint8, device=DEV)
        dq.dq_compress(cfg, r, dq.stage(*st), gd[1], M, perm, msg)
        exp = oracle.compress(cfg_o, a, b, N2, N4, st[0], st[1], gr[1], p.M, p.perm, slot=st[2], n_slots=st[3])
        assert np.array_equal(host(msg), exp), ("compress", a, b)
        # ring DAR (bf16 addend)
        out = torch.zeros(nb, dtype=torch.uint8, device=DEV)
        dq.dq_dar(cfg, r, dq.stage(2, 1), msg, gd[2], False, M, perm, r, out, dq.rng(b, b, N2, E4), None)
        eo, _ = oracle.dar(cfg_o, a, b, N2, N4, 2, 1, exp, gr[2], p.M, p.perm, send=(a, b))
        assert np.array_equal(host(out), eo), ("dar", a, b)
        # butterfly DAR: fp32 addend, send the upper part, keep the lower part
        mid = (a + b) // 2
        addend = np.random.default_rng(a).standard_normal((b - a) * 256).astype(np.float32)
        sr, kr = dq.rng(mid, b, N2, E4), dq.rng(a, mid, N2, E4)
        out2 = torch.zeros(max(1, dq.dq_message_bytes(sr)), dtype=torch.uint8, device=DEV)
        keep = torch.zeros(max(1, (mid - a) * 256), device=DEV)
        dq.dq_dar(cfg, r, dq.stage(3, 2, 1, 2), msg, torch.from_numpy(addend).to(DEV), True, M, perm, sr, out2,
                  kr, keep)
        eo2, ek = oracle.dar(cfg_o, a, b, N2, N4, 3, 2, exp, addend, p.M, p.perm, send=(mid, b),
                             keep=(a, mid), slot=1, n_slots=2)
        assert np.array_equal(host(out2)[: eo2.size], eo2), ("split dar msg", a, b)
        assert np.array_equal(bits32(host(keep)[: ek.size]), bits32(ek)), ("split dar keep", a, b)
        # decode (fp32 and bf16)
        o32 = torch.zeros(p.b.size * 256, device=DEV)
        dq.dq_decode(cfg, r, out, M, perm, o32)
        e32 = oracle.decode(cfg_o, a, b, N2, N4, eo, p.M, p.perm)
        assert np.array_equal(bits32(host(o32)), bits32(e32)), ("decode", a, b)
        o16 = torch.zeros(p.b.size * 256, dtype=torch.bfloat16, device=DEV)
        dq.dq_decode(cfg, r, out, M, perm, o16, out_is_bf16=True)
        assert torch.equal(o16.cpu(), torch.from_numpy(e32).to(torch.bfloat16))
        # an fp32 output 16- but not 32-byte aligned (the decode's bulk copies need 16)
        ob = torch.zeros(p.b.size * 256 + 4, device=DEV)
        o32u = ob[4:]
        assert o32u.data_ptr() % 32 == 16
        dq.dq_decode(cfg, r, out, M, perm, o32u)
        assert np.array_equal(bits32(host(o32u)), bits32(e32)), ("decode, 16-byte aligned output", a, b)


# --------------------------------------------------------------------------- whole all-reduce
def _check_allreduce(name, n, N, butterfly, correlated, B=5.0, seed=0):
    _, gr = grads_for(name, n, N=N, seed=seed)
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J, budget=B, correlated=correlated, butterfly=butterfly, seed=seed)
    outs = ar([dev_u16(g) for g in gr], round=7)
    torch.cuda.synchronize()
    cfg = oracle.Config(N, B, correlated=correlated, seed=seed, round=7)
    p = oracle.plan(cfg, gr)
    assert ar.info.n2 == p.counts[0] and ar.info.n4 == p.counts[1] and ar.info.n8 == p.counts[2]
    assert bits32(np.array([ar.info.T]))[0] == bits32(np.array([p.T]))[0]
    assert np.array_equal(host(ar.perm), p.perm)
    assert np.array_equal(bits32(host(ar.mu)), bits32(p.M / np.float32(N)))
    sel = np.arange(J, dtype=np.int64)
    rows, fin = oracle.allreduce_sg(cfg, butterfly, gr, p.M, p.perm, int(p.counts[0]), int(p.counts[1]),
                                    p.chunk_lo, sel)
    exp = np.zeros(J * 256, np.float32)
    exp.reshape(J, 256)[p.perm] = rows
    o0 = host(outs[0])
    assert np.array_equal(bits32(o0), bits32(exp))
    for o in outs[1:]:
        assert np.array_equal(bits32(host(o)), bits32(o0))   # replicas identical
    # final chunk messages: E, u and codes of every super-group
    lo = ar.chunk_lo()
    N2, N4 = ar.info.n2, ar.info.n4
    for c in range(N):
        a, b = lo[c], lo[c + 1]
        if b == a:
            continue
        m = ar.final_message(c).numpy()
        cnt = b - a
        n2, n4, n8 = oracle.range_counts(a, b, N2, N4)
        off_u = -(-cnt // 16) * 16
        offs = [off_u + 16 * cnt, off_u + 16 * cnt + 64 * n2, off_u + 16 * cnt + 64 * n2 + 128 * n4]
        for s in range(cnt):
            j = a + s
            f = fin[j]
            assert m[s] == f[0]
            assert np.array_equal(m[off_u + 16 * s: off_u + 16 * s + 16], f[1:17])
            if s < n2:
                blk = m[offs[0] + 64 * s: offs[0] + 64 * s + 64]
            elif s < n2 + n4:
                blk = m[offs[1] + 128 * (s - n2): offs[1] + 128 * (s - n2) + 128]
            else:
                blk = m[offs[2] + 256 * (s - n2 - n4): offs[2] + 256 * (s - n2 - n4) + 256]
            assert np.array_equal(blk, f[65:65 + blk.size])
    v_gpu = oracle.vnmse(o0, gr)
    v_orc = oracle.vnmse(exp, gr)
    assert v_gpu == pytest.approx(v_orc, rel=0.01)
    return v_gpu


@pytest.mark.parametrize("correlated", [False, True])
def test_ring4_1m_full_size(correlated):
    """The 4-worker ring on 1,048,576 coordinates per worker, in full."""
    _check_allreduce("ring4_1m", 1_048_576, 4, False, correlated)


@pytest.mark.parametrize("N", [2, 4, 8, 16, 64])
def test_butterfly(N):
    _check_allreduce("llama1b_butterfly8", 256 * 1500 + 77, N, True, True)


@pytest.mark.parametrize("N", [1, 3, 8, 33])
def test_ring_various_ranks(N):
    _check_allreduce("bert_large_ring8", 256 * 999, N, False, True)


@pytest.mark.parametrize("B", [2.0, 4.0, 6.0, 8.0])
def test_budget_sweep(B):
    _check_allreduce("gemma1b_ring16", 256 * 2000, 16, False, True, B=B)


def test_fewer_supergroups_than_ranks():
    """Empty chunks: 3 super-groups over 8 ranks (ring and butterfly), 1 over 4."""
    _check_allreduce("ring4_1m", 3 * 256, 8, False, False)
    _check_allreduce("ring4_1m", 3 * 256, 8, True, True)
    _check_allreduce("ring4_1m", 200, 4, False, True)


@pytest.mark.parametrize("fused", [False, True])
def test_exchange_outputs_16_byte_aligned(fused):
    """Outputs 16- but not 32-byte aligned (the decode's bulk copies need
    16-byte alignment only, in the per-step exchange and in the fused one)
    give the same bits as aligned outputs."""
    N = 4
    _, gr = grads_for("ring4_1m", 256 * 1500, N=N, seed=9)
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J, budget=5.0, correlated=True, seed=0)
    ga = [dev_u16(g) for g in gr]
    ref = [o.clone() for o in ar(ga, round=2, fused=fused)]
    bufs = [torch.zeros(J * 256 + 4, device=DEV) for _ in range(N)]
    outs = [b[4:] for b in bufs]
    assert all(o.data_ptr() % 32 == 16 for o in outs)
    ar(ga, round=2, outs=outs, fused=fused)
    torch.cuda.synchronize()
    if fused:
        ar.check_status()
    for r in range(N):
        assert torch.equal(outs[r].view(torch.int32), ref[r].view(torch.int32)), r



# --------------------------------------------------------------------------- planning: one launch or a chain
@pytest.mark.parametrize("J,B,N", [(1, 5.0, 2), (4097, 2.0, 2), (4097, 8.0, 2), (3000, 3.3, 2), (16384, 5.0, 2),
                                   (16385, 5.0, 2), (40001, 2.0, 3), (40001, 8.0, 3), (40001, 2.37, 3),
                                   (51200, 5.0, 8), (70000, 6.5, 4)])
def test_plan_single_block_and_multi_kernel_paths(J, B, N):
    """dq_plan allocates and reorders up to 16,384 super-groups in one
    single-block launch and above that with a chain of launches (metadata
    all-reduce with the first pass of the radix select, two more passes,
    the bitwidths with the tile scan, the scatter); both give the oracle's
    threshold, bitwidth counts, permutation and means (the two sizes around
    the switch, the all-2-bit and all-8-bit budgets on both sides, and a
    25 MB bucket of 8 ranks)."""
    _, gr = grads_for("bert_large_ring8", J * 256, N=N, seed=J)
    ar = DynamiQAllReduce(N, J, budget=B, correlated=True, seed=0)
    info = ar.plan([dev_u16(g) for g in gr], round=1)
    torch.cuda.synchronize()
    p = oracle.plan(oracle.Config(N, B, correlated=True, seed=0, round=1), gr)
    assert (info.n2, info.n4, info.n8) == tuple(int(c) for c in p.counts)
    assert bits32(np.array([info.T], np.float32))[0] == bits32(np.array([p.T], np.float32))[0]
    assert np.array_equal(host(ar.perm), p.perm)
    assert np.array_equal(bits32(host(ar.mu)), bits32(p.M / np.float32(N)))


@pytest.mark.parametrize("J", [900, 40001])
@pytest.mark.parametrize("fixed_bits", [2, 4, 8])
def test_plan_fixed_bits(J, fixed_bits):
    """The uniform-bitwidth ablation on both planning paths: every
    super-group gets the fixed width, the permutation is the identity, the
    counts are (J, 0, 0), (0, J, 0) or (0, 0, J) and T is reported as NaN
    (no threshold applies)."""
    N = 3
    _, gr = grads_for("bert_large_ring8", J * 256, N=N, seed=J + fixed_bits)
    ar = DynamiQAllReduce(N, J, budget=float(fixed_bits), fixed_bits=fixed_bits)
    info = ar.plan([dev_u16(g) for g in gr], round=1)
    torch.cuda.synchronize()
    assert (info.n2, info.n4, info.n8) == tuple(J if fixed_bits == w else 0 for w in (2, 4, 8))
    assert math.isnan(info.T)
    assert np.array_equal(host(ar.perm), np.arange(J, dtype=np.int32))
    p = oracle.plan(oracle.Config(N, float(fixed_bits), fixed_bits=fixed_bits), gr)
    assert np.array_equal(host(ar.perm), p.perm)
    assert np.array_equal(bits32(host(ar.mu)), bits32(p.M / np.float32(N)))


def test_plan_chain_reports_nonfinite_and_recovers():
    """Above the single-block size the chain's metadata all-reduce raises the
    non-finite flag (a NaN in one rank's gradient), and the next clean plan
    on the same workspace succeeds and equals the oracle's."""
    N, J = 2, 20000
    _, gr = grads_for("bert_large_ring8", J * 256, N=N, seed=11)
    ar = DynamiQAllReduce(N, J, budget=5.0)
    gd = [dev_u16(g) for g in gr]
    gd[1][256 * 17000 + 3] = float("nan")
    with pytest.raises(dq.NonFinite):
        ar.plan(gd, round=1)
    info = ar.plan([dev_u16(g) for g in gr], round=1)
    torch.cuda.synchronize()
    p = oracle.plan(oracle.Config(N, 5.0, round=1), gr)
    assert (info.n2, info.n4, info.n8) == tuple(int(c) for c in p.counts)
    assert np.array_equal(host(ar.perm), p.perm)


@pytest.mark.parametrize("N", [2, 8, 16, 32])
def test_butterfly_decode_outputs_match_fp32_rounded(N):
    """The butterfly's outputs, fp32 and bf16, in every rank equal: bf16 is
    the fp32 result rounded to nearest-even (one decode launch per 16
    outputs: 32 ranks take two)."""
    _, gr = grads_for("llama1b_butterfly8", 256 * 900 + 31, N, seed=N)
    J = gr[0].size // 256
    gd = [dev_u16(g) for g in gr]
    res = {}
    for dt in (torch.float32, torch.bfloat16):
        ar = DynamiQAllReduce(N, J, budget=5.0, correlated=True, butterfly=True, seed=4, out_dtype=dt)
        res[dt] = [o.clone() for o in ar(gd, round=3)]
    torch.cuda.synchronize()
    for a, b in zip(res[torch.float32], res[torch.bfloat16]):
        assert torch.equal(a.to(torch.bfloat16).view(torch.int16), b.view(torch.int16))
        assert torch.equal(a.view(torch.int32), res[torch.float32][0].view(torch.int32))
