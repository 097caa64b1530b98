"""GPU parity of the ablation modes, the larger rank counts and the MXFP8
comparison baseline, through the C ABI, against the oracle.

Bar: bit-exact outputs, plans and final chunk messages (both sides perform
the same correctly rounded fp32 steps and the same integer decisions).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import build, dq, synth
from quantized_hop_gradient_gb300.allreduce import DynamiQAllReduce, MXFP8AllReduce

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    dq.lib()


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def host(t):
    return t.detach().cpu().numpy()


def bits32(a):
    return np.ascontiguousarray(a, np.float32).view(np.int32)


def grads_for(name, n, N=None, seed=0):
    w = synth.WORKLOADS[name].scaled(n)
    if N is not None:
        w = w.__class__(**{**w.__dict__, "n_ranks": N})
    return [synth.as_u16(g) for g in synth.generate(w, "cpu", seed=seed)]


def _final_meta_and_codes(m, cnt, n2, n4, s, scale_fp32):
    """Metadata record (65 bytes, the oracle's layout) and code block of
    local super-group s of a final message."""
    meta = np.zeros(65, np.uint8)
    if scale_fp32:
        meta[1:65] = m[64 * s: 64 * s + 64]
        base = 64 * cnt
    else:
        off_u = -(-cnt // 16) * 16
        meta[0] = m[s]
        meta[1:17] = m[off_u + 16 * s: off_u + 16 * s + 16]
        base = off_u + 16 * cnt
    if s < n2:
        blk = m[base + 64 * s: base + 64 * s + 64]
    elif s < n2 + n4:
        o = base + 64 * n2
        blk = m[o + 128 * (s - n2): o + 128 * (s - n2) + 128]
    else:
        o = base + 64 * n2 + 128 * n4
        blk = m[o + 256 * (s - n2 - n4): o + 256 * (s - n2 - n4) + 256]
    return meta, blk


def _check(gr, N, butterfly, B=5.0, eps=1.0, correlated=True, fixed_bits=0, scale_fp32=False, seed=3):
    J = gr[0].size // 256
    ar = DynamiQAllReduce(N, J, budget=B, eps=eps, correlated=correlated, butterfly=butterfly, seed=seed,
                          fixed_bits=fixed_bits, scale_fp32=scale_fp32)
    outs = ar([dev_u16(g) for g in gr], round=5)
    torch.cuda.synchronize()
    cfg = oracle.Config(N, B, eps=eps, correlated=correlated, seed=seed, round=5, fixed_bits=fixed_bits,
                        scale_fp32=scale_fp32)
    p = oracle.plan(cfg, gr)
    assert [ar.info.n2, ar.info.n4, ar.info.n8] == p.counts.tolist()
    if fixed_bits:
        assert math.isnan(ar.info.T)
    else:
        assert bits32(np.array([ar.info.T]))[0] == bits32(np.array([p.T]))[0]
    assert np.array_equal(host(ar.perm), p.perm)
    sel = np.arange(J, dtype=np.int64)
    rows, fin = oracle.allreduce_sg(cfg, butterfly, gr, p.M, p.perm, int(p.counts[0]), int(p.counts[1]),
                                    p.chunk_lo, sel)
    exp = np.zeros(J * 256, np.float32)
    exp.reshape(J, 256)[p.perm] = rows
    o0 = host(outs[0])
    assert np.array_equal(bits32(o0), bits32(exp))
    assert np.array_equal(bits32(host(outs[-1])), bits32(o0))
    lo = ar.chunk_lo()
    for c in range(N):
        a, b = lo[c], lo[c + 1]
        if b == a:
            continue
        m = ar.final_message(c).numpy()
        n2, n4, _ = oracle.range_counts(a, b, ar.info.n2, ar.info.n4)
        if not scale_fp32:
            assert np.all(m[b - a: -(-(b - a) // 16) * 16] == 0)   # zero E padding, as the oracle writes it
        for s in range(b - a):
            meta, blk = _final_meta_and_codes(m, b - a, n2, n4, s, scale_fp32)
            f = fin[a + s]
            assert np.array_equal(meta, f[:65])
            assert np.array_equal(blk, f[65:65 + blk.size])
    return oracle.vnmse(o0, gr)


# --------------------------------------------------------------------------- ablations
@pytest.mark.parametrize("butterfly", [False, True])
def test_ablation_fp32_scales(butterfly):
    gr = grads_for("llama1b_butterfly8", 256 * 1200 + 99, N=8, seed=1)
    _check(gr, 8, butterfly, scale_fp32=True)
    _check(gr, 8, butterfly, scale_fp32=True, eps=math.inf, correlated=False)


@pytest.mark.parametrize("fixed_bits", [2, 4, 8])
@pytest.mark.parametrize("butterfly", [False, True])
def test_ablation_fixed_bits(fixed_bits, butterfly):
    gr = grads_for("bert_large_ring8", 256 * 900, N=8, seed=2)
    _check(gr, 8, butterfly, B=float(fixed_bits), fixed_bits=fixed_bits)


def test_ablation_uniform_levels_and_independent_rounding():
    gr = grads_for("gemma1b_ring16", 256 * 700, N=16, seed=4)
    _check(gr, 16, False, eps=math.inf)
    _check(gr, 16, True, correlated=False)


def test_single_call_entry_points_fp32_scales():
    """dq_compress / dq_dar / dq_decode in fp32-scale mode, message bytes and
    decoded values against the oracle's range operations."""
    N = 4
    gr = grads_for("ring4_1m", 256 * 500, N=N, seed=6)
    p = oracle.plan(oracle.Config(N, 5.0), gr)
    mu = torch.from_numpy(p.M / np.float32(N)).to(DEV)
    perm = torch.from_numpy(p.perm).to(DEV)
    N2, N4 = int(p.counts[0]), int(p.counts[1])
    cfg_o = oracle.Config(N, 5.0, correlated=True, seed=2, round=9, scale_fp32=True)
    cfg = dq.config(N, 5.0, correlated=True, seed=2, round=9, scale_fp32=True)
    for (a, b) in [(0, 500), (3, 211), (N2 - 2, N2 + N4 + 3), (N2 + N4, 500)]:
        r = dq.rng(a, b, N2, N2 + N4)
        nb = dq.dq_message_bytes(r, True)
        assert nb == oracle.range_message_bytes(a, b, N2, N4, True)
        msg = torch.zeros(nb, dtype=torch.uint8, device=DEV)
        dq.dq_compress(cfg, r, dq.stage(1, 0), dev_u16(gr[1]), mu, perm, msg)
        exp = oracle.compress(cfg_o, a, b, N2, N4, 1, 0, gr[1], p.M, p.perm)
        assert np.array_equal(host(msg), exp)
        mid = (a + b) // 2
        addend = np.random.default_rng(a).standard_normal((b - a) * 256).astype(np.float32)
        sr, kr = dq.rng(a, mid, N2, N2 + N4), dq.rng(mid, b, N2, N2 + N4)
        out = torch.zeros(max(1, dq.dq_message_bytes(sr, True)), dtype=torch.uint8, device=DEV)
        keep = torch.zeros(max(1, (b - mid) * 256), device=DEV)
        dq.dq_dar(cfg, r, dq.stage(2, 1, 0, 2), msg, torch.from_numpy(addend).to(DEV), True, mu, perm, sr, out,
                  kr, keep)
        eo, ek = oracle.dar(cfg_o, a, b, N2, N4, 2, 1, exp, addend, p.M, p.perm, send=(a, mid), keep=(mid, b),
                            slot=0, n_slots=2)
        assert np.array_equal(host(out)[: eo.size], eo)
        assert np.array_equal(bits32(host(keep)[: ek.size]), bits32(ek))
        o32 = torch.zeros(p.b.size * 256, device=DEV)
        dq.dq_decode(cfg, r, msg, mu, perm, o32)
        assert np.array_equal(bits32(host(o32)), bits32(oracle.decode(cfg_o, a, b, N2, N4, exp, p.M, p.perm)))


# --------------------------------------------------------------------------- more ranks
@pytest.mark.parametrize("N", [32, 64])
@pytest.mark.parametrize("butterfly", [False, True])
def test_many_ranks(N, butterfly):
    gr = grads_for("llama1b_butterfly8", 256 * 1024 + 5, N=N, seed=N)
    _check(gr, N, butterfly)


# --------------------------------------------------------------------------- MXFP8 baseline
def _mx_cases():
    rs = np.random.default_rng(0)
    blocks = [rs.normal(size=32) * 10.0 ** rs.uniform(-30, 30) for _ in range(300)]
    blocks.append(np.zeros(32))
    blocks.append(-np.zeros(32))
    t = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (t[:-1] + t[1:]) / 2                       # ties after the scaling (max 448 = 2^8 * 1.75)
    for k in range(0, mids.size - 31, 31):
        b = np.concatenate([[448.0], mids[k:k + 31]]) * rs.choice([-1, 1], 32)
        blocks.append(b * 2.0 ** rs.integers(-20, 20))
    blocks.append(np.concatenate([[480.0, 500.0, -511.0], rs.uniform(-500, 500, 29)]))   # saturation
    blocks.append(np.concatenate([[1.0], -rs.uniform(0, 2.0 ** -11, 31)]))               # signed zeros
    blocks.append(rs.normal(size=32) * 2.0 ** -140)                                      # subnormal max
    blocks.append(rs.normal(size=32) * 2.0 ** 120)
    return np.concatenate(blocks).astype(np.float32)


def test_mx_quantize_dequantize_bit_exact():
    x = _mx_cases()
    n_blk = x.size // 32
    xd = torch.from_numpy(x).to(DEV)
    msg = torch.zeros(dq.dq_mx_message_bytes(n_blk), dtype=torch.uint8, device=DEV)
    dq.dq_mx_quantize(xd, n_blk, msg)
    exp = oracle.mx_quantize(x)
    assert np.array_equal(host(msg), exp)
    out = torch.zeros(x.size, device=DEV)
    dq.dq_mx_dequantize(msg, n_blk, out)
    assert np.array_equal(bits32(host(out)), bits32(oracle.mx_dequantize(exp, n_blk)))


@pytest.mark.parametrize("N,butterfly", [(1, False), (1, True), (3, False), (4, False), (4, True), (8, False),
                                         (8, True), (64, True)])
def test_mx_allreduce_bit_exact(N, butterfly):
    gr = grads_for("llama1b_butterfly8", 256 * 300 + 32 * 5, N=N, seed=N)   # ragged: n_blk not a multiple of N
    n = gr[0].size
    mx = MXFP8AllReduce(N, n, butterfly=butterfly)
    outs = mx([dev_u16(g) for g in gr])
    torch.cuda.synchronize()
    n_blk = n // 32
    rows, fin = oracle.mx_allreduce_blk(N, butterfly, gr, np.arange(n_blk, dtype=np.int64))
    exp = rows.reshape(-1)
    for o in outs:
        assert np.array_equal(bits32(host(o)), bits32(exp))
    lo = mx.chunk_lo()
    for c in range(N):
        a, b = lo[c], lo[c + 1]
        if b == a:
            continue
        m = mx.final_message(c).numpy()
        pad = -(-(b - a) // 16) * 16
        assert np.array_equal(m[: b - a], fin[a:b, 0])
        assert np.all(m[b - a: pad] == 0)                  # zero padding, as the oracle writes it
        assert np.array_equal(m[pad: pad + 32 * (b - a)].reshape(-1, 32), fin[a:b, 1:])


def test_mx_launch_log_and_counts():
    N = 4
    gr = grads_for("ring4_1m", 256 * 64, N=N)
    mx = MXFP8AllReduce(N, gr[0].size)
    log = dq.LaunchLog(64)
    before = dq.dq_launch_count()
    mx([dev_u16(g) for g in gr], log=log)
    torch.cuda.synchronize()
    kinds = [k for k, _, _ in log.launches()]
    assert kinds == [dq.DQ_LAUNCH_MX_HOP] * N + [dq.DQ_LAUNCH_MX_DECODE]
    assert dq.dq_launch_count() - before == N + 1
