"""Pins of the oracle's ablation modes and of its MXFP8 comparison baseline.

MXFP8 follows the OCP Microscaling (MX) v1.0 formats that the pages cite
for their MXFP baselines: E4M3 elements, one E8M0 scale per 32 elements.
The E4M3 code table and in-range rounding are checked against torch's
independent float8_e4m3fn conversion; the block scale against its closed
form; the all-reduce schedule against special cases that are exact and a
message-level restatement.  The ablation modes (fixed bitwidth, fp32 group
scales) are checked against exactness cases, unbiasedness and the identity
with the default path where the two must coincide.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_hop_gradient_gb300 import synth


def _bf16(x) -> np.ndarray:
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32_of_bf16(u) -> np.ndarray:
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- E4M3
def test_e4m3_code_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and np.isnan(ours).sum() == 2
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    # the format's landmarks: largest 448, smallest subnormal 2^-9, smallest normal 2^-6
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6


def test_e4m3_rounding_matches_torch_in_range():
    """Nearest, ties to even: random values over the whole range, every
    midpoint between neighbouring codes and the values just beside them."""
    rs = np.random.default_rng(0)
    mags = np.exp2(rs.uniform(-12, math.log2(460), 20000))
    vals = [mags * rs.choice([-1, 1], mags.size)]
    pos = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mid = (pos[:-1] + pos[1:]) / 2
    for m in (mid, np.nextafter(mid, 0), np.nextafter(mid, 1e9)):
        vals += [m, -m]
    vals.append(np.array([0.0, -0.0, 448.0, -448.0, 463.9, 2.0 ** -10, 2.0 ** -11]))
    v = np.concatenate(vals).astype(np.float32)
    v = v[np.abs(v) < 464]                       # torch turns larger values into NaN
    ref = torch.as_tensor(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(x)) for x in v], np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_keeps_sign():
    for x in (448.0, 464.0, 480.0, 1000.0, 3.0e38):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-9) == 0x80      # rounds to zero, keeps the sign
    # exact ties go to the even code: 1 + 1/16 -> 1, 1 + 3/16 -> 1.25
    assert oracle.e4m3_encode(1.0625) == 0x38
    assert oracle.e4m3_encode(1.1875) == 0x3A
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00 and oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02


# --------------------------------------------------------------------------- MX blocks
@pytest.mark.parametrize("k", [-140, -119, -100, -8, -1, 0, 1, 7, 8, 9, 60, 120])
def test_mx_block_scale_closed_form(k):
    """X = 2^(floor(log2 amax) - 8), clamped at 2^-127; byte = exponent + 127."""
    rs = np.random.default_rng(k + 200)
    amax = np.float32(2.0 ** k * 1.5)
    v = (rs.uniform(-1, 1, 32) * float(amax)).astype(np.float32)
    v[5] = -amax
    X, P = oracle.mx_encode_block(v)
    assert X == max(k - 8, -127) + 127
    x = X - 127
    dec = np.array([oracle.e4m3_value(c) for c in P]) * 2.0 ** x
    if k - 8 >= -127:
        assert dec[5] == -float(amax)             # 1.5 * 2^8 = 384 is a code
    # error bound of one rounding to E4M3 (no saturation: amax / X < 448)
    err = np.abs(dec - v.astype(np.float64))
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** (x - 10))
    assert np.all(err <= bound)


def test_mx_block_zero_and_saturation():
    X, P = oracle.mx_encode_block(np.zeros(32, np.float32))
    assert X == 0 and np.all(P == 0)
    v = np.zeros(32, np.float32)
    v[0], v[1] = 500.0, 300.0                     # amax 500 -> X = 2^0, 500 saturates to 448
    X, P = oracle.mx_encode_block(v)
    assert X == 127 and P[0] == 0x7E and oracle.e4m3_value(P[1]) == 288.0
    # decoding is element x scale: a negative zero stays negative
    msg = oracle.mx_quantize(np.concatenate([[-0.0, 0.0, -1e-30], np.ones(29)]).astype(np.float32))
    d = oracle.mx_dequantize(msg, 1)
    assert list(np.signbit(d[:3])) == [True, False, True] and np.all(d[:3] == 0)


def test_mx_roundtrip_exact_on_representable_blocks():
    rs = np.random.default_rng(3)
    for t in range(50):
        codes = rs.integers(0, 0x7F, 32)          # finite non-negative codes
        codes[rs.integers(0, 32)] = rs.integers(0x78, 0x7F)   # max has exponent 8: X = 2^x exactly
        sgn = rs.choice([1.0, -1.0], 32)
        x = int(rs.integers(-100, 100))
        v = np.array([oracle.e4m3_value(c) for c in codes]) * sgn * 2.0 ** x
        msg = oracle.mx_quantize(v.astype(np.float32))
        assert msg[0] == x + 127
        assert np.array_equal(oracle.mx_dequantize(msg, 1), v.astype(np.float32))


def test_mx_message_layout():
    for n in (1, 15, 16, 17, 100):
        assert oracle.mx_message_bytes(n) == -(-n // 16) * 16 + 32 * n
    x = np.random.default_rng(1).normal(size=32 * 20).astype(np.float32)
    msg = oracle.mx_quantize(x)
    for k in (0, 7, 19):
        X, P = oracle.mx_encode_block(x[32 * k: 32 * k + 32])
        assert msg[k] == X and np.array_equal(msg[32 + 32 * k: 64 + 32 * k], P)


# --------------------------------------------------------------------------- MX all-reduce
def test_mx_allreduce_one_rank_is_quantize_dequantize():
    g = _bf16(np.random.default_rng(5).normal(size=32 * 64) * 3)
    for butterfly in (False, True):
        out = oracle.mx_allreduce(1, [g], butterfly=butterfly)
        assert np.array_equal(out, oracle.mx_dequantize(oracle.mx_quantize(_f32_of_bf16(g)), 64))


@pytest.mark.parametrize("N", [2, 4, 8])
def test_mx_allreduce_single_contributor_is_exact(N):
    """If one worker holds MX-representable values and the others zeros,
    every hop re-encodes the same values: the sum is exact, whichever worker
    holds them (checks that every worker's data enters the sum)."""
    rs = np.random.default_rng(N)
    nb = 4 * N + 3
    codes = rs.integers(0x38, 0x70, 32 * nb)      # values in [1, 256): 4 significant bits, bf16-exact
    codes[(codes & 7) == 7] -= 1                  # no mantissa 1.875: a block max 1.875 * 2^e scales to
                                                  # 480 > 448 and saturates (the format's clipping)
    v = np.array([oracle.e4m3_value(c) for c in codes]) * rs.choice([1.0, -1.0], codes.size)
    v = v.astype(np.float32)
    z = np.zeros_like(v)
    for who in range(N):
        gr = [_bf16(v if r == who else z) for r in range(N)]
        for butterfly in (False, True):
            assert np.array_equal(oracle.mx_allreduce(N, gr, butterfly=butterfly), v)


def test_mx_ring_by_messages_equals_per_block():
    """The ring restated over whole chunk messages (mx_quantize /
    mx_dequantize) gives the per-block result, bit for bit."""
    N, nb = 4, 37
    rs = np.random.default_rng(11)
    gr = [_bf16(rs.standard_t(3, 32 * nb) * np.exp(rs.normal())) for _ in range(N)]
    lo = oracle.mx_chunk_lo(nb, N)
    out = np.zeros(32 * nb, np.float32)
    for c in range(N):
        a, b = lo[c], lo[c + 1]
        x = _f32_of_bf16(gr[(c + 1) % N][32 * a: 32 * b])
        for t in range(1, N):
            msg = oracle.mx_quantize(x)
            x = oracle.mx_dequantize(msg, b - a) + _f32_of_bf16(gr[(c + 1 + t) % N][32 * a: 32 * b])
        out[32 * a: 32 * b] = oracle.mx_dequantize(oracle.mx_quantize(x), b - a)
    assert np.array_equal(out, oracle.mx_allreduce(N, gr))


def test_mx_allreduce_error_within_per_hop_bound():
    """Each of the N encodings adds at most 2^-4 of its input's magnitude (no
    saturation here): |out - s| <= sum over hops of the bound."""
    N = 4
    rs = np.random.default_rng(2)
    gr = [_bf16(rs.normal(size=32 * 50)) for _ in range(N)]
    s = oracle.exact_sum(gr)
    out = oracle.mx_allreduce(N, gr).astype(np.float64)
    absum = sum(np.abs(_f32_of_bf16(g)).astype(np.float64) for g in gr)
    blkmax = np.repeat(absum.reshape(-1, 32).max(axis=1), 32)
    assert np.all(np.abs(out - s) <= N * (2.0 ** -4 * 1.07 * absum + 2.0 ** -10 * blkmax))


# --------------------------------------------------------------------------- ablation: fp32 scales
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_f32_scales_are_group_maxima_and_exact_on_levels(bits):
    rs = np.random.default_rng(bits)
    q = oracle.level_table(bits)
    k = rs.integers(0, 1 << bits, 256)
    m = rs.integers(-20, 20, 16)
    x = (q[k] * np.repeat(2.0 ** m, 16)).astype(np.float32)
    for g in range(16):                           # every group holds its +-2^m (level +-1)
        x[16 * g] = 2.0 ** m[g] * (1 if g % 2 else -1)
        k[16 * g] = (1 << bits) - 1 if g % 2 else 0
    sig, codes = oracle.quantize_sg_f32(x, bits, seed=1)
    assert np.array_equal(sig, np.abs(x).reshape(16, 16).max(axis=1))
    assert np.array_equal(oracle.unpack_codes(codes, bits), k)
    assert np.array_equal(oracle.decode_add_sg_f32(sig, codes, bits, np.zeros(256)), x)


@pytest.mark.parametrize("bits", [2, 4])
def test_f32_scales_unbiased_monte_carlo(bits):
    rs = np.random.default_rng(40 + bits)
    x = (rs.normal(size=256) * np.exp(rs.normal(0, 1, 256))).astype(np.float32)
    xd = x.astype(np.float64)
    R = 3000
    acc = np.zeros(256)
    acc2 = np.zeros(256)
    for r in range(R):
        sig, codes = oracle.quantize_sg_f32(x, bits, seed=9, round=r, n_ranks=4, correlated=True,
                                            rank=r % 4, hop=r % 3, slot=r % 2, n_slots=2)
        dev = oracle.decode_add_sg_f32(sig, codes, bits, np.zeros(256)).astype(np.float64) - xd
        acc += dev
        acc2 += dev * dev
    bias = acc / R
    se = np.sqrt(np.maximum(acc2 / R - bias ** 2, 0) / R)
    sigma = np.repeat(np.abs(x).reshape(16, 16).max(axis=1).astype(np.float64), 16)
    assert np.all(np.abs(bias) <= 5 * se + sigma * 2.0 ** -15 + 1e-6 * np.abs(xd))
    assert abs(bias.sum() / math.sqrt((se ** 2).sum())) < 5


def test_f32_scale_message_layout():
    for n2, n4, n8 in [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 5, 7), (0, 0, 0)]:
        c = n2 + n4 + n8
        assert oracle.message_bytes(n2, n4, n8, True) == 64 * c + 64 * n2 + 128 * n4 + 256 * n8


def _grads(name, n, seed=1, **kw):
    w = synth.WORKLOADS[name].scaled(n, **kw)
    return w, [synth.as_u16(g) for g in synth.generate(w, "cpu", seed=seed)]


def test_f32_scale_message_path_equals_per_supergroup_path():
    """Range-level compress / DAR / decode of a ring in fp32-scale mode
    against the per-super-group walk."""
    w, gr = _grads("ring4_1m", 256 * 40)
    N = w.n_ranks
    cfg = oracle.Config(N, 5.0, correlated=True, round=2, scale_fp32=True)
    p = oracle.plan(cfg, gr)
    N2, N4 = int(p.counts[0]), int(p.counts[1])
    lo = p.chunk_lo
    out = np.zeros(gr[0].size, np.float32)
    for c in range(N):
        a, b = int(lo[c]), int(lo[c + 1])
        msg = oracle.compress(cfg, a, b, N2, N4, (c + 1) % N, 0, gr[(c + 1) % N], p.M, p.perm)
        for t in range(1, N):
            rk = (c + 1 + t) % N
            msg, _ = oracle.dar(cfg, a, b, N2, N4, rk, t, msg, gr[rk], p.M, p.perm, send=(a, b))
        oracle.decode(cfg, a, b, N2, N4, msg, p.M, p.perm, out)
    _, ref = oracle.allreduce(cfg, gr)
    assert np.array_equal(out, ref)


# --------------------------------------------------------------------------- ablation: fixed bitwidth
def test_fixed_bits_plan_and_identity_at_eight_bits():
    w, gr = _grads("bert_large_ring8", 256 * 96)
    for fb in (2, 4, 8):
        p = oracle.plan(oracle.Config(w.n_ranks, 5.0, fixed_bits=fb), gr)
        assert np.all(p.b == fb) and math.isnan(p.T)
        assert np.array_equal(p.perm, np.arange(p.b.size))
        assert p.counts.tolist() == [p.b.size * (fb == k) for k in (2, 4, 8)]
    # budget 8 allocates 8 bits everywhere: the same all-reduce, bit for bit
    for butterfly in (False, True):
        _, a = oracle.allreduce(oracle.Config(8, 8.0, correlated=True, round=4), gr, butterfly)
        _, b = oracle.allreduce(oracle.Config(8, 8.0, correlated=True, round=4, fixed_bits=8), gr, butterfly)
        assert np.array_equal(a, b)


def test_ablations_order_as_the_pages_claim():
    """Variable bitwidth beats uniform bitwidth at the same code bits (4),
    non-uniform levels beat uniform ones, correlated rounding beats
    independent rounding in the butterfly."""
    def v(cfg, gr, butterfly=False, rounds=3):
        return np.mean([oracle.vnmse(oracle.allreduce(oracle.Config(**{**cfg, "round": r}), gr, butterfly)[1], gr)
                        for r in range(rounds)])
    w, gr = _grads("bert_large_ring8", 1 << 16)
    base = dict(n_ranks=8, correlated=True)
    assert v({**base, "budget": 4.0}, gr) < v({**base, "budget": 4.0, "fixed_bits": 4}, gr)
    w, gr = _grads("llama1b_butterfly8", 1 << 16)
    assert v({**base, "budget": 5.0}, gr, True) < v({**base, "budget": 5.0, "eps": math.inf}, gr, True)
    assert v({**base, "budget": 5.0}, gr, True) < v({**base, "budget": 5.0, "correlated": False}, gr, True)
