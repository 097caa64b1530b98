"""Pins of the oracle's generator and its decode-accumulate rounding (CPU only).

* Philox4x32-10 against the published known-answer vectors (no dependency:
  the vectors are in tests/golden/philox4x32_10_kat.txt with their source).
* The decode-accumulate steps x = fl(sigma * q + a) -- the hop's accumulate
  (UINT8 and fp32 group scales, fp32 and bf16 addends) and the final decode's
  add-back of the mean -- against exact rational arithmetic rounded ONCE to
  binary32 by a rounding routine written here.  The inputs are chosen so that
  rounding the product first (two roundings) gives a different answer on many
  coordinates, so a two-rounding slip anywhere in these paths fails here.
"""
import os
from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
SG = 256


# --------------------------------------------------------------------------- Philox known answers
def _kat():
    rows = []
    with open(os.path.join(GOLD, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = [int(x, 16) for x in line.split()]
            assert len(w) == 10
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answer_vectors():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, want in rows:
        got = [int(x) for x in oracle.philox4x32_10(ctr, key)]
        assert got == want, (ctr, key)


def test_uniforms_come_from_the_known_answer_generator():
    """The first stochastic-rounding uniforms of a zero key and counter are
    the 16-bit halves of the first known-answer output (seed 0, round 0,
    stage word 0: independent rounding, hop 0, rank 0)."""
    _, _, want = _kat()[0]
    u = oracle.uniform16(np.arange(16), seed=0, round=0, n_ranks=1, hop=0, rank=0)
    for c in range(16):
        f = c & 7
        v = (want[f >> 1] >> (16 * (f & 1))) & 0xFFFF
        if c >= 8:
            v = (v + 0x8000) & 0xFFFF
        assert int(u[c]) == v, c


# --------------------------------------------------------------------------- exact rounding
def rne32(x: Fr) -> np.float32:
    """x rounded to the nearest binary32, ties to even (normal and subnormal
    range; no overflow in these tests)."""
    if x == 0:
        return np.float32(0.0)
    neg = x < 0
    a = -x if neg else x
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fr(2) ** e > a:
        e -= 1
    assert Fr(2) ** e <= a < Fr(2) ** (e + 1)
    q = max(e, -126) - 23                      # exponent of one unit in the last place
    s = a / Fr(2) ** q
    n = s.numerator // s.denominator
    rem = s - n
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and n % 2 == 1):
        n += 1
    v = float(n) * 2.0 ** q
    assert np.float32(v) == v                   # representable
    return np.float32(-v if neg else v)


def fr(v) -> Fr:
    return Fr(float(np.float32(v)))


def bits_of(a) -> np.ndarray:
    return np.asarray(a, np.float32).view(np.uint32)


def pack(codes, bits) -> np.ndarray:
    """LSB-first packing of 256 codes (coordinate i at bits [b i, b i + b))."""
    out = np.zeros(SG * bits // 8, np.uint8)
    for i, c in enumerate(codes):
        bit = bits * i
        out[bit >> 3] |= (int(c) << (bit & 7)) & 0xFF
    return out


def test_rne32_against_numpy_on_doubles():
    """The rounding routine agrees with the hardware's double -> float
    conversion wherever a double is the exact input."""
    rs = np.random.default_rng(3)
    x = rs.standard_normal(2000) * np.exp2(rs.integers(-140, 40, 2000))
    for v in x:
        assert rne32(Fr(float(v))) == np.float32(v)


def _setup(bits, seed):
    rs = np.random.default_rng(seed)
    q = oracle.level_table(bits)
    codes = rs.integers(0, 1 << bits, SG)
    return rs, q, codes


def _expect(sigma, q, codes, add):
    """(one rounding, two roundings) of sigma_g * q_code + add, exactly."""
    one, two = np.zeros(SG, np.float32), np.zeros(SG, np.float32)
    for i in range(SG):
        p = fr(sigma[i // 16]) * fr(q[codes[i]])
        one[i] = rne32(p + fr(add[i]))
        two[i] = rne32(fr(rne32(p)) + fr(add[i]))
    return one, two


def _cancelling_addends(rs, sigma, q, codes):
    """Half the addends are -fl(sigma q) (the exact sum is then the product's
    rounding error, which two roundings turn into 0), the rest random fp32 of
    the same magnitude."""
    add = np.zeros(SG, np.float32)
    for i in range(SG):
        prod = np.float32(sigma[i // 16]) * np.float32(q[codes[i]])   # IEEE binary32 product
        if i % 2 == 0:
            add[i] = -prod
        else:
            add[i] = np.float32(rs.standard_normal() * float(sigma[i // 16]))
    return add


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_decode_add_uint8_scales_rounds_once(bits):
    rs, q, codes = _setup(bits, 10 + bits)
    e = -3
    E = 127 + e
    u = rs.integers(1, 256, 16).astype(np.uint8)
    sigma = [float(Fr(int(x)) * Fr(2) ** e) for x in u]          # exact in binary32
    add = _cancelling_addends(rs, sigma, q, codes)
    one, two = _expect(sigma, q, codes, add)
    got = oracle.decode_add_sg(E, u, pack(codes, bits), bits, add)
    assert np.array_equal(bits_of(got), bits_of(one))
    assert np.count_nonzero(bits_of(one) != bits_of(two)) >= SG // 8


def test_decode_add_exponent_byte_zero_decodes_to_the_addend():
    rs, q, codes = _setup(4, 5)
    add = rs.standard_normal(SG).astype(np.float32)
    got = oracle.decode_add_sg(0, np.full(16, 200, np.uint8), pack(codes, 4), 4, add)
    assert np.array_equal(bits_of(got), bits_of(add))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_decode_add_fp32_scales_rounds_once(bits):
    rs, q, codes = _setup(bits, 20 + bits)
    sig = (rs.uniform(0.5, 2.0, 16) * 2.0 ** -5).astype(np.float32)   # full 24-bit mantissas
    add = _cancelling_addends(rs, sig, q, codes)
    one, two = _expect(sig, q, codes, add)
    got = oracle.decode_add_sg_f32(sig, pack(codes, bits), bits, add)
    assert np.array_equal(bits_of(got), bits_of(one))
    assert np.count_nonzero(bits_of(one) != bits_of(two)) >= SG // 8


def _message(E, u, codes_packed):
    """Message of one super-group with UINT8 scales: [E padded to 16][16 u][codes]."""
    m = np.zeros(16 + 16 + codes_packed.size, np.uint8)
    m[0] = E
    m[16:32] = u
    m[32:] = codes_packed
    return m


def _counts(bits):
    return {2: (1, 0), 4: (0, 1), 8: (0, 0)}[bits]


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N", [1, 3])
def test_final_decode_adds_back_the_mean_with_one_rounding(bits, N):
    """out = fl(sigma q + fl(mu N)), mu = fl(M / N).  With N = 1 the mean is
    -fl(sigma_0 q_k) for the code k that every coordinate of group 0 carries,
    so two roundings would give exactly 0 there."""
    rs, q, codes = _setup(bits, 30 + bits + N)
    e = 2
    u = rs.integers(1, 256, 16).astype(np.uint8)
    sigma = [float(Fr(int(x)) * Fr(2) ** e) for x in u]
    k = 1                                           # an inner level: sigma * q_k is inexact
    codes[:16] = k
    if N == 1:
        M = -(np.float32(sigma[0]) * np.float32(q[k]))
    else:   # an M for which fl(fl(M / 3) * 3) != M, so the product's rounding shows
        c = (rs.standard_normal(4096) * 300.0).astype(np.float32)
        hit = (c / np.float32(N)) * np.float32(N) != c        # binary32 steps (candidates only)
        M = c[np.argmax(hit)]
    mu = rne32(fr(M) / N)
    back = rne32(fr(mu) * N)
    assert N == 1 or back != M
    one, two = _expect(sigma, q, codes, np.full(SG, back, np.float32))
    N2, N4 = _counts(bits)
    cfg = oracle.Config(N, 5.0)
    got = oracle.decode(cfg, 0, 1, N2, N4, _message(127 + e, u, pack(codes, bits)), np.array([M], np.float32),
                        np.array([0], np.int32))
    assert np.array_equal(bits_of(got), bits_of(one))
    if N == 1:
        assert np.all(two[:16] == 0) and np.all(one[:16] != 0)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_hop_accumulate_of_a_bf16_gradient(bits):
    """A ring hop's accumulate: x = fl(sigma q + fl(float(g) - mu)) over the
    kept range (the fp32 output of a split DAR), mu = fl(M / N)."""
    rs, q, codes = _setup(bits, 40 + bits)
    N, e = 4, 0
    u = rs.integers(1, 256, 16).astype(np.uint8)
    sigma = [float(Fr(int(x)) * Fr(2) ** e) for x in u]
    g = (rs.standard_normal(SG) * 60.0).astype(np.float32)
    g_u16 = (g.view(np.uint32) >> 16).astype(np.uint16)          # truncation: any bf16 will do
    M = np.float32(rs.standard_normal() * 7.0)
    mu = rne32(fr(M) / N)
    a = np.array([rne32(Fr(float(np.uint32(int(h) << 16).view(np.float32))) - fr(mu)) for h in g_u16],
                 np.float32)
    one, two = _expect(sigma, q, codes, a)
    N2, N4 = _counts(bits)
    cfg = oracle.Config(N, 5.0)
    _, keep = oracle.dar(cfg, 0, 1, N2, N4, 1, 1, _message(127 + e, u, pack(codes, bits)), g_u16,
                         np.array([M], np.float32), np.array([0], np.int32), send=(0, 0), keep=(0, 1))
    assert np.array_equal(bits_of(keep), bits_of(one))
    assert np.count_nonzero(bits_of(one) != bits_of(two)) >= 1


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_hop_accumulate_of_an_fp32_partial(bits):
    rs, q, codes = _setup(bits, 50 + bits)
    e = -1
    u = rs.integers(1, 256, 16).astype(np.uint8)
    sigma = [float(Fr(int(x)) * Fr(2) ** e) for x in u]
    add = _cancelling_addends(rs, sigma, q, codes)
    one, two = _expect(sigma, q, codes, add)
    N2, N4 = _counts(bits)
    _, keep = oracle.dar(oracle.Config(8, 5.0), 0, 1, N2, N4, 0, 2, _message(127 + e, u, pack(codes, bits)),
                         add, np.array([0.0], np.float32), np.array([0], np.int32), send=(0, 0), keep=(0, 1))
    assert np.array_equal(bits_of(keep), bits_of(one))
    assert np.count_nonzero(bits_of(one) != bits_of(two)) >= SG // 8
