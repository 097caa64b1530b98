"""Oracle for the DynamiQ quantized multi-hop all-reduce -- TEST INFRASTRUCTURE.

A plain, slow CPU statement of what the hot path computes (``dq_oracle.c``),
wrapped for numpy.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library and never calls it; the library never
imports this package.

Inputs are numpy arrays: bf16 gradients as ``uint16`` bit patterns, fp32 as
``float32``.  See ``dq_oracle.c`` for the method, the readings of the pages
and the citations.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dq_oracle.c")
_SO = os.path.join(_HERE, "_build", "libdq_oracle.so")
_lock = threading.Lock()
_lib = None

SG = 256


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-ffp-contract=off: no FMA contraction)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def _p(a, t):
    return a.ctypes.data_as(C.POINTER(t))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            i64, i32, u64 = C.c_int64, C.c_int32, C.c_uint64
            P = C.c_void_p
            L.or_philox4x32_10.argtypes = [P, P, P]
            L.or_uniform16.argtypes = [P, i64]
            L.or_uniform16.restype = C.c_uint32
            L.or_level_table.argtypes = [C.c_int, C.c_double, P]
            L.or_gap_table.argtypes = [C.c_int, P, P]
            L.or_stats.argtypes = [P, i64, P, P]
            L.or_stats_reduce.argtypes = [P, P, i32, i64, P, P]
            L.or_bits_for.argtypes = [C.c_float, C.c_float]
            L.or_allocate.argtypes = [P, i64, C.c_float, P, P, P]
            L.or_reorder.argtypes = [P, i64, P]
            L.or_chunk_cuts.argtypes = [P, P, i64, i32, P]
            L.or_message_bytes.argtypes = [i64, i64, i64, i32]
            L.or_message_bytes.restype = i64
            L.or_quantize_sg.argtypes = [P, C.c_int, P, P, P, i64, P, P, P]
            L.or_quantize_sg_f32.argtypes = [P, C.c_int, P, P, P, i64, P, P]
            L.or_dequantize_sg.argtypes = [C.c_uint8, P, P, C.c_int, P, P]
            L.or_decode_add_sg.argtypes = [C.c_uint8, P, P, C.c_int, P, P, P]
            L.or_decode_add_sg_f32.argtypes = [P, P, C.c_int, P, P, P]
            L.or_e4m3_value.argtypes = [C.c_uint8]
            L.or_e4m3_value.restype = C.c_double
            L.or_e4m3_encode.argtypes = [C.c_double]
            L.or_e4m3_encode.restype = C.c_uint8
            L.or_mx_encode_block.argtypes = [P, P, P]
            L.or_mx_decode_add_block.argtypes = [C.c_uint8, P, P, P]
            L.or_mx_message_bytes.argtypes = [i64]
            L.or_mx_message_bytes.restype = i64
            L.or_mx_quantize.argtypes = [P, i64, P]
            L.or_mx_dequantize.argtypes = [P, i64, P]
            L.or_mx_allreduce_blk.argtypes = [i32, i32, P, i64, P, i64, P, P]
            L.or_compress.argtypes = [P, i64, i64, i64, i64, i32, i32, i32, i32, P, P, P, P]
            L.or_dar.argtypes = [P, i64, i64, i64, i64, i32, i32, i32, i32, P, P, i32, P, P,
                                 i64, i64, P, i64, i64, P]
            L.or_decode.argtypes = [P, i64, i64, i64, i64, P, P, P, P]
            L.or_allreduce_sg.argtypes = [P, i32, P, P, P, i64, i64, P, P, i64, P, P]
            _lib = L
    return _lib


class _Cfg(C.Structure):
    _fields_ = [("n_ranks", C.c_int32), ("budget", C.c_float), ("eps", C.c_double),
                ("correlated", C.c_int32), ("seed", C.c_uint64), ("round", C.c_uint64),
                ("fixed_bits", C.c_int32), ("scale_fp32", C.c_int32)]


class _Rng(C.Structure):
    _fields_ = [("seed", C.c_uint64), ("round", C.c_uint64), ("n_ranks", C.c_int32),
                ("correlated", C.c_int32), ("hop", C.c_int32), ("rank", C.c_int32),
                ("slot", C.c_int32), ("n_slots", C.c_int32)]


@dataclass
class Config:
    """One all-reduce round.  Ablation switches: ``eps=inf`` (uniform levels),
    ``correlated=False``, ``fixed_bits`` in {2, 4, 8} (uniform bitwidth, no
    allocation) and ``scale_fp32`` (group scales in fp32, no UINT8 level)."""
    n_ranks: int
    budget: float = 5.0
    eps: float = 1.0
    correlated: bool = False
    seed: int = 0
    round: int = 0
    fixed_bits: int = 0
    scale_fp32: bool = False

    def c(self) -> _Cfg:
        return _Cfg(self.n_ranks, self.budget, self.eps, int(self.correlated), self.seed, self.round,
                    int(self.fixed_bits), int(self.scale_fp32))


def _addr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- primitives
def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().or_philox4x32_10(_addr(c), _addr(k), _addr(out))
    return out


def uniform16(idx, *, seed=0, round=0, n_ranks=1, correlated=False, hop=0, rank=0, slot=0,
              n_slots=1) -> np.ndarray:
    r = _Rng(seed, round, n_ranks, int(correlated), hop, rank, slot, n_slots)
    idx = np.asarray(idx, np.int64).ravel()
    f = lib().or_uniform16
    return np.array([f(C.addressof(r), int(i)) for i in idx], np.uint32)


def level_table(bits: int, eps: float = 1.0) -> np.ndarray:
    q = np.zeros(1 << bits, np.float32)
    lib().or_level_table(bits, float(eps), _addr(q))
    return q


def gap_table(bits: int, q: np.ndarray) -> np.ndarray:
    q = _c(q, np.float32)
    G = np.zeros((1 << bits) - 1, np.float32)
    lib().or_gap_table(bits, _addr(q), _addr(G))
    return G


def stats(g_u16: np.ndarray):
    g = _c(g_u16, np.uint16)
    assert g.size % SG == 0
    J = g.size // SG
    mean = np.zeros(J, np.float32)
    sq = np.zeros(J, np.float32)
    lib().or_stats(_addr(g), J, _addr(mean), _addr(sq))
    return mean, sq


def stats_reduce(means, sqs):
    m = _c(means, np.float32)
    s = _c(sqs, np.float32)
    N, J = m.shape
    M = np.zeros(J, np.float32)
    F = np.zeros(J, np.float32)
    lib().or_stats_reduce(_addr(m), _addr(s), N, J, _addr(M), _addr(F))
    return M, F


def bits_for(F: float, T: float) -> int:
    return lib().or_bits_for(F, T)


class BudgetInfeasible(ValueError):
    pass


def allocate(F, budget: float):
    F = _c(F, np.float32)
    J = F.size
    b = np.zeros(J, np.uint8)
    T = np.zeros(1, np.float32)
    counts = np.zeros(3, np.int64)
    rc = lib().or_allocate(_addr(F), J, float(budget), _addr(b), _addr(T), _addr(counts))
    if rc:
        raise BudgetInfeasible(f"budget {budget} < 2 bits per coordinate")
    return b, T[0], counts


def reorder(b) -> np.ndarray:
    b = _c(b, np.uint8)
    perm = np.zeros(b.size, np.int32)
    lib().or_reorder(_addr(b), b.size, _addr(perm))
    return perm


def chunk_cuts(b, perm, n_chunks: int) -> np.ndarray:
    b = _c(b, np.uint8)
    perm = _c(perm, np.int32)
    lo = np.zeros(n_chunks + 1, np.int64)
    lib().or_chunk_cuts(_addr(b), _addr(perm), b.size, n_chunks, _addr(lo))
    return lo


def message_bytes(n2: int, n4: int, n8: int, scale_fp32: bool = False) -> int:
    return lib().or_message_bytes(n2, n4, n8, int(scale_fp32))


def range_counts(lo: int, hi: int, N2: int, N4: int):
    def ov(a, b, c, d):
        return max(0, min(b, d) - max(a, c))
    return ov(lo, hi, 0, N2), ov(lo, hi, N2, N2 + N4), ov(lo, hi, N2 + N4, 1 << 62)


def range_message_bytes(lo, hi, N2, N4, scale_fp32: bool = False) -> int:
    return message_bytes(*range_counts(lo, hi, N2, N4), scale_fp32)


def quantize_sg(x, bits: int, *, eps=1.0, seed=0, round=0, n_ranks=1, correlated=False,
                hop=0, rank=0, slot=0, n_slots=1, idx0=0):
    x = _c(x, np.float32)
    assert x.size == SG
    q = level_table(bits, eps)
    G = gap_table(bits, q)
    r = _Rng(seed, round, n_ranks, int(correlated), hop, rank, slot, n_slots)
    E = np.zeros(1, np.uint8)
    u = np.zeros(16, np.uint8)
    codes = np.zeros(SG * bits // 8, np.uint8)
    lib().or_quantize_sg(_addr(x), bits, _addr(q), _addr(G), C.addressof(r), idx0,
                         _addr(E), _addr(u), _addr(codes))
    return int(E[0]), u, codes


def quantize_sg_f32(x, bits: int, *, eps=1.0, seed=0, round=0, n_ranks=1, correlated=False,
                    hop=0, rank=0, slot=0, n_slots=1, idx0=0):
    """Quantization with fp32 group scales: returns (sigma[16] fp32, codes)."""
    x = _c(x, np.float32)
    assert x.size == SG
    q = level_table(bits, eps)
    G = gap_table(bits, q)
    r = _Rng(seed, round, n_ranks, int(correlated), hop, rank, slot, n_slots)
    sig = np.zeros(16, np.float32)
    codes = np.zeros(SG * bits // 8, np.uint8)
    lib().or_quantize_sg_f32(_addr(x), bits, _addr(q), _addr(G), C.addressof(r), idx0, _addr(sig), _addr(codes))
    return sig, codes


def decode_add_sg(E: int, u, codes, bits: int, add, *, eps=1.0) -> np.ndarray:
    """Decode one super-group with UINT8 scales and add ``add`` (fp32[256])."""
    u = _c(u, np.uint8)
    codes = _c(codes, np.uint8)
    add = _c(add, np.float32)
    q = level_table(bits, eps)
    out = np.zeros(SG, np.float32)
    lib().or_decode_add_sg(E, _addr(u), _addr(codes), bits, _addr(q), _addr(add), _addr(out))
    return out


def decode_add_sg_f32(sig, codes, bits: int, add, *, eps=1.0) -> np.ndarray:
    sig = _c(sig, np.float32)
    codes = _c(codes, np.uint8)
    add = _c(add, np.float32)
    q = level_table(bits, eps)
    out = np.zeros(SG, np.float32)
    lib().or_decode_add_sg_f32(_addr(sig), _addr(codes), bits, _addr(q), _addr(add), _addr(out))
    return out


def dequantize_sg(E: int, u, codes, bits: int, *, eps=1.0) -> np.ndarray:
    u = _c(u, np.uint8)
    codes = _c(codes, np.uint8)
    q = level_table(bits, eps)
    out = np.zeros(SG, np.float32)
    lib().or_dequantize_sg(E, _addr(u), _addr(codes), bits, _addr(q), _addr(out))
    return out


def unpack_codes(codes, bits: int) -> np.ndarray:
    """Codes of the 256 coordinates of one super-group (LSB-first packing)."""
    codes = np.asarray(codes, np.uint8)
    per = 8 // bits
    out = np.zeros(SG, np.int32)
    for i in range(SG):
        out[i] = (int(codes[i // per]) >> ((i % per) * bits)) & ((1 << bits) - 1)
    return out


# --------------------------------------------------------------------------- range ops
def compress(cfg: Config, lo, hi, N2, N4, rank, hop, g_u16, M, perm, slot=0, n_slots=1) -> np.ndarray:
    g = _c(g_u16, np.uint16)
    M = _c(M, np.float32)
    perm = _c(perm, np.int32)
    msg = np.zeros(range_message_bytes(lo, hi, N2, N4, cfg.scale_fp32), np.uint8)
    c = cfg.c()
    lib().or_compress(C.addressof(c), lo, hi, N2, N4, rank, hop, slot, n_slots, _addr(g), _addr(M),
                      _addr(perm), _addr(msg))
    return msg


def dar(cfg: Config, in_lo, in_hi, N2, N4, rank, hop, msg_in, addend, M, perm,
        send=(0, 0), keep=(0, 0), slot=0, n_slots=1):
    """Returns (msg_out, keep_out).  ``addend`` is the full bf16 gradient
    (uint16) of the rank, or an fp32 array of (in_hi-in_lo)*256 partial sums."""
    msg_in = _c(msg_in, np.uint8)
    M = _c(M, np.float32)
    perm = _c(perm, np.int32)
    is32 = addend.dtype == np.float32
    addend = _c(addend, np.float32 if is32 else np.uint16)
    nb = range_message_bytes(send[0], send[1], N2, N4, cfg.scale_fp32)
    msg_out = np.zeros(max(1, nb), np.uint8)
    keep_out = np.zeros(max(1, (keep[1] - keep[0]) * SG), np.float32)
    c = cfg.c()
    lib().or_dar(C.addressof(c), in_lo, in_hi, N2, N4, rank, hop, slot, n_slots, _addr(msg_in), _addr(addend),
                 int(is32), _addr(M), _addr(perm), send[0], send[1], _addr(msg_out),
                 keep[0], keep[1], _addr(keep_out))
    return msg_out[:nb], keep_out[: (keep[1] - keep[0]) * SG]


def decode(cfg: Config, lo, hi, N2, N4, msg, M, perm, out=None) -> np.ndarray:
    msg = _c(msg, np.uint8)
    M = _c(M, np.float32)
    perm = _c(perm, np.int32)
    if out is None:
        out = np.zeros(perm.size * SG, np.float32)
    c = cfg.c()
    lib().or_decode(C.addressof(c), lo, hi, N2, N4, _addr(msg), _addr(M), _addr(perm), _addr(out))
    return out


# --------------------------------------------------------------------------- whole all-reduce
def allreduce_sg(cfg: Config, butterfly: bool, grads, M, perm, N2, N4, chunk_lo, sel):
    """Per-super-group simulation of the all-reduce for reordered super-groups
    ``sel``.  Returns (out[len(sel), 256] fp32, final[len(sel), 321] uint8):
    65 metadata bytes (UINT8 scales: E byte, 16 u bytes, zeros; fp32 scales:
    a zero byte, then the 16 fp32 scales), then 256 code bytes
    (zero-padded)."""
    gs = [_c(g, np.uint16) for g in grads]
    assert len(gs) == cfg.n_ranks
    ptrs = (C.c_void_p * len(gs))(*[_addr(g) for g in gs])
    M = _c(M, np.float32)
    perm = _c(perm, np.int32)
    chunk_lo = _c(chunk_lo, np.int64)
    sel = _c(sel, np.int64)
    out = np.zeros((sel.size, SG), np.float32)
    fin = np.zeros((sel.size, 65 + SG), np.uint8)
    c = cfg.c()
    rc = lib().or_allreduce_sg(C.addressof(c), int(butterfly), C.cast(ptrs, C.c_void_p), _addr(M),
                               _addr(perm), N2, N4, _addr(chunk_lo), _addr(sel), sel.size,
                               _addr(out), _addr(fin))
    if rc:
        raise ValueError("butterfly needs a power-of-two number of ranks")
    return out, fin


@dataclass
class Plan:
    M: np.ndarray
    F: np.ndarray
    b: np.ndarray
    T: float
    counts: np.ndarray
    perm: np.ndarray
    chunk_lo: np.ndarray


def plan(cfg: Config, grads) -> Plan:
    """Statistics, metadata all-reduce, allocation, reordering and chunking."""
    ms, qs = zip(*[stats(g) for g in grads])
    M, F = stats_reduce(np.stack(ms), np.stack(qs))
    if cfg.fixed_bits:
        # uniform-bitwidth ablation: every super-group gets fixed_bits; no
        # threshold applies (T is reported as NaN)
        if cfg.fixed_bits not in (2, 4, 8):
            raise ValueError("fixed_bits must be 2, 4 or 8")
        b = np.full(F.size, cfg.fixed_bits, np.uint8)
        T = np.float32(np.nan)
        counts = np.array([F.size * (cfg.fixed_bits == k) for k in (2, 4, 8)], np.int64)
    else:
        b, T, counts = allocate(F, cfg.budget)
    perm = reorder(b)
    lo = chunk_cuts(b, perm, cfg.n_ranks)
    return Plan(M, F, b, float(T), counts, perm, lo)


def allreduce(cfg: Config, grads, butterfly: bool = False, sel=None):
    """The whole oracle all-reduce.  Returns (plan, out) where out is the
    fp32 sum in original order (or, with ``sel``, rows for those reordered
    super-groups)."""
    p = plan(cfg, grads)
    J = p.b.size
    full = sel is None
    if full:
        sel = np.arange(J, dtype=np.int64)
    rows, _ = allreduce_sg(cfg, butterfly, grads, p.M, p.perm, int(p.counts[0]),
                           int(p.counts[1]), p.chunk_lo, sel)
    if not full:
        return p, rows
    out = np.zeros(J * SG, np.float32)
    out.reshape(J, SG)[p.perm[sel]] = rows
    return p, out


def exact_sum(grads) -> np.ndarray:
    """fp64 sum of bf16 gradients (exact for up to 2^8 workers of bf16 data
    far from overflow: each addend has 8 significant bits)."""
    acc = np.zeros(np.asarray(grads[0]).size, np.float64)
    for g in grads:
        acc += (np.asarray(g, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return acc


def vnmse(out, grads) -> float:
    """vNMSE = ||out - s||^2 / ||s||^2 in fp64, s the exact sum
    [S "Evaluation": compression error measured by vNMSE]."""
    s = exact_sum(grads)
    d = np.asarray(out, np.float64) - s
    den = float(np.dot(s, s))
    return float(np.dot(d, d)) / den if den > 0 else float(np.dot(d, d))


# --------------------------------------------------------------------------- MXFP8 baseline
MXB = 32


def e4m3_value(code: int) -> float:
    return lib().or_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return int(lib().or_e4m3_encode(float(v)))


def mx_encode_block(v):
    v = _c(v, np.float32)
    assert v.size == MXB
    X = np.zeros(1, np.uint8)
    P = np.zeros(MXB, np.uint8)
    lib().or_mx_encode_block(_addr(v), _addr(X), _addr(P))
    return int(X[0]), P


def mx_message_bytes(n_blk: int) -> int:
    return lib().or_mx_message_bytes(n_blk)


def mx_quantize(x) -> np.ndarray:
    x = _c(x, np.float32)
    assert x.size % MXB == 0
    msg = np.zeros(mx_message_bytes(x.size // MXB), np.uint8)
    lib().or_mx_quantize(_addr(x), x.size // MXB, _addr(msg))
    return msg


def mx_dequantize(msg, n_blk: int) -> np.ndarray:
    msg = _c(msg, np.uint8)
    out = np.zeros(n_blk * MXB, np.float32)
    lib().or_mx_dequantize(_addr(msg), n_blk, _addr(out))
    return out


def mx_chunk_lo(n_blk: int, n_ranks: int) -> list:
    """Equal runs of blocks: chunk c = [floor(c B / N), floor((c+1) B / N))."""
    return [c * n_blk // n_ranks for c in range(n_ranks + 1)]


def mx_allreduce_blk(n_ranks: int, butterfly: bool, grads, sel):
    """MXFP8 all-reduce of blocks ``sel`` (32 coords each).  Returns
    (out[len(sel), 32] fp32, final[len(sel), 33] = scale byte + 32 codes)."""
    gs = [_c(g, np.uint16) for g in grads]
    assert len(gs) == n_ranks
    n_blk = gs[0].size // MXB
    ptrs = (C.c_void_p * len(gs))(*[_addr(g) for g in gs])
    sel = _c(sel, np.int64)
    out = np.zeros((sel.size, MXB), np.float32)
    fin = np.zeros((sel.size, 33), np.uint8)
    rc = lib().or_mx_allreduce_blk(n_ranks, int(butterfly), C.cast(ptrs, C.c_void_p), n_blk, _addr(sel),
                                   sel.size, _addr(out), _addr(fin))
    if rc:
        raise ValueError("butterfly needs a power-of-two number of ranks (or a block index is out of range)")
    return out, fin


def mx_allreduce(n_ranks: int, grads, butterfly: bool = False) -> np.ndarray:
    """The whole MXFP8 all-reduce: fp32 sum in original order."""
    n_blk = np.asarray(grads[0]).size // MXB
    out, _ = mx_allreduce_blk(n_ranks, butterfly, grads, np.arange(n_blk, dtype=np.int64))
    return out.reshape(-1)
