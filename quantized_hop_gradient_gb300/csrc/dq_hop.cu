// dq_hop.cu -- fused hop (compress / decompress-accumulate-recompress) and
// final decode kernels.
//
// Work mapping.  A warp takes a work unit of up to 32 consecutive reordered
// super-groups of one task and one bitwidth, and processes them two at a
// time: lanes 0-15 one super-group, lanes 16-31 the next.  Lane l of a half
// owns group l (coordinates 16l .. 16l+15), so a group maximum needs no
// shuffle, a super-group maximum four, and each lane draws one Philox call
// (eight 16-bit fields) for its sixteen coordinates.  The unit's
// permutation entries, means and exponent bytes are loaded once, coalesced,
// and broadcast by shuffles; its message addresses and its send and keep
// masks are computed once per unit.  The incoming codes and UINT8 scales
// of a pair of super-groups are staged in shared memory by cp.async, one
// pair ahead of the computation; the addend (a bf16 gradient or an fp32
// partial sum) goes straight to registers, also one pair ahead.
//
// Per coordinate the quantizer costs a packed fused multiply-add for y, one
// for the bucket index, an AND, two or three shared-memory loads (the
// bucket, then the level and its reciprocal gap), two compares, a subtract
// and a fused multiply-add rounded upward for the rounding decision, and
// the code packing.  For 2 and 4 bits the levels and reciprocal gaps sit in
// separate small tables, so the two operands of each packed operation load
// straight into adjacent registers; for 8 bits one 8-byte load from a
// lane-copied table of {level, gap} pairs gives both without bank conflicts.
// y feeds several instructions; a compiler that fused its multiply into
// the subtract that follows would change the rounding, which the GPU parity
// tests (bit-exact against the oracle) detect.
#include <algorithm>
#include <mutex>

#include "dq_common.cuh"
#include "dq_internal.h"

namespace dq {

namespace {

constexpr int kWarps = 16;      // warps per block
constexpr int kStages = 2;      // pairs of super-groups in flight per warp
constexpr int kHopBlocksPerSM = 1;  // one block per SM (its tables fill most of shared memory); 128 registers

__shared__ __align__(16) Tables g_tab;
// The 4-bit buckets, one copy per half-warp lane: row b (128 bytes) holds
// 16 copies of entry b, and lane l reads copy l mod 16, so the 16 lanes of a
// half-warp always read 16 different bank pairs.
__shared__ __align__(16) BucketEntry g_bk4c[(kMask4 + 1) * kCopies4];

__device__ __forceinline__ void expand_bk4()
{
    for (int i = threadIdx.x; i < (kMask4 + 1) * kCopies4; i += blockDim.x) g_bk4c[i] = g_tab.bk4[i / kCopies4];
}

// The 8-bit tables of the hop kernels, at the start of dynamic shared
// memory, one copy per half-warp lane c: buckets (row b + 256, 128 bytes per
// row) whose entry for copy c holds 128 kb + 8c, and the levels interleaved
// with their reciprocal gaps (128 bytes per level), so the pair {q_k, G16_k}
// of copy c sits at byte 128 k + 8c.  An 8-byte load is served per
// half-warp, whose 16 lanes then always read 16 different bank pairs: one
// conflict-free load per coordinate gives both the level and its gap.
// After them, the decoder's 4-bit pair table: entry p (a code byte: low
// nibble = first coordinate's code) holds the two levels, one copy per
// half-warp lane, copy c of entry p at byte 128 p + 8c.
extern __shared__ __align__(16) uint8_t g_dyn[];
constexpr int kCopies8 = 16;
constexpr int kRows8 = 2 * kOff8 + 1;
constexpr int kBk8cBytes = kRows8 * kCopies8 * 8;
constexpr int kQG8cBytes = 256 * kCopies8 * 8;
constexpr int kQ4pBytes = 256 * kCopies4 * 8;
constexpr int kTab8Bytes = kBk8cBytes + kQG8cBytes;
__host__ __device__ constexpr int tab_bytes(bool) { return kTab8Bytes + kQ4pBytes; }
static_assert(kTab8Bytes % 16 == 0 && kQ4pBytes % 16 == 0, "16-byte aligned staging");
__device__ __forceinline__ const BucketEntry *bk8c() { return reinterpret_cast<const BucketEntry *>(g_dyn); }
__device__ __forceinline__ const float2 *qg8c() { return reinterpret_cast<const float2 *>(g_dyn + kBk8cBytes); }
__device__ __forceinline__ const float2 *q4p() { return reinterpret_cast<const float2 *>(g_dyn + kBk8cBytes + kQG8cBytes); }
// The decoder's 2-bit pair table: entry p (four bits: low two = first
// coordinate's code) holds the two levels; 16 entries of 8 bytes cover the
// 32 banks once, so any lookup pattern is conflict-free.
__shared__ __align__(16) float2 g_q2p[16];

__device__ __forceinline__ void expand_tables(bool pair4)
{
    BucketEntry *bk = reinterpret_cast<BucketEntry *>(g_dyn);
    for (int i = threadIdx.x; i < kRows8 * kCopies8; i += blockDim.x) {
        const BucketEntry e = g_tab.bk8[i / kCopies8];
        bk[i] = BucketEntry{e.boundary, e.kb4 * 32 + (i % kCopies8) * 8};
    }
    float2 *qg = reinterpret_cast<float2 *>(g_dyn + kBk8cBytes);
    for (int i = threadIdx.x; i < 256 * kCopies8; i += blockDim.x)
        qg[i] = make_float2(g_tab.q8[i / kCopies8], g_tab.g8[i / kCopies8]);
    float2 *p4 = reinterpret_cast<float2 *>(g_dyn + kBk8cBytes + kQG8cBytes);
    for (int i = threadIdx.x; pair4 && i < 256 * kCopies4; i += blockDim.x) {
        const int p = i / kCopies4;
        p4[i] = make_float2(g_tab.q4[p & 15], g_tab.q4[p >> 4]);
    }
    for (int i = threadIdx.x; i < 16; i += blockDim.x) g_q2p[i] = make_float2(g_tab.q2[i & 3], g_tab.q2[i >> 2]);
}
// e for S > 0: with S = (1 + f) 2^(eb-127), 255 * 2^e >= S holds first at
// e = eb - 134 when (1 + f) <= 510/256 (mantissa field <= 0x7F0000), else at
// eb - 133; subnormal S (eb = 0) and tiny S clamp to -126.  Byte E = e + 127,
// E = 0 when S = 0.
__device__ __forceinline__ uint32_t exponent_byte(float S)
{
    if (!(S > 0.0f)) return 0u;
    const uint32_t bits = __float_as_uint(S);
    const int eb = (int)(bits >> 23);
    int e = eb - 134 + ((bits & 0x7FFFFFu) > 0x7F0000u ? 1 : 0);
    if (eb == 0 || e < -126) e = -126;
    return (uint32_t)(e + 127);
}

template <int BITS> struct Lvl;
template <> struct Lvl<2> {
    static constexpr int kMask = kMask2;
    __device__ static const float *q() { return g_tab.q2; }
    __device__ static const float *g() { return g_tab.g2; }
    __device__ static const BucketEntry *bk() { return g_tab.bk2; }
    __device__ static float mul() { return g_tab.mul2; }
};
template <> struct Lvl<4> {
    static constexpr int kMask = kMask4;
    __device__ static const float *q() { return g_tab.q4; }
    __device__ static const float *g() { return g_tab.g4; }
    __device__ static const BucketEntry *bk() { return g_bk4c; }
    __device__ static float mul() { return g_tab.mul4; }
};
template <> struct Lvl<8> {
    static constexpr int kMask = kMask8;
    __device__ static const float *q() { return g_tab.q8; }
    __device__ static const float *g() { return g_tab.g8; }
    __device__ static const BucketEntry *bk() { return g_tab.bk8; }
    __device__ static float mul() { return g_tab.mul8; }
};

// shared-memory load at a byte offset from a table
template <typename T>
__device__ __forceinline__ T lds_at(const void *base, uint32_t byte_off)
{
    return *reinterpret_cast<const T *>(reinterpret_cast<const char *>(base) + byte_off);
}

// a * b + c with ONE rounding toward +infinity.
__device__ __forceinline__ float2 f2_fma_rp(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{ .reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\tfma.rp.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d; }"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// k + STEP when a >= b, else k: one compare and one predicated add (the
// select-then-add a compiler makes of the conditional costs one more).  A NaN
// operand compares false either way.
template <uint32_t STEP>
__device__ __forceinline__ uint32_t add_if_ge(uint32_t k, float a, float b)
{
    asm("{ .reg .pred p;\n\tsetp.ge.f32 p, %1, %2;\n\t@p add.u32 %0, %0, %3; }" : "+r"(k) : "f"(a), "f"(b), "n"(STEP));
    return k;
}
// k + STEP when a < b, else k.
template <uint32_t STEP>
__device__ __forceinline__ uint32_t add_if_lt(uint32_t k, float a, float b)
{
    asm("{ .reg .pred p;\n\tsetp.lt.f32 p, %1, %2;\n\t@p add.u32 %0, %0, %3; }" : "+r"(k) : "f"(a), "f"(b), "n"(STEP));
    return k;
}

// Codes of one lane: 16 coordinates of BITS bits, coordinate i at bit BITS*i.
template <int BITS> struct LaneCodes { uint32_t w[BITS / 2]; };

template <int BITS>
__device__ __forceinline__ uint32_t code_of(const LaneCodes<BITS> &c, int i)
{
    return (c.w[(BITS * i) >> 5] >> ((BITS * i) & 31)) & ((1u << BITS) - 1u);
}

// Byte offset of the code block of super-group s of a message (bitwidth BITS).
template <int BITS>
__device__ __forceinline__ int64_t code_block_off(const MsgView &m, int64_t s)
{
    if (BITS == 2) return m.off_c2 + 64 * s;
    if (BITS == 4) return m.off_c4 + 128 * (s - m.n2);
    return m.off_c8 + 256 * (s - m.n2 - m.n4);
}

template <int BITS>
__device__ __forceinline__ const uint8_t *code_block(const MsgView &m, int64_t s)
{
    return m.base + code_block_off<BITS>(m, s);
}

template <int BITS>
__device__ __forceinline__ LaneCodes<BITS> lds_codes(const uint8_t *p)
{
    LaneCodes<BITS> c;
    if (BITS == 2) {
        c.w[0] = *reinterpret_cast<const uint32_t *>(p);
    } else if (BITS == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        c.w[0] = v.x; c.w[1] = v.y;
    } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        c.w[0] = v.x; c.w[1] = v.y; c.w[2] = v.z; c.w[3] = v.w;
    }
    return c;
}

template <int BITS>
__device__ __forceinline__ void stg_codes(uint8_t *p, const LaneCodes<BITS> &c)
{
    if (BITS == 2) *reinterpret_cast<uint32_t *>(p) = c.w[0];
    else if (BITS == 4) *reinterpret_cast<uint2 *>(p) = make_uint2(c.w[0], c.w[1]);
    else *reinterpret_cast<uint4 *>(p) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
}

// x = fl(sigma * q_code + x) with one rounding (fused multiply-add); sigma
// is u * 2^(E-127) (0 when E = 0) with UINT8 scales, the fp32 scale itself
// otherwise.  2 and 4 bits: one 8-byte pair-table load per two codes (both
// tables conflict-free); 8 bits: one lane-copy level load per code.
template <int BITS, bool PAIR4>
__device__ __forceinline__ void decode_add(float2 (&x)[8], float sigma, const LaneCodes<BITS> &c)
{
    const float2 s2 = make_float2(sigma, sigma);
    if constexpr (BITS == 8) {   // lane copies: the level at byte 128 code + 8 (lane mod 16)
        const float2 *q = qg8c();
        const uint32_t c8 = (threadIdx.x & 15u) << 3;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i0 = 2 * k, i1 = 2 * k + 1;
            const uint32_t w0 = c.w[i0 >> 2], w1 = c.w[i1 >> 2];
            const int b0 = 8 * (i0 & 3), b1 = 8 * (i1 & 3);
            const uint32_t o0 = ((b0 >= 7 ? (w0 >> (b0 >= 7 ? b0 - 7 : 0)) : (w0 << 7)) & 0x7F80u) | c8;
            const uint32_t o1 = ((b1 >= 7 ? (w1 >> (b1 >= 7 ? b1 - 7 : 0)) : (w1 << 7)) & 0x7F80u) | c8;
            x[k] = f2_fma(s2, make_float2(lds_at<float>(q, o0), lds_at<float>(q, o1)), x[k]);
        }
    } else if constexpr (BITS == 4 && !PAIR4) {   // one level load per code (16 entries: 16 banks)
        const float *q = Lvl<4>::q();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t w = c.w[k >> 2];
            const int b = 8 * (k & 3);
            const uint32_t o0 = (b >= 2 ? (w >> (b >= 2 ? b - 2 : 0)) : (w << 2)) & 0x3Cu;
            const uint32_t o1 = (w >> (b + 2)) & 0x3Cu;
            x[k] = f2_fma(s2, make_float2(lds_at<float>(q, o0), lds_at<float>(q, o1)), x[k]);
        }
    } else if constexpr (BITS == 4) {   // pair k = code byte k: byte offset 128 byte + 8 (lane mod 16)
        const float2 *q = q4p();
        const uint32_t c8 = (threadIdx.x & 15u) << 3;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t w = c.w[k >> 2];
            const int b = 8 * (k & 3);
            const uint32_t o = ((b >= 7 ? (w >> (b >= 7 ? b - 7 : 0)) : (w << 7)) & 0x7F80u) | c8;
            x[k] = f2_fma(s2, lds_at<float2>(q, o), x[k]);
        }
    } else {   // 2 bits: pair k = bits 4k .. 4k+3, byte offset 8 * nibble
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t w = c.w[0];
            const uint32_t o = (k == 0 ? (w << 3) : (w >> (k == 0 ? 0 : 4 * k - 3))) & 0x78u;
            x[k] = f2_fma(s2, lds_at<float2>(g_q2p, o), x[k]);
        }
    }
}

// Quantization of one lane's group (16 values).  Scale hierarchy: s = group
// max |x|; S = super-group max (half-warp); E from S; u = smallest integer
// with u * 2^e >= s; m = fl(fl(1/u) * 2^-e).  Per coordinate: y = fl(x * m)
// (a fused multiply-add with -0, which adds nothing and rounds once); k =
// the largest level <= y (bucket table, then exact compares); d = fl(y -
// q_k); the code is k + 1 when U < d * G16_k exactly, else k.  The exact
// comparison is t = fl_up(d * G16_k + 2^23) = 2^23 + ceil(d * G16_k) (one
// upward rounding: d * G16_k < 2^16) against the fp32 2^23 + U built from
// U's bits.  y needs no clamp: |y| <= 1 + 2^-23, the top level has G16 = 0,
// and below the bottom level d < 0.
// SF32 (ablation: scales in fp32): sigma = s, y = fl(x / s) (y = 0 when
// s = 0); E_out = 0 and u_out holds the bits of s.
// off: the correlated-rounding offset of this quantizer, in [0, 2^16); OFF =
// false compiles it out (every quantizer of the launch has offset 0).
template <int BITS, bool ONE_LEVEL, bool SF32, bool OFF>
__device__ __forceinline__ LaneCodes<BITS> quantize_group(const float2 (&x)[8], uint32_t ctr0, uint32_t stage_word,
                                                          uint32_t off, const PhiloxKeys &K, uint32_t &E_out,
                                                          uint32_t &u_out)
{
    // group maximum as a three-level tree of three-way maxima (max is exact,
    // so the order does not change the result; 0 joins in as before)
    float a[17];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        a[2 * k] = fabsf(x[k].x);
        a[2 * k + 1] = fabsf(x[k].y);
    }
    a[16] = 0.0f;
    float l1[6];
#pragma unroll
    for (int i = 0; i < 5; ++i) l1[i] = fmaxf(fmaxf(a[3 * i], a[3 * i + 1]), a[3 * i + 2]);
    l1[5] = fmaxf(a[15], a[16]);
    const float s = fmaxf(fmaxf(fmaxf(l1[0], l1[1]), l1[2]), fmaxf(fmaxf(l1[3], l1[4]), l1[5]));
    float m = 0.0f;
    if (SF32) {
        E_out = 0u;
        u_out = __float_as_uint(s);
    } else {
        // super-group maximum: s >= 0, so the bit patterns order like the values
        const bool hi_half = (threadIdx.x & 16u) != 0u;
        const uint32_t sb = __float_as_uint(s);
        const uint32_t m0 = __reduce_max_sync(kFull, hi_half ? 0u : sb);
        const uint32_t m1 = __reduce_max_sync(kFull, hi_half ? sb : 0u);
        const float S = __uint_as_float(hi_half ? m1 : m0);
        const uint32_t E = exponent_byte(S);
        const float inv2e = __uint_as_float((254u - E) << 23);   // 2^-e (any E: finite)
        // u = ceil(s * 2^-e): s * 2^-e is exact and at most 255, so one fused
        // multiply-add rounded upward onto 2^23 leaves 2^23 + u (the clamp
        // only guards non-finite inputs)
        uint32_t u = __float_as_uint(__fmaf_ru(s, inv2e, 8388608.0f)) - 0x4B000000u;
        u = min(u, 255u);
        m = __fmul_rn(g_tab.rcp[u], inv2e);
        E_out = E;
        u_out = u;
    }

    // One Philox call per group: coordinate c takes 16-bit field c mod 8,
    // plus 2^15 (mod 2^16) for c >= 8, plus the correlated offset.  Word A
    // carries coordinate 2i's field in its low half, word B coordinate
    // 2i+1's in its high half (carries out of a half are never read).
    uint32_t r0[4];
    philox4x32_10_keyed(r0, ctr0, stage_word, K);
    const uint32_t offh = off << 16;
    uint32_t A[8], B[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        A[i] = OFF ? r0[i] + off : r0[i];   // !OFF: every offset of the launch is 0
        B[i] = OFF ? r0[i] + offh : r0[i];
        A[i + 4] = A[i] ^ 0x8000u;
        B[i + 4] = B[i] ^ 0x80000000u;
    }

    // 8 bits: lane copies, {level, gap} at byte offsets 128 k + 8 (lane mod 16), steps of 128
    const float *q = BITS == 8 ? reinterpret_cast<const float *>(qg8c()) : Lvl<BITS>::q();
    const float *g = BITS == 8 ? nullptr : Lvl<BITS>::g();
    const BucketEntry *bk = BITS == 8 ? bk8c() : Lvl<BITS>::bk();
    constexpr uint32_t kStep = BITS == 8 ? 128u : 4u;
    // byte offset of bucket b: 8b (2 bits: r = rint(8Hy), 8b = r & ~7) or,
    // for the lane-copied 4- and 8-bit tables, 128b + 8 (lane mod 16)
    // (r = rint(128Hy); 8 bits: b + 256)
    constexpr uint32_t kB = BITS == 2 ? (uint32_t)Lvl<BITS>::kMask << 3 : (uint32_t)Lvl<BITS>::kMask << 7;
    const uint32_t lane_copy = BITS == 2 ? 0u : (threadIdx.x & 15u) << 3;
    const float mul = Lvl<BITS>::mul();
    const float magic = BITS == 8 ? kMagic + (float)(kOff8 * kSub8) : kMagic;
    const float2 mul2 = make_float2(mul, mul), M2 = make_float2(magic, magic);
    const float2 m2 = make_float2(m, m), nz2 = make_float2(-0.0f, -0.0f);
    const float2 C2 = make_float2(8388608.0f, 8388608.0f);   // 2^23
    LaneCodes<BITS> out;
#pragma unroll
    for (int w = 0; w < BITS / 2; ++w) out.w[w] = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float2 y;
        if (SF32) y = s > 0.0f ? make_float2(__fdiv_rn(x[k].x, s), __fdiv_rn(x[k].y, s)) : make_float2(0.0f, 0.0f);
        else y = f2_fma(x[k], m2, nz2);
        const float2 tf = f2_fma(y, mul2, M2);                 // S*H*y is exact: one rounding = rint
        const BucketEntry b0 = lds_at<BucketEntry>(bk, (__float_as_uint(tf.x) & kB) | lane_copy);
        const BucketEntry b1 = lds_at<BucketEntry>(bk, (__float_as_uint(tf.y) & kB) | lane_copy);
        uint32_t k40 = add_if_ge<kStep>((uint32_t)b0.kb4, y.x, b0.boundary);
        uint32_t k41 = add_if_ge<kStep>((uint32_t)b1.kb4, y.y, b1.boundary);
        if (BITS == 8) {   // a non-finite y reaches rows past 512: keep its offsets inside the table
            k40 &= 0x7FF8u;
            k41 &= 0x7FF8u;
        }
        if (!ONE_LEVEL) {  // buckets wider than a gap: walk up (bounded by the top level)
            constexpr uint32_t kTop = kStep * ((1u << BITS) - 1u);
            while (k40 < kTop && y.x >= lds_at<float>(q, k40 + kStep)) k40 += kStep;
            while (k41 < kTop && y.y >= lds_at<float>(q, k41 + kStep)) k41 += kStep;
        }
        float2 t;   // 2^23 + ceil(d * G16)
        if (BITS == 8) {   // one 8-byte load gives the level and its gap
            const float2 e0 = lds_at<float2>(q, k40), e1 = lds_at<float2>(q, k41);
            t = make_float2(__fmaf_ru(__fsub_rn(y.x, e0.x), e0.y, 8388608.0f),
                            __fmaf_ru(__fsub_rn(y.y, e1.x), e1.y, 8388608.0f));
        } else {
            const float2 qv = make_float2(lds_at<float>(q, k40), lds_at<float>(q, k41));
            const float2 gv = make_float2(lds_at<float>(g, k40), lds_at<float>(g, k41));
            t = f2_fma_rp(f2_sub(y, qv), gv, C2);
        }
        const float U0 = __uint_as_float(__byte_perm(A[k], 0x4B00u, 0x5410u));   // 2^23 + U
        const float U1 = __uint_as_float(__byte_perm(B[k], 0x4B00u, 0x5432u));
        k40 = add_if_lt<kStep>(k40, U0, t.x);
        k41 = add_if_lt<kStep>(k41, U1, t.y);
        const int i0 = 2 * k, i1 = 2 * k + 1;
        const int s0 = (BITS * i0) & 31, s1 = (BITS * i1) & 31;
        if (BITS == 8) {   // code = offset / 128 (the lane part is below bit 7)
            out.w[(BITS * i0) >> 5] |= (k40 >> 7) << s0;
            out.w[(BITS * i1) >> 5] |= (k41 >> 7) << s1;
        } else {   // codes never overlap, so adding them packs (a shift-and-add each)
            out.w[(BITS * i0) >> 5] += s0 >= 2 ? (k40 << (s0 >= 2 ? s0 - 2 : 0)) : (k40 >> 2);
            out.w[(BITS * i1) >> 5] += s1 >= 2 ? (k41 << (s1 >= 2 ? s1 - 2 : 0)) : (k41 >> 2);
        }
    }
    return out;
}

// Bytes of one staging slot (a pair of super-groups): addends, incoming
// codes, incoming group scales.
template <bool ADD_F32, bool SF32>
__host__ __device__ constexpr int stage_bytes() { return 512 + (SF32 ? 128 : 32); }
// 8-bit bucket rows up to 1023 (reached by a non-finite y) stay inside the
// smallest dynamic allocation of a hop kernel
static_assert(1024 * kCopies8 * 8 <= tab_bytes(false) + kWarps * kStages * stage_bytes<false, false>() &&
                  1024 * kCopies8 * 8 <= tab_bytes(true) + kWarps * kStages * stage_bytes<true, false>(),
              "garbage rows in bounds");

// One work unit: super-groups j0 .. j0+cnt-1 (one task, one bitwidth).  PP
// supplies perm, mu and the generator key and round.  Message bytes are
// read through L2 (cp.async.cg, ld.cg), never the non-coherent path, so a
// message written earlier in the same launch by other CTAs is read
// correctly after a grid barrier.  A half-warp whose super-group lies past
// the unit's end computes on stale staging data and stores nothing.
template <int BITS, bool HAS_IN, bool ADD_F32, bool ONE_LEVEL, bool SF32, bool OFF, typename PP>
__device__ __forceinline__ void hop_unit(const PP &P, const HopTask &t, uint8_t *stg, int64_t j0, int cnt,
                                         int lane)
{
    constexpr int A_BYTES = 0;   // addends bypass the staging
    constexpr int C_OFF = A_BYTES, U_OFF = A_BYTES + 512, STAGE = stage_bytes<ADD_F32, SF32>();
    constexpr int CB = 32 * BITS;                 // code bytes per super-group
    constexpr int UB = SF32 ? 64 : 16;            // scale bytes per super-group
    const int half = lane >> 4, hl = lane & 15;
    const uint32_t stg_s = smem_addr(stg);

    int32_t old_i = 0;
    float mu_i = 0.0f;
    uint32_t ein_i = 0;
    const int64_t jl = j0 + lane;
    if (lane < cnt) {
        old_i = __ldg(P.perm + jl);
        if (!ADD_F32) mu_i = __ldg(P.mu + old_i);
        if (HAS_IN && !SF32) ein_i = __ldcg(t.in.base + (jl - t.in_lo));
    }
    // super-groups of the unit (bit s) that are sent or kept
    const int64_t send_lo = t.send_lo, send_hi = t.send_hi;
    const unsigned send_m = __ballot_sync(kFull, lane < cnt && jl >= send_lo && jl < send_hi);
    const unsigned keep_m = __ballot_sync(kFull, lane < cnt && jl >= t.keep_lo && jl < t.keep_hi);
    const int npairs = (cnt + 1) >> 1;

    // this lane's addresses for super-group 0 of the unit; super-group s
    // adds s times the per-super-group stride
    const int64_t sl0 = j0 - t.in_lo;
    const uint8_t *in_c = HAS_IN ? t.in.base + code_block_off<BITS>(t.in, sl0) + hl * 16 : nullptr;
    const uint8_t *in_u = HAS_IN ? t.in.base + t.in.off_u + sl0 * UB + hl * 16 : nullptr;
    const char *add_f = ADD_F32 ? static_cast<const char *>(t.addend) + sl0 * 1024 + hl * 64 : nullptr;
    const char *add_b = static_cast<const char *>(t.addend) + hl * 32;
    const int64_t so0 = j0 - send_lo;
    uint8_t *out_c = t.out.base + code_block_off<BITS>(t.out, so0) + hl * (2 * BITS);
    uint8_t *out_u = t.out.base + t.out.off_u + so0 * UB + hl * (SF32 ? 4 : 1);
    float *keep_p = t.keep_out + (j0 - t.keep_lo) * kSG + hl * 16;
    const uint32_t stage_word = t.stage_word, corr = t.corr2 & 0xFFFFu;

    auto issue = [&](int pp) {
        const int s = 2 * pp + half;
        // the compress stages nothing, but this warp-wide shuffle at the top
        // of each pair keeps it 25% faster (measured: 312 against 388 us on
        // the BERT-large compress); the hops with an incoming message drop it
        if (!HAS_IN) (void)__shfl_sync(kFull, old_i, s & 31);
        if (pp < npairs && s < cnt) {
            const uint32_t st = stg_s + (uint32_t)((pp % kStages) * STAGE);
            if (HAS_IN) {
                if (hl < 2 * BITS) cp_async16(st + C_OFF + half * 256 + hl * 16, in_c + (int64_t)s * CB);
                if (SF32) {
                    if (hl < 4) cp_async16(st + U_OFF + half * 64 + hl * 16, in_u + (int64_t)s * UB);
                } else if (hl == 0) {
                    cp_async16(st + U_OFF + half * 16, in_u + (int64_t)s * UB);
                }
            }
        }
        cp_async_commit();
    };

    // bf16 addends go straight to registers, one pair ahead (a lane's 32
    // bytes are two 16-byte loads; no shared-memory round trip)
    uint4 na = make_uint4(0u, 0u, 0u, 0u), nb = na;
    float4 nf[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) nf[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int32_t nold = 0;   // perm entry of the pair that load_add fetched
    auto load_add = [&](int pp) {
        const int s = 2 * pp + half;
        const int32_t old = ADD_F32 ? 0 : __shfl_sync(kFull, old_i, s & 31);
        nold = old;
        if (pp < npairs && s < cnt) {
            if (ADD_F32) {
                const float4 *src = reinterpret_cast<const float4 *>(add_f + (int64_t)s * 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k) nf[k] = __ldg(src + k);
            } else {
                const uint4 *src = reinterpret_cast<const uint4 *>(add_b + (int64_t)old * 512);
                na = __ldg(src);
                nb = __ldg(src + 1);
            }
        }
    };
    load_add(0);
#pragma unroll
    for (int pp = 0; pp < kStages - 1; ++pp) issue(pp);
    uint32_t e_out = 0;
    for (int p = 0; p < npairs; ++p) {
        const uint4 ca = na, cb = nb;
        float4 cf[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) cf[k] = nf[k];
        const int32_t cold = nold;
        load_add(p + 1);
        issue(p + kStages - 1);
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint8_t *st = stg + (p % kStages) * STAGE;
        const int s = 2 * p + half;
        const int32_t old = (ADD_F32 || !HAS_IN) ? __shfl_sync(kFull, old_i, s & 31) : cold;
        const float mu = __shfl_sync(kFull, mu_i, s & 31);
        const uint32_t ein = __shfl_sync(kFull, ein_i, s & 31);

        float2 x[8];
        if (ADD_F32) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[2 * k] = make_float2(cf[k].x, cf[k].y);
                x[2 * k + 1] = make_float2(cf[k].z, cf[k].w);
            }
        } else {
            const uint32_t w[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = make_float2(bf16_lo_minus(w[k], mu), bf16_hi_minus(w[k], mu));
        }
        if (HAS_IN) {
            float sigma;
            if (SF32) {
                sigma = *reinterpret_cast<const float *>(st + U_OFF + half * 64 + hl * 4);
            } else {
                const uint32_t u = st[U_OFF + half * 16 + hl];
                sigma = __fmul_rn((float)u, __uint_as_float(ein << 23));
            }
            const LaneCodes<BITS> c = lds_codes<BITS>(st + C_OFF + half * 256 + hl * 2 * BITS);
            decode_add<BITS, true>(x, sigma, c);
        }
        const bool send = (send_m >> s) & 1u;
        const bool keep = (keep_m >> s) & 1u;
        uint32_t E = 0u, u = 0u;
        if (__any_sync(kFull, send)) {
            const uint32_t ctr0 = (uint32_t)old * 16u + (uint32_t)hl;   // global coordinate index / 16
            const LaneCodes<BITS> q = quantize_group<BITS, ONE_LEVEL, SF32, OFF>(x, ctr0, stage_word, corr, P.ph, E, u);
            if (send) {
                stg_codes<BITS>(out_c + (int64_t)s * CB, q);
                if (SF32) *reinterpret_cast<uint32_t *>(out_u + (int64_t)s * UB) = u;
                else out_u[(int64_t)s * UB] = (uint8_t)u;
            }
        }
        if (keep) {
            float4 *o = reinterpret_cast<float4 *>(keep_p + (int64_t)s * kSG);
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = make_float4(x[2 * k].x, x[2 * k].y, x[2 * k + 1].x, x[2 * k + 1].y);
        }
        const uint32_t e_pair = __shfl_sync(kFull, E, (lane & 1) << 4);
        if ((lane >> 1) == p) e_out = e_pair;
        __syncwarp();
    }
    if (!SF32 && ((send_m >> lane) & 1u)) t.out.base[jl - send_lo] = (uint8_t)e_out;
    // the unit holding the send range's last super-group zeroes the E padding
    if (!SF32 && send_hi > send_lo && send_hi - 1 >= j0 && send_hi - 1 < j0 + cnt) {
        const int64_t c = send_hi - send_lo, pad = (c + 15) / 16 * 16;
        if (lane < pad - c) t.out.base[c + lane] = 0;
    }
}

template <bool HAS_IN, bool ADD_F32, bool ONE_LEVEL, bool SF32, bool OFF>
__global__ void __launch_bounds__(kWarps * 32, kHopBlocksPerSM) hop_kernel(const __grid_constant__ HopParams P)
{
    block_copy(&g_tab, &P.tab);
    __syncthreads();
    expand_bk4();
    expand_tables(HAS_IN);
    __syncthreads();
    uint8_t *dyn = g_dyn + tab_bytes(ADD_F32);
    constexpr int STAGE = stage_bytes<ADD_F32, SF32>();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *stg = dyn + warp * kStages * STAGE;
    const int wpb = (int)(blockDim.x >> 5);   // warps per block: sized to the launch, at most kWarps
    const int64_t nw = (int64_t)gridDim.x * wpb;
    for (int64_t u = (int64_t)blockIdx.x * wpb + warp; u < P.total_units; u += nw) {
        int ti, seg;
        locate_unit(P.task, P.n_tasks, u, ti, seg);
        const HopTask &t = P.task[ti];
        const int64_t j0 = t.seg_lo[seg] + (u - t.unit_begin[seg]) * kUnit;
        const int64_t rem = t.seg_hi[seg] - j0;
        const int cnt = (int)(rem < kUnit ? rem : kUnit);
        if (seg == 0) hop_unit<2, HAS_IN, ADD_F32, ONE_LEVEL, SF32, OFF>(P, t, stg, j0, cnt, lane);
        else if (seg == 1) hop_unit<4, HAS_IN, ADD_F32, ONE_LEVEL, SF32, OFF>(P, t, stg, j0, cnt, lane);
        else hop_unit<8, HAS_IN, ADD_F32, ONE_LEVEL, SF32, OFF>(P, t, stg, j0, cnt, lane);
    }
}

// ---------------------------------------------------------------------------
// Final decode: out[perm[j]*256 + i] = fl(sigma * q_code + fl(mu_j * N)) (one
// rounding), fp32 or bf16.  Output-bound (4 bytes out per 0.69 in): both the
// decode kernel and the fused exchange's last phase hand the stores to the
// bulk-copy engine (decode_unit_bulk).
// ---------------------------------------------------------------------------
constexpr int kDecodeWarps = 16;
// The final decode runs flat: each warp decodes one slice of 32 / kDecodeSplit
// super-groups and exits; short-lived blocks stream their writes to HBM
// faster than a persistent grid-stride loop (7.7 vs 6.6 TB/s measured for
// plain 1 KiB row writes on a GB300).
constexpr int kDecodeSplit = 8;

// Copy only the decode levels (q2, q4, q8: contiguous in Tables) to shared memory.
__device__ __forceinline__ void copy_levels(Tables *dst, const Tables *src)
{
    static_assert(offsetof(Tables, q4) == offsetof(Tables, q2) + 16 && offsetof(Tables, q8) == offsetof(Tables, q4) + 64,
                  "levels contiguous");
    static_assert(offsetof(Tables, q2) % 16 == 0, "16-byte aligned");
    const int4 *s = reinterpret_cast<const int4 *>(src->q2);
    int4 *d = reinterpret_cast<int4 *>(dst->q2);
    for (int i = threadIdx.x; i < (4 + 16 + 256) / 4; i += blockDim.x) d[i] = s[i];
}

// Bulk (TMA) copy of `bytes` from this CTA's shared memory to global
// memory; completion is tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void *gdst, uint32_t ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}

// The decode of up to kDecodeSlice super-groups with the stores handed to
// the bulk-copy engine: the warp writes its decoded rows to shared memory
// (lane l owns coordinates 8l .. 8l+7), makes them visible to the async
// proxy, and each lane issues the copy of one (row, output) pair.  WAIT_ALL:
// then waits until its copies have completed (the shared memory must
// outlive them).  Otherwise the caller alternates two row buffers: before
// writing, every lane waits until at most its latest copy group is still
// reading (the one from the other buffer), and the caller waits for all
// copies at the end.  The global store queue carries none of the output.
constexpr int kDecodeSlice = kUnit / kDecodeSplit;

template <int BITS, bool SF32, bool WAIT_ALL, typename PP>
__device__ __forceinline__ void decode_unit_bulk(const PP &P, const MsgView &msg, int64_t lo, void *const *outs,
                                                 int n_outs, int64_t j0, int cnt, int lane, uint8_t *rows)
{
    if (!WAIT_ALL) {
        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
    }
    int32_t old_i = 0;
    float mu_i = 0.0f;
    uint32_t ein_i = 0;
    if (lane < cnt) {
        old_i = __ldg(P.perm + j0 + lane);
        mu_i = __ldg(P.mu + old_i);
        if (!SF32) ein_i = __ldcg(msg.base + (j0 + lane - lo));
    }
    const float nr = (float)P.n_ranks;
    const float *q = Lvl<BITS>::q();
    const int g = lane >> 1;
    const int row_bytes = P.out_is_bf16 ? 512 : 1024;
    uint32_t c0[kDecodeSlice], c1[kDecodeSlice], ua[kDecodeSlice];
#pragma unroll
    for (int a = 0; a < kDecodeSlice; ++a) {
        c0[a] = c1[a] = ua[a] = 0u;
        if (a < cnt) {
            const int64_t sl = j0 + a - lo;
            const uint8_t *blk = code_block<BITS>(msg, sl);
            if (BITS == 2) {
                c0[a] = __ldcg(reinterpret_cast<const unsigned short *>(blk) + lane);
            } else if (BITS == 4) {
                c0[a] = __ldcg(reinterpret_cast<const unsigned int *>(blk) + lane);
            } else {
                const uint2 v = __ldcg(reinterpret_cast<const uint2 *>(blk) + lane);
                c0[a] = v.x;
                c1[a] = v.y;
            }
            if (SF32) ua[a] = __ldcg(reinterpret_cast<const unsigned int *>(msg.base + msg.off_u + sl * 64) + g);
            else ua[a] = __ldcg(msg.base + msg.off_u + sl * 16 + g);
        }
    }
#pragma unroll
    for (int a = 0; a < kDecodeSlice; ++a) {
        const float mu = __shfl_sync(kFull, mu_i, a);
        const uint32_t E = __shfl_sync(kFull, ein_i, a);
        if (a < cnt) {
            const float back = __fmul_rn(mu, nr);
            const float sigma = SF32 ? __uint_as_float(ua[a]) : __fmul_rn((float)ua[a], __uint_as_float(E << 23));
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w = (BITS == 8 && i >= 4) ? c1[a] : c0[a];
                const int bit = (BITS * i) & 31;
                const uint32_t off = (bit >= 2 ? (w >> (bit >= 2 ? bit - 2 : 0)) : (w << 2)) & (((1u << BITS) - 1u) << 2);
                v[i] = __fmaf_rn(sigma, lds_at<float>(q, off), back);
            }
            if (P.out_is_bf16) {
                uint32_t h[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    h[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i])) |
                           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1])) << 16);
                *reinterpret_cast<uint4 *>(rows + a * 512 + 16 * lane) = make_uint4(h[0], h[1], h[2], h[3]);
            } else {
                float4 *r = reinterpret_cast<float4 *>(rows + a * 1024 + 32 * lane);
                r[0] = make_float4(v[0], v[1], v[2], v[3]);
                r[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    const uint32_t rows_s = smem_addr(rows);
    const int pairs = cnt * n_outs;
    for (int pbase = 0; pbase < pairs; pbase += 32) {
        const int pi = pbase + lane;
        const int a = pi < pairs ? pi / n_outs : 0;
        const int32_t old = __shfl_sync(kFull, old_i, a);
        if (pi < pairs) {
            char *dst = static_cast<char *>(outs[pi - a * n_outs]) + (int64_t)old * row_bytes;
            bulk_store(dst, rows_s + (uint32_t)(a * row_bytes), (uint32_t)row_bytes);
        }
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (WAIT_ALL) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <bool SF32>
__global__ void __launch_bounds__(kDecodeWarps * 32) decode_kernel(const __grid_constant__ DecodeParams P)
{
    extern __shared__ __align__(128) uint8_t drows[];
    copy_levels(&g_tab, &P.tab);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w = (int64_t)blockIdx.x * kDecodeWarps + warp;
    const int64_t u = w / kDecodeSplit;
    if (u >= P.total_units) return;
    int ti, seg;
    locate_unit(P.task, P.n_tasks, u, ti, seg);
    const DecodeTask &t = P.task[ti];
    const int64_t j0 = t.seg_lo[seg] + (u - t.unit_begin[seg]) * kUnit + (w % kDecodeSplit) * (kUnit / kDecodeSplit);
    const int64_t rem = t.seg_hi[seg] - j0;
    if (rem <= 0) return;
    const int cnt = (int)(rem < kUnit / kDecodeSplit ? rem : kUnit / kDecodeSplit);
    void *const *outs = P.n_outs > 0 ? P.outs : &t.out;
    const int n_outs = P.n_outs > 0 ? P.n_outs : 1;
    uint8_t *rows = drows + warp * kDecodeSlice * 1024;
    if (seg == 0) decode_unit_bulk<2, SF32, true>(P, t.msg, t.lo, outs, n_outs, j0, cnt, lane, rows);
    else if (seg == 1) decode_unit_bulk<4, SF32, true>(P, t.msg, t.lo, outs, n_outs, j0, cnt, lane, rows);
    else decode_unit_bulk<8, SF32, true>(P, t.msg, t.lo, outs, n_outs, j0, cnt, lane, rows);
}

// ---------------------------------------------------------------------------
// Grid barrier of a cooperative launch.  Thread 0 of each CTA makes the
// CTA's writes visible (fence), arrives on the counter and waits, with a
// bound, for gridDim.x * (phase + 1) arrivals.  The wait gives up when the
// status word is already set (another CTA timed out) or after
// timeout_cycles of the SM clock, setting the status; every thread of the
// CTA then learns the outcome, and a CTA that gave up returns from the
// kernel, so no CTA waits forever.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool grid_barrier(unsigned *counter, int32_t *status, unsigned target,
                                             long long timeout_cycles)
{
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        const long long t0 = clock64();
        int good = 1;
        while (ld_acquire_u32(counter) < target) {
            if (*(volatile int32_t *)status != 0) { good = 0; break; }
            if (clock64() - t0 > timeout_cycles) {
                atomicCAS(status, 0, kDeviceBarrierTimeout);
                good = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        ok = good;
    }
    __syncthreads();
    return ok != 0;
}

__global__ void barrier_selftest_kernel(unsigned *counter, int32_t *status, unsigned target, long long timeout)
{
    grid_barrier(counter, status, target, timeout);
}

// The ring exchange of one round, fused: at step t every chunk c is handled
// by rank r = (c + 1 + t) mod N, reading rank r-1's message of step t-1 and
// writing its own (buffer parity t & 1); step 0 quantizes the local
// gradient.  After the last step the owners' messages are decoded into every
// output (one read, N writes).  Grid barriers separate the phases.
template <bool ONE_LEVEL, bool SF32>
__global__ void __launch_bounds__(kWarps * 32, 1) fused_ring_kernel(const __grid_constant__ FusedRingParams P)
{
    block_copy(&g_tab, &P.tab);
    __syncthreads();
    expand_bk4();
    expand_tables(true);
    __syncthreads();
    uint8_t *dyn = g_dyn + tab_bytes(false);
    constexpr int STAGE = stage_bytes<false, SF32>();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *stg = dyn + warp * kStages * STAGE;
    const int N = P.n_ranks;
    const int wpb = (int)(blockDim.x >> 5);   // warps per block: sized to the launch, at most kWarps
    const int64_t nw = (int64_t)gridDim.x * wpb;
    for (int t = 0; t <= N; ++t) {
        int slice = 0;   // the final decode alternates two row buffers per warp
        for (int64_t u = (int64_t)blockIdx.x * wpb + warp; u < P.units; u += nw) {
            int c = 0;
            while (c + 1 < N && u >= P.unit_begin[c + 1][0]) ++c;
            int seg = 0;
            while (seg < 2 && u >= P.unit_begin[c][seg + 1]) ++seg;
            const int64_t j0 = P.seg_lo[c][seg] + (u - P.unit_begin[c][seg]) * kUnit;
            const int64_t rem = P.seg_hi[c][seg] - j0;
            const int cnt = (int)(rem < kUnit ? rem : kUnit);
            if (t == N) {   // final decode of chunk c (owner c, step N-1)
                MsgView m = P.chunk[c];
                m.base = P.msgs + (2 * (int64_t)c + ((N - 1) & 1)) * P.msg_stride;
                for (int s0 = 0; s0 < cnt; s0 += kDecodeSlice, ++slice) {
                    const int n = cnt - s0 < kDecodeSlice ? cnt - s0 : kDecodeSlice;
                    // (in the tables' shared memory, dead by then)
                    uint8_t *rb = g_dyn + (2 * warp + (slice & 1)) * kDecodeSlice * 1024;
                    if (seg == 0) decode_unit_bulk<2, SF32, false>(P, m, P.lo[c], P.outs, N, j0 + s0, n, lane, rb);
                    else if (seg == 1) decode_unit_bulk<4, SF32, false>(P, m, P.lo[c], P.outs, N, j0 + s0, n, lane, rb);
                    else decode_unit_bulk<8, SF32, false>(P, m, P.lo[c], P.outs, N, j0 + s0, n, lane, rb);
                }
                continue;
            }
            const int r = (c + 1 + t) % N, src = (r - 1 + N) % N;
            HopTask T;
            T.in = P.chunk[c];
            T.in.base = P.msgs + (2 * (int64_t)src + ((t - 1) & 1)) * P.msg_stride;
            T.out = P.chunk[c];
            T.out.base = P.msgs + (2 * (int64_t)r + (t & 1)) * P.msg_stride;
            T.addend = P.grads[r];
            T.keep_out = nullptr;
            T.in_lo = P.lo[c];
            T.send_lo = P.lo[c];
            T.send_hi = P.lo[c + 1];
            T.keep_lo = T.keep_hi = P.lo[c + 1];
            T.stage_word = (uint32_t)t | (P.correlated ? 0xFFFF0000u : ((uint32_t)r << 16));
            T.corr2 = 0u;   // one quantizer per ring stage: stratum offset 0
            if (t == 0) {
                if (seg == 0) hop_unit<2, false, false, ONE_LEVEL, SF32, false>(P, T, stg, j0, cnt, lane);
                else if (seg == 1) hop_unit<4, false, false, ONE_LEVEL, SF32, false>(P, T, stg, j0, cnt, lane);
                else hop_unit<8, false, false, ONE_LEVEL, SF32, false>(P, T, stg, j0, cnt, lane);
            } else {
                if (seg == 0) hop_unit<2, true, false, ONE_LEVEL, SF32, false>(P, T, stg, j0, cnt, lane);
                else if (seg == 1) hop_unit<4, true, false, ONE_LEVEL, SF32, false>(P, T, stg, j0, cnt, lane);
                else hop_unit<8, true, false, ONE_LEVEL, SF32, false>(P, T, stg, j0, cnt, lane);
            }
        }
        if (t < N && !grid_barrier(P.barrier, P.status, gridDim.x * (unsigned)(t + 1), P.timeout_cycles)) return;
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // the decode's copies
}

// Codes of one lane read from global memory (a message written by an
// earlier launch).
template <int BITS>
__device__ __forceinline__ LaneCodes<BITS> ldg_codes(const uint8_t *p)
{
    LaneCodes<BITS> c;
    if (BITS == 2) {
        c.w[0] = __ldcg(reinterpret_cast<const unsigned int *>(p));
    } else if (BITS == 4) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2 *>(p));
        c.w[0] = v.x; c.w[1] = v.y;
    } else {
        const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(p));
        c.w[0] = v.x; c.w[1] = v.y; c.w[2] = v.z; c.w[3] = v.w;
    }
    return c;
}

constexpr int kRowBytes = 1024;   // row buffer of the in-launch decode, per half-warp

// The final decode of up to kUnit super-groups of one chunk into all N
// outputs: out = fl(sigma * q_code + fl(mu * N)).  The hop's mapping: lanes
// 0-15 decode one super-group, lanes 16-31 the next, lane l of a half the
// coordinates 16l .. 16l+15.  Each half writes its decoded row to its row
// buffer (`rows`, 1 KB per half) and the warp hands the 2N row copies of the
// pair to the bulk-copy engine, one (row, output) per lane; before a row
// buffer is rewritten, each lane waits until its earlier copies have read
// it.  The caller waits for all copies before the block exits.  The codes
// and scales of the next four pairs load while a pair is decoded.  Meant to
// run beside the hop units of a launch, whose shared-memory tables it uses.
template <int BITS, bool SF32, typename PP>
__device__ __forceinline__ void decode_unit_rows(const PP &P, const MsgView &m, int64_t lo, int64_t j0, int cnt,
                                                 int lane, uint8_t *rows)
{
    constexpr int CB = 32 * BITS;
    constexpr int UB = SF32 ? 64 : 16;
    const int half = lane >> 4, hl = lane & 15;
    const int N = P.n_ranks;
    int32_t old_i = 0;
    float back_i = 0.0f;
    uint32_t ein_i = 0;
    if (lane < cnt) {
        old_i = __ldg(P.perm + j0 + lane);
        back_i = __fmul_rn(__ldg(P.mu + old_i), (float)N);
        if (!SF32) ein_i = __ldcg(m.base + (j0 + lane - lo));
    }
    const int64_t sl0 = j0 - lo;
    const uint8_t *cp = m.base + code_block_off<BITS>(m, sl0) + hl * 2 * BITS;
    const uint8_t *up = m.base + m.off_u + sl0 * UB + hl * (SF32 ? 4 : 1);
    uint4 *row = reinterpret_cast<uint4 *>(rows + half * kRowBytes);
    const uint32_t rows_s = smem_addr(rows);
    const int row_bytes = P.out_is_bf16 ? 512 : 1024;
    const int npairs = (cnt + 1) >> 1;
    // codes and scale of pairs p .. p+3 in flight, rotated through q0 .. q3
    LaneCodes<BITS> q0, q1, q2, q3;
    uint32_t u0 = 0, u1 = 0, u2 = 0, u3 = 0;
#pragma unroll
    for (int w = 0; w < BITS / 2; ++w) q0.w[w] = q1.w[w] = q2.w[w] = q3.w[w] = 0u;
    auto load = [&](int pp, LaneCodes<BITS> &qc, uint32_t &uu) {
        const int s = 2 * pp + half;
        if (pp < npairs && s < cnt) {
            qc = ldg_codes<BITS>(cp + (int64_t)s * CB);
            uu = SF32 ? __ldcg(reinterpret_cast<const unsigned int *>(up + (int64_t)s * UB))
                      : (uint32_t)__ldcg(up + (int64_t)s * UB);
        }
    };
    load(0, q0, u0);
    load(1, q1, u1);
    load(2, q2, u2);
    load(3, q3, u3);
    for (int p = 0; p < npairs; ++p) {
        const LaneCodes<BITS> c = q0;
        const uint32_t uc = u0;
        q0 = q1; u0 = u1;
        q1 = q2; u1 = u2;
        q2 = q3; u2 = u3;
        load(p + 4, q3, u3);
        const int s = 2 * p + half;
        const float back = __shfl_sync(kFull, back_i, s & 31);
        const uint32_t E = __shfl_sync(kFull, ein_i, s & 31);
        const float sigma = SF32 ? __uint_as_float(uc) : __fmul_rn((float)uc, __uint_as_float(E << 23));
        float2 x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = make_float2(back, back);
        decode_add<BITS, true>(x, sigma, c);
        // the row buffers are free once this lane's earlier copies have read them
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
        if (P.out_is_bf16) {   // lane l: bytes 32l .. 32l+31 of the 512-byte row
            uint32_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                h[k] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[k].x)) |
                       ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[k].y)) << 16);
            row[2 * hl] = make_uint4(h[0], h[1], h[2], h[3]);
            row[2 * hl + 1] = make_uint4(h[4], h[5], h[6], h[7]);
        } else {               // lane l: bytes 64l .. 64l+63 of the 1 KB row
#pragma unroll
            for (int i = 0; i < 4; ++i)
                row[4 * hl + i] = make_uint4(__float_as_uint(x[2 * i].x), __float_as_uint(x[2 * i].y),
                                             __float_as_uint(x[2 * i + 1].x), __float_as_uint(x[2 * i + 1].y));
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        // copies of the pair: row a (0: lanes 0-15's super-group) to output r
        const int n_rows = 2 * p + 1 < cnt ? 2 : 1;
        const int pairs = n_rows * N;
        for (int pbase = 0; pbase < pairs; pbase += 32) {
            const int pi = pbase + lane;
            const int a = pi < pairs ? pi / N : 0;
            const int32_t old = __shfl_sync(kFull, old_i, (2 * p + a) & 31);
            if (pi < pairs) {
                char *dst = static_cast<char *>(P.outs[pi - a * N]) + (int64_t)old * row_bytes;
                bulk_store(dst, rows_s + (uint32_t)(a * kRowBytes), (uint32_t)row_bytes);
            }
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

// One launch of the pipelined ring exchange (WaveRingParams): hop units of
// several parts, each at its own step, and the decode units of one part,
// spread evenly through the launch's unit list so that every SM keeps
// decoding (bound by HBM writes) beside the hops (bound by instruction
// issue).  Step s of chunk c is handled by rank r = (c + 1 + s) mod N, which
// reads rank r-1's message of step s-1 and writes its own of step s; step 0
// quantizes the local gradient.  The decode reads owner c's message of step
// N-1.  Results are those of the per-step exchange, bit for bit: every
// super-group sees the same operations, only their order in time changes.
template <bool ONE_LEVEL, bool SF32>
__global__ void __launch_bounds__(kWarps * 32, 1) wave_ring_kernel(const __grid_constant__ WaveRingParams P)
{
    // Launched with programmatic stream serialization: the next launch may
    // start its blocks (and their table setup) on the SMs this one frees, and
    // this one's table setup overlaps the previous launch's last units.
    // griddepcontrol.wait returns once the previous launch has completed and
    // its writes are visible; nothing before it touches global memory other
    // than the launch parameters.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    block_copy(&g_tab, &P.tab);
    __syncthreads();
    expand_bk4();
    expand_tables(true);
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    uint8_t *dyn = g_dyn + tab_bytes(false);
    constexpr int STAGE = stage_bytes<false, SF32>();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *stg = dyn + warp * kStages * STAGE;
    uint8_t *rows = dyn + kWarps * kStages * STAGE + warp * 2 * kRowBytes;
    const int N = P.n_ranks;
    // each decode unit is cut into kDecodeSub pieces, so that the launches
    // whose work is mostly decode end evenly
    const int64_t H = P.h_hi - P.h_lo, D = (P.d_hi - P.d_lo) * kDecodeSub, T = H + D;
    // units are taken in turn from the launch's counter, the next one claimed
    // before the current one runs (a static stride would hand every decode
    // unit to the same warps whenever the stride and the decode spacing
    // share a factor)
    auto claim = [&]() -> int64_t {
        unsigned v = 0u;
        if (lane == 0) v = atomicAdd(P.next, 1u);
        return (int64_t)__shfl_sync(kFull, v, 0);
    };
    int64_t k_next = claim();
    while (k_next < T) {
        const int64_t k = k_next;
        k_next = claim();
        // position k is a decode piece when floor(k D / T) steps up at k + 1
        const int64_t f0 = k * D / T, f1 = (k + 1) * D / T;
        const bool dec = f1 > f0;
        const int64_t u = dec ? P.d_lo + f0 / kDecodeSub : P.h_lo + (k - f0);
        int c = 0;
        while (c + 1 < N && u >= P.unit_begin[c + 1][0]) ++c;
        int seg = 0;
        while (seg < 2 && u >= P.unit_begin[c][seg + 1]) ++seg;
        const int64_t j0 = P.seg_lo[c][seg] + (u - P.unit_begin[c][seg]) * kUnit +
                           (dec ? (f0 % kDecodeSub) * (kUnit / kDecodeSub) : 0);
        const int64_t rem = P.seg_hi[c][seg] - j0;
        const int64_t len = dec ? kUnit / kDecodeSub : kUnit;
        if (rem <= 0) continue;   // a piece past the end of a short unit
        const int cnt = (int)(rem < len ? rem : len);
        if (dec) {
            MsgView m = P.chunk[c];
            m.base = P.msgs + ((int64_t)c * N + (N - 1)) * P.msg_stride;
            if (seg == 0) decode_unit_rows<2, SF32>(P, m, P.lo[c], j0, cnt, lane, rows);
            else if (seg == 1) decode_unit_rows<4, SF32>(P, m, P.lo[c], j0, cnt, lane, rows);
            else decode_unit_rows<8, SF32>(P, m, P.lo[c], j0, cnt, lane, rows);
            continue;
        }
        // the part of unit u (largest p with units*p/n_parts <= u) and its step
        const int64_t part = ((u + 1) * P.n_parts - 1) / P.units;
        const int step = P.launch - (int)part;
        const int r = (c + 1 + step) % N, src = (r - 1 + N) % N;
        HopTask t;
        t.in = P.chunk[c];
        t.in.base = step > 0 ? P.msgs + ((int64_t)src * N + (step - 1)) * P.msg_stride : nullptr;
        t.out = P.chunk[c];
        t.out.base = P.msgs + ((int64_t)r * N + step) * P.msg_stride;
        t.addend = P.grads[r];
        t.keep_out = nullptr;
        t.in_lo = P.lo[c];
        t.send_lo = P.lo[c];
        t.send_hi = P.lo[c + 1];
        t.keep_lo = t.keep_hi = P.lo[c + 1];
        t.stage_word = (uint32_t)step | (P.correlated ? 0xFFFF0000u : ((uint32_t)r << 16));
        t.corr2 = 0u;   // one quantizer per ring stage: stratum offset 0
        if (step == 0) {
            if (seg == 0) hop_unit<2, false, false, ONE_LEVEL, SF32, false>(P, t, stg, j0, cnt, lane);
            else if (seg == 1) hop_unit<4, false, false, ONE_LEVEL, SF32, false>(P, t, stg, j0, cnt, lane);
            else hop_unit<8, false, false, ONE_LEVEL, SF32, false>(P, t, stg, j0, cnt, lane);
        } else {
            if (seg == 0) hop_unit<2, true, false, ONE_LEVEL, SF32, false>(P, t, stg, j0, cnt, lane);
            else if (seg == 1) hop_unit<4, true, false, ONE_LEVEL, SF32, false>(P, t, stg, j0, cnt, lane);
            else hop_unit<8, true, false, ONE_LEVEL, SF32, false>(P, t, stg, j0, cnt, lane);
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // the decode's copies
}

// Chunk cuts and work units of one bucket, derived from its plan's counts
// (32-bit: a bucket has fewer than 2^27 super-groups).  The cuts follow
// dq_chunk_cuts: chunk c starts at the first super-group whose code bits
// before it reach ceil(c * total / N).
struct SlotGeom {
    int32_t lo[kMaxStreamRanks + 1];
    int32_t ub[kMaxStreamRanks][4];   // first unit of each segment of chunk c; [3] = its end
    int32_t end2, end4, units, pad;
};

__device__ __forceinline__ void slot_geometry(const BucketSlot &S, int N, SlotGeom &g)
{
    const int64_t J = S.n_sg;
    // counts from a plan whose input was not finite are not trusted: clamped,
    // they still describe J super-groups, so every index stays in range
    const int64_t n2 = min(max(S.counts[0], (int64_t)0), J);
    const int64_t n4 = min(max(S.counts[1], (int64_t)0), J - n2);
    const int64_t n8 = J - n2 - n4;
    const int64_t total = 2 * n2 + 4 * n4 + 8 * n8;
    g.lo[0] = 0;
    for (int c = 1; c < N; ++c) {
        const int64_t target = ((int64_t)c * total + N - 1) / N;
        int64_t i;
        if (target <= 2 * n2) i = (target + 1) / 2;
        else if (target <= 2 * n2 + 4 * n4) i = n2 + (target - 2 * n2 + 3) / 4;
        else i = n2 + n4 + (target - 2 * n2 - 4 * n4 + 7) / 8;
        g.lo[c] = (int32_t)i;
    }
    g.lo[N] = (int32_t)J;
    g.end2 = (int32_t)n2;
    g.end4 = (int32_t)(n2 + n4);
    int32_t u = 0;
    for (int c = 0; c < N; ++c) {
        const int32_t a = g.lo[c], b = g.lo[c + 1];
        const int32_t cuts[4] = {a, max(a, min(b, g.end2)), max(a, min(b, g.end4)), b};
        for (int s = 0; s < 3; ++s) {
            g.ub[c][s] = u;
            u += (cuts[s + 1] - cuts[s] + kUnit - 1) / kUnit;
        }
        g.ub[c][3] = u;
    }
    g.units = u;
}

// Message layout of chunk [a, b) of a bucket (msg_view on the device).
__device__ __forceinline__ MsgView chunk_view(uint8_t *base, int32_t a, int32_t b, int32_t end2, int32_t end4,
                                              bool sf32)
{
    auto overlap = [](int32_t x0, int32_t x1, int32_t y0, int32_t y1) {
        const int32_t l = max(x0, y0), h = min(x1, y1);
        return h > l ? h - l : 0;
    };
    MsgView m;
    m.base = base;
    m.c = b - a;
    m.n2 = overlap(a, b, 0, end2);
    m.n4 = overlap(a, b, end2, end4);
    m.off_u = sf32 ? 0 : (m.c + 15) / 16 * 16;
    m.off_c2 = m.off_u + (sf32 ? 64 : 16) * m.c;
    m.off_c4 = m.off_c2 + 64 * m.n2;
    m.off_c8 = m.off_c4 + 128 * m.n4;
    return m;
}

// One launch of the bucket stream (StreamRingParams).  Every block first
// derives the chunk cuts and work units of the launch's buckets from their
// plans' counts (shared memory).  The tasks are the work units of every
// bucket at a ring step and the decode pieces of the bucket at its final
// decode, spread evenly through the task list; warps claim them in turn from
// the launch's counter, one ahead.  Step s of chunk c of a bucket is handled
// by rank r = (c + 1 + s) mod N, which reads rank r-1's message of step s-1
// and writes its own of step s (step 0 quantizes the local gradient); the
// decode reads owner c's message of step N-1.  Launched with programmatic
// stream serialization, as the pipelined exchange's kernel.
template <bool ONE_LEVEL, bool SF32>
__global__ void __launch_bounds__(kWarps * 32, 1) stream_ring_kernel(const __grid_constant__ StreamRingParams P)
{
    __shared__ SlotGeom geo[kMaxStreamRanks + 1];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    block_copy(&g_tab, &P.tab);
    __syncthreads();
    expand_bk4();
    expand_tables(true);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the plans' counts and the previous launch's messages
    const int N = P.n_ranks;
    if (threadIdx.x < (unsigned)P.n_slots) slot_geometry(P.slot[threadIdx.x], N, geo[threadIdx.x]);
    __syncthreads();
    uint8_t *dyn = g_dyn + tab_bytes(false);
    constexpr int STAGE = stage_bytes<false, SF32>();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *stg = dyn + warp * kStages * STAGE;
    uint8_t *rows = dyn + kWarps * kStages * STAGE + warp * 2 * kRowBytes;
    // hop tasks H (units of the buckets at a ring step) and decode pieces D
    uint32_t H = 0, D = 0;
    int dslot = -1;
    for (int i = 0; i < P.n_slots; ++i) {
        if (P.slot[i].step == N) {
            dslot = i;
            D = (uint32_t)geo[i].units * kDecodeSub;
        } else {
            H += (uint32_t)geo[i].units;
        }
    }
    const uint32_t T = H + D, stride = D > 0 ? T / D : 1u;
    uint32_t k_next = 0u;
    if (lane == 0) k_next = atomicAdd(P.next, 1u);
    k_next = __shfl_sync(kFull, k_next, 0);
    while (k_next < T) {
        const uint32_t k = k_next;
        if (lane == 0) k_next = atomicAdd(P.next, 1u);
        k_next = __shfl_sync(kFull, k_next, 0);
        // position k is a decode piece when k = i * stride + stride - 1 with i < D
        const uint32_t q = k / stride, in_step = k - q * stride;
        const bool dec = D > 0 && q < D && in_step == stride - 1;
        int si;
        uint32_t u, piece = 0;
        if (dec) {
            si = dslot;
            u = q / kDecodeSub;
            piece = q % kDecodeSub;
        } else {
            u = k - min(q, D);   // the hop tasks before k: k minus the pieces before it
            si = 0;
            while (si == dslot || u >= (uint32_t)geo[si].units) {
                if (si != dslot) u -= (uint32_t)geo[si].units;
                ++si;
            }
        }
        const BucketSlot &S = P.slot[si];
        const SlotGeom &g = geo[si];
        int c = 0;
        while (c + 1 < N && (int32_t)u >= g.ub[c + 1][0]) ++c;
        int seg = 0;
        while (seg < 2 && (int32_t)u >= g.ub[c][seg + 1]) ++seg;
        const int32_t a = g.lo[c], b = g.lo[c + 1];
        const int32_t c2 = max(a, min(b, g.end2)), c4 = max(a, min(b, g.end4));   // the segments' cuts
        const int32_t seg_lo = seg == 0 ? a : (seg == 1 ? c2 : c4), seg_hi = seg == 0 ? c2 : (seg == 1 ? c4 : b);
        const int32_t j0 = seg_lo + ((int32_t)u - g.ub[c][seg]) * kUnit + (int32_t)piece * (kUnit / kDecodeSub);
        const int32_t len = dec ? kUnit / kDecodeSub : kUnit;
        const int32_t rem = seg_hi - j0;
        if (rem <= 0) continue;   // a piece past the end of a short unit
        const int cnt = rem < len ? rem : len;
        if (dec) {
            const MsgView m = chunk_view(S.msgs + ((int64_t)c * N + (N - 1)) * S.msg_stride, a, b, g.end2, g.end4, SF32);
            if (seg == 0) decode_unit_rows<2, SF32>(S, m, a, j0, cnt, lane, rows);
            else if (seg == 1) decode_unit_rows<4, SF32>(S, m, a, j0, cnt, lane, rows);
            else decode_unit_rows<8, SF32>(S, m, a, j0, cnt, lane, rows);
            continue;
        }
        const int step = S.step;
        const int r = (c + 1 + step) % N, src = (r - 1 + N) % N;
        HopTask t;
        t.in = chunk_view(step > 0 ? S.msgs + ((int64_t)src * N + (step - 1)) * S.msg_stride : nullptr, a, b, g.end2,
                          g.end4, SF32);
        t.out = chunk_view(S.msgs + ((int64_t)r * N + step) * S.msg_stride, a, b, g.end2, g.end4, SF32);
        t.addend = S.grads[r];
        t.keep_out = nullptr;
        t.in_lo = a;
        t.send_lo = a;
        t.send_hi = b;
        t.keep_lo = t.keep_hi = b;
        t.stage_word = (uint32_t)step | (P.correlated ? 0xFFFF0000u : ((uint32_t)r << 16));
        t.corr2 = 0u;   // one quantizer per ring stage: stratum offset 0
        if (step == 0) {
            if (seg == 0) hop_unit<2, false, false, ONE_LEVEL, SF32, false>(S, t, stg, j0, cnt, lane);
            else if (seg == 1) hop_unit<4, false, false, ONE_LEVEL, SF32, false>(S, t, stg, j0, cnt, lane);
            else hop_unit<8, false, false, ONE_LEVEL, SF32, false>(S, t, stg, j0, cnt, lane);
        } else {
            if (seg == 0) hop_unit<2, true, false, ONE_LEVEL, SF32, false>(S, t, stg, j0, cnt, lane);
            else if (seg == 1) hop_unit<4, true, false, ONE_LEVEL, SF32, false>(S, t, stg, j0, cnt, lane);
            else hop_unit<8, true, false, ONE_LEVEL, SF32, false>(S, t, stg, j0, cnt, lane);
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // the decode's copies
}

// Opts a kernel in to `dyn` bytes of dynamic shared memory (needed once its
// static plus dynamic shared memory passes 48 KB), once per device; `done`
// is the caller's per-kernel record.
template <typename K>
cudaError_t allow_dyn_smem(K kernel, size_t dyn, bool (&done)[128])
{
    static std::mutex mu;   // first calls from several host threads may meet here
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

// Warps per block of a hop launch: one block per SM (its tables fill most of
// shared memory), as many warps as spread the launch's units over all SMs,
// at most kWarps.  The dynamic allocation always covers kWarps warps of
// staging, so a bucket row read for a non-finite value stays inside it.
inline int hop_block_warps(int64_t units)
{
    const int64_t sms = sm_count();
    const int64_t w = (units + sms - 1) / sms;
    return (int)std::max<int64_t>(1, std::min<int64_t>(kWarps, w));
}

template <typename K>
int grid_for(K kernel, int warps, size_t dyn_smem, int64_t units)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, warps * 32, dyn_smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int64_t need = (units + warps - 1) / warps;
    return (int)(need < cap ? (need < 1 ? 1 : need) : cap);
}

template <bool HAS_IN, bool ADD_F32, bool ONE_LEVEL, bool SF32, bool OFF = true>
cudaError_t launch_hop_t(const HopParams &P, cudaStream_t st)
{
    const size_t dyn = (size_t)tab_bytes(ADD_F32) + (size_t)kWarps * kStages * stage_bytes<ADD_F32, SF32>();
    auto k = hop_kernel<HAS_IN, ADD_F32, ONE_LEVEL, SF32, OFF>;
    static bool opted[128] = {false};   // one record per instantiation of this launcher
    const cudaError_t ea = allow_dyn_smem(k, dyn, opted);
    if (ea != cudaSuccess) return ea;
    const int wpb = hop_block_warps(P.total_units);
    k<<<grid_for(k, wpb, dyn, P.total_units), wpb * 32, dyn, st>>>(P);
    note_launches(1);
    return cudaGetLastError();
}

template <bool SF32>
cudaError_t launch_hop_s(const HopParams &P, bool has_in, bool add_f32, cudaStream_t st)
{
    const bool one = P.tab.one_level != 0;
    bool off = false;   // some task shifts its uniforms (correlated rounding with several slots)
    for (int i = 0; i < P.n_tasks; ++i) off = off || P.task[i].corr2 != 0u;
    if (!SF32 && one && !add_f32 && !off)   // the ring's kernels: no offsets to add
        return has_in ? launch_hop_t<true, false, true, SF32, false>(P, st) : launch_hop_t<false, false, true, SF32, false>(P, st);
    if (!has_in)
        return one ? launch_hop_t<false, false, true, SF32>(P, st) : launch_hop_t<false, false, false, SF32>(P, st);
    if (add_f32)
        return one ? launch_hop_t<true, true, true, SF32>(P, st) : launch_hop_t<true, true, false, SF32>(P, st);
    return one ? launch_hop_t<true, false, true, SF32>(P, st) : launch_hop_t<true, false, false, SF32>(P, st);
}

template <bool SF32>
cudaError_t launch_decode_s(const DecodeParams &P, cudaStream_t st)
{
    auto k = decode_kernel<SF32>;
    const size_t dyn = (size_t)kDecodeWarps * kDecodeSlice * 1024;
    static bool opted[128] = {false};   // one record per instantiation of this launcher
    const cudaError_t ea = allow_dyn_smem(k, dyn, opted);
    if (ea != cudaSuccess) return ea;
    const int64_t warps = P.total_units * kDecodeSplit;
    k<<<(unsigned)((warps + kDecodeWarps - 1) / kDecodeWarps), kDecodeWarps * 32, dyn, st>>>(P);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hop(const HopParams &P, bool has_in, bool add_f32, cudaStream_t st)
{
    if (P.total_units <= 0) return cudaSuccess;
    return P.scale_fp32 ? launch_hop_s<true>(P, has_in, add_f32, st) : launch_hop_s<false>(P, has_in, add_f32, st);
}

cudaError_t launch_decode(const DecodeParams &P, cudaStream_t st)
{
    if (P.total_units <= 0) return cudaSuccess;
    return P.scale_fp32 ? launch_decode_s<true>(P, st) : launch_decode_s<false>(P, st);
}

namespace {

template <bool ONE_LEVEL, bool SF32>
cudaError_t launch_fused_t(const FusedRingParams &P, cudaStream_t st)
{
    const size_t dyn = (size_t)tab_bytes(false) + (size_t)kWarps * kStages * stage_bytes<false, SF32>();
    auto k = fused_ring_kernel<ONE_LEVEL, SF32>;
    static bool opted[128] = {false};   // one record per instantiation of this launcher
    cudaError_t e = allow_dyn_smem(k, dyn, opted);
    if (e != cudaSuccess) return e;
    const int wpb = hop_block_warps(P.units);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, wpb * 32, dyn);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    // every CTA must be resident at once (cooperative launch): at most the
    // CTAs that fit, and no more than the work needs
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int64_t need = std::max<int64_t>(1, (P.units + wpb - 1) / wpb);
    const int grid = (int)std::min(cap, need);
    void *args[] = {const_cast<FusedRingParams *>(&P)};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(k), dim3(grid), dim3(wpb * 32), args, dyn, st);
    note_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_ring(const FusedRingParams &P, cudaStream_t st)
{
    const bool one = P.tab.one_level != 0;
    if (P.scale_fp32) return one ? launch_fused_t<true, true>(P, st) : launch_fused_t<false, true>(P, st);
    return one ? launch_fused_t<true, false>(P, st) : launch_fused_t<false, false>(P, st);
}

namespace {

template <bool ONE_LEVEL, bool SF32>
cudaError_t launch_wave_t(const WaveRingParams &P, int64_t units, cudaStream_t st)
{
    const size_t dyn = (size_t)tab_bytes(false) + (size_t)kWarps * kStages * stage_bytes<false, SF32>() +
                       (size_t)kWarps * 2 * kRowBytes;
    auto k = wave_ring_kernel<ONE_LEVEL, SF32>;
    static bool opted[128] = {false};   // one record per instantiation of this launcher
    const cudaError_t e = allow_dyn_smem(k, dyn, opted);
    if (e != cudaSuccess) return e;
    const int wpb = hop_block_warps(units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid_for(k, wpb, dyn, units));
    cfg.blockDim = dim3((unsigned)(wpb * 32));
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t el = cudaLaunchKernelEx(&cfg, k, P);
    note_launches(1);
    return el != cudaSuccess ? el : cudaGetLastError();
}

}  // namespace

namespace {

template <bool ONE_LEVEL, bool SF32>
cudaError_t launch_stream_t(const StreamRingParams &P, int64_t tasks, cudaStream_t st, int free_sms)
{
    const size_t dyn = (size_t)tab_bytes(false) + (size_t)kWarps * kStages * stage_bytes<false, SF32>() +
                       (size_t)kWarps * 2 * kRowBytes;
    auto k = stream_ring_kernel<ONE_LEVEL, SF32>;
    static bool opted[128] = {false};   // one record per instantiation of this launcher
    const cudaError_t e = allow_dyn_smem(k, dyn, opted);
    if (e != cudaSuccess) return e;
    const int wpb = hop_block_warps(tasks);
    cudaLaunchConfig_t cfg = {};
    // one block per SM; free_sms SMs are left to other streams' kernels
    cfg.gridDim = dim3((unsigned)std::max(1, std::min(grid_for(k, wpb, dyn, tasks), sm_count() - free_sms)));
    cfg.blockDim = dim3((unsigned)(wpb * 32));
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t el = cudaLaunchKernelEx(&cfg, k, P);
    note_launches(1);
    return el != cudaSuccess ? el : cudaGetLastError();
}

}  // namespace

cudaError_t launch_stream_ring(const StreamRingParams &P, int64_t tasks_hint, cudaStream_t st, int free_sms)
{
    const bool one = P.tab.one_level != 0;
    if (P.scale_fp32)
        return one ? launch_stream_t<true, true>(P, tasks_hint, st, free_sms)
                   : launch_stream_t<false, true>(P, tasks_hint, st, free_sms);
    return one ? launch_stream_t<true, false>(P, tasks_hint, st, free_sms)
               : launch_stream_t<false, false>(P, tasks_hint, st, free_sms);
}

cudaError_t launch_wave_ring(const WaveRingParams &P, cudaStream_t st)
{
    const int64_t units = (P.h_hi - P.h_lo) + (P.d_hi - P.d_lo);
    if (units <= 0) return cudaSuccess;
    const bool one = P.tab.one_level != 0;
    if (P.scale_fp32) return one ? launch_wave_t<true, true>(P, units, st) : launch_wave_t<false, true>(P, units, st);
    return one ? launch_wave_t<true, false>(P, units, st) : launch_wave_t<false, false>(P, units, st);
}

cudaError_t launch_barrier_selftest(int32_t n_blocks, int32_t missing, long long timeout_cycles, unsigned *counter,
                                    int32_t *status, cudaStream_t st)
{
    unsigned target = (unsigned)n_blocks + (unsigned)missing;
    void *args[] = {&counter, &status, &target, &timeout_cycles};
    const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(barrier_selftest_kernel),
                                                      dim3(n_blocks), dim3(32), args, 0, st);
    note_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dq
