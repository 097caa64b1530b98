// dq_codec.cu -- statistics, fused hop (compress / decompress-accumulate-
// recompress) and final decode kernels.
//
// Work mapping: one warp per super-group, lane l owning coordinates
// 8l .. 8l+7 (16 bytes of bf16, one 128-bit load).  Lanes 2g and 2g+1 form
// group g, so a group maximum is one xor-1 shuffle and a super-group maximum
// four more.  Lane l's codes are the b contiguous bytes at b*l of the
// super-group's code block, so the codes of a super-group are written by one
// coalesced warp store, and lane l draws one Philox call (128 bits = eight
// 16-bit uniforms) for its eight coordinates.
#include "dq_common.cuh"
#include "dq_internal.h"

namespace dq {

// ---------------------------------------------------------------------------
// Statistics: per super-group sum and sum of squares over the raw bf16
// values, fp32, fixed tree.  Tree within a group: a[i] += a[i+h] for
// h = 8, 4, 2, 1 (h = 8 pairs the two lanes of a group: one xor-1 shuffle;
// h = 4, 2, 1 stay in the lane).  Then the 16 group partials by the same
// tree: h = 8, 4, 2, 1 groups apart = lanes xor 16, 8, 4, 2.  fp32 addition
// is commutative, so the lane on either side of a shuffle computes the same
// value.  mean = sum * 2^-8.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float lane_tree8(float (&a)[8])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __fadd_rn(a[i], __shfl_xor_sync(kFull, a[i], 1));
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) a[i] = __fadd_rn(a[i], a[i + h]);
    float v = a[0];
#pragma unroll
    for (int m = 16; m >= 2; m >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

__global__ void __launch_bounds__(256) stats_kernel(const uint16_t *__restrict__ g, int64_t n_sg,
                                                    float *__restrict__ mean, float *__restrict__ sq)
{
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t j = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; j < n_sg; j += nw) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(g + j * kSG) + lane);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float a[8], b[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            a[2 * k] = bf16_lo(w[k]);
            a[2 * k + 1] = bf16_hi(w[k]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = __fmul_rn(a[i], a[i]);
        const float s = lane_tree8(a);
        const float q = lane_tree8(b);
        if (lane == 0) {
            mean[j] = __fmul_rn(s, 0.00390625f);
            sq[j] = q;
        }
    }
}

// Metadata all-reduce: M_j and F_j summed over ranks 0..N-1 in order.
__global__ void __launch_bounds__(256) stats_reduce_kernel(const float *__restrict__ mean_all,
                                                           const float *__restrict__ sq_all, int32_t n,
                                                           int64_t n_sg, float *__restrict__ M,
                                                           float *__restrict__ F)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n_sg; j += stride) {
        float m = mean_all[j], f = sq_all[j];
        for (int32_t w = 1; w < n; ++w) {
            m = __fadd_rn(m, mean_all[(int64_t)w * n_sg + j]);
            f = __fadd_rn(f, sq_all[(int64_t)w * n_sg + j]);
        }
        M[j] = m;
        F[j] = f;
    }
}

// ---------------------------------------------------------------------------
// Quantization of one lane's eight values (the lane's share of one
// super-group).  Scale hierarchy: s_g = group max |x|; S = super-group max;
// e = smallest integer >= -126 with 255 * 2^e >= S (E = e + 127, E = 0 when
// S = 0); u_g = smallest integer with u_g * 2^e >= s_g; m_g =
// fl(fl(1/u_g) * 2^-e).  Per coordinate: y = clamp(fl(x * m_g), -1, 1);
// k = largest level <= y (bucket table, then exact compares); p =
// fl(fl(y - q_k) * G_k); code = k + (U * 2^-16 < p).
// ---------------------------------------------------------------------------
struct LaneQuant {
    uint32_t E;     // exponent byte of the super-group
    uint32_t u;     // UINT8 scale of this lane's group
    uint64_t codes; // 8 codes, BITS bits each, coordinate i at bits BITS*i
};

// e for S > 0: with S = (1 + f) 2^(eb-127), 255 * 2^e >= S holds first at
// e = eb - 134 when (1 + f) <= 510/256 (mantissa field <= 0x7F0000), else at
// eb - 133; subnormal S (eb = 0) and tiny S clamp to -126.
__device__ __forceinline__ uint32_t exponent_byte(float S)
{
    if (!(S > 0.0f)) return 0u;
    const uint32_t bits = __float_as_uint(S);
    const int eb = (int)(bits >> 23);
    int e = eb - 134 + ((bits & 0x7FFFFFu) > 0x7F0000u ? 1 : 0);
    if (eb == 0 || e < -126) e = -126;
    return (uint32_t)(e + 127);
}

template <int BITS>
__device__ __forceinline__ LaneQuant quantize_lane(const float (&x)[8], const Tables &T, uint32_t ctr0,
                                                   uint32_t stage_word, uint32_t corr_off,
                                                   uint32_t key0, uint32_t key1, uint32_t round0,
                                                   uint32_t round1)
{
    const float2 *qg = BITS == 2 ? T.qg2 : (BITS == 4 ? T.qg4 : T.qg8);
    const BucketEntry *bk = BITS == 2 ? T.bk2 : (BITS == 4 ? T.bk4 : T.bk8);
    const int Hi = BITS == 2 ? T.H2 : (BITS == 4 ? T.H4 : T.H8);
    const float H = (float)Hi;

    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s = fmaxf(s, fabsf(x[i]));
    s = fmaxf(s, __shfl_xor_sync(kFull, s, 1));
    float S = s;
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) S = fmaxf(S, __shfl_xor_sync(kFull, S, m));

    LaneQuant r;
    r.E = exponent_byte(S);
    r.u = 0u;
    float mult = 0.0f;
    if (s > 0.0f) {
        const float inv2e = __uint_as_float((254u - r.E) << 23);  // 2^-e, a normal float
        const float t = __fmul_rn(s, inv2e);                         // exact unless subnormal
        int u = (int)ceilf(t);
        u = u < 1 ? 1 : u;
        r.u = (uint32_t)u;
        mult = __fmul_rn(__frcp_rn((float)u), inv2e);
    }

    uint32_t c[4] = {ctr0, stage_word, round0, round1};
    philox4x32_10(c, key0, key1);

    uint64_t codes = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float y = __fmul_rn(x[i], mult);
        y = fminf(fmaxf(y, -1.0f), 1.0f);
        const int t = __float2int_rd(__fmul_rn(y, H)) + Hi;
        const BucketEntry be = bk[t];
        int k = be.kb;
        if (y >= be.boundary) {
            ++k;
            while (y >= qg[k + 1].x) ++k;
        }
        const float2 lv = qg[k];
        const float p = __fmul_rn(__fsub_rn(y, lv.x), lv.y);
        const uint32_t w = c[i >> 1];
        uint32_t U = (i & 1) ? (w >> 16) : (w & 0xFFFFu);
        U = (U + corr_off) & 0xFFFFu;
        const float uf = __fsub_rn(__uint_as_float(0x3F800000u | (U << 7)), 1.0f);  // U * 2^-16
        const int code = k + (uf < p ? 1 : 0);
        codes |= (uint64_t)(uint32_t)code << (BITS * i);
    }
    r.codes = codes;
    return r;
}

// Decoded values of one lane: fl(sigma_g * q_code), sigma_g = u_g * 2^(E-127).
template <int BITS>
__device__ __forceinline__ void decode_lane(uint64_t codes, uint32_t E, uint32_t u, const Tables &T,
                                            float (&d)[8])
{
    const float2 *qg = BITS == 2 ? T.qg2 : (BITS == 4 ? T.qg4 : T.qg8);
    const float sigma = E ? __fmul_rn((float)u, __uint_as_float(E << 23)) : 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t code = (uint32_t)(codes >> (BITS * i)) & ((1u << BITS) - 1u);
        d[i] = __fmul_rn(sigma, qg[code].x);
    }
}

// Code block of local super-group s of a message, and the lane's part of it.
template <int BITS>
__device__ __forceinline__ const uint8_t *code_block(const MsgView &m, int64_t s)
{
    if (BITS == 2) return m.base + m.off_c2 + 64 * s;
    if (BITS == 4) return m.base + m.off_c4 + 128 * (s - m.n2);
    return m.base + m.off_c8 + 256 * (s - m.n2 - m.n4);
}

template <int BITS>
__device__ __forceinline__ uint64_t load_codes(const uint8_t *blk, int lane)
{
    if (BITS == 2) return __ldcs(reinterpret_cast<const unsigned short *>(blk) + lane);
    if (BITS == 4) return __ldcs(reinterpret_cast<const unsigned int *>(blk) + lane);
    const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(blk) + lane);
    return (uint64_t)v.x | ((uint64_t)v.y << 32);
}

template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t *blk, int lane, uint64_t codes)
{
    if (BITS == 2) reinterpret_cast<unsigned short *>(blk)[lane] = (unsigned short)codes;
    else if (BITS == 4) reinterpret_cast<unsigned int *>(blk)[lane] = (unsigned int)codes;
    else reinterpret_cast<uint2 *>(blk)[lane] = make_uint2((uint32_t)codes, (uint32_t)(codes >> 32));
}

// ---------------------------------------------------------------------------
// Fused hop over one super-group (reordered index j) of one task.
// HAS_IN: decode the incoming message and add (DAR); otherwise compress.
// ADD_F32: the addend is fp32 partial sums (butterfly); otherwise the bf16
// local gradient read through perm, minus mu_j = fl(M_j / N).
// ---------------------------------------------------------------------------
template <int BITS, bool HAS_IN, bool ADD_F32>
__device__ __forceinline__ void hop_sg(const HopParams &P, const HopTask &t, const Tables &T, int64_t j,
                                       int lane)
{
    const int64_t old = __ldg(P.perm + j);
    const int64_t s_in = j - t.in_lo;
    float x[8];
    if (ADD_F32) {
        const float4 *a = reinterpret_cast<const float4 *>(static_cast<const float *>(t.addend) +
                                                          s_in * kSG) + 2 * lane;
        const float4 a0 = __ldcs(a), a1 = __ldcs(a + 1);
        x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w;
        x[4] = a1.x; x[5] = a1.y; x[6] = a1.z; x[7] = a1.w;
    } else {
        const float mu = __fdiv_rn(__ldg(P.M + old), (float)P.n_ranks);
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(t.addend) +
                                                               old * kSG) + lane);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __fsub_rn(bf16_lo(w[k]), mu);
            x[2 * k + 1] = __fsub_rn(bf16_hi(w[k]), mu);
        }
    }
    if (HAS_IN) {
        const uint8_t *mb = t.in.base;
        const uint32_t E = __ldg(mb + s_in);
        const uint32_t u = __ldg(mb + t.in.off_u + s_in * 16 + (lane >> 1));
        const uint64_t codes = load_codes<BITS>(code_block<BITS>(t.in, s_in), lane);
        float d[8];
        decode_lane<BITS>(codes, E, u, T, d);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __fadd_rn(d[i], x[i]);
    }
    if (j >= t.send_lo && j < t.send_hi) {
        const int64_t so = j - t.send_lo;
        const uint32_t ctr0 = (uint32_t)((uint64_t)old * 32u + (uint64_t)lane);
        const LaneQuant qz = quantize_lane<BITS>(x, T, ctr0, t.stage_word, t.corr_off, P.key0, P.key1,
                                                 P.round0, P.round1);
        uint8_t *ob = t.out.base;
        if (lane == 0) ob[so] = (uint8_t)qz.E;
        if ((lane & 1) == 0) ob[t.out.off_u + so * 16 + (lane >> 1)] = (uint8_t)qz.u;
        store_codes<BITS>(const_cast<uint8_t *>(code_block<BITS>(t.out, so)), lane, qz.codes);
    } else if (j >= t.keep_lo && j < t.keep_hi) {
        float4 *k = reinterpret_cast<float4 *>(t.keep_out + (j - t.keep_lo) * kSG) + 2 * lane;
        k[0] = make_float4(x[0], x[1], x[2], x[3]);
        k[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
}

template <bool HAS_IN, bool ADD_F32>
__global__ void __launch_bounds__(256) hop_kernel(const __grid_constant__ HopParams P)
{
    __shared__ __align__(16) Tables T;
    block_copy(&T, &P.tab);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < P.total_sg; g += nw) {
        int ti = 0;
        while (ti + 1 < P.n_tasks && g >= P.task[ti + 1].sg_begin) ++ti;
        const HopTask &t = P.task[ti];
        const int64_t j = t.in_lo + (g - t.sg_begin);
        if (j < P.end2) hop_sg<2, HAS_IN, ADD_F32>(P, t, T, j, lane);
        else if (j < P.end4) hop_sg<4, HAS_IN, ADD_F32>(P, t, T, j, lane);
        else hop_sg<8, HAS_IN, ADD_F32>(P, t, T, j, lane);
    }
}

// ---------------------------------------------------------------------------
// Final decode: out[perm[j]*256 + i] = fl(dec + fl(fl(M_j / N) * N)).
// ---------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ void decode_sg(const DecodeParams &P, const DecodeTask &t, const Tables &T,
                                          int64_t j, int lane)
{
    const int64_t old = __ldg(P.perm + j);
    const int64_t s = j - t.lo;
    const uint8_t *mb = t.msg.base;
    const uint32_t E = __ldg(mb + s);
    const uint32_t u = __ldg(mb + t.msg.off_u + s * 16 + (lane >> 1));
    const uint64_t codes = load_codes<BITS>(code_block<BITS>(t.msg, s), lane);
    float d[8];
    decode_lane<BITS>(codes, E, u, T, d);
    const float mu = __fdiv_rn(__ldg(P.M + old), (float)P.n_ranks);
    const float back = __fmul_rn(mu, (float)P.n_ranks);
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = __fadd_rn(d[i], back);
    if (P.out_is_bf16) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(d[2 * k]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(d[2 * k + 1]));
            w[k] = lo | (hi << 16);
        }
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(P.out) + old * kSG) + lane;
        __stcs(o, make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(P.out) + old * kSG) + 2 * lane;
        __stcs(o, make_float4(d[0], d[1], d[2], d[3]));
        __stcs(o + 1, make_float4(d[4], d[5], d[6], d[7]));
    }
}

__global__ void __launch_bounds__(256) decode_kernel(const __grid_constant__ DecodeParams P)
{
    __shared__ __align__(16) Tables T;
    block_copy(&T, &P.tab);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < P.total_sg; g += nw) {
        int ti = 0;
        while (ti + 1 < P.n_tasks && g >= P.task[ti + 1].sg_begin) ++ti;
        const DecodeTask &t = P.task[ti];
        const int64_t j = t.lo + (g - t.sg_begin);
        if (j < P.end2) decode_sg<2>(P, t, T, j, lane);
        else if (j < P.end4) decode_sg<4>(P, t, T, j, lane);
        else decode_sg<8>(P, t, T, j, lane);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
static int grid_for(int64_t work_warps)
{
    const int64_t blocks = (work_warps + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

cudaError_t launch_stats(const uint16_t *g, int64_t n_sg, float *mean, float *sq, cudaStream_t st)
{
    stats_kernel<<<grid_for(n_sg), 256, 0, st>>>(g, n_sg, mean, sq);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_stats_reduce(const float *mean_all, const float *sq_all, int32_t n, int64_t n_sg,
                                float *M, float *F, cudaStream_t st)
{
    int64_t blocks = (n_sg + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    blocks = blocks < 1 ? 1 : (blocks < cap ? blocks : cap);
    stats_reduce_kernel<<<(int)blocks, 256, 0, st>>>(mean_all, sq_all, n, n_sg, M, F);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_hop(const HopParams &P, bool has_in, bool add_f32, cudaStream_t st)
{
    if (P.total_sg <= 0) return cudaSuccess;
    const int grid = grid_for(P.total_sg);
    if (!has_in) hop_kernel<false, false><<<grid, 256, 0, st>>>(P);
    else if (add_f32) hop_kernel<true, true><<<grid, 256, 0, st>>>(P);
    else hop_kernel<true, false><<<grid, 256, 0, st>>>(P);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams &P, cudaStream_t st)
{
    if (P.total_sg <= 0) return cudaSuccess;
    decode_kernel<<<grid_for(P.total_sg), 256, 0, st>>>(P);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace dq
