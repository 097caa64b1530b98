// dq_mx.cu -- the MXFP8 comparison baseline: OCP Microscaling (MX) v1.0
// MXFP8 encoding (blocks of 32 E4M3 elements sharing one E8M0 scale) inside
// the same N-rank ring / butterfly schedule as DynamiQ, every hop decoding,
// adding in fp32 and re-encoding.  DynamiQ's pages compare their error with
// MXFP8's (Abstract; scribe notes "Evaluation"); this path measures that
// comparison and the cost of an MXFP8 hop on the same hardware.
//
// Encoding of a block (the conversion rule of the MX specification): the
// shared exponent x = floor(log2(max |V_i|)) - 8 (8 being the exponent of
// E4M3's largest normal, 448), clamped at -127, stored as the byte x + 127
// (0 for an all-zero block); P_i = V_i * 2^-x converted to E4M3 with
// round-to-nearest-even, saturating at +-448 (cvt .satfinite).  For a normal
// max with biased fp32 exponent field f the byte is max(f - 8, 0); V_i * 2^-x
// is a power-of-two scaling (exact wherever the result can round to a
// non-zero E4M3 value).  Decoding: P_i * 2^x is exact in fp32 (E4M3 values
// have 4 significant bits and the smallest product is 2^-136).
//
// Work mapping: a warp takes 16 consecutive blocks (512 coordinates) of one
// task; lane l handles elements 4(l mod 8) .. +3 of block 4i + l/8 in
// sub-step i = 0..3, so every load and store instruction of the warp covers
// contiguous memory, and a block's maximum takes three shuffles inside its
// 8 lanes.  All loads of the 16 blocks are issued before any arithmetic.
#include <cuda_fp8.h>
#include <string.h>

#include <algorithm>
#include <memory>
#include <vector>

#include "dq_common.cuh"
#include "dq_internal.h"
#include "dq_sched.h"

namespace dq {
namespace {

constexpr int kMxBlk = 32;      // elements per block
constexpr int kMxUnit = 16;     // blocks per warp work unit
constexpr int kMxWarps = 8;     // warps per CTA
constexpr int kMxMaxOuts = 64;  // outputs written by one decode launch

struct MxTask {
    const uint8_t *in;          // incoming message over blocks [lo, hi) (unused for the first hop)
    const void *addend;         // bf16 gradient (block b at b*32) or fp32 rows (b - lo)
    uint8_t *out;               // message over [send_lo, send_hi)
    float *keep;                // fp32 rows (b - keep_lo)
    int64_t lo, hi, send_lo, send_hi, keep_lo, keep_hi;
    int64_t in_pad, out_pad;    // offset of the element section (block count padded to 16)
    int64_t unit_begin;         // first global work unit
};

struct MxParams {
    MxTask task[kMaxTasks];
    int32_t n_tasks;
    int64_t total_units;
};

struct MxDecodeTask {
    const uint8_t *msg;         // final message over blocks [lo, hi)
    int64_t lo, hi, pad, unit_begin;
};

struct MxDecodeParams {
    MxDecodeTask task[kMaxTasks];
    int32_t n_tasks;
    int64_t total_units;
    float *outs[kMxMaxOuts];    // every output receives every decoded block
    int32_t n_outs;
};

int64_t pad16(int64_t n) { return (n + 15) / 16 * 16; }

// 2^(X-127) for a scale byte X in [0, 254] (X = 0: the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t X)
{
    return X ? __uint_as_float(X << 23) : __uint_as_float(0x00200000u);
}

// Four E4M3 codes (byte k = element k) -> fp32, exactly (via f16, which
// holds every E4M3 value).
__device__ __forceinline__ float4 e4m3x4_to_f32(uint32_t w)
{
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Four fp32 -> E4M3 codes (byte k = element k), nearest-even, saturating.
__device__ __forceinline__ uint32_t f32x4_to_e4m3(float a, float b, float c, float d)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi << 16);
}

template <typename Task>
__device__ __forceinline__ int mx_locate(const Task *tasks, int n, int64_t u)
{
    int ti = 0;
    while (ti + 1 < n && u >= tasks[ti + 1].unit_begin) ++ti;
    return ti;
}

// One hop over all tasks: x = fl(dec(msg_in) + addend) (or x = addend for
// the first hop), then re-encode (send range) or keep as fp32 (keep range).
template <bool HAS_IN, bool ADD_F32>
__global__ void __launch_bounds__(kMxWarps * 32) mx_hop_kernel(const __grid_constant__ MxParams P)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, bq = lane >> 3;
    const int64_t nw = (int64_t)gridDim.x * kMxWarps;
    for (int64_t u = (int64_t)blockIdx.x * kMxWarps + warp; u < P.total_units; u += nw) {
        const MxTask &t = P.task[mx_locate(P.task, P.n_tasks, u)];
        const int64_t b0 = t.lo + (u - t.unit_begin) * kMxUnit;
        uint32_t code[4], xin[4];
        float4 add[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t b = b0 + 4 * i + bq;
            code[i] = 0u;
            xin[i] = 0u;
            add[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (b < t.hi) {
                const int64_t bl = b - t.lo;
                if (HAS_IN) {
                    code[i] = __ldg(reinterpret_cast<const uint32_t *>(t.in + t.in_pad + bl * kMxBlk) + sub);
                    xin[i] = __ldg(t.in + bl);
                }
                if (ADD_F32) {
                    add[i] = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(t.addend) + bl * kMxBlk) +
                                   sub);
                } else {
                    const uint2 w =
                        __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(t.addend) + b * kMxBlk) +
                              sub);
                    add[i] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t b = b0 + 4 * i + bq;
            float4 x = add[i];
            if (HAS_IN) {
                const float sc = e8m0_value(xin[i]);
                const float4 v = e4m3x4_to_f32(code[i]);
                x = make_float4(__fadd_rn(__fmul_rn(v.x, sc), x.x), __fadd_rn(__fmul_rn(v.y, sc), x.y),
                                __fadd_rn(__fmul_rn(v.z, sc), x.z), __fadd_rn(__fmul_rn(v.w, sc), x.w));
            }
            float a = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 1));
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 2));
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 4));
            if (b >= t.hi) continue;
            if (b >= t.send_lo && b < t.send_hi) {
                const uint32_t f = __float_as_uint(a) >> 23;
                const uint32_t X = f > 8u ? f - 8u : 0u;
                const float inv = __uint_as_float((254u - X) << 23);   // 2^(127 - X)
                const uint32_t w = f32x4_to_e4m3(__fmul_rn(x.x, inv), __fmul_rn(x.y, inv), __fmul_rn(x.z, inv),
                                                 __fmul_rn(x.w, inv));
                const int64_t so = b - t.send_lo;
                reinterpret_cast<uint32_t *>(t.out + t.out_pad + so * kMxBlk)[sub] = w;
                if (sub == 0) t.out[so] = (uint8_t)X;
                if (b == t.send_hi - 1 && sub > 0) {   // zero the scale section's padding
                    const int64_t c = t.send_hi - t.send_lo;
                    for (int64_t q = c + sub - 1; q < t.out_pad; q += 7) t.out[q] = 0;
                }
            } else if (b >= t.keep_lo && b < t.keep_hi) {
                reinterpret_cast<float4 *>(t.keep + (b - t.keep_lo) * kMxBlk)[sub] = x;
            }
        }
    }
}

// Final decode: every task's blocks to every output (one read, n_outs writes).
__global__ void __launch_bounds__(kMxWarps * 32) mx_decode_kernel(const __grid_constant__ MxDecodeParams P)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, bq = lane >> 3;
    const int64_t nw = (int64_t)gridDim.x * kMxWarps;
    for (int64_t u = (int64_t)blockIdx.x * kMxWarps + warp; u < P.total_units; u += nw) {
        const MxDecodeTask &t = P.task[mx_locate(P.task, P.n_tasks, u)];
        const int64_t b0 = t.lo + (u - t.unit_begin) * kMxUnit;
        uint32_t code[4], xin[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t b = b0 + 4 * i + bq;
            code[i] = xin[i] = 0u;
            if (b < t.hi) {
                code[i] = __ldg(reinterpret_cast<const uint32_t *>(t.msg + t.pad + (b - t.lo) * kMxBlk) + sub);
                xin[i] = __ldg(t.msg + (b - t.lo));
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t b = b0 + 4 * i + bq;
            if (b >= t.hi) continue;
            const float sc = e8m0_value(xin[i]);
            const float4 v = e4m3x4_to_f32(code[i]);
            const float4 y = make_float4(__fmul_rn(v.x, sc), __fmul_rn(v.y, sc), __fmul_rn(v.z, sc), __fmul_rn(v.w, sc));
            for (int o = 0; o < P.n_outs; ++o) __stcs(reinterpret_cast<float4 *>(P.outs[o] + b * kMxBlk) + sub, y);
        }
    }
}

template <typename K>
int mx_grid(K kernel, int64_t units)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kMxWarps * 32, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int64_t need = (units + kMxWarps - 1) / kMxWarps;
    return (int)std::max<int64_t>(1, std::min(need, cap));
}

cudaError_t launch_mx_hop(const MxParams &P, bool has_in, bool add_f32, cudaStream_t st)
{
    if (P.total_units <= 0) return cudaSuccess;
    if (has_in && add_f32) mx_hop_kernel<true, true><<<mx_grid(mx_hop_kernel<true, true>, P.total_units), kMxWarps * 32, 0, st>>>(P);
    else if (has_in) mx_hop_kernel<true, false><<<mx_grid(mx_hop_kernel<true, false>, P.total_units), kMxWarps * 32, 0, st>>>(P);
    else if (add_f32) mx_hop_kernel<false, true><<<mx_grid(mx_hop_kernel<false, true>, P.total_units), kMxWarps * 32, 0, st>>>(P);
    else mx_hop_kernel<false, false><<<mx_grid(mx_hop_kernel<false, false>, P.total_units), kMxWarps * 32, 0, st>>>(P);
    note_launches(1);
    return cudaGetLastError();
}

// The decode is launched flat (one unit per warp, grid sized to the work):
// short-lived blocks stream its writes faster than a persistent loop.
cudaError_t launch_mx_decode(const MxDecodeParams &P, cudaStream_t st)
{
    if (P.total_units <= 0) return cudaSuccess;
    mx_decode_kernel<<<(unsigned)((P.total_units + kMxWarps - 1) / kMxWarps), kMxWarps * 32, 0, st>>>(P);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------- host side
constexpr int64_t kMxMaxBlk = (int64_t)1 << 40;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Launches hop tasks in batches of at most kMaxTasks (empty ones dropped).
cudaError_t run_mx_hops(const std::vector<MxTask> &tasks, bool has_in, bool add_f32, cudaStream_t st,
                        dq_launch_log *log)
{
    std::unique_ptr<MxParams> P(new MxParams());
    size_t i = 0;
    while (i < tasks.size()) {
        memset(P.get(), 0, sizeof(MxParams));
        int n = 0;
        int64_t units = 0, blocks = 0;
        while (i < tasks.size() && n < kMaxTasks) {
            MxTask t = tasks[i++];
            if (t.hi <= t.lo) continue;
            t.unit_begin = units;
            units += (t.hi - t.lo + kMxUnit - 1) / kMxUnit;
            blocks += t.hi - t.lo;
            P->task[n++] = t;
        }
        P->n_tasks = n;
        P->total_units = units;
        if (n > 0) {
            const LogSlot slot = log_begin(log, DQ_LAUNCH_MX_HOP, blocks * kMxBlk / kSG, st);
            const cudaError_t e = launch_mx_hop(*P, has_in, add_f32, st);
            log_end(slot, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

struct MxChunk {
    const uint8_t *msg;
    int64_t lo, hi;
};

cudaError_t run_mx_decodes(const std::vector<MxChunk> &chunks, float *const *outs, int32_t n_outs, cudaStream_t st,
                           dq_launch_log *log)
{
    std::unique_ptr<MxDecodeParams> D(new MxDecodeParams());
    for (int32_t o0 = 0; o0 < n_outs; o0 += kMxMaxOuts) {
        size_t i = 0;
        while (i < chunks.size()) {
            memset(D.get(), 0, sizeof(MxDecodeParams));
            D->n_outs = std::min(n_outs - o0, kMxMaxOuts);
            for (int32_t o = 0; o < D->n_outs; ++o) D->outs[o] = outs[o0 + o];
            int n = 0;
            int64_t units = 0, blocks = 0;
            while (i < chunks.size() && n < kMaxTasks) {
                const MxChunk &c = chunks[i++];
                if (c.hi <= c.lo) continue;
                MxDecodeTask &t = D->task[n++];
                t.msg = c.msg;
                t.lo = c.lo;
                t.hi = c.hi;
                t.pad = pad16(c.hi - c.lo);
                t.unit_begin = units;
                units += (c.hi - c.lo + kMxUnit - 1) / kMxUnit;
                blocks += c.hi - c.lo;
            }
            D->n_tasks = n;
            D->total_units = units;
            if (n > 0) {
                const LogSlot slot = log_begin(log, DQ_LAUNCH_MX_DECODE, blocks * kMxBlk / kSG * D->n_outs, st);
                const cudaError_t e = launch_mx_decode(*D, st);
                log_end(slot, st);
                if (e != cudaSuccess) return e;
            }
        }
    }
    return cudaSuccess;
}

struct MxLayout {
    std::vector<int64_t> lo;
    size_t msg_stride = 0, keep_stride = 0, msgs = 0, keeps = 0, finals = 0, total = 0;
    Schedule S;
};

bool mx_layout(int32_t N, int32_t butterfly, int64_t n_blk, MxLayout &X)
{
    if (N < 1 || N > 65535 || n_blk < 1 || n_blk >= kMxMaxBlk) return false;
    if (!build_schedule(N, butterfly != 0, X.S)) return false;
    X.lo.resize((size_t)N + 1);
    for (int32_t c = 0; c <= N; ++c) X.lo[c] = (int64_t)c * n_blk / N;
    size_t mmax = 16, kmax = 16;
    for (const SchedStep &st : X.S.steps)
        for (const SchedHop &h : st.hops) {
            const int64_t ns = X.lo[h.send.b] - X.lo[h.send.a], nk = X.lo[h.keep.b] - X.lo[h.keep.a];
            mmax = std::max(mmax, (size_t)(pad16(ns) + kMxBlk * ns));
            kmax = std::max(kmax, (size_t)(nk * kMxBlk) * sizeof(float));
        }
    auto r256 = [](size_t b) { return (b + 255) / 256 * 256; };
    X.msg_stride = r256(mmax);
    X.keep_stride = butterfly ? r256(kmax) : 0;
    size_t o = 0;
    X.msgs = o;   o += 2 * (size_t)N * X.msg_stride;
    X.keeps = o;  o += 2 * (size_t)N * X.keep_stride;
    X.finals = o; o += butterfly ? (size_t)N * X.msg_stride : 0;
    X.total = o;
    return true;
}

}  // namespace
}  // namespace dq

using namespace dq;

extern "C" {

size_t dq_mx_message_bytes(int64_t n_blk)
{
    if (n_blk < 0 || n_blk >= kMxMaxBlk) return 0;
    return (size_t)(pad16(n_blk) + kMxBlk * n_blk);
}

dq_status dq_mx_quantize(const float *x, int64_t n_blk, uint8_t *msg, void *stream)
{
    if (n_blk < 0 || n_blk >= kMxMaxBlk) return DQ_ERR_INVALID_ARG;
    if (n_blk == 0) return DQ_OK;
    if (!x || !msg) return DQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(msg)) return DQ_ERR_ALIGNMENT;
    MxTask t;
    memset(&t, 0, sizeof(t));
    t.addend = x;
    t.out = msg;
    t.lo = 0;
    t.hi = n_blk;
    t.send_lo = 0;
    t.send_hi = n_blk;
    t.keep_lo = t.keep_hi = n_blk;
    t.out_pad = pad16(n_blk);
    return run_mx_hops({t}, false, true, static_cast<cudaStream_t>(stream), nullptr) == cudaSuccess ? DQ_OK
                                                                                                   : DQ_ERR_CUDA;
}

dq_status dq_mx_dequantize(const uint8_t *msg, int64_t n_blk, float *out, void *stream)
{
    if (n_blk < 0 || n_blk >= kMxMaxBlk) return DQ_ERR_INVALID_ARG;
    if (n_blk == 0) return DQ_OK;
    if (!msg || !out) return DQ_ERR_INVALID_ARG;
    if (!aligned16(msg) || !aligned16(out)) return DQ_ERR_ALIGNMENT;
    float *outs[1] = {out};
    return run_mx_decodes({MxChunk{msg, 0, n_blk}}, outs, 1, static_cast<cudaStream_t>(stream), nullptr) ==
                   cudaSuccess
               ? DQ_OK
               : DQ_ERR_CUDA;
}

size_t dq_mx_exchange_workspace_bytes(int32_t n_ranks, int32_t butterfly, int64_t n_blk)
{
    MxLayout X;
    return mx_layout(n_ranks, butterfly, n_blk, X) ? X.total : 0;
}

dq_status dq_mx_exchange(int32_t n_ranks, int32_t butterfly, const void *const *grads, int64_t n_blk, void *ws,
                         size_t ws_bytes, void *const *outs, const uint8_t **final_msgs, dq_launch_log *log,
                         void *stream)
{
    MxLayout X;
    if (!grads || !ws || !outs || !mx_layout(n_ranks, butterfly, n_blk, X)) return DQ_ERR_INVALID_ARG;
    if (ws_bytes < X.total) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    const int32_t N = n_ranks;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r] || !outs[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r]) || !aligned16(outs[r])) return DQ_ERR_ALIGNMENT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    auto msg = [&](int32_t r, int32_t par) {
        return par < 0 ? w + X.finals + (size_t)r * X.msg_stride : w + X.msgs + (size_t)(2 * r + par) * X.msg_stride;
    };
    auto keepb = [&](int32_t r, int32_t par) {
        return reinterpret_cast<float *>(w + X.keeps + (size_t)(2 * r + par) * X.keep_stride);
    };
    const std::vector<int64_t> &lo = X.lo;
    std::vector<MxTask> tasks;
    for (const SchedStep &step : X.S.steps) {
        tasks.clear();
        for (const SchedHop &h : step.hops) {
            MxTask t;
            memset(&t, 0, sizeof(t));
            const int64_t a = lo[h.in.a], b = lo[h.in.b];
            const int64_t sa = lo[h.send.a], sb = lo[h.send.b], ka = lo[h.keep.a], kb = lo[h.keep.b];
            t.in = h.in_rank < 0 ? nullptr : msg(h.in_rank, h.in_par);
            t.addend = h.add_par < 0 ? grads[h.rank] : (const void *)keepb(h.rank, h.add_par);
            t.out = msg(h.rank, h.out_par);
            t.keep = kb > ka ? keepb(h.rank, h.keep_par) : nullptr;
            t.lo = a;
            t.hi = b;
            t.send_lo = sb > sa ? sa : b;
            t.send_hi = sb > sa ? sb : b;
            t.keep_lo = kb > ka ? ka : b;
            t.keep_hi = kb > ka ? kb : b;
            t.in_pad = pad16(b - a);
            t.out_pad = pad16(sb - sa);
            tasks.push_back(t);
        }
        if (run_mx_hops(tasks, step.has_in, step.add_f32, st, log) != cudaSuccess) return DQ_ERR_CUDA;
    }
    std::vector<MxChunk> chunks;
    for (int32_t c = 0; c < N; ++c) chunks.push_back(MxChunk{msg(X.S.fin_rank[c], X.S.fin_par[c]), lo[c], lo[c + 1]});
    std::vector<float *> o((size_t)N);
    for (int32_t r = 0; r < N; ++r) o[r] = static_cast<float *>(outs[r]);
    if (run_mx_decodes(chunks, o.data(), N, st, log) != cudaSuccess) return DQ_ERR_CUDA;
    if (final_msgs)
        for (int32_t c = 0; c < N; ++c) final_msgs[c] = chunks[c].msg;
    return DQ_OK;
}

}  // extern "C"
