// dq_common.cuh -- shared definitions of the libdq CUDA kernels (sm_103a).
//
// Floating point: all codec arithmetic uses explicitly rounded fp32
// operations: scalar __fmul_rn-style intrinsics (never contracted) and the
// packed .f32x2 instructions with .rn rounding; the library is built with
// -fmad=false.  ptxas does contract a packed multiply that feeds a packed
// add into one fused multiply-add even under .rn, so the kernels use a
// packed multiply only where its result feeds a compare or a multiply, and
// write every intended fused multiply-add explicitly.  Each result is then
// the correctly rounded binary32 of each step as written, reproducible bit
// for bit by any IEEE implementation that performs the same steps.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dq.h"

namespace dq {

constexpr int kSG = 256;        // coordinates per super-group
constexpr int kGroup = 16;      // coordinates per group (one UINT8 scale each)
constexpr int kUnit = 32;       // super-groups per work unit of a warp
constexpr unsigned kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// Level tables for one eps, built on the host and copied to shared memory.
//
// q*[k]   : the levels (decode and search).
// g*[k]   : G16_k = fl(1/fl(q_{k+1} - q_k)) * 2^16 (exact scaling), 0 for the
//           top level.
// bk*[i]  : level-search buckets.  For y in [-1, 1] and H a power of two,
//           r = rint(S*H*y) (ties to even; S = 8 for 2 and 8 bits, 128 for 4
//           bits) sits in the low bits of the bit pattern of
//           fl(S*H*y + 1.5*2^23); bucket b = floor(r / S) covers
//           [(b - 1/(2S))/H, (b + 1 - 1/(2S))/H).  The entry of bucket b sits
//           at index b & MASK, found as the bit pattern ANDed with a constant
//           -- so any bit pattern (NaN included) indexes inside the table.
//           It holds the next level above the bucket's lower edge
//           (boundary) and 4x the index kb of the largest level at or below
//           that edge (a byte offset into q* and g*).  The 4-bit table is
//           expanded in shared memory to 16 copies, one per lane of a
//           half-warp, so its lookups never meet in a bank.
// rcp[u]  : fl(1/u) for the UINT8 scales, rcp[0] = 0.
// mul*    : S*H of each bitwidth.
// ---------------------------------------------------------------------------
constexpr int kMask2 = 63, kMask4 = 127, kMask8 = 1023;   // tables of MASK+1 entries
constexpr int kSub2 = 8, kSub4 = 128, kSub8 = 128;        // S of each bitwidth
constexpr int kOff8 = 256;   // 8-bit buckets are stored at b + 256 (0 .. 512 for y in [-1, 1])
constexpr int kCopies4 = 16;                              // lane copies of the 4-bit table
// H is a power of two with 2H + 1 <= MASK + 1: at most 16, 32 and 256.
constexpr float kMagic = 12582912.0f;                     // 1.5 * 2^23

struct BucketEntry {
    float boundary;
    int32_t kb4;
};

struct Tables {
    BucketEntry bk8[kMask8 + 1];
    BucketEntry bk4[kMask4 + 1];
    BucketEntry bk2[kMask2 + 1];
    float q2[4], q4[16], q8[256];
    float g2[4], g4[16], g8[256];
    float rcp[256];
    float mul2, mul4, mul8;
    int32_t one_level;   // every bucket holds at most one level above its lower edge
};

// One message (the bytes that carry a range of reordered super-groups).
// UINT8 scales: E bytes at 0, u bytes at off_u (16 per SG); fp32 scales
// (ablation): 16 floats per SG at off_u = 0 and no E bytes.
struct MsgView {
    uint8_t *base;
    int64_t c, n2, n4;                    // SGs in range; of them 2-bit, 4-bit
    int64_t off_u, off_c2, off_c4, off_c8;
};

// One fused hop (one rank's dq_compress or dq_dar) inside a batched launch.
// Its super-groups [in_lo, in_hi) are cut into three bitwidth-pure segments,
// each split into work units of up to kUnit consecutive super-groups.
struct HopTask {
    MsgView in;                 // incoming message (unused for compress)
    MsgView out;                // message for the send range
    const void *addend;         // bf16 gradient (by perm) or fp32 rows (j - in_lo)
    float *keep_out;            // fp32 rows (j - keep_lo)
    int64_t in_lo;
    int64_t send_lo, send_hi, keep_lo, keep_hi;
    int64_t seg_lo[3], seg_hi[3];
    int64_t unit_begin[4];      // first global unit of each segment; [3] = end
    uint32_t stage_word;        // generator counter word 1
    uint32_t corr2;             // correlated offset in both 16-bit halves
};

constexpr int kMaxTasks = 32;

// Philox4x32-10 with key (seed low, seed high) and counter words 2, 3 =
// (round low, round high), prepared once per launch on the host: the round
// keys of rounds 1..9 (the key plus r times the Weyl constants) and round 0's
// part that involves no lane value (the product of word 2, its high half
// xored with the key).  The kernels then read every key straight from the
// launch parameters.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];    // round keys (k0[0], k1[0] = the seed)
    uint32_t a0;                // mulhi(M1, round low) ^ k0[0]
    uint32_t l1;                // M1 * round low
    uint32_t r1k;               // round high ^ k1[0]
};

struct HopParams {
    Tables tab;
    HopTask task[kMaxTasks];
    int32_t n_tasks;
    int32_t n_ranks;
    int64_t total_units;
    const float *mu;
    const int32_t *perm;
    PhiloxKeys ph;              // generator key schedule (seed, round)
    int32_t scale_fp32;         // group scales in fp32 (ablation) instead of UINT8
};

// One chunk decoded by the final decode (same unit structure).
struct DecodeTask {
    MsgView msg;
    void *out;                  // this task's output (a rank's full gradient buffer)
    int64_t lo;
    int64_t seg_lo[3], seg_hi[3];
    int64_t unit_begin[4];
};

constexpr int kMaxDecodeOuts = 16;

struct DecodeParams {
    Tables tab;
    DecodeTask task[kMaxTasks];
    int32_t n_tasks;
    int32_t n_ranks;
    int64_t total_units;
    const float *mu;
    const int32_t *perm;
    int32_t out_is_bf16;
    int32_t scale_fp32;
    // n_outs > 0: every task is decoded into all of outs[0..n_outs) (one
    // read of the message, n_outs writes) and the tasks' `out` is unused
    int32_t n_outs;
    void *outs[kMaxDecodeOuts];
};

// Statistics of several ranks in one launch.
constexpr int kMaxStatsRanks = 64;
struct StatsParams {
    const uint16_t *g[kMaxStatsRanks];
    int32_t n_ranks;
    int64_t n_sg;
    float *mean_all;   // n_ranks x n_sg
    float *sq_all;
};

// The whole ring exchange of one round in one cooperative launch: N hop
// steps and the final decode, separated by grid barriers.  Chunk c's
// message layout, units and range are the same at every step; only the
// message buffers and the quantizing rank rotate.
constexpr int kMaxFusedRanks = 64;
constexpr int32_t kDeviceBarrierTimeout = 1;   // status word: a barrier wait ran out

struct FusedRingParams {
    Tables tab;
    MsgView chunk[kMaxFusedRanks];             // message layout of chunk c (base unset)
    int64_t lo[kMaxFusedRanks + 1];            // chunk cuts (reordered super-groups)
    int64_t seg_lo[kMaxFusedRanks][3], seg_hi[kMaxFusedRanks][3];
    int64_t unit_begin[kMaxFusedRanks][4];     // first unit of each segment of chunk c; [3] = end
    const void *grads[kMaxFusedRanks];
    void *outs[kMaxFusedRanks];
    uint8_t *msgs;                             // two message buffers per rank, msg_stride apart
    int64_t msg_stride;
    int64_t units;                             // work units per phase
    int32_t n_ranks;
    int32_t correlated;
    const float *mu;
    const int32_t *perm;
    PhiloxKeys ph;                             // generator key schedule (seed, round)
    int32_t out_is_bf16;
    int32_t scale_fp32;
    unsigned int *barrier;                     // arrival counter, zero at launch
    int32_t *status;                           // zero at launch; kDeviceBarrierTimeout on a timeout
    long long timeout_cycles;                  // bound of every barrier wait (SM clock cycles)
};

// One launch of the pipelined ring exchange.  The work units of one step
// (numbered across the chunks as in FusedRingParams) are cut into n_parts
// parts of consecutive units, part p = [units*p/n_parts, units*(p+1)/n_parts);
// launch t runs every part p at step t - p (0 <= t - p < N) and decodes part
// t - N, so N + n_parts launches carry a round.  Warps take the launch's
// units in turn from a counter, one unit ahead of their work.  A part's units go through
// the steps in order, one launch apart; rank r's message of step s has its
// own buffer (r*N + s), so no launch overwrites bytes another part has still
// to read.
constexpr int kMaxWaveParts = 256;
constexpr int kDecodeSub = 4;   // decode pieces per work unit in the pipelined exchanges (8 super-groups each)
constexpr int kWaveCounterBytes = 2048;   // one unit counter per launch: (kMaxFusedRanks + kMaxWaveParts) x 4 bytes
static_assert((kMaxFusedRanks + kMaxWaveParts) * 4 <= kWaveCounterBytes, "wave counters");

struct WaveRingParams {
    Tables tab;
    MsgView chunk[kMaxFusedRanks];             // message layout of chunk c (base unset)
    int64_t lo[kMaxFusedRanks + 1];
    int64_t seg_lo[kMaxFusedRanks][3], seg_hi[kMaxFusedRanks][3];
    int64_t unit_begin[kMaxFusedRanks][4];
    const void *grads[kMaxFusedRanks];
    void *outs[kMaxFusedRanks];
    uint8_t *msgs;                             // N*N message buffers, msg_stride apart
    int64_t msg_stride;
    int64_t units;                             // work units of one step (all chunks)
    int64_t h_lo, h_hi;                        // this launch's hop units [h_lo, h_hi)
    int64_t d_lo, d_hi;                        // this launch's decode units [d_lo, d_hi)
    unsigned int *next;                        // this launch's unit counter, zero at launch
    int32_t n_parts;
    int32_t launch;                            // t
    int32_t n_ranks;
    int32_t correlated;
    const float *mu;
    const int32_t *perm;
    PhiloxKeys ph;
    int32_t out_is_bf16;
    int32_t scale_fp32;
};

// One launch of the bucket stream (dq_exchange_stream_step): a ring
// exchange pipelined across DDP buckets.  Launch t runs ring step t - b of
// every bucket b in flight and the final decode of bucket t - N, so N + 1
// buckets share each launch.  A bucket's chunk cuts and work units are
// derived on the device from the 2/4/8 counts its (asynchronous) planning
// left in device memory: the host never waits for a plan.
constexpr int kMaxStreamRanks = 8;

struct BucketSlot {
    const void *grads[kMaxStreamRanks];
    void *outs[kMaxStreamRanks];
    const int64_t *counts;      // device: n2, n4, n8 of the bucket's plan
    const float *mu;
    const int32_t *perm;
    uint8_t *msgs;              // N*N message buffers of the bucket, msg_stride apart
    int64_t msg_stride;
    PhiloxKeys ph;              // the bucket's generator round
    int32_t n_sg;
    int32_t step;               // 0 .. N-1: ring step; N: the final decode
    int32_t n_ranks;            // the launch's, so that a slot serves as
    int32_t out_is_bf16;        //   the kernels' parameter view
};

struct StreamRingParams {
    Tables tab;
    BucketSlot slot[kMaxStreamRanks + 1];
    int32_t n_slots;
    int32_t n_ranks;
    int32_t correlated;
    int32_t scale_fp32;
    unsigned int *next;         // task counter, zero at launch
};

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC 2011): ten rounds; each multiplies words
// 0 and 2 by the Philox constants (full 64-bit products), xors the high
// halves into words 1 and 3 with the round key, and bumps the key by the
// Weyl constants between rounds.  Here on the counter (c0, c1, round low,
// round high) with the key schedule K prepared on the host (PhiloxKeys).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x32_10_keyed(uint32_t c[4], uint32_t c0, uint32_t c1, const PhiloxKeys &K)
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    c[0] = K.a0 ^ c1;              // round 0
    c[1] = K.l1;
    c[2] = __umulhi(M0, c0) ^ K.r1k;
    c[3] = M0 * c0;
#pragma unroll
    for (int r = 1; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(M0, c[0]), lo0 = M0 * c[0];
        const uint32_t hi1 = __umulhi(M1, c[2]), lo1 = M1 * c[2];
        const uint32_t n0 = hi1 ^ c[1] ^ K.k0[r];
        const uint32_t n2 = hi0 ^ c[3] ^ K.k1[r];
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

// bf16 pair (low half = first element) -> two fp32, exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fl(float(b) - c) for the bf16 b in the low / high half of w: the
// mixed-precision subtract widens b exactly and rounds once.
__device__ __forceinline__ float bf16_lo_minus(uint32_t w, float c)
{
    float r;
    asm("{ .reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tsub.rn.f32.bf16 %0, l, %2; }" : "=f"(r) : "r"(w), "f"(c));
    return r;
}
__device__ __forceinline__ float bf16_hi_minus(uint32_t w, float c)
{
    float r;
    asm("{ .reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tsub.rn.f32.bf16 %0, h, %2; }" : "=f"(r) : "r"(w), "f"(c));
    return r;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (Blackwell .f32x2): two IEEE binary32 operations with the
// given rounding in one instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b)
{
    float2 r;
    asm("{ .reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d; }"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 f2_sub(float2 a, float2 b)
{
    float2 r;
    asm("{ .reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d; }"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// a * b + c with ONE rounding.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{ .reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d; }"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// ---------------------------------------------------------------------------
// cp.async staging (16-byte global -> shared copies, L2 only)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst_smem), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Copy a POD struct from parameter space to shared memory with the whole block.
template <typename T>
__device__ __forceinline__ void block_copy(T *dst, const T *src)
{
    static_assert(sizeof(T) % 16 == 0, "16-byte multiple");
    const int4 *s = reinterpret_cast<const int4 *>(src);
    int4 *d = reinterpret_cast<int4 *>(dst);
    for (int i = threadIdx.x; i < (int)(sizeof(T) / 16); i += blockDim.x) d[i] = s[i];
}

// Which task and bitwidth segment a work unit belongs to.
template <typename Task>
__device__ __forceinline__ void locate_unit(const Task *tasks, int n_tasks, int64_t u, int &ti, int &seg)
{
    ti = 0;
    while (ti + 1 < n_tasks && u >= tasks[ti + 1].unit_begin[0]) ++ti;
    seg = 0;
    while (seg < 2 && u >= tasks[ti].unit_begin[seg + 1]) ++seg;
}

}  // namespace dq
