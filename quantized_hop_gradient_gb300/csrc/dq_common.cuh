// dq_common.cuh -- shared definitions of the libdq CUDA kernels (sm_103a).
//
// Floating point: all codec arithmetic uses explicitly rounded fp32
// intrinsics (__fadd_rn, __fsub_rn, __fmul_rn, __fdiv_rn, __frcp_rn) and the
// library is built with -fmad=false, so no multiply-add is contracted and
// every result is the correctly rounded binary32 of each step.  That makes
// codes, scales and decoded values reproducible bit for bit by any IEEE
// implementation that performs the same steps.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dq.h"

namespace dq {

constexpr int kSG = 256;        // coordinates per super-group
constexpr int kGroup = 16;      // coordinates per group (one UINT8 scale each)
constexpr int kLaneCoords = 8;  // one warp per super-group: 8 coordinates per lane
constexpr unsigned kFull = 0xFFFFFFFFu;

// Bucket tables for the level search: bucket t of bitwidth b covers
// y in [t/H - 1, (t+1)/H - 1); kb is the largest level index with
// q_kb <= t/H - 1 and boundary = q_{kb+1} (+inf for the top level).
constexpr int kMaxH2 = 64, kMaxH4 = 128, kMaxH8 = 512;

struct BucketEntry {
    int32_t kb;
    float boundary;
};

// Level tables for one eps, built on the host.
// qg*[k] = {q_k, G_k}: the level and the reciprocal gap fl(1/fl(q_{k+1}-q_k));
// G of the top level is 0, and one sentinel entry {+inf, 0} follows it.
struct Tables {
    float2 qg2[5];
    float2 qg4[17];
    float2 qg8[257];
    int32_t H2, H4, H8, pad_;
    BucketEntry bk2[2 * kMaxH2 + 1];
    BucketEntry bk4[2 * kMaxH4 + 1];
    BucketEntry bk8[2 * kMaxH8 + 1];
};

// One message (the bytes that carry a range of reordered super-groups).
struct MsgView {
    uint8_t *base;
    int64_t c, n2, n4;                    // SGs in range; of them 2-bit, 4-bit
    int64_t off_u, off_c2, off_c4, off_c8;
};

// One fused hop (one rank's dq_compress or dq_dar) inside a batched launch.
struct HopTask {
    MsgView in;                 // incoming message (unused for compress)
    MsgView out;                // message for the send range
    const void *addend;         // bf16 gradient (by perm) or fp32 rows (j - in_lo)
    float *keep_out;            // fp32 rows (j - keep_lo)
    int64_t in_lo;
    int64_t send_lo, send_hi, keep_lo, keep_hi;
    int64_t sg_begin;           // first batched super-group index of this task
    uint32_t stage_word;        // generator counter word 1: hop | rank << 16, 0 if correlated
    uint32_t corr_off;          // floor(rank * 2^16 / N) if correlated, else 0
};

constexpr int kMaxTasks = 32;

struct HopParams {
    Tables tab;
    HopTask task[kMaxTasks];
    int32_t n_tasks;
    int32_t n_ranks;
    int64_t total_sg;
    int64_t end2, end4;
    const float *M;
    const int32_t *perm;
    uint32_t key0, key1;        // seed
    uint32_t round0, round1;    // round
};

// One chunk decoded by the final decode.
struct DecodeTask {
    MsgView msg;
    int64_t lo;
    int64_t sg_begin;
};

struct DecodeParams {
    Tables tab;
    DecodeTask task[kMaxTasks];
    int32_t n_tasks;
    int32_t n_ranks;
    int64_t total_sg;
    int64_t end2, end4;
    const float *M;
    const int32_t *perm;
    void *out;
    int32_t out_is_bf16;
};

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC 2011): ten rounds; each multiplies words
// 0 and 2 by the Philox constants (full 64-bit products), xors the high
// halves into words 1 and 3 with the round key, and bumps the key by the
// Weyl constants between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1)
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += W0; k1 += W1; }
        const uint32_t hi0 = __umulhi(M0, c[0]), lo0 = M0 * c[0];
        const uint32_t hi1 = __umulhi(M1, c[2]), lo1 = M1 * c[2];
        const uint32_t n0 = hi1 ^ c[1] ^ k0;
        const uint32_t n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

// bf16 pair (low half = first element) -> two fp32, exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Copy a POD struct from parameter space to shared memory with the whole block.
template <typename T>
__device__ __forceinline__ void block_copy(T *dst, const T *src)
{
    static_assert(sizeof(T) % 16 == 0, "16-byte multiple");
    const int4 *s = reinterpret_cast<const int4 *>(src);
    int4 *d = reinterpret_cast<int4 *>(dst);
    for (int i = threadIdx.x; i < (int)(sizeof(T) / 16); i += blockDim.x) d[i] = s[i];
}

}  // namespace dq
