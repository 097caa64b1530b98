// dq_codec.cu -- per-super-group statistics and the simulated metadata
// all-reduce.
//
// Work mapping: one warp per super-group, lane l owning coordinates
// 8l .. 8l+7 (16 bytes of bf16, one 128-bit load); lanes 2g and 2g+1 hold
// group g.
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
    constexpr int kAhead = 4;   // super-groups loaded before any is reduced
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    for (int64_t jb = w0; jb < n_sg; jb += nw * kAhead) {
        uint4 v[kAhead];
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            const int64_t j = jb + a * nw;
            v[a] = j < n_sg ? __ldcs(reinterpret_cast<const uint4 *>(g + j * kSG) + lane) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            const int64_t j = jb + a * nw;
            const uint32_t w[4] = {v[a].x, v[a].y, v[a].z, v[a].w};
            float x[8], y[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[2 * k] = bf16_lo(w[k]);
                x[2 * k + 1] = bf16_hi(w[k]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(x[i], x[i]);
            const float s = lane_tree8(x);
            const float q = lane_tree8(y);
            if (lane == 0 && j < n_sg) {
                mean[j] = __fmul_rn(s, 0.00390625f);
                sq[j] = q;
            }
        }
    }
}

// Metadata all-reduce: M_j and F_j summed over ranks 0..N-1 in order, and
// the mean every worker subtracts, mu_j = fl(M_j / N).
__global__ void __launch_bounds__(256) stats_reduce_kernel(const float *__restrict__ mean_all,
                                                           const float *__restrict__ sq_all, int32_t n,
                                                           int64_t n_sg, float *__restrict__ M,
                                                           float *__restrict__ F, float *__restrict__ mu)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const float nf = (float)n;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n_sg; j += stride) {
        float m = mean_all[j], f = sq_all[j];
        for (int32_t w = 1; w < n; ++w) {
            m = __fadd_rn(m, mean_all[(int64_t)w * n_sg + j]);
            f = __fadd_rn(f, sq_all[(int64_t)w * n_sg + j]);
        }
        if (M) M[j] = m;
        F[j] = f;
        mu[j] = __fdiv_rn(m, nf);
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
                                float *M, float *F, float *mu, cudaStream_t st)
{
    int64_t blocks = (n_sg + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    blocks = blocks < 1 ? 1 : (blocks < cap ? blocks : cap);
    stats_reduce_kernel<<<(int)blocks, 256, 0, st>>>(mean_all, sq_all, n, n_sg, M, F, mu);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace dq
