// dq_codec.cu -- per-super-group statistics and the simulated metadata
// all-reduce.
//
// Work mapping of the statistics: half a warp per super-group, one group of
// 16 coordinates per lane.
#include "dq_common.cuh"
#include "dq_internal.h"

namespace dq {

// ---------------------------------------------------------------------------
// Statistics: per super-group sum and sum of squares over the raw bf16
// values, fp32, fixed tree.  Tree within a group: a[i] += a[i+h] for
// h = 8, 4, 2, 1; then the 16 group partials by the same tree.  Mapping:
// half a warp per super-group, lane l of the half owning group l (two
// 128-bit loads of 8 bf16), so the group tree stays in the lane and the tree
// over groups is four xor shuffles (h = 8, 4, 2, 1 lanes apart) per sum.
// fp32 addition is commutative, so the lanes on both sides of a shuffle
// compute the same value.  mean = sum * 2^-8.
// ---------------------------------------------------------------------------
constexpr int kStatsAhead = 8;   // pairs of super-groups a warp loads before it reduces any

__device__ __forceinline__ float group_tree16(float (&a)[16])
{
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) a[i] = __fadd_rn(a[i], a[i + h]);
    return a[0];
}

__device__ __forceinline__ float half_tree16(float v)
{
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, h));
    return v;
}

// Pairs of super-groups of one rank: super-groups 2p, 2p+1 of gradient g.
__device__ __forceinline__ void stats_pairs(const uint16_t *__restrict__ g, int64_t n_sg, float *__restrict__ mean,
                                            float *__restrict__ sq, int64_t pb, int64_t stride, int lane)
{
    constexpr int kAhead = kStatsAhead;
    const int half = lane >> 4, hl = lane & 15;
    uint4 v[kAhead][2];
#pragma unroll
    for (int a = 0; a < kAhead; ++a) {
        const int64_t j = 2 * (pb + a * stride) + half;
        if (j < n_sg) {
            const uint4 *src = reinterpret_cast<const uint4 *>(g + j * kSG + hl * 16);
            v[a][0] = __ldg(src);
            v[a][1] = __ldg(src + 1);
        } else {
            v[a][0] = v[a][1] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int a = 0; a < kAhead; ++a) {
        const int64_t j = 2 * (pb + a * stride) + half;
        const uint32_t w[8] = {v[a][0].x, v[a][0].y, v[a][0].z, v[a][0].w,
                               v[a][1].x, v[a][1].y, v[a][1].z, v[a][1].w};
        float x[16], y[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            x[2 * k] = bf16_lo(w[k]);
            x[2 * k + 1] = bf16_hi(w[k]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(x[i], x[i]);
        const float s = half_tree16(group_tree16(x));
        const float q = half_tree16(group_tree16(y));
        if (hl == 0 && j < n_sg) {
            mean[j] = __fmul_rn(s, 0.00390625f);
            sq[j] = q;
        }
    }
}

// Both kernels run flat: each warp reduces one block of kStatsAhead pairs
// and exits (short-lived blocks stream from HBM faster than a persistent
// grid-stride loop).
__global__ void __launch_bounds__(256) stats_kernel(const uint16_t *__restrict__ g, int64_t n_sg,
                                                    float *__restrict__ mean, float *__restrict__ sq)
{
    const int lane = threadIdx.x & 31;
    const int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_pairs = (n_sg + 1) >> 1;
    if (b * kStatsAhead < n_pairs) stats_pairs(g, n_sg, mean, sq, b * kStatsAhead, 1, lane);
}

// Several ranks: warp-blocks of pairs are numbered rank by rank.
__global__ void __launch_bounds__(256) stats_batched_kernel(const __grid_constant__ StatsParams S)
{
    const int lane = threadIdx.x & 31;
    const int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_pairs = (S.n_sg + 1) >> 1;
    const int64_t per_rank = (n_pairs + kStatsAhead - 1) / kStatsAhead;   // blocks of kStatsAhead pairs per rank
    if (b >= per_rank * S.n_ranks) return;
    const int r = (int)(b / per_rank);
    const int64_t pb = (b - (int64_t)r * per_rank) * kStatsAhead;
    stats_pairs(S.g[r], S.n_sg, S.mean_all + (int64_t)r * S.n_sg, S.sq_all + (int64_t)r * S.n_sg, pb, 1, lane);
}

// Metadata all-reduce: M_j and F_j summed over ranks 0..N-1 in order, and
// the mean every worker subtracts, mu_j = fl(M_j / N).  `nonfinite`
// (optional) is set to 1 when some M_j or F_j is not finite: a NaN or
// infinite gradient value, or squares or sums beyond the fp32 range, which
// the allocation cannot take.
__global__ void __launch_bounds__(256) stats_reduce_kernel(const float *__restrict__ mean_all,
                                                           const float *__restrict__ sq_all, int32_t n,
                                                           int64_t n_sg, float *__restrict__ M,
                                                           float *__restrict__ F, float *__restrict__ mu,
                                                           int32_t *__restrict__ nonfinite)
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
        if (nonfinite && !(isfinite(m) && isfinite(f))) atomicOr(nonfinite, 1);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
static unsigned flat_grid(int64_t work_warps)
{
    const int64_t blocks = (work_warps + 7) / 8;
    return (unsigned)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_stats(const uint16_t *g, int64_t n_sg, float *mean, float *sq, cudaStream_t st)
{
    const int64_t n_pairs = (n_sg + 1) >> 1;
    stats_kernel<<<flat_grid((n_pairs + kStatsAhead - 1) / kStatsAhead), 256, 0, st>>>(g, n_sg, mean, sq);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_stats_batched(const StatsParams &S, cudaStream_t st)
{
    const int64_t n_pairs = (S.n_sg + 1) >> 1;
    stats_batched_kernel<<<flat_grid((n_pairs + kStatsAhead - 1) / kStatsAhead * S.n_ranks), 256, 0, st>>>(S);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_stats_reduce(const float *mean_all, const float *sq_all, int32_t n, int64_t n_sg,
                                float *M, float *F, float *mu, cudaStream_t st, int32_t *nonfinite)
{
    int64_t blocks = (n_sg + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    blocks = blocks < 1 ? 1 : (blocks < cap ? blocks : cap);
    stats_reduce_kernel<<<(int)blocks, 256, 0, st>>>(mean_all, sq_all, n, n_sg, M, F, mu, nonfinite);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace dq
