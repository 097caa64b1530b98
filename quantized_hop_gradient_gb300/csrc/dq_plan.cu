// dq_plan.cu -- bitwidth allocation and reordering kernels.
//
// Allocation.  With T = T_{2,4}, super-group j gets 8 bits when
// 17 F_j >= 512 T, 4 bits when F_j >= T, else 2.  For non-negative fp32 the
// order of values is the order of bit patterns, and for fp32 T
//   F >= T        <=>  bits(T) <= key4 = bits(F)
//   17 F >= 512 T <=>  bits(T) <= key8 = bits(rd(F * 17/512))
// (17/512 is exact in fp32, so one multiply rounded toward -inf gives the
// largest fp32 not above 17F/512).  The code bits beyond 2 per super-group
// are W(t) = 2 #{key4 >= t} + 4 #{key8 >= t}, non-increasing in t.  The
// smallest t with W(t) <= R = floor(B J) - 2J is v + 1, where v is the
// largest key at which the weight of keys >= v first exceeds R: a weighted
// radix select over the 2J keys, three passes of 11-, 11- and 10-bit digits
// from the top.  Each pass is one launch: every block adds its histogram to
// a global one, and the block that arrives last picks the digit (no block
// waits for another).
//
// Reordering.  A stable counting sort of the super-groups by bitwidth
// (2, 4, 8): per-tile counts, one scan over tiles, then a stable scatter.
// In the planning chain the bitwidths and the per-tile counts come from one
// launch whose last block also scans the tiles.
#include <mutex>

#include "dq_common.cuh"
#include "dq_internal.h"

namespace dq {

namespace {

constexpr int kAllocThreads = 256;
constexpr int kTile = kReorderTile;    // super-groups per reorder tile
constexpr int kTileThreads = 256;      // 8 super-groups per thread
constexpr int64_t kSmallPlanMaxSG = 16384;   // single-block plan: F in 64 KB of shared memory; above this the multi-kernel path is faster
constexpr int kBins = 2048;            // digits of up to 11 bits
constexpr int kSelectPasses = 3;

// first bit and width mask of the digit of each pass (bits 21..31, 10..20, 0..9)
__host__ __device__ constexpr int digit_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__host__ __device__ constexpr uint32_t digit_mask(int pass) { return pass == 2 ? 1023u : 2047u; }

struct AllocState {
    unsigned int hist[kBins];          // weights by digit of the current pass (zero between passes)
    long long above;                   // weight of keys above the current prefix
    long long R;                       // remaining budget of extra code bits
    uint32_t prefix;                   // determined high digits of v
    uint32_t t;                        // final threshold bit pattern
    int32_t all8;                      // 1: budget >= 8 bits, T = 0
    unsigned int arrived;              // blocks of the current launch that have finished their part
};
constexpr size_t kAllocStateBytes = (sizeof(AllocState) + 255) / 256 * 256;

__device__ __forceinline__ uint32_t key4_of(float F) { return __float_as_uint(F); }
__device__ __forceinline__ uint32_t key8_of(float F) { return __float_as_uint(__fmul_rd(F, 0.033203125f)); }

// Bin of a key in pass `pass` (kBins: not in this pass, its higher digits
// differ from the prefix found so far).
__device__ __forceinline__ uint32_t bin_of(uint32_t key, uint32_t prefix, int pass)
{
    const int shift = digit_shift(pass);
    if (pass > 0) {
        const int hs = digit_shift(pass - 1);
        if ((key >> hs) != (prefix >> hs)) return (uint32_t)kBins;
    }
    return (key >> shift) & digit_mask(pass);
}

__global__ void alloc_init_kernel(AllocState *st, long long R, int all8, int64_t *counts, int32_t *flag)
{
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) st->hist[i] = 0u;
    if (threadIdx.x == 0) {
        st->above = 0;
        st->R = R;
        st->prefix = 0u;
        st->t = 0u;
        st->all8 = all8;
        st->arrived = 0u;
        if (counts) counts[0] = counts[1] = counts[2] = 0;
        if (flag) *flag = 0;
    }
}

// Called by the last block of a pass: the largest digit d with
// above + sum_{d' >= d} hist[d'] > R becomes the pass's digit of v; the
// histogram and the arrival count are cleared for the next pass.  Thread i
// owns bins 8i .. 8i+7 (blockDim = kAllocThreads).
__device__ void select_digit(AllocState *st, int pass)
{
    static_assert(kAllocThreads * 8 == kBins, "8 bins per thread");
    __shared__ long long warp_tot[kAllocThreads / 32];
    __shared__ int dstar;
    __shared__ long long dhigher;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    unsigned int h[8];
    long long loc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        h[i] = __ldcg(&st->hist[8 * tid + i]);
        loc += h[i];
    }
    // weight of the bins of this thread and every thread above it
    long long incl = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_down_sync(kFull, incl, off);
        if (lane + off < 32) incl += o;
    }
    if (lane == 0) warp_tot[wid] = incl;
    if (tid == 0) dstar = -1;
    __syncthreads();
    for (int w = wid + 1; w < kAllocThreads / 32; ++w) incl += warp_tot[w];
    const long long above = __ldcg(&st->above), R = __ldcg(&st->R);
    long long gt = incl - loc;   // weight of the bins above 8*tid + i
    int best = -1;
    long long best_gt = 0;
#pragma unroll
    for (int i = 7; i >= 0; --i) {
        if (best < 0 && above + gt + (long long)h[i] > R) {
            best = 8 * tid + i;
            best_gt = gt;
        }
        gt += h[i];
    }
    if (best >= 0) atomicMax(&dstar, best);
    __syncthreads();
    if (best >= 0 && best == dstar) dhigher = best_gt;
    if (tid == 0 && dstar < 0) dhigher = incl - (long long)h[0];   // no digit qualifies: d = 0 (cannot happen unless all8)
    __syncthreads();
    if (tid == 0) {
        const int d = dstar < 0 ? 0 : dstar;
        st->above = above + dhigher;
        const uint32_t prefix = __ldcg(&st->prefix) | ((uint32_t)d << digit_shift(pass));
        st->prefix = prefix;
        if (pass == kSelectPasses - 1) st->t = prefix + 1u;
        st->arrived = 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) st->hist[8 * tid + i] = 0u;
}

// One pass of the select: the weighted histogram (by the digit at `pass`) of
// the keys whose higher digits equal the prefix, added into the global one;
// the last block to finish picks the digit.  REDUCE (pass 0 of the planning
// chain): F is first computed from the ranks' per-super-group statistics,
// as the metadata all-reduce does (M_j, F_j summed over ranks 0..N-1 in
// order, mu_j = fl(M_j / N)), and written with M and mu; a non-finite M_j
// or F_j sets *nonfinite and, if given, the caller's *sticky flag (which
// collects the planning of many buckets).  hist = false (REDUCE only:
// budget >= 8 bits or a fixed bitwidth) skips the histogram.
template <bool REDUCE>
__global__ void __launch_bounds__(kAllocThreads) alloc_pass_kernel(const float *__restrict__ Fin, int64_t n,
                                                                   AllocState *st, int pass, bool hist,
                                                                   const float *__restrict__ mean_all,
                                                                   const float *__restrict__ sq_all, int32_t n_ranks,
                                                                   float *__restrict__ M, float *__restrict__ Fout,
                                                                   float *__restrict__ mu,
                                                                   int32_t *__restrict__ nonfinite,
                                                                   int32_t *__restrict__ sticky)
{
    __shared__ unsigned int h[kBins];
    __shared__ bool last;
    const int tid = threadIdx.x, lane = tid & 31;
    const bool do_hist = hist && !st->all8;
    if (do_hist)
        for (int i = tid; i < kBins; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    const uint32_t prefix = do_hist ? st->prefix : 0u;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // whole warps run every iteration (the match below needs all 32 lanes)
    const int64_t n_warp = (n + 31) & ~(int64_t)31;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + tid; j < n_warp; j += stride) {
        uint32_t b4 = (uint32_t)kBins, b8 = (uint32_t)kBins;
        if (j < n) {
            float f;
            if (REDUCE) {
                float m = mean_all[j];
                f = sq_all[j];
                int32_t w = 1;
                for (; w + 4 <= n_ranks; w += 4) {   // four ranks' loads in flight, then the sums in rank order
                    float a[4], c[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        a[k] = mean_all[(int64_t)(w + k) * n + j];
                        c[k] = sq_all[(int64_t)(w + k) * n + j];
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        m = __fadd_rn(m, a[k]);
                        f = __fadd_rn(f, c[k]);
                    }
                }
                for (; w < n_ranks; ++w) {
                    m = __fadd_rn(m, mean_all[(int64_t)w * n + j]);
                    f = __fadd_rn(f, sq_all[(int64_t)w * n + j]);
                }
                if (M) M[j] = m;
                Fout[j] = f;
                mu[j] = __fdiv_rn(m, (float)n_ranks);
                if (nonfinite && !(isfinite(m) && isfinite(f))) {
                    atomicOr(nonfinite, 1);
                    if (sticky) atomicOr(sticky, 1);
                }
            } else {
                f = __ldg(Fin + j);
            }
            if (do_hist) {
                b4 = bin_of(key4_of(f), prefix, pass);
                b8 = bin_of(key8_of(f), prefix, pass);
            }
        }
        if (do_hist) {   // the top digits are mostly the exponent: combine equal bins of a warp first
            const unsigned p4 = __match_any_sync(kFull, b4);
            if (b4 < (uint32_t)kBins && lane == __ffs(p4) - 1) atomicAdd(&h[b4], 2u * (unsigned)__popc(p4));
            const unsigned p8 = __match_any_sync(kFull, b8);
            if (b8 < (uint32_t)kBins && lane == __ffs(p8) - 1) atomicAdd(&h[b8], 4u * (unsigned)__popc(p8));
        }
    }
    if (!do_hist) return;
    __syncthreads();
    for (int i = tid; i < kBins; i += blockDim.x)
        if (h[i]) atomicAdd(&st->hist[i], h[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(&st->arrived, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    select_digit(st, pass);
}

// --------------------------------------------------------------------------- reorder
__device__ __forceinline__ int class_of(uint8_t bits) { return bits == 2 ? 0 : (bits == 4 ? 1 : 2); }

__global__ void __launch_bounds__(kTileThreads) reorder_count_kernel(const uint8_t *__restrict__ b, int64_t n,
                                                                     long long *tile_counts)
{
    __shared__ unsigned int c[3];
    if (threadIdx.x < 3) c[threadIdx.x] = 0u;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kTile;
    unsigned int l[3] = {0u, 0u, 0u};
    for (int i = threadIdx.x; i < kTile; i += blockDim.x) {
        const int64_t j = base + i;
        if (j < n) ++l[class_of(b[j])];
    }
    for (int k = 0; k < 3; ++k) atomicAdd(&c[k], l[k]);
    __syncthreads();
    if (threadIdx.x < 3) tile_counts[(int64_t)blockIdx.x * 4 + threadIdx.x] = c[threadIdx.x];
}

// Exclusive scan over tiles, per class, plus the class bases: replaces
// tile_counts[tile*4+c] by the first output position of (tile, class) and
// returns the class totals.  Any block size that is a multiple of 32 (up to
// 1024); the whole block calls it.
__device__ void scan_tiles(long long *tile_counts, int64_t n_tiles, long long (&tot)[3])
{
    __shared__ long long s_tot[3];
    __shared__ long long warp_sum[32][3];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = (int)(blockDim.x >> 5);
    // pass 1: class totals
    long long part[3] = {0, 0, 0};
    for (int64_t i = tid; i < n_tiles; i += blockDim.x)
        for (int k = 0; k < 3; ++k) part[k] += __ldcg(&tile_counts[i * 4 + k]);
    for (int k = 0; k < 3; ++k)
        for (int m = 16; m >= 1; m >>= 1) part[k] += __shfl_xor_sync(kFull, part[k], m);
    if (lane == 0)
        for (int k = 0; k < 3; ++k) warp_sum[wid][k] = part[k];
    __syncthreads();
    if (tid == 0) {
        for (int k = 0; k < 3; ++k) {
            long long s = 0;
            for (int w = 0; w < nw; ++w) s += warp_sum[w][k];
            s_tot[k] = s;
        }
    }
    __syncthreads();
    for (int k = 0; k < 3; ++k) tot[k] = s_tot[k];
    long long carry[3] = {0, tot[0], tot[0] + tot[1]};
    // pass 2: chunked exclusive scan
    for (int64_t base = 0; base < n_tiles; base += blockDim.x) {
        const int64_t i = base + tid;
        long long v[3];
        for (int k = 0; k < 3; ++k) v[k] = i < n_tiles ? __ldcg(&tile_counts[i * 4 + k]) : 0;
        long long inc[3] = {v[0], v[1], v[2]};
        for (int off = 1; off < 32; off <<= 1)
            for (int k = 0; k < 3; ++k) {
                const long long o = __shfl_up_sync(kFull, inc[k], off);
                if (lane >= off) inc[k] += o;
            }
        __syncthreads();   // the previous chunk's reads of warp_sum are done
        if (lane == 31)
            for (int k = 0; k < 3; ++k) warp_sum[wid][k] = inc[k];
        __syncthreads();
        long long wpre[3] = {0, 0, 0}, chunk[3] = {0, 0, 0};
        for (int w = 0; w < nw; ++w)
            for (int k = 0; k < 3; ++k) {
                if (w < wid) wpre[k] += warp_sum[w][k];
                chunk[k] += warp_sum[w][k];
            }
        if (i < n_tiles)
            for (int k = 0; k < 3; ++k) tile_counts[i * 4 + k] = carry[k] + wpre[k] + inc[k] - v[k];
        for (int k = 0; k < 3; ++k) carry[k] += chunk[k];
    }
}

__global__ void __launch_bounds__(1024) reorder_scan_kernel(long long *tile_counts, int64_t n_tiles)
{
    long long tot[3];
    scan_tiles(tile_counts, n_tiles, tot);
}

// Bitwidths of one tile of super-groups (from F and the threshold, or the
// fixed width) and the tile's count per class; the block that finishes last
// scans the tiles (the first output position of each tile and class, as
// reorder_scan_kernel) and writes the class totals and T.
__global__ void __launch_bounds__(kTileThreads) tile_assign_kernel(const float *__restrict__ F, int64_t n,
                                                                   AllocState *st, int32_t fixed_bits,
                                                                   uint8_t *__restrict__ b, long long *tile_counts,
                                                                   int64_t *counts, float *T)
{
    constexpr int kPer = kTile / kTileThreads;  // 8 consecutive super-groups per thread
    __shared__ unsigned long long warp_tot[kTileThreads / 32];
    __shared__ bool last;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t t = st->all8 ? 0u : st->t;
    const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)tid * kPer;
    unsigned long long mine = 0ull;  // packed counts: class k in bits [21k, 21k+21)
    for (int i = 0; i < kPer; ++i) {
        const int64_t j = base + i;
        if (j < n) {
            uint8_t bits;
            if (fixed_bits) {
                bits = (uint8_t)fixed_bits;
            } else {
                const float f = __ldg(F + j);
                bits = key8_of(f) >= t ? 8 : (key4_of(f) >= t ? 4 : 2);
            }
            b[j] = bits;
            mine += 1ull << (21 * class_of(bits));
        }
    }
    for (int off = 16; off >= 1; off >>= 1) mine += __shfl_xor_sync(kFull, mine, off);
    if (lane == 0) warp_tot[wid] = mine;
    __syncthreads();
    if (tid == 0) {
        unsigned long long all = 0ull;
        for (int w = 0; w < kTileThreads / 32; ++w) all += warp_tot[w];
        for (int k = 0; k < 3; ++k) tile_counts[(int64_t)blockIdx.x * 4 + k] = (long long)((all >> (21 * k)) & 0x1FFFFFull);
        __threadfence();
        last = atomicAdd(&st->arrived, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    long long tot[3];
    scan_tiles(tile_counts, (int64_t)gridDim.x, tot);
    if (tid == 0) {
        counts[0] = tot[0];
        counts[1] = tot[1];
        counts[2] = tot[2];
        *T = __uint_as_float(t);
        st->arrived = 0u;
    }
}

__global__ void __launch_bounds__(kTileThreads) reorder_scatter_kernel(const uint8_t *__restrict__ b, int64_t n,
                                                                       const long long *tile_off,
                                                                       int32_t *__restrict__ perm)
{
    constexpr int kPer = kTile / kTileThreads;  // 8 consecutive super-groups per thread
    __shared__ unsigned long long warp_tot[kTileThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)tid * kPer;
    uint8_t cls[kPer];
    unsigned long long mine = 0ull;  // packed counts: class k in bits [21k, 21k+21)
    for (int i = 0; i < kPer; ++i) {
        const int64_t j = base + i;
        cls[i] = j < n ? (uint8_t)class_of(b[j]) : (uint8_t)3;
        if (cls[i] < 3) mine += 1ull << (21 * cls[i]);
    }
    unsigned long long inc = mine;
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(kFull, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    unsigned long long pre = inc - mine;
    for (int w = 0; w < wid; ++w) pre += warp_tot[w];
    long long pos[3];
    for (int k = 0; k < 3; ++k)
        pos[k] = tile_off[(int64_t)blockIdx.x * 4 + k] + (long long)((pre >> (21 * k)) & 0x1FFFFFull);
    for (int i = 0; i < kPer; ++i) {
        if (cls[i] < 3) perm[pos[cls[i]]++] = (int32_t)(base + i);
    }
}

// --------------------------------------------------------------------------- small problems
// Allocation and reorder in one block, for up to kSmallPlanMaxSG super-groups
// (F held in shared memory): a weighted radix select (four passes of 8-bit
// digits, the threshold the chain above finds) and the same stable
// partition, without the chain's launches.  Histogram
// updates are combined per warp (__match_any_sync) before the shared
// atomic, since the top digit of F is mostly its exponent and few bins
// take most keys.  fixed_bits != 0 gives every super-group that width.
constexpr int kSmallPlanThreads = 1024;

__global__ void __launch_bounds__(kSmallPlanThreads) plan_small_kernel(const float *__restrict__ F, int32_t n,
                                                                       long long R, int32_t all8, int32_t fixed_bits,
                                                                       uint8_t *__restrict__ b, float *T,
                                                                       int64_t *counts, int32_t *__restrict__ perm,
                                                                       const int32_t *nonfinite, int32_t *sticky)
{
    extern __shared__ float sF[];
    __shared__ unsigned int hist[256];
    __shared__ int s_d;
    __shared__ unsigned long long s_higher;
    __shared__ unsigned long long warp_tot[kSmallPlanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nth = blockDim.x;
    for (int j = tid; j < n; j += nth) sF[j] = F[j];
    __syncthreads();

    uint32_t t = 0u;
    if (!fixed_bits && !all8) {
        uint32_t prefix = 0u;
        long long above = 0;
        for (int pass = 0; pass < 4; ++pass) {
            for (int i = tid; i < 256; i += nth) hist[i] = 0u;
            __syncthreads();
            const int shift = 24 - 8 * pass;
            for (int base = wid * 32; base < n; base += nth) {
                const int j = base + lane;
                uint32_t bin4 = 256u, bin8 = 256u;   // 256: no bin
                if (j < n) {
                    const float f = sF[j];
                    const uint32_t k4 = key4_of(f), k8 = key8_of(f);
                    if (pass == 0 || (k4 >> (shift + 8)) == (prefix >> (shift + 8))) bin4 = (k4 >> shift) & 255u;
                    if (pass == 0 || (k8 >> (shift + 8)) == (prefix >> (shift + 8))) bin8 = (k8 >> shift) & 255u;
                }
                const unsigned p4 = __match_any_sync(kFull, bin4);
                if (bin4 < 256u && lane == __ffs(p4) - 1) atomicAdd(&hist[bin4], 2u * (unsigned)__popc(p4));
                const unsigned p8 = __match_any_sync(kFull, bin8);
                if (bin8 < 256u && lane == __ffs(p8) - 1) atomicAdd(&hist[bin8], 4u * (unsigned)__popc(p8));
            }
            __syncthreads();
            if (wid == 0) {   // the largest digit d with above + sum_{d' >= d} hist[d'] > R
                unsigned long long h[8], loc = 0ull;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    h[i] = hist[8 * lane + i];
                    loc += h[i];
                }
                unsigned long long incl = loc;   // weight of lanes >= this lane
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const unsigned long long o = __shfl_down_sync(kFull, incl, off);
                    if (lane + off < 32) incl += o;
                }
                unsigned long long gt = incl - loc;   // weight of the bins above 8*lane + i
                int best = -1;
                unsigned long long best_gt = 0ull;
#pragma unroll
                for (int i = 7; i >= 0; --i) {
                    if (best < 0 && above + (long long)(gt + h[i]) > R) {
                        best = 8 * lane + i;
                        best_gt = gt;
                    }
                    gt += h[i];
                }
                const unsigned q = __ballot_sync(kFull, best >= 0);
                const int src = q ? 31 - __clz((int)q) : 0;
                const int d = __shfl_sync(kFull, best, src);
                const unsigned long long dgt = __shfl_sync(kFull, best_gt, src);
                const unsigned long long total = __shfl_sync(kFull, incl, 0);
                const unsigned long long h0 = __shfl_sync(kFull, h[0], 0);
                if (lane == 0) {
                    s_d = q ? d : 0;
                    s_higher = q ? dgt : total - h0;
                }
            }
            __syncthreads();
            prefix |= (uint32_t)s_d << shift;
            above += (long long)s_higher;
            __syncthreads();
        }
        t = prefix + 1u;
    }

    // assign and count: thread tid takes a contiguous run of super-groups
    const int per = (n + nth - 1) / nth;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    unsigned long long mine = 0ull;   // packed counts: class k in bits [21k, 21k+21)
    for (int j = lo; j < hi; ++j) {
        const float f = sF[j];
        uint8_t bits;
        if (fixed_bits) bits = (uint8_t)fixed_bits;
        else bits = key8_of(f) >= t ? 8 : (key4_of(f) >= t ? 4 : 2);
        b[j] = bits;
        mine += 1ull << (21 * class_of(bits));
    }
    unsigned long long inc = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(kFull, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    unsigned long long pre = inc - mine, all = 0ull;
    for (int w = 0; w < nth / 32; ++w) {
        if (w < wid) pre += warp_tot[w];
        all += warp_tot[w];
    }
    const long long tot0 = (long long)(all & 0x1FFFFFull), tot1 = (long long)((all >> 21) & 0x1FFFFFull),
                    tot2 = (long long)((all >> 42) & 0x1FFFFFull);
    long long pos[3] = {(long long)(pre & 0x1FFFFFull), tot0 + (long long)((pre >> 21) & 0x1FFFFFull),
                        tot0 + tot1 + (long long)((pre >> 42) & 0x1FFFFFull)};
    for (int j = lo; j < hi; ++j) perm[pos[class_of(b[j])]++] = j;
    if (tid == 0) {
        counts[0] = tot0;
        counts[1] = tot1;
        counts[2] = tot2;
        *T = __uint_as_float(t);
        if (sticky && nonfinite && *nonfinite) atomicOr(sticky, 1);   // the reduce before this launch set it
    }
}

}  // namespace

size_t reorder_scratch_bytes(int64_t n_sg)
{
    const int64_t n_tiles = (n_sg + kTile - 1) / kTile;
    return (size_t)(n_tiles > 0 ? n_tiles : 1) * 4 * sizeof(long long);
}

// [allocation state][per-tile counts]
size_t plan_scratch_bytes(int64_t n_sg) { return kAllocStateBytes + (reorder_scratch_bytes(n_sg) + 255) / 256 * 256; }

static int alloc_blocks(int64_t n_sg)
{
    // about two super-groups per thread, at most eight blocks per SM
    int64_t blocks = (n_sg + 2 * kAllocThreads - 1) / (2 * kAllocThreads);
    const int64_t cap = (int64_t)sm_count() * 8;
    return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

cudaError_t launch_allocate(const float *F, int64_t n_sg, int64_t cap_bits, uint8_t *b, float *T,
                            int64_t *counts, void *ws, cudaStream_t st)
{
    AllocState *s = static_cast<AllocState *>(ws);
    long long *tiles = reinterpret_cast<long long *>(static_cast<uint8_t *>(ws) + kAllocStateBytes);
    const long long R = (long long)(cap_bits - 2 * n_sg);
    const int all8 = R >= 6 * (long long)n_sg ? 1 : 0;
    alloc_init_kernel<<<1, 256, 0, st>>>(s, R, all8, counts, nullptr);
    if (!all8) {
        const int blocks = alloc_blocks(n_sg);
        for (int pass = 0; pass < kSelectPasses; ++pass)
            alloc_pass_kernel<false><<<blocks, kAllocThreads, 0, st>>>(F, n_sg, s, pass, true, nullptr, nullptr, 0,
                                                                       nullptr, nullptr, nullptr, nullptr, nullptr);
    }
    const int64_t n_tiles = (n_sg + kTile - 1) / kTile;
    tile_assign_kernel<<<(unsigned)n_tiles, kTileThreads, 0, st>>>(F, n_sg, s, 0, b, tiles, counts, T);
    note_launches(all8 ? 2 : 2 + kSelectPasses);
    return cudaGetLastError();
}

cudaError_t launch_reorder(const uint8_t *b, int64_t n_sg, int32_t *perm, void *ws, cudaStream_t st)
{
    long long *tiles = static_cast<long long *>(ws);
    const int64_t n_tiles = (n_sg + kTile - 1) / kTile;
    reorder_count_kernel<<<(int)n_tiles, kTileThreads, 0, st>>>(b, n_sg, tiles);
    reorder_scan_kernel<<<1, 1024, 0, st>>>(tiles, n_tiles);
    reorder_scatter_kernel<<<(int)n_tiles, kTileThreads, 0, st>>>(b, n_sg, tiles, perm);
    note_launches(3);
    return cudaGetLastError();
}

cudaError_t launch_plan_chain(const float *mean_all, const float *sq_all, int32_t n_ranks, int64_t n_sg,
                              int64_t cap_bits, int32_t fixed_bits, float *M, float *F, float *mu,
                              int32_t *nonfinite, uint8_t *b, float *T, int64_t *counts, int32_t *perm, void *ws,
                              cudaStream_t st, int32_t *sticky)
{
    AllocState *s = static_cast<AllocState *>(ws);
    long long *tiles = reinterpret_cast<long long *>(static_cast<uint8_t *>(ws) + kAllocStateBytes);
    const long long R = (long long)(cap_bits - 2 * n_sg);
    const int all8 = (fixed_bits || R >= 6 * (long long)n_sg) ? 1 : 0;
    const int blocks = alloc_blocks(n_sg);
    const int64_t n_tiles = (n_sg + kTile - 1) / kTile;
    alloc_init_kernel<<<1, 256, 0, st>>>(s, R, all8, counts, nonfinite);
    alloc_pass_kernel<true><<<blocks, kAllocThreads, 0, st>>>(nullptr, n_sg, s, 0, !all8, mean_all, sq_all, n_ranks,
                                                              M, F, mu, nonfinite, sticky);
    for (int pass = 1; pass < kSelectPasses && !all8; ++pass)
        alloc_pass_kernel<false><<<blocks, kAllocThreads, 0, st>>>(F, n_sg, s, pass, true, nullptr, nullptr, 0,
                                                                   nullptr, nullptr, nullptr, nullptr, nullptr);
    tile_assign_kernel<<<(unsigned)n_tiles, kTileThreads, 0, st>>>(F, n_sg, s, fixed_bits, b, tiles, counts, T);
    reorder_scatter_kernel<<<(unsigned)n_tiles, kTileThreads, 0, st>>>(b, n_sg, tiles, perm);
    note_launches(all8 ? 4 : 3 + kSelectPasses);
    return cudaGetLastError();
}

int64_t small_plan_max_sg() { return kSmallPlanMaxSG; }

cudaError_t launch_plan_small(const float *F, int64_t n_sg, int64_t cap_bits, int32_t fixed_bits, uint8_t *b,
                              float *T, int64_t *counts, int32_t *perm, cudaStream_t st, const int32_t *nonfinite,
                              int32_t *sticky)
{
    if (n_sg < 1 || n_sg > kSmallPlanMaxSG) return cudaErrorInvalidValue;
    const size_t smem = (size_t)n_sg * sizeof(float);
    // the attribute is set once per device; the lock makes first calls from
    // several host threads safe
    static std::mutex mu;
    static bool attr_set[128] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(plan_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)(kSmallPlanMaxSG * sizeof(float)));
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const long long R = (long long)(cap_bits - 2 * n_sg);
    const int all8 = R >= 6 * (long long)n_sg ? 1 : 0;
    plan_small_kernel<<<1, kSmallPlanThreads, smem, st>>>(F, (int32_t)n_sg, R, all8, fixed_bits, b, T, counts, perm,
                                                          nonfinite, sticky);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace dq
