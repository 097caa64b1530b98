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
// radix select over the 2J keys, four passes of 8-bit digits from the top.
//
// Reordering.  A stable counting sort of the super-groups by bitwidth
// (2, 4, 8): per-tile counts, one scan over tiles, then a stable scatter.
#include <mutex>

#include "dq_common.cuh"
#include "dq_internal.h"

namespace dq {

namespace {

constexpr int kAllocThreads = 256;
constexpr int kTile = kReorderTile;    // super-groups per reorder tile
constexpr int kTileThreads = 256;      // 8 super-groups per thread
constexpr int64_t kSmallPlanMaxSG = 16384;   // single-block plan: F in 64 KB of shared memory; above this the multi-kernel path is faster

struct AllocState {
    unsigned long long hist[256];
    long long above;                   // weight of keys above the current prefix
    long long R;                       // remaining budget of extra code bits
    uint32_t prefix;                   // determined high digits of v
    uint32_t t;                        // final threshold bit pattern
    int32_t all8;                      // 1: budget >= 8 bits, T = 0
    int32_t pad_;
};

__device__ __forceinline__ uint32_t key4_of(float F) { return __float_as_uint(F); }
__device__ __forceinline__ uint32_t key8_of(float F) { return __float_as_uint(__fmul_rd(F, 0.033203125f)); }

__global__ void alloc_init_kernel(AllocState *st, long long R, int all8, int64_t *counts)
{
    for (int i = threadIdx.x; i < 256; i += blockDim.x) st->hist[i] = 0ull;
    if (threadIdx.x == 0) {
        st->above = 0;
        st->R = R;
        st->prefix = 0u;
        st->t = 0u;
        st->all8 = all8;
        counts[0] = counts[1] = counts[2] = 0;
    }
}

// Histogram (by the digit at `pass`) of the weights of keys whose higher
// digits equal the prefix found so far.
__global__ void __launch_bounds__(kAllocThreads) alloc_hist_kernel(const float *__restrict__ F, int64_t n,
                                                                   AllocState *st, int pass)
{
    __shared__ unsigned int h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    if (!st->all8) {
        const uint32_t prefix = st->prefix;
        const int shift = 24 - 8 * pass;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
            const float f = __ldg(F + j);
            const uint32_t k4 = key4_of(f), k8 = key8_of(f);
            if (pass == 0 || (k4 >> (shift + 8)) == (prefix >> (shift + 8)))
                atomicAdd(&h[(k4 >> shift) & 255u], 2u);
            if (pass == 0 || (k8 >> (shift + 8)) == (prefix >> (shift + 8)))
                atomicAdd(&h[(k8 >> shift) & 255u], 4u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (h[i]) atomicAdd(&st->hist[i], (unsigned long long)h[i]);
}

// Picks the digit at `pass`: the largest d with above + sum_{d' >= d} h[d'] > R.
__global__ void __launch_bounds__(256) alloc_select_kernel(AllocState *st, int pass)
{
    __shared__ unsigned long long suf[256];
    __shared__ int dstar;
    const int d = threadIdx.x;
    if (st->all8) return;
    suf[d] = st->hist[d];
    if (d == 0) dstar = -1;
    __syncthreads();
    // suffix sums (Hillis-Steele over 256 entries)
    for (int off = 1; off < 256; off <<= 1) {
        const unsigned long long v = d + off < 256 ? suf[d + off] : 0ull;
        __syncthreads();
        suf[d] += v;
        __syncthreads();
    }
    const long long above = st->above, R = st->R;
    if (above + (long long)suf[d] > R) atomicMax(&dstar, d);
    __syncthreads();
    if (d == 0) {
        const int ds = dstar < 0 ? 0 : dstar;
        const unsigned long long higher = ds + 1 < 256 ? suf[ds + 1] : 0ull;
        st->above = above + (long long)higher;
        st->prefix |= (uint32_t)ds << (24 - 8 * pass);
        if (pass == 3) st->t = st->prefix + 1u;
    }
    __syncthreads();
    st->hist[d] = 0ull;
}

__global__ void __launch_bounds__(kAllocThreads) alloc_assign_kernel(const float *__restrict__ F, int64_t n,
                                                                     const AllocState *st, uint8_t *__restrict__ b,
                                                                     float *T, int64_t *counts)
{
    __shared__ unsigned long long cnt[3];
    if (threadIdx.x < 3) cnt[threadIdx.x] = 0ull;
    __syncthreads();
    const uint32_t t = st->all8 ? 0u : st->t;
    if (blockIdx.x == 0 && threadIdx.x == 0) *T = __uint_as_float(t);
    unsigned int c2 = 0, c4 = 0, c8 = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
        const float f = __ldg(F + j);
        uint8_t bits = 2;
        if (key8_of(f) >= t) { bits = 8; ++c8; }
        else if (key4_of(f) >= t) { bits = 4; ++c4; }
        else ++c2;
        b[j] = bits;
    }
    atomicAdd(&cnt[0], (unsigned long long)c2);
    atomicAdd(&cnt[1], (unsigned long long)c4);
    atomicAdd(&cnt[2], (unsigned long long)c8);
    __syncthreads();
    if (threadIdx.x < 3 && cnt[threadIdx.x])
        atomicAdd(reinterpret_cast<unsigned long long *>(counts) + threadIdx.x, cnt[threadIdx.x]);
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

// Exclusive scan over tiles, per class, plus the class bases: writes the
// first output position of each (tile, class) into tile_counts[tile*4+c].
__global__ void __launch_bounds__(1024) reorder_scan_kernel(long long *tile_counts, int64_t n_tiles)
{
    __shared__ long long tot[3];
    __shared__ long long warp_sum[32][3];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    long long carry[3] = {0, 0, 0};
    // pass 1: class totals
    long long part[3] = {0, 0, 0};
    for (int64_t i = tid; i < n_tiles; i += blockDim.x)
        for (int k = 0; k < 3; ++k) part[k] += tile_counts[i * 4 + k];
    for (int k = 0; k < 3; ++k)
        for (int m = 16; m >= 1; m >>= 1) part[k] += __shfl_xor_sync(kFull, part[k], m);
    if (lane == 0)
        for (int k = 0; k < 3; ++k) warp_sum[wid][k] = part[k];
    __syncthreads();
    if (tid == 0) {
        for (int k = 0; k < 3; ++k) {
            long long s = 0;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += warp_sum[w][k];
            tot[k] = s;
        }
    }
    __syncthreads();
    carry[0] = 0;
    carry[1] = tot[0];
    carry[2] = tot[0] + tot[1];
    __syncthreads();
    // pass 2: chunked exclusive scan
    for (int64_t base = 0; base < n_tiles; base += blockDim.x) {
        const int64_t i = base + tid;
        long long v[3];
        for (int k = 0; k < 3; ++k) v[k] = i < n_tiles ? tile_counts[i * 4 + k] : 0;
        long long inc[3] = {v[0], v[1], v[2]};
        for (int off = 1; off < 32; off <<= 1)
            for (int k = 0; k < 3; ++k) {
                const long long o = __shfl_up_sync(kFull, inc[k], off);
                if (lane >= off) inc[k] += o;
            }
        if (lane == 31)
            for (int k = 0; k < 3; ++k) warp_sum[wid][k] = inc[k];
        __syncthreads();
        long long wpre[3] = {0, 0, 0}, chunk[3] = {0, 0, 0};
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            for (int k = 0; k < 3; ++k) {
                if (w < wid) wpre[k] += warp_sum[w][k];
                chunk[k] += warp_sum[w][k];
            }
        if (i < n_tiles)
            for (int k = 0; k < 3; ++k) tile_counts[i * 4 + k] = carry[k] + wpre[k] + inc[k] - v[k];
        for (int k = 0; k < 3; ++k) carry[k] += chunk[k];
        __syncthreads();
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
// (F held in shared memory): the same weighted radix select and stable
// partition as the kernels above, without their 12 launches.  Histogram
// updates are combined per warp (__match_any_sync) before the shared
// atomic, since the top digit of F is mostly its exponent and few bins
// take most keys.  fixed_bits != 0 gives every super-group that width.
constexpr int kSmallPlanThreads = 1024;

__global__ void __launch_bounds__(kSmallPlanThreads) plan_small_kernel(const float *__restrict__ F, int32_t n,
                                                                       long long R, int32_t all8, int32_t fixed_bits,
                                                                       uint8_t *__restrict__ b, float *T,
                                                                       int64_t *counts, int32_t *__restrict__ perm)
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
    }
}

}  // namespace

size_t reorder_scratch_bytes(int64_t n_sg)
{
    const int64_t n_tiles = (n_sg + kTile - 1) / kTile;
    return (size_t)(n_tiles > 0 ? n_tiles : 1) * 4 * sizeof(long long);
}

size_t plan_scratch_bytes(int64_t n_sg)
{
    const size_t reorder = reorder_scratch_bytes(n_sg);
    const size_t alloc = sizeof(AllocState);
    const size_t m = reorder > alloc ? reorder : alloc;
    return (m + 255) / 256 * 256;
}

cudaError_t launch_allocate(const float *F, int64_t n_sg, int64_t cap_bits, uint8_t *b, float *T,
                            int64_t *counts, void *ws, cudaStream_t st)
{
    AllocState *s = static_cast<AllocState *>(ws);
    const long long R = (long long)(cap_bits - 2 * n_sg);
    const int all8 = R >= 6 * (long long)n_sg ? 1 : 0;
    alloc_init_kernel<<<1, 256, 0, st>>>(s, R, all8, counts);
    int64_t blocks = (n_sg + kAllocThreads - 1) / kAllocThreads;
    const int64_t cap = (int64_t)sm_count() * 4;
    blocks = blocks < 1 ? 1 : (blocks < cap ? blocks : cap);
    if (!all8) {
        for (int pass = 0; pass < 4; ++pass) {
            alloc_hist_kernel<<<(int)blocks, kAllocThreads, 0, st>>>(F, n_sg, s, pass);
            alloc_select_kernel<<<1, 256, 0, st>>>(s, pass);
        }
    }
    alloc_assign_kernel<<<(int)blocks, kAllocThreads, 0, st>>>(F, n_sg, s, b, T, counts);
    note_launches(all8 ? 2 : 10);
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

int64_t small_plan_max_sg() { return kSmallPlanMaxSG; }

cudaError_t launch_plan_small(const float *F, int64_t n_sg, int64_t cap_bits, int32_t fixed_bits, uint8_t *b,
                              float *T, int64_t *counts, int32_t *perm, cudaStream_t st)
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
    plan_small_kernel<<<1, kSmallPlanThreads, smem, st>>>(F, (int32_t)n_sg, R, all8, fixed_bits, b, T, counts, perm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace dq
