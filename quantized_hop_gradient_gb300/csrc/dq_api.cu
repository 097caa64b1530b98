// dq_api.cu -- the C ABI of libdq: argument validation, level tables,
// message layout, single-call entry points and the N-rank schedule.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "dq_common.cuh"
#include "dq_internal.h"
#include "dq_sched.h"

namespace dq {

// --------------------------------------------------------------------------- device info
static std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int sm_count()
{
    static std::atomic<int> cache[128];   // zero-initialised (static storage); 0 = not yet read
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 152;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// --------------------------------------------------------------------------- level tables
// Levels: r_k = -1 + 2k/(L-1), q_k = sign(r_k) * a(eps + a)/(1 + eps) with
// a = |r_k|, evaluated in binary64 in that order, rounded once to fp32;
// eps = +inf gives q_k = r_k.
static void levels(int bits, double eps, float *q)
{
    const int L = 1 << bits;
    for (int k = 0; k < L; ++k) {
        const double r = -1.0 + (2.0 * (double)k) / (double)(L - 1);
        const double a = fabs(r);
        const double f = isinf(eps) ? a : (a * (eps + a)) / (1.0 + eps);
        q[k] = (float)(r < 0.0 ? -f : f);
    }
}

// Levels, G16_k = fl(1/fl(q_{k+1}-q_k)) * 2^16 (0 for the top level) and the
// level-search buckets of one bitwidth.  H is the smallest power of two with
// 1/H <= the smallest gap (capped at the table's capacity); with r =
// rint(sub H y), bucket b = floor(r/sub) covers [(b - 1/(2 sub))/H,
// (b + 1 - 1/(2 sub))/H) (a tie at the lower edge rounds to the even r =
// sub b) and is stored at index b & mask.  Returns whether every bucket
// holds at most one level above its lower edge.
static bool fill_bitwidth(int bits, double eps, float *qdec, float *g16, BucketEntry *bk, int mask, int sub,
                          int off, float *mul_out)
{
    const int L = 1 << bits;
    float q[256];
    levels(bits, eps, q);
    float min_gap = INFINITY;
    for (int k = 0; k < L; ++k) {
        float G = 0.0f;
        if (k + 1 < L) {
            const float gap = q[k + 1] - q[k];
            G = (1.0f / gap) * 65536.0f;
            if (gap < min_gap) min_gap = gap;
        }
        qdec[k] = q[k];
        g16[k] = G;
    }
    const int hmax = mask / 2;   // 2H + 1 buckets must fit in the mask + 1 slots
    int H = 2;
    while (2 * H <= hmax && 1.0 / (double)H > (double)min_gap) H *= 2;
    *mul_out = (float)(sub * H);
    for (int i = 0; i <= mask; ++i) {   // unused slots: harmless entries
        bk[i].boundary = INFINITY;
        bk[i].kb4 = 0;
    }
    bool one = true;
    for (int b = -H; b <= H; ++b) {
        const double half = 0.5 / (double)sub;
        const double lo = ((double)b - half) / (double)H, hi = ((double)b + 1.0 - half) / (double)H;
        int kb = 0;
        for (int k = 0; k < L; ++k)
            if ((double)q[k] <= lo) kb = k;
        int above = 0;
        for (int k = 0; k < L; ++k)
            if ((double)q[k] > lo && (double)q[k] < hi) ++above;
        if (above > 1) one = false;
        BucketEntry &e = bk[(b + off) & mask];
        e.kb4 = 4 * kb;
        e.boundary = kb + 1 < L ? q[kb + 1] : INFINITY;
    }
    return one;
}

bool build_tables(double eps, Tables *out)
{
    if (!(eps > 0.0)) return false;  // rejects NaN, zero and negatives; +inf allowed
    static std::mutex mu;
    static std::map<uint64_t, std::unique_ptr<Tables>> cache;
    uint64_t key;
    memcpy(&key, &eps, sizeof(key));
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it == cache.end()) {
        std::unique_ptr<Tables> t(new Tables());
        memset(t.get(), 0, sizeof(Tables));
        bool one = fill_bitwidth(2, eps, t->q2, t->g2, t->bk2, kMask2, kSub2, 0, &t->mul2);
        one = fill_bitwidth(4, eps, t->q4, t->g4, t->bk4, kMask4, kSub4, 0, &t->mul4) && one;
        one = fill_bitwidth(8, eps, t->q8, t->g8, t->bk8, kMask8, kSub8, kOff8, &t->mul8) && one;
        t->one_level = one ? 1 : 0;
        t->rcp[0] = 0.0f;
        for (int u = 1; u < 256; ++u) t->rcp[u] = 1.0f / (float)u;
        if (cache.size() > 16) cache.clear();
        it = cache.emplace(key, std::move(t)).first;
    }
    *out = *it->second;
    return true;
}

// --------------------------------------------------------------------------- message layout
static int64_t overlap(int64_t a, int64_t b, int64_t c, int64_t d)
{
    const int64_t lo = a > c ? a : c, hi = b < d ? b : d;
    return hi > lo ? hi - lo : 0;
}

size_t msg_bytes(int64_t c, int64_t n2, int64_t n4, int64_t n8, bool scale_fp32)
{
    const int64_t meta = scale_fp32 ? 64 * c : (c + 15) / 16 * 16 + 16 * c;
    return (size_t)(meta + 64 * n2 + 128 * n4 + 256 * n8);
}

MsgView msg_view(uint8_t *base, int64_t lo, int64_t hi, int64_t end2, int64_t end4, bool scale_fp32)
{
    MsgView m;
    m.base = base;
    m.c = hi - lo;
    m.n2 = overlap(lo, hi, 0, end2);
    m.n4 = overlap(lo, hi, end2, end4);
    m.off_u = scale_fp32 ? 0 : (m.c + 15) / 16 * 16;
    m.off_c2 = m.off_u + (scale_fp32 ? 64 : 16) * m.c;
    m.off_c4 = m.off_c2 + 64 * m.n2;
    m.off_c8 = m.off_c4 + 128 * m.n4;
    return m;
}

// Bitwidth-pure segments of [lo, hi) and their work units, numbered from
// `first`; returns the number of units.
template <typename Task>
static int64_t set_units(Task &t, int64_t lo, int64_t hi, int64_t end2, int64_t end4, int64_t first)
{
    const int64_t cuts[4] = {lo, std::max(lo, std::min(hi, end2)), std::max(lo, std::min(hi, end4)), hi};
    int64_t u = first;
    for (int s = 0; s < 3; ++s) {
        t.seg_lo[s] = cuts[s];
        t.seg_hi[s] = cuts[s + 1];
        t.unit_begin[s] = u;
        u += (cuts[s + 1] - cuts[s] + kUnit - 1) / kUnit;
    }
    t.unit_begin[3] = u;
    return u - first;
}

}  // namespace dq

using namespace dq;

// --------------------------------------------------------------------------- host helpers
namespace {

constexpr int64_t kMaxSG = (int64_t)1 << 27;  // keeps the generator counter in 32 bits

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool range_ok(const dq_range &r)
{
    return r.lo >= 0 && r.lo <= r.hi && r.hi - r.lo < kMaxSG && r.hi <= kMaxSG && r.end2 >= 0 &&
           r.end2 <= r.end4 && r.end4 <= kMaxSG;
}

bool cfg_ok(const dq_config *c)
{
    return c && c->n_ranks >= 1 && c->n_ranks <= 65535 && (c->eps > 0.0) &&
           (c->fixed_bits == 0 || c->fixed_bits == 2 || c->fixed_bits == 4 || c->fixed_bits == 8) &&
           (c->scale_fp32 == 0 || c->scale_fp32 == 1);
}

bool stage_ok(const dq_config *cfg, const dq_stage &s)
{
    return s.rank >= 0 && s.rank < cfg->n_ranks && s.hop >= 0 && s.hop <= 0xFFFF && s.n_slots >= 1 &&
           s.n_slots <= 65536 && s.slot >= 0 && s.slot < s.n_slots;
}

dq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DQ_OK : DQ_ERR_CUDA; }

// Generator counter word 1 and the correlated-rounding offset of a stage:
// independent rounding keys the stream by (hop, rank); correlated rounding
// shares one stream per hop (rank field 0xFFFF, above any rank) and shifts
// it by floor(slot * 2^16 / n_slots), in both 16-bit halves of a word.
HopTask make_task(const dq_config *cfg, const dq_stage &s)
{
    HopTask t;
    memset(&t, 0, sizeof(t));
    if (cfg->correlated) {
        const uint32_t off = (uint32_t)(((uint64_t)(uint32_t)s.slot << 16) / (uint64_t)(uint32_t)s.n_slots);
        t.stage_word = (uint32_t)s.hop | (0xFFFFu << 16);
        t.corr2 = off | (off << 16);
    } else {
        t.stage_word = (uint32_t)s.hop | ((uint32_t)s.rank << 16);
        t.corr2 = 0u;
    }
    return t;
}

// The Philox key schedule of a launch (seed as key, round as counter words 2
// and 3): round keys and round 0's lane-independent part.
PhiloxKeys philox_keys(uint64_t seed, uint64_t round)
{
    const uint32_t M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    PhiloxKeys K;
    for (int r = 0; r < 10; ++r) {
        K.k0[r] = (uint32_t)seed + (uint32_t)r * W0;
        K.k1[r] = (uint32_t)(seed >> 32) + (uint32_t)r * W1;
    }
    const uint64_t p = (uint64_t)M1 * (uint32_t)round;
    K.a0 = (uint32_t)(p >> 32) ^ K.k0[0];
    K.l1 = (uint32_t)p;
    K.r1k = (uint32_t)(round >> 32) ^ K.k1[0];
    return K;
}

void fill_common(HopParams &P, const dq_config *cfg, const float *mu, const int32_t *perm)
{
    P.n_ranks = cfg->n_ranks;
    P.mu = mu;
    P.perm = perm;
    P.ph = philox_keys(cfg->seed, cfg->round);
    P.scale_fp32 = cfg->scale_fp32;
}

// A hop task with its input range [in_lo, in_hi).
struct PendingHop {
    HopTask t;
    int64_t in_hi;
};

}  // namespace

namespace dq {

LogSlot log_begin(dq_launch_log *log, int32_t kind, int64_t sgs, cudaStream_t st)
{
    if (!log || !log->events || log->count < 0 || log->count >= log->capacity) return {nullptr, -1};
    const int32_t i = log->count++;
    if (log->kinds) log->kinds[i] = kind;
    if (log->sgs) log->sgs[i] = sgs;
    cudaEventRecord(static_cast<cudaEvent_t>(log->events[2 * i]), st);
    return {log, i};
}

void log_end(const LogSlot &s, cudaStream_t st)
{
    if (s.log) cudaEventRecord(static_cast<cudaEvent_t>(s.log->events[2 * s.i + 1]), st);
}

}  // namespace dq

namespace {

// Launches hop tasks in batches of at most kMaxTasks (empty tasks dropped).
cudaError_t run_hops(HopParams &P, const std::vector<PendingHop> &tasks, int64_t end2, int64_t end4, bool has_in,
                     bool add_f32, cudaStream_t st, dq_launch_log *log)
{
    size_t i = 0;
    while (i < tasks.size()) {
        int n = 0;
        int64_t units = 0, sgs = 0;
        while (i < tasks.size() && n < kMaxTasks) {
            const PendingHop &ph = tasks[i++];
            if (ph.in_hi <= ph.t.in_lo) continue;
            HopTask t = ph.t;
            units += set_units(t, t.in_lo, ph.in_hi, end2, end4, units);
            sgs += ph.in_hi - t.in_lo;
            P.task[n++] = t;
        }
        P.n_tasks = n;
        P.total_units = units;
        if (n > 0) {
            const LogSlot slot = log_begin(log, has_in ? DQ_LAUNCH_DAR : DQ_LAUNCH_COMPRESS, sgs, st);
            const cudaError_t e = launch_hop(P, has_in, add_f32, st);
            log_end(slot, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

// A chunk to decode: its message, reordered range and output.
struct PendingDecode {
    const uint8_t *msg;
    int64_t lo, hi;
    void *out;
};

cudaError_t run_decodes(DecodeParams &D, const std::vector<PendingDecode> &chunks, int64_t end2, int64_t end4,
                        cudaStream_t st, dq_launch_log *log)
{
    size_t i = 0;
    while (i < chunks.size()) {
        int n = 0;
        int64_t units = 0, sgs = 0;
        while (i < chunks.size() && n < kMaxTasks) {
            const PendingDecode &c = chunks[i++];
            if (c.hi <= c.lo) continue;
            DecodeTask &t = D.task[n++];
            memset(&t, 0, sizeof(t));
            t.msg = msg_view(const_cast<uint8_t *>(c.msg), c.lo, c.hi, end2, end4, D.scale_fp32 != 0);
            t.out = c.out;
            t.lo = c.lo;
            units += set_units(t, c.lo, c.hi, end2, end4, units);
            sgs += (c.hi - c.lo) * std::max(1, D.n_outs);   // super-groups written
        }
        D.n_tasks = n;
        D.total_units = units;
        if (n > 0) {
            const LogSlot slot = log_begin(log, DQ_LAUNCH_DECODE, sgs, st);
            const cudaError_t e = launch_decode(D, st);
            log_end(slot, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

std::unique_ptr<DecodeParams> decode_params(const dq_config *cfg, const float *mu, const int32_t *perm,
                                            int32_t out_is_bf16, const Tables &tab)
{
    std::unique_ptr<DecodeParams> D(new DecodeParams());
    memset(D.get(), 0, sizeof(DecodeParams));
    D->tab = tab;
    D->n_ranks = cfg->n_ranks;
    D->mu = mu;
    D->perm = perm;
    D->out_is_bf16 = out_is_bf16 ? 1 : 0;
    D->scale_fp32 = cfg->scale_fp32;
    return D;
}

}  // namespace

// --------------------------------------------------------------------------- single-call entry points
extern "C" {

const char *dq_version(void) { return "libdq 0.2 (sm_103a)"; }

uint64_t dq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *dq_status_string(dq_status s)
{
    switch (s) {
    case DQ_OK: return "ok";
    case DQ_ERR_INVALID_ARG: return "invalid argument";
    case DQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case DQ_ERR_BUDGET_INFEASIBLE: return "budget below 2 bits per coordinate";
    case DQ_ERR_CUDA: return "CUDA error";
    case DQ_ERR_NONFINITE: return "non-finite gradient statistics (NaN or infinite input)";
    }
    return "unknown status";
}

size_t dq_message_bytes(dq_range r, int32_t scale_fp32)
{
    if (!range_ok(r) || (scale_fp32 != 0 && scale_fp32 != 1)) return 0;
    const MsgView m = msg_view(nullptr, r.lo, r.hi, r.end2, r.end4, scale_fp32 != 0);
    return msg_bytes(m.c, m.n2, m.n4, m.c - m.n2 - m.n4, scale_fp32 != 0);
}

dq_status dq_level_table(int32_t bits, double eps, float *q_host)
{
    if ((bits != 2 && bits != 4 && bits != 8) || !q_host) return DQ_ERR_INVALID_ARG;
    Tables t;
    if (!build_tables(eps, &t)) return DQ_ERR_INVALID_ARG;
    const float *q = bits == 2 ? t.q2 : (bits == 4 ? t.q4 : t.q8);
    for (int k = 0; k < (1 << bits); ++k) q_host[k] = q[k];
    return DQ_OK;
}

dq_status dq_stats(const void *g_bf16, int64_t n_sg, float *mean, float *sq, void *stream)
{
    if (n_sg < 0 || n_sg >= kMaxSG) return DQ_ERR_INVALID_ARG;
    if (n_sg == 0) return DQ_OK;
    if (!g_bf16 || !mean || !sq) return DQ_ERR_INVALID_ARG;
    if (!aligned16(g_bf16)) return DQ_ERR_ALIGNMENT;
    return cuda_status(launch_stats(static_cast<const uint16_t *>(g_bf16), n_sg, mean, sq,
                                    static_cast<cudaStream_t>(stream)));
}

dq_status dq_stats_reduce(const float *mean_all, const float *sq_all, int32_t n_ranks, int64_t n_sg, float *M,
                          float *F, float *mu, void *stream)
{
    if (n_sg < 0 || n_sg >= kMaxSG || n_ranks < 1 || n_ranks > 65535) return DQ_ERR_INVALID_ARG;
    if (n_sg == 0) return DQ_OK;
    if (!mean_all || !sq_all || !F || !mu) return DQ_ERR_INVALID_ARG;
    return cuda_status(launch_stats_reduce(mean_all, sq_all, n_ranks, n_sg, M, F, mu,
                                           static_cast<cudaStream_t>(stream)));
}

size_t dq_workspace_bytes(int64_t n_sg) { return plan_scratch_bytes(n_sg < 0 ? 0 : n_sg); }

dq_status dq_allocate(const float *F, int64_t n_sg, float budget, uint8_t *b, float *T_dev, int64_t *counts_dev,
                      void *ws, size_t ws_bytes, void *stream)
{
    if (n_sg < 1 || n_sg >= kMaxSG) return DQ_ERR_INVALID_ARG;
    if (!F || !b || !T_dev || !counts_dev || !ws) return DQ_ERR_INVALID_ARG;
    if (!(budget >= 2.0f)) return DQ_ERR_BUDGET_INFEASIBLE;
    if (ws_bytes < plan_scratch_bytes(n_sg)) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws) || ((uintptr_t)counts_dev & 7u)) return DQ_ERR_ALIGNMENT;
    // floor(B * J) is exact in binary64 for J < 2^27
    const int64_t cap = (int64_t)floor((double)budget * (double)n_sg);
    return cuda_status(launch_allocate(F, n_sg, cap, b, T_dev, counts_dev, ws, static_cast<cudaStream_t>(stream)));
}

dq_status dq_reorder(const uint8_t *b, int64_t n_sg, int32_t *perm, void *ws, size_t ws_bytes, void *stream)
{
    if (n_sg < 1 || n_sg >= kMaxSG) return DQ_ERR_INVALID_ARG;
    if (!b || !perm || !ws) return DQ_ERR_INVALID_ARG;
    if (ws_bytes < plan_scratch_bytes(n_sg)) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    return cuda_status(launch_reorder(b, n_sg, perm, ws, static_cast<cudaStream_t>(stream)));
}

dq_status dq_chunk_cuts(int64_t n2, int64_t n4, int64_t n8, int32_t n_chunks, int64_t *lo)
{
    if (n2 < 0 || n4 < 0 || n8 < 0 || n_chunks < 1 || !lo) return DQ_ERR_INVALID_ARG;
    const int64_t J = n2 + n4 + n8;
    if (J >= kMaxSG) return DQ_ERR_INVALID_ARG;
    const int64_t total = 2 * n2 + 4 * n4 + 8 * n8;
    lo[0] = 0;
    for (int32_t c = 1; c < n_chunks; ++c) {
        const int64_t target = ((int64_t)c * total + n_chunks - 1) / n_chunks;  // ceil
        int64_t i;
        if (target <= 2 * n2) i = (target + 1) / 2;
        else if (target <= 2 * n2 + 4 * n4) i = n2 + (target - 2 * n2 + 3) / 4;
        else i = n2 + n4 + (target - 2 * n2 - 4 * n4 + 7) / 8;
        lo[c] = i;
    }
    lo[n_chunks] = J;
    return DQ_OK;
}

dq_status dq_compress(const dq_config *cfg, dq_range r, dq_stage stage, const void *g_bf16, const float *mu,
                      const int32_t *perm, uint8_t *msg_out, void *stream)
{
    if (!cfg_ok(cfg) || !range_ok(r) || !stage_ok(cfg, stage)) return DQ_ERR_INVALID_ARG;
    if (r.hi == r.lo) return DQ_OK;
    if (!g_bf16 || !mu || !perm || !msg_out) return DQ_ERR_INVALID_ARG;
    if (!aligned16(g_bf16) || !aligned16(msg_out)) return DQ_ERR_ALIGNMENT;
    std::unique_ptr<HopParams> P(new HopParams());
    memset(P.get(), 0, sizeof(HopParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    fill_common(*P, cfg, mu, perm);
    PendingHop h;
    h.t = make_task(cfg, stage);
    h.t.out = msg_view(msg_out, r.lo, r.hi, r.end2, r.end4, cfg->scale_fp32 != 0);
    h.t.addend = g_bf16;
    h.t.in_lo = r.lo;
    h.t.send_lo = r.lo;
    h.t.send_hi = r.hi;
    h.t.keep_lo = h.t.keep_hi = r.hi;
    h.in_hi = r.hi;
    return cuda_status(run_hops(*P, {h}, r.end2, r.end4, false, false, static_cast<cudaStream_t>(stream), nullptr));
}

dq_status dq_dar(const dq_config *cfg, dq_range in, dq_stage stage, const uint8_t *msg_in, const void *addend,
                 int32_t addend_is_fp32, const float *mu, const int32_t *perm, dq_range send, uint8_t *msg_out,
                 dq_range keep, float *keep_out, void *stream)
{
    if (!cfg_ok(cfg) || !range_ok(in) || !range_ok(send) || !range_ok(keep) || !stage_ok(cfg, stage))
        return DQ_ERR_INVALID_ARG;
    if (send.end2 != in.end2 || send.end4 != in.end4 || keep.end2 != in.end2 || keep.end4 != in.end4)
        return DQ_ERR_INVALID_ARG;
    const int64_t ns = send.hi - send.lo, nk = keep.hi - keep.lo, ni = in.hi - in.lo;
    if (ns + nk != ni) return DQ_ERR_INVALID_ARG;
    if (ns > 0 && (send.lo < in.lo || send.hi > in.hi)) return DQ_ERR_INVALID_ARG;
    if (nk > 0 && (keep.lo < in.lo || keep.hi > in.hi)) return DQ_ERR_INVALID_ARG;
    if (ns > 0 && nk > 0 && !(send.hi == keep.lo || keep.hi == send.lo)) return DQ_ERR_INVALID_ARG;
    if (ni == 0) return DQ_OK;
    if (!msg_in || !addend || !perm || (!addend_is_fp32 && !mu)) return DQ_ERR_INVALID_ARG;
    if ((ns > 0 && !msg_out) || (nk > 0 && !keep_out)) return DQ_ERR_INVALID_ARG;
    if (!aligned16(msg_in) || !aligned16(addend) || (ns > 0 && !aligned16(msg_out)) ||
        (nk > 0 && !aligned16(keep_out)))
        return DQ_ERR_ALIGNMENT;
    std::unique_ptr<HopParams> P(new HopParams());
    memset(P.get(), 0, sizeof(HopParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    fill_common(*P, cfg, mu, perm);
    PendingHop h;
    h.t = make_task(cfg, stage);
    h.t.in = msg_view(const_cast<uint8_t *>(msg_in), in.lo, in.hi, in.end2, in.end4, cfg->scale_fp32 != 0);
    h.t.out = msg_view(msg_out, send.lo, send.hi, send.end2, send.end4, cfg->scale_fp32 != 0);
    h.t.addend = addend;
    h.t.keep_out = keep_out;
    h.t.in_lo = in.lo;
    h.t.send_lo = ns > 0 ? send.lo : in.hi;
    h.t.send_hi = ns > 0 ? send.hi : in.hi;
    h.t.keep_lo = nk > 0 ? keep.lo : in.hi;
    h.t.keep_hi = nk > 0 ? keep.hi : in.hi;
    h.in_hi = in.hi;
    return cuda_status(run_hops(*P, {h}, in.end2, in.end4, true, addend_is_fp32 != 0,
                                static_cast<cudaStream_t>(stream), nullptr));
}

dq_status dq_decode(const dq_config *cfg, dq_range r, const uint8_t *msg, const float *mu, const int32_t *perm,
                    void *out, int32_t out_is_bf16, void *stream)
{
    if (!cfg_ok(cfg) || !range_ok(r)) return DQ_ERR_INVALID_ARG;
    if (r.hi == r.lo) return DQ_OK;
    if (!msg || !mu || !perm || !out) return DQ_ERR_INVALID_ARG;
    if (!aligned16(msg) || !aligned16(out)) return DQ_ERR_ALIGNMENT;
    Tables tab;
    if (!build_tables(cfg->eps, &tab)) return DQ_ERR_INVALID_ARG;
    std::unique_ptr<DecodeParams> D = decode_params(cfg, mu, perm, out_is_bf16, tab);
    return cuda_status(run_decodes(*D, {PendingDecode{msg, r.lo, r.hi, out}}, r.end2, r.end4,
                                   static_cast<cudaStream_t>(stream), nullptr));
}

}  // extern "C"

// --------------------------------------------------------------------------- N-rank schedule
namespace {

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

struct PlanLayout {
    size_t mean_all, sq_all, M, F, b, T, counts, scratch, total;
};

PlanLayout plan_layout(int32_t n, int64_t J)
{
    PlanLayout L;
    size_t o = 0;
    L.mean_all = o; o += round256(sizeof(float) * (size_t)n * (size_t)J);
    L.sq_all = o;   o += round256(sizeof(float) * (size_t)n * (size_t)J);
    L.M = o;        o += round256(sizeof(float) * (size_t)J);
    L.F = o;        o += round256(sizeof(float) * (size_t)J);
    L.b = o;        o += round256((size_t)J);
    L.T = o;        o += 256;
    L.counts = o;   o += 256;
    L.scratch = o;  o += round256(plan_scratch_bytes(J));
    L.total = o;
    return L;
}

struct ExchangeLayout {
    std::vector<int64_t> lo;    // chunk cuts
    size_t msg_stride = 0;      // bytes per message buffer
    size_t keep_stride = 0;     // bytes per fp32 keep buffer
    size_t msgs = 0, keeps = 0, finals = 0, total = 0;
    Schedule S;
};

bool exchange_layout(const dq_config *cfg, int32_t butterfly, const dq_plan_info *info, ExchangeLayout &X)
{
    const int32_t N = cfg->n_ranks;
    X.lo.assign((size_t)N + 1, 0);
    if (dq_chunk_cuts(info->n2, info->n4, info->n8, N, X.lo.data()) != DQ_OK) return false;
    if (!build_schedule(N, butterfly != 0, X.S)) return false;
    const int64_t end2 = info->n2, end4 = info->n2 + info->n4;
    const bool sf = cfg->scale_fp32 != 0;
    size_t mmax = 16, kmax = 16;
    for (const SchedStep &st : X.S.steps)
        for (const SchedHop &h : st.hops) {
            const int64_t a = X.lo[h.send.a], b = X.lo[h.send.b];
            const MsgView m = msg_view(nullptr, a, b, end2, end4, sf);
            mmax = std::max(mmax, msg_bytes(m.c, m.n2, m.n4, m.c - m.n2 - m.n4, sf));
            kmax = std::max(kmax, (size_t)(X.lo[h.keep.b] - X.lo[h.keep.a]) * kSG * sizeof(float));
        }
    X.msg_stride = round256(mmax);
    X.keep_stride = butterfly ? round256(kmax) : 0;
    size_t o = 0;
    X.msgs = o;   o += 2 * (size_t)N * X.msg_stride;
    X.keeps = o;  o += 2 * (size_t)N * X.keep_stride;
    X.finals = o; o += butterfly ? (size_t)N * X.msg_stride : 0;
    X.total = o;
    return true;
}

}  // namespace

namespace {

// What dq_plan reads back to the host: the stream counts, the threshold and
// the non-finite flag.
struct PlanReadback {
    int64_t counts[3];
    float T;
    int32_t nonfinite;
    int32_t status;   // dq_get_device_status
};

// One thread copies the plan's results into host memory mapped into the
// device address space.  The host then reads them after synchronising the
// plan's stream: no copy-engine transfer is involved, so the read cannot
// queue behind large host<->device copies that other streams have in flight
// (a pageable cudaMemcpyAsync could, and stalled the planning of a round
// until the next round's gradient upload had finished).
__global__ void plan_readback_kernel(const int64_t *counts, const float *T, const int32_t *nonfinite,
                                     PlanReadback *out)
{
    if (threadIdx.x == 0) {
        out->counts[0] = counts[0];
        out->counts[1] = counts[1];
        out->counts[2] = counts[2];
        out->T = T ? *T : 0.0f;
        out->nonfinite = *nonfinite;
    }
}

// Zeroes a few 32-bit words in stream order.  A kernel, not
// cudaMemsetAsync: a small memset may be carried out by a copy engine and
// then wait behind large host<->device copies queued by other streams.
__global__ void zero_words_kernel(uint32_t *a, int na, uint32_t *b)
{
    for (int i = threadIdx.x; i < na; i += blockDim.x) a[i] = 0u;
    if (threadIdx.x == 0 && b) *b = 0u;
}

// a[0 .. na) and, if b is not null, b[0]
cudaError_t zero_words(void *a, int na, void *b, cudaStream_t st)
{
    zero_words_kernel<<<1, 32, 0, st>>>(static_cast<uint32_t *>(a), na, static_cast<uint32_t *>(b));
    note_launches(1);
    return cudaGetLastError();
}

// Zeroes n 32-bit words (any count) in one launch.
__global__ void zero_many_kernel(uint32_t *p, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0u;
}

cudaError_t zero_many(void *p, int64_t n, cudaStream_t st)
{
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4 * (int64_t)sm_count());
    zero_many_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<uint32_t *>(p), n);
    note_launches(1);
    return cudaGetLastError();
}

// One thread copies a device status word into host memory mapped into the
// device address space (the readback of dq_get_device_status).
__global__ void status_readback_kernel(const int32_t *src, int32_t *out)
{
    if (threadIdx.x == 0) *out = *src;
}

// The calling thread's pinned, device-mapped readback buffer (allocated on
// the thread's first dq_plan, kept until the process exits).
PlanReadback *plan_readback_buffer()
{
    thread_local PlanReadback *buf = nullptr;
    if (!buf) {
        void *p = nullptr;
        if (cudaHostAlloc(&p, sizeof(PlanReadback), cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
            return nullptr;
        buf = static_cast<PlanReadback *>(p);
    }
    return buf;
}

// Enqueues the readback on st, synchronises st and returns the host copy.
dq_status plan_read(const int64_t *counts, const float *T, const int32_t *nonfinite, cudaStream_t st,
                    PlanReadback *out)
{
    PlanReadback *buf = plan_readback_buffer();
    if (!buf) return DQ_ERR_CUDA;
    PlanReadback *dev = nullptr;
    if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&dev), buf, 0) != cudaSuccess) return DQ_ERR_CUDA;
    plan_readback_kernel<<<1, 32, 0, st>>>(counts, T, nonfinite, dev);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return DQ_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DQ_ERR_CUDA;
    const volatile PlanReadback *v = buf;   // written by the device: read it afresh
    for (int i = 0; i < 3; ++i) out->counts[i] = v->counts[i];
    out->T = v->T;
    out->nonfinite = v->nonfinite;
    return DQ_OK;
}

}  // namespace

extern "C" {

size_t dq_plan_workspace_bytes(int32_t n_ranks, int64_t n_sg)
{
    if (n_ranks < 1 || n_sg < 1) return 0;
    return plan_layout(n_ranks, n_sg).total;
}

}  // extern "C"

namespace {

// Where a plan leaves its results on the device.
struct PlanDev {
    int64_t *counts;     // n2, n4, n8
    float *T;
    int32_t *nonfinite;
};

// Enqueues the whole plan (statistics, reduce, allocation, reorder) on st;
// nothing is read back.
dq_status plan_enqueue(const dq_config *cfg, const void *const *grads, int64_t n_sg, float *mu, int32_t *perm,
                       void *ws, size_t ws_bytes, void *const *rank_ready, dq_launch_log *log, cudaStream_t st,
                       PlanDev &out, int32_t *sticky = nullptr)
{
    if (!cfg_ok(cfg) || !grads || !mu || !perm || !ws || n_sg < 1 || n_sg >= kMaxSG) return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    const PlanLayout L = plan_layout(N, n_sg);
    if (ws_bytes < L.total) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    if (!cfg->fixed_bits && !(cfg->budget_bits >= 2.0f)) return DQ_ERR_BUDGET_INFEASIBLE;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r])) return DQ_ERR_ALIGNMENT;
    }
    uint8_t *w = static_cast<uint8_t *>(ws);
    float *mean_all = reinterpret_cast<float *>(w + L.mean_all);
    float *sq_all = reinterpret_cast<float *>(w + L.sq_all);
    float *M = reinterpret_cast<float *>(w + L.M);
    float *F = reinterpret_cast<float *>(w + L.F);
    uint8_t *b = w + L.b;
    float *T = reinterpret_cast<float *>(w + L.T);
    int64_t *counts = reinterpret_cast<int64_t *>(w + L.counts);
    int32_t *nonfinite = reinterpret_cast<int32_t *>(w + L.counts + 32);   // inside the counts slot
    void *scratch = w + L.scratch;
    out = PlanDev{counts, T, nonfinite};
    const bool small = n_sg <= small_plan_max_sg();
    // the flag is cleared before the statistics reduce sets it (the chain clears it itself)
    if (small && zero_words(nonfinite, 1, nullptr, st) != cudaSuccess) return DQ_ERR_CUDA;
    if (rank_ready) {  // one launch per rank, each after its rank's event
        for (int32_t r = 0; r < N; ++r) {
            if (rank_ready[r] && cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(rank_ready[r]), 0) != cudaSuccess)
                return DQ_ERR_CUDA;
            const LogSlot slot = log_begin(log, DQ_LAUNCH_STATS, n_sg, st);
            const cudaError_t e = launch_stats(static_cast<const uint16_t *>(grads[r]), n_sg,
                                               mean_all + (size_t)r * n_sg, sq_all + (size_t)r * n_sg, st);
            log_end(slot, st);
            if (e != cudaSuccess) return DQ_ERR_CUDA;
        }
    } else {           // all ranks in launches of up to kMaxStatsRanks
        for (int32_t r0 = 0; r0 < N; r0 += kMaxStatsRanks) {
            StatsParams S;
            memset(&S, 0, sizeof(S));
            S.n_ranks = std::min(N - r0, kMaxStatsRanks);
            for (int32_t r = 0; r < S.n_ranks; ++r) S.g[r] = static_cast<const uint16_t *>(grads[r0 + r]);
            S.n_sg = n_sg;
            S.mean_all = mean_all + (size_t)r0 * n_sg;
            S.sq_all = sq_all + (size_t)r0 * n_sg;
            const LogSlot slot = log_begin(log, DQ_LAUNCH_STATS, n_sg * S.n_ranks, st);
            const cudaError_t e = launch_stats_batched(S, st);
            log_end(slot, st);
            if (e != cudaSuccess) return DQ_ERR_CUDA;
        }
    }
    const int64_t cap = (int64_t)floor((double)cfg->budget_bits * (double)n_sg);
    const LogSlot slot = log_begin(log, DQ_LAUNCH_ALLOCATE_REORDER, n_sg, st);
    if (small) {
        // small problems: the metadata all-reduce, then allocation and reorder in one launch
        if (launch_stats_reduce(mean_all, sq_all, N, n_sg, M, F, mu, st, nonfinite) != cudaSuccess) return DQ_ERR_CUDA;
        if (launch_plan_small(F, n_sg, cap, cfg->fixed_bits, b, T, counts, perm, st, nonfinite, sticky) != cudaSuccess)
            return DQ_ERR_CUDA;
    } else if (launch_plan_chain(mean_all, sq_all, N, n_sg, cap, cfg->fixed_bits, M, F, mu, nonfinite, b, T, counts,
                                 perm, scratch, st, sticky) != cudaSuccess) {
        return DQ_ERR_CUDA;
    }
    log_end(slot, st);
    return DQ_OK;
}

}  // namespace

extern "C" {

dq_status dq_plan(const dq_config *cfg, const void *const *grads, int64_t n_sg, float *mu, int32_t *perm, void *ws,
                  size_t ws_bytes, dq_plan_info *info, void *const *rank_ready, dq_launch_log *log, void *stream)
{
    if (!info) return DQ_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PlanDev d;
    const dq_status s = plan_enqueue(cfg, grads, n_sg, mu, perm, ws, ws_bytes, rank_ready, log, st, d);
    if (s != DQ_OK) return s;
    PlanReadback h;
    const dq_status rs = plan_read(d.counts, cfg->fixed_bits ? nullptr : d.T, d.nonfinite, st, &h);
    if (rs != DQ_OK) return rs;
    if (h.nonfinite) return DQ_ERR_NONFINITE;
    info->T = cfg->fixed_bits ? NAN : h.T;
    info->n2 = h.counts[0];
    info->n4 = h.counts[1];
    info->n8 = h.counts[2];
    return DQ_OK;
}

dq_status dq_plan_async(const dq_config *cfg, const void *const *grads, int64_t n_sg, float *mu, int32_t *perm,
                        void *ws, size_t ws_bytes, const int64_t **counts_dev, const int32_t **nonfinite_dev,
                        void *const *rank_ready, dq_launch_log *log, void *stream)
{
    if (!counts_dev) return DQ_ERR_INVALID_ARG;
    PlanDev d;
    const dq_status s =
        plan_enqueue(cfg, grads, n_sg, mu, perm, ws, ws_bytes, rank_ready, log, static_cast<cudaStream_t>(stream), d);
    if (s != DQ_OK) return s;
    *counts_dev = d.counts;
    if (nonfinite_dev) *nonfinite_dev = d.nonfinite;
    return DQ_OK;
}

size_t dq_exchange_workspace_bytes(const dq_config *cfg, int32_t butterfly, int64_t n_sg, const dq_plan_info *info)
{
    if (!cfg_ok(cfg) || !info || n_sg < 1) return 0;
    ExchangeLayout X;
    if (!exchange_layout(cfg, butterfly, info, X)) return 0;
    return X.total;
}

dq_status dq_exchange(const dq_config *cfg, int32_t butterfly, const void *const *grads, int64_t n_sg, const float *mu,
                      const int32_t *perm, const dq_plan_info *info, void *ws, size_t ws_bytes, void *const *outs,
                      int32_t out_is_bf16, const uint8_t **final_msgs, dq_launch_log *log, void *stream)
{
    if (!cfg_ok(cfg) || !grads || !mu || !perm || !info || !ws || !outs || n_sg < 1 || n_sg >= kMaxSG)
        return DQ_ERR_INVALID_ARG;
    if (info->n2 < 0 || info->n4 < 0 || info->n8 < 0 || info->n2 + info->n4 + info->n8 != n_sg)
        return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    ExchangeLayout X;
    if (!exchange_layout(cfg, butterfly, info, X)) return DQ_ERR_INVALID_ARG;
    if (ws_bytes < X.total) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r] || !outs[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r]) || !aligned16(outs[r])) return DQ_ERR_ALIGNMENT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t end2 = info->n2, end4 = info->n2 + info->n4;
    const bool sf = cfg->scale_fp32 != 0;
    uint8_t *w = static_cast<uint8_t *>(ws);
    auto msg = [&](int32_t r, int32_t par) {
        return par < 0 ? w + X.finals + (size_t)r * X.msg_stride : w + X.msgs + (size_t)(2 * r + par) * X.msg_stride;
    };
    auto keepb = [&](int32_t r, int32_t par) {
        return reinterpret_cast<float *>(w + X.keeps + (size_t)(2 * r + par) * X.keep_stride);
    };
    const std::vector<int64_t> &lo = X.lo;

    std::unique_ptr<HopParams> P(new HopParams());
    memset(P.get(), 0, sizeof(HopParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    fill_common(*P, cfg, mu, perm);

    std::vector<PendingHop> tasks;
    for (const SchedStep &step : X.S.steps) {
        tasks.clear();
        for (const SchedHop &h : step.hops) {
            const int64_t a = lo[h.in.a], b = lo[h.in.b];
            const int64_t sa = lo[h.send.a], sb = lo[h.send.b], ka = lo[h.keep.a], kb = lo[h.keep.b];
            PendingHop ph;
            ph.t = make_task(cfg, dq_stage{h.rank, h.stage, h.slot, h.n_slots});
            ph.t.in = msg_view(h.in_rank < 0 ? nullptr : msg(h.in_rank, h.in_par), a, b, end2, end4, sf);
            ph.t.out = msg_view(msg(h.rank, h.out_par), sa, sb, end2, end4, sf);
            ph.t.addend = h.add_par < 0 ? grads[h.rank] : (const void *)keepb(h.rank, h.add_par);
            ph.t.keep_out = kb > ka ? keepb(h.rank, h.keep_par) : nullptr;
            ph.t.in_lo = a;
            ph.t.send_lo = sb > sa ? sa : b;
            ph.t.send_hi = sb > sa ? sb : b;
            ph.t.keep_lo = kb > ka ? ka : b;
            ph.t.keep_hi = kb > ka ? kb : b;
            ph.in_hi = b;
            tasks.push_back(ph);
        }
        if (run_hops(*P, tasks, end2, end4, step.has_in, step.add_f32, st, log) != cudaSuccess) return DQ_ERR_CUDA;
    }

    // All-gather hands the final chunks to every rank unchanged; every rank
    // decodes all of them into its own output.  Each launch reads the chunk
    // messages once and writes up to kMaxDecodeOuts ranks' outputs.
    std::vector<const uint8_t *> fin((size_t)N, nullptr);
    for (int32_t c = 0; c < N; ++c) fin[c] = msg(X.S.fin_rank[c], X.S.fin_par[c]);
    std::vector<PendingDecode> chunks;
    for (int32_t c = 0; c < N; ++c) chunks.push_back(PendingDecode{fin[c], lo[c], lo[c + 1], nullptr});
    std::unique_ptr<DecodeParams> D = decode_params(cfg, mu, perm, out_is_bf16, P->tab);
    for (int32_t r0 = 0; r0 < N; r0 += kMaxDecodeOuts) {
        D->n_outs = std::min(N - r0, kMaxDecodeOuts);
        for (int32_t i = 0; i < D->n_outs; ++i) D->outs[i] = outs[r0 + i];
        if (run_decodes(*D, chunks, end2, end4, st, log) != cudaSuccess) return DQ_ERR_CUDA;
    }
    if (final_msgs)
        for (int32_t c = 0; c < N; ++c) final_msgs[c] = fin[c];
    return DQ_OK;
}

}  // extern "C"

// --------------------------------------------------------------------------- fused ring exchange
namespace {

constexpr long long kBarrierTimeoutCycles = 2000000000LL;   // about one second at the SM clock

bool fused_ok(const dq_config *cfg) { return cfg_ok(cfg) && cfg->n_ranks <= kMaxFusedRanks; }

}  // namespace

extern "C" {

size_t dq_exchange_fused_workspace_bytes(const dq_config *cfg, int64_t n_sg, const dq_plan_info *info)
{
    if (!fused_ok(cfg) || !info || n_sg < 1) return 0;
    ExchangeLayout X;
    if (!exchange_layout(cfg, 0, info, X)) return 0;
    return X.total + 256;   // + the barrier's arrival counter
}

dq_status dq_exchange_fused(const dq_config *cfg, const void *const *grads, int64_t n_sg, const float *mu,
                            const int32_t *perm, const dq_plan_info *info, void *ws, size_t ws_bytes,
                            void *const *outs, int32_t out_is_bf16, int32_t *status_dev,
                            const uint8_t **final_msgs, dq_launch_log *log, void *stream)
{
    if (!fused_ok(cfg) || !grads || !mu || !perm || !info || !ws || !outs || !status_dev || n_sg < 1 ||
        n_sg >= kMaxSG)
        return DQ_ERR_INVALID_ARG;
    if (info->n2 < 0 || info->n4 < 0 || info->n8 < 0 || info->n2 + info->n4 + info->n8 != n_sg)
        return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    ExchangeLayout X;
    if (!exchange_layout(cfg, 0, info, X)) return DQ_ERR_INVALID_ARG;
    if (ws_bytes < X.total + 256) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    if ((uintptr_t)status_dev & 3u) return DQ_ERR_ALIGNMENT;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r] || !outs[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r]) || !aligned16(outs[r])) return DQ_ERR_ALIGNMENT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t end2 = info->n2, end4 = info->n2 + info->n4;
    const bool sf = cfg->scale_fp32 != 0;
    uint8_t *w = static_cast<uint8_t *>(ws);

    std::unique_ptr<FusedRingParams> P(new FusedRingParams());
    memset(P.get(), 0, sizeof(FusedRingParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    int64_t units = 0;
    for (int32_t c = 0; c < N; ++c) {
        const int64_t a = X.lo[c], b = X.lo[c + 1];
        P->chunk[c] = msg_view(nullptr, a, b, end2, end4, sf);
        P->lo[c] = a;
        HopTask t;   // segment and unit bookkeeping of chunk c
        memset(&t, 0, sizeof(t));
        units += set_units(t, a, b, end2, end4, units);
        for (int s = 0; s < 3; ++s) {
            P->seg_lo[c][s] = t.seg_lo[s];
            P->seg_hi[c][s] = t.seg_hi[s];
            P->unit_begin[c][s] = t.unit_begin[s];
        }
        P->unit_begin[c][3] = t.unit_begin[3];
        P->grads[c] = grads[c];
        P->outs[c] = outs[c];
    }
    P->lo[N] = X.lo[N];
    P->msgs = w + X.msgs;
    P->msg_stride = (int64_t)X.msg_stride;
    P->units = units;
    P->n_ranks = N;
    P->correlated = cfg->correlated ? 1 : 0;
    P->mu = mu;
    P->perm = perm;
    P->ph = philox_keys(cfg->seed, cfg->round);
    P->out_is_bf16 = out_is_bf16 ? 1 : 0;
    P->scale_fp32 = cfg->scale_fp32;
    P->barrier = reinterpret_cast<unsigned int *>(w + X.total);
    P->status = status_dev;
    P->timeout_cycles = kBarrierTimeoutCycles;
    if (zero_words(P->barrier, 1, status_dev, st) != cudaSuccess) return DQ_ERR_CUDA;
    const LogSlot slot = log_begin(log, DQ_LAUNCH_FUSED_RING, n_sg * (N + 1), st);
    const cudaError_t e = launch_fused_ring(*P, st);
    log_end(slot, st);
    if (e != cudaSuccess) return DQ_ERR_CUDA;
    if (final_msgs)
        for (int32_t c = 0; c < N; ++c) final_msgs[c] = w + X.msgs + (size_t)(2 * c + ((N - 1) & 1)) * X.msg_stride;
    return DQ_OK;
}

size_t dq_exchange_pipelined_workspace_bytes(const dq_config *cfg, int64_t n_sg, const dq_plan_info *info)
{
    if (!fused_ok(cfg) || !info || n_sg < 1) return 0;
    ExchangeLayout X;
    if (!exchange_layout(cfg, 0, info, X)) return 0;
    return (size_t)cfg->n_ranks * (size_t)cfg->n_ranks * X.msg_stride + kWaveCounterBytes;
}

dq_status dq_exchange_pipelined(const dq_config *cfg, const void *const *grads, int64_t n_sg, const float *mu,
                                const int32_t *perm, const dq_plan_info *info, void *ws, size_t ws_bytes,
                                void *const *outs, int32_t out_is_bf16, int32_t n_parts,
                                const uint8_t **final_msgs, dq_launch_log *log, void *stream)
{
    if (!fused_ok(cfg) || !grads || !mu || !perm || !info || !ws || !outs || n_sg < 1 || n_sg >= kMaxSG ||
        n_parts < 1)
        return DQ_ERR_INVALID_ARG;
    if (info->n2 < 0 || info->n4 < 0 || info->n8 < 0 || info->n2 + info->n4 + info->n8 != n_sg)
        return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    ExchangeLayout X;
    if (!exchange_layout(cfg, 0, info, X)) return DQ_ERR_INVALID_ARG;
    const size_t msgs_bytes = (size_t)N * (size_t)N * X.msg_stride;
    if (ws_bytes < msgs_bytes + kWaveCounterBytes) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r] || !outs[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r]) || !aligned16(outs[r])) return DQ_ERR_ALIGNMENT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t end2 = info->n2, end4 = info->n2 + info->n4;
    const bool sf = cfg->scale_fp32 != 0;
    uint8_t *w = static_cast<uint8_t *>(ws);

    std::unique_ptr<WaveRingParams> P(new WaveRingParams());
    memset(P.get(), 0, sizeof(WaveRingParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    int64_t units = 0;
    for (int32_t c = 0; c < N; ++c) {
        const int64_t a = X.lo[c], b = X.lo[c + 1];
        P->chunk[c] = msg_view(nullptr, a, b, end2, end4, sf);
        P->lo[c] = a;
        HopTask t;   // segment and unit bookkeeping of chunk c
        memset(&t, 0, sizeof(t));
        units += set_units(t, a, b, end2, end4, units);
        for (int s = 0; s < 3; ++s) {
            P->seg_lo[c][s] = t.seg_lo[s];
            P->seg_hi[c][s] = t.seg_hi[s];
            P->unit_begin[c][s] = t.unit_begin[s];
        }
        P->unit_begin[c][3] = t.unit_begin[3];
        P->grads[c] = grads[c];
        P->outs[c] = outs[c];
    }
    P->lo[N] = X.lo[N];
    P->msgs = w;
    P->msg_stride = (int64_t)X.msg_stride;
    P->units = units;
    const int32_t parts = (int32_t)std::min<int64_t>(std::min<int64_t>(n_parts, kMaxWaveParts), units);
    P->n_parts = parts;
    P->n_ranks = N;
    P->correlated = cfg->correlated ? 1 : 0;
    P->mu = mu;
    P->perm = perm;
    P->ph = philox_keys(cfg->seed, cfg->round);
    P->out_is_bf16 = out_is_bf16 ? 1 : 0;
    P->scale_fp32 = cfg->scale_fp32;

    // first unit of part p, and the super-groups in units [ua, ub)
    auto part_lo = [&](int64_t p) { return units * p / parts; };
    auto sgs_in = [&](int64_t ua, int64_t ub) {
        int64_t n = 0;
        for (int32_t c = 0; c < N; ++c)
            for (int s = 0; s < 3; ++s) {
                const int64_t b0 = P->unit_begin[c][s], b1 = P->unit_begin[c][s + 1];
                const int64_t x = std::max(ua, b0), y = std::min(ub, b1);
                if (y > x)
                    n += std::min(P->seg_hi[c][s], P->seg_lo[c][s] + kUnit * (y - b0)) -
                         (P->seg_lo[c][s] + kUnit * (x - b0));
            }
        return n;
    };
    // one unit counter per launch, all zeroed here
    unsigned int *next = reinterpret_cast<unsigned int *>(w + msgs_bytes);
    if (zero_words(next, N + parts, nullptr, st) != cudaSuccess) return DQ_ERR_CUDA;
    for (int32_t t = 0; t < N + parts; ++t) {
        const int32_t plo = std::max(0, t - N + 1), phi = std::min(t, parts - 1), pd = t - N;
        P->launch = t;
        P->next = next + t;
        P->h_lo = P->h_hi = 0;
        if (plo <= phi) {
            P->h_lo = part_lo(plo);
            P->h_hi = part_lo(phi + 1);
        }
        P->d_lo = P->d_hi = 0;
        if (pd >= 0 && pd < parts) {
            P->d_lo = part_lo(pd);
            P->d_hi = part_lo(pd + 1);
        }
        const LogSlot slot =
            log_begin(log, DQ_LAUNCH_PIPELINED, sgs_in(P->h_lo, P->h_hi) + sgs_in(P->d_lo, P->d_hi), st);
        const cudaError_t e = launch_wave_ring(*P, st);
        log_end(slot, st);
        if (e != cudaSuccess) return DQ_ERR_CUDA;
    }
    if (final_msgs)
        for (int32_t c = 0; c < N; ++c) final_msgs[c] = w + ((size_t)c * N + (size_t)(N - 1)) * X.msg_stride;
    return DQ_OK;
}

}  // extern "C"

namespace {

// Bytes of one chunk message of a bucket of J super-groups, for any
// allocation: at most J super-groups of scale metadata, and at most
// 8J/N + 9 code bits per super-group-coordinate (the cut gives a chunk at
// most ceil(total/N) + 8 of the bucket's total code bits), 32 bytes each.
size_t bucket_msg_stride(int32_t N, int64_t J, bool sf)
{
    const int64_t meta = sf ? 64 * J : (J + 15) / 16 * 16 + 16 * J;
    const int64_t codes = 32 * (8 * J / N + 9) + 256;
    return round256((size_t)(meta + codes));
}

bool stream_cfg_ok(const dq_config *cfg) { return cfg_ok(cfg) && cfg->n_ranks <= kMaxStreamRanks; }

}  // namespace

extern "C" {

size_t dq_bucket_msgs_bytes(const dq_config *cfg, int64_t n_sg)
{
    if (!stream_cfg_ok(cfg) || n_sg < 1 || n_sg >= kMaxSG) return 0;
    const size_t N = (size_t)cfg->n_ranks;
    return N * N * bucket_msg_stride(cfg->n_ranks, n_sg, cfg->scale_fp32 != 0);
}

}  // extern "C"

namespace {

// Fills P (tables aside) for one launch of the bucket stream and launches it.
dq_status stream_step(const dq_config *cfg, StreamRingParams *P, const dq_bucket_step *steps, int32_t n_steps,
                      unsigned int *counter_dev, int32_t out_is_bf16, dq_launch_log *log, cudaStream_t st,
                      int32_t free_sms = 0)
{
    const int32_t N = cfg->n_ranks;
    if (n_steps < 1 || n_steps > N + 1) return DQ_ERR_INVALID_ARG;
    if (!counter_dev) return DQ_ERR_INVALID_ARG;
    if ((uintptr_t)counter_dev & 3u) return DQ_ERR_ALIGNMENT;
    const bool sf = cfg->scale_fp32 != 0;
    int decodes = 0;
    int64_t tasks = 0, sgs = 0;
    for (int32_t i = 0; i < n_steps; ++i) {
        const dq_bucket_step &b = steps[i];
        if (b.step < 0 || b.step > N || b.n_sg < 1 || b.n_sg >= kMaxSG || !b.counts_dev || !b.grads_host ||
            !b.outs_host || !b.mu || !b.perm || !b.msgs)
            return DQ_ERR_INVALID_ARG;
        if (b.step == N && ++decodes > 1) return DQ_ERR_INVALID_ARG;
        if (b.msgs_bytes < dq_bucket_msgs_bytes(cfg, b.n_sg)) return DQ_ERR_INVALID_ARG;
        if (((uintptr_t)b.counts_dev & 7u) || !aligned16(b.mu) || !aligned16(b.perm) || !aligned16(b.msgs))
            return DQ_ERR_ALIGNMENT;
        BucketSlot &S = P->slot[i];
        for (int32_t r = 0; r < N; ++r) {
            if (!b.grads_host[r] || !b.outs_host[r]) return DQ_ERR_INVALID_ARG;
            if (!aligned16(b.grads_host[r]) || !aligned16(b.outs_host[r])) return DQ_ERR_ALIGNMENT;
            S.grads[r] = b.grads_host[r];
            S.outs[r] = b.outs_host[r];
        }
        S.counts = b.counts_dev;
        S.mu = b.mu;
        S.perm = b.perm;
        S.msgs = static_cast<uint8_t *>(b.msgs);
        S.msg_stride = (int64_t)bucket_msg_stride(N, b.n_sg, sf);
        S.ph = philox_keys(cfg->seed, b.round);
        S.n_sg = (int32_t)b.n_sg;
        S.step = b.step;
        S.n_ranks = N;
        S.out_is_bf16 = out_is_bf16 ? 1 : 0;
        // grid sizing only: the units of one step (the device finds the exact count)
        const int64_t units = (b.n_sg + kUnit - 1) / kUnit + 3 * N;
        tasks += b.step == N ? units * kDecodeSub : units;
        sgs += b.n_sg;
    }
    P->n_slots = n_steps;
    P->n_ranks = N;
    P->correlated = cfg->correlated ? 1 : 0;
    P->scale_fp32 = cfg->scale_fp32;
    P->next = counter_dev;
    const LogSlot slot = log_begin(log, DQ_LAUNCH_STREAM, sgs, st);
    const cudaError_t e = launch_stream_ring(*P, tasks, st, free_sms);
    log_end(slot, st);
    return cuda_status(e);
}

// CUDA events of one dq_allreduce_stream call, destroyed when it returns
// (destruction waits for nothing: an event still pending in a stream is
// released once it completes).
struct EventPool {
    std::vector<cudaEvent_t> ev;
    ~EventPool()
    {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
    bool make(size_t n)
    {
        for (size_t i = 0; i < n; ++i) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
            ev.push_back(e);
        }
        return true;
    }
};

}  // namespace

extern "C" {

dq_status dq_exchange_stream_step(const dq_config *cfg, const dq_bucket_step *steps, int32_t n_steps,
                                  unsigned int *counter_dev, int32_t out_is_bf16, dq_launch_log *log, void *stream)
{
    if (!stream_cfg_ok(cfg) || !steps) return DQ_ERR_INVALID_ARG;
    std::unique_ptr<StreamRingParams> P(new StreamRingParams());
    memset(P.get(), 0, sizeof(StreamRingParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    return stream_step(cfg, P.get(), steps, n_steps, counter_dev, out_is_bf16, log, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// The bucket stream's driver (dq_allreduce_stream, and with host staging
// dq_allreduce_stream_io).  Host iteration t enqueues the planning of bucket
// t + lookahead (after its upload, if any) and exchange launch t.
dq_status allreduce_stream(const dq_config *cfg, const dq_bucket *buckets, const dq_bucket_io *io,
                           int32_t n_buckets, const dq_stream_set *sets, int32_t n_sets, int32_t lookahead,
                           int32_t plan_sms, unsigned int *counters_dev, int32_t out_is_bf16, int32_t *nonfinite_dev,
                           cudaStream_t cin, cudaStream_t cout, cudaStream_t ps, cudaStream_t st, dq_launch_log *log)
{
    if (!stream_cfg_ok(cfg) || !buckets || !sets || !counters_dev || n_buckets < 1) return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    if (lookahead < 1 || n_sets < N + lookahead + 1 || plan_sms < 0 || plan_sms >= sm_count()) return DQ_ERR_INVALID_ARG;
    if (((uintptr_t)counters_dev & 3u) || ((uintptr_t)nonfinite_dev & 3u)) return DQ_ERR_ALIGNMENT;
    for (int32_t k = 0; k < n_buckets; ++k)
        if (buckets[k].n_sg < 1 || buckets[k].n_sg >= kMaxSG || !buckets[k].grads_host || !buckets[k].outs_host)
            return DQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_sets; ++i)
        if (!sets[i].mu || !sets[i].perm || !sets[i].plan_ws || !sets[i].msgs) return DQ_ERR_INVALID_ARG;
    // host staging: which earlier bucket last read each device gradient
    // buffer (up to the launch of its last ring step), and which earlier
    // download last read each output buffer a decode writes; the reuse
    // waits for it, and an upload must be enqueued after that launch
    const int64_t out_elem = out_is_bf16 ? 2 : 4;
    std::vector<int32_t> reads_done_by((size_t)n_buckets, -1), out_prev((size_t)n_buckets, -1);
    if (io) {
        std::unordered_map<const void *, int32_t> last_grad, last_out;
        for (int32_t k = 0; k < n_buckets; ++k) {
            if (io[k].src_host) {
                for (int32_t r = 0; r < N; ++r) {
                    if (!io[k].src_host[r] || !buckets[k].grads_host[r]) return DQ_ERR_INVALID_ARG;
                    auto it = last_grad.find(buckets[k].grads_host[r]);
                    if (it != last_grad.end()) {
                        // that bucket's last read (launch b + N - 1) precedes this planning's enqueue (k - lookahead)
                        if (it->second + N - 1 >= k - lookahead) return DQ_ERR_INVALID_ARG;
                        reads_done_by[k] = std::max(reads_done_by[k], it->second);
                    }
                }
            }
            for (int32_t r = 0; r < N; ++r) last_grad[buckets[k].grads_host[r]] = k;
            // any output this bucket's decode writes may be a buffer an earlier download still reads
            for (int32_t r = 0; r < N; ++r) {
                auto it = last_out.find(buckets[k].outs_host[r]);
                if (it != last_out.end()) out_prev[k] = std::max(out_prev[k], it->second);
            }
            if (io[k].dst_host) {
                if (!buckets[k].outs_host[0]) return DQ_ERR_INVALID_ARG;
                last_out[buckets[k].outs_host[0]] = k;
            }
        }
    }
    const int32_t R = n_sets;   // ring of events per kind (a wait on a later record of a slot waits longer, never less)
    EventPool E;   // per set: planned, free again; rings: uploaded, last read, decoded, downloaded; the call's start; the end
    if (!E.make(2 * (size_t)n_sets + (io ? 4 * (size_t)R : 0) + 2)) return DQ_ERR_CUDA;
    auto ev_plan = [&](int32_t i) { return E.ev[2 * i]; };
    auto ev_free = [&](int32_t i) { return E.ev[2 * i + 1]; };
    auto ev_up = [&](int32_t k) { return E.ev[2 * n_sets + (k % R)]; };
    auto ev_read = [&](int32_t k) { return E.ev[2 * n_sets + R + (k % R)]; };
    auto ev_dec = [&](int32_t k) { return E.ev[2 * n_sets + 2 * R + (k % R)]; };
    auto ev_out = [&](int32_t k) { return E.ev[2 * n_sets + 3 * R + (k % R)]; };
    cudaEvent_t ev_start = E.ev[E.ev.size() - 2], ev_end = E.ev.back();
    // the pass's non-finite flag is cleared before any planning starts
    if (nonfinite_dev && zero_words(nonfinite_dev, 1, nullptr, st) != cudaSuccess) return DQ_ERR_CUDA;
    // the other streams start after everything already enqueued on `stream`
    // (earlier work may still use the sets, the staging or the outputs)
    if (cudaEventRecord(ev_start, st) != cudaSuccess) return DQ_ERR_CUDA;
    for (cudaStream_t o : {ps, cin, cout})
        if (io && o != st && cudaStreamWaitEvent(o, ev_start, 0) != cudaSuccess) return DQ_ERR_CUDA;
    if (!io && ps != st && cudaStreamWaitEvent(ps, ev_start, 0) != cudaSuccess) return DQ_ERR_CUDA;
    std::unique_ptr<StreamRingParams> P(new StreamRingParams());
    memset(P.get(), 0, sizeof(StreamRingParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    if (zero_many(counters_dev, (int64_t)n_buckets + N, st) != cudaSuccess) return DQ_ERR_CUDA;
    std::vector<const int64_t *> counts((size_t)n_buckets, nullptr);
    std::vector<uint8_t> used((size_t)n_sets, 0);
    auto upload = [&](int32_t k) -> dq_status {
        if (!io || !io[k].src_host) return DQ_OK;
        if (reads_done_by[k] >= 0 && cudaStreamWaitEvent(cin, ev_read(reads_done_by[k]), 0) != cudaSuccess)
            return DQ_ERR_CUDA;
        const size_t bytes = (size_t)buckets[k].n_sg * kSG * 2;
        for (int32_t r = 0; r < N; ++r)
            if (cudaMemcpyAsync(const_cast<void *>(buckets[k].grads_host[r]), io[k].src_host[r], bytes,
                                cudaMemcpyHostToDevice, cin) != cudaSuccess)
                return DQ_ERR_CUDA;
        if (cudaEventRecord(ev_up(k), cin) != cudaSuccess || cudaStreamWaitEvent(ps, ev_up(k), 0) != cudaSuccess)
            return DQ_ERR_CUDA;
        return DQ_OK;
    };
    auto plan = [&](int32_t k) -> dq_status {
        const int32_t si = k % n_sets;
        if (used[si] && cudaStreamWaitEvent(ps, ev_free(si), 0) != cudaSuccess) return DQ_ERR_CUDA;
        used[si] = 1;
        dq_status s = upload(k);
        if (s != DQ_OK) return s;
        dq_config c = *cfg;
        c.round = buckets[k].round;
        PlanDev d;
        const dq_stream_set &S = sets[si];
        s = plan_enqueue(&c, buckets[k].grads_host, buckets[k].n_sg, S.mu, S.perm, S.plan_ws, S.plan_ws_bytes,
                         nullptr, log, ps, d, nonfinite_dev);
        if (s != DQ_OK) return s;
        counts[k] = d.counts;
        return cudaEventRecord(ev_plan(si), ps) == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
    };
    dq_status s = DQ_OK;
    for (int32_t k = 0; k < std::min(lookahead, n_buckets); ++k)
        if ((s = plan(k)) != DQ_OK) return s;
    dq_bucket_step steps[kMaxStreamRanks + 1];
    for (int32_t t = 0; t < n_buckets + N; ++t) {
        if (t + lookahead < n_buckets && (s = plan(t + lookahead)) != DQ_OK) return s;
        if (t < n_buckets && cudaStreamWaitEvent(st, ev_plan(t % n_sets), 0) != cudaSuccess) return DQ_ERR_CUDA;
        // this launch decodes bucket t - N: a download of its rank-0 output buffer still in flight comes first
        if (io && t >= N && out_prev[t - N] >= 0 && cudaStreamWaitEvent(st, ev_out(out_prev[t - N]), 0) != cudaSuccess)
            return DQ_ERR_CUDA;
        int32_t n = 0;
        for (int32_t b = std::max(0, t - N); b <= std::min(t, n_buckets - 1); ++b) {
            const dq_stream_set &S = sets[b % n_sets];
            steps[n++] = dq_bucket_step{buckets[b].n_sg, counts[b], buckets[b].grads_host, buckets[b].outs_host,
                                        S.mu, S.perm, S.msgs, S.msgs_bytes, buckets[b].round, t - b};
        }
        if ((s = stream_step(cfg, P.get(), steps, n, counters_dev + t, out_is_bf16, log, st, plan_sms)) != DQ_OK)
            return s;
        if (t >= N && cudaEventRecord(ev_free((t - N) % n_sets), st) != cudaSuccess) return DQ_ERR_CUDA;
        if (!io) continue;
        // bucket t - N + 1 ran its last ring step: its gradients are no longer read
        if (t - N + 1 >= 0 && t - N + 1 < n_buckets && cudaEventRecord(ev_read(t - N + 1), st) != cudaSuccess)
            return DQ_ERR_CUDA;
        const int32_t b = t - N;   // decoded by this launch
        if (b >= 0 && io[b].dst_host) {
            if (cudaEventRecord(ev_dec(b), st) != cudaSuccess || cudaStreamWaitEvent(cout, ev_dec(b), 0) != cudaSuccess ||
                cudaMemcpyAsync(io[b].dst_host, buckets[b].outs_host[0], (size_t)buckets[b].n_sg * kSG * out_elem,
                                cudaMemcpyDeviceToHost, cout) != cudaSuccess ||
                cudaEventRecord(ev_out(b), cout) != cudaSuccess)
                return DQ_ERR_CUDA;
        }
    }
    // `stream` covers the whole call: the downloads join it at the end
    if (io && cout != st &&
        (cudaEventRecord(ev_end, cout) != cudaSuccess || cudaStreamWaitEvent(st, ev_end, 0) != cudaSuccess))
        return DQ_ERR_CUDA;
    return DQ_OK;
}

}  // namespace

extern "C" {

dq_status dq_allreduce_stream(const dq_config *cfg, const dq_bucket *buckets, int32_t n_buckets,
                              const dq_stream_set *sets, int32_t n_sets, int32_t lookahead, int32_t plan_sms,
                              unsigned int *counters_dev, int32_t out_is_bf16, int32_t *nonfinite_dev,
                              void *plan_stream, void *stream, dq_launch_log *log)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t ps = plan_stream ? static_cast<cudaStream_t>(plan_stream) : st;
    return allreduce_stream(cfg, buckets, nullptr, n_buckets, sets, n_sets, lookahead, plan_sms, counters_dev,
                            out_is_bf16, nonfinite_dev, st, st, ps, st, log);
}

dq_status dq_allreduce_stream_io(const dq_config *cfg, const dq_bucket *buckets, const dq_bucket_io *io,
                                 int32_t n_buckets, const dq_stream_set *sets, int32_t n_sets, int32_t lookahead,
                                 int32_t plan_sms, unsigned int *counters_dev, int32_t out_is_bf16,
                                 int32_t *nonfinite_dev, void *copy_in_stream, void *copy_out_stream,
                                 void *plan_stream, void *stream, dq_launch_log *log)
{
    if (!io) return DQ_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t ps = plan_stream ? static_cast<cudaStream_t>(plan_stream) : st;
    cudaStream_t cin = copy_in_stream ? static_cast<cudaStream_t>(copy_in_stream) : ps;
    cudaStream_t cout = copy_out_stream ? static_cast<cudaStream_t>(copy_out_stream) : st;
    return allreduce_stream(cfg, buckets, io, n_buckets, sets, n_sets, lookahead, plan_sms, counters_dev, out_is_bf16,
                            nonfinite_dev, cin, cout, ps, st, log);
}

dq_status dq_get_device_status(const int32_t *status_dev, int32_t *status_host, void *stream)
{
    if (!status_dev || !status_host) return DQ_ERR_INVALID_ARG;
    if ((uintptr_t)status_dev & 3u) return DQ_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PlanReadback *buf = plan_readback_buffer();
    if (!buf) return DQ_ERR_CUDA;
    PlanReadback *dev = nullptr;
    if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&dev), buf, 0) != cudaSuccess) return DQ_ERR_CUDA;
    status_readback_kernel<<<1, 32, 0, st>>>(status_dev, &dev->status);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return DQ_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DQ_ERR_CUDA;
    *status_host = *reinterpret_cast<volatile int32_t *>(&buf->status);
    return DQ_OK;
}

dq_status dq_barrier_selftest(int32_t n_blocks, int32_t missing, int64_t timeout_cycles, void *scratch,
                              int32_t *status_dev, void *stream)
{
    if (n_blocks < 1 || n_blocks > 1024 || missing < 0 || missing > 1024 || timeout_cycles < 1 ||
        timeout_cycles > 4 * kBarrierTimeoutCycles || !scratch || !status_dev)
        return DQ_ERR_INVALID_ARG;
    if (((uintptr_t)scratch & 3u) || ((uintptr_t)status_dev & 3u)) return DQ_ERR_ALIGNMENT;
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return DQ_ERR_CUDA;
    if (n_blocks > sm_count()) return DQ_ERR_INVALID_ARG;   // one small CTA per SM at most: all resident
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int *counter = static_cast<unsigned int *>(scratch);
    if (zero_words(counter, 1, status_dev, st) != cudaSuccess) return DQ_ERR_CUDA;
    return cuda_status(launch_barrier_selftest(n_blocks, missing, (long long)timeout_cycles, counter, status_dev, st));
}

}  // extern "C"

// Kernel parameters are limited to 32,764 bytes.
static_assert(sizeof(dq::HopParams) <= 32764, "HopParams exceeds the kernel parameter limit");
static_assert(sizeof(dq::DecodeParams) <= 32764, "DecodeParams exceeds the kernel parameter limit");
static_assert(sizeof(dq::FusedRingParams) <= 32764, "FusedRingParams exceeds the kernel parameter limit");
static_assert(sizeof(dq::WaveRingParams) <= 32764, "WaveRingParams exceeds the kernel parameter limit");
static_assert(sizeof(dq::StreamRingParams) <= 32764, "StreamRingParams exceeds the kernel parameter limit");
