// dq_api.cu -- the C ABI of libdq: argument validation, level tables,
// message layout, single-call entry points and the N-rank schedule.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

#include "dq_common.cuh"
#include "dq_internal.h"

namespace dq {

// --------------------------------------------------------------------------- device info
static std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int sm_count()
{
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 152;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
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

// {q_k, G_k} with G_k = fl(1/fl(q_{k+1} - q_k)), G of the top level 0,
// sentinel {+inf, 0}; bucket table for t = 0 .. 2H (H the smallest power of
// two with 1/H <= min gap, capped at hmax; with the cap a bucket may hold
// more than one level and the kernel's exact compares walk over them).
static void fill_bitwidth(int bits, double eps, float2 *qg, BucketEntry *bk, int32_t *H_out, int hmax)
{
    const int L = 1 << bits;
    float q[256];
    levels(bits, eps, q);
    float min_gap = INFINITY;
    for (int k = 0; k < L; ++k) {
        float G = 0.0f;
        if (k + 1 < L) {
            const float gap = q[k + 1] - q[k];
            G = 1.0f / gap;
            if (gap < min_gap) min_gap = gap;
        }
        qg[k] = make_float2(q[k], G);
    }
    qg[L] = make_float2(INFINITY, 0.0f);
    int H = 2;
    while (H < hmax && 1.0 / (double)H > (double)min_gap) H *= 2;
    *H_out = H;
    for (int t = 0; t <= 2 * H; ++t) {
        const double edge = (double)t / (double)H - 1.0;
        int kb = 0;
        for (int k = 0; k < L; ++k)
            if ((double)q[k] <= edge) kb = k;
        bk[t].kb = kb;
        bk[t].boundary = kb + 1 < L ? q[kb + 1] : INFINITY;
    }
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
        fill_bitwidth(2, eps, t->qg2, t->bk2, &t->H2, kMaxH2);
        fill_bitwidth(4, eps, t->qg4, t->bk4, &t->H4, kMaxH4);
        fill_bitwidth(8, eps, t->qg8, t->bk8, &t->H8, kMaxH8);
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

size_t msg_bytes(int64_t c, int64_t n2, int64_t n4, int64_t n8)
{
    return (size_t)((c + 15) / 16 * 16 + 16 * c + 64 * n2 + 128 * n4 + 256 * n8);
}

MsgView msg_view(uint8_t *base, int64_t lo, int64_t hi, int64_t end2, int64_t end4)
{
    MsgView m;
    m.base = base;
    m.c = hi - lo;
    m.n2 = overlap(lo, hi, 0, end2);
    m.n4 = overlap(lo, hi, end2, end4);
    m.off_u = (m.c + 15) / 16 * 16;
    m.off_c2 = m.off_u + 16 * m.c;
    m.off_c4 = m.off_c2 + 64 * m.n2;
    m.off_c8 = m.off_c4 + 128 * m.n4;
    return m;
}

}  // namespace dq

using namespace dq;

// --------------------------------------------------------------------------- validation helpers
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
    return c && c->n_ranks >= 1 && c->n_ranks <= 65535 && (c->eps > 0.0);
}

dq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DQ_OK : DQ_ERR_CUDA; }

bool stage_ok(const dq_config *cfg, const dq_stage &s)
{
    return s.rank >= 0 && s.rank < cfg->n_ranks && s.hop >= 0 && s.hop <= 0xFFFF && s.n_slots >= 1 &&
           s.n_slots <= 65536 && s.slot >= 0 && s.slot < s.n_slots;
}

// Generator counter word 1 and the correlated-rounding offset of a stage:
// independent rounding keys the stream by (hop, rank); correlated rounding
// shares one stream per hop (rank field 0xFFFF, above any rank) and shifts
// it by floor(slot * 2^16 / n_slots).
HopTask make_task(const dq_config *cfg, const dq_stage &s)
{
    HopTask t;
    memset(&t, 0, sizeof(t));
    if (cfg->correlated) {
        t.stage_word = (uint32_t)s.hop | (0xFFFFu << 16);
        t.corr_off = (uint32_t)(((uint64_t)(uint32_t)s.slot << 16) / (uint64_t)(uint32_t)s.n_slots);
    } else {
        t.stage_word = (uint32_t)s.hop | ((uint32_t)s.rank << 16);
        t.corr_off = 0u;
    }
    return t;
}

void fill_common(HopParams &P, const dq_config *cfg, const float *M, const int32_t *perm, int64_t end2,
                 int64_t end4)
{
    P.n_ranks = cfg->n_ranks;
    P.end2 = end2;
    P.end4 = end4;
    P.M = M;
    P.perm = perm;
    P.key0 = (uint32_t)cfg->seed;
    P.key1 = (uint32_t)(cfg->seed >> 32);
    P.round0 = (uint32_t)cfg->round;
    P.round1 = (uint32_t)(cfg->round >> 32);
}

}  // namespace

// --------------------------------------------------------------------------- single-call entry points
extern "C" {

const char *dq_version(void) { return "libdq 0.1 (sm_103a)"; }

uint64_t dq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *dq_status_string(dq_status s)
{
    switch (s) {
    case DQ_OK: return "ok";
    case DQ_ERR_INVALID_ARG: return "invalid argument";
    case DQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case DQ_ERR_BUDGET_INFEASIBLE: return "budget below 2 bits per coordinate";
    case DQ_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

size_t dq_message_bytes(dq_range r)
{
    if (!range_ok(r)) return 0;
    const MsgView m = msg_view(nullptr, r.lo, r.hi, r.end2, r.end4);
    return msg_bytes(m.c, m.n2, m.n4, m.c - m.n2 - m.n4);
}

dq_status dq_level_table(int32_t bits, double eps, float *q_host)
{
    if ((bits != 2 && bits != 4 && bits != 8) || !q_host) return DQ_ERR_INVALID_ARG;
    Tables t;
    if (!build_tables(eps, &t)) return DQ_ERR_INVALID_ARG;
    const float2 *qg = bits == 2 ? t.qg2 : (bits == 4 ? t.qg4 : t.qg8);
    for (int k = 0; k < (1 << bits); ++k) q_host[k] = qg[k].x;
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

dq_status dq_stats_reduce(const float *mean_all, const float *sq_all, int32_t n_ranks, int64_t n_sg,
                          float *M, float *F, void *stream)
{
    if (n_sg < 0 || n_sg >= kMaxSG || n_ranks < 1) return DQ_ERR_INVALID_ARG;
    if (n_sg == 0) return DQ_OK;
    if (!mean_all || !sq_all || !M || !F) return DQ_ERR_INVALID_ARG;
    return cuda_status(launch_stats_reduce(mean_all, sq_all, n_ranks, n_sg, M, F,
                                           static_cast<cudaStream_t>(stream)));
}

size_t dq_workspace_bytes(int64_t n_sg) { return plan_scratch_bytes(n_sg < 0 ? 0 : n_sg); }

dq_status dq_allocate(const float *F, int64_t n_sg, float budget, uint8_t *b, float *T_dev,
                      int64_t *counts_dev, void *ws, size_t ws_bytes, void *stream)
{
    if (n_sg < 1 || n_sg >= kMaxSG) return DQ_ERR_INVALID_ARG;
    if (!F || !b || !T_dev || !counts_dev || !ws) return DQ_ERR_INVALID_ARG;
    if (!(budget >= 2.0f)) return DQ_ERR_BUDGET_INFEASIBLE;
    if (ws_bytes < plan_scratch_bytes(n_sg)) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws) || ((uintptr_t)counts_dev & 7u)) return DQ_ERR_ALIGNMENT;
    // floor(B * J) is exact in binary64 for J < 2^27
    const int64_t cap = (int64_t)floor((double)budget * (double)n_sg);
    return cuda_status(launch_allocate(F, n_sg, cap, b, T_dev, counts_dev, ws,
                                       static_cast<cudaStream_t>(stream)));
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

dq_status dq_compress(const dq_config *cfg, dq_range r, dq_stage stage, const void *g_bf16, const float *M,
                      const int32_t *perm, uint8_t *msg_out, void *stream)
{
    if (!cfg_ok(cfg) || !range_ok(r) || !stage_ok(cfg, stage)) return DQ_ERR_INVALID_ARG;
    if (r.hi == r.lo) return DQ_OK;
    if (!g_bf16 || !M || !perm || !msg_out) return DQ_ERR_INVALID_ARG;
    if (!aligned16(g_bf16) || !aligned16(msg_out)) return DQ_ERR_ALIGNMENT;
    std::unique_ptr<HopParams> P(new HopParams());
    memset(P.get(), 0, sizeof(HopParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    fill_common(*P, cfg, M, perm, r.end2, r.end4);
    HopTask t = make_task(cfg, stage);
    t.out = msg_view(msg_out, r.lo, r.hi, r.end2, r.end4);
    t.addend = g_bf16;
    t.in_lo = r.lo;
    t.send_lo = r.lo;
    t.send_hi = r.hi;
    t.keep_lo = t.keep_hi = r.hi;
    t.sg_begin = 0;
    P->task[0] = t;
    P->n_tasks = 1;
    P->total_sg = r.hi - r.lo;
    return cuda_status(launch_hop(*P, false, false, static_cast<cudaStream_t>(stream)));
}

dq_status dq_dar(const dq_config *cfg, dq_range in, dq_stage stage, const uint8_t *msg_in, const void *addend,
                 int32_t addend_is_fp32, const float *M, const int32_t *perm, dq_range send, uint8_t *msg_out,
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
    if (!msg_in || !addend || !M || !perm) return DQ_ERR_INVALID_ARG;
    if ((ns > 0 && !msg_out) || (nk > 0 && !keep_out)) return DQ_ERR_INVALID_ARG;
    if (!aligned16(msg_in) || !aligned16(addend) || (ns > 0 && !aligned16(msg_out)) ||
        (nk > 0 && !aligned16(keep_out)))
        return DQ_ERR_ALIGNMENT;
    std::unique_ptr<HopParams> P(new HopParams());
    memset(P.get(), 0, sizeof(HopParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    fill_common(*P, cfg, M, perm, in.end2, in.end4);
    HopTask t = make_task(cfg, stage);
    t.in = msg_view(const_cast<uint8_t *>(msg_in), in.lo, in.hi, in.end2, in.end4);
    t.out = msg_view(msg_out, send.lo, send.hi, send.end2, send.end4);
    t.addend = addend;
    t.keep_out = keep_out;
    t.in_lo = in.lo;
    t.send_lo = ns > 0 ? send.lo : in.hi;
    t.send_hi = ns > 0 ? send.hi : in.hi;
    t.keep_lo = nk > 0 ? keep.lo : in.hi;
    t.keep_hi = nk > 0 ? keep.hi : in.hi;
    t.sg_begin = 0;
    P->task[0] = t;
    P->n_tasks = 1;
    P->total_sg = ni;
    return cuda_status(launch_hop(*P, true, addend_is_fp32 != 0, static_cast<cudaStream_t>(stream)));
}

dq_status dq_decode(const dq_config *cfg, dq_range r, const uint8_t *msg, const float *M, const int32_t *perm,
                    void *out, int32_t out_is_bf16, void *stream)
{
    if (!cfg_ok(cfg) || !range_ok(r)) return DQ_ERR_INVALID_ARG;
    if (r.hi == r.lo) return DQ_OK;
    if (!msg || !M || !perm || !out) return DQ_ERR_INVALID_ARG;
    if (!aligned16(msg) || !aligned16(out)) return DQ_ERR_ALIGNMENT;
    std::unique_ptr<DecodeParams> P(new DecodeParams());
    memset(P.get(), 0, sizeof(DecodeParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    P->n_ranks = cfg->n_ranks;
    P->end2 = r.end2;
    P->end4 = r.end4;
    P->M = M;
    P->perm = perm;
    P->out = out;
    P->out_is_bf16 = out_is_bf16 ? 1 : 0;
    P->task[0].msg = msg_view(const_cast<uint8_t *>(msg), r.lo, r.hi, r.end2, r.end4);
    P->task[0].lo = r.lo;
    P->task[0].sg_begin = 0;
    P->n_tasks = 1;
    P->total_sg = r.hi - r.lo;
    return cuda_status(launch_decode(*P, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// --------------------------------------------------------------------------- N-rank schedule
namespace {

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

struct PlanLayout {
    size_t mean_all, sq_all, F, b, T, counts, scratch, total;
};

PlanLayout plan_layout(int32_t n, int64_t J)
{
    PlanLayout L;
    size_t o = 0;
    L.mean_all = o; o += round256(sizeof(float) * (size_t)n * (size_t)J);
    L.sq_all = o;   o += round256(sizeof(float) * (size_t)n * (size_t)J);
    L.F = o;        o += round256(sizeof(float) * (size_t)J);
    L.b = o;        o += round256((size_t)J);
    L.T = o;        o += 256;
    L.counts = o;   o += 256;
    L.scratch = o;  o += round256(plan_scratch_bytes(J));
    L.total = o;
    return L;
}

// Chunk sets of the butterfly: at step s rank r holds chunks
// [base, base + 2^(L-s)), base = (r >> (L-s)) << (L-s); it keeps the half
// whose bit (L-1-s) equals its own and sends the other half.
struct ChunkSpan { int32_t a, b; };

ChunkSpan bfly_keep(int32_t L, int32_t s, int32_t r)
{
    const int32_t width = 1 << (L - s), half = width >> 1, base = (r >> (L - s)) << (L - s);
    const int32_t my = (r >> (L - 1 - s)) & 1;
    return {base + my * half, base + my * half + half};
}

ChunkSpan bfly_send(int32_t L, int32_t s, int32_t r)
{
    const int32_t width = 1 << (L - s), half = width >> 1, base = (r >> (L - s)) << (L - s);
    const int32_t my = (r >> (L - 1 - s)) & 1;
    return {base + (1 - my) * half, base + (1 - my) * half + half};
}

int32_t log2_exact(int32_t n)
{
    int32_t L = 0;
    while ((1 << L) < n) ++L;
    return (1 << L) == n ? L : -1;
}

struct ExchangeLayout {
    std::vector<int64_t> lo;    // chunk cuts
    size_t msg_stride = 0;      // bytes per message buffer
    size_t keep_stride = 0;     // bytes per fp32 keep buffer
    size_t msgs = 0, keeps = 0, finals = 0, total = 0;
    int32_t L = 0;
};

bool exchange_layout(const dq_config *cfg, int32_t butterfly, int64_t J, const dq_plan_info *info,
                     ExchangeLayout &X)
{
    const int32_t N = cfg->n_ranks;
    X.lo.assign((size_t)N + 1, 0);
    if (dq_chunk_cuts(info->n2, info->n4, info->n8, N, X.lo.data()) != DQ_OK) return false;
    const int64_t end2 = info->n2, end4 = info->n2 + info->n4;
    auto bytes = [&](int64_t a, int64_t b) {
        const MsgView m = msg_view(nullptr, a, b, end2, end4);
        return msg_bytes(m.c, m.n2, m.n4, m.c - m.n2 - m.n4);
    };
    size_t mmax = 16, kmax = 16;
    for (int32_t c = 0; c < N; ++c) mmax = std::max(mmax, bytes(X.lo[c], X.lo[c + 1]));
    if (butterfly) {
        X.L = log2_exact(N);
        if (X.L < 0) return false;
        for (int32_t s = 0; s < X.L; ++s)
            for (int32_t r = 0; r < N; ++r) {
                const ChunkSpan S = bfly_send(X.L, s, r), K = bfly_keep(X.L, s, r);
                mmax = std::max(mmax, bytes(X.lo[S.a], X.lo[S.b]));
                kmax = std::max(kmax, (size_t)(X.lo[K.b] - X.lo[K.a]) * kSG * sizeof(float));
            }
    }
    X.msg_stride = round256(mmax);
    X.keep_stride = butterfly ? round256(kmax) : 0;
    size_t o = 0;
    X.msgs = o;   o += 2 * (size_t)N * X.msg_stride;
    X.keeps = o;  o += 2 * (size_t)N * X.keep_stride;
    X.finals = o; o += butterfly ? (size_t)N * X.msg_stride : 0;
    X.total = o;
    (void)J;
    return true;
}

// Brackets one launch with the caller's events (if a log has room).
struct LogSlot {
    dq_launch_log *log;
    int32_t i;
};

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

// Launches a batch of hop tasks (split into launches of at most kMaxTasks).
cudaError_t run_hops(HopParams &P, std::vector<HopTask> &tasks, bool has_in, bool add_f32, cudaStream_t st,
                     dq_launch_log *log)
{
    size_t i = 0;
    while (i < tasks.size()) {
        int n = 0;
        int64_t total = 0;
        while (i < tasks.size() && n < kMaxTasks) {
            HopTask t = tasks[i++];
            const int64_t cnt = (t.send_hi - t.send_lo) + (t.keep_hi - t.keep_lo);
            if (cnt <= 0) continue;
            t.sg_begin = total;
            total += cnt;
            P.task[n++] = t;
        }
        P.n_tasks = n;
        P.total_sg = total;
        if (n > 0) {
            const LogSlot slot = log_begin(log, has_in ? DQ_LAUNCH_DAR : DQ_LAUNCH_COMPRESS, total, st);
            const cudaError_t e = launch_hop(P, has_in, add_f32, st);
            log_end(slot, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t dq_plan_workspace_bytes(int32_t n_ranks, int64_t n_sg)
{
    if (n_ranks < 1 || n_sg < 1) return 0;
    return plan_layout(n_ranks, n_sg).total;
}

dq_status dq_plan(const dq_config *cfg, const void *const *grads, int64_t n_sg, float *M, int32_t *perm,
                  void *ws, size_t ws_bytes, dq_plan_info *info, void *stream)
{
    if (!cfg_ok(cfg) || !grads || !M || !perm || !ws || !info || n_sg < 1 || n_sg >= kMaxSG)
        return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    const PlanLayout L = plan_layout(N, n_sg);
    if (ws_bytes < L.total) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    if (!(cfg->budget_bits >= 2.0f)) return DQ_ERR_BUDGET_INFEASIBLE;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r])) return DQ_ERR_ALIGNMENT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    float *mean_all = reinterpret_cast<float *>(w + L.mean_all);
    float *sq_all = reinterpret_cast<float *>(w + L.sq_all);
    float *F = reinterpret_cast<float *>(w + L.F);
    uint8_t *b = w + L.b;
    float *T = reinterpret_cast<float *>(w + L.T);
    int64_t *counts = reinterpret_cast<int64_t *>(w + L.counts);
    void *scratch = w + L.scratch;
    for (int32_t r = 0; r < N; ++r) {
        const cudaError_t e = launch_stats(static_cast<const uint16_t *>(grads[r]), n_sg,
                                           mean_all + (size_t)r * n_sg, sq_all + (size_t)r * n_sg, st);
        if (e != cudaSuccess) return DQ_ERR_CUDA;
    }
    if (launch_stats_reduce(mean_all, sq_all, N, n_sg, M, F, st) != cudaSuccess) return DQ_ERR_CUDA;
    dq_status s = dq_allocate(F, n_sg, cfg->budget_bits, b, T, counts, scratch, plan_scratch_bytes(n_sg), stream);
    if (s != DQ_OK) return s;
    s = dq_reorder(b, n_sg, perm, scratch, plan_scratch_bytes(n_sg), stream);
    if (s != DQ_OK) return s;
    int64_t hc[3];
    float hT = 0.0f;
    if (cudaMemcpyAsync(hc, counts, sizeof(hc), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DQ_ERR_CUDA;
    if (cudaMemcpyAsync(&hT, T, sizeof(hT), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DQ_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DQ_ERR_CUDA;
    info->T = hT;
    info->n2 = hc[0];
    info->n4 = hc[1];
    info->n8 = hc[2];
    return DQ_OK;
}

size_t dq_exchange_workspace_bytes(const dq_config *cfg, int32_t butterfly, int64_t n_sg, const dq_plan_info *info)
{
    if (!cfg_ok(cfg) || !info) return 0;
    ExchangeLayout X;
    if (!exchange_layout(cfg, butterfly, n_sg, info, X)) return 0;
    return X.total;
}

dq_status dq_exchange(const dq_config *cfg, int32_t butterfly, const void *const *grads, int64_t n_sg,
                      const float *M, const int32_t *perm, const dq_plan_info *info, void *ws, size_t ws_bytes,
                      void *const *outs, int32_t out_is_bf16, const uint8_t **final_msgs, dq_launch_log *log,
                      void *stream)
{
    if (!cfg_ok(cfg) || !grads || !M || !perm || !info || !ws || !outs || n_sg < 1 || n_sg >= kMaxSG)
        return DQ_ERR_INVALID_ARG;
    if (info->n2 < 0 || info->n4 < 0 || info->n8 < 0 || info->n2 + info->n4 + info->n8 != n_sg)
        return DQ_ERR_INVALID_ARG;
    const int32_t N = cfg->n_ranks;
    ExchangeLayout X;
    if (!exchange_layout(cfg, butterfly, n_sg, info, X)) return DQ_ERR_INVALID_ARG;
    if (ws_bytes < X.total) return DQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DQ_ERR_ALIGNMENT;
    for (int32_t r = 0; r < N; ++r) {
        if (!grads[r] || !outs[r]) return DQ_ERR_INVALID_ARG;
        if (!aligned16(grads[r]) || !aligned16(outs[r])) return DQ_ERR_ALIGNMENT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t end2 = info->n2, end4 = info->n2 + info->n4;
    uint8_t *w = static_cast<uint8_t *>(ws);
    auto msg = [&](int32_t r, int32_t par) { return w + X.msgs + (size_t)(2 * r + par) * X.msg_stride; };
    auto keepb = [&](int32_t r, int32_t par) {
        return reinterpret_cast<float *>(w + X.keeps + (size_t)(2 * r + par) * X.keep_stride);
    };
    auto finb = [&](int32_t r) { return w + X.finals + (size_t)r * X.msg_stride; };
    const std::vector<int64_t> &lo = X.lo;

    std::unique_ptr<HopParams> P(new HopParams());
    memset(P.get(), 0, sizeof(HopParams));
    if (!build_tables(cfg->eps, &P->tab)) return DQ_ERR_INVALID_ARG;
    fill_common(*P, cfg, M, perm, end2, end4);

    // A task over SG range [a, b): send [sa, sb) to `out`, keep [ka, kb) to `keep`.
    auto task = [&](dq_stage stage, const uint8_t *in, int64_t a, int64_t b, const void *addend, uint8_t *out,
                    int64_t sa, int64_t sb, float *keep, int64_t ka, int64_t kb) {
        HopTask t = make_task(cfg, stage);
        t.in = msg_view(const_cast<uint8_t *>(in), a, b, end2, end4);
        t.out = msg_view(out, sa, sb, end2, end4);
        t.addend = addend;
        t.keep_out = keep;
        t.in_lo = a;
        t.send_lo = sb > sa ? sa : b;
        t.send_hi = sb > sa ? sb : b;
        t.keep_lo = kb > ka ? ka : b;
        t.keep_hi = kb > ka ? kb : b;
        return t;
    };

    std::vector<const uint8_t *> fin((size_t)N, nullptr);
    std::vector<HopTask> tasks;
    cudaError_t e = cudaSuccess;
    if (!butterfly) {
        // Ring reduce-scatter: at step t rank r handles chunk (r - 1 - t) mod N;
        // step 0 compresses it, later steps decode the message of rank r - 1,
        // add the local gradient and recompress (stage t, quantizing rank r).
        for (int32_t t = 0; t < N && e == cudaSuccess; ++t) {
            tasks.clear();
            for (int32_t r = 0; r < N; ++r) {
                const int32_t c = (int32_t)((((int64_t)r - 1 - t) % N + N) % N);
                const int32_t src = (r - 1 + N) % N;
                tasks.push_back(task(dq_stage{r, t, 0, 1}, t ? msg(src, (t - 1) & 1) : nullptr, lo[c], lo[c + 1], grads[r],
                                     msg(r, t & 1), lo[c], lo[c + 1], nullptr, 0, 0));
            }
            e = run_hops(*P, tasks, t > 0, false, st, log);
        }
        for (int32_t c = 0; c < N; ++c) fin[c] = msg(c, (N - 1) & 1);  // owner c, step N-1
    } else {
        const int32_t L = X.L;
        if (L == 0) {
            tasks.push_back(task(dq_stage{0, 0, 0, 1}, nullptr, lo[0], lo[1], grads[0], finb(0), lo[0], lo[1], nullptr, 0, 0));
            e = run_hops(*P, tasks, false, false, st, log);
        } else {
            // step 0: compress the half that is sent
            for (int32_t r = 0; r < N; ++r) {
                const ChunkSpan S = bfly_send(L, 0, r);
                const int32_t ns = 1 << (L - 1);
                tasks.push_back(task(dq_stage{r, 0, r & (ns - 1), ns}, nullptr, lo[S.a], lo[S.b], grads[r], msg(r, 0), lo[S.a], lo[S.b],
                                     nullptr, 0, 0));
            }
            e = run_hops(*P, tasks, false, false, st, log);
            // steps 1 .. L-1: decode the partner's half, add, send one half, keep the other
            for (int32_t s = 1; s < L && e == cudaSuccess; ++s) {
                tasks.clear();
                for (int32_t r = 0; r < N; ++r) {
                    const ChunkSpan K0 = bfly_keep(L, s - 1, r), S = bfly_send(L, s, r), K = bfly_keep(L, s, r);
                    const int32_t p = r ^ (N >> s);
                    const void *add = s == 1 ? grads[r] : (const void *)keepb(r, (s - 1) & 1);
                    const int32_t ns = 1 << (L - 1 - s);
                    tasks.push_back(task(dq_stage{r, s, r & (ns - 1), ns}, msg(p, (s - 1) & 1), lo[K0.a], lo[K0.b], add, msg(r, s & 1),
                                         lo[S.a], lo[S.b], keepb(r, s & 1), lo[K.a], lo[K.b]));
                }
                e = run_hops(*P, tasks, true, s >= 2, st, log);
            }
            // the owner adds the last half it receives and compresses its chunk once
            if (e == cudaSuccess) {
                tasks.clear();
                for (int32_t r = 0; r < N; ++r) {
                    const void *add = L == 1 ? grads[r] : (const void *)keepb(r, (L - 1) & 1);
                    tasks.push_back(task(dq_stage{r, L, 0, 1}, msg(r ^ 1, (L - 1) & 1), lo[r], lo[r + 1], add, finb(r), lo[r],
                                         lo[r + 1], nullptr, 0, 0));
                }
                e = run_hops(*P, tasks, true, L >= 2, st, log);
            }
        }
        for (int32_t r = 0; r < N; ++r) fin[r] = finb(r);
    }
    if (e != cudaSuccess) return DQ_ERR_CUDA;

    // All-gather hands the final chunks to every rank unchanged; each rank
    // decodes all of them into its own output.
    std::unique_ptr<DecodeParams> D(new DecodeParams());
    memset(D.get(), 0, sizeof(DecodeParams));
    D->tab = P->tab;
    D->n_ranks = N;
    D->end2 = end2;
    D->end4 = end4;
    D->M = M;
    D->perm = perm;
    D->out_is_bf16 = out_is_bf16 ? 1 : 0;
    for (int32_t r = 0; r < N; ++r) {
        D->out = outs[r];
        int32_t c = 0;
        while (c < N) {
            int n = 0;
            int64_t total = 0;
            while (c < N && n < kMaxTasks) {
                if (lo[c + 1] > lo[c]) {
                    D->task[n].msg = msg_view(const_cast<uint8_t *>(fin[c]), lo[c], lo[c + 1], end2, end4);
                    D->task[n].lo = lo[c];
                    D->task[n].sg_begin = total;
                    total += lo[c + 1] - lo[c];
                    ++n;
                }
                ++c;
            }
            D->n_tasks = n;
            D->total_sg = total;
            if (n > 0) {
                const LogSlot slot = log_begin(log, DQ_LAUNCH_DECODE, total, st);
                const cudaError_t e2 = launch_decode(*D, st);
                log_end(slot, st);
                if (e2 != cudaSuccess) return DQ_ERR_CUDA;
            }
        }
    }
    if (final_msgs)
        for (int32_t c = 0; c < N; ++c) final_msgs[c] = fin[c];
    return DQ_OK;
}

}  // extern "C"
