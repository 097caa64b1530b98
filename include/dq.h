/*
 * dq.h -- C ABI of libdq, a GB300 (sm_103a) implementation of the
 * data-parallel hot path of DynamiQ, a gradient-quantization scheme for
 * multi-hop all-reduce (arXiv 2602.08923).
 *
 * Sources, cited per entry point below:
 *   [S] everythinginsigcomm.group scribe notes, "DynamiQ: Accelerating
 *       Gradient Synchronization using Compressed Multi-hop All-reduce",
 *       sections "Key idea and contribution" and "Evaluation".
 *   [P] pith.science review of the same paper: "What carries the argument",
 *       "Referee Report" (Summary, major comment 1, minor comment 1),
 *       "Axiom & Free-Parameter Ledger", Fig. 2 and Fig. 3 captions.
 *   [A] mlsanity.com page of the paper, Abstract.
 *
 * Vocabulary.  A group is 16 consecutive coordinates sharing one scale; a
 * super-group (SG) is 16 groups = 256 consecutive coordinates sharing a
 * bitwidth, a mean and a squared norm [P "What carries the argument"].
 * n_sg = J is the number of super-groups of one worker's gradient (the
 * gradient length is J * 256; pad with zeros).  N = n_ranks workers are
 * simulated on one GPU: each worker's buffers are ordinary device buffers and
 * a "hop" hands a message buffer from one simulated rank to the next.
 *
 * Conventions (all entry points):
 *   - Device pointers are cudaMalloc/PyTorch device memory on the current
 *     device; "host" marks the few host pointers.  The caller owns every
 *     buffer; the library never allocates device memory.  dq_plan and
 *     dq_get_device_status read their results back through one small
 *     pinned host buffer mapped into the device address space, one per
 *     calling thread (under 64 bytes, allocated on the thread's first such
 *     call, kept until the process exits): the readback is a one-thread
 *     kernel write, so it never waits behind copies queued on other streams.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; only dq_plan synchronises (it reads three
 *     counts back to the host).
 *   - Gradient, message, mean and output pointers must be 16-byte aligned
 *     (DQ_ERR_ALIGNMENT otherwise).
 *   - The return value reports argument validation and the launch status
 *     (cudaGetLastError); nothing is launched when validation fails.
 *   - Calls on one stream are ordered; calls that share output buffers must
 *     not overlap on different streams.
 *   - Non-finite gradient values are outside the method's domain.  dq_plan
 *     detects them (they make a super-group's squared-norm sum F_j NaN or
 *     infinite) and returns DQ_ERR_NONFINITE; the other entry points do not
 *     check, and their results are then unspecified (no fault, no hang).
 */
#ifndef DQ_H
#define DQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DQ_OK = 0,
    DQ_ERR_INVALID_ARG = 1,        /* null pointer, bad size, bad range, bad N   */
    DQ_ERR_ALIGNMENT = 2,          /* a pointer is not 16-byte aligned           */
    DQ_ERR_BUDGET_INFEASIBLE = 3,  /* budget below 2 bits per coordinate         */
    DQ_ERR_CUDA = 4,               /* a CUDA call or kernel launch failed        */
    DQ_ERR_NONFINITE = 5           /* dq_plan: a super-group's statistics are not
                                      finite (NaN or infinite gradient values, or
                                      squares beyond the fp32 range)             */
} dq_status;

/* Parameters of one all-reduce round.  The last two fields, with eps and
 * correlated, switch off one technique each for ablation [S "Key idea and
 * contribution": variable bitwidth, non-uniform levels, hierarchical scale
 * quantization, correlated rounding; P Referee Report minor comment 1:
 * variable vs uniform bitwidth]; zero is the method as published. */
typedef struct {
    int32_t  n_ranks;      /* N, 1 .. 65535 (butterfly: a power of two)              */
    float    budget_bits;  /* B, average code bits per coordinate, >= 2             */
    double   eps;          /* level shape: q = sign(r) |r|(eps+|r|)/(1+eps); > 0, or
                              +inf for uniform levels; 1.0 by default              */
    int32_t  correlated;   /* 1: correlated rounding across ranks, 0: independent  */
    uint64_t seed;         /* key of the counter-based generator                    */
    uint64_t round;        /* training round (part of the generator counter)        */
    int32_t  fixed_bits;   /* 0: variable allocation; 2, 4 or 8: every super-group
                              gets that width (dq_plan skips the allocation; the
                              budget is not used)                                   */
    int32_t  scale_fp32;   /* 0: UINT8 group scales (E byte + u per group);
                              1: group scales sent as fp32, sigma = max |x|,
                              y = x / sigma (no second-level quantization)          */
} dq_config;

/* Who quantizes, for the stochastic-rounding generator.  Independent
 * rounding draws from a stream keyed by (seed, round, hop, rank, coordinate).
 * Correlated rounding [S "Key idea and contribution": shared randomness
 * across workers so that rounding errors cancel, up to 2x lower variance]
 * draws one uniform per (seed, round, hop, coordinate), shared by all
 * workers, and worker `slot` of the n_slots workers that quantize the same
 * coordinates at the same stage shifts it by slot/n_slots (one uniform per
 * stratum).  A fresh uniform per stage keeps every hop exactly unbiased.
 * Ring stages and the owner's final quantization have n_slots = 1;
 * butterfly step s (of L = log2 N) has n_slots = 2^(L-1-s), slot = the low
 * L-1-s bits of the rank. */
typedef struct {
    int32_t rank;     /* quantizing worker, 0 .. N-1                       */
    int32_t hop;      /* quantization stage of these coordinates, 0..65535 */
    int32_t slot;     /* 0 .. n_slots-1                                    */
    int32_t n_slots;  /* >= 1                                              */
} dq_stage;

/* A range of REORDERED super-groups [lo, hi).  After reordering, SGs
 * [0, end2) are 2-bit, [end2, end4) 4-bit and [end4, J) 8-bit. */
typedef struct {
    int64_t lo, hi;
    int64_t end2, end4;
} dq_range;

/* Version string of the library. */
const char *dq_version(void);

/* Human-readable name of a status code (static string). */
const char *dq_status_string(dq_status s);

/* Bytes of the message that carries range r (host, pure).  Layout, for
 * c = hi - lo SGs of which n2, n4, n8 have 2, 4, 8 bits:
 *   [E: c exponent bytes, padded to a multiple of 16][u: 16 bytes per SG]
 *   [2-bit codes, 64 B per SG][4-bit codes, 128 B per SG][8-bit, 256 B per SG]
 * With scale_fp32 = 1 the E and u sections are replaced by 16 fp32 scales
 * (64 B) per SG.  Coordinate i of an SG occupies bits [b*i, b*i+b) of the
 * SG's code block, least significant bits first.  [S "Key idea and
 * contribution": groups and super-groups; P Referee Report summary:
 * hierarchical UINT8 group scaling]  Returns 0 for an invalid range. */
size_t dq_message_bytes(dq_range r, int32_t scale_fp32);

/* Level table of the library for b in {2, 4, 8} (host, pure): writes 2^b
 * fp32 levels to q_host.  [P ledger: Q = {f(eps, r)}; S "Key idea and
 * contribution": more levels near zero] */
dq_status dq_level_table(int32_t bits, double eps, float *q_host);

/* Per-super-group statistics of ONE worker [S "Key idea and contribution":
 * each worker computes the mean and squared l2 norm of each super-group;
 * P major comment 1: F is computed before the mean is subtracted].
 *   g_bf16: device, J*256 bf16 values.  mean, sq: device, J floats each.
 *   Sums are fp32 in a fixed halving tree (16 coords of a group, then the 16
 *   group partials); mean = sum / 256. */
dq_status dq_stats(const void *g_bf16, int64_t n_sg, float *mean, float *sq, void *stream);

/* Metadata all-reduce, simulated [S "Key idea and contribution": a
 * lightweight all-reduce of the statistics; P Fig. 2(b)].
 *   mean_all, sq_all: device, N x J row-major (row r = rank r's dq_stats).
 *   M, F: device, J floats: M_j = sum of means, F_j = sum of squared norms,
 *   each added in rank order 0..N-1 in fp32 (M may be NULL).
 *   mu: device, J floats: the mean every worker subtracts, fl(M_j / N). */
dq_status dq_stats_reduce(const float *mean_all, const float *sq_all, int32_t n_ranks,
                          int64_t n_sg, float *M, float *F, float *mu, void *stream);

/* Device scratch needed by dq_allocate and dq_reorder for J super-groups. */
size_t dq_workspace_bytes(int64_t n_sg);

/* Bitwidth allocation [P "What carries the argument" and Fig. 3 caption:
 * thresholds tied by T_{2,4} = 17/512 T_{4,8}, one scalar meets any budget].
 *   b_j = 8 if 17 F_j >= 512 T, 4 if F_j >= T, else 2, where T is the
 *   smallest non-negative fp32 with sum_j b_j <= floor(B * J).
 *   F: device, J floats (finite, >= 0).  b: device, J bytes.  T_dev: device,
 *   1 float.  counts_dev: device, 3 int64 (number of 2-, 4-, 8-bit SGs).
 *   ws: device scratch of at least dq_workspace_bytes(J) bytes.
 *   Errors: DQ_ERR_BUDGET_INFEASIBLE if budget < 2; J must be < 2^27. */
dq_status dq_allocate(const float *F, int64_t n_sg, float budget, uint8_t *b, float *T_dev,
                      int64_t *counts_dev, void *ws, size_t ws_bytes, void *stream);

/* Reordering by bitwidth [S "Key idea and contribution": reorder the
 * super-groups by bitwidth, same bitwidth contiguous; P Fig. 2(c)].
 *   Stable partition 2-bit, 4-bit, 8-bit.  perm: device, J int32,
 *   perm[new] = old.  ws as for dq_allocate. */
dq_status dq_reorder(const uint8_t *b, int64_t n_sg, int32_t *perm, void *ws, size_t ws_bytes,
                     void *stream);

/* dq_reorder for callers that cannot allocate device memory.  No passage of
 * the paper corresponds to it: it exists for code that must not, or cannot,
 * call cudaMalloc when it reorders -- e.g. an application that reserved all
 * device memory for its own pool at start-up, a loop that forbids allocation
 * while it runs, or a caller that holds the input and output buffers but no
 * handle to the allocator that owns them.  Same result as dq_reorder; the
 * scratch is a 128 KiB array inside the library, resident on every GPU that
 * loads it until the process exits, so the call allocates nothing.
 *   b: device, n_sg bytes; perm: device, n_sg int32 (caller-owned).
 *   n_sg must be 1 .. DQ_REORDER_STATIC_MAX_SG; larger sizes return
 *   DQ_ERR_INVALID_ARG without touching the GPU (use dq_reorder then).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process: after cudaDeviceReset (or any teardown of the device's primary
 *   context) later calls on that device are invalid.  All calls share the one
 *   array: calls that overlap on the GPU (different streams, or different host
 *   threads without ordering) race and must not be made. */
#define DQ_REORDER_STATIC_MAX_SG 8388608
dq_status dq_reorder_static(const uint8_t *b, int64_t n_sg, int32_t *perm, void *stream);

/* Chunk cuts of the reordered stream among n_chunks workers (host, pure):
 * chunk_lo_host[c] = the smallest reordered index whose prefix of code bits
 * reaches ceil(c * total / n_chunks); chunk_lo_host[n_chunks] = J.  Chunks
 * carry near-equal code bits (equal bytes per hop). */
dq_status dq_chunk_cuts(int64_t n2, int64_t n4, int64_t n8, int32_t n_chunks,
                        int64_t *chunk_lo_host);

/* First hop: quantize one worker's normalised gradient over range r
 * [S "Key idea and contribution": each worker normalises by the global mean
 * and quantizes; non-uniform levels, UINT8 second-level scales, correlated
 * rounding].  x = fl(float(g[perm[j]*256 + i]) - mu[perm[j]]), mu as written
 * by dq_stats_reduce.
 *   hop: quantization stage index; rank: the quantizing rank (generator
 *   counter and correlated offset).  msg_out: device, dq_message_bytes(r). */
dq_status dq_compress(const dq_config *cfg, dq_range r, dq_stage stage, const void *g_bf16,
                      const float *mu, const int32_t *perm, uint8_t *msg_out, void *stream);

/* One hop: decompress - accumulate - recompress, fused [S "Key idea and
 * contribution": decompress the incoming partial sum, accumulate the local
 * gradient, recompress, forward; S: a fused CUDA kernel; A].
 *   x = fl(dec(msg_in) + addend) over range in.
 *   addend: addend_is_fp32 = 0: the worker's bf16 gradient (full J*256, read
 *   through perm, mean subtracted); = 1: fp32 partial sums, row j - in.lo.
 *   SGs in `send` are requantized into msg_out (dq_message_bytes(send));
 *   SGs in `keep` are written as fp32 to keep_out (row j - keep.lo).
 *   send and keep must split `in` into two adjacent ranges (either may be
 *   empty): a ring hop sends everything, a butterfly step sends one half and
 *   keeps the other. */
dq_status dq_dar(const dq_config *cfg, dq_range in, dq_stage stage, const uint8_t *msg_in,
                 const void *addend, int32_t addend_is_fp32, const float *mu, const int32_t *perm, dq_range send, uint8_t *msg_out,
                 dq_range keep, float *keep_out, void *stream);

/* Final decode [S "Key idea and contribution": restore the original
 * super-group order and add back the subtracted mean; P Referee Report
 * summary: the receiver unnormalises].  out[perm[j]*256 + i] =
 * fl(dec + fl(mu_j * N)), fp32 (out_is_bf16 = 0) or rounded to bf16. */
dq_status dq_decode(const dq_config *cfg, dq_range r, const uint8_t *msg, const float *mu,
                    const int32_t *perm, void *out, int32_t out_is_bf16, void *stream);

/* ---- the whole round: statistics to decode, N simulated ranks ---------- */

/* Result of the planning phase, filled by dq_plan. */
typedef struct {
    float   T;            /* the threshold T_{2,4}; NaN when fixed_bits is set */
    int64_t n2, n4, n8;   /* SGs per bitwidth */
} dq_plan_info;

/* Device bytes dq_plan needs in plan_ws for N ranks and J super-groups. */
size_t dq_plan_workspace_bytes(int32_t n_ranks, int64_t n_sg);

/* Planning phase of one all-reduce round over N ranks [S "Key idea and
 * contribution", statistics collection phase; P Fig. 2(a)-(c)]: per-rank
 * statistics, metadata all-reduce, allocation and reordering.
 *   grads_host: host array of N device pointers (J*256 bf16 each).
 *   mu, perm: device outputs (J floats, J int32) used by dq_exchange.
 *   info_host: host output.  Synchronises `stream` once to read the counts.
 *   plan_ws: device scratch of dq_plan_workspace_bytes(N, J).
 *   rank_ready_host: NULL, or a host array of N cudaEvent_t (entries may
 *   be NULL): the statistics of rank r wait on event r, so a rank's
 *   statistics start as soon as its gradient is ready (e.g. its upload or
 *   its backward pass finished) while other ranks' are still in flight.
 *   log: NULL or a dq_launch_log to fill (see below).
 *   Returns DQ_ERR_NONFINITE (after the sync) when some M_j or F_j is not
 *   finite; mu, perm and info are then not meaningful. */
typedef struct dq_launch_log dq_launch_log;
dq_status dq_plan(const dq_config *cfg, const void *const *grads_host, int64_t n_sg,
                  float *mu, int32_t *perm, void *plan_ws, size_t plan_ws_bytes,
                  dq_plan_info *info_host, void *const *rank_ready_host, dq_launch_log *log,
                  void *stream);

/* dq_plan without the readback: the same launches, enqueued on `stream`, and
 * no synchronisation.  The plan's 2/4/8 counts stay on the device, for
 * dq_exchange_stream_step, which derives the bucket's chunk cuts from them.
 *   counts_dev_host: host output: the device address (inside plan_ws) of the
 *   three int64 counts n2, n4, n8, written by the enqueued work.
 *   nonfinite_dev_host: NULL, or host output: the device address (inside
 *   plan_ws) of an int32 that the enqueued work leaves nonzero when some M_j
 *   or F_j is not finite (read it with dq_get_device_status after the work;
 *   the round's results are then not meaningful, though no kernel faults).
 *   Other arguments as for dq_plan.  Errors: as dq_plan's argument checks. */
dq_status dq_plan_async(const dq_config *cfg, const void *const *grads_host, int64_t n_sg,
                        float *mu, int32_t *perm, void *plan_ws, size_t plan_ws_bytes,
                        const int64_t **counts_dev_host, const int32_t **nonfinite_dev_host,
                        void *const *rank_ready_host, dq_launch_log *log, void *stream);

/* Optional record of the kernel launches of dq_plan and dq_exchange, for timing them on
 * the launching stream.  events: host array of 2*capacity cudaEvent_t created
 * by the caller (timing enabled); launch i is bracketed by events[2i] and
 * events[2i+1].  kinds[i]: DQ_LAUNCH_*; sgs[i]: super-groups it processed
 * (a decode launch counts each super-group once per output it writes: the
 * exchange decodes each chunk once into up to 16 ranks' outputs).
 * count: in, first free slot; out, slots used.  Launches beyond capacity
 * are not recorded (they still run). */
enum { DQ_LAUNCH_COMPRESS = 0, DQ_LAUNCH_DAR = 1, DQ_LAUNCH_DECODE = 2, DQ_LAUNCH_STATS = 3,
       DQ_LAUNCH_ALLOCATE_REORDER = 4, /* statistics reduce, allocation and reorder, one bracket */
       DQ_LAUNCH_MX_HOP = 5, DQ_LAUNCH_MX_DECODE = 6, /* MXFP8 baseline; sgs = coordinates / 256 */
       DQ_LAUNCH_FUSED_RING = 7, /* dq_exchange_fused: all hops and the decode; sgs = J * (N + 1) */
       DQ_LAUNCH_PIPELINED = 8,  /* one launch of dq_exchange_pipelined; sgs = super-groups its hop
                                    units process plus super-groups it decodes (each once) */
       DQ_LAUNCH_STREAM = 9      /* one dq_exchange_stream_step; sgs = the super-groups of its
                                    buckets (each once) */ };
struct dq_launch_log {
    void   **events;
    int32_t *kinds;
    int64_t *sgs;
    int32_t  capacity;
    int32_t  count;
};

/* Number of kernels libdq has launched in this process (all entry points). */
uint64_t dq_launch_count(void);

/* Device bytes dq_exchange needs (messages and butterfly partial sums). */
size_t dq_exchange_workspace_bytes(const dq_config *cfg, int32_t butterfly, int64_t n_sg,
                                   const dq_plan_info *info);

/* Main all-reduce phase [S "Key idea and contribution": hop-by-hop
 * decompress-accumulate-recompress, then restore order and add the mean;
 * S "Evaluation": ring and butterfly topologies].  Ring: reduce-scatter of
 * N-1 DAR hops, the owner's DAR giving the final chunk, all-gather forwarding
 * the bytes unchanged.  Butterfly: recursive halving with split DAR (one half
 * sent compressed, the other kept in fp32), the owner compressing its chunk
 * once.  Every rank then decodes all chunks into outs_host[r] (device, J*256
 * fp32, or bf16 if out_is_bf16).  final_msgs_host, if not NULL, receives the
 * N device pointers (inside ws) of the final chunk messages.  log: NULL or
 * a dq_launch_log to fill.  No sync. */
dq_status dq_exchange(const dq_config *cfg, int32_t butterfly, const void *const *grads_host,
                      int64_t n_sg, const float *mu, const int32_t *perm,
                      const dq_plan_info *info, void *ws, size_t ws_bytes,
                      void *const *outs_host, int32_t out_is_bf16,
                      const uint8_t **final_msgs_host, dq_launch_log *log, void *stream);

/* ---- the ring exchange in one launch -------------------------------------
 * Device status words (int32) written by the fused exchange: */
#define DQ_DEVICE_OK 0
#define DQ_DEVICE_BARRIER_TIMEOUT 1   /* a grid-barrier wait ran out; outputs are invalid */

/* Device bytes dq_exchange_fused needs (ring; 1 <= N <= 64), 0 otherwise. */
size_t dq_exchange_fused_workspace_bytes(const dq_config *cfg, int64_t n_sg, const dq_plan_info *info);

/* The ring exchange of dq_exchange (same results, bit for bit) as ONE
 * cooperative launch: the N hop steps and the final decode run in a
 * persistent kernel, separated by device-wide barriers instead of kernel
 * boundaries [S "Key idea and contribution": hop-by-hop fused decompress-
 * accumulate-recompress; the barrier replaces the network hand-off].  It
 * removes the per-step launches, which dominate small buckets.
 *   Ring only, 1 <= N <= 64; arguments as for dq_exchange; ws of
 *   dq_exchange_fused_workspace_bytes bytes.
 *   status_dev: device int32 (4-byte aligned), set to DQ_DEVICE_OK before
 *   the launch; every barrier wait is bounded (about a second of SM
 *   clock) and, when it runs out, the kernel sets DQ_DEVICE_BARRIER_TIMEOUT
 *   and returns instead of waiting on.  Read it after the stream is
 *   synchronised; the outputs are valid only when it is DQ_DEVICE_OK.
 *   Every CTA is resident at once (cudaLaunchCooperativeKernel); other work
 *   running on the GPU at the same time delays the launch, it cannot
 *   deadlock it. */
dq_status dq_exchange_fused(const dq_config *cfg, const void *const *grads_host, int64_t n_sg,
                            const float *mu, const int32_t *perm, const dq_plan_info *info, void *ws,
                            size_t ws_bytes, void *const *outs_host, int32_t out_is_bf16,
                            int32_t *status_dev, const uint8_t **final_msgs_host, dq_launch_log *log,
                            void *stream);

/* ---- the ring exchange, pipelined over parts -------------------------------
 * Device bytes dq_exchange_pipelined needs: N*N chunk messages and 2 KB of
 * unit counters (ring; 1 <= N <= 64), 0 otherwise. */
size_t dq_exchange_pipelined_workspace_bytes(const dq_config *cfg, int64_t n_sg, const dq_plan_info *info);

/* The ring exchange of dq_exchange (same results, bit for bit: final
 * messages and outputs) with the reduce-scatter pipelined over parts of the
 * super-groups, the way a ring all-reduce is pipelined over slices of its
 * chunks [S "Evaluation": ring all-reduce; S "Key idea and contribution":
 * hop-by-hop fused decompress-accumulate-recompress, then restore order and
 * add the mean].  The work units of one step (all chunks, 32 reordered
 * super-groups each, in chunk order) are cut into n_parts parts of
 * consecutive units; launch t (t = 0 .. N + n_parts - 1) runs step t - p of
 * every part p with 0 <= t - p < N and the final decode of part t - N.  So
 * the decode of early parts (bound by HBM writes: N outputs of 4 bytes per
 * coordinate) runs in the same launches as the hops of later parts (bound by
 * instruction issue), on every SM at once.
 *   Ring only, 1 <= N <= 64; arguments as for dq_exchange.
 *   n_parts: >= 1; cut to at most 256 and to the work units of one step.
 *   n_parts = 1 is N + 1 launches with the per-step work of dq_exchange.
 *   ws: dq_exchange_pipelined_workspace_bytes bytes (device, 16-byte
 *   aligned): rank r's message of step s in its own buffer, so a launch never
 *   overwrites bytes that another part has still to read, then one unit
 *   counter per launch (zeroed by the call; one extra small launch).
 *   final_msgs_host: as for dq_exchange (owner c's message of step N-1).
 *   Errors: DQ_ERR_INVALID_ARG (bad config, N > 64, n_parts < 1, null
 *   pointer, small ws), DQ_ERR_ALIGNMENT, DQ_ERR_CUDA (a launch failed).  No
 *   sync. */
dq_status dq_exchange_pipelined(const dq_config *cfg, const void *const *grads_host, int64_t n_sg,
                                const float *mu, const int32_t *perm, const dq_plan_info *info, void *ws,
                                size_t ws_bytes, void *const *outs_host, int32_t out_is_bf16, int32_t n_parts,
                                const uint8_t **final_msgs_host, dq_launch_log *log, void *stream);

/* ---- DDP buckets: the ring exchange pipelined across buckets -------------
 * Data-parallel training all-reduces its gradient as a stream of buckets
 * [S "Evaluation": DDP gradient buckets; review "What carries the
 * argument": each bucket is compressed with its own statistics and
 * allocation].  A bucket of a 25 MB DDP stream gives each ring step too few
 * work units to fill the GPU, so the exchange is pipelined across buckets:
 * launch t runs ring step t - b of every bucket b in flight (N of them) and
 * the final decode of bucket t - N, the way the ring pipelines its chunks.
 * Each bucket's planning is dq_plan_async (no host round trip); the launch
 * derives the bucket's chunk cuts and work units on the device from the
 * counts the plan left there.  Results are those of dq_exchange for each
 * bucket, bit for bit. */

/* One bucket's part in a launch. */
typedef struct {
    int64_t            n_sg;        /* super-groups of the bucket (J), 1 .. 2^27-1 */
    const int64_t     *counts_dev;  /* device: n2, n4, n8 (dq_plan_async's counts_dev) */
    const void *const *grads_host;  /* host array of N device bf16 gradients (J*256) */
    void *const       *outs_host;   /* host array of N device outputs (J*256 fp32 or bf16) */
    const float       *mu;          /* device, J floats, from the bucket's plan */
    const int32_t     *perm;        /* device, J int32, from the bucket's plan */
    void              *msgs;        /* device, 16-byte aligned: the bucket's messages */
    size_t             msgs_bytes;  /* >= dq_bucket_msgs_bytes(cfg, n_sg) */
    uint64_t           round;       /* the bucket's generator round */
    int32_t            step;        /* 0 .. N-1: this launch runs ring step `step` of
                                       the bucket; N: its final decode */
} dq_bucket_step;

/* Device bytes of one bucket's message buffers (N*N chunk messages, sized
 * for any allocation of n_sg super-groups); 0 for a bad config, a butterfly
 * or more than 8 ranks. */
size_t dq_bucket_msgs_bytes(const dq_config *cfg, int64_t n_sg);

/* One launch of the bucket stream: the ring steps and the final decode
 * listed in steps[0 .. n_steps) (1 <= n_steps <= N + 1, at most one decode,
 * ring only, N <= 8; cfg's round is not used: each bucket carries its own).
 * A bucket's step s must follow its step s-1 on the same stream (and its
 * decode its step N-1); its plan must precede its step 0 (stream order or an
 * event).  The bucket's messages, mu, perm and gradients must stay untouched
 * from its step 0 to its decode.
 *   counter_dev: device uint32, zero at the launch (one per launch; the
 *   launch counts it up).
 *   Errors: DQ_ERR_INVALID_ARG (bad config, N > 8, a bad step list, a null
 *   pointer, small msgs), DQ_ERR_ALIGNMENT, DQ_ERR_CUDA.  No sync. */
dq_status dq_exchange_stream_step(const dq_config *cfg, const dq_bucket_step *steps, int32_t n_steps,
                                  unsigned int *counter_dev, int32_t out_is_bf16, dq_launch_log *log,
                                  void *stream);

/* A whole bucket stream in one call: every bucket's dq_plan_async on
 * plan_stream (lookahead buckets ahead of the exchange) and the N + n_buckets
 * launches of dq_exchange_stream_step on `stream`, ordered by CUDA events
 * the call creates and releases (no device memory is allocated, and the
 * host never waits).  Each bucket's results equal a dq_plan + dq_exchange
 * round of that bucket with cfg's round replaced by the bucket's.
 *   buckets[k]: the bucket's size, its N gradients and outputs (host arrays
 *   of device pointers, as for dq_plan and dq_exchange) and its round.
 *   lookahead: >= 1, how many buckets ahead of the exchange the planning
 *   is enqueued.
 *   plan_sms: SMs the exchange's launches leave free for the planning
 *   stream's kernels (0 .. SMs - 1).
 *   sets[0 .. n_sets): caller-owned buffer sets, n_sets >= N + lookahead + 1:
 *   bucket k uses set k % n_sets, which is reused once bucket k - n_sets has
 *   been decoded.  A set holds
 *   mu and perm (bucket_sg floats and int32), a plan workspace
 *   (dq_plan_workspace_bytes(N, bucket_sg)) and the messages
 *   (dq_bucket_msgs_bytes(cfg, bucket_sg)), bucket_sg >= every n_sg.
 *   counters_dev: device, n_buckets + N uint32 (zeroed by the call).
 *   nonfinite_dev: NULL, or a device int32 (4-byte aligned) that the call
 *   clears and that becomes 1 when any bucket's statistics are not finite
 *   (what dq_plan reports as DQ_ERR_NONFINITE: that bucket's results are
 *   meaningless, the others are unaffected); read it after the work, e.g.
 *   with dq_get_device_status.
 *   plan_stream: the planning stream (NULL: `stream`); give it a higher
 *   priority than `stream`, so that its short kernels take SMs as the
 *   exchange's launches free them.
 *   Errors: as dq_exchange_stream_step and dq_plan's argument checks, and
 *   DQ_ERR_INVALID_ARG for a bad lookahead, plan_sms or n_sets.  No sync. */
typedef struct {
    int64_t            n_sg;
    const void *const *grads_host;
    void *const       *outs_host;
    uint64_t           round;
} dq_bucket;

typedef struct {
    float   *mu;
    int32_t *perm;
    void    *plan_ws;
    size_t   plan_ws_bytes;
    void    *msgs;
    size_t   msgs_bytes;
} dq_stream_set;

dq_status dq_allreduce_stream(const dq_config *cfg, const dq_bucket *buckets, int32_t n_buckets,
                              const dq_stream_set *sets, int32_t n_sets, int32_t lookahead, int32_t plan_sms,
                              unsigned int *counters_dev, int32_t out_is_bf16, int32_t *nonfinite_dev,
                              void *plan_stream, void *stream, dq_launch_log *log);

/* dq_allreduce_stream with the host staging of every bucket done by the
 * library: the DDP bucket stream end to end, gradients arriving from host
 * memory and rank 0's result leaving to it (the paper's all-reduce runs on
 * gradients each worker holds and hands back [S "Key idea and
 * contribution"]; here the host side of that hand-over is part of the
 * call, with no host round trip per bucket).
 *   io[k].src_host: host array of N pinned host pointers; rank r's bf16
 *   gradient of bucket k (n_sg * 256 values) is copied into
 *   buckets[k].grads_host[r] on copy_in_stream, right before the bucket's
 *   planning is enqueued (lookahead buckets ahead of the exchange), and the
 *   planning waits for it.  NULL: the gradients are already on the device.
 *   A device gradient buffer used by an earlier bucket b is refilled once
 *   b's last ring step has run; that launch must come before the planning
 *   of bucket k in the call's order, i.e. k >= b + N + lookahead (e.g.
 *   staging sets cycled k mod S with S >= N + lookahead), else
 *   DQ_ERR_INVALID_ARG.
 *   io[k].dst_host: pinned host buffer for rank 0's result of bucket k
 *   (n_sg * 256 fp32, or bf16 with out_is_bf16), copied on copy_out_stream
 *   after the bucket's decode; a later decode that writes the same device
 *   buffer waits for that copy.  NULL: no download.
 *   copy_in_stream, copy_out_stream: the copy streams (NULL: plan_stream
 *   and `stream`).  Everything the call enqueues on the other streams
 *   starts after the work already on `stream`, and `stream` ends after the
 *   last download, so one synchronisation of `stream` covers the pass.
 *   Other arguments and errors: as dq_allreduce_stream.  No sync. */
typedef struct {
    const void *const *src_host;
    void              *dst_host;
} dq_bucket_io;

dq_status dq_allreduce_stream_io(const dq_config *cfg, const dq_bucket *buckets, const dq_bucket_io *io,
                                 int32_t n_buckets, const dq_stream_set *sets, int32_t n_sets, int32_t lookahead,
                                 int32_t plan_sms, unsigned int *counters_dev, int32_t out_is_bf16,
                                 int32_t *nonfinite_dev, void *copy_in_stream, void *copy_out_stream,
                                 void *plan_stream, void *stream, dq_launch_log *log);

/* Reads a device status word into host memory [boundary of the hot path:
 * device-side errors of an asynchronous call are reported through a status
 * word that the caller reads after the work; the paper itself defines no
 * interface].  status_dev: device int32, 4-byte aligned -- the word passed
 * to dq_exchange_fused or dq_barrier_selftest (caller-owned).  status_host:
 * host int32 that receives it: DQ_DEVICE_OK or DQ_DEVICE_BARRIER_TIMEOUT.
 * Enqueues a 4-byte device-to-host copy on `stream` and synchronises that
 * stream, so the value read includes every kernel enqueued on the stream
 * before the call.  This entry point and dq_plan are the only ones that
 * synchronise.  Errors: DQ_ERR_INVALID_ARG (null pointer), DQ_ERR_ALIGNMENT,
 * DQ_ERR_CUDA (the copy or the synchronisation failed, e.g. an earlier
 * kernel on the stream faulted; *status_host is then left unchanged). */
dq_status dq_get_device_status(const int32_t *status_dev, int32_t *status_host, void *stream);

/* Test of the failure path of the fused exchange's barrier, with no
 * counterpart in the paper: n_blocks CTAs (1 .. number of SMs) run one
 * barrier that waits for n_blocks + missing arrivals, each wait bounded by
 * timeout_cycles (<= 8e9).  missing = 0: every CTA passes, *status_dev stays
 * DQ_DEVICE_OK.  missing > 0: the wait runs out, *status_dev becomes
 * DQ_DEVICE_BARRIER_TIMEOUT and the kernel returns; the context stays
 * usable.  scratch: device, 4 bytes (the arrival counter). */
dq_status dq_barrier_selftest(int32_t n_blocks, int32_t missing, int64_t timeout_cycles, void *scratch,
                              int32_t *status_dev, void *stream);

/* ---- comparison baseline: MXFP8 ------------------------------------------
 * The pages compare DynamiQ's error with MXFP8's [A Abstract; S
 * "Evaluation"], citing the OCP Microscaling (MX) v1.0 specification.  This
 * is that baseline, run over the same N-rank schedules on the GPU: blocks of
 * 32 coordinates (n_blk blocks = n_blk * 32 coordinates, in original order)
 * share one E8M0 scale byte X (2^(X-127)); elements are FP8 E4M3.  Encode:
 * X - 127 = floor(log2 max|v|) - 8, clamped at -127 (X = 0 for an all-zero
 * block); element = v * 2^(127-X) rounded to nearest-even, saturating at
 * +-448.  A hop decodes, adds in fp32 (x = fl(dec + addend)) and re-encodes;
 * there is no mean, allocation or reordering.  Chunk c of N is blocks
 * [floor(c n_blk / N), floor((c+1) n_blk / N)).
 * Message of c blocks: [X: c bytes, padded to a multiple of 16]
 *                      [elements: 32 bytes per block]. */

/* Bytes of the MXFP8 message of n_blk blocks (host, pure; 0 if invalid). */
size_t dq_mx_message_bytes(int64_t n_blk);

/* Encode n_blk blocks of fp32 x (device, 32 * n_blk floats) into msg
 * (device, dq_mx_message_bytes(n_blk)). */
dq_status dq_mx_quantize(const float *x, int64_t n_blk, uint8_t *msg, void *stream);

/* Decode msg into out (device, 32 * n_blk floats). */
dq_status dq_mx_dequantize(const uint8_t *msg, int64_t n_blk, float *out, void *stream);

/* Device bytes dq_mx_exchange needs (0 for invalid arguments). */
size_t dq_mx_exchange_workspace_bytes(int32_t n_ranks, int32_t butterfly, int64_t n_blk);

/* The MXFP8 all-reduce of N simulated ranks: grads_host[r] is rank r's bf16
 * gradient (device, 32 * n_blk values), outs_host[r] its fp32 output (the
 * sum, identical on every rank).  Ring (butterfly = 0) or butterfly (N a
 * power of two) with the same hop schedule as dq_exchange.  ws: device
 * scratch of dq_mx_exchange_workspace_bytes bytes.  final_msgs_host, if not
 * NULL, receives the N device pointers of the final chunk messages. */
dq_status dq_mx_exchange(int32_t n_ranks, int32_t butterfly, const void *const *grads_host, int64_t n_blk,
                         void *ws, size_t ws_bytes, void *const *outs_host, const uint8_t **final_msgs_host,
                         dq_launch_log *log, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DQ_H */
