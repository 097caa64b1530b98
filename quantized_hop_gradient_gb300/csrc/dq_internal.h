// dq_internal.h -- declarations shared by the libdq translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dq_common.cuh"

namespace dq {

int sm_count();            // SMs of the current device (cached per device)
void note_launches(int n);  // adds to the library's launch counter

// Level tables for eps (host; cached).  Returns false for an invalid eps.
bool build_tables(double eps, Tables *out);

// Message view of range [lo, hi) with stream boundaries end2, end4.
MsgView msg_view(uint8_t *base, int64_t lo, int64_t hi, int64_t end2, int64_t end4, bool scale_fp32);
size_t msg_bytes(int64_t c, int64_t n2, int64_t n4, int64_t n8, bool scale_fp32);

cudaError_t launch_stats(const uint16_t *g, int64_t n_sg, float *mean, float *sq, cudaStream_t st);
cudaError_t launch_stats_batched(const StatsParams &S, cudaStream_t st);
cudaError_t launch_stats_reduce(const float *mean_all, const float *sq_all, int32_t n, int64_t n_sg,
                                float *M, float *F, float *mu, cudaStream_t st, int32_t *nonfinite = nullptr);
cudaError_t launch_hop(const HopParams &P, bool has_in, bool add_f32, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams &P, cudaStream_t st);
// Cooperative launches (every CTA resident): the fused ring exchange, and a
// lone grid barrier whose target is `missing` arrivals more than the grid
// provides (missing > 0 makes the bounded wait run out).
cudaError_t launch_fused_ring(const FusedRingParams &P, cudaStream_t st);
cudaError_t launch_barrier_selftest(int32_t n_blocks, int32_t missing, long long timeout_cycles,
                                    unsigned int *counter, int32_t *status, cudaStream_t st);
// One launch of the pipelined ring exchange (ordinary launch).
cudaError_t launch_wave_ring(const WaveRingParams &P, cudaStream_t st);
// One launch of the bucket stream; tasks_hint sizes the grid (the exact
// task count is known only on the device), free_sms SMs are left free.
cudaError_t launch_stream_ring(const StreamRingParams &P, int64_t tasks_hint, cudaStream_t st, int free_sms = 0);

// Allocation (radix select of T) and reordering; ws is device scratch.
constexpr int kReorderTile = 2048;   // super-groups per reorder tile (4 int64 of scratch each)
size_t plan_scratch_bytes(int64_t n_sg);
size_t reorder_scratch_bytes(int64_t n_sg);   // bytes of ws that launch_reorder uses
cudaError_t launch_allocate(const float *F, int64_t n_sg, int64_t cap_bits, uint8_t *b, float *T,
                            int64_t *counts, void *ws, cudaStream_t st);
cudaError_t launch_reorder(const uint8_t *b, int64_t n_sg, int32_t *perm, void *ws, cudaStream_t st);
// The planning after the statistics, for any size: metadata all-reduce
// (M, F, mu from the ranks' per-super-group statistics), allocation and
// reorder in 3 + passes launches; ws holds plan_scratch_bytes(n_sg).
// fixed_bits != 0 gives every super-group that width.  sticky (optional):
// set to 1, and never cleared, when the statistics are not finite.
cudaError_t launch_plan_chain(const float *mean_all, const float *sq_all, int32_t n_ranks, int64_t n_sg,
                              int64_t cap_bits, int32_t fixed_bits, float *M, float *F, float *mu,
                              int32_t *nonfinite, uint8_t *b, float *T, int64_t *counts, int32_t *perm, void *ws,
                              cudaStream_t st, int32_t *sticky = nullptr);
// allocation and reorder of up to small_plan_max_sg() super-groups in one launch
int64_t small_plan_max_sg();
// nonfinite: the flag the statistics reduce before this launch set;
// sticky (optional) receives it as launch_plan_chain's.
cudaError_t launch_plan_small(const float *F, int64_t n_sg, int64_t cap_bits, int32_t fixed_bits, uint8_t *b,
                              float *T, int64_t *counts, int32_t *perm, cudaStream_t st,
                              const int32_t *nonfinite = nullptr, int32_t *sticky = nullptr);

// Brackets one launch with the caller's events (if a log has room).
struct LogSlot {
    dq_launch_log *log;
    int32_t i;
};
LogSlot log_begin(dq_launch_log *log, int32_t kind, int64_t sgs, cudaStream_t st);
void log_end(const LogSlot &s, cudaStream_t st);

}  // namespace dq
