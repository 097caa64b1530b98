// dq_sched.h -- the N-rank hop schedules (host only), shared by the DynamiQ
// exchange and the MXFP8 comparison exchange.
//
// Ring [scribe notes "Evaluation": ring all-reduce]: reduce-scatter in N
// steps; at step t rank r handles chunk (r - 1 - t) mod N: step 0 quantizes
// it from the local gradient, later steps decode rank r-1's message, add the
// local gradient and requantize (stage t); the message of step N-1 is the
// owner's final chunk, which the all-gather forwards unchanged.
// Butterfly (recursive halving, N = 2^L) [same, butterfly all-reduce]: at
// step s rank r holds chunks [base, base + 2^(L-s)), keeps the half whose bit
// (L-1-s) equals its own and sends the other half to r XOR 2^(L-1-s); the
// sender quantizes (stage s), the receiver decodes and adds to its partial
// sum (the local gradient at s = 1, its fp32 kept half after that).  After L
// steps the owner quantizes its chunk once (stage L).
// Messages live in two buffers per rank (parity of the step), the butterfly's
// kept fp32 halves likewise, and the butterfly's final chunks in one final
// buffer per rank.
#pragma once

#include <stdint.h>

#include <vector>

namespace dq {

struct ChunkSpan {
    int32_t a, b;   // chunks [a, b)
};

struct SchedHop {
    int32_t rank;          // the rank that runs this hop (and quantizes)
    int32_t stage;         // quantization stage (generator counter)
    int32_t slot, n_slots; // correlated-rounding stratum
    int32_t in_rank;       // -1: no incoming message; else message (in_rank, in_par)
    int32_t in_par;
    ChunkSpan in;          // chunks processed
    ChunkSpan send;        // chunks quantized into the out message (may be empty)
    ChunkSpan keep;        // chunks written as fp32 to keep buffer (rank, keep_par)
    int32_t add_par;       // -1: addend = the rank's gradient; else keep buffer (rank, add_par)
    int32_t out_par;       // out message (rank, out_par); -1: the rank's final buffer
    int32_t keep_par;
};

struct SchedStep {
    std::vector<SchedHop> hops;
    bool has_in;   // every hop decodes an incoming message
    bool add_f32;  // every hop's addend is an fp32 kept half
};

struct Schedule {
    std::vector<SchedStep> steps;
    // final chunk c: message (fin_rank[c], fin_par[c]); fin_par -1 = final buffer
    std::vector<int32_t> fin_rank, fin_par;
    int32_t L = 0;  // butterfly levels
};

inline int32_t sched_log2(int32_t n)
{
    int32_t L = 0;
    while ((1 << L) < n) ++L;
    return (1 << L) == n ? L : -1;
}

// Butterfly chunk halves of rank r at step s (keep: its own half).
inline ChunkSpan bfly_half(int32_t L, int32_t s, int32_t r, bool keep)
{
    const int32_t width = 1 << (L - s), half = width >> 1, base = (r >> (L - s)) << (L - s);
    const int32_t my = (r >> (L - 1 - s)) & 1;
    const int32_t h = keep ? my : 1 - my;
    return {base + h * half, base + h * half + half};
}

// Returns false when the butterfly is asked for a non-power-of-two N.
inline bool build_schedule(int32_t N, bool butterfly, Schedule &S)
{
    S.steps.clear();
    S.fin_rank.assign((size_t)N, 0);
    S.fin_par.assign((size_t)N, 0);
    const ChunkSpan none{0, 0};
    if (!butterfly) {
        for (int32_t t = 0; t < N; ++t) {
            SchedStep st;
            st.has_in = t > 0;
            st.add_f32 = false;
            for (int32_t r = 0; r < N; ++r) {
                const int32_t c = (int32_t)((((int64_t)r - 1 - t) % N + N) % N);
                SchedHop h;
                h.rank = r;
                h.stage = t;
                h.slot = 0;
                h.n_slots = 1;
                h.in_rank = t ? (r - 1 + N) % N : -1;
                h.in_par = (t - 1) & 1;
                h.in = {c, c + 1};
                h.send = {c, c + 1};
                h.keep = none;
                h.add_par = -1;
                h.out_par = t & 1;
                h.keep_par = 0;
                st.hops.push_back(h);
            }
            S.steps.push_back(st);
        }
        for (int32_t c = 0; c < N; ++c) {
            S.fin_rank[c] = c;
            S.fin_par[c] = (N - 1) & 1;
        }
        return true;
    }
    const int32_t L = sched_log2(N);
    if (L < 0) return false;
    S.L = L;
    for (int32_t c = 0; c < N; ++c) {
        S.fin_rank[c] = c;
        S.fin_par[c] = -1;
    }
    if (L == 0) {
        SchedStep st;
        st.has_in = false;
        st.add_f32 = false;
        st.hops.push_back(SchedHop{0, 0, 0, 1, -1, 0, {0, 1}, {0, 1}, none, -1, -1, 0});
        S.steps.push_back(st);
        return true;
    }
    {   // step 0: quantize the half that is sent
        SchedStep st;
        st.has_in = false;
        st.add_f32 = false;
        const int32_t ns = 1 << (L - 1);
        for (int32_t r = 0; r < N; ++r) {
            const ChunkSpan Sd = bfly_half(L, 0, r, false);
            st.hops.push_back(SchedHop{r, 0, r & (ns - 1), ns, -1, 0, Sd, Sd, none, -1, 0, 0});
        }
        S.steps.push_back(st);
    }
    for (int32_t s = 1; s < L; ++s) {   // decode the partner's half, add, send one half, keep the other
        SchedStep st;
        st.has_in = true;
        st.add_f32 = s >= 2;
        const int32_t ns = 1 << (L - 1 - s);
        for (int32_t r = 0; r < N; ++r) {
            const ChunkSpan K0 = bfly_half(L, s - 1, r, true), Sd = bfly_half(L, s, r, false),
                            K = bfly_half(L, s, r, true);
            st.hops.push_back(SchedHop{r, s, r & (ns - 1), ns, r ^ (N >> s), (s - 1) & 1, K0, Sd, K,
                                       s == 1 ? -1 : (s - 1) & 1, s & 1, s & 1});
        }
        S.steps.push_back(st);
    }
    {   // the owner adds the last half it receives and quantizes its chunk once
        SchedStep st;
        st.has_in = true;
        st.add_f32 = L >= 2;
        for (int32_t r = 0; r < N; ++r)
            st.hops.push_back(SchedHop{r, L, 0, 1, r ^ 1, (L - 1) & 1, {r, r + 1}, {r, r + 1}, none,
                                       L == 1 ? -1 : (L - 1) & 1, -1, 0});
        S.steps.push_back(st);
    }
    return true;
}

}  // namespace dq
