// dq_static.cu -- dq_reorder_static: the bitwidth reordering of dq_reorder
// for callers that cannot allocate device memory, with its scratch in a
// file-scope device array instead of a caller-supplied workspace.
//
// The array lives in every GPU that loads the library, for the life of the
// process.  In host code its name is only a host-side stand-in; the device
// address is looked up with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and passed to the kernels.
#include <mutex>

#include "dq_common.cuh"
#include "dq_internal.h"

namespace {

// one scratch slot of 4 int64 per reorder tile (the tile size is dq_reorder's)
constexpr int64_t kMaxTiles = (DQ_REORDER_STATIC_MAX_SG + dq::kReorderTile - 1) / dq::kReorderTile;

// Per-tile counts and offsets of the reorder: 4 int64 per tile.  Every entry
// a call reads is written earlier in the same call, so nothing needs to be
// cleared between calls.
static __device__ __align__(256) long long g_reorder_scratch[kMaxTiles * 4];

std::mutex g_mu;
void *g_addr[256] = {nullptr};

// Device address of the scratch array on the current device.
dq_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DQ_ERR_CUDA;
    if (dev < 0 || dev >= 256) return DQ_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_reorder_scratch) != cudaSuccess || !p) return DQ_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return DQ_OK;
}

}  // namespace

extern "C" dq_status dq_reorder_static(const uint8_t *b, int64_t n_sg, int32_t *perm, void *stream)
{
    if (n_sg < 1 || n_sg > DQ_REORDER_STATIC_MAX_SG) return DQ_ERR_INVALID_ARG;
    if (!b || !perm) return DQ_ERR_INVALID_ARG;
    // the reorder must fit the array (holds by construction; checked so that
    // a change of the tile layout fails here instead of writing past it)
    if (dq::reorder_scratch_bytes(n_sg) > sizeof(g_reorder_scratch)) return DQ_ERR_INVALID_ARG;
    void *ws = nullptr;
    const dq_status s = scratch_address(&ws);
    if (s != DQ_OK) return s;
    return dq::launch_reorder(b, n_sg, perm, ws, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DQ_OK
                                                                                                      : DQ_ERR_CUDA;
}
