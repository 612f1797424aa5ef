// layout_noalloc.cu -- ep_get_layout_noalloc: the dispatch layout with its
// scratch in a fixed device array owned by this library, for callers that
// cannot allocate device memory at call time.
//
// Who needs it: code that runs inside another runtime whose memory pool owns
// all device memory (a plugin or custom operator that may not call
// cudaMalloc itself), and serving loops with a memory budget fixed at start
// up, where a per-call allocation could fail mid-request or stall the device
// (cudaMalloc may synchronise).  Those callers still own and pass every
// input and output; only the layout's scratch moves here.
//
// The scratch is one file-scope __device__ array of kStaticScratchBytes
// (1 MiB).  Every GPU that loads the library holds it until the process
// exits.  Host code cannot use the array's name as a device address (it
// names a host-side stand-in), so the first call on each device, with that
// device current, looks the address up with cudaGetSymbolAddress and caches
// it; make that first call before any stream capture.  All calls on a
// device share the one array: calls whose work overlaps on the GPU (two
// streams, or two host threads) race on it and must be serialised by the
// caller.  The layout kernels write every scratch word they later read, so
// nothing needs clearing between calls and the previous call's contents do
// not matter.
#include <mutex>

#include "ep.h"
#include "ep_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_layout_scratch on the current device (looked up once
// per device); nullptr on failure.
void *scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess)
            return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" ep_status ep_get_layout_noalloc(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E,
                                           int32_t experts_per_rank, int32_t *expert_count, int32_t *expert_off,
                                           int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                                           int32_t *pos, int32_t *src, int32_t *err_flag, void *stream)
{
    const size_t need = ep_layout_workspace_bytes(T, k, E, experts_per_rank);
    if (need == 0)
        return (T < 0 || k < 1 || E < 1 || experts_per_rank < 1 || E % experts_per_rank != 0) ? EP_ERR_INVALID_ARG
                                                                                              : EP_ERR_UNSUPPORTED;
    if (need > kStaticScratchBytes)
        return EP_ERR_UNSUPPORTED;  // the sizes need more scratch than the fixed array holds
    void *scratch = scratch_on_current_device();
    if (scratch == nullptr)
        return EP_ERR_CUDA;
    return ep_get_layout(topk_idx, T, k, E, experts_per_rank, expert_count, expert_off, rank_count, rank_off,
                         rank_tokens, pos, src, err_flag, scratch, kStaticScratchBytes, stream);
}
