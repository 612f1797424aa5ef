// ep_api.cu -- the C ABI declared in include/ep.h: argument checks, then the
// launches.  No allocation, no host synchronisation.
#include <stdint.h>

#include "ep.h"
#include "ep_internal.cuh"

namespace ep {

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    return dev;
}

int device_sm_count()
{
    // Cached per device; the attribute never changes for a device.
    static PerDeviceCache<1> cache;
    return cache.get([] {
        const int dev = current_device();
        int n = 1;
        if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        return n;
    });
}

}  // namespace ep

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

ep_status launched(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

constexpr int kMaxGateExperts = 512;
constexpr int kMaxGateK = 32;
constexpr int kMaxGroups = 32;
constexpr int kMaxKin = 4;
constexpr int kMaxLayoutExperts = 1024;
constexpr int kMaxRowK = 64;  // slots per token accepted by layout, dispatch and combine

ep_status check_layout_args(int32_t T, int32_t k, int32_t E, int32_t epr)
{
    if (T < 0 || k < 1 || E < 1 || epr < 1 || E % epr != 0)
        return EP_ERR_INVALID_ARG;
    if (E > kMaxLayoutExperts || k > kMaxRowK || (int64_t)T * k >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

}  // namespace

extern "C" {

const char *ep_status_str(ep_status s)
{
    switch (s) {
    case EP_OK:
        return "ok";
    case EP_ERR_INVALID_ARG:
        return "invalid argument";
    case EP_ERR_UNSUPPORTED:
        return "unsupported size or configuration";
    case EP_ERR_ALIGNMENT:
        return "misaligned pointer";
    case EP_ERR_CUDA:
        return "CUDA launch error";
    }
    return "unknown status";
}

}  // extern "C"

namespace {

ep_status check_gate_cfg(const ep_gate_cfg *cfg)
{
    if (!cfg)
        return EP_ERR_INVALID_ARG;
    const int E = cfg->num_experts, k = cfg->top_k, G = cfg->n_groups, Kg = cfg->topk_group;
    const int kin = cfg->topk_in_group;
    if (E < 1 || k < 1 || k > E || G < 1 || E % G != 0 || Kg < 1 || Kg > G || kin < 1 || kin > E / G)
        return EP_ERR_INVALID_ARG;
    if ((int64_t)Kg * (E / G) < k)
        return EP_ERR_INVALID_ARG;
    if (cfg->score_fn != EP_SCORE_RAW && cfg->score_fn != EP_SCORE_SOFTMAX)
        return EP_ERR_INVALID_ARG;
    if (cfg->normalize != 0 && cfg->normalize != 1)
        return EP_ERR_INVALID_ARG;
    if (E > kMaxGateExperts || k > kMaxGateK || G > kMaxGroups || kin > kMaxKin)
        return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

ep::GateParams gate_params(const ep_gate_cfg *cfg)
{
    return ep::GateParams{cfg->num_experts, cfg->top_k, cfg->n_groups, cfg->topk_group, cfg->topk_in_group,
                          cfg->score_fn, cfg->normalize};
}

}  // namespace

extern "C" {

ep_status ep_gate(const float *scores, const float *bias, int32_t T, const ep_gate_cfg *cfg, int32_t *topk_idx,
                  float *topk_w, void *stream)
{
    if (T < 0)
        return EP_ERR_INVALID_ARG;
    const ep_status c = check_gate_cfg(cfg);
    if (c != EP_OK)
        return c;
    if ((int64_t)T * cfg->num_experts >= (int64_t)1 << 40)
        return EP_ERR_UNSUPPORTED;
    if (T == 0)
        return EP_OK;
    if (!scores || !topk_idx || !topk_w)
        return EP_ERR_INVALID_ARG;
    if (!aligned(scores, 4) || (bias && !aligned(bias, 4)) || !aligned(topk_idx, 4) || !aligned(topk_w, 4))
        return EP_ERR_ALIGNMENT;
    return launched(
        ep::launch_gate(scores, bias, T, gate_params(cfg), topk_idx, topk_w, static_cast<cudaStream_t>(stream)));
}

size_t ep_layout_workspace_bytes(int32_t T, int32_t k, int32_t E, int32_t experts_per_rank)
{
    if (check_layout_args(T, k, E, experts_per_rank) != EP_OK)
        return 0;
    return ep::layout_workspace_bytes(T, k, E, experts_per_rank);
}

ep_status ep_get_layout(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E, int32_t experts_per_rank,
                        int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                        int32_t *rank_tokens, int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    const ep_status a = check_layout_args(T, k, E, experts_per_rank);
    if (a != EP_OK)
        return a;
    if (!expert_count || !expert_off || !rank_count || !rank_off || !rank_tokens || !workspace)
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !pos || !src))
        return EP_ERR_INVALID_ARG;
    if (workspace_bytes < ep::layout_workspace_bytes(T, k, E, experts_per_rank))
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {topk_idx, expert_count, expert_off, rank_count, rank_off, rank_tokens, pos, src, err_flag};
    for (const void *q : ptrs)
        if (q && !aligned(q, 4))
            return EP_ERR_ALIGNMENT;
    if (!aligned(workspace, 16))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_layout(topk_idx, T, k, E, experts_per_rank, expert_count, expert_off, rank_count,
                                      rank_off, rank_tokens, pos, src, err_flag, workspace,
                                      static_cast<cudaStream_t>(stream)));
}

ep_status ep_gate_layout(const float *scores, const float *bias, int32_t T, const ep_gate_cfg *cfg,
                         int32_t experts_per_rank, int32_t *topk_idx, float *topk_w, int32_t *expert_count,
                         int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                         int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, size_t workspace_bytes,
                         void *stream)
{
    if (T < 0)
        return EP_ERR_INVALID_ARG;
    const ep_status c = check_gate_cfg(cfg);
    if (c != EP_OK)
        return c;
    const int E = cfg->num_experts, k = cfg->top_k;
    const ep_status l = check_layout_args(T, k, E, experts_per_rank);
    if (l != EP_OK)
        return l;
    if (!expert_count || !expert_off || !rank_count || !rank_off || !rank_tokens || !workspace)
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (!scores || !topk_idx || !topk_w || !pos || !src))
        return EP_ERR_INVALID_ARG;
    if (workspace_bytes < ep::layout_workspace_bytes(T, k, E, experts_per_rank))
        return EP_ERR_INVALID_ARG;
    const void *p4[] = {scores, bias, topk_idx, topk_w, expert_count, expert_off, rank_count, rank_off, rank_tokens,
                        pos,    src,  err_flag};
    for (const void *q : p4)
        if (q && !aligned(q, 4))
            return EP_ERR_ALIGNMENT;
    if (!aligned(workspace, 16))
        return EP_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ep::GateParams gp = gate_params(cfg);
    // The grid-wide launch with lane-segment gating for group-limited
    // batches past decode size and for batches past one cluster's layout;
    // decode-sized batches in one clustered launch; otherwise the gate
    // kernel then the layout (one CTA, or one cluster).
    const long long entries = (long long)T * k;
    const bool grouped = gp.Kg < gp.G;
    if (T > 0 && entries > ep::kSmallLayoutEntries && (grouped || entries > ep::kClusterLayoutEntries) &&
        ep::route_supported(T, k, E, experts_per_rank, true) && ep::gate_fast_supported(gp, scores, bias))
        return launched(ep::launch_route(scores, bias, &gp, nullptr, topk_idx, topk_w, T, k, E, experts_per_rank,
                                         expert_count, expert_off, rank_count, rank_off, rank_tokens, pos, src,
                                         err_flag, workspace, st));
    // decode-sized batches (at most 4096 entries, 512 tokens): one
    // clustered launch with no grid barrier
    if (T > 0 && entries <= ep::kSmallLayoutEntries && ep::gate_layout_small_supported(T, k))
        return launched(ep::launch_gate_layout_small(scores, bias, T, gp, experts_per_rank, topk_idx, topk_w,
                                                     expert_count, expert_off, rank_count, rank_off, rank_tokens,
                                                     pos, src, st));
    // configurations the lane-segment gating does not serve, batches too
    // large for one grid of one CTA per SM, and those between: the two
    // steps' own kernels
    cudaError_t e = ep::launch_gate(scores, bias, T, gp, topk_idx, topk_w, st);
    if (e == cudaSuccess)
        e = ep::launch_layout(topk_idx, T, k, E, experts_per_rank, expert_count, expert_off, rank_count, rank_off,
                              rank_tokens, pos, src, err_flag, workspace, st);
    return launched(e);
}

ep_status ep_dispatch(const void *x, int32_t T, int32_t H, int32_t k, const int32_t *pos, int32_t dtype, void *recv,
                      int32_t recv_rows, void *recv_scales, int32_t *err_flag, void *stream)
{
    if (T < 0 || H < 1 || k < 1 || recv_rows < 0)
        return EP_ERR_INVALID_ARG;
    if (dtype != EP_DTYPE_BF16 && dtype != EP_DTYPE_FP8_E4M3_B128 && dtype != EP_DTYPE_MXFP8_E4M3_B32)
        return EP_ERR_INVALID_ARG;
    if (H % 8 != 0 || k > kMaxRowK || (int64_t)T * k >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    if ((dtype == EP_DTYPE_FP8_E4M3_B128 && H % 128 != 0) || (dtype == EP_DTYPE_MXFP8_E4M3_B32 && H % 32 != 0))
        return EP_ERR_UNSUPPORTED;
    if (T == 0)
        return EP_OK;
    if (!x || !pos || (recv_rows > 0 && (!recv || (dtype != EP_DTYPE_BF16 && !recv_scales))))
        return EP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(pos, 4) ||
        (dtype == EP_DTYPE_FP8_E4M3_B128 && !aligned(recv_scales, 4)) || (err_flag && !aligned(err_flag, 4)))
        return EP_ERR_ALIGNMENT;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t *xs = static_cast<const uint16_t *>(x);
    if (dtype == EP_DTYPE_BF16)
        return launched(
            ep::launch_dispatch_bf16(xs, T, H, k, pos, static_cast<uint16_t *>(recv), recv_rows, err_flag, st));
    if (dtype == EP_DTYPE_FP8_E4M3_B128)
        return launched(ep::launch_dispatch_fp8(xs, T, H, k, pos, static_cast<uint8_t *>(recv),
                                                static_cast<float *>(recv_scales), recv_rows, err_flag, st));
    return launched(ep::launch_dispatch_mxfp8(xs, T, H, k, pos, static_cast<uint8_t *>(recv),
                                              static_cast<uint8_t *>(recv_scales), recv_rows, err_flag, st));
}

ep_status ep_combine(const void *y, int32_t y_rows, const int32_t *pos, const float *topk_w, int32_t T, int32_t H,
                     int32_t k, void *out, int32_t *err_flag, void *stream)
{
    if (T < 0 || H < 1 || k < 1 || y_rows < 0)
        return EP_ERR_INVALID_ARG;
    if (H % 8 != 0 || k > kMaxRowK || (int64_t)T * k >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    if (T == 0)
        return EP_OK;
    if ((y_rows > 0 && !y) || !pos || !topk_w || !out)
        return EP_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(pos, 4) || !aligned(topk_w, 4) ||
        (err_flag && !aligned(err_flag, 4)))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_combine(static_cast<const uint16_t *>(y), y_rows, pos, topk_w, T, H, k,
                                       static_cast<uint16_t *>(out), err_flag, static_cast<cudaStream_t>(stream)));
}

ep_status ep_combine_fp8(const void *yq, const void *yscales, int32_t scale_dtype, int32_t y_rows, const int32_t *pos,
                         const float *topk_w, int32_t T, int32_t H, int32_t k, void *out, int32_t *err_flag,
                         void *stream)
{
    if (T < 0 || H < 1 || k < 1 || y_rows < 0)
        return EP_ERR_INVALID_ARG;
    if (scale_dtype != EP_DTYPE_FP8_E4M3_B128 && scale_dtype != EP_DTYPE_MXFP8_E4M3_B32)
        return EP_ERR_INVALID_ARG;
    const int bs = scale_dtype == EP_DTYPE_FP8_E4M3_B128 ? 128 : 32;
    if (H % bs != 0 || k > kMaxRowK || (int64_t)T * k >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    if (T == 0)
        return EP_OK;
    if ((y_rows > 0 && (!yq || !yscales)) || !pos || !topk_w || !out)
        return EP_ERR_INVALID_ARG;
    if (!aligned(yq, 16) || !aligned(out, 16) || !aligned(pos, 4) || !aligned(topk_w, 4) ||
        (bs == 128 && !aligned(yscales, 4)) || (err_flag && !aligned(err_flag, 4)))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_combine_fp8(static_cast<const uint8_t *>(yq), yscales, bs == 32 ? 1 : 0, y_rows, pos,
                                           topk_w, T, H, k, static_cast<uint16_t *>(out), err_flag,
                                           static_cast<cudaStream_t>(stream)));
}

ep_status ep_get_layout_capacity(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E, int32_t experts_per_rank,
                                 int32_t capacity, int32_t *expert_count, int32_t *expert_off, int32_t *rank_count,
                                 int32_t *rank_off, int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos,
                                 int32_t *src, int32_t *err_flag, void *workspace, size_t workspace_bytes,
                                 void *stream)
{
    const ep_status a = check_layout_args(T, k, E, experts_per_rank);
    if (a != EP_OK)
        return a;
    if (capacity < 0)
        return EP_ERR_INVALID_ARG;
    if ((int64_t)E * capacity >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    if (!expert_count || !expert_off || !rank_count || !rank_off || !rank_tokens || !expert_dropped || !workspace)
        return EP_ERR_INVALID_ARG;
    if ((T > 0 && (!topk_idx || !pos)) || ((int64_t)E * capacity > 0 && !src))
        return EP_ERR_INVALID_ARG;
    if (workspace_bytes < ep::layout_workspace_bytes(T, k, E, experts_per_rank))
        return EP_ERR_INVALID_ARG;
    const void *ptrs[] = {topk_idx, expert_count, expert_off, rank_count, rank_off, rank_tokens, expert_dropped,
                          pos,      src,          err_flag};
    for (const void *q : ptrs)
        if (q && !aligned(q, 4))
            return EP_ERR_ALIGNMENT;
    if (!aligned(workspace, 16))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_layout_capacity(topk_idx, T, k, E, experts_per_rank, capacity, expert_count,
                                               expert_off, rank_count, rank_off, rank_tokens, expert_dropped, pos,
                                               src, err_flag, workspace, static_cast<cudaStream_t>(stream)));
}

ep_status ep_dispatch_backward(const void *grad_recv, int32_t recv_rows, const int32_t *pos, int32_t T, int32_t H,
                               int32_t k, void *grad_x, int32_t *err_flag, void *stream)
{
    if (T < 0 || H < 1 || k < 1 || recv_rows < 0)
        return EP_ERR_INVALID_ARG;
    if (H % 8 != 0 || k > kMaxRowK || (int64_t)T * k >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    if (T == 0)
        return EP_OK;
    if ((recv_rows > 0 && !grad_recv) || !pos || !grad_x)
        return EP_ERR_INVALID_ARG;
    if (!aligned(grad_recv, 16) || !aligned(grad_x, 16) || !aligned(pos, 4) || (err_flag && !aligned(err_flag, 4)))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_combine(static_cast<const uint16_t *>(grad_recv), recv_rows, pos, nullptr, T, H, k,
                                       static_cast<uint16_t *>(grad_x), err_flag, static_cast<cudaStream_t>(stream)));
}

ep_status ep_combine_backward(const void *grad_out, const void *y, int32_t y_rows, const int32_t *pos,
                              const float *topk_w, int32_t T, int32_t H, int32_t k, void *grad_y, float *grad_w,
                              int32_t *err_flag, void *stream)
{
    if (T < 0 || H < 1 || k < 1 || y_rows < 0)
        return EP_ERR_INVALID_ARG;
    if (H % 8 != 0 || k > kMaxRowK || (int64_t)T * k >= (int64_t)INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    if (T == 0)
        return EP_OK;
    if (!grad_out || (y_rows > 0 && (!y || !grad_y)) || !pos || !topk_w || !grad_w)
        return EP_ERR_INVALID_ARG;
    if (!aligned(grad_out, 16) || !aligned(y, 16) || !aligned(grad_y, 16) || !aligned(pos, 4) ||
        !aligned(topk_w, 4) || !aligned(grad_w, 4) || (err_flag && !aligned(err_flag, 4)))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_combine_backward(static_cast<const uint16_t *>(grad_out),
                                                static_cast<const uint16_t *>(y), y_rows, pos, topk_w, T, H, k,
                                                static_cast<uint16_t *>(grad_y), grad_w, err_flag,
                                                static_cast<cudaStream_t>(stream)));
}

ep_status ep_decode_dispatch(const float *scores, const float *bias, int32_t T, const ep_gate_cfg *cfg,
                             int32_t experts_per_rank, const void *x, int32_t H, int32_t dtype, int32_t *topk_idx,
                             float *topk_w, int32_t *expert_count, int32_t *expert_off, int32_t *rank_count,
                             int32_t *rank_off, int32_t *rank_tokens, int32_t *pos, int32_t *src, void *recv,
                             int32_t recv_rows, void *recv_scales, int32_t *err_flag, void *workspace,
                             size_t workspace_bytes, void *stream)
{
    if (T < 1 || H < 1 || recv_rows < 0)
        return EP_ERR_INVALID_ARG;
    const ep_status c = check_gate_cfg(cfg);
    if (c != EP_OK)
        return c;
    const int E = cfg->num_experts, k = cfg->top_k;
    const ep_status l = check_layout_args(T, k, E, experts_per_rank);
    if (l != EP_OK)
        return l;
    if (dtype != EP_DTYPE_BF16 && dtype != EP_DTYPE_FP8_E4M3_B128 && dtype != EP_DTYPE_MXFP8_E4M3_B32)
        return EP_ERR_INVALID_ARG;
    if (H % 8 != 0 || (dtype == EP_DTYPE_FP8_E4M3_B128 && H % 128 != 0) ||
        (dtype == EP_DTYPE_MXFP8_E4M3_B32 && H % 32 != 0))
        return EP_ERR_UNSUPPORTED;
    if ((size_t)T * k > ep::decode_max_entries())
        return EP_ERR_UNSUPPORTED;  // the fused path is for decode-sized batches
    if (!expert_count || !expert_off || !rank_count || !rank_off || !rank_tokens || !workspace ||
        workspace_bytes < 2 * sizeof(unsigned))
        return EP_ERR_INVALID_ARG;
    if (!scores || !x || !topk_idx || !topk_w || !pos || !src ||
        (recv_rows > 0 && (!recv || (dtype != EP_DTYPE_BF16 && !recv_scales))))
        return EP_ERR_INVALID_ARG;
    const void *p4[] = {scores, bias, topk_idx, topk_w, expert_count, expert_off, rank_count, rank_off, rank_tokens,
                        pos,    src,  err_flag, workspace};
    for (const void *q : p4)
        if (q && !aligned(q, 4))
            return EP_ERR_ALIGNMENT;
    if (!aligned(x, 16) || !aligned(recv, 16))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_decode(scores, bias, T, gate_params(cfg), experts_per_rank,
                                      static_cast<const uint16_t *>(x), H, dtype, topk_idx, topk_w, expert_count,
                                      expert_off, rank_count, rank_off, rank_tokens, pos, src, recv, recv_scales,
                                      recv_rows, err_flag, workspace, static_cast<cudaStream_t>(stream)));
}

ep_status ep_selftest_grid_barrier(int32_t missing_arrivals, int64_t spin_limit, int32_t *err_flag, void *workspace,
                                   size_t workspace_bytes, void *stream)
{
    if (missing_arrivals < 0 || spin_limit < 1 || spin_limit > ((int64_t)1 << 24) || !err_flag || !workspace ||
        workspace_bytes < 2 * sizeof(unsigned))
        return EP_ERR_INVALID_ARG;
    if (!aligned(err_flag, 4) || !aligned(workspace, 4))
        return EP_ERR_ALIGNMENT;
    return launched(ep::launch_barrier_selftest((unsigned)missing_arrivals, spin_limit, err_flag, workspace,
                                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
