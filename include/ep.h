/*
 * ep.h -- C ABI of the MoE expert-parallel dispatch/combine hot path on one
 * GB300 (sm_103a): group-limited top-k gating, dispatch layout,
 * permute-scatter (BF16, or FP8 e4m3 with 1x128 block scales), inverse gather
 * and router-weighted combine.
 *
 * The operation follows the pages' statement of expert parallelism:
 *  - "Expert Parallelism (Parallelisme d'experts)" (polydesk.ai glossary),
 *    section "Le principe de base": whole experts live on a rank, E experts
 *    over E/experts_per_rank ranks; section "Le pattern de communication
 *    all-to-all": Phase 1 Dispatch sends each token to the holders of its
 *    chosen experts, Phase 2 Combine returns the expert outputs and sums them
 *    weighted by the router scores.
 *  - "DeepEP de DeepSeek : la lib open source qui optimise la communication
 *    GPU pour les modeles MoE a l'echelle" (ai-master.dev), section
 *    "Group-limited gating algorithm" (experts chosen inside a few groups),
 *    section "Support FP8 et MXFP8" (FP8 payload at half the BF16 bytes).
 *  - hyper.ai story on NVIDIA Hybrid-EP (hyper.ai/fr/stories/b564891f...):
 *    dispatch/combine operators callable from PyTorch over pre-allocated
 *    buffers; sizing them must not need a host round trip when a fixed
 *    maximum is known.
 *
 * On one GPU the "ranks" are logical: rank r owns experts
 * [r*experts_per_rank, (r+1)*experts_per_rank) and the rows of one receive
 * buffer between rank_off[r] and rank_off[r+1].  A send is a store.
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers owned by the caller.  The library never
 *    allocates or frees device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*,
 *    NULL = legacy default stream) and never synchronise the host.
 *  - Problems that the host can see (bad sizes, bad configuration, NULL or
 *    misaligned pointers) return an error status and launch nothing.
 *    A failed launch returns EP_ERR_CUDA (the CUDA error is left to
 *    cudaGetLastError's caller to inspect or clear).
 *  - Problems only the device can see never trap: the offending entry is
 *    skipped and a bit is OR-ed into *err_flag (a device int32, may be NULL):
 *      EP_FLAG_BAD_EXPERT  an expert index neither -1 nor in [0, E)
 *      EP_FLAG_BAD_ROW     a receive row outside the buffer's rows
 *      EP_FLAG_TIMEOUT     a bounded device-side wait ran out (the grid
 *                          barrier of a cooperative launch); that work stopped
 *  - bf16 tensors are raw 16-bit bfloat16 patterns, row-major.
 *  - T*k rows always suffice for a receive buffer (top-k picks k distinct
 *    experts per token), so buffers are sized without reading any count
 *    back to the host.  Calls that read or write a receive buffer take its
 *    row count (recv_rows / y_rows): T*k after ep_get_layout, E*capacity
 *    after ep_get_layout_capacity.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1, /* a size, pointer or configuration field is invalid */
    EP_ERR_UNSUPPORTED = 2, /* valid in principle but outside this library's limits */
    EP_ERR_ALIGNMENT = 3,   /* a pointer is not aligned as the call requires */
    EP_ERR_CUDA = 4         /* the CUDA runtime reported an error at launch */
} ep_status;

enum { EP_FLAG_BAD_EXPERT = 1, EP_FLAG_BAD_ROW = 2, EP_FLAG_TIMEOUT = 4 };

typedef enum {
    EP_SCORE_RAW = 0,    /* scores are affinities used as given (e.g. sigmoid outputs) */
    EP_SCORE_SOFTMAX = 1 /* scores are logits; weights come from their softmax */
} ep_score_fn;

typedef enum {
    EP_DTYPE_BF16 = 0,          /* receive rows are bf16 copies of x */
    EP_DTYPE_FP8_E4M3_B128 = 1, /* e4m3 codes + one fp32 scale per 128 columns */
    EP_DTYPE_MXFP8_E4M3_B32 = 2 /* MXFP8: e4m3 codes + one E8M0 (power-of-two) scale byte per 32 columns */
} ep_dtype;

/* Gating configuration (see ep_gate). */
typedef struct {
    int32_t num_experts;   /* E, 1..512 */
    int32_t top_k;         /* k, 1..min(E, 32) */
    int32_t n_groups;      /* G, 1..32, divides E; groups are contiguous blocks of E/G experts */
    int32_t topk_group;    /* groups kept per token, 1..G; topk_group * E/G >= k */
    int32_t topk_in_group; /* keys summed into a group's score, 1..min(4, E/G) */
    int32_t score_fn;      /* ep_score_fn */
    int32_t normalize;     /* 1: weights of a token sum to one; 0: unnormalised */
} ep_gate_cfg;

/*
 * Step 1 -- router top-k with the group limit ("DeepEP de DeepSeek ...",
 * section "Group-limited gating algorithm"; hyper.ai Hybrid-EP story: each
 * token activates only its top-k experts).
 *
 * scores   [T, E] fp32 row-major: affinities (RAW) or logits (SOFTMAX).
 * bias     [E] fp32 or NULL: added to the score to form the selection key
 *          (key = score + bias, fp32); it never enters the weights.
 * T        tokens, >= 0.
 * topk_idx [T, k] int32 out: chosen experts in slot order = selection order
 *          (descending key; equal keys -> lower expert index first).
 * topk_w   [T, k] fp32 out: RAW: score (normalize=0) or score / sum of the
 *          chosen scores in slot order (normalize=1). SOFTMAX: the full
 *          softmax probability (normalize=0) or exp(l - m) / sum over the
 *          chosen k of exp(l - m), m = largest chosen logit (normalize=1).
 * Group score = sum of the group's topk_in_group largest keys, largest
 * first, in fp32; the topk_group best groups are kept (ties -> lower group
 * index) and the k experts are chosen among them.  With n_groups = 1 this is
 * plain top-k.  Scores must be finite.
 * Errors: EP_ERR_INVALID_ARG (NULL pointer with T > 0, cfg fields out of
 * range), EP_ERR_UNSUPPORTED (E > 512, k > 32, G > 32, topk_in_group > 4),
 * EP_ERR_ALIGNMENT (scores, bias, outputs not 4-byte aligned), EP_ERR_CUDA.
 */
ep_status ep_gate(const float *scores, const float *bias, int32_t T, const ep_gate_cfg *cfg,
                  int32_t *topk_idx, float *topk_w, void *stream);

/* Bytes of device workspace ep_get_layout needs for these sizes (a multiple
 * of 256; 0 if the sizes are invalid). */
size_t ep_layout_workspace_bytes(int32_t T, int32_t k, int32_t E, int32_t experts_per_rank);

/*
 * Step 2 -- dispatch layout for logical ranks of experts_per_rank contiguous
 * experts ("Expert Parallelism ...", section "Le principe de base"; the
 * hyper.ai Hybrid-EP story's buffer sizing step).
 *
 * topk_idx      [T, k] int32: expert per (token, slot); -1 = empty slot.
 * expert_count  [E] out: entries per expert.
 * expert_off    [E+1] out: exclusive prefix sum of expert_count.
 * rank_count    [R] out (R = E / experts_per_rank): entries per rank.
 * rank_off      [R+1] out: exclusive prefix sum of rank_count.
 * rank_tokens   [R] out: distinct tokens with at least one entry on the rank.
 * pos           [T, k] out: receive row of entry (t, j) = expert_off[e] +
 *               number of entries of expert e with a smaller flat index
 *               t*k+j (a stable order), or -1 for a skipped entry.
 * src           [T*k] out: inverse of pos (flat entry index per receive
 *               row); rows at or past expert_off[E] hold -1.
 * err_flag      device int32 or NULL: EP_FLAG_BAD_EXPERT is OR-ed in when an
 *               index is neither -1 nor in [0, E); that entry is skipped.
 * workspace     device scratch of at least ep_layout_workspace_bytes(...)
 *               bytes, 16-byte aligned; contents need no initialisation.
 *               Afterwards its first 4 bytes are zero (this call clears
 *               them when it uses them) and the rest is garbage.  It must not be
 *               shared by layouts in flight at the same time.
 * Batches of more than 4096 entries run as one cooperative launch while a
 * grid of one CTA per SM covers them with at most 4096 entries per CTA (a
 * bounded grid barrier; if its wait runs out EP_FLAG_TIMEOUT is OR-ed into
 * *err_flag and the outputs are incomplete), else as three launches.
 * Limits: 1 <= E <= 1024, experts_per_rank divides E, 1 <= k <= 64, T >= 0,
 * T*k < 2^31.  Errors: EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED,
 * EP_ERR_ALIGNMENT, EP_ERR_CUDA.
 */
ep_status ep_get_layout(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E,
                        int32_t experts_per_rank, int32_t *expert_count, int32_t *expert_off,
                        int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                        int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Steps 1 and 2 in one call: ep_gate, then ep_get_layout of the experts it
 * chose, with the outputs of those two calls bit for bit ("DeepEP de DeepSeek
 * ...", section "Group-limited gating algorithm"; "Expert Parallelism ...",
 * section "Le principe de base").  Each is short and latency-bound.  Which
 * kernels run depends on the batch:
 *  - at most 4096 entries (T*k) and 512 tokens (decode-sized): one launch
 *    of one thread-block cluster, whose CTAs gate a slice of the tokens each
 *    and exchange per-expert token masks through distributed shared memory;
 *  - group-limited gating past that, and any gating past 65536 entries,
 *    while a grid of one CTA per SM covers the batch with at most 128
 *    tokens per CTA: one cooperative launch whose CTAs gate and count their
 *    own tokens, meet at one grid barrier and then place them;
 *  - otherwise the two calls' own kernels.
 *
 * Arguments: those of ep_gate (scores, bias, T, cfg, topk_idx, topk_w) and
 * of ep_get_layout (experts_per_rank, expert_count .. src, err_flag), with
 * the same layouts, limits and errors, except:
 * workspace     at least ep_layout_workspace_bytes(T, cfg->top_k,
 *               cfg->num_experts, experts_per_rank) bytes, 16-byte aligned,
 *               whose first 4 bytes (the grid barrier's arrival count) are
 *               zero before the call.  Every call that completes leaves the
 *               count zero (so do ep_get_layout and ep_get_layout_capacity
 *               on the same workspace): clear it once when the workspace is
 *               allocated.  If the barrier's bounded wait runs out,
 *               EP_FLAG_TIMEOUT is OR-ed into *err_flag, the outputs are
 *               incomplete and the count must be cleared again.  Calls in
 *               flight at the same time need separate workspaces.
 */
ep_status ep_gate_layout(const float *scores, const float *bias, int32_t T, const ep_gate_cfg *cfg,
                         int32_t experts_per_rank, int32_t *topk_idx, float *topk_w, int32_t *expert_count,
                         int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                         int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, size_t workspace_bytes,
                         void *stream);

/*
 * ep_get_layout without a workspace argument, for callers that cannot
 * allocate device memory at call time: code running inside another
 * runtime whose memory pool owns the device memory (a plugin or custom
 * operator that may not call cudaMalloc itself), or a serving loop with a
 * memory budget fixed at start-up, where an allocation per call could fail
 * mid-request or stall the device.  The source pages have no counterpart to
 * this call; it exists for those callers only.
 *
 * Arguments, outputs and errors are those of ep_get_layout.  The scratch is
 * a fixed 1 MiB device array inside this library (every GPU that loads the
 * library keeps it until the process exits); sizes whose
 * ep_layout_workspace_bytes exceeds 1 MiB are rejected with
 * EP_ERR_UNSUPPORTED (T*k up to about 465 thousand entries fit at E = 256,
 * experts_per_rank = 8).  The call allocates nothing.  The first
 * call on a device looks up the array's device address (with that device
 * current) and caches it: make that first call before any stream capture.
 * Every call on a device shares the one array, so calls whose work overlaps
 * on the GPU (other streams, other host threads) race and must be
 * serialised by the caller; the array needs no clearing between calls.
 */
ep_status ep_get_layout_noalloc(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E,
                                int32_t experts_per_rank, int32_t *expert_count, int32_t *expert_off,
                                int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                                int32_t *pos, int32_t *src, int32_t *err_flag, void *stream);

/*
 * Step 3 -- permute-scatter ("Expert Parallelism ...", section "Le pattern
 * de communication all-to-all", Phase 1; FP8 modes from "DeepEP de DeepSeek
 * ...", section "Support FP8 et MXFP8").
 *
 * x            [T, H] bf16, 16-byte aligned; H % 8 == 0.
 * pos          [T, k] int32 receive row per entry (from ep_get_layout);
 *              entries < 0 are skipped; rows >= recv_rows are skipped and
 *              flagged EP_FLAG_BAD_ROW.  1 <= k <= 64.
 * recv_rows    rows of recv (and of recv_scales), >= 0.
 * dtype        EP_DTYPE_BF16: recv [T*k, H] bf16, recv[pos[t,j]] = x[t];
 *              recv_scales unused (may be NULL).
 *              EP_DTYPE_FP8_E4M3_B128 (needs H % 128 == 0): recv [T*k, H]
 *              e4m3 bytes and recv_scales fp32 [T*k, H/128]; per token and
 *              128-column block b: s = amax|x[t, b]| / 448 (fp32 IEEE
 *              division), code = e4m3(x / s) with an fp32 IEEE division and
 *              round-to-nearest-even saturating to +-448; a block with
 *              amax = 0 gets s = 0 and signed-zero codes.
 *              EP_DTYPE_MXFP8_E4M3_B32 (needs H % 32 == 0; the OCP
 *              Microscaling MXFP8 format): recv [T*k, H] e4m3 bytes and
 *              recv_scales uint8 [T*k, H/32] E8M0 bytes; per 32-column block
 *              e = floor(log2 amax) - 8 clamped to [-127, 127] (amax = 0:
 *              -127), byte = e + 127, code = e4m3(x * 2^-e) nearest-even,
 *              saturating.
 *              Every copy of a token carries the same codes and scales.
 * recv         16-byte aligned.  recv_scales: 4-byte aligned for fp32.
 * Rows of recv not named by pos are left untouched.
 * Errors: EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED (H % 8, H % 128 for FP8,
 * H % 32 for MXFP8, k > 64), EP_ERR_ALIGNMENT, EP_ERR_CUDA.
 */
ep_status ep_dispatch(const void *x, int32_t T, int32_t H, int32_t k, const int32_t *pos,
                      int32_t dtype, void *recv, int32_t recv_rows, void *recv_scales,
                      int32_t *err_flag, void *stream);

/*
 * Steps 4 and 5 -- inverse gather and weighted combine ("Expert Parallelism
 * ...", section "Le pattern de communication all-to-all", Phase 2: results
 * return to their token and are combined weighted by the router scores).
 *
 * y       [y_rows, H] bf16 expert outputs in receive-row order, 16-byte
 *         aligned (y_rows = T*k after ep_get_layout).
 * pos     [T, k] int32 (from ep_get_layout); entries < 0 contribute nothing,
 *         rows >= y_rows contribute nothing and are flagged EP_FLAG_BAD_ROW.
 * topk_w  [T, k] fp32 router weights.
 * out     [T, H] bf16, 16-byte aligned:
 *         out[t, h] = bf16_rne( fma chain over j = 0..k-1 in slot order of
 *         w[t, j] * y[pos[t, j], h], accumulated in fp32 from 0 ).
 * H % 8 == 0.  Errors: EP_ERR_INVALID_ARG, EP_ERR_ALIGNMENT, EP_ERR_CUDA.
 */
ep_status ep_combine(const void *y, int32_t y_rows, const int32_t *pos, const float *topk_w, int32_t T,
                     int32_t H, int32_t k, void *out, int32_t *err_flag, void *stream);

/*
 * Steps 4 and 5 on FP8 expert outputs ("DeepEP de DeepSeek ...", section
 * "Support FP8 et MXFP8": FP8 payloads in both directions halve the bytes).
 *
 * yq           [y_rows, H] e4m3 codes, 16-byte aligned.
 * yscales      scale_dtype EP_DTYPE_FP8_E4M3_B128: fp32 [y_rows, H/128];
 *              EP_DTYPE_MXFP8_E4M3_B32: E8M0 bytes [y_rows, H/32].
 * pos, topk_w, out, err_flag as in ep_combine.
 * out[t, h] = bf16_rne( fp32 fma chain over j of (w[t,j] * block scale,
 * rounded to fp32 once per slot) * e4m3 value of yq[pos[t,j], h] ).  Errors
 * as ep_combine, plus EP_ERR_UNSUPPORTED when H is not a multiple of the
 * block width.
 */
ep_status ep_combine_fp8(const void *yq, const void *yscales, int32_t scale_dtype, int32_t y_rows,
                         const int32_t *pos, const float *topk_w, int32_t T, int32_t H, int32_t k,
                         void *out, int32_t *err_flag, void *stream);

/*
 * Capacity-limited layout: the capacity factor / token dropping lever of
 * "Expert Parallelism ...", section "Defis et optimisations" (Load
 * balancing).  Expert e owns the fixed receive rows [e*capacity,
 * (e+1)*capacity); entries are taken in flat (token, slot) order and an
 * expert's entries past its first `capacity` are dropped (pos = -1; a
 * combine then gives them no weight).  capacity >= 0; a capacity factor f
 * gives capacity = ceil(f * T * k / E).
 *
 * Outputs as ep_get_layout, except: expert_count[E] = kept entries;
 * expert_off[e] = e*capacity; rank_count[R] = kept entries of the rank;
 * rank_off[r] = r*experts_per_rank*capacity; rank_tokens[R] = distinct
 * tokens with a kept entry on the rank; expert_dropped[E] = entries past
 * capacity; src has E*capacity rows (-1 for an empty row).  The receive
 * buffer needs E*capacity rows.  workspace as ep_get_layout.  Limits as
 * ep_get_layout and E*capacity < 2^31.  Like ep_get_layout's larger
 * batches, this runs as one cooperative launch with a bounded grid barrier
 * (EP_FLAG_TIMEOUT if its wait runs out) unless one CTA per SM would hold
 * more than 4096 entries, then as three launches.
 */
ep_status ep_get_layout_capacity(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E,
                                 int32_t experts_per_rank, int32_t capacity, int32_t *expert_count,
                                 int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                                 int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos,
                                 int32_t *src, int32_t *err_flag, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Backward of the BF16 dispatch (a k-fold copy): the gradient of a source
 * row is the sum of its copies' gradients,
 *   grad_x[t, h] = bf16_rne( fp32 sum over j in slot order of grad_recv[pos[t,j], h] ),
 * a token with no copy getting zeros.  grad_recv [recv_rows, H] bf16, grad_x
 * [T, H] bf16, both 16-byte aligned; pos, k, H, err_flag as in ep_combine.
 * (Training is the pages' main setting: "DeepEP de DeepSeek ...", forward
 * and backward passes of pretraining.)
 */
ep_status ep_dispatch_backward(const void *grad_recv, int32_t recv_rows, const int32_t *pos, int32_t T,
                               int32_t H, int32_t k, void *grad_x, int32_t *err_flag, void *stream);

/*
 * Backward of the weighted combine out[t] = sum_j w[t,j] * y[pos[t,j]]:
 *   grad_y[pos[t,j], h] = bf16_rne(w[t,j] * grad_out[t, h])  (the exact product
 *                         rounded once, for products in fp32's normal range)
 *   grad_w[t, j]        = sum_h grad_out[t, h] * y[pos[t,j], h]  (fp32, fixed
 *                         reduction order; 0 for an empty slot)
 * grad_out [T, H] bf16, y and grad_y [y_rows, H] bf16 (16-byte aligned; rows
 * of grad_y not named by pos untouched), topk_w and grad_w [T, k] fp32.
 */
ep_status ep_combine_backward(const void *grad_out, const void *y, int32_t y_rows, const int32_t *pos,
                              const float *topk_w, int32_t T, int32_t H, int32_t k, void *grad_y,
                              float *grad_w, int32_t *err_flag, void *stream);

/*
 * Fused low-latency path for decode-sized batches ("DeepEP de DeepSeek
 * ...", section "Kernels low-latency dispatch et combine"; "Expert
 * Parallelism ...": decode messages of 100 KB - 2 MB): ep_gate,
 * ep_get_layout and ep_dispatch in ONE launch, with results identical to
 * the three separate calls.  Up to 512 tokens the launch is a grid of
 * thread-block clusters with no grid barrier: every cluster gates and lays
 * out the whole batch (its CTAs exchange per-expert token masks through
 * distributed shared memory) and scatters its share of the tokens.  Larger
 * batches take one cooperative launch with a grid barrier between gating
 * and layout.
 *
 * Arguments as those calls (cfg as ep_gate; experts_per_rank and the layout
 * outputs as ep_get_layout; x, H, dtype, recv, recv_rows, recv_scales as
 * ep_dispatch).  1 <= T and T*k <= 4096 (larger batches use the separate
 * calls: EP_ERR_UNSUPPORTED).  workspace: >= 8 bytes of device memory,
 * 4-byte aligned, whose first 4 bytes hold the grid barrier's arrival count:
 * zero it once before the first call; each call leaves it zero for the
 * next (calls sharing it must not overlap on the GPU).  The grid barrier
 * (batches past 512 tokens) waits at most about a second; if that ran out,
 * EP_FLAG_TIMEOUT is set in *err_flag, the outputs are incomplete and the
 * workspace must be zeroed again.
 * A device without cooperative launch returns EP_ERR_CUDA.
 */
ep_status ep_decode_dispatch(const float *scores, const float *bias, int32_t T, const ep_gate_cfg *cfg,
                             int32_t experts_per_rank, const void *x, int32_t H, int32_t dtype,
                             int32_t *topk_idx, float *topk_w, int32_t *expert_count,
                             int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                             int32_t *rank_tokens, int32_t *pos, int32_t *src, void *recv,
                             int32_t recv_rows, void *recv_scales, int32_t *err_flag, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * Check of the fused path's bounded grid barrier: one cooperative launch
 * whose CTAs wait for missing_arrivals arrivals that never come (0: none
 * missing, the barrier completes).  With missing_arrivals > 0 every CTA
 * polls spin_limit times (1 <= spin_limit <= 2^24; each poll sleeps about
 * 32 ns plus a global load), then sets EP_FLAG_TIMEOUT in *err_flag and
 * returns -- the wait ends on its own and the context stays usable.
 * workspace: >= 8 bytes, 4-byte aligned, cleared by this call.  The pages
 * have no counterpart to this call; it exists so that the timeout path is
 * tested on the GPU without a hang.
 */
ep_status ep_selftest_grid_barrier(int32_t missing_arrivals, int64_t spin_limit, int32_t *err_flag,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Static description of a status code. */
const char *ep_status_str(ep_status s);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
