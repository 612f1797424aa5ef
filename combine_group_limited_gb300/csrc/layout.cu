// layout.cu -- step 2: dispatch layout (counts, prefix sums, stable rows).
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le principe de
// base": whole experts per rank, here experts_per_rank contiguous experts per
// logical rank.  The hyper.ai Hybrid-EP story notes that sizing the receive
// buffers needs a synchronisation unless a fixed maximum is used; top-k with
// distinct experts fills at most T*k rows, so nothing here is read back to
// the host.
//
// Three launches over tiles of whole tokens (about 2048 entries each):
//  1. count:  per tile, per-expert entry counts and per-rank distinct-token
//             counts (shared-memory integer atomics; the totals do not depend
//             on their order).
//  2. scan:   one CTA: per expert, an exclusive scan over tiles (warp scans);
//             then an exclusive scan over experts and the per-rank sums.
//  3. place:  per tile, the stable row of every entry: 8 warps take
//             contiguous slices in flat order; __match_any_sync groups equal
//             experts inside a 32-entry chunk, so an entry's rank is the
//             popcount of lower lanes in its group plus the running count of
//             its warp, whose base is the tile's base plus the lower warps'
//             counts.  The result is the order a sequential walk gives.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kTileEntries = 2048;
constexpr int kScanThreads = 1024;
constexpr int kMaxExperts = 1024;

__device__ __forceinline__ bool valid_expert(int e, int E) { return (unsigned)e < (unsigned)E; }

__global__ void __launch_bounds__(kLayoutThreads) layout_count_kernel(
    const int32_t *__restrict__ idx, int T, int k, int E, int epr, int tile_tok, int nt,
    int32_t *__restrict__ ws_cnt, int32_t *__restrict__ ws_rt, int32_t *__restrict__ err_flag)
{
    extern __shared__ int32_t cnt_smem[];  // [E] expert counts, [R] rank token counts
    const int R = E / epr;
    for (int i = threadIdx.x; i < E + R; i += blockDim.x)
        cnt_smem[i] = 0;
    __syncthreads();

    const int tile = blockIdx.x;
    const int t0 = tile * tile_tok;
    const int t1 = min(T, t0 + tile_tok);
    int bad = 0;
    for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
        const int e = __ldg(idx + i);
        if (valid_expert(e, E))
            atomicAdd(&cnt_smem[e], 1);
        else if (e != -1)
            bad = 1;
    }
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        const int32_t *r_ = idx + (size_t)t * k;
        for (int j = 0; j < k; ++j) {
            const int e = __ldg(r_ + j);
            if (!valid_expert(e, E))
                continue;
            const int r = e / epr;
            bool first = true;
            for (int jj = 0; jj < j; ++jj) {
                const int e2 = __ldg(r_ + jj);
                if (valid_expert(e2, E) && e2 / epr == r) {
                    first = false;
                    break;
                }
            }
            if (first)
                atomicAdd(&cnt_smem[E + r], 1);
        }
    }
    if (bad && err_flag)
        atomicOr(err_flag, (int)1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        ws_cnt[(size_t)e * nt + tile] = cnt_smem[e];
    for (int r = threadIdx.x; r < R; r += blockDim.x)
        ws_rt[(size_t)r * nt + tile] = cnt_smem[E + r];
}

// Inclusive warp scan.
__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off)
            v += n;
    }
    return v;
}

__global__ void __launch_bounds__(kScanThreads) layout_scan_kernel(
    int T, int k, int E, int epr, int nt, int32_t *__restrict__ ws_cnt, const int32_t *__restrict__ ws_rt,
    int32_t *__restrict__ expert_count, int32_t *__restrict__ expert_off, int32_t *__restrict__ rank_count,
    int32_t *__restrict__ rank_off, int32_t *__restrict__ rank_tokens, int32_t *__restrict__ src)
{
    __shared__ int32_t s_cnt[kMaxExperts];
    __shared__ int32_t s_wsum[kScanThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int R = E / epr;

    // Per expert: exclusive scan over tiles, in place; total = expert count.
    for (int e = warp; e < E; e += nwarps) {
        int32_t *col = ws_cnt + (size_t)e * nt;
        int running = 0;
        for (int base = 0; base < nt; base += 32) {
            const int tl = base + lane;
            const int v = tl < nt ? col[tl] : 0;
            const int incl = warp_incl_scan(v, lane);
            if (tl < nt)
                col[tl] = running + incl - v;
            running += __shfl_sync(kFullMask, incl, 31);
        }
        if (lane == 0) {
            s_cnt[e] = running;
            expert_count[e] = running;
        }
    }
    // Per rank: distinct tokens summed over tiles.
    for (int r = warp; r < R; r += nwarps) {
        const int32_t *col = ws_rt + (size_t)r * nt;
        int acc = 0;
        for (int tl = lane; tl < nt; tl += 32)
            acc += col[tl];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc += __shfl_xor_sync(kFullMask, acc, off);
        if (lane == 0)
            rank_tokens[r] = acc;
    }
    __syncthreads();

    // Exclusive scan over experts (E <= 1024 = one value per thread).
    const int e = threadIdx.x;
    const int v = e < E ? s_cnt[e] : 0;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31)
        s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int ws = lane < nwarps ? s_wsum[lane] : 0;
        const int wi = warp_incl_scan(ws, lane);
        if (lane < nwarps)
            s_wsum[lane] = wi - ws;
    }
    __syncthreads();
    const int excl = s_wsum[warp] + incl - v;
    __syncthreads();
    if (e < E)
        s_cnt[e] = excl;  // reuse as offsets
    __shared__ int32_t s_total;
    if (e == E - 1)
        s_total = excl + v;
    __syncthreads();
    const int total = s_total;
    if (e < E)
        expert_off[e] = excl;
    if (e == 0)
        expert_off[E] = total;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int lo = s_cnt[r * epr];
        const int hi = (r + 1) * epr < E ? s_cnt[(r + 1) * epr] : total;
        rank_off[r] = lo;
        rank_count[r] = hi - lo;
    }
    if (threadIdx.x == 0)
        rank_off[R] = total;
    // Rows no entry lands on.
    for (int i = total + threadIdx.x; i < T * k; i += blockDim.x)
        src[i] = -1;
}

__global__ void __launch_bounds__(kLayoutThreads) layout_place_kernel(
    const int32_t *__restrict__ idx, int T, int k, int E, int tile_tok, int nt, const int32_t *__restrict__ ws_cnt,
    const int32_t *__restrict__ expert_off, int32_t *__restrict__ pos, int32_t *__restrict__ src,
    int32_t *__restrict__ err_flag)
{
    extern __shared__ int32_t hist[];  // [kLayoutWarps][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x;
    const int n0 = tile * tile_tok * k;
    const int n1 = min(T, (tile + 1) * tile_tok) * k;
    const int per_warp = (((n1 - n0) + kLayoutWarps * 32 - 1) / (kLayoutWarps * 32)) * 32;
    const int w0 = n0 + warp * per_warp;
    const int w1 = min(n1, w0 + per_warp);
    int32_t *my = hist + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int n_total = T * k;

    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x)
        hist[i] = 0;
    __syncthreads();

    // A: each warp's per-expert counts.
    for (int c = w0; c < w1; c += 32) {
        const int i = c + lane;
        const int e = i < w1 ? __ldg(idx + i) : -1;
        const int key = valid_expert(e, E) ? e : E;
        const unsigned grp = __match_any_sync(kFullMask, key);
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();

    // B: warp bases = expert offset + tile base + counts of the lower warps.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int base = __ldg(expert_off + e) + __ldg(ws_cnt + (size_t)e * nt + tile);
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = base;
            base += c;
        }
    }
    __syncthreads();

    // C: rows in flat order.
    for (int c = w0; c < w1; c += 32) {
        const int i = c + lane;
        const bool in = i < w1;
        const int e = in ? __ldg(idx + i) : -1;
        const int key = valid_expert(e, E) ? e : E;
        const unsigned grp = __match_any_sync(kFullMask, key);
        if (key < E) {
            const int p = my[key] + __popc(grp & lt_mask);
            // p < T*k by construction; checked so that an index tensor
            // changed between the launches cannot send a store astray.
            if (p >= 0 && p < n_total) {
                pos[i] = p;
                src[p] = i;
            } else {
                pos[i] = -1;
                if (err_flag)
                    atomicOr(err_flag, 2);
            }
        } else if (in) {
            pos[i] = -1;
        }
        __syncwarp();
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
}

}  // namespace

int layout_tile_tokens(int k)
{
    const int tt = kTileEntries / (k > 0 ? k : 1);
    return tt < 1 ? 1 : tt;
}

int layout_num_tiles(int T, int k)
{
    const int tt = layout_tile_tokens(k);
    return (T + tt - 1) / tt;
}

size_t layout_workspace_bytes(int T, int k, int E, int epr)
{
    const size_t nt = (size_t)layout_num_tiles(T, k);
    const size_t R = (size_t)(E / epr);
    const size_t bytes = nt * ((size_t)E + R) * sizeof(int32_t);
    return ((bytes + 255) / 256) * 256 + 256;
}

cudaError_t launch_layout(const int32_t *topk_idx, int T, int k, int E, int epr, int32_t *expert_count,
                          int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                          int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, cudaStream_t st)
{
    const int tile_tok = layout_tile_tokens(k);
    const int nt = layout_num_tiles(T, k);
    const int R = E / epr;
    int32_t *ws_cnt = static_cast<int32_t *>(workspace);
    int32_t *ws_rt = ws_cnt + (size_t)nt * E;
    if (nt > 0) {
        layout_count_kernel<<<nt, kLayoutThreads, (E + R) * sizeof(int32_t), st>>>(
            topk_idx, T, k, E, epr, tile_tok, nt, ws_cnt, ws_rt, err_flag);
    }
    layout_scan_kernel<<<1, kScanThreads, 0, st>>>(T, k, E, epr, nt, ws_cnt, ws_rt, expert_count, expert_off,
                                                   rank_count, rank_off, rank_tokens, src);
    if (nt > 0) {
        layout_place_kernel<<<nt, kLayoutThreads, kLayoutWarps * E * sizeof(int32_t), st>>>(
            topk_idx, T, k, E, tile_tok, nt, ws_cnt, expert_off, pos, src, err_flag);
    }
    return cudaGetLastError();
}

}  // namespace ep
