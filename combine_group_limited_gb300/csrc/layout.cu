// layout.cu -- step 2: dispatch layout (counts, prefix sums, stable rows).
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le principe de
// base": whole experts per rank, here experts_per_rank contiguous experts per
// logical rank.  The hyper.ai Hybrid-EP story notes that sizing the receive
// buffers needs a synchronisation unless a fixed maximum is used; top-k with
// distinct experts fills at most T*k rows, so nothing here is read back to
// the host.
//
// Batches of up to 4096 entries take one launch (layout_small_kernel).  Larger
// ones, and capacity mode, take one cooperative launch (route.cu) while a
// grid of one CTA per SM covers them with at most 4096 entries per CTA;
// beyond that they take three launches over tiles of whole tokens (about 512
// entries each):
//  1. count:  per tile, per-expert entry counts and per-rank distinct-token
//             counts (shared-memory integer atomics; the totals do not depend
//             on their order).  Workspace columns [E][tiles], [R][tiles].
//  2. scan:   one warp per column: experts get an exclusive scan over tiles
//             (in place) and their total; ranks get their distinct-token sum.
//  3. place:  every CTA scans the E expert totals itself (a block scan of at
//             most 1024 values, 4 per thread) to get expert_off, then gives each entry its
//             stable row: 8 warps take contiguous slices in flat order;
//             a ballot per key bit groups equal experts inside a 32-entry chunk,
//             so an entry's row is its expert's offset + the tile's base + the
//             lower warps' counts + the running count of its warp + the
//             popcount of lower lanes in its group -- the order a sequential
//             walk gives.  CTA 0 also writes the offsets and the per-rank
//             arrays; all CTAs fill src past the last row with -1.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kTileEntries = 512;
constexpr int kPlaceThreads = 256;
constexpr int kPlaceWarps = kPlaceThreads / 32;
constexpr int kMaxExperts = 1024;
constexpr int kSmallThreads = 512;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallEntries = kSmallLayoutEntries;
constexpr int kSmallChunks = kSmallEntries / (kSmallWarps * 32);  // 32-entry chunks per warp

__device__ __forceinline__ bool valid_expert(int e, int E) { return (unsigned)e < (unsigned)E; }

__global__ void __launch_bounds__(kLayoutThreads) layout_count_kernel(
    const int32_t *__restrict__ idx, int T, int k, int E, int epr, int tile_tok, int nt,
    int32_t *__restrict__ ws_cnt, int32_t *__restrict__ ws_rt, int32_t *__restrict__ err_flag)
{
    // [E] expert counts, [R] rank token counts, [kTileEntries] the tile's ranks
    extern __shared__ int32_t cnt_smem[];
    const int R = E / epr;
    int32_t *s_rank = cnt_smem + E + R;
    for (int i = threadIdx.x; i < E + R; i += blockDim.x)
        cnt_smem[i] = 0;
    __syncthreads();

    const int tile = blockIdx.x;
    const int n0 = tile * tile_tok * k;
    const int n1 = min(T, (tile + 1) * tile_tok) * k;
    const int lane = threadIdx.x & 31;
    const int eb = key_bits((unsigned)E), rb = key_bits((unsigned)R);
    int bad = 0;
    // Warp-uniform loops: the counts are warp-aggregated (warp_count).
    for (int base = n0 + (threadIdx.x & ~31); base < n1; base += blockDim.x) {
        const int i = base + lane;
        const bool in = i < n1;
        const int e = in ? __ldg(idx + i) : -1;
        const bool ok = valid_expert(e, E);
        bad |= in && !ok && e != -1;
        warp_count(cnt_smem, ok ? (unsigned)e : 0u, ok, eb);
        if (in)
            s_rank[i - n0] = ok ? e / epr : -1;
    }
    __syncthreads();
    // Distinct tokens per rank: an entry counts if no earlier slot of its
    // token is on the same rank.
    for (int base = n0 + (threadIdx.x & ~31); base < n1; base += blockDim.x) {
        const int i = base + lane;
        const int r = i < n1 ? s_rank[i - n0] : -1;
        bool first = r >= 0;
        if (first) {
            const int j = (i - n0) % k;
            const int32_t *tok = s_rank + (i - n0 - j);
            for (int jj = 0; jj < j; ++jj)
                first &= tok[jj] != r;
        }
        warp_count(cnt_smem + E, first ? (unsigned)r : 0u, first, rb);
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

// One warp per column: columns [0, E) are expert columns (scanned in place,
// total to expert_count), columns [E, E+R) are rank columns (summed into
// rank_tokens).
__global__ void __launch_bounds__(kLayoutThreads) layout_scan_kernel(
    int E, int R, int nt, int zero_rank_tokens, int32_t *__restrict__ ws_cnt, const int32_t *__restrict__ ws_rt,
    int32_t *__restrict__ expert_count, int32_t *__restrict__ rank_tokens)
{
    const int lane = threadIdx.x & 31;
    const int col = blockIdx.x * kLayoutWarps + (threadIdx.x >> 5);
    if (col >= E + R)
        return;
    if (col < E) {
        int32_t *c = ws_cnt + (size_t)col * nt;
        int running = 0;
        for (int base = 0; base < nt; base += 128) {
            int v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int tl = base + 32 * u + lane;
                v[u] = tl < nt ? c[tl] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int tl = base + 32 * u + lane;
                const int incl = warp_incl_scan(v[u], lane);
                if (tl < nt)
                    c[tl] = running + incl - v[u];
                running += __shfl_sync(kFullMask, incl, 31);
            }
        }
        if (lane == 0)
            expert_count[col] = running;
    } else {
        const int r = col - E;
        const int32_t *c = ws_rt + (size_t)r * nt;
        int acc = 0;
        for (int tl = lane; tl < nt; tl += 32)
            acc += c[tl];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc += __shfl_xor_sync(kFullMask, acc, off);
        if (lane == 0)
            rank_tokens[r] = zero_rank_tokens ? 0 : acc;
    }
}

// kCap: capacity mode -- expert e owns the fixed rows [e*cap, (e+1)*cap); an
// entry whose stable rank within its expert is >= cap is dropped (pos = -1).
template <bool kCap>
__global__ void __launch_bounds__(kPlaceThreads) layout_place_kernel(
    const int32_t *__restrict__ idx, int T, int k, int E, int epr, int tile_tok, int nt, int cap,
    const int32_t *__restrict__ ws_cnt, int32_t *__restrict__ expert_count, int32_t *__restrict__ expert_off,
    int32_t *__restrict__ rank_count, int32_t *__restrict__ rank_off, int32_t *__restrict__ rank_tokens,
    int32_t *__restrict__ expert_dropped, int32_t *__restrict__ pos, int32_t *__restrict__ src,
    int32_t *__restrict__ err_flag)
{
    // hist [kPlaceWarps][E], off [E]; capacity mode adds kept ranks
    // [kTileEntries] and kept distinct-token counts [R]
    extern __shared__ int32_t place_smem[];
    int32_t *hist = place_smem;
    int32_t *s_off = place_smem + kPlaceWarps * E;
    int32_t *s_krank = s_off + E;
    int32_t *s_rt = s_krank + kTileEntries;
    __shared__ int32_t s_wsum[kPlaceWarps];
    __shared__ int32_t s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x;
    const int R = E / epr;
    const int n_total = T * k;
    const int n_rows = kCap ? E * cap : n_total;

    if (kCap) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            s_off[e] = e * cap;
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            s_rt[r] = 0;
        if (threadIdx.x == 0)
            s_total = E * cap;
    } else {
        // Expert offsets: exclusive scan of the E <= 1024 totals, kPerThread
        // consecutive experts per thread.
        constexpr int kPerThread = kMaxExperts / kPlaceThreads;
        const int e0 = threadIdx.x * kPerThread;
        int v[kPerThread];
        int sum = 0;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            v[u] = e0 + u < E ? __ldg(expert_count + e0 + u) : 0;
            sum += v[u];
        }
        const int incl = warp_incl_scan(sum, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = lane < kPlaceWarps ? s_wsum[lane] : 0;
            const int wi = warp_incl_scan(ws, lane);
            if (lane < kPlaceWarps)
                s_wsum[lane] = wi - ws;
        }
        __syncthreads();
        int run = s_wsum[warp] + incl - sum;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            if (e0 + u < E)
                s_off[e0 + u] = run;
            if (e0 + u == E - 1)
                s_total = run + v[u];
            run += v[u];
        }
    }
    for (int i = threadIdx.x; i < kPlaceWarps * E; i += blockDim.x)
        hist[i] = 0;
    __syncthreads();
    const int total = s_total;
    if (tile == 0 && kCap) {
        // The scan left each expert's total entries in expert_count; keep
        // at most cap of them.  s_off is free for the kept counts here.
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int all = expert_count[e];
            const int kept = all < cap ? all : cap;
            s_off[e] = kept;
            expert_dropped[e] = all - kept;
            expert_off[e] = e * cap;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            expert_count[e] = s_off[e];
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            int c = 0;
            for (int e = r * epr; e < (r + 1) * epr; ++e)
                c += s_off[e];
            rank_count[r] = c;
            rank_off[r] = r * epr * cap;
        }
        if (threadIdx.x == 0) {
            expert_off[E] = E * cap;
            rank_off[R] = R * epr * cap;
        }
    } else if (tile == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            expert_off[e] = s_off[e];
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            const int lo = s_off[r * epr];
            const int hi = (r + 1) * epr < E ? s_off[(r + 1) * epr] : total;
            rank_off[r] = lo;
            rank_count[r] = hi - lo;
        }
        if (threadIdx.x == 0) {
            expert_off[E] = total;
            rank_off[R] = total;
        }
    }
    // Rows no entry lands on (capacity mode: the launcher cleared src).
    if (!kCap)
        for (int i = total + blockIdx.x * blockDim.x + threadIdx.x; i < n_total; i += gridDim.x * blockDim.x)
            src[i] = -1;

    const int n0 = tile * tile_tok * k;
    const int n1 = min(T, (tile + 1) * tile_tok) * k;
    const int per_warp = (((n1 - n0) + kPlaceWarps * 32 - 1) / (kPlaceWarps * 32)) * 32;
    const int w0 = n0 + warp * per_warp;
    const int w1 = min(n1, w0 + per_warp);
    int32_t *my = hist + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int eb = key_bits((unsigned)E);  // keys 0..E (E marks an invalid entry)

    // A: each warp's per-expert counts.
    for (int c = w0; c < w1; c += 32) {
        const int i = c + lane;
        const int e = i < w1 ? __ldg(idx + i) : -1;
        const int key = valid_expert(e, E) ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();

    // B: warp bases = tile base within the expert + counts of the lower warps
    // (+ the expert's offset outside capacity mode).
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int base = (kCap ? 0 : s_off[e]) + __ldg(ws_cnt + (size_t)e * nt + tile);
        for (int w = 0; w < kPlaceWarps; ++w) {
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
        const unsigned grp = peer_mask((unsigned)key, eb);
        int kept_rank = -1;
        if (key < E) {
            const int r = my[key] + __popc(grp & lt_mask);
            // In capacity mode r is the rank within the expert; otherwise the
            // row.  Rows stay below the row count by construction; checked so
            // that an index tensor changed between the launches cannot send a
            // store astray.
            const int p = kCap ? (r < cap ? e * cap + r : -1) : r;
            if (p >= 0 && p < n_rows) {
                pos[i] = p;
                src[p] = i;
                kept_rank = e / epr;
            } else {
                pos[i] = -1;
                if (!kCap && err_flag)
                    atomicOr(err_flag, 2);
            }
        } else if (in) {
            pos[i] = -1;
        }
        if (kCap && in)
            s_krank[i - n0] = kept_rank;
        __syncwarp();
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }

    if (kCap) {
        // Distinct tokens with a kept entry, per rank.
        __syncthreads();
        const int rb = key_bits((unsigned)R);
        for (int base = n0 + (threadIdx.x & ~31); base < n1; base += blockDim.x) {
            const int i = base + lane;
            const int r = i < n1 ? s_krank[i - n0] : -1;
            bool first = r >= 0;
            if (first) {
                const int j = (i - n0) % k;
                const int32_t *tok = s_krank + (i - n0 - j);
                for (int jj = 0; jj < j; ++jj)
                    first &= tok[jj] != r;
            }
            warp_count(s_rt, first ? (unsigned)r : 0u, first, rb);
        }
        __syncthreads();
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            if (s_rt[r])
                atomicAdd(rank_tokens + r, s_rt[r]);
    }
}

// Small batches (T*k <= kSmallEntries): the whole layout in one CTA and one
// launch -- the three-launch path is latency-bound there.  Same results.
// Each warp owns a contiguous slice of at most kSmallChunks x 32 entries and
// loads it into registers once (no load waits inside the passes): counts and
// distinct tokens by warp-aggregated shared counters, an exclusive scan of
// the counts, then stable rows -- ballot peer masks rank equal experts inside
// a 32-entry chunk, per-warp running counts start at the lower warps' counts.
__global__ void __launch_bounds__(kSmallThreads) layout_small_kernel(
    const int32_t *__restrict__ idx, int T, int k, int E, int epr, int32_t *__restrict__ expert_count,
    int32_t *__restrict__ expert_off, int32_t *__restrict__ rank_count, int32_t *__restrict__ rank_off,
    int32_t *__restrict__ rank_tokens, int32_t *__restrict__ pos, int32_t *__restrict__ src,
    int32_t *__restrict__ err_flag)
{
    extern __shared__ int32_t ssm[];  // off [E], rank tokens [R], hist [kSmallWarps][E], ranks [N]
    const int R = E / epr;
    const int N = T * k;
    int32_t *s_off = ssm;
    int32_t *s_rt = s_off + E;
    int32_t *hist = s_rt + R;
    int32_t *s_rank = hist + kSmallWarps * E;
    __shared__ int32_t s_wsum[kSmallWarps];
    __shared__ int32_t s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < E + R + kSmallWarps * E; i += blockDim.x)
        ssm[i] = 0;
    const int per_warp = ((N + kSmallWarps * 32 - 1) / (kSmallWarps * 32)) * 32;  // <= kSmallChunks * 32
    const int w0 = warp * per_warp;
    // ev: the entry's expert, -1 for an empty slot, -2 outside the slice.  An
    // index outside [0, E) other than -1 (including -2) is flagged here and
    // becomes an empty slot, so -2 never comes from the caller's indices.
    int ev[kSmallChunks];
    int bad = 0;
#pragma unroll
    for (int c = 0; c < kSmallChunks; ++c) {
        const int i = w0 + 32 * c + lane;
        int e = -2;
        if (32 * c < per_warp && i < N) {
            e = __ldg(idx + i);
            if (e != -1 && !valid_expert(e, E)) {
                bad = 1;
                e = -1;
            }
        }
        ev[c] = e;
    }
    __syncthreads();
    const int eb = key_bits((unsigned)E), rb = key_bits((unsigned)R);
#pragma unroll
    for (int c = 0; c < kSmallChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int e = ev[c];
        const bool ok = valid_expert(e, E);
        warp_count(s_off, ok ? (unsigned)e : 0u, ok, eb);
        if (e != -2)
            s_rank[i] = ok ? e / epr : -1;
    }
    if (bad && err_flag)
        atomicOr(err_flag, 1);
    __syncthreads();
    // Distinct tokens per rank: an entry counts if no earlier slot of its
    // token is on the same rank (ranks read from shared memory).
#pragma unroll
    for (int c = 0; c < kSmallChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int r = (ev[c] != -2) ? s_rank[i] : -1;
        bool first = r >= 0;
        if (first) {
            const int j = i % k;
            for (int jj = 0; jj < j; ++jj)
                first &= s_rank[i - j + jj] != r;
        }
        warp_count(s_rt, first ? (unsigned)r : 0u, first, rb);
    }
    __syncthreads();
    {
        constexpr int kPerThread = kMaxExperts / kSmallThreads;
        const int e0 = threadIdx.x * kPerThread;
        int v[kPerThread];
        int sum = 0;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            v[u] = e0 + u < E ? s_off[e0 + u] : 0;
            sum += v[u];
        }
        const int incl = warp_incl_scan(sum, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = lane < kSmallWarps ? s_wsum[lane] : 0;
            const int wi = warp_incl_scan(ws, lane);
            if (lane < kSmallWarps)
                s_wsum[lane] = wi - ws;
        }
        __syncthreads();
        int run = s_wsum[warp] + incl - sum;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            if (e0 + u < E) {
                s_off[e0 + u] = run;
                expert_count[e0 + u] = v[u];
                expert_off[e0 + u] = run;
            }
            if (e0 + u == E - 1)
                s_total = run + v[u];
            run += v[u];
        }
    }
    __syncthreads();
    const int total = s_total;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int lo = s_off[r * epr];
        const int hi = (r + 1) * epr < E ? s_off[(r + 1) * epr] : total;
        rank_off[r] = lo;
        rank_count[r] = hi - lo;
        rank_tokens[r] = s_rt[r];
    }
    if (threadIdx.x == 0) {
        expert_off[E] = total;
        rank_off[R] = total;
    }
    for (int i = total + threadIdx.x; i < N; i += blockDim.x)
        src[i] = -1;

    int32_t *my = hist + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int c = 0; c < kSmallChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int e = ev[c];
        const int key = valid_expert(e, E) ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int base = s_off[e];
        for (int w = 0; w < kSmallWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = base;
            base += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kSmallChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int e = ev[c];
        const int key = valid_expert(e, E) ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (key < E) {
            const int p = my[key] + __popc(grp & lt_mask);
            if (p >= 0 && p < N) {
                pos[i] = p;
                src[p] = i;
            } else {
                pos[i] = -1;
            }
        } else if (e == -1 || (e != -2 && i < N)) {
            pos[i] = -1;
        }
        __syncwarp();
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
}

// Zero counts for an empty batch (no tile runs).
__global__ void layout_empty_kernel(int E, int epr, int cap, int32_t *expert_count, int32_t *expert_off,
                                    int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                                    int32_t *expert_dropped)
{
    const int R = E / epr;
    const int c = cap < 0 ? 0 : cap;  // capacity mode keeps its fixed offsets
    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
        if (i < E) {
            expert_count[i] = 0;
            if (expert_dropped)
                expert_dropped[i] = 0;
        }
        expert_off[i] = i * c;
    }
    for (int i = threadIdx.x; i <= R; i += blockDim.x) {
        if (i < R) {
            rank_count[i] = 0;
            rank_tokens[i] = 0;
        }
        rank_off[i] = i * epr * c;
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

// Workspace: 256 bytes whose first 4 are the single-launch path's grid
// barrier count (no other path touches them), then either the per-tile
// counts of the three-launch path or the per-CTA rows of the single-launch
// one.
size_t layout_workspace_bytes(int T, int k, int E, int epr)
{
    const size_t nt = (size_t)layout_num_tiles(T, k);
    const size_t R = (size_t)(E / epr);
    const size_t bytes = ((nt * ((size_t)E + R) * sizeof(int32_t) + 255) / 256) * 256 + 256;
    const size_t single = route_workspace_bytes(E);
    return bytes > single ? bytes : single;
}

cudaError_t launch_layout_impl(const int32_t *topk_idx, int T, int k, int E, int epr, int cap,
                               int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                               int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos, int32_t *src,
                               int32_t *err_flag, void *workspace, cudaStream_t st)
{
    const bool capped = cap >= 0;
    const int tile_tok = layout_tile_tokens(k);
    const int nt = layout_num_tiles(T, k);
    const int R = E / epr;
    if (nt == 0) {
        if (capped && (size_t)E * cap > 0) {
            cudaError_t e = cudaMemsetAsync(src, 0xFF, (size_t)E * cap * sizeof(int32_t), st);  // -1
            if (e != cudaSuccess)
                return e;
        }
        layout_empty_kernel<<<1, 256, 0, st>>>(E, epr, cap, expert_count, expert_off, rank_count, rank_off,
                                               rank_tokens, expert_dropped);
        return cudaGetLastError();
    }
    if (!capped && T * k <= kSmallEntries) {
        const size_t smem = ((size_t)E + R + (size_t)kSmallWarps * E + (size_t)T * k) * sizeof(int32_t);
        if (smem > 48 * 1024) {
            static PerDeviceCache<1> attr;  // the largest size any call can need, once per device
            const cudaError_t e = raise_smem_limit(
                attr, (const void *)layout_small_kernel,
                ((size_t)kMaxExperts * (kSmallWarps + 2) + kSmallEntries) * sizeof(int32_t));
            if (e != cudaSuccess)
                return e;
        }
        layout_small_kernel<<<1, kSmallThreads, smem, st>>>(topk_idx, T, k, E, epr, expert_count, expert_off,
                                                            rank_count, rank_off, rank_tokens, pos, src, err_flag);
        return cudaGetLastError();
    }
    // Mid-size batches (up to 16 CTAs of 4096 entries) and small capacity
    // layouts: one thread-block cluster, no barrier and no workspace.
    // Measured on GB300 it beats the grid-wide launch there (Mixtral shape
    // 9.8 against 13.0 us cold; decode-sized capacity layout 4.9 against
    // 16.5 us back to back); larger batches spread their scattered stores
    // over every SM with the grid-wide launch instead.
    if ((capped || T * k > kSmallEntries) && (long long)T * k <= kClusterLayoutEntries &&
        layout_cluster_supported(T, k, E, epr))
        return launch_layout_cluster(topk_idx, T, k, E, epr, cap, expert_count, expert_off, rank_count, rank_off,
                                     rank_tokens, expert_dropped, pos, src, err_flag, st);
    if (route_supported(T, k, E, epr, false) && (capped || T * k > kSmallEntries)) {
        // one cooperative launch; its barrier's arrival count starts at zero
        cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(unsigned), st);
        if (e != cudaSuccess)
            return e;
        return launch_route(nullptr, nullptr, nullptr, topk_idx, nullptr, nullptr, T, k, E, epr, expert_count,
                            expert_off, rank_count, rank_off, rank_tokens, pos, src, err_flag, workspace, st,
                            capped ? cap : -1, expert_dropped);
    }
    if (capped && (size_t)E * cap > 0) {
        cudaError_t e = cudaMemsetAsync(src, 0xFF, (size_t)E * cap * sizeof(int32_t), st);  // -1
        if (e != cudaSuccess)
            return e;
    }
    int32_t *ws_cnt = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + 256);
    int32_t *ws_rt = ws_cnt + (size_t)nt * E;
    layout_count_kernel<<<nt, kLayoutThreads, (E + R + kTileEntries) * sizeof(int32_t), st>>>(
        topk_idx, T, k, E, epr, tile_tok, nt, ws_cnt, ws_rt, err_flag);
    const int scan_grid = (E + R + kLayoutWarps - 1) / kLayoutWarps;
    layout_scan_kernel<<<scan_grid, kLayoutThreads, 0, st>>>(E, R, nt, capped ? 1 : 0, ws_cnt, ws_rt, expert_count,
                                                             rank_tokens);
    const size_t place_smem =
        ((size_t)kPlaceWarps * E + E + (capped ? (size_t)kTileEntries + R : 0)) * sizeof(int32_t);
    if (capped)
        layout_place_kernel<true><<<nt, kPlaceThreads, place_smem, st>>>(
            topk_idx, T, k, E, epr, tile_tok, nt, cap, ws_cnt, expert_count, expert_off, rank_count, rank_off,
            rank_tokens, expert_dropped, pos, src, err_flag);
    else
        layout_place_kernel<false><<<nt, kPlaceThreads, place_smem, st>>>(
            topk_idx, T, k, E, epr, tile_tok, nt, 0, ws_cnt, expert_count, expert_off, rank_count, rank_off,
            rank_tokens, expert_dropped, pos, src, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_layout(const int32_t *topk_idx, int T, int k, int E, int epr, int32_t *expert_count,
                          int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                          int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, cudaStream_t st)
{
    return launch_layout_impl(topk_idx, T, k, E, epr, -1, expert_count, expert_off, rank_count, rank_off,
                              rank_tokens, nullptr, pos, src, err_flag, workspace, st);
}

cudaError_t launch_layout_capacity(const int32_t *topk_idx, int T, int k, int E, int epr, int cap,
                                   int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                                   int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos, int32_t *src,
                                   int32_t *err_flag, void *workspace, cudaStream_t st)
{
    return launch_layout_impl(topk_idx, T, k, E, epr, cap, expert_count, expert_off, rank_count, rank_off,
                              rank_tokens, expert_dropped, pos, src, err_flag, workspace, st);
}

}  // namespace ep
