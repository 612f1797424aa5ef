// route.cu -- routing of a whole batch in one cooperative launch: the
// group-limited gating (optional) and the dispatch layout.
//
// "DeepEP de DeepSeek ...", section "Group-limited gating algorithm" (the
// gating); "Expert Parallelism (Parallelisme d'experts)", section "Le
// principe de base" (a rank's experts are contiguous; the counts and offsets
// the dispatch writes into).  Done separately, these are four short,
// latency-bound launches at full size (gating, then count / scan / place);
// here one grid of one CTA per SM does all of it:
//   1. each CTA owns a contiguous range of whole tokens; with gating on it
//      gates them (gate_impl.cuh), else it reads their chosen experts;
//   2. it counts its entries per expert in per-warp shared counters (ballot
//      peer masks; no atomics), turns them into per-warp offsets (a warp scan
//      per expert), counts its distinct tokens per rank, and publishes its
//      per-expert count row;
//   3. a grid barrier (bounded wait; past its limit EP_FLAG_TIMEOUT);
//   4. it sums the count rows of the CTAs before it and of all CTAs (16-byte
//      loads through L2), scans the totals into expert offsets and gives
//      each of its entries its stable row: the expert's offset + the
//      entries of earlier CTAs + those of earlier warps + the equal lower
//      lanes.  CTA 0 writes the counts and offsets.
// Results are those of the separate calls, bit for bit.
#include "coop.cuh"
#include "gate_impl.cuh"

namespace ep {

namespace {

constexpr int kRtThreads = 1024;
constexpr int kRtWarps = kRtThreads / 32;
constexpr int kRtChunks = 4;                            // 32-entry chunks per warp
constexpr int kRtMaxRange = kRtWarps * 32 * kRtChunks;  // entries per CTA
constexpr int kRtMaxExperts = 1024;                     // == kRtThreads: one thread per expert in the scan
constexpr int kRtMaxCtas = 160;
constexpr int kRtWhStride = kRtWarps + 1;  // per-expert row of per-warp counts, padded against bank conflicts
constexpr int kRtMaxPhases = 32;           // CTA rows summed per thread in the column sums: C / phases

struct RouteArgs {
    const float *scores;
    const float *bias;
    GateParams gp;
    int group_lanes, vec_rows;
    int32_t *topk_idx;  // out when gating, else in
    float *topk_w;
    int T, k, E, E4, epr;
    int32_t *expert_count, *expert_off, *rank_count, *rank_off, *rank_tokens, *pos, *src;
    int32_t *err_flag;
    int cap;                  // >= 0: capacity mode (expert e owns rows [e*cap, (e+1)*cap)); -1: dropless
    int32_t *expert_dropped;  // [E], capacity mode
    unsigned *barrier;  // arrival count, zero at launch
    int32_t *rows;      // [gridDim.x][E4] per-CTA expert counts
    long long spin_limit;
};

__host__ __device__ inline int round4(int v) { return (v + 3) & ~3; }

// Threads per 4-expert column in the column sums.
__host__ __device__ inline int route_phases(int E4)
{
    const int p = kRtThreads / (E4 / 4);
    return p < kRtMaxPhases ? p : kRtMaxPhases;
}

// Capacity mode after the column sums (s_tot: every entry per expert; s_pre:
// entries of earlier CTAs): expert e keeps its first cap entries in flat
// order, in rows [e*cap, (e+1)*cap); later ones are dropped (pos = -1).
// src was cleared to -1 before the launch.  Distinct tokens per rank count
// kept entries only.
__device__ __forceinline__ void route_place_capped(const RouteArgs &a, const int32_t *s_tot, const int32_t *s_pre,
                                                   int32_t *s_wh, int32_t *s_rk, int32_t *s_rt,
                                                   const int (&ev)[kRtChunks], int per_warp, int w0, int n_lo,
                                                   int eb, int rb)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E, epr = a.epr, R = E / epr, cap = a.cap, k = a.k;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int tot = s_tot[e], kept = tot < cap ? tot : cap;
            a.expert_count[e] = kept;
            a.expert_dropped[e] = tot - kept;
            a.expert_off[e] = e * cap;
        }
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            int kept = 0;
            for (int e = r * epr; e < (r + 1) * epr; ++e)
                kept += s_tot[e] < cap ? s_tot[e] : cap;
            a.rank_count[r] = kept;
            a.rank_off[r] = r * epr * cap;
        }
        if (threadIdx.x == 0) {
            a.expert_off[E] = E * cap;
            a.rank_off[R] = E * cap;
        }
    }
    // each warp's first rank within the expert: earlier CTAs + earlier warps
    for (int e = warp; e < E; e += kRtWarps)
        s_wh[e * kRtWhStride + lane] += s_pre[e];
    __syncthreads();
    int32_t *my = s_wh + warp;
    const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int c = 0; c < kRtChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int e = ev[c];
        const bool ok = (unsigned)e < (unsigned)E;
        const int key = ok ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (e != -2) {
            const int rank = ok ? my[key * kRtWhStride] + __popc(grp & lt_mask) : cap;
            const int p = rank < cap ? key * cap + rank : -1;
            if (p >= 0)
                a.src[p] = n_lo + i;
            else
                s_rk[i] = -1;  // dropped: no distinct-token count
            a.pos[n_lo + i] = p;
        }
        __syncwarp();
        if (ok && lane == __ffs(grp) - 1)
            my[key * kRtWhStride] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kRtChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int r = ev[c] != -2 ? s_rk[i] : -1;
        bool first = r >= 0;
        if (first) {
            const int j = i % k;
            for (int jj = 0; jj < j; ++jj)
                first &= s_rk[i - j + jj] != r;
        }
        warp_count(s_rt, first ? (unsigned)r : 0u, first, rb);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x)
        if (s_rt[r])
            atomicAdd(a.rank_tokens + r, s_rt[r]);
}

template <bool kGate, int EPL>
__global__ void __launch_bounds__(kRtThreads) route_kernel(const RouteArgs a)
{
    extern __shared__ __align__(16) int32_t rsm[];
    __shared__ int32_t s_wsum[kRtWarps];
    __shared__ int32_t s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, k = a.k, E = a.E, E4 = a.E4, epr = a.epr, R = E / epr;
    const int C = gridDim.x, cta = blockIdx.x;
    const int t_lo = (int)((long long)T * cta / C);
    const int t_hi = (int)((long long)T * (cta + 1) / C);
    const int n_lo = t_lo * k, n = (t_hi - t_lo) * k;

    // 1. this CTA's tokens: gate them, or take their experts as given
    if (kGate) {
        for (int t = t_lo + warp; t < t_hi; t += kRtWarps)
            gate_token<EPL>(a.scores, a.bias, t, a.gp, a.group_lanes, a.vec_rows,
                            reinterpret_cast<uint32_t *>(rsm) + warp * gate_warp_words<EPL>(), a.topk_idx,
                            a.topk_w);
        __syncthreads();  // experts written (read back below through L2); gate scratch free
    }
    if (cta == 0)
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            a.rank_tokens[r] = 0;  // every CTA adds its share after the barrier

    int32_t *s_rt = rsm;                   // [R] this range's distinct tokens per rank
    int32_t *s_rk = s_rt + R;              // [n] rank of each entry of the range (-1: none)
    int32_t *s_wh = s_rk + n;                 // [E][kRtWhStride] per-warp counts, then row bases
    int32_t *s_pre = s_wh + kRtWhStride * E;  // [E4] entries of earlier CTAs
    int32_t *s_tot = s_pre + E4;              // [E4] all entries, then expert offsets
    int4 *s_part = reinterpret_cast<int4 *>(rsm + round4(R + n + kRtWhStride * E + 2 * E4));
    for (int i = threadIdx.x; i < R; i += blockDim.x)
        s_rt[i] = 0;
    for (int i = threadIdx.x; i < kRtWhStride * E; i += blockDim.x)
        s_wh[i] = 0;

    // each warp owns a contiguous slice of at most kRtChunks x 32 entries
    const int per_warp = ((n + kRtWarps * 32 - 1) / (kRtWarps * 32)) * 32;
    const int w0 = warp * per_warp;
    // ev: the entry's expert, -1 for an empty slot, -2 outside the slice.  An
    // index outside [0, E) other than -1 (including -2) is flagged here and
    // becomes an empty slot, so -2 never comes from the caller's indices.
    int ev[kRtChunks];
    int bad = 0;
#pragma unroll
    for (int c = 0; c < kRtChunks; ++c) {
        const int i = w0 + 32 * c + lane;
        int e = -2;
        if (32 * c < per_warp && i < n) {
            e = __ldcg(a.topk_idx + n_lo + i);
            if (e != -1 && (unsigned)e >= (unsigned)E) {
                bad = 1;
                e = -1;
            }
        }
        ev[c] = e;
    }
    __syncthreads();

    // 2. per-warp counts (a warp's own column: no atomics) and entry ranks
    const int eb = key_bits((unsigned)E), rb = key_bits((unsigned)R);
    int32_t *my = s_wh + warp;  // my[key * kRtWhStride]
#pragma unroll
    for (int c = 0; c < kRtChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int e = ev[c];
        const bool ok = (unsigned)e < (unsigned)E;
        const int key = ok ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (ok && lane == __ffs(grp) - 1)
            my[key * kRtWhStride] += __popc(grp);
        if (e != -2)
            s_rk[i] = ok ? e / epr : -1;
        __syncwarp();
    }
    if (bad && a.err_flag)
        atomicOr(a.err_flag, 1);
    __syncthreads();
    // distinct tokens per rank: an entry counts if no earlier slot of its
    // token is on the same rank (ranges hold whole tokens).  In capacity
    // mode only kept entries count, known after the barrier.
    const bool capped = a.cap >= 0;
#pragma unroll
    for (int c = 0; c < kRtChunks; ++c) {
        if (32 * c >= per_warp || capped)
            break;
        const int i = w0 + 32 * c + lane;
        const int r = ev[c] != -2 ? s_rk[i] : -1;
        bool first = r >= 0;
        if (first) {
            const int j = i % k;
            for (int jj = 0; jj < j; ++jj)
                first &= s_rk[i - j + jj] != r;
        }
        warp_count(s_rt, first ? (unsigned)r : 0u, first, rb);
    }
    // per-warp counts -> exclusive per-warp offsets (a warp scan per
    // expert, lane w = warp w's count); publish the CTA's row
    for (int e = warp; e < E; e += kRtWarps) {
        const int c = s_wh[e * kRtWhStride + lane];
        const int incl = warp_incl_scan(c, lane);
        s_wh[e * kRtWhStride + lane] = incl - c;
        if (lane == 31)
            a.rows[(size_t)cta * E4 + e] = incl;
    }
    for (int e = E + threadIdx.x; e < E4; e += blockDim.x)
        a.rows[(size_t)cta * E4 + e] = 0;

    // 3. every CTA's row is published
    if (!grid_barrier(a.barrier, (unsigned)C, a.spin_limit, a.err_flag))
        return;

    // 4. sums over the rows of the CTAs before this one, and of all
    const int G4 = E4 / 4;
    const int P = route_phases(E4);  // threads per column, each summing every P-th row
    int4 *s_pp = s_part, *s_pt = s_part + P * G4;
    if ((int)threadIdx.x < P * G4) {
        const int g = threadIdx.x % G4, ph = threadIdx.x / G4;
        const int4 *col = reinterpret_cast<const int4 *>(a.rows) + g;
        int4 pre = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
        int r = ph;
        for (; r + 3 * P < C; r += 4 * P) {
            int4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = __ldcg(col + (size_t)(r + u * P) * G4);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                tot.x += v[u].x, tot.y += v[u].y, tot.z += v[u].z, tot.w += v[u].w;
                if (r + u * P < cta)
                    pre.x += v[u].x, pre.y += v[u].y, pre.z += v[u].z, pre.w += v[u].w;
            }
        }
        for (; r < C; r += P) {
            const int4 v = __ldcg(col + (size_t)r * G4);
            tot.x += v.x, tot.y += v.y, tot.z += v.z, tot.w += v.w;
            if (r < cta)
                pre.x += v.x, pre.y += v.y, pre.z += v.z, pre.w += v.w;
        }
        s_pp[ph * G4 + g] = pre;
        s_pt[ph * G4 + g] = tot;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int g = e >> 2, q = e & 3;
        int pre = 0, tot = 0;
#pragma unroll 8
        for (int ph = 0; ph < P; ++ph) {
            pre += reinterpret_cast<const int32_t *>(s_pp + ph * G4 + g)[q];
            tot += reinterpret_cast<const int32_t *>(s_pt + ph * G4 + g)[q];
        }
        s_pre[e] = pre;
        s_tot[e] = tot;
    }
    __syncthreads();
    if (capped) {
        route_place_capped(a, s_tot, s_pre, s_wh, s_rk, s_rt, ev, per_warp, w0, n_lo, eb, rb);
        return;
    }
    // exclusive scan of the totals: one thread per expert
    {
        const int e = threadIdx.x;
        const int v = e < E ? s_tot[e] : 0;
        const int incl = warp_incl_scan(v, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = s_wsum[lane];
            const int wi = warp_incl_scan(ws, lane);
            s_wsum[lane] = wi - ws;
            if (lane == 31)
                s_total = wi;
        }
        __syncthreads();
        if (e < E) {
            const int off = s_wsum[warp] + incl - v;
            s_tot[e] = off;
            if (cta == 0) {
                a.expert_count[e] = v;
                a.expert_off[e] = off;
            }
        }
    }
    __syncthreads();
    const int total = s_total;
    const int N = T * k;
    if (cta == 0) {
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            const int lo = s_tot[r * epr];
            const int hi = (r + 1) * epr < E ? s_tot[(r + 1) * epr] : total;
            a.rank_off[r] = lo;
            a.rank_count[r] = hi - lo;
        }
        if (threadIdx.x == 0) {
            a.expert_off[E] = total;
            a.rank_off[R] = total;
        }
    }
    for (long long i = total + (long long)cta * blockDim.x + threadIdx.x; i < N; i += (long long)C * blockDim.x)
        a.src[i] = -1;
    for (int r = threadIdx.x; r < R; r += blockDim.x)
        if (s_rt[r])
            atomicAdd(a.rank_tokens + r, s_rt[r]);
    // row bases of each warp: offset + earlier CTAs + earlier warps
    for (int e = warp; e < E; e += kRtWarps)
        s_wh[e * kRtWhStride + lane] += s_tot[e] + s_pre[e];
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int c = 0; c < kRtChunks; ++c) {
        if (32 * c >= per_warp)
            break;
        const int i = w0 + 32 * c + lane;
        const int e = ev[c];
        const bool ok = (unsigned)e < (unsigned)E;
        const int key = ok ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (e != -2) {
            int p = ok ? my[key * kRtWhStride] + __popc(grp & lt_mask) : -1;
            if (p >= N)  // unreachable with consistent counts; never write outside src
                p = -1;
            if (p >= 0)
                a.src[p] = n_lo + i;
            a.pos[n_lo + i] = p;
        }
        __syncwarp();
        if (ok && lane == __ffs(grp) - 1)
            my[key * kRtWhStride] += __popc(grp);
        __syncwarp();
    }
}

size_t route_smem_bytes(int range, int E, int epr, int warp_floats)
{
    const int E4 = round4(E);
    const int G4 = E4 / 4;
    const int P = route_phases(E4);
    const size_t lay = (size_t)round4(E / epr + range + kRtWhStride * E + 2 * E4) * sizeof(int32_t) +
                       (size_t)2 * P * G4 * sizeof(int4);
    const size_t gate = (size_t)kRtWarps * warp_floats * sizeof(float);
    return gate > lay ? gate : lay;
}

int route_grid(int T)
{
    int c = device_sm_count();
    if (c > kRtMaxCtas)
        c = kRtMaxCtas;
    return T < c ? T : c;
}

template <bool kGate, int EPL>
cudaError_t launch_route_impl(RouteArgs a, cudaStream_t st)
{
    int warp_floats = 0;
    if (kGate)
        gate_plan<EPL>(a.gp, a.scores, a.bias, a.group_lanes, a.vec_rows, warp_floats);
    const int grid = route_grid(a.T);
    const int range = ((a.T + grid - 1) / grid) * a.k;
    const size_t smem = route_smem_bytes(range, a.E, a.epr, warp_floats);
    const void *fn = (const void *)route_kernel<kGate, EPL>;
    static bool attr_set = false;  // per instantiation: allow the largest size any call can need
    if (!attr_set) {
        const size_t most = route_smem_bytes(kRtMaxRange, kRtMaxExperts, 1, kGate ? kRtMaxExperts : 0);
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kRtThreads), args, smem, st);
}

}  // namespace

size_t route_workspace_bytes(int E) { return 256 + (size_t)kRtMaxCtas * round4(E) * sizeof(int32_t); }

bool route_supported(int T, int k, int E)
{
    if (T < 1 || E > kRtMaxExperts)
        return false;
    const int grid = route_grid(T);
    return (long long)((T + grid - 1) / grid) * k <= kRtMaxRange;
}

cudaError_t launch_route(const float *scores, const float *bias, const GateParams *gp, const int32_t *topk_idx_in,
                         int32_t *topk_idx, float *topk_w, int T, int k, int E, int epr, int32_t *expert_count,
                         int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                         int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, cudaStream_t st, int cap,
                         int32_t *expert_dropped)
{
    RouteArgs a{};
    a.cap = gp ? -1 : cap;
    a.expert_dropped = expert_dropped;
    a.scores = scores;
    a.bias = bias;
    if (gp)
        a.gp = *gp;
    a.topk_idx = gp ? topk_idx : const_cast<int32_t *>(topk_idx_in);
    a.topk_w = topk_w;
    a.T = T;
    a.k = k;
    a.E = E;
    a.E4 = round4(E);
    a.epr = epr;
    a.expert_count = expert_count;
    a.expert_off = expert_off;
    a.rank_count = rank_count;
    a.rank_off = rank_off;
    a.rank_tokens = rank_tokens;
    a.pos = pos;
    a.src = src;
    a.err_flag = err_flag;
    a.barrier = static_cast<unsigned *>(workspace);
    a.rows = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + 256);
    a.spin_limit = kGridSpinLimit;
    if (!gp)
        return launch_route_impl<false, 1>(a, st);
    if (E <= 32)
        return launch_route_impl<true, 1>(a, st);
    if (E <= 64)
        return launch_route_impl<true, 2>(a, st);
    if (E <= 128)
        return launch_route_impl<true, 4>(a, st);
    if (E <= 256)
        return launch_route_impl<true, 8>(a, st);
    return launch_route_impl<true, 16>(a, st);
}

}  // namespace ep
