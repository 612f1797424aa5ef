// route.cu -- routing of a whole batch in one cooperative launch: the
// group-limited gating (optional) and the dispatch layout (dropless or with
// a per-expert capacity).
//
// "DeepEP de DeepSeek ...", section "Group-limited gating algorithm" (the
// gating); "Expert Parallelism (Parallelisme d'experts)", section "Le
// principe de base" (a rank holds whole experts, so receive rows go rank by
// rank, expert by expert, in flat (token, slot) order); section "Defis et
// optimisations" (a per-expert capacity bounds the load).
//
// One CTA per SM, in thread-block clusters of cs CTAs where the device can
// co-schedule them (else cs = 1).  CTA c owns a contiguous range of whole
// tokens, cut into ranking blocks of 32 tokens (one bit each in a 32-bit
// mask):
//   1. it gates its tokens with lane segments (gate_fast.cuh; the score
//      loads are issued first, so their latency overlaps the prologue),
//      keeping the chosen experts in shared memory -- or loads the given
//      ones, flagging and skipping indices outside [0, E) other than -1;
//   2. each valid entry sets its token's bit in the (block, expert) and
//      (block, rank) masks (shared-memory atomic ORs: their order does not
//      matter); a token's experts being distinct, an entry's rank among its
//      expert's entries of the block is the popcount of the mask below its
//      token's bit (indices that repeat an expert inside a token take a
//      counting path instead); the block counts give each block's base
//      within the CTA and the CTA's per-expert totals;
//   3. the cluster's CTAs read each other's totals through distributed
//      shared memory: the entries of lower CTAs of the cluster, and the
//      cluster's totals, which its first CTA publishes as one row;
//   4. one grid barrier (bounded wait; past its limit EP_FLAG_TIMEOUT);
//   5. the column sums of the rows of lower clusters and of all clusters,
//      a scan of the totals into expert offsets;
//   6. every entry's row = offset + lower clusters + lower CTAs of the
//      cluster + lower blocks + its rank in the block.  CTA 0 writes the
//      counts and offsets.
// Results are those of the separate calls, bit for bit.
#include "coop.cuh"
#include "gate_fast.cuh"

namespace ep {

namespace {

constexpr int kRtThreads = 1024;
constexpr int kRtWarps = kRtThreads / 32;
constexpr int kBlk = 32;                // tokens per ranking block
constexpr int kRtMaxCtas = 160;
constexpr int kRtMaxTok = 128;          // tokens per CTA
constexpr int kRtMaxExperts = 1024;     // == kRtThreads: one thread per expert in the scan
constexpr int kRtMaxCluster = 8;
constexpr int kRtMaxPhases = 32;        // cluster rows summed per thread in the column sums: rows / phases
constexpr int kRtRowBatch = 8;          // rows a thread loads at once in the column sums

struct RouteArgs {
    GateFastArgs g;      // gating: scores, bias, parameters, outputs (unused when idx is given)
    const int32_t *idx;  // layout only: the experts per (token, slot); NULL when gating
    int T, k, E, E4, epr;
    int cap;  // >= 0: capacity mode (expert e owns rows [e*cap, (e+1)*cap)); -1: dropless
    int32_t *expert_count, *expert_off, *rank_count, *rank_off, *rank_tokens, *expert_dropped, *pos, *src;
    int32_t *err_flag;
    unsigned *barrier;  // arrival count, zero at launch
    int32_t *rows;      // [clusters][E4] per-cluster expert totals
    long long spin_limit;
};

__host__ __device__ inline int round4(int v) { return (v + 3) & ~3; }

// Phases of the column sums: threads per 4-expert column, a power of two.
__host__ __device__ inline int route_phases(int E4)
{
    int p = kRtThreads / (E4 / 4);
    if (p > kRtMaxPhases)
        p = kRtMaxPhases;
    int q = 1;
    while (q * 2 <= p)
        q *= 2;
    return q;
}

// Shared-memory words: [gating: bias rows (floats), candidate lists (2 words
// each), chosen experts and scores], then, 16-byte aligned, [layout: this
// CTA's totals, pre, totals (all three take 16-byte accesses), distinct
// tokens, entries, masks, rank masks, block bases].
struct RouteSmem {
    size_t gate_words, lay_words;
};

__host__ __device__ inline RouteSmem route_smem(int tpc, int k, int E, int R, int L, int EPL, int cap, bool gate)
{
    RouteSmem s;
    const int tpw = 32 / L;
    const int tslots = ((tpc + tpw - 1) / tpw) * tpw;  // tokens of the gating warps, whole warps
    s.gate_words = gate ? (size_t)L * (EPL + 4) + (size_t)tslots * cap * 2 + (size_t)tslots * k * 2 : 0;
    s.gate_words = (s.gate_words + 3) & ~(size_t)3;
    const int nb = (tpc + kBlk - 1) / kBlk;
    const int E4 = round4(E);
    s.lay_words = 3 * (size_t)E4 + round4(R) + (size_t)tpc * k + (size_t)nb * (2 * E + R);
    return s;
}

template <bool kGate, int EPL, int L, int Q>
__global__ void __launch_bounds__(kRtThreads, 1) route_kernel(const RouteArgs a)
{
    extern __shared__ __align__(16) int32_t rsm[];
    __shared__ int32_t s_wsum[kRtWarps];
    __shared__ int32_t s_total;
    constexpr int TPW = 32 / L;  // tokens a gating warp serves
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, k = a.k, E = a.E, E4 = a.E4, epr = a.epr, R = E / epr;
    const int C = gridDim.x, cta = blockIdx.x;
    const int t_lo = (int)((long long)T * cta / C), t_hi = (int)((long long)T * (cta + 1) / C);
    const int ntok = t_hi - t_lo, n_lo = t_lo * k, n = ntok * k;

    // 1a. the gating warps' score loads go first
    const bool gating = kGate && warp * TPW < ntok;
    const int tl = tid / L;
    const int tg = tl < ntok ? t_lo + tl : T;  // a lane segment past the range stores nothing
    float4 sv[EPL / 4];
    if (gating)
        gate_load<EPL, L>(a.g, tg, sv);

    const unsigned cs = cluster_nctarank(), cr = cluster_ctarank();
    const int ncl = C / (int)cs, cl = cta / (int)cs;
    const int tpc = (T + C - 1) / C;  // the most tokens a CTA holds (shared-memory sizing)
    const int nb = (ntok + kBlk - 1) / kBlk, NB = (tpc + kBlk - 1) / kBlk;
    const bool capped = !kGate && a.cap >= 0;  // routing with gating is always dropless
    const RouteSmem sz = route_smem(tpc, k, E, R, L, EPL, a.g.cap, kGate);
    int32_t *s_row = rsm + sz.gate_words;  // [E4] this CTA's entries per expert (read by the cluster)
    int32_t *s_pre = s_row + E4;           // [E4] entries of lower CTAs
    int32_t *s_tot = s_pre + E4;           // [E4] all entries, then offsets
    int32_t *s_rt = s_tot + E4;            // [R] distinct tokens per rank
    int32_t *s_tk = s_rt + round4(R);      // [n] this CTA's entries
    unsigned *s_mask = reinterpret_cast<unsigned *>(s_tk + (size_t)tpc * k);  // [NB][E]
    unsigned *s_rmask = s_mask + (size_t)NB * E;                             // [NB][R]
    int32_t *s_cpre = reinterpret_cast<int32_t *>(s_rmask + (size_t)NB * R);  // [NB][E] entries of lower blocks

    for (int i = tid; i < NB * (E + R); i += kRtThreads)
        s_mask[i] = 0u;  // s_mask and s_rmask are contiguous
    if (cta == 0)
        for (int r = tid; r < R; r += kRtThreads)
            a.rank_tokens[r] = 0;  // every CTA adds its share after the grid barrier
    if (capped) {
        // rows no kept entry lands on read -1: this CTA's slice (ordered
        // before every CTA's placements by the grid barrier)
        const long long rows = (long long)E * a.cap;
        for (long long r = rows * cta / C + tid; r < rows * (cta + 1) / C; r += kRtThreads)
            a.src[r] = -1;
    }

    // 1b. this CTA's entries
    if (kGate) {
        float *s_bias = reinterpret_cast<float *>(rsm);
        const int tslots = ((tpc + TPW - 1) / TPW) * TPW;
        // the bias block is L*(EPL+4) words, a multiple of 4: the 8-byte lists stay aligned
        unsigned long long *s_list = reinterpret_cast<unsigned long long *>(s_bias + L * (EPL + 4));
        int32_t *s_sel = reinterpret_cast<int32_t *>(s_list + (size_t)tslots * a.g.cap);
        float *s_ssc = reinterpret_cast<float *>(s_sel + (size_t)tslots * k);
        stage_bias<EPL>(a.g.bias, E, s_bias, tid, kRtThreads);
        __syncthreads();
        if (gating)
            gate_segment<EPL, L, Q>(a.g, tg, sv, s_bias, s_list + (size_t)tl * a.g.cap, s_sel + (size_t)tl * k,
                                    s_ssc + (size_t)tl * k, tl < ntok ? s_tk + (size_t)tl * k : nullptr);
    } else {
        int bad = 0;
        for (int i = tid; i < n; i += kRtThreads) {
            int e = __ldcg(a.idx + n_lo + i);
            if (e != -1 && (unsigned)e >= (unsigned)E) {
                bad = 1;
                e = -1;
            }
            s_tk[i] = e;
        }
        if (bad && a.err_flag)
            atomicOr(a.err_flag, 1);
    }
    __syncthreads();

    // 2. masks, block counts, the CTA's totals
    int dup = 0;
    for (int i = tid; i < n; i += kRtThreads) {
        const int e = s_tk[i];
        if (e < 0)
            continue;
        const int tk = i / k, j = i - tk * k;
        if (!kGate)
            for (int jj = 0; jj < j; ++jj)
                dup |= s_tk[i - j + jj] == e ? 1 : 0;
        const unsigned bit = 1u << (tk & (kBlk - 1));
        const int blk = tk / kBlk;
        atomicOr(s_mask + (size_t)blk * E + e, bit);
        atomicOr(s_rmask + (size_t)blk * R + e / epr, bit);
    }
    // gating chooses distinct experts per token: no repeats to count
    bool any_dup = false;
    if (kGate)
        __syncthreads();
    else
        any_dup = __syncthreads_or(dup) != 0;
    if (any_dup) {
        // an expert repeated within a token: count the entries one by one
        for (int i = tid; i < NB * E; i += kRtThreads)
            s_cpre[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kRtThreads) {
            const int e = s_tk[i];
            if (e >= 0)
                atomicAdd(s_cpre + (size_t)(i / k / kBlk) * E + e, 1);
        }
        __syncthreads();
    }
    for (int e = tid; e < E4; e += kRtThreads) {
        int run = 0;
        for (int blk = 0; blk < nb; ++blk) {
            const size_t at = (size_t)blk * E + e;
            const int cnt = e >= E ? 0 : (any_dup ? s_cpre[at] : __popc(s_mask[at]));
            if (e < E)
                s_cpre[at] = run;
            run += cnt;
        }
        s_row[e] = run;
    }
    if (!capped)
        for (int r = tid; r < R; r += kRtThreads) {
            int cnt = 0;
            for (int blk = 0; blk < nb; ++blk)
                cnt += __popc(s_rmask[(size_t)blk * R + r]);
            s_rt[r] = cnt;
        }

    // 3. the cluster's totals: lower CTAs of the cluster, and all of them
    cluster_arrive();
    cluster_wait();
    for (int e = tid; e < E4; e += kRtThreads) {
        int v[kRtMaxCluster];
#pragma unroll
        for (int q = 0; q < kRtMaxCluster; ++q)
            v[q] = q < (int)cs ? cluster_peer(s_row, (unsigned)q)[e] : 0;
        int pre = 0, tot = 0;
#pragma unroll
        for (int q = 0; q < kRtMaxCluster; ++q) {
            tot += v[q];
            pre += q < (int)cr ? v[q] : 0;
        }
        s_pre[e] = pre;
        if (cr == 0)
            a.rows[(size_t)cl * E4 + e] = tot;
    }
    cluster_arrive();  // this CTA is done reading the others' shared memory

    // 4. every cluster's row is published
    if (!grid_barrier(a.barrier, (unsigned)C, a.spin_limit, a.err_flag)) {
        cluster_wait();
        return;
    }

    // 5. column sums over the rows of lower clusters and of all clusters:
    // thread (g, ph) sums the 4-expert column g over rows ph, ph + P, ...;
    // the P phases of a column are adjacent lanes, reduced by xor shuffles
    {
        const int G4 = E4 / 4, P = route_phases(E4);
        const int g = tid / P, ph = tid % P;
        int4 pre = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
        if (g < G4) {
            const int4 *col = reinterpret_cast<const int4 *>(a.rows) + g;
            for (int r0 = ph; r0 < ncl; r0 += P * kRtRowBatch) {
                int4 v[kRtRowBatch];
#pragma unroll
                for (int u = 0; u < kRtRowBatch; ++u) {
                    const int r = r0 + u * P;
                    v[u] = r < ncl ? __ldcg(col + (size_t)r * G4) : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kRtRowBatch; ++u) {
                    const int r = r0 + u * P;
                    tot.x += v[u].x, tot.y += v[u].y, tot.z += v[u].z, tot.w += v[u].w;
                    if (r < cl)
                        pre.x += v[u].x, pre.y += v[u].y, pre.z += v[u].z, pre.w += v[u].w;
                }
            }
        }
        for (int off = 1; off < P; off <<= 1) {
            pre.x += __shfl_xor_sync(kFullMask, pre.x, off);
            pre.y += __shfl_xor_sync(kFullMask, pre.y, off);
            pre.z += __shfl_xor_sync(kFullMask, pre.z, off);
            pre.w += __shfl_xor_sync(kFullMask, pre.w, off);
            tot.x += __shfl_xor_sync(kFullMask, tot.x, off);
            tot.y += __shfl_xor_sync(kFullMask, tot.y, off);
            tot.z += __shfl_xor_sync(kFullMask, tot.z, off);
            tot.w += __shfl_xor_sync(kFullMask, tot.w, off);
        }
        if (g < G4 && ph == 0) {
            int4 p4 = reinterpret_cast<int4 *>(s_pre)[g];
            p4.x += pre.x, p4.y += pre.y, p4.z += pre.z, p4.w += pre.w;
            reinterpret_cast<int4 *>(s_pre)[g] = p4;
            reinterpret_cast<int4 *>(s_tot)[g] = tot;
        }
    }
    if (!capped)
        for (int r = tid; r < R; r += kRtThreads)
            if (s_rt[r])
                atomicAdd(a.rank_tokens + r, s_rt[r]);
    __syncthreads();

    const long long N = (long long)T * k;
    if (!capped) {
        // exclusive scan of the totals: one thread per expert (E <= 1024)
        const int e = tid;
        const int v = e < E ? s_tot[e] : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int nv = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off)
                incl += nv;
        }
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = s_wsum[lane];
            int wi = ws;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int nv = __shfl_up_sync(kFullMask, wi, off);
                if (lane >= off)
                    wi += nv;
            }
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
        __syncthreads();
        const int total = s_total;
        if (cta == 0) {
            for (int r = tid; r < R; r += kRtThreads) {
                const int lo = s_tot[r * epr];
                const int hi = (r + 1) * epr < E ? s_tot[(r + 1) * epr] : total;
                a.rank_off[r] = lo;
                a.rank_count[r] = hi - lo;
            }
            if (tid == 0) {
                a.expert_off[E] = total;
                a.rank_off[R] = total;
            }
        }
        // rows past the last entry (only when entries were skipped) read -1
        for (long long r = total + (long long)cta * kRtThreads + tid; r < N; r += (long long)C * kRtThreads)
            a.src[r] = -1;
    } else {
        const int cap = a.cap;
        if (cta == 0) {
            for (int e = tid; e < E; e += kRtThreads) {
                const int tot = s_tot[e], kept = tot < cap ? tot : cap;
                a.expert_count[e] = kept;
                a.expert_dropped[e] = tot - kept;
                a.expert_off[e] = e * cap;
            }
            for (int r = tid; r < R; r += kRtThreads) {
                int kept = 0;
                for (int e = r * epr; e < (r + 1) * epr; ++e)
                    kept += s_tot[e] < cap ? s_tot[e] : cap;
                a.rank_count[r] = kept;
                a.rank_off[r] = r * epr * cap;
            }
            if (tid == 0) {
                a.expert_off[E] = E * cap;
                a.rank_off[R] = E * cap;
            }
        }
        // the rank masks now collect tokens with a kept entry
        for (int i = tid; i < NB * R; i += kRtThreads)
            s_rmask[i] = 0u;
        __syncthreads();
    }

    // 6. rows in flat order
    for (int i = tid; i < n; i += kRtThreads) {
        const int e = s_tk[i];
        int p = -1;
        if (e >= 0) {
            const int tk = i / k, blk = tk / kBlk;
            int lr;
            if (!any_dup) {
                lr = __popc(s_mask[(size_t)blk * E + e] & ((1u << (tk & (kBlk - 1))) - 1u));
            } else {
                lr = 0;
                for (int i2 = blk * kBlk * k; i2 < i; ++i2)
                    lr += s_tk[i2] == e ? 1 : 0;
            }
            const int rank = s_pre[e] + s_cpre[(size_t)blk * E + e] + lr;  // within the expert, flat order
            if (!capped) {
                p = s_tot[e] + rank;
                if ((long long)p >= N)  // unreachable with consistent counts; never write outside src
                    p = -1;
            } else if (rank < a.cap) {
                p = e * a.cap + rank;
                atomicOr(s_rmask + (size_t)blk * R + e / epr, 1u << (tk & (kBlk - 1)));
            }
            if (p >= 0)
                a.src[p] = n_lo + i;
        }
        a.pos[n_lo + i] = p;
    }
    if (capped) {
        __syncthreads();
        for (int r = tid; r < R; r += kRtThreads) {
            int cnt = 0;
            for (int blk = 0; blk < nb; ++blk)
                cnt += __popc(s_rmask[(size_t)blk * R + r]);
            if (cnt)
                atomicAdd(a.rank_tokens + r, cnt);
        }
    }
    cluster_wait();  // no CTA leaves while a peer may still read its shared memory
}

// Launch shapes on this device: for each cluster size cs in {8, 4, 2}, the
// most CTAs (one per SM) a cooperative grid of such clusters can hold,
// found once per device.  A batch takes the largest cluster size whose grid
// covers at least half the SMs and still gives every CTA at most kRtMaxTok
// tokens, else single CTAs on every SM.  Larger clusters leave fewer rows
// for the column sums: measured on GB300 (152 SMs, DeepSeek-V3 shape), 120
// CTAs in clusters of 8 beat 152 in clusters of 2 or single CTAs, despite
// the SMs left idle.
PerDeviceCache<1> g_no_clusters;  // 1 once a clustered cooperative launch failed on the device

void route_no_clusters()
{
    g_no_clusters.get([] { return 1; });
}

int route_cluster_ctas(int cs)
{
    static PerDeviceCache<kRtMaxCluster + 1> cache;
    return cache.get(
        [cs] {
            const int sms = device_sm_count();
            const int cap = sms < kRtMaxCtas ? sms : kRtMaxCtas;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cs);
            cfg.blockDim = dim3(kRtThreads);
            cfg.dynamicSmemBytes = 16 * 1024;  // within the default limit; one CTA per SM either way
            cudaLaunchAttribute at;
            at.id = cudaLaunchAttributeClusterDimension;
            at.val.clusterDim.x = cs;
            at.val.clusterDim.y = 1;
            at.val.clusterDim.z = 1;
            cfg.attrs = &at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, (const void *)route_kernel<false, 8, 1, 1>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                return -1;  // not cached: asked again next time
            }
            int c = cs * n;
            if (c > cap)
                c = (cap / cs) * cs;
            return c > 0 ? c : -1;
        },
        cs);
}

// Grid size and cluster size for T tokens: every CTA gets at least one
// token; the grid is a multiple of the cluster size.
void route_grid(int T, int &grid, int &cs)
{
    const int sms = device_sm_count();
    const int cap = sms < kRtMaxCtas ? sms : kRtMaxCtas;
    cs = 1;
    grid = cap;
    if (g_no_clusters.get([] { return 0; }) <= 0) {
        for (int c : {kRtMaxCluster, 4, 2}) {
            const int ctas = route_cluster_ctas(c);
            if (ctas < 1 || 2 * ctas < cap || (T + ctas - 1) / ctas > kRtMaxTok)
                continue;
            cs = c;
            grid = ctas;
            break;
        }
    }
    int g = grid < T ? grid : T;
    if (cs > 1 && g < cs)
        cs = 1;
    g = (g / cs) * cs;
    grid = g < 1 ? 1 : g;
}

template <bool kGate, int EPL, int L, int Q>
cudaError_t launch_route_impl(RouteArgs a, cudaStream_t st)
{
    int grid, cs;
    route_grid(a.T, grid, cs);
    const int tpc = (a.T + grid - 1) / grid;
    // a CTA gates all its tokens in one pass of L lanes each: its token count
    // must fit (tokens past kRtThreads / L would keep unset experts)
    if (tpc > kRtMaxTok || (kGate && tpc > kRtThreads / L))
        return cudaErrorInvalidConfiguration;
    const RouteSmem sz = route_smem(tpc, a.k, a.E, a.E / a.epr, L, EPL, a.g.cap, kGate);
    const size_t smem = (sz.gate_words + sz.lay_words) * sizeof(int32_t);
    const void *fn = (const void *)route_kernel<kGate, EPL, L, Q>;
    static PerDeviceCache<1> attr;  // per instantiation and device: the most any call can need
    const RouteSmem most = route_smem(kRtMaxTok, kGate ? kGfMaxK : 64, kRtMaxExperts, kRtMaxExperts, L, EPL,
                                      kGate ? kGfCap : 0, kGate);
    const cudaError_t e = raise_smem_limit(attr, fn, (most.gate_words + most.lay_words) * sizeof(int32_t));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kRtThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = cs;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, route_kernel<kGate, EPL, L, Q>, a);
    if (err != cudaSuccess && cs > 1) {
        // this device (or driver) does not take a cooperative launch in
        // clusters: run without, and remember it for later calls
        cudaGetLastError();
        route_no_clusters();
        route_grid(a.T, grid, cs);
        cfg.gridDim = dim3(grid);
        at[1].val.clusterDim.x = 1;
        const int tpc1 = (a.T + grid - 1) / grid;
        const RouteSmem sz1 = route_smem(tpc1, a.k, a.E, a.E / a.epr, L, EPL, a.g.cap, kGate);
        cfg.dynamicSmemBytes = (sz1.gate_words + sz1.lay_words) * sizeof(int32_t);
        err = cudaLaunchKernelEx(&cfg, route_kernel<kGate, EPL, L, Q>, a);
    }
    return err;
}

template <int EPL, int L>
cudaError_t launch_gate_route(RouteArgs a, int Q, cudaStream_t st)
{
    if (Q == 1)
        return launch_route_impl<true, EPL, L, 1>(a, st);
    if (Q == 2)
        return launch_route_impl<true, EPL, L, 2>(a, st);
    return launch_route_impl<true, EPL, L, 4>(a, st);
}

}  // namespace

size_t route_workspace_bytes(int E) { return 256 + (size_t)kRtMaxCtas * round4(E) * sizeof(int32_t); }

void route_launch_shape(int T, int *grid, int *cluster)
{
    route_grid(T, *grid, *cluster);
}

bool route_supported(int T, int k, int E, int epr, bool gate)
{
    if (T < 1 || k < 1 || E < 1 || E > kRtMaxExperts || epr < 1 || E % epr != 0)
        return false;
    if (gate && k > kGfMaxK)
        return false;
    int grid, cs;
    route_grid(T, grid, cs);
    return (T + grid - 1) / grid <= kRtMaxTok;
}

cudaError_t launch_route(const float *scores, const float *bias, const GateParams *gp, const int32_t *topk_idx_in,
                         int32_t *topk_idx, float *topk_w, int T, int k, int E, int epr, int32_t *expert_count,
                         int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                         int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, cudaStream_t st, int cap,
                         int32_t *expert_dropped)
{
    RouteArgs a{};
    a.idx = gp ? nullptr : topk_idx_in;
    a.T = T;
    a.k = k;
    a.E = E;
    a.E4 = round4(E);
    a.epr = epr;
    a.cap = gp ? -1 : cap;
    a.expert_count = expert_count;
    a.expert_off = expert_off;
    a.rank_count = rank_count;
    a.rank_off = rank_off;
    a.rank_tokens = rank_tokens;
    a.expert_dropped = expert_dropped;
    a.pos = pos;
    a.src = src;
    a.err_flag = err_flag;
    a.barrier = static_cast<unsigned *>(workspace);
    a.rows = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + 256);
    a.spin_limit = kGridSpinLimit;
    if (!gp)
        return launch_route_impl<false, 8, 1, 1>(a, st);
    GateFastPlan f;
    if (!gate_fast_plan(*gp, scores, bias, f))
        return cudaErrorNotSupported;
    a.g.scores = scores;
    a.g.bias = bias;
    a.g.T = T;
    a.g.p = *gp;
    a.g.m = f.m;
    a.g.q = f.q;
    a.g.cap = f.cap;
    a.g.topk_idx = topk_idx;
    a.g.topk_w = topk_w;
    switch (E) {
    case 8: return launch_gate_route<8, 1>(a, f.Q, st);
    case 16: return launch_gate_route<8, 2>(a, f.Q, st);
    case 32: return launch_gate_route<8, 4>(a, f.Q, st);
    case 64: return launch_gate_route<8, 8>(a, f.Q, st);
    case 128: return launch_gate_route<16, 8>(a, f.Q, st);
    default: return launch_gate_route<32, 8>(a, f.Q, st);
    }
}

}  // namespace ep
