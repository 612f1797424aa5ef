// layout_cluster.cu -- step 2, the dispatch layout, by one thread-block
// cluster: no grid barrier, no workspace, one launch.
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le principe de
// base": a rank holds whole experts, here experts_per_rank contiguous ones,
// so the receive rows are grouped by rank, then expert, then in flat
// (token, slot) order.  The layout is a stable counting sort of the T*k
// expert indices.
//
// The cluster's C CTAs (16 where the device allows, else 8) each own a
// contiguous range of whole 32-token ranking blocks.  Per CTA:
//  1. its entries go to shared memory; each valid one sets its token's bit
//     in the (block, expert) and (block, rank) masks -- shared-memory
//     atomic ORs, whose order does not matter;
//  2. an entry's rank among its expert's entries of the same block is the
//     popcount of that mask below its token's bit (a token's k experts are
//     distinct; caller-given indices that repeat an expert within a token
//     take a counting path instead), the block's count is the popcount;
//     a column prefix over the CTA's blocks gives each block's base;
//  3. the CTA's per-expert totals and per-rank distinct-token counts sit in
//     its shared memory; after one cluster barrier every CTA reads all of
//     them through distributed shared memory: the entries of lower CTAs and
//     the totals, scanned into the expert offsets;
//  4. each entry's row = expert offset + lower CTAs + lower blocks + its
//     rank in the block.
// Launched with programmatic stream serialisation: the prologue (clearing
// shared memory) may overlap the previous kernel; griddepcontrol.wait comes
// before any global memory access.  Results equal the other layout paths'
// bit for bit.
#include "coop.cuh"

namespace ep {

namespace {

constexpr int kLcThreads = 1024;
constexpr int kLcWarps = kLcThreads / 32;
constexpr int kBlk = 32;  // tokens per ranking block: one bit each in a 32-bit mask
constexpr int kLcMaxCluster = 16;
constexpr int kLcMaxExperts = kLcThreads;  // one thread per expert in the offset scan
constexpr size_t kLcMaxSmem = 220 * 1024;  // below the 227 KB a CTA may hold, with room for the static part

struct LcArgs {
    const int32_t *idx;
    int T, k, E, epr;
    int cap;  // >= 0: capacity mode (expert e owns rows [e*cap, (e+1)*cap)); -1: dropless
    int nb;   // ranking blocks per CTA at most (shared-memory sizing)
    int32_t *expert_count, *expert_off, *rank_count, *rank_off, *rank_tokens, *expert_dropped, *pos, *src;
    int32_t *err_flag;
};

__device__ __forceinline__ int warp_incl_sum(int v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off)
            v += n;
    }
    return v;
}

__host__ __device__ inline size_t lc_smem_words(int nb, int E, int R, int k)
{
    return (size_t)nb * (2 * E + R) + 3 * (size_t)E + R + (size_t)nb * kBlk * k;
}

// kCap: capacity mode (a.cap >= 0); the dropless instance is compiled
// without the capacity paths (a smaller body to fetch on a cold call).
template <bool kCap>
__global__ void __launch_bounds__(kLcThreads, 1) layout_cluster_kernel(const LcArgs a)
{
    extern __shared__ __align__(16) int32_t lsm[];
    __shared__ int32_t s_wsum[kLcWarps];
    __shared__ int32_t s_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, k = a.k, E = a.E, epr = a.epr, R = E / epr, NB = a.nb;
    const bool capped = kCap;
    const unsigned C = cluster_nctarank(), c = cluster_ctarank();
    const int B = (T + kBlk - 1) / kBlk;
    const int b0 = (int)((long long)B * c / C), b1 = (int)((long long)B * (c + 1) / C);
    const int nb = b1 - b0;
    const int t0 = b0 * kBlk, t1 = min(T, b1 * kBlk);
    const int n0 = t0 * k, n = (t1 - t0) * k;
    const long long N = (long long)T * k;

    unsigned *s_mask = reinterpret_cast<unsigned *>(lsm);  // [NB][E] tokens of a block that chose expert e
    unsigned *s_rmask = s_mask + (size_t)NB * E;           // [NB][R] tokens of a block with an entry on rank r
    int32_t *s_cpre = reinterpret_cast<int32_t *>(s_rmask + (size_t)NB * R);  // [NB][E] entries of lower blocks
    int32_t *s_part = s_cpre + (size_t)NB * E;  // [E] this CTA's entries per expert (read by the cluster)
    int32_t *s_prt = s_part + E;                // [R] this CTA's distinct tokens per rank (read by CTA 0)
    int32_t *s_pre = s_prt + R;                 // [E] entries of lower CTAs
    int32_t *s_off = s_pre + E;                 // [E] totals, then each expert's first row
    int32_t *s_ev = s_off + E;                  // [n] this CTA's entries

    for (int i = tid; i < NB * (E + R); i += kLcThreads)
        s_mask[i] = 0u;  // s_mask and s_rmask are contiguous

    // Every global access below comes after the previous kernel's results
    // are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (capped) {
        // rows no kept entry lands on read -1: this CTA clears its slice
        // (ordered before every CTA's stores by the cluster barrier)
        const long long rows = (long long)E * a.cap;
        for (long long r = rows * c / C + tid; r < rows * (c + 1) / C; r += kLcThreads)
            a.src[r] = -1;
        if (c == 0)
            for (int r = tid; r < R; r += kLcThreads)
                a.rank_tokens[r] = 0;  // every CTA adds its share after the barrier
    }

    // 1. entries; an index neither -1 nor in [0, E) is flagged and skipped
    int bad = 0;
    for (int i = tid; i < n; i += kLcThreads) {
        int e = __ldcg(a.idx + n0 + i);
        if (e != -1 && (unsigned)e >= (unsigned)E) {
            bad = 1;
            e = -1;
        }
        s_ev[i] = e;
    }
    if (bad && a.err_flag)
        atomicOr(a.err_flag, 1);
    __syncthreads();
    int dup = 0;
    for (int i = tid; i < n; i += kLcThreads) {
        const int e = s_ev[i];
        if (e < 0)
            continue;
        const int tl = i / k, j = i - tl * k;
        for (int jj = 0; jj < j; ++jj)
            dup |= s_ev[i - j + jj] == e ? 1 : 0;
        const unsigned bit = 1u << (tl & (kBlk - 1));
        const int blk = tl / kBlk;
        atomicOr(s_mask + (size_t)blk * E + e, bit);
        atomicOr(s_rmask + (size_t)blk * R + e / epr, bit);
    }
    const bool any_dup = __syncthreads_or(dup) != 0;
    if (any_dup) {
        // an expert repeated within a token: count entries one by one
        for (int i = tid; i < NB * E; i += kLcThreads)
            s_cpre[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kLcThreads) {
            const int e = s_ev[i];
            if (e >= 0)
                atomicAdd(s_cpre + (size_t)(i / k / kBlk) * E + e, 1);
        }
        __syncthreads();
    }

    // 2. per-block counts -> bases within the CTA; the CTA's totals
    for (int e = tid; e < E; e += kLcThreads) {
        int run = 0;
        for (int blk = 0; blk < nb; ++blk) {
            const size_t at = (size_t)blk * E + e;
            const int cnt = any_dup ? s_cpre[at] : __popc(s_mask[at]);
            s_cpre[at] = run;
            run += cnt;
        }
        s_part[e] = run;
    }
    for (int r = tid; r < R; r += kLcThreads) {
        int cnt = 0;
        for (int blk = 0; blk < nb; ++blk)
            cnt += __popc(s_rmask[(size_t)blk * R + r]);
        s_prt[r] = cnt;
    }

    // 3. every CTA's totals are published
    cluster_arrive();
    cluster_wait();
    for (int e = tid; e < E; e += kLcThreads) {
        int v[kLcMaxCluster];
#pragma unroll
        for (int q = 0; q < kLcMaxCluster; ++q)
            v[q] = q < (int)C ? cluster_peer(s_part, (unsigned)q)[e] : 0;
        int pre = 0, tot = 0;
#pragma unroll
        for (int q = 0; q < kLcMaxCluster; ++q) {
            tot += v[q];
            pre += q < (int)c ? v[q] : 0;
        }
        s_pre[e] = pre;
        s_off[e] = tot;
    }
    if (!capped && c == 0)
        for (int r = tid; r < R; r += kLcThreads) {
            int v[kLcMaxCluster];
#pragma unroll
            for (int q = 0; q < kLcMaxCluster; ++q)
                v[q] = q < (int)C ? cluster_peer(s_prt, (unsigned)q)[r] : 0;
            int tot = 0;
#pragma unroll
            for (int q = 0; q < kLcMaxCluster; ++q)
                tot += v[q];
            a.rank_tokens[r] = tot;
        }
    cluster_arrive();  // this CTA is done reading the others' shared memory
    __syncthreads();

    int total = 0;
    if (!capped) {
        // exclusive scan of the totals, one expert per thread (E <= 1024)
        const int e = tid;
        const int v = e < E ? s_off[e] : 0;
        const int incl = warp_incl_sum(v, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = s_wsum[lane];
            const int wi = warp_incl_sum(ws, lane);
            s_wsum[lane] = wi - ws;
            if (lane == 31)
                s_total = wi;
        }
        __syncthreads();
        if (e < E) {
            const int off = s_wsum[warp] + incl - v;
            s_off[e] = off;
            if (c == 0) {
                a.expert_count[e] = v;
                a.expert_off[e] = off;
            }
        }
        __syncthreads();
        total = s_total;
        if (c == 0) {
            for (int r = tid; r < R; r += kLcThreads) {
                const int lo = s_off[r * epr];
                const int hi = (r + 1) * epr < E ? s_off[(r + 1) * epr] : total;
                a.rank_off[r] = lo;
                a.rank_count[r] = hi - lo;
            }
            if (tid == 0) {
                a.expert_off[E] = total;
                a.rank_off[R] = total;
            }
        }
        // rows past the last entry (only when entries were skipped) read -1
        for (long long r = total + (long long)c * kLcThreads + tid; r < N; r += (long long)C * kLcThreads)
            a.src[r] = -1;
    } else {
        const int cap = a.cap;
        if (c == 0) {
            for (int e = tid; e < E; e += kLcThreads) {
                const int tot = s_off[e], kept = tot < cap ? tot : cap;
                a.expert_count[e] = kept;
                a.expert_dropped[e] = tot - kept;
                a.expert_off[e] = e * cap;
            }
            for (int r = tid; r < R; r += kLcThreads) {
                int kept = 0;
                for (int e = r * epr; e < (r + 1) * epr; ++e)
                    kept += s_off[e] < cap ? s_off[e] : cap;
                a.rank_count[r] = kept;
                a.rank_off[r] = r * epr * cap;
            }
            if (tid == 0) {
                a.expert_off[E] = E * cap;
                a.rank_off[R] = E * cap;
            }
        }
        // the rank masks now collect tokens with a kept entry
        for (int i = tid; i < NB * R; i += kLcThreads)
            s_rmask[i] = 0u;
        __syncthreads();
    }

    // 4. rows in flat order
    for (int i = tid; i < n; i += kLcThreads) {
        const int e = s_ev[i];
        int p = -1;
        if (e >= 0) {
            const int tl = i / k, blk = tl / kBlk;
            int lr;
            if (!any_dup) {
                lr = __popc(s_mask[(size_t)blk * E + e] & ((1u << (tl & (kBlk - 1))) - 1u));
            } else {
                lr = 0;
                for (int i2 = blk * kBlk * k; i2 < i; ++i2)
                    lr += s_ev[i2] == e ? 1 : 0;
            }
            const int rank = s_pre[e] + s_cpre[(size_t)blk * E + e] + lr;  // within the expert, flat order
            if (!capped) {
                p = s_off[e] + rank;
                if ((long long)p >= N)  // unreachable with consistent counts; never write outside src
                    p = -1;
            } else if (rank < a.cap) {
                p = e * a.cap + rank;
                atomicOr(s_rmask + (size_t)blk * R + e / epr, 1u << (tl & (kBlk - 1)));
            }
            if (p >= 0)
                a.src[p] = n0 + i;
        }
        a.pos[n0 + i] = p;
    }
    if (capped) {
        __syncthreads();
        for (int r = tid; r < R; r += kLcThreads) {
            int cnt = 0;
            for (int blk = 0; blk < nb; ++blk)
                cnt += __popc(s_rmask[(size_t)blk * R + r]);
            if (cnt)
                atomicAdd(a.rank_tokens + r, cnt);
        }
    }
    cluster_wait();  // no CTA leaves while another may still read its shared memory
}

// The cluster size this device runs the kernel at: 16 CTAs of one SM each
// where the device allows non-portable cluster sizes and can co-schedule
// them, else 8; 0 if neither fits.  One answer for both instances (the
// smaller of the two), so that the support check and the launch agree.
template <bool kCap>
int cluster_size_of()
{
    const void *fn = (const void *)layout_cluster_kernel<kCap>;
    static PerDeviceCache<1> attr;
    const cudaError_t ae = raise_smem_limit(attr, fn, kLcMaxSmem);
    if (ae != cudaSuccess)
        return 0;
    static PerDeviceCache<1> sizes;
    return sizes.get([fn] {
        for (int cs : {kLcMaxCluster, 8}) {
            if (cs > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
                cudaGetLastError();
                continue;
            }
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cs);
            cfg.blockDim = dim3(kLcThreads);
            cfg.dynamicSmemBytes = kLcMaxSmem;
            cudaLaunchAttribute at;
            at.id = cudaLaunchAttributeClusterDimension;
            at.val.clusterDim.x = cs;
            at.val.clusterDim.y = 1;
            at.val.clusterDim.z = 1;
            cfg.attrs = &at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0)
                return cs;
            cudaGetLastError();
        }
        return -1;  // cached: this device cannot run the kernel as a cluster
    });
}

int cluster_size_for()
{
    const int a = cluster_size_of<false>(), b = cluster_size_of<true>();
    return a < b ? a : b;
}

}  // namespace

bool layout_cluster_supported(int T, int k, int E, int epr)
{
    if (T < 1 || k < 1 || E < 1 || E > kLcMaxExperts || epr < 1 || E % epr != 0)
        return false;
    const int cs = cluster_size_for();
    if (cs < 1)
        return false;
    const int B = (T + kBlk - 1) / kBlk;
    const int C = B < cs ? B : cs;
    const int nb = (B + C - 1) / C;
    return lc_smem_words(nb, E, E / epr, k) * sizeof(int32_t) <= kLcMaxSmem;
}

cudaError_t launch_layout_cluster(const int32_t *topk_idx, int T, int k, int E, int epr, int cap,
                                  int32_t *expert_count, int32_t *expert_off, int32_t *rank_count,
                                  int32_t *rank_off, int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos,
                                  int32_t *src, int32_t *err_flag, cudaStream_t st)
{
    const int cs = cluster_size_for();
    if (cs < 1)
        return cudaErrorNotSupported;
    const int B = (T + kBlk - 1) / kBlk;
    const int C = B < cs ? B : cs;
    LcArgs a{};
    a.idx = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.epr = epr;
    a.cap = cap;
    a.nb = (B + C - 1) / C;
    a.expert_count = expert_count;
    a.expert_off = expert_off;
    a.rank_count = rank_count;
    a.rank_off = rank_off;
    a.rank_tokens = rank_tokens;
    a.expert_dropped = expert_dropped;
    a.pos = pos;
    a.src = src;
    a.err_flag = err_flag;
    const size_t smem = lc_smem_words(a.nb, E, E / epr, k) * sizeof(int32_t);
    if (smem > kLcMaxSmem)
        return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kLcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cap >= 0)
        return cudaLaunchKernelEx(&cfg, layout_cluster_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, layout_cluster_kernel<false>, a);
}

}  // namespace ep
