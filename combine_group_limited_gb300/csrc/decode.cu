// decode.cu -- fused low-latency path for decode-sized batches: gating,
// layout and dispatch in one launch.
//
// "DeepEP de DeepSeek ...", section "Kernels low-latency dispatch et
// combine": separate latency-optimised kernels for small (decode) batches;
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all": decode messages of 100 KB to 2 MB, where the
// exchange is 10-30 % of end-to-end latency.  At T = 128 the three separate
// steps are several short launches; here they are one.
//
// Up to 512 tokens: the clustered kernel further down (no grid barrier).
// Past that (T*k <= 4096 with k < 8), the cooperative kernel: each CTA (one
// per SM) owns a contiguous range of tokens:
//   1. it gates its tokens (gate_impl.cuh);
//   2. a grid barrier (every CTA is resident: cooperative launch), with a
//      bounded wait -- past its limit a CTA sets EP_FLAG_TIMEOUT and stops;
//   3. it counts all T*k <= 4096 chosen experts and those before its range
//      (warp-aggregated shared counters), scans the totals into expert
//      offsets, and gives its own entries their stable rows (offset +
//      earlier entries of the expert + equal lower lanes, ballot peer
//      masks); CTA 0 writes the offsets and counts, every CTA its rows and
//      its share of the distinct-token counts;
//   4. it scatters its own tokens' rows (dispatch_impl.cuh).
// Results are the ones the separate calls give, bit for bit.
#include "coop.cuh"
#include "dispatch_impl.cuh"
#include "gate_impl.cuh"

namespace ep {

namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxEntries = 4096;                           // T*k of the fused path
constexpr int kDecChunks = kMaxEntries / (kDecWarps * 32);  // 32-entry chunks per warp

struct DecodeArgs {
    const float *scores;
    const float *bias;
    int T;
    GateParams gp;
    int group_lanes, vec_rows;
    int epr;
    const uint16_t *x;
    int H;
    int dtype;  // ep_dtype
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_count, *expert_off, *rank_count, *rank_off, *rank_tokens, *pos, *src;
    void *recv;
    void *recv_scales;
    long long rows;
    int32_t *err_flag;
    unsigned *barrier;
    unsigned barrier_extra;  // arrivals expected beyond the grid (0; >0 only in the self-test)
    long long spin_limit;
};

template <int EPL>
__global__ void __launch_bounds__(kDecThreads) decode_fused_kernel(const DecodeArgs a)
{
    extern __shared__ int32_t dsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.gp.E, k = a.gp.k, T = a.T, N = T * k, R = E / a.epr;
    // This CTA's tokens: a contiguous range, so that its entries' rows only
    // need the counts of the entries before the range.
    const int t_lo = (int)((long long)T * blockIdx.x / gridDim.x);
    const int t_hi = (int)((long long)T * (blockIdx.x + 1) / gridDim.x);
    const int n_lo = t_lo * k, n_hi = t_hi * k;

    // 1. gating of this CTA's tokens
    for (int t = t_lo + warp; t < t_hi; t += kDecWarps)
        gate_token<EPL>(a.scores, a.bias, t, a.gp, a.group_lanes, a.vec_rows,
                        reinterpret_cast<uint32_t *>(dsm) + warp * gate_warp_words<EPL>(), a.topk_idx, a.topk_w);
    if (blockIdx.x == 0)
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            a.rank_tokens[r] = 0;  // accumulated by every CTA after the barrier

    // 2. every CTA's experts are written
    if (!grid_barrier(a.barrier, gridDim.x + a.barrier_extra, a.spin_limit, a.err_flag))
        return;

    // 3. counts of all entries and of the entries before this CTA's range
    int32_t *s_tot = dsm;                 // [E] totals, then offsets
    int32_t *s_pre = s_tot + E;           // [E] entries before n_lo
    int32_t *s_rt = s_pre + E;            // [R] this range's distinct tokens per rank
    int32_t *s_idx = s_rt + R;            // [n_hi - n_lo] this range's experts
    int32_t *s_rows = s_idx + (n_hi - n_lo);  // [n_hi - n_lo] their receive rows
    __shared__ int32_t s_wsum[kDecWarps];
    __shared__ int32_t s_total;
    for (int i = threadIdx.x; i < 2 * E + R; i += blockDim.x)
        dsm[i] = 0;
    __syncthreads();
    const int eb = key_bits((unsigned)E), rb = key_bits((unsigned)R);
    {
        // each warp loads its slice of all N experts at once (written by
        // other CTAs: read through L2), then counts it
        const int per_warp = ((N + kDecWarps * 32 - 1) / (kDecWarps * 32)) * 32;  // <= kDecChunks * 32
        const int w0 = warp * per_warp;
        int ev[kDecChunks];
#pragma unroll
        for (int c = 0; c < kDecChunks; ++c) {
            const int i = w0 + 32 * c + lane;
            ev[c] = (32 * c < per_warp && i < N) ? __ldcg(a.topk_idx + i) : -1;
        }
#pragma unroll
        for (int c = 0; c < kDecChunks; ++c) {
            if (32 * c >= per_warp)
                break;
            const int i = w0 + 32 * c + lane;
            const int e = ev[c];
            const bool ok = (unsigned)e < (unsigned)E;
            warp_count(s_tot, ok ? (unsigned)e : 0u, ok, eb);
            warp_count(s_pre, ok ? (unsigned)e : 0u, ok && i < n_lo, eb);
            if (i >= n_lo && i < n_hi)
                s_idx[i - n_lo] = e;
        }
    }
    __syncthreads();
    {
        constexpr int kPerThread = kMaxExperts / kDecThreads;
        const int e0 = threadIdx.x * kPerThread;
        int v[kPerThread];
        int sum = 0;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            v[u] = e0 + u < E ? s_tot[e0 + u] : 0;
            sum += v[u];
        }
        const int incl = warp_incl_scan(sum, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = lane < kDecWarps ? s_wsum[lane] : 0;
            const int wi = warp_incl_scan(ws, lane);
            if (lane < kDecWarps)
                s_wsum[lane] = wi - ws;
        }
        __syncthreads();
        int run = s_wsum[warp] + incl - sum;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            if (e0 + u < E) {
                s_tot[e0 + u] = run;
                if (blockIdx.x == 0) {
                    a.expert_off[e0 + u] = run;
                    a.expert_count[e0 + u] = v[u];
                }
            }
            if (e0 + u == E - 1)
                s_total = run + v[u];
            run += v[u];
        }
    }
    __syncthreads();
    const int total = s_total;
    if (blockIdx.x == 0) {
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            const int lo = s_tot[r * a.epr];
            const int hi = (r + 1) * a.epr < E ? s_tot[(r + 1) * a.epr] : total;
            a.rank_off[r] = lo;
            a.rank_count[r] = hi - lo;
        }
        if (threadIdx.x == 0) {
            a.expert_off[E] = total;
            a.rank_off[R] = total;
        }
    }
    for (int i = total + blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
        a.src[i] = -1;
    // Rows of this range's entries, in flat order: warp 0 walks the range in
    // 32-entry chunks; a lane's row is its expert's offset + the entries of
    // that expert before the range + the equal lower lanes so far.
    if (warp == 0) {
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int c = n_lo; c < n_hi; c += 32) {
            const int i = c + lane;
            const bool in = i < n_hi;
            const int e = in ? s_idx[i - n_lo] : -1;
            const int key = (unsigned)e < (unsigned)E ? e : E;
            const unsigned grp = peer_mask((unsigned)key, key_bits((unsigned)E));
            int p = -1;
            if (key < E)
                p = s_tot[key] + s_pre[key] + __popc(grp & lt_mask);
            if (in) {
                a.pos[i] = p;
                s_rows[i - n_lo] = p;
                if (p >= 0)
                    a.src[p] = i;
            }
            __syncwarp();
            if (key < E && lane == __ffs(grp) - 1)
                s_pre[key] += __popc(grp);
            __syncwarp();
        }
    }
    // distinct tokens per rank, from this range's experts (shared memory)
    for (int base = n_lo + (threadIdx.x & ~31); base < n_hi; base += blockDim.x) {
        const int i = base + lane;
        const int e = i < n_hi ? s_idx[i - n_lo] : -1;
        const bool ok = (unsigned)e < (unsigned)E;
        const int r = ok ? e / a.epr : 0;
        bool first = ok;
        if (ok) {
            const int j = (i - n_lo) % k;
            for (int jj = 0; jj < j; ++jj) {
                const int e2 = s_idx[i - n_lo - j + jj];
                first &= !((unsigned)e2 < (unsigned)E && e2 / a.epr == r);
            }
        }
        warp_count(s_rt, (unsigned)r, first, rb);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x)
        if (s_rt[r])
            atomicAdd(a.rank_tokens + r, s_rt[r]);

    // 4. scatter this CTA's rows: warp items over (token, row segment)
    const int segs = a.dtype == 0 ? bf16_segs(a.H) : fp8_segs(a.H);
    const int items = (t_hi - t_lo) * segs;
    for (int item = warp; item < items; item += kDecWarps) {
        const int t = t_lo + item / segs;
        const int seg = item - (t - t_lo) * segs;
        int p0 = -1, p1 = -1;
        if (lane < k)
            p0 = s_rows[(t - t_lo) * k + lane];
        if (lane + 32 < k)
            p1 = s_rows[(t - t_lo) * k + lane + 32];
        if (p0 >= a.rows || p1 >= a.rows) {
            if (a.err_flag)
                atomicOr(a.err_flag, 2);
            p0 = p0 >= a.rows ? -1 : p0;
            p1 = p1 >= a.rows ? -1 : p1;
        }
        if (a.dtype == 0)
            dispatch_bf16_item(a.x, a.H, k, t, seg, p0, p1, static_cast<uint16_t *>(a.recv));
        else if (a.dtype == 1)
            dispatch_fp8_item(a.x, a.H, k, t, seg, p0, p1, static_cast<uint8_t *>(a.recv),
                              static_cast<float *>(a.recv_scales));
        else
            dispatch_mxfp8_item(a.x, a.H, k, t, seg, p0, p1, static_cast<uint8_t *>(a.recv),
                                static_cast<uint8_t *>(a.recv_scales));
    }
}

// ---------------------------------------------------------------------------
// Clustered decode path: no grid barrier.
//
// The gating and the layout of a decode batch are small next to its
// dispatch, so every cluster of CS = 8 CTAs computes both for the WHOLE batch
// (CTA r of a cluster gates tokens [T*r/CS, T*(r+1)/CS), one warp per
// token), and the clusters then share the dispatch: of CTA r's warp items
// (its tokens' row segments, in order), cluster c scatters items c, c + G,
// c + 2G, ... (G clusters, at most as many as are resident at once), and it
// writes the outputs of CTA r's tokens j with j % G == c.  The only
// exchange is inside a cluster, through distributed shared memory:
//   1. each CTA marks, per expert and per rank, which of its tokens chose
//      it (64-bit token masks, shared-memory atomicOr), and stores the
//      popcounts into slot [r] of every cluster CTA's count table (remote
//      shared-memory stores; ranks only to CTA 0 of cluster 0);
//   2. one cluster barrier; then, locally, the entries of each expert in
//      lower CTAs (pre) and in all (total), and one warp scans the totals
//      into expert offsets;
//   3. the row of entry (token j, slot) for expert e is
//      offset[e] + pre[e] + popc(mask[e] & below(j)) -- the stable
//      flat-order rank, since a token names an expert at most once;
//   4. CTA 0 of cluster 0 writes the counts, offsets and distinct tokens per
//      rank; the dispatching CTA of a token writes its experts, weights,
//      rows and src entries and scatters its rows (dispatch_impl.cuh).  Each
//      warp loads its first row segment before it gates, so that load
//      overlaps the gating, and converts it (FP8 / MXFP8) between arriving
//      at the cluster barrier and waiting on it.
// Every cluster computes the same layout, so results equal the separate
// calls bit for bit.  With dtype < 0 nothing is dispatched and one cluster
// writes everything: the gating + layout of ep_gate_layout.  Launched with
// programmatic stream serialisation: clearing shared memory may overlap
// the previous kernel; griddepcontrol.wait precedes every global access.
constexpr int kDcMaxTpc = 64;  // tokens per CTA: one bit each in a 64-bit mask
constexpr int kDcMaxCluster = 8;
constexpr int kDcMaxTokens = kDcMaxCluster * kDcMaxTpc;

struct DcSmem {
    size_t gate, e, w, mask, rmask, cnt, rcnt, pre, off, total;
};

// Byte offsets of the clustered kernel's shared memory: gating scratch,
// entries' experts and weights, expert and rank masks (8-byte aligned), the
// cluster's per-CTA expert and rank counts, entries before this CTA per
// expert, offsets.
__host__ __device__ inline DcSmem dc_smem(int tpc, int k, int E, int R, int cs, int warp_words)
{
    DcSmem m{};
    m.gate = 0;
    m.e = (size_t)kDecWarps * warp_words * 4;
    m.w = m.e + (size_t)tpc * k * 4;
    m.mask = (m.w + (size_t)tpc * k * 4 + 15) & ~(size_t)15;
    m.rmask = m.mask + (size_t)E * 8;
    m.cnt = m.rmask + (size_t)R * 8;
    m.rcnt = m.cnt + (size_t)cs * E * 4;
    m.pre = m.rcnt + (size_t)cs * R * 4;
    m.off = m.pre + (size_t)E * 4;
    m.total = m.off + (size_t)E * 4;
    return m;
}

// The receive row of this CTA's local token j for slot `lane` (lane < k),
// or -1.
__device__ __forceinline__ int dc_row(const int32_t *s_e, const int32_t *s_pre, const int32_t *s_off,
                                      const unsigned long long *s_mask, int E, int k, int j, int lane)
{
    const int e = s_e[j * k + lane];
    if ((unsigned)e >= (unsigned)E)
        return -1;
    return s_off[e] + s_pre[e] + __popcll(s_mask[e] & ((1ull << j) - 1ull));
}

// kDt: the payload the body is compiled for: -1 none (gating and layout
// only), 1 FP8 1x128 (the decode path's usual payload), kDtAny the others
// (BF16, MXFP8), taken from a.dtype at run time.  A body specialised to FP8
// measured 7.28 against 7.48 us a call back to back (decode shape).
constexpr int kDtAny = 3;

template <int EPL, int kDt>
__global__ void __launch_bounds__(kDecThreads, 1) decode_cluster_kernel(const DecodeArgs a)
{
    const int dtype = kDt == kDtAny ? a.dtype : kDt;
    extern __shared__ __align__(16) unsigned char dc_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.gp.E, k = a.gp.k, T = a.T, R = E / a.epr;
    const unsigned cs = cluster_nctarank(), cr = cluster_ctarank();
    const int cid = (int)cluster_id_x(), G = (int)(gridDim.x / cs);
    // T <= 512 and cs <= 8: 32-bit products and divisions
    const int t_lo = T * (int)cr / (int)cs, t_hi = T * ((int)cr + 1) / (int)cs;
    const int n_loc = t_hi - t_lo;
    const int tpc = (T + (int)cs - 1) / (int)cs;
    const DcSmem L = dc_smem(tpc, k, E, R, (int)cs, gate_warp_words<EPL>());
    int32_t *s_e = reinterpret_cast<int32_t *>(dc_raw + L.e);
    float *s_w = reinterpret_cast<float *>(dc_raw + L.w);
    unsigned long long *s_mask = reinterpret_cast<unsigned long long *>(dc_raw + L.mask);
    unsigned long long *s_rmask = reinterpret_cast<unsigned long long *>(dc_raw + L.rmask);
    int32_t *s_cnt = reinterpret_cast<int32_t *>(dc_raw + L.cnt);    // [cs][E]
    int32_t *s_rcnt = reinterpret_cast<int32_t *>(dc_raw + L.rcnt);  // [cs][R], CTA 0 of cluster 0
    int32_t *s_pre = reinterpret_cast<int32_t *>(dc_raw + L.pre);
    int32_t *s_off = reinterpret_cast<int32_t *>(dc_raw + L.off);
    __shared__ int32_t s_wsum[kDecWarps];
    __shared__ int32_t s_total;
    const bool writer = cid == 0 && cr == 0;  // counts, offsets, distinct tokens

    for (int i = threadIdx.x; i < E + R; i += kDecThreads)
        (i < E ? s_mask[i] : s_rmask[i - E]) = 0ull;
    pdl_wait();

    // this CTA's warp items (token, row segment); this cluster's share is
    // items i0, i0 + G * warps, ... for each warp, whose first row segment
    // is loaded now
    const int segs = dtype < 0 ? 0 : dtype == 0 ? bf16_segs(a.H) : fp8_segs(a.H);
    const int n_items = n_loc * segs;
    const int i0 = cid + G * warp;
    uint4 v[kBf16Unroll];
    if (i0 < n_items) {
        const int t = t_lo + i0 / segs, seg = i0 % segs;
        if (dtype == 0)
            bf16_item_load(a.x, a.H, t, seg, v);
        else
            q8_item_load(a.x, a.H, t, seg, v[0], v[1]);
    }
    __syncthreads();

    // 1. gating of this CTA's tokens, and their masks
    for (int j = warp; j < n_loc; j += kDecWarps) {
        int e;
        float w;
        gate_token_slots<EPL>(a.scores, a.bias, t_lo + j, a.gp, a.group_lanes, a.vec_rows,
                              reinterpret_cast<uint32_t *>(dc_raw + L.gate) + warp * gate_warp_words<EPL>(), e, w);
        if (lane < k) {
            s_e[j * k + lane] = e;
            s_w[j * k + lane] = w;
            if ((unsigned)e < (unsigned)E) {
                atomicOr(s_mask + e, 1ull << j);
                atomicOr(s_rmask + e / a.epr, 1ull << j);
            }
        }
    }
    pdl_trigger();
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kDecThreads) {
        const int c = __popcll(s_mask[e]);
        for (unsigned q = 0; q < cs; ++q)
            cluster_store(s_cnt + cr * E + e, q, c);
    }
    if (cid == 0)
        for (int r = threadIdx.x; r < R; r += kDecThreads)
            cluster_store(s_rcnt + cr * R + r, 0, __popcll(s_rmask[r]));
    cluster_arrive();
    // while the cluster's counts arrive: this warp's first row segment in
    // FP8 / MXFP8 (codes and scale depend on the row alone)
    uint4 qv = v[0];
    float qs = 0.0f;
    uint8_t qe = 0;
    if (i0 < n_items && dtype == 1)
        qv = fp8_quant16_regs(v[0], v[1], qs);
    else if (i0 < n_items && dtype == 2)
        qv = mx_quant16_regs(v[0], v[1], qe);
    cluster_wait();  // every CTA's counts are here; no remote access follows

    // 2. entries per expert in lower CTAs and in all (thread e owns expert e:
    //    E <= kDecThreads), scanned across the block into offsets
    int tot = 0;
    if ((int)threadIdx.x < E) {
        int pre = 0;
        for (int q = 0; q < (int)cs; ++q) {
            const int c = s_cnt[q * E + threadIdx.x];
            pre += q < (int)cr ? c : 0;
            tot += c;
        }
        s_pre[threadIdx.x] = pre;
    }
    const int incl = warp_incl_scan(tot, lane);
    if (lane == 31)
        s_wsum[warp] = incl;
    if (writer)
        for (int r = threadIdx.x; r < R; r += kDecThreads) {
            int n = 0;
            for (int q = 0; q < (int)cs; ++q)
                n += s_rcnt[q * R + r];
            a.rank_tokens[r] = n;
        }
    __syncthreads();
    int base = lane < warp ? s_wsum[lane] : 0;  // the warps below this one
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        base += __shfl_xor_sync(kFullMask, base, o);
    if ((int)threadIdx.x < E) {
        const int off = base + incl - tot;
        s_off[threadIdx.x] = off;
        if (writer) {
            a.expert_off[threadIdx.x] = off;
            a.expert_count[threadIdx.x] = tot;
        }
        if ((int)threadIdx.x == E - 1)
            s_total = off + tot;
    }
    __syncthreads();
    if (writer) {
        const int total = s_total;
        for (int r = threadIdx.x; r < R; r += kDecThreads) {
            const int lo = s_off[r * a.epr];
            const int hi = (r + 1) * a.epr < E ? s_off[(r + 1) * a.epr] : total;
            a.rank_off[r] = lo;
            a.rank_count[r] = hi - lo;
        }
        if (threadIdx.x == 0) {
            a.expert_off[E] = total;
            a.rank_off[R] = total;
        }
    }
    const int total = s_total, N = T * k;
    if (cid == 0)  // rows no entry fills (none unless an expert index was out of range)
        for (int i = total + (int)(cr * kDecThreads + threadIdx.x); i < N; i += (int)cs * kDecThreads)
            a.src[i] = -1;

    // 3. this cluster's share of this CTA's tokens: experts, weights, rows
    const int n_my = n_loc > cid ? (n_loc - cid + G - 1) / G : 0;
    for (int i = threadIdx.x; i < n_my * k; i += kDecThreads) {
        const int j = cid + (i / k) * G, slot = i - (i / k) * k;
        const long long f = (long long)(t_lo + j) * k + slot;
        const int p = dc_row(s_e, s_pre, s_off, s_mask, E, k, j, slot);
        a.topk_idx[f] = s_e[j * k + slot];
        a.topk_w[f] = s_w[j * k + slot];
        a.pos[f] = p;
        if (p >= 0)
            a.src[p] = (int)f;
    }
    // 4. this cluster's share of this CTA's row segments
    for (int item = i0; item < n_items; item += G * kDecWarps) {
        const int j = item / segs, seg = item - j * segs;
        const int t = t_lo + j;
        const bool first = item == i0;  // its row segment is loaded (and converted) already
        if (!first) {
            if (dtype == 0)
                bf16_item_load(a.x, a.H, t, seg, v);
            else
                q8_item_load(a.x, a.H, t, seg, v[0], v[1]);
        }
        int p0 = lane < k ? dc_row(s_e, s_pre, s_off, s_mask, E, k, j, lane) : -1;
        if (p0 >= a.rows) {
            if (a.err_flag)
                atomicOr(a.err_flag, 2);
            p0 = -1;
        }
        if (dtype == 0)
            bf16_item_store(a.H, k, seg, p0, -1, v, static_cast<uint16_t *>(a.recv));
        else if (dtype == 1 && first)
            fp8_item_put(a.H, k, seg, p0, -1, qv, qs, static_cast<uint8_t *>(a.recv),
                         static_cast<float *>(a.recv_scales));
        else if (dtype == 1)
            fp8_item_store(a.H, k, seg, p0, -1, v[0], v[1], static_cast<uint8_t *>(a.recv),
                           static_cast<float *>(a.recv_scales));
        else if (first)
            mxfp8_item_put(a.H, k, seg, p0, -1, qv, qe, static_cast<uint8_t *>(a.recv),
                           static_cast<uint8_t *>(a.recv_scales));
        else
            mxfp8_item_store(a.H, k, seg, p0, -1, v[0], v[1], static_cast<uint8_t *>(a.recv),
                             static_cast<uint8_t *>(a.recv_scales));
    }
}

// Barrier check: one cooperative launch that only arrives at the barrier,
// expecting `extra` arrivals that never come when extra > 0.
__global__ void __launch_bounds__(kDecThreads) barrier_selftest_kernel(unsigned *counter, unsigned extra,
                                                                       long long spin_limit, int32_t *err_flag)
{
    grid_barrier(counter, gridDim.x + extra, spin_limit, err_flag);
}

size_t decode_smem_bytes(int range_entries, int E, int epr, int warp_floats)
{
    const size_t gate = (size_t)kDecWarps * warp_floats * sizeof(float);
    const size_t lay = ((size_t)2 * E + E / epr + 2 * (size_t)range_entries) * sizeof(int32_t);
    return gate > lay ? gate : lay;
}

template <int EPL>
cudaError_t launch_epl(DecodeArgs a, cudaStream_t st)
{
    int warp_floats;
    gate_plan<EPL>(a.gp, a.scores, a.bias, a.group_lanes, a.vec_rows, warp_floats);
    // One CTA per SM, at most one per token: every CTA is resident, as the
    // grid barrier requires (the cooperative launch refuses a larger grid).
    const int sms = device_sm_count();
    const int grid = a.T < sms ? a.T : sms;
    const int range_entries = ((a.T + grid - 1) / grid) * a.gp.k;
    const size_t smem = decode_smem_bytes(range_entries, a.gp.E, a.epr, warp_floats);
    const void *fn = (const void *)decode_fused_kernel<EPL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kDecThreads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kDecThreads), args, smem, st);
}

constexpr size_t kDcMaxSmem = 100 * 1024;

template <int EPL>
cudaError_t launch_cluster_epl(DecodeArgs a, cudaStream_t st)
{
    int warp_floats;
    gate_plan<EPL>(a.gp, a.scores, a.bias, a.group_lanes, a.vec_rows, warp_floats);
    // the body for this payload, and its per-device launch caches
    const int var = a.dtype < 0 ? 0 : a.dtype == 1 ? 1 : 2;
    void (*const kern)(DecodeArgs) = var == 0   ? decode_cluster_kernel<EPL, -1>
                                     : var == 1 ? decode_cluster_kernel<EPL, 1>
                                                : decode_cluster_kernel<EPL, kDtAny>;
    const void *fn = (const void *)kern;
    static PerDeviceCache<1> smem_attr[3];
    const cudaError_t e = raise_smem_limit(smem_attr[var], fn, kDcMaxSmem);
    if (e != cudaSuccess)
        return e;
    const int cs = a.T < kDcMaxCluster ? a.T : kDcMaxCluster;
    const int tpc = (a.T + cs - 1) / cs;
    const size_t smem = dc_smem(tpc, a.gp.k, a.gp.E, a.gp.E / a.epr, cs, warp_floats).total;
    if (smem > kDcMaxSmem)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // clusters: as many as are resident at once (a cluster that waits for
    // another to finish doubles the latency; fewer leave SMs idle while the
    // rows are written), at most one per row segment of a CTA; one cluster
    // when nothing is dispatched
    int G = 1;
    if (a.dtype >= 0) {
        const int segs = a.dtype == 0 ? bf16_segs(a.H) : fp8_segs(a.H);
        G = tpc * segs;
        static PerDeviceCache<kDcMaxCluster + 1> resident[3];
        const int most = resident[var].get(
            [&] {
                cudaLaunchConfig_t q = {};
                q.gridDim = dim3((unsigned)cs);
                q.blockDim = dim3(kDecThreads);
                q.dynamicSmemBytes = kDcMaxSmem;
                q.attrs = attr;
                q.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, fn, &q) != cudaSuccess || n < 1) {
                    (void)cudaGetLastError();
                    n = 1;
                }
                return n;
            },
            cs);
        G = G < most ? G : most;
        G = G < 1 ? 1 : G;
    }
    cfg.gridDim = dim3((unsigned)(G * cs));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// The clustered kernel when the batch fits its token masks, else (or if the
// clustered launch is refused) the cooperative one.  dtype < 0 (gating and
// layout only) takes the clustered kernel alone.
template <int EPL>
cudaError_t launch_args(DecodeArgs a, cudaStream_t st)
{
    if (a.T <= kDcMaxTokens) {
        const cudaError_t e = launch_cluster_epl<EPL>(a, st);
        if (e == cudaSuccess || a.dtype < 0)
            return e;
        (void)cudaGetLastError();  // a refused launch leaves no sticky error
    }
    if (a.dtype < 0)
        return cudaErrorInvalidConfiguration;
    return launch_epl<EPL>(a, st);
}

cudaError_t launch_by_experts(const DecodeArgs &a, cudaStream_t st)
{
    if (a.gp.E <= 32)
        return launch_args<1>(a, st);
    if (a.gp.E <= 64)
        return launch_args<2>(a, st);
    if (a.gp.E <= 128)
        return launch_args<4>(a, st);
    if (a.gp.E <= 256)
        return launch_args<8>(a, st);
    return launch_args<16>(a, st);
}

}  // namespace


size_t decode_max_entries() { return kMaxEntries; }

bool gate_layout_small_supported(int T, int k) { return T >= 1 && T <= kDcMaxTokens && (long long)T * k <= kMaxEntries; }

cudaError_t launch_gate_layout_small(const float *scores, const float *bias, int T, const GateParams &gp, int epr,
                                     int32_t *topk_idx, float *topk_w, int32_t *expert_count, int32_t *expert_off,
                                     int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens, int32_t *pos,
                                     int32_t *src, cudaStream_t st)
{
    DecodeArgs a{};
    a.scores = scores;
    a.bias = bias;
    a.T = T;
    a.gp = gp;
    a.epr = epr;
    a.dtype = -1;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.expert_count = expert_count;
    a.expert_off = expert_off;
    a.rank_count = rank_count;
    a.rank_off = rank_off;
    a.rank_tokens = rank_tokens;
    a.pos = pos;
    a.src = src;
    return launch_by_experts(a, st);
}

cudaError_t launch_decode(const float *scores, const float *bias, int T, const GateParams &gp, int epr,
                          const uint16_t *x, int H, int dtype, int32_t *topk_idx, float *topk_w,
                          int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                          int32_t *rank_tokens, int32_t *pos, int32_t *src, void *recv, void *recv_scales,
                          long long rows, int32_t *err_flag, void *barrier_word, cudaStream_t st)
{
    DecodeArgs a{};
    a.scores = scores;
    a.bias = bias;
    a.T = T;
    a.gp = gp;
    a.epr = epr;
    a.x = x;
    a.H = H;
    a.dtype = dtype;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.expert_count = expert_count;
    a.expert_off = expert_off;
    a.rank_count = rank_count;
    a.rank_off = rank_off;
    a.rank_tokens = rank_tokens;
    a.pos = pos;
    a.src = src;
    a.recv = recv;
    a.recv_scales = recv_scales;
    a.rows = rows;
    a.err_flag = err_flag;
    a.barrier = static_cast<unsigned *>(barrier_word);
    a.barrier_extra = 0;
    a.spin_limit = kGridSpinLimit;
    return launch_by_experts(a, st);
}

cudaError_t launch_barrier_selftest(unsigned extra, long long spin_limit, int32_t *err_flag, void *barrier_word,
                                    cudaStream_t st)
{
    // the check starts from cleared words (a timed-out barrier leaves them mid-way)
    cudaError_t e = cudaMemsetAsync(barrier_word, 0, 2 * sizeof(unsigned), st);
    if (e != cudaSuccess)
        return e;
    unsigned *counter = static_cast<unsigned *>(barrier_word);
    void *args[] = {&counter, &extra, &spin_limit, &err_flag};
    return cudaLaunchCooperativeKernel((const void *)barrier_selftest_kernel, dim3(device_sm_count()),
                                       dim3(kDecThreads), args, 0, st);
}

}  // namespace ep
