// gate_fast.cuh -- group-limited top-k gating with a lane segment per token.
//
// "DeepEP de DeepSeek : la lib open source qui optimise la communication GPU
// pour les modeles MoE a l'echelle", section "Group-limited gating
// algorithm": a token's experts are chosen inside its best few groups.  The
// results are those of gate_token (gate_impl.cuh) bit for bit; this body
// serves the common shapes with far fewer instructions per token.
//
// A token is served by L lanes (a segment of the warp), lane s owning the
// EPL contiguous experts [s*EPL, (s+1)*EPL); a warp serves 32/L tokens, so
// the cross-lane steps are shared by several tokens instead of taking a
// whole warp each.  Per token:
//  1. keys: order-preserving uint32 of score + bias, and each lane's Q
//     largest keys;
//  2. groups (when topk_group < n_groups): a group is m whole lanes; its
//     score is the sum of its topk_in_group largest keys (largest first, in
//     fp32), merged over its lanes by xor shuffles; a group is kept when
//     fewer than topk_group groups beat it (higher score, or equal score and
//     lower index);
//  3. a bound: the smallest q-th largest key over the kept lanes, where
//     q * (kept lanes) >= k, so at least k kept keys reach it and no key
//     below it can be among the top k;
//  4. the keys that reach the bound (the candidates, a handful per token)
//     go into a shared list as 64-bit (key, inverted expert index) words, so
//     that a larger word is exactly a better choice (higher key, or equal key
//     and lower index);
//  5. each candidate's slot is the number of candidates larger than it;
//     those below k are the chosen experts, in selection order;
//  6. weights from the unbiased scores of the chosen experts, summed in slot
//     order.
// When more than `cap` keys reach the bound (massive ties) the token finds
// the exact k-th largest key instead (a bitwise search over the key space),
// takes every larger key and the lowest-index equal ones, and ranks those.
// The loops are laid out for instruction-level parallelism: the row loads
// are all issued before any is used, and the shuffles, list reads and slot
// sums are unrolled so that their latencies overlap.
#pragma once

#include "gate_impl.cuh"

namespace ep {

constexpr int kGfThreads = 256;
constexpr int kGfCap = 64;     // candidate words per token
constexpr int kGfMaxK = 32;    // slots per token

struct GateFastArgs {
    const float *scores;
    const float *bias;  // may be NULL
    int T;
    GateParams p;
    int m;    // lanes per group when grouped (topk_group < n_groups), else 0
    int q;    // keys per kept lane that make up the bound
    int cap;  // candidate words per token in shared memory (min(kGfCap, E))
    int32_t *topk_idx;
    float *topk_w;
};

// Inclusive sum over the L lanes of the caller's segment (L a power of two,
// segments aligned to L within the warp).
template <int L>
__device__ __forceinline__ int seg_incl_sum(int v, int seg)
{
#pragma unroll
    for (int off = 1; off < L; off <<= 1) {
        const int n = __shfl_up_sync(kFullMask, v, off, L);
        if (seg >= off)
            v += n;
    }
    return v;
}

template <int L>
__device__ __forceinline__ int seg_sum(int v)
{
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1)
        v += __shfl_xor_sync(kFullMask, v, off);
    return v;
}

// Keeps top[0..Q) sorted descending after offering v.
template <int Q>
__device__ __forceinline__ void offer_top(uint32_t (&top)[Q], uint32_t v)
{
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const uint32_t hi = max(top[i], v);
        v = min(top[i], v);
        top[i] = hi;
    }
}

__device__ __forceinline__ float4 ld_nc_f4(const float *p)
{
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// Padded bias rows, one per lane segment position (conflict-free 16-byte
// reads): word (e / EPL) * (EPL + 4) + e % EPL.
template <int EPL>
__device__ __forceinline__ void stage_bias(const float *bias, int E, float *s_bias, int tid, int nthreads)
{
    for (int i = tid; i < E; i += nthreads)
        s_bias[(i / EPL) * (EPL + 4) + i % EPL] = bias ? __ldg(bias + i) : 0.0f;
}

// Issues the loads of the calling lane's EPL scores of token t (the last
// token when t >= T); called first in a kernel so that their latency
// overlaps the kernel's prologue.
template <int EPL, int L>
__device__ __forceinline__ void gate_load(const GateFastArgs &a, int t, float4 (&sv)[EPL / 4])
{
    const int seg = (threadIdx.x & 31) % L;
    const int tc = t < a.T ? t : a.T - 1;
    const float *row = a.scores + (size_t)tc * a.p.E + seg * EPL;
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i)
        sv[i] = ld_nc_f4(row + 4 * i);
}

// Gates token t with the calling lane segment, from the scores gate_load
// fetched (every lane of the warp must call it together; lanes of a segment
// whose t >= T compute on the last token and store nothing).  lst: the
// token's `cap` candidate words; sel, ssc: its k chosen experts and their
// unbiased scores (shared memory).  The chosen experts also go to s_tk[j]
// when s_tk is given.
template <int EPL, int L, int Q>
__device__ __forceinline__ void gate_segment(const GateFastArgs &a, int t, const float4 (&sv)[EPL / 4],
                                             const float *s_bias, unsigned long long *lst, int32_t *sel, float *ssc,
                                             int32_t *s_tk)
{
    constexpr int KR = EPL + 4;
    const int E = a.p.E, T = a.T, k = a.p.k, cap = a.cap;
    const int seg = (threadIdx.x & 31) % L;
    const int tc = t < T ? t : T - 1;
    const int e0 = seg * EPL;

    // 1. keys (score + bias, or score + 0 -- which also turns -0 into +0)
    uint32_t ord[EPL];
    const float4 *b4 = reinterpret_cast<const float4 *>(s_bias + seg * KR);
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i) {
        const float4 b = b4[i];
        ord[4 * i] = ordered_key(sv[i].x + b.x);
        ord[4 * i + 1] = ordered_key(sv[i].y + b.y);
        ord[4 * i + 2] = ordered_key(sv[i].z + b.z);
        ord[4 * i + 3] = ordered_key(sv[i].w + b.w);
    }
    // top-Q by a tree over runs of four keys (short dependency chains)
    uint32_t top[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i)
        top[i] = 0u;
    {
        uint32_t part[EPL / 4][Q];
#pragma unroll
        for (int r = 0; r < EPL / 4; ++r) {
#pragma unroll
            for (int i = 0; i < Q; ++i)
                part[r][i] = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                offer_top<Q>(part[r], ord[4 * r + i]);
        }
#pragma unroll
        for (int r = 0; r < EPL / 4; ++r)
#pragma unroll
            for (int i = 0; i < Q; ++i)
                offer_top<Q>(top, part[r][i]);
    }

    // 2. groups of m whole lanes
    bool kept = true;
    if (a.m > 0) {
        const int m = a.m, G = L / m, kin = a.p.kin;
        uint32_t g[Q];
#pragma unroll
        for (int i = 0; i < Q; ++i)
            g[i] = top[i];
#pragma unroll
        for (int off = 1; off < L; off <<= 1) {
            if (off >= m)
                break;
            uint32_t o[Q];
#pragma unroll
            for (int i = 0; i < Q; ++i)
                o[i] = __shfl_xor_sync(kFullMask, g[i], off);
#pragma unroll
            for (int i = 0; i < Q; ++i)
                offer_top<Q>(g, o[i]);
        }
        float gs = key_value(g[0]);
#pragma unroll
        for (int i = 1; i < Q; ++i)
            if (i < kin)
                gs = gs + key_value(g[i]);
        const uint32_t gk = ordered_key(gs);
        const int my_g = seg / m;
        uint32_t og[L];
#pragma unroll
        for (int gg = 0; gg < L; ++gg)
            og[gg] = __shfl_sync(kFullMask, gk, (gg * m) & (L - 1), L);
        int beaten = 0;
#pragma unroll
        for (int gg = 0; gg < L; ++gg)
            if (gg < G)
                beaten += (og[gg] > gk || (og[gg] == gk && gg < my_g)) ? 1 : 0;
        kept = beaten < a.p.Kg;
    }

    // 3. the bound: the smallest q-th largest key of the kept lanes
    uint32_t bnd = top[0];
#pragma unroll
    for (int i = 1; i < Q; ++i)
        if (i == a.q - 1)
            bnd = top[i];
    if (!kept)
        bnd = 0xFFFFFFFFu;
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1)
        bnd = min(bnd, __shfl_xor_sync(kFullMask, bnd, off));

    // 4. candidates: the kept keys that reach the bound
    uint32_t cm = 0u;
    if (kept) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            cm |= (ord[i] >= bnd ? 1u : 0u) << i;
    }
    int incl = seg_incl_sum<L>(__popc(cm), seg);
    int ntot = __shfl_sync(kFullMask, incl, L - 1, L);
    const bool over = ntot > cap;
    if (__any_sync(kFullMask, over)) {
        // The exact k-th largest kept key th: the largest value with at
        // least k kept keys at or above it, found bit by bit.
        uint32_t th = 0u;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t x = th | (1u << bit);
            int c = 0;
            if (kept) {
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    c += ord[i] >= x ? 1 : 0;
            }
            if (seg_sum<L>(c) >= k)
                th = x;
        }
        uint32_t gtm = 0u, eqm = 0u;
        if (kept) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                gtm |= (ord[i] > th ? 1u : 0u) << i;
                eqm |= (ord[i] == th ? 1u : 0u) << i;
            }
        }
        const int ngt = seg_sum<L>(__popc(gtm));
        const int eq_before = seg_incl_sum<L>(__popc(eqm), seg) - __popc(eqm);
        int take = k - ngt - eq_before;  // equal keys this lane still takes, lowest index first
        uint32_t em = 0u, rest = eqm;
        while (take > 0 && rest != 0u) {
            em |= rest & (0u - rest);
            rest &= rest - 1u;
            --take;
        }
        if (over)
            cm = gtm | em;
        incl = seg_incl_sum<L>(__popc(cm), seg);
        ntot = __shfl_sync(kFullMask, incl, L - 1, L);
    }

    for (int j = seg; j < k; j += L) {
        sel[j] = 0;  // a slot no candidate fills (impossible for finite scores) stays in range
        ssc[j] = 0.0f;
    }
    {
        int w = incl - __popc(cm);
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((cm >> i) & 1u)
                lst[w++] = ((unsigned long long)ord[i] << 32) | (uint32_t)(0xFFFFu - (unsigned)(e0 + i));
    }
    __syncwarp();

    // 5. slot of each candidate = candidates larger than it
    const float *srow = a.scores + (size_t)tc * E;
    for (int c = seg; c < ntot; c += 2 * L) {
        const unsigned long long me0 = lst[c];
        const bool two = c + L < ntot;
        const unsigned long long me1 = two ? lst[c + L] : ~0ull;
        int r0 = 0, r1 = 0;
        int c2 = 0;
        for (; c2 + 4 <= ntot; c2 += 4) {
            const unsigned long long v0 = lst[c2], v1 = lst[c2 + 1], v2 = lst[c2 + 2], v3 = lst[c2 + 3];
            r0 += (v0 > me0 ? 1 : 0) + (v1 > me0 ? 1 : 0) + (v2 > me0 ? 1 : 0) + (v3 > me0 ? 1 : 0);
            r1 += (v0 > me1 ? 1 : 0) + (v1 > me1 ? 1 : 0) + (v2 > me1 ? 1 : 0) + (v3 > me1 ? 1 : 0);
        }
        for (; c2 < ntot; ++c2) {
            const unsigned long long v = lst[c2];
            r0 += v > me0 ? 1 : 0;
            r1 += v > me1 ? 1 : 0;
        }
        if (r0 < k) {
            const int e = (int)(0xFFFFu - (uint32_t)(me0 & 0xFFFFu));
            sel[r0] = e;
            ssc[r0] = __ldg(srow + e);
        }
        if (two && r1 < k) {
            const int e = (int)(0xFFFFu - (uint32_t)(me1 & 0xFFFFu));
            sel[r1] = e;
            ssc[r1] = __ldg(srow + e);
        }
    }
    __syncwarp();

    // 6. weights from the unbiased scores, sums in slot order (the slot
    // scores are read eight at a time so that their loads overlap)
    if (t < T) {
        float den = 0.0f, mx = ssc[0];
        if (a.p.score_fn != 0) {  // softmax renormalised over the chosen k
            for (int j0 = 0; j0 < k; j0 += 8) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    v[u] = j0 + u < k ? ssc[j0 + u] : -INFINITY;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    mx = fmaxf(mx, v[u]);
            }
        }
        for (int j0 = 0; j0 < k; j0 += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = j0 + u < k ? ssc[j0 + u] : 0.0f;
            if (a.p.score_fn == 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (j0 + u < k)
                        den += v[u];
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (j0 + u < k)
                        den += expf(v[u] - mx);
            }
        }
        for (int j = seg; j < k; j += L) {
            const float sj = ssc[j];
            float w;
            if (a.p.score_fn == 0)
                w = a.p.normalize ? sj / den : sj;
            else
                w = expf(sj - mx) / den;
            const int e = sel[j];
            a.topk_idx[(size_t)t * k + j] = e;
            a.topk_w[(size_t)t * k + j] = w;
            if (s_tk)
                s_tk[j] = e;
        }
    }
}

// Launch plan of the lane-segment body: a token takes L lanes of EPL
// experts each.  Shapes: E in {8, 16, 32, 64, 128, 256}; groups, when they
// limit the choice, of whole lanes; the softmax mode only renormalised; at
// most 4 keys per lane for the group score and the bound; k <= 32; 16-byte
// score rows and bias.
struct GateFastPlan {
    int EPL, L, Q, m, q, cap;
};

inline bool gate_fast_plan(const GateParams &p, const float *scores, const float *bias, GateFastPlan &f)
{
    f = GateFastPlan{};
    const int E = p.E;
    switch (E) {
    case 8: f.EPL = 8; f.L = 1; break;
    case 16: f.EPL = 8; f.L = 2; break;
    case 32: f.EPL = 8; f.L = 4; break;
    case 64: f.EPL = 8; f.L = 8; break;
    case 128: f.EPL = 16; f.L = 8; break;
    case 256: f.EPL = 32; f.L = 8; break;
    default: return false;
    }
    if (p.k > kGfMaxK || (p.score_fn != 0 && !p.normalize))
        return false;  // the full softmax needs every score's exponential
    if ((reinterpret_cast<uintptr_t>(scores) & 15) != 0 || (reinterpret_cast<uintptr_t>(bias) & 15) != 0)
        return false;
    const bool grouped = p.Kg < p.G;
    f.m = 0;
    int kept_lanes = f.L;
    int need = 1;
    if (grouped) {
        const int gsize = E / p.G;
        if (gsize % f.EPL != 0)
            return false;
        f.m = gsize / f.EPL;  // divides L, a power of two
        kept_lanes = p.Kg * f.m;
        need = p.kin;
    }
    f.q = (p.k + kept_lanes - 1) / kept_lanes;
    if (f.q > need)
        need = f.q;
    if (need > 4 || f.q > f.EPL)
        return false;
    f.Q = need <= 1 ? 1 : (need <= 2 ? 2 : 4);
    f.cap = E < kGfCap ? E : kGfCap;
    return true;
}

// Shared-memory bytes of the standalone kernel: candidate lists, chosen
// experts and their scores, the padded bias.
template <int EPL, int L>
__host__ __device__ constexpr size_t gate_fast_smem(int cap, int k)
{
    return (size_t)(kGfThreads / L) * cap * 8 + (size_t)(kGfThreads / L) * k * 8 + (size_t)L * (EPL + 4) * 4;
}

template <int EPL, int L, int Q>
__global__ void __launch_bounds__(kGfThreads) gate_fast_kernel(const GateFastArgs a)
{
    constexpr int TPC = kGfThreads / L;  // tokens per CTA
    extern __shared__ __align__(16) unsigned long long gsm8[];
    const int cap = a.cap, k = a.p.k;
    unsigned long long *s_list = gsm8;                                 // [TPC][cap]
    int32_t *s_sel = reinterpret_cast<int32_t *>(s_list + TPC * cap);  // [TPC][k]
    float *s_ssc = reinterpret_cast<float *>(s_sel + TPC * k);         // [TPC][k]
    float *s_bias = s_ssc + TPC * k;                                   // [L][EPL + 4]
    const int tl = threadIdx.x / L;
    const int t = blockIdx.x * TPC + tl;
    float4 sv[EPL / 4];
    gate_load<EPL, L>(a, t, sv);
    stage_bias<EPL>(a.bias, a.p.E, s_bias, threadIdx.x, kGfThreads);
    __syncthreads();
    gate_segment<EPL, L, Q>(a, t, sv, s_bias, s_list + tl * cap, s_sel + tl * k, s_ssc + tl * k, nullptr);
}

}  // namespace ep
