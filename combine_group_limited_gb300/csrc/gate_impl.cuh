// gate_impl.cuh -- the per-token body of the group-limited top-k gating,
// shared by the gating kernel and the fused low-latency decode kernel.
//
// "DeepEP de DeepSeek : la lib open source qui optimise la communication GPU
// pour les modeles MoE a l'echelle", section "Group-limited gating
// algorithm".  One warp gates one token; see gate.cu for the layout.
#pragma once

#include <math.h>

#include "ep_internal.cuh"

namespace ep {

constexpr int kMaxKin = 4;

// Keep top[0..3] sorted descending after offering v.
__device__ __forceinline__ void offer(float (&top)[kMaxKin], float v)
{
#pragma unroll
    for (int q = 0; q < kMaxKin; ++q) {
        const float hi = fmaxf(top[q], v);
        v = fminf(top[q], v);
        top[q] = hi;
    }
}

__device__ __forceinline__ void offer_u(uint32_t (&top)[kMaxKin], uint32_t v)
{
#pragma unroll
    for (int q = 0; q < kMaxKin; ++q) {
        const uint32_t hi = max(top[q], v);
        v = min(top[q], v);
        top[q] = hi;
    }
}

// Inverse of ordered_key.
__device__ __forceinline__ float key_value(uint32_t o)
{
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Descending bitonic sort of N (a power of two) keys; each compare-exchange
// is one max and one min.
template <int N>
__device__ __forceinline__ void sort_desc(uint32_t (&a)[N])
{
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size / 2; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint32_t hi = max(a[i], a[j]), lo = min(a[i], a[j]);
                    const bool desc = (i & size) == 0;
                    a[i] = desc ? hi : lo;
                    a[j] = desc ? lo : hi;
                }
            }
        }
    }
}

// Words of per-warp shared scratch gate_token needs: every lane's sorted
// keys, then the chosen experts of the k slots, then their raw scores.
// (The general group path also stages the row's keys there first: E <= 32 *
// EPL words.)
template <int EPL>
__host__ __device__ constexpr int gate_warp_words()
{
    return 32 * EPL + 64;
}

// Gates token t with the calling warp (all 32 lanes).  wsm: the warp's
// gate_warp_words<EPL>() words of shared memory.  Lane j < k writes slot j.
//
// Lane l owns experts [l*EPL, (l+1)*EPL).  It maps its keys to
// order-preserving uint32s (0 = no candidate) and sorts a copy descending.
// Group scores: for groups that are power-of-two runs of whole lanes, the
// largest keys of a group are among its lanes' sorted heads (merged with xor
// shuffles); other groups are scanned by one lane each from shared memory.
// Each top-k round is a warp max over the lanes' current heads; among lanes
// holding that key the lowest lane wins (its experts have the lower
// indices), and it advances to its next sorted key (read from shared
// memory).  A lane's wins took its sorted keys in order, so at the end it
// finds each won key among its unsorted keys -- equal keys go lowest index
// first, the order the tie rule asks for -- and writes the expert of that
// round's slot.
//
// gate_token_slots leaves slot `lane`'s expert and weight in out_e and out_w
// of lane lane < k; gate_token writes them to topk_idx and topk_w.
template <int EPL>
__device__ __forceinline__ void gate_token_slots(const float *__restrict__ scores, const float *__restrict__ bias,
                                                 int t, const GateParams &p, int group_lanes, int vec_rows,
                                                 uint32_t *wsm, int &out_e, float &out_w)
{
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int e0 = lane * EPL;
    const float *row = scores + (size_t)t * E;

    // sc: the raw scores (kept for the weights, so that the row is read
    // once); key: the selection keys score + bias
    float sc[EPL], key[EPL];
    if (EPL % 4 == 0 && vec_rows) {
#pragma unroll
        for (int i = 0; i < EPL; i += 4) {
            const float4 s4 = __ldg(reinterpret_cast<const float4 *>(row + e0 + i));
            sc[i] = s4.x;
            sc[i + 1] = s4.y;
            sc[i + 2] = s4.z;
            sc[i + 3] = s4.w;
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            key[i] = sc[i];
        if (bias) {
#pragma unroll
            for (int i = 0; i < EPL; i += 4) {
                const float4 b4 = __ldg(reinterpret_cast<const float4 *>(bias + e0 + i));
                key[i] = sc[i] + b4.x;
                key[i + 1] = sc[i + 1] + b4.y;
                key[i + 2] = sc[i + 2] + b4.z;
                key[i + 3] = sc[i + 3] + b4.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = e0 + i;
            sc[i] = e < E ? __ldg(row + e) : 0.0f;
            key[i] = e < E ? (bias ? sc[i] + __ldg(bias + e) : sc[i]) : -INFINITY;
        }
    }
    uint32_t ord[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        ord[i] = (e0 + i < E) ? ordered_key(key[i]) : 0u;

    uint32_t srt[EPL];
    bool lane_kept = true;
    const bool grouped = p.Kg < p.G;
    if (grouped && group_lanes == 0) {
        // General groups: lane g scans group g's keys in shared memory.
        const int gsize = E / p.G;
        float *skey = reinterpret_cast<float *>(wsm);
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (e0 + i < E)
                skey[e0 + i] = key[i];
        __syncwarp();
        float gs = -INFINITY;
        if (lane < p.G) {
            float top[kMaxKin];
#pragma unroll
            for (int q = 0; q < kMaxKin; ++q)
                top[q] = -INFINITY;
            for (int e = lane * gsize; e < (lane + 1) * gsize; ++e)
                offer(top, skey[e]);
            gs = top[0];
#pragma unroll
            for (int q = 1; q < kMaxKin; ++q)
                if (q < p.kin)
                    gs = gs + top[q];
        }
        uint32_t kept = 0u;
        for (int r = 0; r < p.Kg; ++r) {
            const bool c = lane < p.G && !((kept >> lane) & 1u);
            const uint32_t o = c ? ordered_key(gs) : 0u;
            const uint32_t mx = __reduce_max_sync(kFullMask, o);
            const uint32_t g = __reduce_min_sync(kFullMask, (c && o == mx) ? (uint32_t)lane : 0xFFFFFFFFu);
            if (g < 32u)
                kept |= 1u << g;
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (e0 + i < E && !((kept >> ((e0 + i) / gsize)) & 1u))
                ord[i] = 0u;
        __syncwarp();  // the staged keys are dead; wsm now holds the lists
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            srt[i] = ord[i];
        sort_desc(srt);
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            srt[i] = ord[i];
        sort_desc(srt);
        if (grouped) {
            // Groups are runs of group_lanes whole lanes (a power of two): the
            // group's largest keys are among its lanes' sorted heads.
            float gs;
            if (p.kin <= 2) {
                uint32_t a0 = srt[0], a1 = EPL > 1 ? srt[EPL > 1 ? 1 : 0] : 0u;
#pragma unroll 4
                for (int off = 1; off < group_lanes; off <<= 1) {
                    const uint32_t b0 = __shfl_xor_sync(kFullMask, a0, off);
                    const uint32_t b1 = __shfl_xor_sync(kFullMask, a1, off);
                    const uint32_t n1 = max(min(a0, b0), max(a1, b1));
                    a0 = max(a0, b0);
                    a1 = n1;
                }
                gs = key_value(a0);
                if (p.kin == 2)
                    gs = gs + key_value(a1);
            } else {
                uint32_t top[kMaxKin];
#pragma unroll
                for (int q = 0; q < kMaxKin; ++q)
                    top[q] = (q < EPL) ? srt[q < EPL ? q : 0] : 0u;
                for (int off = 1; off < group_lanes; off <<= 1) {
                    uint32_t other[kMaxKin];
#pragma unroll
                    for (int q = 0; q < kMaxKin; ++q)
                        other[q] = __shfl_xor_sync(kFullMask, top[q], off);
#pragma unroll
                    for (int q = 0; q < kMaxKin; ++q)
                        offer_u(top, other[q]);
                }
                gs = key_value(top[0]);
#pragma unroll
                for (int q = 1; q < kMaxKin; ++q)
                    if (q < p.kin)
                        gs = gs + key_value(top[q]);
            }
            const int my_group = lane / group_lanes;
            const bool leader = (lane % group_lanes) == 0 && my_group < p.G;
            uint32_t kept = 0u;
#pragma unroll 4
            for (int r = 0; r < p.Kg; ++r) {
                const bool c = leader && !((kept >> my_group) & 1u);
                const uint32_t o = c ? ordered_key(gs) : 0u;
                const uint32_t mx = __reduce_max_sync(kFullMask, o);
                const uint32_t g =
                    __reduce_min_sync(kFullMask, (c && o == mx) ? (uint32_t)my_group : 0xFFFFFFFFu);
                if (g < 32u)
                    kept |= 1u << g;
            }
            lane_kept = (kept >> my_group) & 1u;
        }
    }

    // This lane's sorted keys, for the rounds to read past the head.
    uint32_t *lst = wsm + lane * EPL;
    int32_t *s_e = reinterpret_cast<int32_t *>(wsm + 32 * EPL);
    float *s_raw = reinterpret_cast<float *>(wsm + 32 * EPL + 32);
    if (EPL % 4 == 0) {
#pragma unroll
        for (int i = 0; i < EPL; i += 4)
            *reinterpret_cast<uint4 *>(lst + i) = make_uint4(srt[i], srt[i + 1], srt[i + 2], srt[i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            lst[i] = srt[i];
    }
    // a slot no round fills (impossible for finite scores) names expert 0
    s_e[lane] = 0;
    s_raw[lane] = __shfl_sync(kFullMask, sc[0], 0);
    __syncwarp();

    // Top-k rounds over the lanes' heads.
    const int k = p.k;
    uint32_t hk = lane_kept ? srt[0] : 0u;
    int h = 0;
    uint32_t won = 0u;  // bit j: this lane won round j
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
        const uint32_t mx = __reduce_max_sync(kFullMask, hk);
        const unsigned bal = __ballot_sync(kFullMask, hk == mx && mx != 0u);
        if (bal != 0u && lane == __ffs(bal) - 1) {
            won |= 1u << j;
            ++h;
            hk = h < EPL ? lst[h] : 0u;
        }
    }
    // Experts of the won rounds: the n-th win took sorted key n; the lowest
    // unused index holding that key is its expert.
    uint32_t used = 0u;
    int n = 0;
    while (__any_sync(kFullMask, won != 0u)) {
        if (won != 0u) {
            const int j = __ffs(won) - 1;
            won &= won - 1u;
            const uint32_t kv = lst[n++];
            uint32_t m = 0u;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                m |= (ord[i] == kv ? 1u : 0u) << i;
            m &= ~used;
            const int i = __ffs(m) - 1;
            used |= 1u << i;
            float v = sc[0];
#pragma unroll
            for (int ii = 1; ii < EPL; ++ii)
                v = ii == i ? sc[ii] : v;
            s_e[j] = e0 + i;
            s_raw[j] = v;
        }
    }
    __syncwarp();
    int my_e = 0;
    float my_s = 0.0f;  // the unbiased score of slot `lane`
    if (lane < k) {
        const int e = s_e[lane];
        my_e = (unsigned)e < (unsigned)E ? e : 0;
        my_s = s_raw[lane];
    }
    __syncwarp();  // the scratch may be reused by the warp's next token

    // Weights from the unbiased score, sums taken in slot order.
    float w;
    if (p.score_fn == 0) {
        if (p.normalize) {
            float den = 0.0f;
#pragma unroll 8
            for (int jj = 0; jj < k; ++jj)
                den += __shfl_sync(kFullMask, my_s, jj);
            w = my_s / den;
        } else {
            w = my_s;
        }
    } else if (p.normalize) {
        float m = (lane < k) ? my_s : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
        const float ex = (lane < k) ? expf(my_s - m) : 0.0f;
        float den = 0.0f;
#pragma unroll 8
        for (int jj = 0; jj < k; ++jj)
            den += __shfl_sync(kFullMask, ex, jj);
        w = ex / den;
    } else {
        float raw[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            raw[i] = (e0 + i < E) ? sc[i] : 0.0f;
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (e0 + i < E)
                m = fmaxf(m, raw[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
        float z = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (e0 + i < E)
                z += expf(raw[i] - m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            z += __shfl_xor_sync(kFullMask, z, off);
        w = expf(my_s - m) / z;
    }
    out_e = my_e;
    out_w = w;
}

template <int EPL>
__device__ __forceinline__ void gate_token(const float *__restrict__ scores, const float *__restrict__ bias, int t,
                                           const GateParams &p, int group_lanes, int vec_rows, uint32_t *wsm,
                                           int32_t *__restrict__ topk_idx, float *__restrict__ topk_w)
{
    int e;
    float w;
    gate_token_slots<EPL>(scores, bias, t, p, group_lanes, vec_rows, wsm, e, w);
    const int lane = threadIdx.x & 31;
    if (lane < p.k) {
        topk_idx[(size_t)t * p.k + lane] = e;
        topk_w[(size_t)t * p.k + lane] = w;
    }
}


// Host-side launch plan shared by the gating launchers: whether groups are
// power-of-two runs of whole lanes (group_lanes > 0), whether 16-byte row
// loads are allowed, and the shared memory words per warp gate_token needs.
template <int EPL>
inline void gate_plan(const GateParams &p, const float *scores, const float *bias, int &group_lanes, int &vec_rows,
                      int &warp_floats)
{
    group_lanes = 0;
    if (p.Kg < p.G) {
        const int gsize = p.E / p.G;
        if (gsize % EPL == 0) {
            const int L = gsize / EPL;
            if (L <= 32 && (L & (L - 1)) == 0)
                group_lanes = L;
        }
    }
    vec_rows = (EPL % 4 == 0 && p.E == 32 * EPL && (reinterpret_cast<uintptr_t>(scores) & 15) == 0 &&
                (reinterpret_cast<uintptr_t>(bias) & 15) == 0)
                   ? 1
                   : 0;
    warp_floats = gate_warp_words<EPL>();
}

}  // namespace ep
