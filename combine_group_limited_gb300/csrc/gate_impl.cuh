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

// Descending bitonic sort of N (a power of two) packed candidates.
template <int N>
__device__ __forceinline__ void sort_desc(unsigned long long (&a)[N])
{
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size / 2; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long x = a[i], y = a[j];
                    if (desc ? (x < y) : (x > y)) {
                        a[i] = y;
                        a[j] = x;
                    }
                }
            }
        }
    }
}

// Candidate = key in the high word, (EPL-1-i) in the low word: the larger
// key wins, then the lower index.  0 marks "no candidate".
template <int EPL>
__device__ __forceinline__ unsigned long long pack_cand(uint32_t ord, int i)
{
    return ord ? ((unsigned long long)ord << 32) | (unsigned)(EPL - 1 - i) : 0ull;
}

// Gates token t with the calling warp (all 32 lanes).  warp_smem: E floats
// of shared memory for this warp, used only when group_lanes == 0 and the
// groups are limited.  Lane j < k writes slot j.
template <int EPL>
__device__ __forceinline__ void gate_token(const float *__restrict__ scores, const float *__restrict__ bias, int t,
                                           const GateParams &p, int group_lanes, int vec_rows, float *warp_smem,
                                           int32_t *__restrict__ topk_idx, float *__restrict__ topk_w)
{
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int e0 = lane * EPL;
    const float *row = scores + (size_t)t * E;

    float key[EPL];
    if (EPL % 4 == 0 && vec_rows) {
#pragma unroll
        for (int i = 0; i < EPL; i += 4) {
            const float4 s4 = __ldg(reinterpret_cast<const float4 *>(row + e0 + i));
            key[i] = s4.x;
            key[i + 1] = s4.y;
            key[i + 2] = s4.z;
            key[i + 3] = s4.w;
        }
        if (bias) {
#pragma unroll
            for (int i = 0; i < EPL; i += 4) {
                const float4 b4 = __ldg(reinterpret_cast<const float4 *>(bias + e0 + i));
                key[i] = key[i] + b4.x;
                key[i + 1] = key[i + 1] + b4.y;
                key[i + 2] = key[i + 2] + b4.z;
                key[i + 3] = key[i + 3] + b4.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = e0 + i;
            key[i] = e < E ? (bias ? __ldg(row + e) + __ldg(bias + e) : __ldg(row + e)) : -INFINITY;
        }
    }
    uint32_t ord[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        ord[i] = (e0 + i < E) ? ordered_key(key[i]) : 0u;

    unsigned long long cand[EPL];
    const bool grouped = p.Kg < p.G;
    if (grouped && group_lanes == 0) {
        // General groups: lane g scans group g's keys in shared memory.
        const int gsize = E / p.G;
        float *skey = warp_smem;
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
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            cand[i] = pack_cand<EPL>(ord[i], i);
        sort_desc(cand);
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            cand[i] = pack_cand<EPL>(ord[i], i);
        sort_desc(cand);
        if (grouped) {
            // Groups are runs of group_lanes whole lanes (a power of two): the
            // group's largest keys are among its lanes' sorted heads.
            uint32_t top[kMaxKin];
#pragma unroll
            for (int q = 0; q < kMaxKin; ++q)
                top[q] = (q < EPL) ? (uint32_t)(cand[q < EPL ? q : 0] >> 32) : 0u;
            for (int off = 1; off < group_lanes; off <<= 1) {
                uint32_t other[kMaxKin];
#pragma unroll
                for (int q = 0; q < kMaxKin; ++q)
                    other[q] = __shfl_xor_sync(kFullMask, top[q], off);
#pragma unroll
                for (int q = 0; q < kMaxKin; ++q)
                    offer_u(top, other[q]);
            }
            const int my_group = lane / group_lanes;
            const bool leader = (lane % group_lanes) == 0 && my_group < p.G;
            float gs = key_value(top[0]);
#pragma unroll
            for (int q = 1; q < kMaxKin; ++q)
                if (q < p.kin)
                    gs = gs + key_value(top[q]);
            uint32_t kept = 0u;
            for (int r = 0; r < p.Kg; ++r) {
                const bool c = leader && !((kept >> my_group) & 1u);
                const uint32_t o = c ? ordered_key(gs) : 0u;
                const uint32_t mx = __reduce_max_sync(kFullMask, o);
                const uint32_t g =
                    __reduce_min_sync(kFullMask, (c && o == mx) ? (uint32_t)my_group : 0xFFFFFFFFu);
                if (g < 32u)
                    kept |= 1u << g;
            }
            if (!((kept >> my_group) & 1u)) {
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    cand[i] = 0ull;
            }
        }
    }

    // Top-k rounds over the lanes' sorted heads.
    int my_e = 0;
    for (int j = 0; j < p.k; ++j) {
        const uint32_t hk = (uint32_t)(cand[0] >> 32);
        const uint32_t mx = __reduce_max_sync(kFullMask, hk);
        const uint32_t mine = (hk == mx && hk != 0u) ? (uint32_t)(e0 + EPL - 1 - (int)(cand[0] & 0xFFFFFFFFull))
                                                     : 0xFFFFFFFFu;
        const uint32_t wu = __reduce_min_sync(kFullMask, mine);
        if (wu == mine && wu != 0xFFFFFFFFu) {
#pragma unroll
            for (int i = 0; i + 1 < EPL; ++i)
                cand[i] = cand[i + 1];
            cand[EPL - 1] = 0ull;
        }
        // Always a valid expert for finite scores; clamped so that even
        // unsupported (NaN) input cannot index outside the score row.
        if (lane == j)
            my_e = wu < (uint32_t)E ? (int)wu : 0;
    }

    // Weights from the unbiased score, sums taken in slot order.
    const int k = p.k;
    const float my_s = (lane < k) ? __ldg(row + my_e) : 0.0f;
    float w;
    if (p.score_fn == 0) {
        if (p.normalize) {
            float den = 0.0f;
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
        for (int jj = 0; jj < k; ++jj)
            den += __shfl_sync(kFullMask, ex, jj);
        w = ex / den;
    } else {
        float raw[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            raw[i] = (e0 + i < E) ? __ldg(row + e0 + i) : 0.0f;
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
    if (lane < k) {
        topk_idx[(size_t)t * k + lane] = my_e;
        topk_w[(size_t)t * k + lane] = w;
    }
}


// Host-side launch plan shared by the gating launchers: whether groups are
// power-of-two runs of whole lanes (group_lanes > 0), whether 16-byte row
// loads are allowed, and the shared memory (floats per warp) the general
// group path needs.
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
    warp_floats = (p.Kg < p.G && group_lanes == 0) ? p.E : 0;
}

}  // namespace ep
