// gate.cu -- step 1: group-limited top-k gating, one warp per token.
//
// "DeepEP de DeepSeek : la lib open source qui optimise la communication GPU
// pour les modeles MoE a l'echelle", section "Group-limited gating
// algorithm": each token's experts are chosen inside a few groups instead of
// over all experts.  Groups are contiguous blocks of E/G experts; a group's
// score is the sum of its topk_in_group largest keys (largest first, fp32);
// the topk_group best groups are kept and the top-k experts are chosen among
// them.  key = score + bias selects; the unbiased score weighs.  Ties go to
// the lower index.
//
// Layout: lane l of the token's warp owns experts l, l+32, l+64, ... (EPL of
// them, coalesced loads of the score row).  Each selection round is a warp
// max over order-preserving uint32 keys (redux.sync), then a warp min over
// the indices that reach the max, so ties resolve to the lower index without
// 64-bit shuffles.  Keys and raw scores also go to shared memory for the
// per-group scan (lane g scores group g) and for the weight lookup.
#include <math.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;
constexpr int kMaxKin = 4;

template <int EPL>
__global__ void __launch_bounds__(kGateThreads) gate_kernel(const float *__restrict__ scores,
                                                            const float *__restrict__ bias, int T,
                                                            GateParams p, int32_t *__restrict__ topk_idx,
                                                            float *__restrict__ topk_w)
{
    extern __shared__ float gate_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kGateWarps + warp;
    if (t >= T)
        return;  // the whole warp leaves together
    const int E = p.E;
    float *skey = gate_smem + warp * 2 * E;
    float *sraw = skey + E;
    const float *row = scores + (size_t)t * E;

    float key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        float kv = -INFINITY;
        if (e < E) {
            const float s = __ldg(row + e);
            kv = bias ? s + __ldg(bias + e) : s;
            skey[e] = kv;
            sraw[e] = s;
        }
        key[i] = kv;
    }
    __syncwarp();

    const int gsize = E / p.G;
    uint32_t kept = 0xFFFFFFFFu;
    if (p.Kg < p.G) {
        // Group score: lane g scans group g's keys, keeping the largest kin.
        float gs = -INFINITY;
        if (lane < p.G) {
            float top[kMaxKin];
#pragma unroll
            for (int q = 0; q < kMaxKin; ++q)
                top[q] = -INFINITY;
            for (int e = lane * gsize; e < (lane + 1) * gsize; ++e) {
                float v = skey[e];
#pragma unroll
                for (int q = 0; q < kMaxKin; ++q)
                    if (v > top[q]) {
                        const float tmp = top[q];
                        top[q] = v;
                        v = tmp;
                    }
            }
            gs = top[0];
#pragma unroll
            for (int q = 1; q < kMaxKin; ++q)
                if (q < p.kin)
                    gs = gs + top[q];
        }
        kept = 0u;
        for (int r = 0; r < p.Kg; ++r) {
            const bool cand = lane < p.G && !((kept >> lane) & 1u);
            const uint32_t o = cand ? ordered_key(gs) : 0u;
            const uint32_t mx = __reduce_max_sync(kFullMask, o);
            const uint32_t g = __reduce_min_sync(kFullMask, (cand && o == mx) ? (uint32_t)lane : 0xFFFFFFFFu);
            if (g < 32u)
                kept |= 1u << g;
        }
    }

    // Top-k experts inside the kept groups.
    uint32_t taken = 0u;
    int my_e = 0;
    for (int j = 0; j < p.k; ++j) {
        uint32_t bo = 0u;
        uint32_t be = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            const bool ok = e < E && !((taken >> i) & 1u) && ((kept >> (e / gsize)) & 1u);
            const uint32_t o = ok ? ordered_key(key[i]) : 0u;
            if (ok && o > bo) {  // i ascending: the first maximum is the lowest index
                bo = o;
                be = (uint32_t)e;
            }
        }
        const uint32_t mx = __reduce_max_sync(kFullMask, bo);
        const uint32_t wu = __reduce_min_sync(kFullMask, (bo == mx) ? be : 0xFFFFFFFFu);
        // Always a valid expert for finite scores; clamped so that even
        // unsupported (NaN) input cannot index outside the score row.
        const int win = wu < (uint32_t)E ? (int)wu : 0;
        if ((win & 31) == lane)
            taken |= 1u << (win >> 5);
        if (lane == j)
            my_e = win;
    }

    // Weights from the unbiased score, sums taken in slot order.
    const int k = p.k;
    const float my_s = (lane < k) ? sraw[my_e] : 0.0f;
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
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32)
            m = fmaxf(m, sraw[e]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
        float z = 0.0f;
        for (int e = lane; e < E; e += 32)
            z += expf(sraw[e] - m);
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

template <int EPL>
cudaError_t launch_epl(const float *scores, const float *bias, int T, const GateParams &p, int32_t *idx,
                       float *w, cudaStream_t st)
{
    const size_t smem = (size_t)kGateWarps * 2 * p.E * sizeof(float);
    const int grid = (T + kGateWarps - 1) / kGateWarps;
    gate_kernel<EPL><<<grid, kGateThreads, smem, st>>>(scores, bias, T, p, idx, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate(const float *scores, const float *bias, int T, const GateParams &p,
                        int32_t *topk_idx, float *topk_w, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    if (p.E <= 32)
        return launch_epl<1>(scores, bias, T, p, topk_idx, topk_w, st);
    if (p.E <= 64)
        return launch_epl<2>(scores, bias, T, p, topk_idx, topk_w, st);
    if (p.E <= 128)
        return launch_epl<4>(scores, bias, T, p, topk_idx, topk_w, st);
    if (p.E <= 256)
        return launch_epl<8>(scores, bias, T, p, topk_idx, topk_w, st);
    return launch_epl<16>(scores, bias, T, p, topk_idx, topk_w, st);
}

}  // namespace ep
