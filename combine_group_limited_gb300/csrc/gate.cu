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
// Layout: lane l of the token's warp owns the EPL contiguous experts
// [l*EPL, (l+1)*EPL), loaded as 16-byte vectors when the row allows.  Each
// lane sorts its order-preserving uint32 keys once (a bitonic network of
// max/min pairs).  When a group is a power-of-two run of whole lanes (E=256,
// G=8: 4 lanes of 8), the group's largest keys come from the lanes' sorted
// heads merged by xor shuffles; otherwise lane g scans group g in shared
// memory.  Each top-k round is one warp max over the lanes' heads; the
// lowest lane holding it wins (lower lanes own lower indices) and steps to
// its next key.  Only at the end does a lane find which of its experts its
// won keys were (equal keys lowest index first).  The unbiased score of each
// chosen expert is re-read from the (cached) score row.
#include "gate_fast.cuh"

namespace ep {

namespace {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;

template <int EPL>
__global__ void __launch_bounds__(kGateThreads, 1) gate_kernel(const float *__restrict__ scores,
                                                            const float *__restrict__ bias, int T,
                                                            GateParams p, int group_lanes, int vec_rows,
                                                            int32_t *__restrict__ topk_idx,
                                                            float *__restrict__ topk_w)
{
    extern __shared__ uint32_t gate_smem[];  // gate_warp_words<EPL>() per warp
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kGateWarps + warp;
    if (t >= T)
        return;  // the whole warp leaves together
    gate_token<EPL>(scores, bias, t, p, group_lanes, vec_rows, gate_smem + warp * gate_warp_words<EPL>(), topk_idx,
                    topk_w);
}

template <int EPL>
cudaError_t launch_epl(const float *scores, const float *bias, int T, const GateParams &p, int32_t *idx,
                       float *w, cudaStream_t st)
{
    int group_lanes, vec_rows, warp_floats;
    gate_plan<EPL>(p, scores, bias, group_lanes, vec_rows, warp_floats);
    const size_t smem = (size_t)kGateWarps * warp_floats * sizeof(float);
    const int grid = (T + kGateWarps - 1) / kGateWarps;
    gate_kernel<EPL><<<grid, kGateThreads, smem, st>>>(scores, bias, T, p, group_lanes, vec_rows, idx, w);
    return cudaGetLastError();
}

template <int EPL, int L, int Q>
cudaError_t launch_fast_q(const GateFastPlan &f, const float *scores, const float *bias, int T, const GateParams &p,
                          int32_t *idx, float *w, cudaStream_t st)
{
    GateFastArgs a{};
    a.scores = scores;
    a.bias = bias;
    a.T = T;
    a.p = p;
    a.m = f.m;
    a.q = f.q;
    a.topk_idx = idx;
    a.topk_w = w;
    a.cap = f.cap;
    const size_t smem = gate_fast_smem<EPL, L>(a.cap, p.k);
    const void *fn = (const void *)gate_fast_kernel<EPL, L, Q>;
    static PerDeviceCache<1> attr;  // the largest size any call can need (k = 32), once per device
    const cudaError_t e = raise_smem_limit(attr, fn, gate_fast_smem<EPL, L>(kGfCap, 32));
    if (e != cudaSuccess)
        return e;
    constexpr int TPC = kGfThreads / L;
    gate_fast_kernel<EPL, L, Q><<<(T + TPC - 1) / TPC, kGfThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int EPL, int L>
cudaError_t launch_fast_l(const GateFastPlan &f, const float *scores, const float *bias, int T, const GateParams &p,
                          int32_t *idx, float *w, cudaStream_t st)
{
    if (f.Q == 1)
        return launch_fast_q<EPL, L, 1>(f, scores, bias, T, p, idx, w, st);
    if (f.Q == 2)
        return launch_fast_q<EPL, L, 2>(f, scores, bias, T, p, idx, w, st);
    return launch_fast_q<EPL, L, 4>(f, scores, bias, T, p, idx, w, st);
}

cudaError_t launch_fast(const GateFastPlan &f, const float *scores, const float *bias, int T, const GateParams &p,
                        int32_t *idx, float *w, cudaStream_t st)
{
    switch (p.E) {
    case 8: return launch_fast_l<8, 1>(f, scores, bias, T, p, idx, w, st);
    case 16: return launch_fast_l<8, 2>(f, scores, bias, T, p, idx, w, st);
    case 32: return launch_fast_l<8, 4>(f, scores, bias, T, p, idx, w, st);
    case 64: return launch_fast_l<8, 8>(f, scores, bias, T, p, idx, w, st);
    case 128: return launch_fast_l<16, 8>(f, scores, bias, T, p, idx, w, st);
    default: return launch_fast_l<32, 8>(f, scores, bias, T, p, idx, w, st);
    }
}

}  // namespace

bool gate_fast_supported(const GateParams &p, const float *scores, const float *bias)
{
    GateFastPlan f;
    return gate_fast_plan(p, scores, bias, f);
}

// The lane-segment kernel serves group-limited gating of batches of 2048 or
// more tokens: measured on GB300 it is faster there (DeepSeek-V3 shape:
// 12.1 against 13.1 us cold, 8.3 against 10.4 us back to back).  Elsewhere
// the warp-per-token kernel measured as fast or faster: its shorter chains
// win on decode-sized batches (3.2 against 6.4 us back to back), and
// without groups it loses nothing to the lane segments' per-lane work.
bool use_gate_fast(const GateParams &p, int T, const float *scores, const float *bias)
{
    GateFastPlan f;
    return T >= 2048 && p.Kg < p.G && gate_fast_plan(p, scores, bias, f);
}

cudaError_t launch_gate(const float *scores, const float *bias, int T, const GateParams &p,
                        int32_t *topk_idx, float *topk_w, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    GateFastPlan f;
    if (use_gate_fast(p, T, scores, bias) && gate_fast_plan(p, scores, bias, f))
        return launch_fast(f, scores, bias, T, p, topk_idx, topk_w, st);
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
