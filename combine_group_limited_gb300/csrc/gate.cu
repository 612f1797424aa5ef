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
#include "gate_impl.cuh"

namespace ep {

namespace {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;

template <int EPL>
__global__ void __launch_bounds__(kGateThreads) gate_kernel(const float *__restrict__ scores,
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
