// combine.cu -- steps 4 and 5: inverse gather and router-weighted combine.
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all", Phase 2 Combine: each token's expert outputs
// come back to it and are summed weighted by the router scores.
//
// out[t, h] = bf16_rne(fma(w[t,k-1], y[pos[t,k-1], h], ... fma(w[t,0],
// y[pos[t,0], h], 0.0f))): an fp32 fma chain in slot order, so the result
// does not depend on the launch shape.  The gather is never materialised:
// pos (token-major) names the k rows to read.  HBM-bound: 2Hk bytes in and
// 2H out per token.  A CTA takes one token at a time; a thread owns a
// 16-byte column chunk and first issues the loads of up to 8 slots, then
// runs their fmas in order, so eight 16-byte loads are in flight per thread.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kCombThreads = 256;
constexpr int kMaxK = 64;
constexpr int kSlotBatch = 8;

__global__ void __launch_bounds__(kCombThreads) combine_kernel(const uint16_t *__restrict__ y,
                                                               const int32_t *__restrict__ pos,
                                                               const float *__restrict__ w, int T, int H, int k,
                                                               uint16_t *__restrict__ out,
                                                               int32_t *__restrict__ err_flag)
{
    __shared__ int32_t s_pos[kMaxK];
    __shared__ float s_w[kMaxK];
    const int C = H / 8;
    const long long rows = (long long)T * k;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();
        if (threadIdx.x < k) {
            int p = __ldg(pos + (size_t)t * k + threadIdx.x);
            if (p >= rows) {
                if (err_flag)
                    atomicOr(err_flag, 2);
                p = -1;
            }
            s_pos[threadIdx.x] = p;
            s_w[threadIdx.x] = __ldg(w + (size_t)t * k + threadIdx.x);
        }
        __syncthreads();
        for (int c = threadIdx.x; c < C; c += kCombThreads) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[i] = 0.0f;
            for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
                uint4 v[kSlotBatch];
#pragma unroll
                for (int u = 0; u < kSlotBatch; ++u) {
                    const int j = j0 + u;
                    const int p = j < k ? s_pos[j] : -1;
                    if (p >= 0)
                        v[u] = ld_stream16(y + (size_t)p * H + (size_t)c * 8);
                }
#pragma unroll
                for (int u = 0; u < kSlotBatch; ++u) {
                    const int j = j0 + u;
                    const int p = j < k ? s_pos[j] : -1;
                    if (p >= 0) {
                        const float wj = s_w[j];
                        const uint32_t vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc[2 * i] = fmaf(wj, bf16_lo(vv[i]), acc[2 * i]);
                            acc[2 * i + 1] = fmaf(wj, bf16_hi(vv[i]), acc[2 * i + 1]);
                        }
                    }
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            st_stream16(out + (size_t)t * H + (size_t)c * 8, o);
        }
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t *y, const int32_t *pos, const float *w, int T, int H, int k,
                           uint16_t *out, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    static int per_sm = 0;
    if (per_sm < 1) {
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void *)combine_kernel, kCombThreads, 0);
        if (per_sm < 1)
            per_sm = 1;
    }
    int grid = device_sm_count() * per_sm;
    if (grid > T)
        grid = T;
    combine_kernel<<<grid, kCombThreads, 0, st>>>(y, pos, w, T, H, k, out, err_flag);
    return cudaGetLastError();
}

}  // namespace ep
