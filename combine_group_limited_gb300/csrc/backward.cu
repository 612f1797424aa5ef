// backward.cu -- backward of the weighted combine.
//
// The combine of "Expert Parallelism (Parallelisme d'experts)", section "Le
// pattern de communication all-to-all" (Phase 2: the expert outputs come back
// and are summed weighted by the router scores) is out[t] = sum_j w[t,j] *
// y[pos[t,j]].  Its gradients, for training (the setting of "DeepEP de
// DeepSeek ...": forward and backward passes), are
//   grad_y[pos[t,j], :] = w[t,j] * grad_out[t, :]        (a weighted dispatch)
//   grad_w[t, j]        = <grad_out[t, :], y[pos[t,j], :]>
// (The backward of the BF16 dispatch is the combine with unit weights; see
// combine.cu.)
//
// One CTA per token at a time (at k <= 2 on large batches, one warp per
// token instead: combine_backward_warp_kernel): each thread owns 16-byte
// column chunks; per
// chunk it reads grad_out once and the k expert rows, writes the k scaled
// rows, and keeps k partial dot products.  grad_y is rounded once to bf16:
// the fp32 product p = w*g is corrected with its exact residual
// fma(w, g, -p) (the FMA-based TwoProduct of Ogita, Rump and Oishi,
// "Accurate sum and dot product", SIAM J. Sci. Comput. 2005) whenever p sits
// exactly on a bf16 rounding midpoint, so the result is the correctly rounded
// bf16 of the exact product (for products in the normal fp32 range).  The
// dots are reduced in a fixed order (each thread's chunks in sequence, a warp
// xor-tree, then the warps in order), so grad_w does not depend on timing.
// As in the combine, the next token's rows and weights are fetched while
// one is processed, and the block size spreads a row evenly over the warps
// (the reduction order then depends on H, never on timing).
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kMaxK = 64;
constexpr int kSlotBatch = 8;

// bf16 nearest-even of the exact product w*g (see the file comment).
__device__ __forceinline__ float exact_product_for_bf16(float w, float g)
{
    float p = w * g;
    const float e = fmaf(w, g, -p);
    uint32_t u = __float_as_uint(p);
    if ((u & 0xFFFFu) == 0x8000u && e != 0.0f) {
        // p is a bf16 midpoint but the true product is not: step one fp32 ulp
        // toward the true product so that rounding picks its side.
        const bool away = (e > 0.0f) == (p > 0.0f);
        u = away ? u + 1u : u - 1u;
        p = __uint_as_float(u);
    }
    return p;
}

__global__ void __launch_bounds__(kBwdThreads, 3) combine_backward_kernel(
    const uint16_t *__restrict__ grad_out, const uint16_t *__restrict__ y, const int32_t *__restrict__ pos,
    const float *__restrict__ w, int T, int H, int k, uint16_t *__restrict__ grad_y, float *__restrict__ grad_w,
    long long rows, int32_t *__restrict__ err_flag)
{
    __shared__ int32_t s_pos[kMaxK];
    __shared__ float s_w[kMaxK];
    __shared__ float s_part[kSlotBatch][kBwdWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int C = H / 8;
    const bool loader = threadIdx.x < k;
    int np = -1;
    float nw = 0.0f;
    if (loader && blockIdx.x < T) {
        np = __ldg(pos + (size_t)blockIdx.x * k + threadIdx.x);
        nw = __ldg(w + (size_t)blockIdx.x * k + threadIdx.x);
    }
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();
        if (loader) {
            int p = np;
            if (p >= rows) {
                if (err_flag)
                    atomicOr(err_flag, 2);
                p = -1;
            }
            s_pos[threadIdx.x] = p;
            s_w[threadIdx.x] = nw;
        }
        __syncthreads();
        const int tn = t + gridDim.x;  // prefetch the next token's rows and weights
        if (loader && tn < T) {
            np = __ldg(pos + (size_t)tn * k + threadIdx.x);
            nw = __ldg(w + (size_t)tn * k + threadIdx.x);
        }
        const uint16_t *grow = grad_out + (size_t)t * H;
        for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
            float dot[kSlotBatch];
#pragma unroll
            for (int u = 0; u < kSlotBatch; ++u)
                dot[u] = 0.0f;
            for (int c = threadIdx.x; c < C; c += blockDim.x) {
                const uint4 gv = ld_stream16(grow + (size_t)c * 8);
                const uint32_t gw4[4] = {gv.x, gv.y, gv.z, gv.w};
                float g[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    g[2 * i] = bf16_lo(gw4[i]);
                    g[2 * i + 1] = bf16_hi(gw4[i]);
                }
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
                    if (p < 0)
                        continue;
                    const float wj = s_w[j];
                    const uint32_t yv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        dot[u] = fmaf(g[2 * i], bf16_lo(yv[i]), dot[u]);
                        dot[u] = fmaf(g[2 * i + 1], bf16_hi(yv[i]), dot[u]);
                    }
                    // Products; a bf16 rounding midpoint among them (low 16
                    // bits 0x8000, about one in 2^16) takes the exact path.
                    float pr[8];
                    uint32_t mid = 0xFFFFu;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        pr[i] = wj * g[i];
                        mid = min(mid, (__float_as_uint(pr[i]) & 0xFFFFu) ^ 0x8000u);
                    }
                    if (mid == 0u) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            pr[i] = exact_product_for_bf16(wj, g[i]);
                    }
                    uint4 o;
                    o.x = pack_bf16x2(pr[0], pr[1]);
                    o.y = pack_bf16x2(pr[2], pr[3]);
                    o.z = pack_bf16x2(pr[4], pr[5]);
                    o.w = pack_bf16x2(pr[6], pr[7]);
                    st_plain16(grad_y + (size_t)p * H + (size_t)c * 8, o);
                }
            }
            // Fixed-order reduction of the batch's dots.
#pragma unroll
            for (int u = 0; u < kSlotBatch; ++u) {
                float d = dot[u];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    d += __shfl_xor_sync(kFullMask, d, off);
                if (lane == 0)
                    s_part[u][warp] = d;
            }
            __syncthreads();
            if (threadIdx.x < kSlotBatch && j0 + threadIdx.x < k) {
                const int j = j0 + threadIdx.x;
                float d = 0.0f;
                for (int wi = 0; wi < nwarps; ++wi)
                    d += s_part[threadIdx.x][wi];
                grad_w[(size_t)t * k + j] = s_pos[j] >= 0 ? d : 0.0f;
            }
            __syncthreads();
        }
    }
}

// grad_y of one 16-byte chunk for one slot: the 8 products w * g rounded
// once to bf16 (midpoints among them take the exact path, as in
// combine_backward_kernel), and the slot's dot product advanced by the chunk.
__device__ __forceinline__ uint4 backward_chunk(float wj, const float (&g)[8], const uint4 &yv4, float &dot)
{
    const uint32_t yv[4] = {yv4.x, yv4.y, yv4.z, yv4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dot = fmaf(g[2 * i], bf16_lo(yv[i]), dot);
        dot = fmaf(g[2 * i + 1], bf16_hi(yv[i]), dot);
    }
    float pr[8];
    uint32_t mid = 0xFFFFu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        pr[i] = wj * g[i];
        mid = min(mid, (__float_as_uint(pr[i]) & 0xFFFFu) ^ 0x8000u);
    }
    if (mid == 0u) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            pr[i] = exact_product_for_bf16(wj, g[i]);
    }
    uint4 o;
    o.x = pack_bf16x2(pr[0], pr[1]);
    o.y = pack_bf16x2(pr[2], pr[3]);
    o.z = pack_bf16x2(pr[4], pr[5]);
    o.w = pack_bf16x2(pr[6], pr[7]);
    return o;
}

// k <= 2 on large batches: one warp per token and no block barriers.  A
// CTA-per-token pass pays a memory round trip and four barriers per token,
// which at two slots is most of the token's time.  Each lane takes
// kBwdWarpChunks 16-byte chunks at once (grad_out and both slots' rows
// loaded before any arithmetic), and the next token's rows and weights are
// fetched while one is processed.  Each lane's dots run over its chunks in
// order and are then summed by a warp xor-tree: a fixed order, so grad_w
// does not depend on timing.  Blocks of 4 warps at up to 64 registers keep
// 32 warps on an SM.
constexpr int kBwdWarpThreads = 128;
constexpr int kBwdWarpChunks = 2;

__global__ void __launch_bounds__(kBwdWarpThreads, 8) combine_backward_warp_kernel(
    const uint16_t *__restrict__ grad_out, const uint16_t *__restrict__ y, const int32_t *__restrict__ pos,
    const float *__restrict__ w, int T, int H, int k, uint16_t *__restrict__ grad_y, float *__restrict__ grad_w,
    long long rows, int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    const int warp = (int)balanced_warp();  // grid <= T blocks
    const int nwarps = (int)grid_warps();
    const int C = H / 8;
    int np = -1;
    float nw = 0.0f;
    if (warp < T && lane < k) {
        np = __ldg(pos + (size_t)warp * k + lane);
        nw = __ldg(w + (size_t)warp * k + lane);
    }
    for (int t = warp; t < T; t += nwarps) {
        int p = np;
        if (lane < k && p >= rows) {
            if (err_flag)
                atomicOr(err_flag, 2);
            p = -1;
        }
        const int p0 = __shfl_sync(kFullMask, p, 0), p1 = __shfl_sync(kFullMask, p, 1);
        const float w0 = __shfl_sync(kFullMask, nw, 0), w1 = __shfl_sync(kFullMask, nw, 1);
        const int q1 = k > 1 ? p1 : -1;
        const int tn = t + nwarps;  // < 2T: no overflow
        if (tn < T && lane < k) {
            np = __ldg(pos + (size_t)tn * k + lane);
            nw = __ldg(w + (size_t)tn * k + lane);
        }
        const uint16_t *grow = grad_out + (size_t)t * H;
        float d0 = 0.0f, d1 = 0.0f;
        for (int c0 = lane; c0 < C; c0 += 32 * kBwdWarpChunks) {
            uint4 gv[kBwdWarpChunks], v0[kBwdWarpChunks], v1[kBwdWarpChunks];
#pragma unroll
            for (int m = 0; m < kBwdWarpChunks; ++m) {
                const int c = c0 + 32 * m;
                if (c >= C)
                    continue;
                gv[m] = ld_stream16(grow + (size_t)c * 8);
                if (p0 >= 0)
                    v0[m] = ld_stream16(y + (size_t)p0 * H + (size_t)c * 8);
                if (q1 >= 0)
                    v1[m] = ld_stream16(y + (size_t)q1 * H + (size_t)c * 8);
            }
#pragma unroll
            for (int m = 0; m < kBwdWarpChunks; ++m) {
                const int c = c0 + 32 * m;
                if (c >= C)
                    continue;
                const uint32_t gw4[4] = {gv[m].x, gv[m].y, gv[m].z, gv[m].w};
                float g[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    g[2 * i] = bf16_lo(gw4[i]);
                    g[2 * i + 1] = bf16_hi(gw4[i]);
                }
                if (p0 >= 0)
                    st_plain16(grad_y + (size_t)p0 * H + (size_t)c * 8, backward_chunk(w0, g, v0[m], d0));
                if (q1 >= 0)
                    st_plain16(grad_y + (size_t)q1 * H + (size_t)c * 8, backward_chunk(w1, g, v1[m], d1));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            d0 += __shfl_xor_sync(kFullMask, d0, off);
            d1 += __shfl_xor_sync(kFullMask, d1, off);
        }
        if (lane == 0)
            grad_w[(size_t)t * k] = p0 >= 0 ? d0 : 0.0f;
        if (lane == 1 && k > 1)
            grad_w[(size_t)t * k + 1] = q1 >= 0 ? d1 : 0.0f;
    }
}

}  // namespace

cudaError_t launch_combine_backward(const uint16_t *grad_out, const uint16_t *y, long long rows, const int32_t *pos,
                                    const float *w, int T, int H, int k, uint16_t *grad_y, float *grad_w,
                                    int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    if (k <= 2 && T >= 2048) {
        static PerDeviceCache<1> occ;
        const int per_sm = occupancy_per_sm(occ, (const void *)combine_backward_warp_kernel, kBwdWarpThreads, 0);
        long long g = (long long)device_sm_count() * per_sm;  // one token per CTA at least (balanced_warp)
        if (g > T)
            g = T;
        combine_backward_warp_kernel<<<(int)g, kBwdWarpThreads, 0, st>>>(grad_out, y, pos, w, T, H, k, grad_y,
                                                                          grad_w, rows, err_flag);
        return cudaGetLastError();
    }
    const int threads = chunk_threads(H / 8, k);  // <= kBwdThreads (k <= 64)
    static PerDeviceCache<33> occ;
    const int grid = row_grid((const void *)combine_backward_kernel, threads, T, occ);
    combine_backward_kernel<<<grid, threads, 0, st>>>(grad_out, y, pos, w, T, H, k, grad_y, grad_w, rows,
                                                      err_flag);
    return cudaGetLastError();
}

}  // namespace ep
