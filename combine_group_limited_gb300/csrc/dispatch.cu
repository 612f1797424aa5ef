// dispatch.cu -- step 3: permute-scatter of token rows into the receive
// buffer, BF16 copy or FP8 e4m3 with one fp32 scale per 128 columns.
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all", Phase 1 Dispatch: each token goes to the
// holders of its chosen experts.  "DeepEP de DeepSeek ...", section "Support
// FP8 et MXFP8": an FP8 payload halves the bytes against BF16.
//
// HBM-bound: every source row is read once and written k times (BF16: 2H
// bytes in, 2Hk out; FP8: 2H in, k(H + H/32) out).  A CTA takes one token at
// a time; its threads cover the row in 16-byte chunks with streaming loads,
// hold them in registers and issue the k stores (the row is never re-read
// per copy).  FP8: 8 consecutive lanes own one 128-column block (16 columns
// each); the block's amax is a 3-step xor-shuffle max, the scale an IEEE
// fp32 division by 448, each code an IEEE fp32 division then a
// round-to-nearest-even saturating e4m3 conversion (cvt.rn.satfinite).
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kDispThreads = 256;
constexpr int kMaxK = 64;
constexpr int kBf16Unroll = 4;

// Loads the token's k receive rows into shared memory; bad rows are dropped
// and flagged.  Ends with a block barrier.
__device__ __forceinline__ void load_rows(const int32_t *__restrict__ pos, int t, int k, long long rows,
                                          int32_t *s_pos, int32_t *err_flag)
{
    __syncthreads();  // the previous token's readers are done
    if (threadIdx.x < k) {
        int p = __ldg(pos + (size_t)t * k + threadIdx.x);
        if (p >= rows) {
            if (err_flag)
                atomicOr(err_flag, 2);
            p = -1;
        }
        s_pos[threadIdx.x] = p;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kDispThreads) dispatch_bf16_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                     int k, const int32_t *__restrict__ pos,
                                                                     uint16_t *__restrict__ recv,
                                                                     int32_t *__restrict__ err_flag)
{
    __shared__ int32_t s_pos[kMaxK];
    const int C = H / 8;  // 16-byte chunks per row
    const long long rows = (long long)T * k;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        load_rows(pos, t, k, rows, s_pos, err_flag);
        const uint16_t *xrow = x + (size_t)t * H;
        for (int c0 = threadIdx.x; c0 < C; c0 += kDispThreads * kBf16Unroll) {
            uint4 v[kBf16Unroll];
#pragma unroll
            for (int u = 0; u < kBf16Unroll; ++u) {
                const int c = c0 + u * kDispThreads;
                if (c < C)
                    v[u] = ld_stream16(xrow + (size_t)c * 8);
            }
            for (int j = 0; j < k; ++j) {
                const int p = s_pos[j];
                if (p < 0)
                    continue;
                uint16_t *dst = recv + (size_t)p * H;
#pragma unroll
                for (int u = 0; u < kBf16Unroll; ++u) {
                    const int c = c0 + u * kDispThreads;
                    if (c < C)
                        st_stream16(dst + (size_t)c * 8, v[u]);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kDispThreads) dispatch_fp8_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                    int k, const int32_t *__restrict__ pos,
                                                                    uint8_t *__restrict__ recv_q,
                                                                    float *__restrict__ recv_s,
                                                                    int32_t *__restrict__ err_flag)
{
    __shared__ int32_t s_pos[kMaxK];
    const int C16 = H / 16;    // 16-column groups per row; 8 per 128-column block
    const int nb = H / 128;    // scales per row
    const long long rows = (long long)T * k;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        load_rows(pos, t, k, rows, s_pos, err_flag);
        const uint16_t *xrow = x + (size_t)t * H;
        // The trip count is the same for every thread, so whole 8-lane
        // groups are active or idle together and the shuffles see all lanes.
        for (int base = 0; base < C16; base += kDispThreads) {
            const int c = base + threadIdx.x;
            const bool act = c < C16;
            uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
            if (act) {
                a = ld_stream16(xrow + (size_t)c * 16);
                b = ld_stream16(xrow + (size_t)c * 16 + 8);
            }
            const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float f[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                f[2 * i] = bf16_lo(wv[i]);
                f[2 * i + 1] = bf16_hi(wv[i]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                amax = fmaxf(amax, fabsf(f[i]));
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
            const float s = __fdiv_rn(amax, 448.0f);
            uint32_t q[4];
            if (amax == 0.0f) {
                // all zeros: keep each element's sign bit (bf16 bit 15 -> code bit 7)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t w0 = wv[2 * i], w1 = wv[2 * i + 1];
                    q[i] = ((w0 >> 8) & 0x80u) | ((w0 >> 16) & 0x8000u) | ((w1 << 8) & 0x800000u) |
                           (w1 & 0x80000000u);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t lo = pack_e4m3x2(__fdiv_rn(f[4 * i], s), __fdiv_rn(f[4 * i + 1], s));
                    const uint32_t hi = pack_e4m3x2(__fdiv_rn(f[4 * i + 2], s), __fdiv_rn(f[4 * i + 3], s));
                    q[i] = lo | (hi << 16);
                }
            }
            if (act) {
                const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                for (int j = 0; j < k; ++j) {
                    const int p = s_pos[j];
                    if (p < 0)
                        continue;
                    st_stream16(recv_q + (size_t)p * H + (size_t)c * 16, qv);
                    if ((c & 7) == 0)
                        recv_s[(size_t)p * nb + (c >> 3)] = s;
                }
            }
        }
    }
}

// A grid of (resident CTAs per SM) x (SMs), capped at one CTA per token.
int dispatch_grid(const void *kernel, int &per_sm_cache, int T)
{
    if (per_sm_cache < 1) {
        int per_sm = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kDispThreads, 0);
        per_sm_cache = per_sm < 1 ? 1 : per_sm;
    }
    const int g = device_sm_count() * per_sm_cache;
    return T < g ? T : g;
}

int g_bf16_per_sm = 0;
int g_fp8_per_sm = 0;

}  // namespace

cudaError_t launch_dispatch_bf16(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint16_t *recv,
                                 int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    const int grid = dispatch_grid((const void *)dispatch_bf16_kernel, g_bf16_per_sm, T);
    dispatch_bf16_kernel<<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint8_t *recv_q,
                                float *recv_s, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    const int grid = dispatch_grid((const void *)dispatch_fp8_kernel, g_fp8_per_sm, T);
    dispatch_fp8_kernel<<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_s, err_flag);
    return cudaGetLastError();
}

}  // namespace ep
