// dispatch.cu -- step 3: permute-scatter of token rows into the receive
// buffer, BF16 copy, FP8 e4m3 with one fp32 scale per 128 columns, or MXFP8
// (e4m3 with one power-of-two E8M0 scale per 32 columns).
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all", Phase 1 Dispatch: each token goes to the
// holders of its chosen experts.  "DeepEP de DeepSeek ...", section "Support
// FP8 et MXFP8": an FP8 payload halves the bytes against BF16.
//
// HBM-bound: every source row is read once and written k times (BF16: 2H
// bytes in, 2Hk out; FP8: 2H in, k(H + H/32) out).  Work is split into warp
// items -- one token's row segment of 32 lanes x 16 bytes (x U) -- handed out
// grid-stride to a persistent grid of (resident CTAs per SM) x (SMs).  There
// is no block barrier: lane j of the warp holds the token's j-th receive row
// (and lane j of a second register slot j+32) and shuffles it to the others,
// so every warp streams independently.  Loads bypass L1; stores are plain.
// The row is held in registers and never re-read per copy.
// FP8: 8 consecutive lanes own one 128-column block (16 columns each); the
// block's amax is a 3-step xor-shuffle max, the scale an IEEE fp32 division
// by 448, each code an IEEE fp32 division then a round-to-nearest-even
// saturating e4m3 conversion (cvt.rn.satfinite).
#include "dispatch_impl.cuh"

namespace ep {

namespace {

constexpr int kDispThreads = 256;

__global__ void __launch_bounds__(kDispThreads) dispatch_bf16_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                     int k, const int32_t *__restrict__ pos,
                                                                     uint16_t *__restrict__ recv, long long rows,
                                                                     int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    for (ItemWalk it(T, bf16_segs(H)); it.valid(); it.next()) {
        int p0, p1;
        token_rows(pos, it.t, k, rows, lane, err_flag, p0, p1);
        dispatch_bf16_item(x, H, k, it.t, it.seg, p0, p1, recv);
    }
}

__global__ void __launch_bounds__(kDispThreads) dispatch_fp8_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                    int k, const int32_t *__restrict__ pos,
                                                                    uint8_t *__restrict__ recv_q,
                                                                    float *__restrict__ recv_s, long long rows,
                                                                    int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    for (ItemWalk it(T, fp8_segs(H)); it.valid(); it.next()) {
        int p0, p1;
        token_rows(pos, it.t, k, rows, lane, err_flag, p0, p1);
        dispatch_fp8_item(x, H, k, it.t, it.seg, p0, p1, recv_q, recv_s);
    }
}

// MXFP8 (OCP Microscaling v1.0, E4M3 elements): a 32-column block is two
// lanes of 16 columns.  Its scale is 2^e, e = floor(log2(amax)) - 8 (the
// exponent of 448) clamped to [-127, 127] and stored as the E8M0 byte e + 127
// (amax = 0 gives e = -127).  x * 2^-e is exact in fp32 (a power-of-two
// product; only values far below the smallest e4m3 subnormal can round, and
// they code to a signed zero either way), then cvt.rn.satfinite to e4m3.
__global__ void __launch_bounds__(kDispThreads) dispatch_mxfp8_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                      int k, const int32_t *__restrict__ pos,
                                                                      uint8_t *__restrict__ recv_q,
                                                                      uint8_t *__restrict__ recv_e, long long rows,
                                                                      int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    for (ItemWalk it(T, fp8_segs(H)); it.valid(); it.next()) {
        int p0, p1;
        token_rows(pos, it.t, k, rows, lane, err_flag, p0, p1);
        dispatch_mxfp8_item(x, H, k, it.t, it.seg, p0, p1, recv_q, recv_e);
    }
}

// A persistent grid of (resident CTAs per SM) x (SMs), capped by the work.
int persistent_grid(const void *kernel, int &per_sm_cache, long long warp_items)
{
    if (per_sm_cache < 1) {
        int per_sm = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kDispThreads, 0);
        per_sm_cache = per_sm < 1 ? 1 : per_sm;
    }
    const long long g = (long long)device_sm_count() * per_sm_cache;
    const long long need = (warp_items + kDispThreads / 32 - 1) / (kDispThreads / 32);
    return (int)(need < g ? need : g);
}

int g_bf16_per_sm = 0;
int g_fp8_per_sm = 0;
int g_mx_per_sm = 0;

}  // namespace

cudaError_t launch_dispatch_mxfp8(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint8_t *recv_q,
                                  uint8_t *recv_e, long long rows, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    const long long items = (long long)T * fp8_segs(H);
    const int grid = persistent_grid((const void *)dispatch_mxfp8_kernel, g_mx_per_sm, items);
    dispatch_mxfp8_kernel<<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_e, rows, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_bf16(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint16_t *recv,
                                 long long rows, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    const long long items = (long long)T * bf16_segs(H);
    const int grid = persistent_grid((const void *)dispatch_bf16_kernel, g_bf16_per_sm, items);
    dispatch_bf16_kernel<<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv, rows, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint8_t *recv_q,
                                float *recv_s, long long rows, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    const long long items = (long long)T * fp8_segs(H);
    const int grid = persistent_grid((const void *)dispatch_fp8_kernel, g_fp8_per_sm, items);
    dispatch_fp8_kernel<<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_s, rows, err_flag);
    return cudaGetLastError();
}

}  // namespace ep
