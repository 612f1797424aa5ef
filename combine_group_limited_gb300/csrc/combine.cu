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
// runs their fmas in order, so eight 16-byte loads are in flight per thread;
// the next token's rows and weights are fetched while one is summed.
// With w == NULL every weight is 1: the backward of the BF16 dispatch (a
// copy), whose source-row gradient is the sum of its copies' gradients.
//
// combine_fp8_kernel: the same reduction over FP8 expert outputs (e4m3 codes
// with fp32 1x128 or E8M0 1x32 block scales).  A code converts exactly to
// fp32 (cvt.rn.f16x2.e4m3x2, then f16 -> f32); the slot's weight times its
// block scale is formed once (exact for E8M0 powers of two, one fp32
// rounding for fp32 scales) and the codes enter the same fp32 fma chain in
// slot order.  2 bytes of FP8 payload per column per slot
// instead of 2 bytes of BF16 halves the bytes the combine reads.
#include <cuda_fp16.h>

#include "coop.cuh"

namespace ep {

namespace {

constexpr int kCombThreads = 256;
constexpr int kMaxK = 64;
constexpr int kSlotBatch = 8;

}  // namespace

// Threads per CTA for a row of c column chunks and k slots: the fewest
// passes of at most kCombThreads threads, spread evenly over whole warps
// (H = 7168: 896 BF16 chunks = 4 passes of 224, not 3.5 passes of 256), and
// never fewer threads than slots (thread j < k loads slot j's row and
// weight).
int chunk_threads(int c, int k)
{
    const int passes = (c + kCombThreads - 1) / kCombThreads;
    const int per_pass = (c + passes - 1) / passes;
    const int t = ((per_pass + 31) / 32) * 32;
    const int tk = ((k + 31) / 32) * 32;
    return t > tk ? t : tk;
}

// Column segments per token for the CTA-per-row kernels: a batch too small
// to give every resident CTA a token (decode-sized) splits each row into S
// segments of at least half a pass of kCombThreads chunks, so more CTAs
// share the rows and each runs fewer dependent passes.
int column_segments(int T, int chunks, int resident)
{
    if (T <= 0 || T >= resident)
        return 1;
    int S = (resident + T - 1) / T;
    const int most = chunks / (kCombThreads / 2);
    if (S > most)
        S = most;
    return S < 1 ? 1 : S;
}

// A persistent grid of every resident CTA of the kernel at this block size
// (at most one per row); the occupancy is cached per device and per block
// size (a multiple of 32, at most 1024).
int row_grid(const void *kern, int threads, int T, PerDeviceCache<33> &cache)
{
    const int per_sm = occupancy_per_sm(cache, kern, threads, 0, threads / 32);
    const long long g = (long long)device_sm_count() * per_sm;
    return (int)(g < T ? g : T);
}

namespace {

template <bool kSplit>  // false: S == 1 (one item per token, no division per item)
__global__ void __launch_bounds__(kCombThreads) combine_kernel(const uint16_t *__restrict__ y,
                                                               const int32_t *__restrict__ pos,
                                                               const float *__restrict__ w, int T, int H, int k,
                                                               uint16_t *__restrict__ out, long long rows,
                                                               int32_t *__restrict__ err_flag, int S)
{
    __shared__ int32_t s_pos[kMaxK];
    __shared__ float s_w[kMaxK];
    const int C = H / 8;
    const long long items = (long long)T * S;  // (token, column segment) pairs
    const bool loader = threadIdx.x < k;        // k <= 64 < blockDim.x
    int np = -1;
    float nw = 0.0f;
    if (loader && blockIdx.x < items) {
        const long long t0 = kSplit ? blockIdx.x / S : blockIdx.x;
        np = __ldg(pos + t0 * k + threadIdx.x);
        nw = w ? __ldg(w + t0 * k + threadIdx.x) : 1.0f;
    }
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const long long t = kSplit ? it / S : it;
        const int seg = kSplit ? (int)(it - t * S) : 0;
        const int c_lo = kSplit ? (int)((long long)C * seg / S) : 0;
        const int c_hi = kSplit ? (int)((long long)C * (seg + 1) / S) : C;
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
        const long long itn = it + gridDim.x;  // the next item's rows and weights load while this one is summed
        if (loader && itn < items) {
            const long long tn = kSplit ? itn / S : itn;
            np = __ldg(pos + tn * k + threadIdx.x);
            nw = w ? __ldg(w + tn * k + threadIdx.x) : 1.0f;
        }
        for (int c = c_lo + threadIdx.x; c < c_hi; c += kCombThreads) {
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

__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float &a, float &b, float &c, float &d)
{
    uint32_t h0, h1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    const __half2 p0 = *reinterpret_cast<const __half2 *>(&h0);
    const __half2 p1 = *reinterpret_cast<const __half2 *>(&h1);
    a = __low2float(p0);
    b = __high2float(p0);
    c = __low2float(p1);
    d = __high2float(p1);
}

// E8M0 byte -> 2^(byte - 127) as fp32 (byte 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b)
{
    return b == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// acc (16 columns as 8 packed fp32x2 pairs) += ws * decode(16 codes): the
// fp32 fma chain of every column, two columns per packed instruction.
__device__ __forceinline__ void fma_codes16(uint64_t ws2, const uint4 &v, uint64_t (&acc)[8])
{
    const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float d0, d1, d2, d3;
        e4m3x4_to_f32(vv[i], d0, d1, d2, d3);
        acc[2 * i] = f2_fma(ws2, f2_pack(d0, d1), acc[2 * i]);
        acc[2 * i + 1] = f2_fma(ws2, f2_pack(d2, d3), acc[2 * i + 1]);
    }
}

// The 16 accumulated columns rounded to bf16 as two 16-byte words.
__device__ __forceinline__ void pack_acc16(const uint64_t (&acc)[8], uint4 &o0, uint4 &o1)
{
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float lo, hi;
        f2_unpack(acc[i], lo, hi);
        w[i] = pack_bf16x2(lo, hi);
    }
    o0 = make_uint4(w[0], w[1], w[2], w[3]);
    o1 = make_uint4(w[4], w[5], w[6], w[7]);
}

// kMx: scales are E8M0 bytes per 32 columns; else fp32 per 128 columns.
// Slots are summed kFp8SlotBatch at a time (all loads of a batch issued
// before its conversions), and the kernel is held to five CTAs per SM: the
// decode arithmetic per byte is about twice the BF16 combine's, and more
// resident warps overlap it with the loads better than more loads in flight
// per thread.  DSV3 shape (ncu, L2 flushed): 96.3 us against 102.7 us with
// batches of 8 slots at three CTAs per SM, 98.5 us at four CTAs per SM.
constexpr int kFp8SlotBatch = 4;

template <bool kMx, bool kSplit>
__global__ void __launch_bounds__(kCombThreads, 5) combine_fp8_kernel(const uint8_t *__restrict__ yq,
                                                                   const void *__restrict__ yscale,
                                                                   const int32_t *__restrict__ pos,
                                                                   const float *__restrict__ w, int T, int H, int k,
                                                                   uint16_t *__restrict__ out, long long rows,
                                                                   int32_t *__restrict__ err_flag, int S)
{
    __shared__ int32_t s_pos[kMaxK];
    __shared__ float s_w[kMaxK];
    const int C16 = H / 16;
    const int nb = kMx ? H / 32 : H / 128;
    const long long items = (long long)T * S;  // (token, column segment) pairs
    const bool loader = threadIdx.x < k;        // k <= 64 < blockDim.x
    int np = -1;
    float nw = 0.0f;
    if (loader && blockIdx.x < items) {
        const long long t0 = kSplit ? blockIdx.x / S : blockIdx.x;
        np = __ldg(pos + t0 * k + threadIdx.x);
        nw = __ldg(w + t0 * k + threadIdx.x);
    }
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const long long t = kSplit ? it / S : it;
        const int seg = kSplit ? (int)(it - t * S) : 0;
        const int c_lo = kSplit ? (int)((long long)C16 * seg / S) : 0;
        const int c_hi = kSplit ? (int)((long long)C16 * (seg + 1) / S) : C16;
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
        const long long itn = it + gridDim.x;  // the next item's rows and weights load while this one is summed
        if (loader && itn < items) {
            const long long tn = kSplit ? itn / S : itn;
            np = __ldg(pos + tn * k + threadIdx.x);
            nw = __ldg(w + tn * k + threadIdx.x);
        }
        for (int c = c_lo + threadIdx.x; c < c_hi; c += kCombThreads) {
            uint64_t acc[8];  // column pairs, packed fp32x2
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[i] = 0ull;
            const int sb = kMx ? (c >> 1) : (c >> 3);  // this lane's scale block
            for (int j0 = 0; j0 < k; j0 += kFp8SlotBatch) {
                // First issue every load of the batch (codes and raw scale
                // words), then convert: no load waits behind a conversion.
                uint4 v[kFp8SlotBatch];
                uint32_t sraw[kFp8SlotBatch];
#pragma unroll
                for (int u = 0; u < kFp8SlotBatch; ++u) {
                    const int j = j0 + u;
                    const int p = j < k ? s_pos[j] : -1;
                    if (p >= 0) {
                        v[u] = ld_stream16(yq + (size_t)p * H + (size_t)c * 16);
                        sraw[u] = kMx ? (uint32_t)__ldg(static_cast<const uint8_t *>(yscale) + (size_t)p * nb + sb)
                                      : __float_as_uint(__ldg(static_cast<const float *>(yscale) + (size_t)p * nb + sb));
                    }
                }
#pragma unroll
                for (int u = 0; u < kFp8SlotBatch; ++u) {
                    const int j = j0 + u;
                    const int p = j < k ? s_pos[j] : -1;
                    if (p >= 0) {
                        // weight times block scale once per slot: one fp32
                        // rounding per term, as scaling each code would be
                        const float sc = kMx ? e8m0_to_f32(sraw[u]) : __uint_as_float(sraw[u]);
                        const float ws = s_w[j] * sc;
                        fma_codes16(f2_pack(ws, ws), v[u], acc);
                    }
                }
            }
            uint4 o0, o1;
            pack_acc16(acc, o0, o1);
            uint16_t *dst = out + (size_t)t * H + (size_t)c * 16;
            st_stream16(dst, o0);
            st_stream16(dst + 8, o1);
        }
    }
}

// Decode-sized batches (flat_sized below): one thread per column chunk
// of one token (8 BF16 columns, or 16 FP8 codes), with no
// shared memory and no block barrier.  Each thread reads its token's rows
// and weights itself (the lanes of a warp read the same words, one request)
// and then its chunk of up to 8 slots at once, so a call is two dependent
// memory round trips.  The CTA kernels stage rows and weights in shared
// memory behind two block barriers and, at this size, leave most of each
// CTA idle.  Launched with programmatic stream serialisation: the launch
// may overlap the previous kernel's tail; griddepcontrol.wait precedes
// every global access.  The same fp32 fma chain in slot order, so the
// results equal the CTA kernels' bit for bit.
constexpr int kFlatThreads = 256;

// Rows and weights of slots [j0, j0 + 8) of token t; a row outside [0, rows)
// is flagged (by the token's first chunk) and skipped.
__device__ __forceinline__ void flat_slots(const int32_t *__restrict__ pos, const float *__restrict__ w, long long t,
                                           int k, int j0, long long rows, int32_t *err_flag, bool first,
                                           int (&p)[kSlotBatch], float (&ww)[kSlotBatch])
{
#pragma unroll
    for (int u = 0; u < kSlotBatch; ++u) {
        const int j = j0 + u;
        p[u] = j < k ? __ldg(pos + t * k + j) : -1;
        ww[u] = j < k ? (w ? __ldg(w + t * k + j) : 1.0f) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kSlotBatch; ++u)
        if (p[u] >= rows) {
            if (first && err_flag)
                atomicOr(err_flag, 2);
            p[u] = -1;
        }
}

__global__ void __launch_bounds__(kFlatThreads) combine_flat_kernel(const uint16_t *__restrict__ y,
                                                                    const int32_t *__restrict__ pos,
                                                                    const float *__restrict__ w, int T, int H, int k,
                                                                    uint16_t *__restrict__ out, long long rows,
                                                                    int32_t *__restrict__ err_flag)
{
    pdl_wait();
    const int C = H / 8;
    const long long g = (long long)blockIdx.x * kFlatThreads + threadIdx.x;
    if (g >= (long long)T * C)
        return;
    const long long t = g / C;
    const int c = (int)(g - t * C);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
        int p[kSlotBatch];
        float ww[kSlotBatch];
        flat_slots(pos, w, t, k, j0, rows, err_flag, c == 0, p, ww);
        uint4 v[kSlotBatch];
#pragma unroll
        for (int u = 0; u < kSlotBatch; ++u)
            if (p[u] >= 0)
                v[u] = ld_stream16(y + (size_t)p[u] * H + (size_t)c * 8);
#pragma unroll
        for (int u = 0; u < kSlotBatch; ++u)
            if (p[u] >= 0) {
                const uint32_t vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(ww[u], bf16_lo(vv[i]), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(ww[u], bf16_hi(vv[i]), acc[2 * i + 1]);
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

template <bool kMx>
__global__ void __launch_bounds__(kFlatThreads) combine_fp8_flat_kernel(const uint8_t *__restrict__ yq,
                                                                        const void *__restrict__ yscale,
                                                                        const int32_t *__restrict__ pos,
                                                                        const float *__restrict__ w, int T, int H,
                                                                        int k, uint16_t *__restrict__ out,
                                                                        long long rows, int32_t *__restrict__ err_flag)
{
    pdl_wait();
    const int C16 = H / 16;
    const int nb = kMx ? H / 32 : H / 128;
    const long long g = (long long)blockIdx.x * kFlatThreads + threadIdx.x;
    if (g >= (long long)T * C16)
        return;
    const long long t = g / C16;
    const int c = (int)(g - t * C16);
    const int sb = kMx ? (c >> 1) : (c >> 3);
    uint64_t acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = 0ull;
    for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
        int p[kSlotBatch];
        float ww[kSlotBatch];
        flat_slots(pos, w, t, k, j0, rows, err_flag, c == 0, p, ww);
        uint4 v[kSlotBatch];
        uint32_t sraw[kSlotBatch];
#pragma unroll
        for (int u = 0; u < kSlotBatch; ++u)
            if (p[u] >= 0) {
                v[u] = ld_stream16(yq + (size_t)p[u] * H + (size_t)c * 16);
                sraw[u] = kMx ? (uint32_t)__ldg(static_cast<const uint8_t *>(yscale) + (size_t)p[u] * nb + sb)
                              : __float_as_uint(__ldg(static_cast<const float *>(yscale) + (size_t)p[u] * nb + sb));
            }
#pragma unroll
        for (int u = 0; u < kSlotBatch; ++u)
            if (p[u] >= 0) {
                const float sc = kMx ? e8m0_to_f32(sraw[u]) : __uint_as_float(sraw[u]);
                const float ws = ww[u] * sc;
                fma_codes16(f2_pack(ws, ws), v[u], acc);
            }
    }
    uint4 o0, o1;
    pack_acc16(acc, o0, o1);
    uint16_t *dst = out + (size_t)t * H + (size_t)c * 16;
    st_stream16(dst, o0);
    st_stream16(dst + 8, o1);
}

// Batches that take the thread-per-chunk kernels: at most two tokens per
// SM.  Measured on GB300 (H = 7168, k = 8): at 128 tokens they take 3.2 us
// a call back to back against 5.7 for the CTA kernel (FP8 input: 3.5
// against 4.1); at 512 tokens, 16.0 us against 14.6 (ncu, cold).
inline bool flat_sized(int T) { return T <= 2 * device_sm_count(); }

// Launches a flat kernel with programmatic stream serialisation.
template <class... P, class... A>
cudaError_t launch_flat(void (*kern)(P...), long long threads, cudaStream_t st, A... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((threads + kFlatThreads - 1) / kFlatThreads));
    cfg.blockDim = dim3(kFlatThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Few slots per token (k <= 2, Mixtral-like routing): one warp per token and
// no block barrier.  A CTA-per-token combine keeps only k loads in flight
// per thread there and waits at two barriers per token; here each lane
// takes kWarpChunks 16-byte column chunks of the row at once (k * kWarpChunks
// loads in flight), and warps move to their next token independently, its
// rows and weights fetched while the current one is summed.  Each column's
// fma chain is the one combine_kernel runs.
constexpr int kWarpChunks = 4;

__global__ void __launch_bounds__(kCombThreads) combine_warp_kernel(const uint16_t *__restrict__ y,
                                                                    const int32_t *__restrict__ pos,
                                                                    const float *__restrict__ w, int T, int H, int k,
                                                                    uint16_t *__restrict__ out, long long rows,
                                                                    int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    const long long warp = balanced_warp();
    const long long nwarps = grid_warps();
    const int C = H / 8;
    // lane j < k holds slot j's row and weight (k <= 2)
    int np = -1;
    float nw = 0.0f;
    if (warp < T && lane < k) {
        np = __ldg(pos + warp * k + lane);
        nw = w ? __ldg(w + warp * k + lane) : 1.0f;
    }
    for (long long t = warp; t < T; t += nwarps) {
        int p = np;
        if (lane < k && p >= rows) {
            if (err_flag)
                atomicOr(err_flag, 2);
            p = -1;
        }
        const int p0 = __shfl_sync(kFullMask, p, 0), p1 = __shfl_sync(kFullMask, p, 1);
        const float w0 = __shfl_sync(kFullMask, nw, 0), w1 = __shfl_sync(kFullMask, nw, 1);
        const int q0 = k > 0 ? p0 : -1, q1 = k > 1 ? p1 : -1;
        const long long tn = t + nwarps;  // the next token's rows and weights
        if (tn < T && lane < k) {
            np = __ldg(pos + tn * k + lane);
            nw = w ? __ldg(w + tn * k + lane) : 1.0f;
        }
        for (int c0 = lane; c0 < C; c0 += 32 * kWarpChunks) {
            uint4 v0[kWarpChunks], v1[kWarpChunks];
#pragma unroll
            for (int m = 0; m < kWarpChunks; ++m) {
                const int c = c0 + 32 * m;
                if (c < C) {
                    if (q0 >= 0)
                        v0[m] = ld_stream16(y + (size_t)q0 * H + (size_t)c * 8);
                    if (q1 >= 0)
                        v1[m] = ld_stream16(y + (size_t)q1 * H + (size_t)c * 8);
                }
            }
#pragma unroll
            for (int m = 0; m < kWarpChunks; ++m) {
                const int c = c0 + 32 * m;
                if (c >= C)
                    continue;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = 0.0f;
                if (q0 >= 0) {
                    const uint32_t vv[4] = {v0[m].x, v0[m].y, v0[m].z, v0[m].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = fmaf(w0, bf16_lo(vv[i]), acc[2 * i]);
                        acc[2 * i + 1] = fmaf(w0, bf16_hi(vv[i]), acc[2 * i + 1]);
                    }
                }
                if (q1 >= 0) {
                    const uint32_t vv[4] = {v1[m].x, v1[m].y, v1[m].z, v1[m].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = fmaf(w1, bf16_lo(vv[i]), acc[2 * i]);
                        acc[2 * i + 1] = fmaf(w1, bf16_hi(vv[i]), acc[2 * i + 1]);
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
}

// Blocks of 4 warps at up to 72 registers a thread keep 28 warps on an SM
// (7 blocks), so a 4096-token batch finishes in one round of warps.
constexpr int kFp8WarpThreads = 128;

// The FP8 / MXFP8-input combine with one warp per token for k <= 2, as
// combine_warp_kernel: each lane takes kWarpChunks 16-column chunks at once
// (16 codes and their block scale per slot); the arithmetic is
// combine_fp8_kernel's (w * s once per slot and block, then the fma chain).
template <bool kMx>
__global__ void __launch_bounds__(kFp8WarpThreads, 7) combine_fp8_warp_kernel(const uint8_t *__restrict__ yq,
                                                                        const void *__restrict__ yscale,
                                                                        const int32_t *__restrict__ pos,
                                                                        const float *__restrict__ w, int T, int H,
                                                                        int k, uint16_t *__restrict__ out,
                                                                        long long rows,
                                                                        int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    const long long warp = balanced_warp();
    const long long nwarps = grid_warps();
    const int C16 = H / 16;
    const int nb = kMx ? H / 32 : H / 128;
    int np = -1;
    float nw = 0.0f;
    if (warp < T && lane < k) {
        np = __ldg(pos + warp * k + lane);
        nw = __ldg(w + warp * k + lane);
    }
    for (long long t = warp; t < T; t += nwarps) {
        int p = np;
        if (lane < k && p >= rows) {
            if (err_flag)
                atomicOr(err_flag, 2);
            p = -1;
        }
        const int p0 = __shfl_sync(kFullMask, p, 0), p1 = __shfl_sync(kFullMask, p, 1);
        const float w0 = __shfl_sync(kFullMask, nw, 0), w1 = __shfl_sync(kFullMask, nw, 1);
        const int q0 = k > 0 ? p0 : -1, q1 = k > 1 ? p1 : -1;
        const long long tn = t + nwarps;
        if (tn < T && lane < k) {
            np = __ldg(pos + tn * k + lane);
            nw = __ldg(w + tn * k + lane);
        }
        for (int c0 = lane; c0 < C16; c0 += 32 * kWarpChunks) {
            uint4 v0[kWarpChunks], v1[kWarpChunks];
            uint32_t s0[kWarpChunks], s1[kWarpChunks];
#pragma unroll
            for (int m = 0; m < kWarpChunks; ++m) {
                const int c = c0 + 32 * m;
                if (c >= C16)
                    continue;
                const int sb = kMx ? (c >> 1) : (c >> 3);
                if (q0 >= 0) {
                    v0[m] = ld_stream16(yq + (size_t)q0 * H + (size_t)c * 16);
                    s0[m] = kMx ? (uint32_t)__ldg(static_cast<const uint8_t *>(yscale) + (size_t)q0 * nb + sb)
                                : __float_as_uint(__ldg(static_cast<const float *>(yscale) + (size_t)q0 * nb + sb));
                }
                if (q1 >= 0) {
                    v1[m] = ld_stream16(yq + (size_t)q1 * H + (size_t)c * 16);
                    s1[m] = kMx ? (uint32_t)__ldg(static_cast<const uint8_t *>(yscale) + (size_t)q1 * nb + sb)
                                : __float_as_uint(__ldg(static_cast<const float *>(yscale) + (size_t)q1 * nb + sb));
                }
            }
#pragma unroll
            for (int m = 0; m < kWarpChunks; ++m) {
                const int c = c0 + 32 * m;
                if (c >= C16)
                    continue;
                uint64_t acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = 0ull;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int q = j == 0 ? q0 : q1;
                    if (q < 0)
                        continue;
                    const uint32_t sr = j == 0 ? s0[m] : s1[m];
                    const float sc = kMx ? e8m0_to_f32(sr) : __uint_as_float(sr);
                    const float ws = (j == 0 ? w0 : w1) * sc;
                    fma_codes16(f2_pack(ws, ws), j == 0 ? v0[m] : v1[m], acc);
                }
                uint4 o0, o1;
                pack_acc16(acc, o0, o1);
                uint16_t *dst = out + (size_t)t * H + (size_t)c * 16;
                st_stream16(dst, o0);
                st_stream16(dst + 8, o1);
            }
        }
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t *y, long long rows, const int32_t *pos, const float *w, int T, int H,
                           int k, uint16_t *out, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    if (k <= 2 && T >= 2048) {
        static PerDeviceCache<1> occ;
        const int wps = occupancy_per_sm(occ, (const void *)combine_warp_kernel, kCombThreads, 0);
        long long g = (long long)device_sm_count() * wps;  // one token per CTA at least (balanced_warp)
        if (g > T)
            g = T;
        combine_warp_kernel<<<(int)g, kCombThreads, 0, st>>>(y, pos, w, T, H, k, out, rows, err_flag);
        return cudaGetLastError();
    }
    static PerDeviceCache<1> occ;  // the same registers either way: sized on the unsplit kernel
    const int per_sm = occupancy_per_sm(occ, (const void *)combine_kernel<false>, kCombThreads, 0);
    if (flat_sized(T))  // decode-sized: one thread per chunk
        return launch_flat(combine_flat_kernel, (long long)T * (H / 8), st, y, pos, w, T, H, k, out, rows, err_flag);
    const int S = column_segments(T, H / 8, device_sm_count() * per_sm);
    long long grid = (long long)device_sm_count() * per_sm;
    if (grid > (long long)T * S)
        grid = (long long)T * S;
    if (S > 1)
        combine_kernel<true><<<(int)grid, kCombThreads, 0, st>>>(y, pos, w, T, H, k, out, rows, err_flag, S);
    else
        combine_kernel<false><<<(int)grid, kCombThreads, 0, st>>>(y, pos, w, T, H, k, out, rows, err_flag, 1);
    return cudaGetLastError();
}

}  // namespace ep

namespace ep {

cudaError_t launch_combine_fp8(const uint8_t *yq, const void *yscale, int mx, long long rows, const int32_t *pos,
                               const float *w, int T, int H, int k, uint16_t *out, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    if (k <= 2 && T >= 2048) {
        static PerDeviceCache<2> occ;
        const void *wk = mx ? (const void *)combine_fp8_warp_kernel<true> : (const void *)combine_fp8_warp_kernel<false>;
        const int ps = occupancy_per_sm(occ, wk, kFp8WarpThreads, 0, mx ? 1 : 0);
        long long g = (long long)device_sm_count() * ps;  // one token per CTA at least (balanced_warp)
        if (g > T)
            g = T;
        if (mx)
            combine_fp8_warp_kernel<true><<<(int)g, kFp8WarpThreads, 0, st>>>(yq, yscale, pos, w, T, H, k, out, rows,
                                                                          err_flag);
        else
            combine_fp8_warp_kernel<false><<<(int)g, kFp8WarpThreads, 0, st>>>(yq, yscale, pos, w, T, H, k, out, rows,
                                                                           err_flag);
        return cudaGetLastError();
    }
    static PerDeviceCache<2> occ;
    const void *kern =
        mx ? (const void *)combine_fp8_kernel<true, false> : (const void *)combine_fp8_kernel<false, false>;
    const int per_sm = occupancy_per_sm(occ, kern, kCombThreads, 0, mx ? 1 : 0);
    if (flat_sized(T)) {  // decode-sized: one thread per chunk
        const long long n = (long long)T * (H / 16);
        return mx ? launch_flat(combine_fp8_flat_kernel<true>, n, st, yq, yscale, pos, w, T, H, k, out, rows, err_flag)
                  : launch_flat(combine_fp8_flat_kernel<false>, n, st, yq, yscale, pos, w, T, H, k, out, rows,
                                err_flag);
    }
    const int S = column_segments(T, H / 16, device_sm_count() * per_sm);
    long long gl = (long long)device_sm_count() * per_sm;
    if (gl > (long long)T * S)
        gl = (long long)T * S;
    const int grid = (int)gl;
    if (mx && S > 1)
        combine_fp8_kernel<true, true><<<grid, kCombThreads, 0, st>>>(yq, yscale, pos, w, T, H, k, out, rows,
                                                                      err_flag, S);
    else if (mx)
        combine_fp8_kernel<true, false><<<grid, kCombThreads, 0, st>>>(yq, yscale, pos, w, T, H, k, out, rows,
                                                                       err_flag, 1);
    else if (S > 1)
        combine_fp8_kernel<false, true><<<grid, kCombThreads, 0, st>>>(yq, yscale, pos, w, T, H, k, out, rows,
                                                                       err_flag, S);
    else
        combine_fp8_kernel<false, false><<<grid, kCombThreads, 0, st>>>(yq, yscale, pos, w, T, H, k, out, rows,
                                                                        err_flag, 1);
    return cudaGetLastError();
}

}  // namespace ep
