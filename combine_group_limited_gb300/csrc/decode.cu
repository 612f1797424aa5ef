// decode.cu -- fused low-latency path for decode-sized batches: gating,
// layout and dispatch in one cooperative launch.
//
// "DeepEP de DeepSeek ...", section "Kernels low-latency dispatch et
// combine": separate latency-optimised kernels for small (decode) batches;
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all": decode messages of 100 KB to 2 MB, where the
// exchange is 10-30 % of end-to-end latency.  At T = 128 the three separate
// steps are five short launches; here they are one:
//   1. gating: warps over the tokens, grid-wide (gate_impl.cuh);
//   2. a grid barrier (every CTA is resident: cooperative launch), with a
//      bounded wait -- past its limit a CTA sets EP_FLAG_TIMEOUT and stops;
//   3. every CTA rebuilds the whole layout of the T*k <= 4096 entries in
//      shared memory (warp-aggregated histogram, exclusive scan, stable
//      ranks from ballot peer masks) from the chosen experts; CTA 0 writes
//      the layout outputs;
//   4. warp items over (token, row segment) grid-wide scatter the rows
//      (dispatch_impl.cuh), reading each token's receive rows from shared
//      memory.
// Results are the ones the separate calls give, bit for bit.
#include "dispatch_impl.cuh"
#include "gate_impl.cuh"

namespace ep {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxExperts = 1024;

struct DecodeArgs {
    const float *scores;
    const float *bias;
    int T;
    GateParams gp;
    int group_lanes, vec_rows;
    int epr;
    const uint16_t *x;
    int H;
    int dtype;  // ep_dtype
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_count, *expert_off, *rank_count, *rank_off, *rank_tokens, *pos, *src;
    void *recv;
    void *recv_scales;
    long long rows;
    int32_t *err_flag;
    unsigned *barrier;
    unsigned barrier_extra;  // arrivals expected beyond the grid (0; >0 only in the self-test)
    long long spin_limit;
};

// All CTAs of the (cooperative) grid arrive once; the wait is bounded.
// Returns false, with EP_FLAG_TIMEOUT set, if the limit ran out.
__device__ bool grid_barrier(unsigned *counter, unsigned expected, long long spin_limit, int32_t *err_flag)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's global writes before its arrival
        atomicAdd(counter, 1u);
        unsigned v = 0;
        long long it = 0;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= expected || ++it >= spin_limit)
                break;
            __nanosleep(64);
        }
        s_ok = v >= expected;
        if (!s_ok && err_flag)
            atomicOr(err_flag, 4);
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off)
            v += n;
    }
    return v;
}

template <int EPL>
__global__ void __launch_bounds__(kDecThreads) decode_fused_kernel(const DecodeArgs a)
{
    extern __shared__ int32_t dsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.gp.E, k = a.gp.k, T = a.T, N = T * k, R = E / a.epr;

    // 1. gating
    for (int t = blockIdx.x * kDecWarps + warp; t < T; t += gridDim.x * kDecWarps)
        gate_token<EPL>(a.scores, a.bias, t, a.gp, a.group_lanes, a.vec_rows, reinterpret_cast<float *>(dsm) + warp * E,
                        a.topk_idx, a.topk_w);

    // 2. every CTA's experts are written
    if (!grid_barrier(a.barrier, gridDim.x + a.barrier_extra, a.spin_limit, a.err_flag))
        return;

    // 3. layout of all N entries in shared memory
    int32_t *s_idx = dsm;                  // [N]
    int32_t *s_pos = s_idx + N;            // [N]
    int32_t *s_off = s_pos + N;            // [E] counts, then offsets
    int32_t *hist = s_off + E;             // [kDecWarps][E]
    int32_t *s_rt = hist + kDecWarps * E;  // [R]
    __shared__ int32_t s_wsum[kDecWarps];
    __shared__ int32_t s_total;
    for (int i = threadIdx.x; i < N; i += blockDim.x)
        s_idx[i] = __ldcg(a.topk_idx + i);  // written by other CTAs: read through L2
    for (int i = threadIdx.x; i < E + kDecWarps * E + R; i += blockDim.x)
        s_off[i] = 0;
    __syncthreads();
    const int eb = key_bits((unsigned)E), rb = key_bits((unsigned)R);
    for (int base = threadIdx.x & ~31; base < N; base += blockDim.x) {
        const int i = base + lane;
        const int e = i < N ? s_idx[i] : -1;
        const bool ok = (unsigned)e < (unsigned)E;
        warp_count(s_off, ok ? (unsigned)e : 0u, ok, eb);
    }
    __syncthreads();
    {
        constexpr int kPerThread = kMaxExperts / kDecThreads;
        const int e0 = threadIdx.x * kPerThread;
        int v[kPerThread];
        int sum = 0;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            v[u] = e0 + u < E ? s_off[e0 + u] : 0;
            sum += v[u];
        }
        const int incl = warp_incl_scan(sum, lane);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = lane < kDecWarps ? s_wsum[lane] : 0;
            const int wi = warp_incl_scan(ws, lane);
            if (lane < kDecWarps)
                s_wsum[lane] = wi - ws;
        }
        __syncthreads();
        int run = s_wsum[warp] + incl - sum;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            if (e0 + u < E)
                s_off[e0 + u] = run;
            if (e0 + u == E - 1)
                s_total = run + v[u];
            run += v[u];
        }
    }
    __syncthreads();
    const int per_warp = ((N + kDecWarps * 32 - 1) / (kDecWarps * 32)) * 32;
    const int w0 = warp * per_warp;
    const int w1 = min(N, w0 + per_warp);
    int32_t *my = hist + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int c = w0; c < w1; c += 32) {
        const int i = c + lane;
        const int e = i < w1 ? s_idx[i] : -1;
        const int key = (unsigned)e < (unsigned)E ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int base = s_off[e];
        for (int w = 0; w < kDecWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = base;
            base += c;
        }
    }
    __syncthreads();
    for (int c = w0; c < w1; c += 32) {
        const int i = c + lane;
        const bool in = i < w1;
        const int e = in ? s_idx[i] : -1;
        const int key = (unsigned)e < (unsigned)E ? e : E;
        const unsigned grp = peer_mask((unsigned)key, eb);
        if (in)
            s_pos[i] = key < E ? my[key] + __popc(grp & lt_mask) : -1;
        __syncwarp();
        if (key < E && lane == __ffs(grp) - 1)
            my[key] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();
    const int total = s_total;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int hi = e + 1 < E ? s_off[e + 1] : total;
            a.expert_off[e] = s_off[e];
            a.expert_count[e] = hi - s_off[e];
        }
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            const int lo = s_off[r * a.epr];
            const int hi = (r + 1) * a.epr < E ? s_off[(r + 1) * a.epr] : total;
            a.rank_off[r] = lo;
            a.rank_count[r] = hi - lo;
        }
        if (threadIdx.x == 0) {
            a.expert_off[E] = total;
            a.rank_off[R] = total;
        }
        for (int base = threadIdx.x & ~31; base < N; base += blockDim.x) {
            const int i = base + lane;
            const bool in = i < N;
            const int p = in ? s_pos[i] : -1;
            if (in) {
                a.pos[i] = p;
                if (p >= 0)
                    a.src[p] = i;
            }
            const int e = in ? s_idx[i] : -1;
            const bool ok = (unsigned)e < (unsigned)E;
            // distinct tokens per rank: the token's first slot on the rank counts
            const int r = ok ? e / a.epr : 0;
            bool first = ok;
            if (ok) {
                const int j = i % k;
                for (int jj = 0; jj < j; ++jj) {
                    const int e2 = s_idx[i - j + jj];
                    first &= !((unsigned)e2 < (unsigned)E && e2 / a.epr == r);
                }
            }
            warp_count(s_rt, (unsigned)r, first, rb);
        }
        for (int i = total + threadIdx.x; i < N; i += blockDim.x)
            a.src[i] = -1;
        __syncthreads();
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            a.rank_tokens[r] = s_rt[r];
    }

    // 4. scatter the rows
    const int segs = a.dtype == 0 ? bf16_segs(a.H) : fp8_segs(a.H);
    for (ItemWalk it(T, segs); it.valid(); it.next()) {
        int p0 = -1, p1 = -1;
        if (lane < k)
            p0 = s_pos[it.t * k + lane];
        if (lane + 32 < k)
            p1 = s_pos[it.t * k + lane + 32];
        if (p0 >= a.rows || p1 >= a.rows) {
            if (a.err_flag)
                atomicOr(a.err_flag, 2);
            p0 = p0 >= a.rows ? -1 : p0;
            p1 = p1 >= a.rows ? -1 : p1;
        }
        if (a.dtype == 0)
            dispatch_bf16_item(a.x, a.H, k, it.t, it.seg, p0, p1, static_cast<uint16_t *>(a.recv));
        else if (a.dtype == 1)
            dispatch_fp8_item(a.x, a.H, k, it.t, it.seg, p0, p1, static_cast<uint8_t *>(a.recv),
                              static_cast<float *>(a.recv_scales));
        else
            dispatch_mxfp8_item(a.x, a.H, k, it.t, it.seg, p0, p1, static_cast<uint8_t *>(a.recv),
                                static_cast<uint8_t *>(a.recv_scales));
    }
}

// Barrier check: one cooperative launch that only arrives at the barrier,
// expecting `extra` arrivals that never come when extra > 0.
__global__ void __launch_bounds__(kDecThreads) barrier_selftest_kernel(unsigned *counter, unsigned extra,
                                                                       long long spin_limit, int32_t *err_flag)
{
    grid_barrier(counter, gridDim.x + extra, spin_limit, err_flag);
}

size_t decode_smem_bytes(int T, int k, int E, int epr, int warp_floats)
{
    const size_t gate = (size_t)kDecWarps * warp_floats * sizeof(float);
    const size_t lay = ((size_t)2 * T * k + E + (size_t)kDecWarps * E + E / epr) * sizeof(int32_t);
    return gate > lay ? gate : lay;
}

template <int EPL>
cudaError_t launch_epl(DecodeArgs a, cudaStream_t st)
{
    int warp_floats;
    gate_plan<EPL>(a.gp, a.scores, a.bias, a.group_lanes, a.vec_rows, warp_floats);
    const size_t smem = decode_smem_bytes(a.T, a.gp.k, a.gp.E, a.epr, warp_floats);
    const void *fn = (const void *)decode_fused_kernel<EPL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kDecThreads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    // At most the resident CTAs per SM (up to 3, for the scatter's bytes in
    // flight) times the SMs: every CTA is resident, as the grid barrier
    // requires (the cooperative launch refuses a larger grid).
    const int grid = device_sm_count() * (per_sm < 3 ? per_sm : 3);
    e = cudaMemsetAsync(a.barrier, 0, sizeof(unsigned), st);
    if (e != cudaSuccess)
        return e;
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kDecThreads), args, smem, st);
}

}  // namespace

constexpr long long kDecodeSpinLimit = 1LL << 21;  // about a second of polling

size_t decode_max_entries() { return 4096; }

cudaError_t launch_decode(const float *scores, const float *bias, int T, const GateParams &gp, int epr,
                          const uint16_t *x, int H, int dtype, int32_t *topk_idx, float *topk_w,
                          int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                          int32_t *rank_tokens, int32_t *pos, int32_t *src, void *recv, void *recv_scales,
                          long long rows, int32_t *err_flag, void *barrier_word, cudaStream_t st)
{
    DecodeArgs a{};
    a.scores = scores;
    a.bias = bias;
    a.T = T;
    a.gp = gp;
    a.epr = epr;
    a.x = x;
    a.H = H;
    a.dtype = dtype;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.expert_count = expert_count;
    a.expert_off = expert_off;
    a.rank_count = rank_count;
    a.rank_off = rank_off;
    a.rank_tokens = rank_tokens;
    a.pos = pos;
    a.src = src;
    a.recv = recv;
    a.recv_scales = recv_scales;
    a.rows = rows;
    a.err_flag = err_flag;
    a.barrier = static_cast<unsigned *>(barrier_word);
    a.barrier_extra = 0;
    a.spin_limit = kDecodeSpinLimit;
    if (gp.E <= 32)
        return launch_epl<1>(a, st);
    if (gp.E <= 64)
        return launch_epl<2>(a, st);
    if (gp.E <= 128)
        return launch_epl<4>(a, st);
    if (gp.E <= 256)
        return launch_epl<8>(a, st);
    return launch_epl<16>(a, st);
}

cudaError_t launch_barrier_selftest(unsigned extra, long long spin_limit, int32_t *err_flag, void *barrier_word,
                                    cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(barrier_word, 0, sizeof(unsigned), st);
    if (e != cudaSuccess)
        return e;
    unsigned *counter = static_cast<unsigned *>(barrier_word);
    void *args[] = {&counter, &extra, &spin_limit, &err_flag};
    return cudaLaunchCooperativeKernel((const void *)barrier_selftest_kernel, dim3(device_sm_count()),
                                       dim3(kDecThreads), args, 0, st);
}

}  // namespace ep
