// decode.cu -- fused low-latency path for decode-sized batches: gating,
// layout and dispatch in one cooperative launch.
//
// "DeepEP de DeepSeek ...", section "Kernels low-latency dispatch et
// combine": separate latency-optimised kernels for small (decode) batches;
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all": decode messages of 100 KB to 2 MB, where the
// exchange is 10-30 % of end-to-end latency.  At T = 128 the three separate
// steps are five short launches; here they are one:
// each CTA (one per SM) owns a contiguous range of tokens:
//   1. it gates its tokens (gate_impl.cuh);
//   2. a grid barrier (every CTA is resident: cooperative launch), with a
//      bounded wait -- past its limit a CTA sets EP_FLAG_TIMEOUT and stops;
//   3. it counts all T*k <= 4096 chosen experts and those before its range
//      (warp-aggregated shared counters), scans the totals into expert
//      offsets, and gives its own entries their stable rows (offset +
//      earlier entries of the expert + equal lower lanes, ballot peer
//      masks); CTA 0 writes the offsets and counts, every CTA its rows and
//      its share of the distinct-token counts;
//   4. it scatters its own tokens' rows (dispatch_impl.cuh).
// Results are the ones the separate calls give, bit for bit.
#include "coop.cuh"
#include "dispatch_impl.cuh"
#include "gate_impl.cuh"

namespace ep {

namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxEntries = 4096;                           // T*k of the fused path
constexpr int kDecChunks = kMaxEntries / (kDecWarps * 32);  // 32-entry chunks per warp

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

template <int EPL>
__global__ void __launch_bounds__(kDecThreads) decode_fused_kernel(const DecodeArgs a)
{
    extern __shared__ int32_t dsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.gp.E, k = a.gp.k, T = a.T, N = T * k, R = E / a.epr;
    // This CTA's tokens: a contiguous range, so that its entries' rows only
    // need the counts of the entries before the range.
    const int t_lo = (int)((long long)T * blockIdx.x / gridDim.x);
    const int t_hi = (int)((long long)T * (blockIdx.x + 1) / gridDim.x);
    const int n_lo = t_lo * k, n_hi = t_hi * k;

    // 1. gating of this CTA's tokens
    for (int t = t_lo + warp; t < t_hi; t += kDecWarps)
        gate_token<EPL>(a.scores, a.bias, t, a.gp, a.group_lanes, a.vec_rows,
                        reinterpret_cast<uint32_t *>(dsm) + warp * gate_warp_words<EPL>(), a.topk_idx, a.topk_w);
    if (blockIdx.x == 0)
        for (int r = threadIdx.x; r < R; r += blockDim.x)
            a.rank_tokens[r] = 0;  // accumulated by every CTA after the barrier

    // 2. every CTA's experts are written
    if (!grid_barrier(a.barrier, gridDim.x + a.barrier_extra, a.spin_limit, a.err_flag))
        return;

    // 3. counts of all entries and of the entries before this CTA's range
    int32_t *s_tot = dsm;                 // [E] totals, then offsets
    int32_t *s_pre = s_tot + E;           // [E] entries before n_lo
    int32_t *s_rt = s_pre + E;            // [R] this range's distinct tokens per rank
    int32_t *s_idx = s_rt + R;            // [n_hi - n_lo] this range's experts
    int32_t *s_rows = s_idx + (n_hi - n_lo);  // [n_hi - n_lo] their receive rows
    __shared__ int32_t s_wsum[kDecWarps];
    __shared__ int32_t s_total;
    for (int i = threadIdx.x; i < 2 * E + R; i += blockDim.x)
        dsm[i] = 0;
    __syncthreads();
    const int eb = key_bits((unsigned)E), rb = key_bits((unsigned)R);
    {
        // each warp loads its slice of all N experts at once (written by
        // other CTAs: read through L2), then counts it
        const int per_warp = ((N + kDecWarps * 32 - 1) / (kDecWarps * 32)) * 32;  // <= kDecChunks * 32
        const int w0 = warp * per_warp;
        int ev[kDecChunks];
#pragma unroll
        for (int c = 0; c < kDecChunks; ++c) {
            const int i = w0 + 32 * c + lane;
            ev[c] = (32 * c < per_warp && i < N) ? __ldcg(a.topk_idx + i) : -1;
        }
#pragma unroll
        for (int c = 0; c < kDecChunks; ++c) {
            if (32 * c >= per_warp)
                break;
            const int i = w0 + 32 * c + lane;
            const int e = ev[c];
            const bool ok = (unsigned)e < (unsigned)E;
            warp_count(s_tot, ok ? (unsigned)e : 0u, ok, eb);
            warp_count(s_pre, ok ? (unsigned)e : 0u, ok && i < n_lo, eb);
            if (i >= n_lo && i < n_hi)
                s_idx[i - n_lo] = e;
        }
    }
    __syncthreads();
    {
        constexpr int kPerThread = kMaxExperts / kDecThreads;
        const int e0 = threadIdx.x * kPerThread;
        int v[kPerThread];
        int sum = 0;
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            v[u] = e0 + u < E ? s_tot[e0 + u] : 0;
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
            if (e0 + u < E) {
                s_tot[e0 + u] = run;
                if (blockIdx.x == 0) {
                    a.expert_off[e0 + u] = run;
                    a.expert_count[e0 + u] = v[u];
                }
            }
            if (e0 + u == E - 1)
                s_total = run + v[u];
            run += v[u];
        }
    }
    __syncthreads();
    const int total = s_total;
    if (blockIdx.x == 0) {
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            const int lo = s_tot[r * a.epr];
            const int hi = (r + 1) * a.epr < E ? s_tot[(r + 1) * a.epr] : total;
            a.rank_off[r] = lo;
            a.rank_count[r] = hi - lo;
        }
        if (threadIdx.x == 0) {
            a.expert_off[E] = total;
            a.rank_off[R] = total;
        }
    }
    for (int i = total + blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
        a.src[i] = -1;
    // Rows of this range's entries, in flat order: warp 0 walks the range in
    // 32-entry chunks; a lane's row is its expert's offset + the entries of
    // that expert before the range + the equal lower lanes so far.
    if (warp == 0) {
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int c = n_lo; c < n_hi; c += 32) {
            const int i = c + lane;
            const bool in = i < n_hi;
            const int e = in ? s_idx[i - n_lo] : -1;
            const int key = (unsigned)e < (unsigned)E ? e : E;
            const unsigned grp = peer_mask((unsigned)key, key_bits((unsigned)E));
            int p = -1;
            if (key < E)
                p = s_tot[key] + s_pre[key] + __popc(grp & lt_mask);
            if (in) {
                a.pos[i] = p;
                s_rows[i - n_lo] = p;
                if (p >= 0)
                    a.src[p] = i;
            }
            __syncwarp();
            if (key < E && lane == __ffs(grp) - 1)
                s_pre[key] += __popc(grp);
            __syncwarp();
        }
    }
    // distinct tokens per rank, from this range's experts (shared memory)
    for (int base = n_lo + (threadIdx.x & ~31); base < n_hi; base += blockDim.x) {
        const int i = base + lane;
        const int e = i < n_hi ? s_idx[i - n_lo] : -1;
        const bool ok = (unsigned)e < (unsigned)E;
        const int r = ok ? e / a.epr : 0;
        bool first = ok;
        if (ok) {
            const int j = (i - n_lo) % k;
            for (int jj = 0; jj < j; ++jj) {
                const int e2 = s_idx[i - n_lo - j + jj];
                first &= !((unsigned)e2 < (unsigned)E && e2 / a.epr == r);
            }
        }
        warp_count(s_rt, (unsigned)r, first, rb);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x)
        if (s_rt[r])
            atomicAdd(a.rank_tokens + r, s_rt[r]);

    // 4. scatter this CTA's rows: warp items over (token, row segment)
    const int segs = a.dtype == 0 ? bf16_segs(a.H) : fp8_segs(a.H);
    const int items = (t_hi - t_lo) * segs;
    for (int item = warp; item < items; item += kDecWarps) {
        const int t = t_lo + item / segs;
        const int seg = item - (t - t_lo) * segs;
        int p0 = -1, p1 = -1;
        if (lane < k)
            p0 = s_rows[(t - t_lo) * k + lane];
        if (lane + 32 < k)
            p1 = s_rows[(t - t_lo) * k + lane + 32];
        if (p0 >= a.rows || p1 >= a.rows) {
            if (a.err_flag)
                atomicOr(a.err_flag, 2);
            p0 = p0 >= a.rows ? -1 : p0;
            p1 = p1 >= a.rows ? -1 : p1;
        }
        if (a.dtype == 0)
            dispatch_bf16_item(a.x, a.H, k, t, seg, p0, p1, static_cast<uint16_t *>(a.recv));
        else if (a.dtype == 1)
            dispatch_fp8_item(a.x, a.H, k, t, seg, p0, p1, static_cast<uint8_t *>(a.recv),
                              static_cast<float *>(a.recv_scales));
        else
            dispatch_mxfp8_item(a.x, a.H, k, t, seg, p0, p1, static_cast<uint8_t *>(a.recv),
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

size_t decode_smem_bytes(int range_entries, int E, int epr, int warp_floats)
{
    const size_t gate = (size_t)kDecWarps * warp_floats * sizeof(float);
    const size_t lay = ((size_t)2 * E + E / epr + 2 * (size_t)range_entries) * sizeof(int32_t);
    return gate > lay ? gate : lay;
}

template <int EPL>
cudaError_t launch_epl(DecodeArgs a, cudaStream_t st)
{
    int warp_floats;
    gate_plan<EPL>(a.gp, a.scores, a.bias, a.group_lanes, a.vec_rows, warp_floats);
    // One CTA per SM, at most one per token: every CTA is resident, as the
    // grid barrier requires (the cooperative launch refuses a larger grid).
    const int sms = device_sm_count();
    const int grid = a.T < sms ? a.T : sms;
    const int range_entries = ((a.T + grid - 1) / grid) * a.gp.k;
    const size_t smem = decode_smem_bytes(range_entries, a.gp.E, a.epr, warp_floats);
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
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kDecThreads), args, smem, st);
}

}  // namespace


size_t decode_max_entries() { return kMaxEntries; }

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
    a.spin_limit = kGridSpinLimit;
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
    // the check starts from cleared words (a timed-out barrier leaves them mid-way)
    cudaError_t e = cudaMemsetAsync(barrier_word, 0, 2 * sizeof(unsigned), st);
    if (e != cudaSuccess)
        return e;
    unsigned *counter = static_cast<unsigned *>(barrier_word);
    void *args[] = {&counter, &extra, &spin_limit, &err_flag};
    return cudaLaunchCooperativeKernel((const void *)barrier_selftest_kernel, dim3(device_sm_count()),
                                       dim3(kDecThreads), args, 0, st);
}

}  // namespace ep
