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
// bytes in, 2Hk out; FP8: 2H in, k(H + H/32) out).  The standalone calls use
// the bulk-copy kernel below (rows staged in shared memory, copies issued as
// cp.async.bulk transfers); rows too long to stage, and the fused decode
// path, use the warp-item bodies.  Warp-item path: work is split into warp
// items -- one token's row segment of 32 lanes x 16 bytes (x U) -- handed out
// grid-stride to a persistent grid of (resident CTAs per SM) x (SMs).  There
// is no block barrier: lane j of the warp holds the token's j-th receive row
// (and lane j of a second register slot j+32) and shuffles it to the others,
// so every warp streams independently.  Loads bypass L1; stores are plain.
// The row is held in registers and never re-read per copy.
// FP8: 8 consecutive lanes own one 128-column block (16 columns each); the
// block's amax is a 3-step xor-shuffle max, the scale an IEEE fp32 division
// by 448, each code the IEEE fp32 quotient x / s (formed without a division
// per element; see fp8_quant16_regs) then a round-to-nearest-even saturating
// e4m3 conversion (cvt.rn.satfinite).
#include "dispatch_impl.cuh"

namespace ep {

namespace {

constexpr int kDispThreads = 256;

// The item kernels are software-pipelined: a warp issues the next item's
// row and pos loads before it checks, converts and stores the current one,
// so the check of pos (a branch on a loaded value, which stalls in-order
// issue) and the row loads of one item never form two round trips in a row.
__global__ void __launch_bounds__(kDispThreads) dispatch_bf16_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                     int k, const int32_t *__restrict__ pos,
                                                                     uint16_t *__restrict__ recv, long long rows,
                                                                     int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    ItemWalk it(T, bf16_segs(H));
    if (!it.valid())
        return;
    int p0, p1;
    uint4 v[kBf16Unroll];
    load_token_rows(pos, it.t, k, lane, p0, p1);
    bf16_item_load(x, H, it.t, it.seg, v);
    for (;;) {
        ItemWalk nx = it;
        nx.next();
        const bool more = nx.valid();  // warp-uniform
        int n0 = -1, n1 = -1;
        uint4 nv[kBf16Unroll];
        if (more) {
            load_token_rows(pos, nx.t, k, lane, n0, n1);
            bf16_item_load(x, H, nx.t, nx.seg, nv);
        }
        check_token_rows(rows, err_flag, p0, p1);
        bf16_item_store(H, k, it.seg, p0, p1, v, recv);
        if (!more)
            break;
        it = nx;
        p0 = n0;
        p1 = n1;
#pragma unroll
        for (int u = 0; u < kBf16Unroll; ++u)
            v[u] = nv[u];
    }
}

__global__ void __launch_bounds__(kDispThreads) dispatch_fp8_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                    int k, const int32_t *__restrict__ pos,
                                                                    uint8_t *__restrict__ recv_q,
                                                                    float *__restrict__ recv_s, long long rows,
                                                                    int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    ItemWalk it(T, fp8_segs(H));
    if (!it.valid())
        return;
    int p0, p1;
    uint4 a, b;
    load_token_rows(pos, it.t, k, lane, p0, p1);
    q8_item_load(x, H, it.t, it.seg, a, b);
    for (;;) {
        ItemWalk nx = it;
        nx.next();
        const bool more = nx.valid();  // warp-uniform
        int n0 = -1, n1 = -1;
        uint4 na = make_uint4(0, 0, 0, 0), nb = make_uint4(0, 0, 0, 0);
        if (more) {
            load_token_rows(pos, nx.t, k, lane, n0, n1);
            q8_item_load(x, H, nx.t, nx.seg, na, nb);
        }
        check_token_rows(rows, err_flag, p0, p1);
        fp8_item_store(H, k, it.seg, p0, p1, a, b, recv_q, recv_s);
        if (!more)
            break;
        it = nx;
        p0 = n0;
        p1 = n1;
        a = na;
        b = nb;
    }
}

// FP8 / MXFP8 for few slots per token (k <= kQ8RowMaxK, Mixtral-like
// routing): a warp walks whole tokens, their row segments in order, so a
// token's receive rows are loaded and shuffled to the lanes once (kept in
// registers) rather than once per segment, and the segment loop carries no
// token bookkeeping; the next segment's row load (and at a token's last
// segment, the next token's pos) is issued before the current one is
// converted and stored.  The same per-segment arithmetic as the item
// kernels (fp8_quant16_regs, mx_quant16_regs).
constexpr int kQ8RowMaxK = 4;

template <bool kMx>
__global__ void __launch_bounds__(kDispThreads) dispatch_q8_rows_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                        int k, const int32_t *__restrict__ pos,
                                                                        uint8_t *__restrict__ recv_q,
                                                                        void *__restrict__ recv_sc, long long rows,
                                                                        int32_t *__restrict__ err_flag)
{
    const int lane = threadIdx.x & 31;
    const long long nw = grid_warps();
    long long t = balanced_warp();
    if (t >= T)
        return;
    const int segs = fp8_segs(H);
    const int C16 = H / 16;
    const int nb = kMx ? H / 32 : H / 128;
    int pl = lane < k ? __ldg(pos + t * k + lane) : -1;  // slot `lane`'s row, as loaded
    int seg = 0;
    uint4 a, b;
    q8_item_load(x, H, t, 0, a, b);
    for (;;) {
        // this token's rows, checked, in every lane
        int p[kQ8RowMaxK];
        if (pl >= rows) {
            if (err_flag)
                atomicOr(err_flag, 2);
            pl = -1;
        }
#pragma unroll
        for (int j = 0; j < kQ8RowMaxK; ++j)
            p[j] = __shfl_sync(kFullMask, pl, j);
        for (;;) {
            const bool last_seg = seg + 1 == segs;
            const long long tn = last_seg ? t + nw : t;
            const int sn = last_seg ? 0 : seg + 1;
            const bool more = tn < T;  // warp-uniform
            uint4 na = make_uint4(0, 0, 0, 0), nb4 = make_uint4(0, 0, 0, 0);
            if (more)
                q8_item_load(x, H, tn, sn, na, nb4);
            if (more && last_seg)
                pl = lane < k ? __ldg(pos + tn * k + lane) : -1;
            const int c = seg * 32 + lane;
            const bool act = c < C16;
            float s = 0.0f;
            uint8_t eb = 0;
            const uint4 qv = kMx ? mx_quant16_regs(a, b, eb) : fp8_quant16_regs(a, b, s);
            if (act) {
#pragma unroll
                for (int j = 0; j < kQ8RowMaxK; ++j) {
                    if (j >= k || p[j] < 0)
                        continue;
                    st_plain16(recv_q + (size_t)p[j] * H + (size_t)c * 16, qv);
                    if (kMx) {
                        if ((c & 1) == 0)
                            static_cast<uint8_t *>(recv_sc)[(size_t)p[j] * nb + (c >> 1)] = eb;
                    } else if ((c & 7) == 0) {
                        static_cast<float *>(recv_sc)[(size_t)p[j] * nb + (c >> 3)] = s;
                    }
                }
            }
            if (!more)
                return;
            t = tn;
            seg = sn;
            a = na;
            b = nb4;
            if (last_seg)
                break;
        }
    }
}

// The same walk with kQ8Depth row segments in flight per warp (MXFP8, whose
// conversion is light enough that the walk waits on its loads; the FP8
// conversion keeps the issue slots busy and gains nothing): each lane
// copies its 32 bytes of the next segments into a per-warp ring in shared
// memory with cp.async (no registers held), waits for the oldest with
// cp.async.wait_group and reads back only what it copied itself (so no
// warp barrier is needed).  Mixtral shape: 9.4 -> 8.6 us a call back to
// back (FP8 with the ring: 10.9 -> 11.5, so FP8 keeps the register walk).
// Needs fp8_segs(H) >= kQ8Depth, so
// that the copies in flight span at most the next token, whose pos is then
// the one prefetched.
constexpr int kQ8Depth = 4;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool act)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = act ? 16 : 0;  // src-size 0: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}

template <bool kMx>
__global__ void __launch_bounds__(kDispThreads) dispatch_q8_ring_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                        int k, const int32_t *__restrict__ pos,
                                                                        uint8_t *__restrict__ recv_q,
                                                                        void *__restrict__ recv_sc, long long rows,
                                                                        int32_t *__restrict__ err_flag)
{
    __shared__ __align__(16) uint4 ring[kDispThreads / 32][kQ8Depth][32][2];
    const int lane = threadIdx.x & 31;
    uint4(*my)[32][2] = ring[threadIdx.x >> 5];
    const long long nw = grid_warps();
    const long long t0 = balanced_warp();
    if (t0 >= T)
        return;
    const int segs = fp8_segs(H);
    const int C16 = H / 16;
    const int nb = kMx ? H / 32 : H / 128;
    // producer position (the next segment to copy) and consumer position
    long long tp = t0, tc = t0;
    int sp = 0, sc = 0;
    int pl_next = -1;  // pos of the producer's token when it is ahead of the consumer's
    auto issue = [&](int slot) {
        if (tp < T) {
            const int c = sp * 32 + lane;
            const bool act = c < C16;
            const uint16_t *src = x + (size_t)tp * H + (size_t)(act ? c : 0) * 16;
            cp_async16(&my[slot][lane][0], src, act);
            cp_async16(&my[slot][lane][1], src + 8, act);
            if (sp == 0 && tp != tc)
                pl_next = lane < k ? __ldg(pos + tp * k + lane) : -1;
            if (++sp == segs) {
                sp = 0;
                tp += nw;
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");  // an empty group past the end keeps the count
    };
    int pl = lane < k ? __ldg(pos + tc * k + lane) : -1;
#pragma unroll
    for (int d = 0; d < kQ8Depth; ++d)
        issue(d);
    int p[kQ8RowMaxK];
    int slot = 0;
    for (;;) {
        if (sc == 0) {  // the consumer enters token tc: its checked rows in every lane
            if (pl >= rows) {
                if (err_flag)
                    atomicOr(err_flag, 2);
                pl = -1;
            }
#pragma unroll
            for (int j = 0; j < kQ8RowMaxK; ++j)
                p[j] = __shfl_sync(kFullMask, pl, j);
        }
        asm volatile("cp.async.wait_group %0;" ::"n"(kQ8Depth - 1) : "memory");
        const uint4 a = my[slot][lane][0], b = my[slot][lane][1];
        const int c = sc * 32 + lane;
        const bool act = c < C16;
        float s = 0.0f;
        uint8_t eb = 0;
        const uint4 qv = kMx ? mx_quant16_regs(a, b, eb) : fp8_quant16_regs(a, b, s);
        if (act) {
#pragma unroll
            for (int j = 0; j < kQ8RowMaxK; ++j) {
                if (j >= k || p[j] < 0)
                    continue;
                st_plain16(recv_q + (size_t)p[j] * H + (size_t)c * 16, qv);
                if (kMx) {
                    if ((c & 1) == 0)
                        static_cast<uint8_t *>(recv_sc)[(size_t)p[j] * nb + (c >> 1)] = eb;
                } else if ((c & 7) == 0) {
                    static_cast<float *>(recv_sc)[(size_t)p[j] * nb + (c >> 3)] = s;
                }
            }
        }
        // the slot is consumed (this lane read its own copies): refill it
        issue(slot);
        slot = slot + 1 == kQ8Depth ? 0 : slot + 1;
        if (++sc == segs) {
            sc = 0;
            tc += nw;
            if (tc >= T)
                break;
            pl = pl_next;
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
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
    ItemWalk it(T, fp8_segs(H));
    if (!it.valid())
        return;
    int p0, p1;
    uint4 a, b;
    load_token_rows(pos, it.t, k, lane, p0, p1);
    q8_item_load(x, H, it.t, it.seg, a, b);
    for (;;) {
        ItemWalk nx = it;
        nx.next();
        const bool more = nx.valid();  // warp-uniform
        int n0 = -1, n1 = -1;
        uint4 na = make_uint4(0, 0, 0, 0), nb = make_uint4(0, 0, 0, 0);
        if (more) {
            load_token_rows(pos, nx.t, k, lane, n0, n1);
            q8_item_load(x, H, nx.t, nx.seg, na, nb);
        }
        check_token_rows(rows, err_flag, p0, p1);
        mxfp8_item_store(H, k, it.seg, p0, p1, a, b, recv_q, recv_e);
        if (!more)
            break;
        it = nx;
        p0 = n0;
        p1 = n1;
        a = na;
        b = nb;
    }
}

// Bulk-copy dispatch: a CTA stages one token's receive row in shared memory
// (the BF16 row as is, or its FP8 / MXFP8 codes and scales, computed there
// once), then one thread issues the k copies as cp.async.bulk
// shared->global transfers -- whole rows handed to the copy engine instead
// of 16-byte stores from every lane.  Two staging buffers alternate, so the
// next token is loaded and quantised while the previous token's copies are
// in flight (a bulk group is waited for, reads only, before its buffer is
// reused).  Scale rows that are not a multiple of 16 bytes, or whose buffer
// is not 16-byte aligned, are written with plain stores instead.
constexpr int kBulkThreads = 256;
constexpr int kBulkMaxK = 64;

__device__ __forceinline__ void bulk_s2g(void *dst, unsigned src_smem, unsigned bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}

template <int kMode>  // 0: BF16, 1: FP8 e4m3 1x128 (fp32 scales), 2: MXFP8 1x32 (E8M0 scales)
__global__ void __launch_bounds__(kBulkThreads) dispatch_bulk_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                                      int k, const int32_t *__restrict__ pos,
                                                                      uint8_t *__restrict__ recv,
                                                                      uint8_t *__restrict__ recv_sc, int bulk_sc,
                                                                      long long rows, int32_t *__restrict__ err_flag)
{
    extern __shared__ __align__(128) unsigned char bsm[];
    __shared__ int32_t s_pos[2][kBulkMaxK];
    const int row_bytes = kMode == 0 ? 2 * H : H;
    const int nsc = kMode == 1 ? H / 128 : H / 32;        // scales per row
    const int sc_bytes = kMode == 0 ? 0 : H / 32;         // fp32 per 128 columns or one byte per 32
    const int stage = row_bytes + ((sc_bytes + 15) & ~15);
    int buf = 0;
    for (long long t = blockIdx.x; t < T; t += gridDim.x, buf ^= 1) {
        unsigned char *row = bsm + (size_t)buf * stage;
        unsigned char *sc = row + row_bytes;
        // this buffer was last read by the copies of two tokens ago
        if (threadIdx.x == 0)
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        if ((int)threadIdx.x < k) {
            int p = __ldg(pos + t * k + threadIdx.x);
            if (p >= rows) {
                if (err_flag)
                    atomicOr(err_flag, 2);
                p = -1;
            }
            s_pos[buf][threadIdx.x] = p;
        }
        const uint16_t *xrow = x + (size_t)t * H;
        if (kMode == 0) {
            for (int c = threadIdx.x; c < H / 8; c += kBulkThreads)
                reinterpret_cast<uint4 *>(row)[c] = ld_stream16(xrow + (size_t)c * 8);
        } else {
            const int C16 = H / 16;
            for (int c0 = 0; c0 < C16; c0 += kBulkThreads) {  // whole warps in every pass
                const int c = c0 + threadIdx.x;
                const bool act = c < C16;
                if (kMode == 1) {
                    float sv;
                    const uint4 q = fp8_quant16(xrow, c, act, sv);
                    if (act) {
                        reinterpret_cast<uint4 *>(row)[c] = q;
                        if ((c & 7) == 0)
                            reinterpret_cast<float *>(sc)[c >> 3] = sv;
                    }
                } else {
                    uint8_t ev;
                    const uint4 q = mx_quant16(xrow, c, act, ev);
                    if (act) {
                        reinterpret_cast<uint4 *>(row)[c] = q;
                        if ((c & 1) == 0)
                            sc[c >> 1] = ev;
                    }
                }
            }
        }
        // the staged row is read by the copy engine (the async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned srow = (unsigned)__cvta_generic_to_shared(row);
            const unsigned ssc = (unsigned)__cvta_generic_to_shared(sc);
            for (int j = 0; j < k; ++j) {
                const int p = s_pos[buf][j];
                if (p < 0)
                    continue;
                bulk_s2g(recv + (size_t)p * row_bytes, srow, (unsigned)row_bytes);
                if (kMode != 0 && bulk_sc)
                    bulk_s2g(recv_sc + (size_t)p * sc_bytes, ssc, (unsigned)sc_bytes);
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (kMode != 0 && !bulk_sc) {
            for (int i = threadIdx.x; i < k * nsc; i += kBulkThreads) {
                const int j = i / nsc, b = i - j * nsc;
                const int p = s_pos[buf][j];
                if (p < 0)
                    continue;
                if (kMode == 1)
                    reinterpret_cast<float *>(recv_sc)[(size_t)p * nsc + b] = reinterpret_cast<const float *>(sc)[b];
                else
                    recv_sc[(size_t)p * nsc + b] = sc[b];
            }
        }
    }
    // the copies must have completed (written, not only read) before exit
    if (threadIdx.x == 0)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Staging bytes of the bulk-copy kernel (two rows plus their scales).
size_t bulk_smem(int H, int mode)
{
    const size_t row_bytes = mode == 0 ? 2 * (size_t)H : (size_t)H;
    const size_t sc_bytes = mode == 0 ? 0 : (size_t)H / 32;
    return 2 * (row_bytes + ((sc_bytes + 15) & ~(size_t)15));
}

// The bulk-copy kernel pays a staging round trip per token, repaid by the
// k copies it hands to the copy engine: measured on GB300 it wins at k >= 4
// on full batches (DeepSeek-V3 and Qwen3 shapes: FP8 3-9 % faster, BF16 up
// to 4 %) and loses at k = 2 (Mixtral shape) and on decode-sized batches,
// which keep the warp-item kernels -- as do rows too long to stage twice in
// shared memory.
constexpr size_t kBulkMaxSmem = 200 * 1024;

bool use_bulk(int T, int H, int k, int mode)
{
    return k >= 4 && T >= 2048 && bulk_smem(H, mode) <= kBulkMaxSmem;
}

template <int kMode>
cudaError_t launch_bulk(const uint16_t *x, int T, int H, int k, const int32_t *pos, void *recv, void *recv_sc,
                        long long rows, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    const int sc_bytes = kMode == 0 ? 0 : H / 32;
    const size_t smem = bulk_smem(H, kMode);
    const int bulk_sc = kMode != 0 && sc_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(recv_sc) & 15) == 0;
    const void *fn = (const void *)dispatch_bulk_kernel<kMode>;
    static PerDeviceCache<1> attr;  // per mode: the largest staging use_bulk admits, once per device
    const cudaError_t ae = raise_smem_limit(attr, fn, kBulkMaxSmem);
    if (ae != cudaSuccess)
        return ae;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBulkThreads, smem);
    if (e != cudaSuccess)
        return e;
    const int cap = kMode == 0 ? 2 : 4;  // CTAs per SM: in flight rows vs. staging latency (measured)
    per_sm = per_sm < 1 ? 1 : (per_sm > cap ? cap : per_sm);
    const long long g = (long long)device_sm_count() * per_sm;
    const int grid = (int)(g < T ? g : T);
    dispatch_bulk_kernel<kMode><<<grid, kBulkThreads, smem, st>>>(
        x, T, H, k, pos, static_cast<uint8_t *>(recv), static_cast<uint8_t *>(recv_sc), bulk_sc, rows, err_flag);
    return cudaGetLastError();
}

// A persistent grid of (resident CTAs per SM) x (SMs), capped at one CTA per
// warp item (the warps are numbered across CTAs, balanced_warp, so a small
// batch spreads over as many SMs as it has items); the occupancy is cached
// per device.
int persistent_grid(const void *kernel, PerDeviceCache<1> &per_sm_cache, long long warp_items)
{
    const int per_sm = occupancy_per_sm(per_sm_cache, kernel, kDispThreads, 0);
    const long long g = (long long)device_sm_count() * per_sm;
    return (int)(warp_items < g ? warp_items : g);
}

PerDeviceCache<1> g_bf16_per_sm;
PerDeviceCache<1> g_fp8_per_sm;
PerDeviceCache<1> g_mx_per_sm;
PerDeviceCache<1> g_fp8_rows_per_sm;
PerDeviceCache<1> g_mx_rows_per_sm;
PerDeviceCache<1> g_mx_ring_per_sm;

}  // namespace

cudaError_t launch_dispatch_mxfp8(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint8_t *recv_q,
                                  uint8_t *recv_e, long long rows, int32_t *err_flag, cudaStream_t st)
{
    if (T == 0)
        return cudaSuccess;
    if (use_bulk(T, H, k, 2))
        return launch_bulk<2>(x, T, H, k, pos, recv_q, recv_e, rows, err_flag, st);
    if (k <= kQ8RowMaxK && fp8_segs(H) >= kQ8Depth) {
        const int grid = persistent_grid((const void *)dispatch_q8_ring_kernel<true>, g_mx_ring_per_sm, T);
        dispatch_q8_ring_kernel<true><<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_e, rows, err_flag);
        return cudaGetLastError();
    }
    if (k <= kQ8RowMaxK) {
        const int grid = persistent_grid((const void *)dispatch_q8_rows_kernel<true>, g_mx_rows_per_sm, T);
        dispatch_q8_rows_kernel<true><<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_e, rows, err_flag);
        return cudaGetLastError();
    }
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
    if (use_bulk(T, H, k, 0))
        return launch_bulk<0>(x, T, H, k, pos, recv, nullptr, rows, err_flag, st);
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
    if (use_bulk(T, H, k, 1))
        return launch_bulk<1>(x, T, H, k, pos, recv_q, recv_s, rows, err_flag, st);
    if (k <= kQ8RowMaxK) {
        const int grid = persistent_grid((const void *)dispatch_q8_rows_kernel<false>, g_fp8_rows_per_sm, T);
        dispatch_q8_rows_kernel<false><<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_s, rows,
                                                                      err_flag);
        return cudaGetLastError();
    }
    const long long items = (long long)T * fp8_segs(H);
    const int grid = persistent_grid((const void *)dispatch_fp8_kernel, g_fp8_per_sm, items);
    dispatch_fp8_kernel<<<grid, kDispThreads, 0, st>>>(x, T, H, k, pos, recv_q, recv_s, rows, err_flag);
    return cudaGetLastError();
}

}  // namespace ep
