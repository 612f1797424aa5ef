// ep_internal.cuh -- shared device helpers and kernel launchers of the
// MoE dispatch/combine library (sm_103a).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace ep {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

// Order-preserving map of a binary32 value onto uint32: a < b as floats
// iff key(a) < key(b) as integers.  -0.0 maps like +0.0 so that equal floats
// give equal keys (ties are then broken by index).  NaN inputs are
// unsupported.
__device__ __forceinline__ uint32_t ordered_key(float v)
{
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two bf16 (round to nearest even) packed lo | hi << 16.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 values -> two e4m3 codes (round to nearest even, saturating to
// the largest finite magnitude) packed lo | hi << 8.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Two fp32 values in one 64-bit register (low, high) for the packed fp32x2
// arithmetic of sm_100-family GPUs: each lane of a packed op is the IEEE
// round-to-nearest-even result of the scalar op, so packing changes no bit.
// The largest magnitude of the 16 bf16 values in a and b, as fp32: a tree
// of packed max-of-magnitude operations on the bf16 pairs (the sign of each
// result is not used), then the larger half.  Exact: every candidate is one
// of the inputs' magnitudes.
__device__ __forceinline__ float bf16x16_amax(const uint4 &a, const uint4 &b)
{
    uint32_t m0, m1, m2, m3;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m0) : "r"(a.x), "r"(a.y));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m1) : "r"(a.z), "r"(a.w));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(b.x), "r"(b.y));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m3) : "r"(b.z), "r"(b.w));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m0) : "r"(m0), "r"(m1));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(m3));
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m0) : "r"(m0), "r"(m2));
    return fmaxf(__uint_as_float((m0 << 16) & 0x7FFF0000u), __uint_as_float(m0 & 0x7FFF0000u));
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 16-byte global load that bypasses L1 allocation (each byte is read once).
// Warp numbering of the persistent warp kernels: warp w of CTA b is global
// warp w * gridDim.x + b, so consecutive work units (tokens, row segments)
// go to different CTAs -- with a grid of whole waves, to different SMs --
// and every CTA gets the same share of them to within one unit.  (Numbered
// CTA by CTA, a grid smaller than a full wave left some SMs a CTA more
// than others, a third more work on Mixtral-sized batches.)
__device__ __forceinline__ long long balanced_warp()
{
    return (long long)(threadIdx.x >> 5) * gridDim.x + blockIdx.x;
}
__device__ __forceinline__ long long grid_warps() { return ((long long)gridDim.x * blockDim.x) >> 5; }

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte global store with the streaming (evict-first) cache hint.
__device__ __forceinline__ void st_stream16(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Plain 16-byte global store (default L2 policy).  Measured on GB300 it is
// slightly faster than the streaming hint for the k-fold scatter stores of
// the dispatch, whose rows are completed by neighbouring warps while still
// in L2.
__device__ __forceinline__ void st_plain16(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Lanes of the warp whose key equals this lane's key, for keys in
// [0, 2^nbits): one ballot per key bit (every lane must call it).  Unlike
// __match_any_sync its cost does not grow with the number of distinct keys.
__device__ __forceinline__ unsigned peer_mask(unsigned key, int nbits)
{
    unsigned m = kFullMask;
    for (int b = 0; b < nbits; ++b) {
        const unsigned bit = (key >> b) & 1u;
        const unsigned bal = __ballot_sync(kFullMask, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

// Bits needed for keys 0..max_key.
__host__ __device__ __forceinline__ int key_bits(unsigned max_key)
{
    int b = 1;
    while ((max_key >> b) != 0u)
        ++b;
    return b;
}

// Warp-aggregated shared-memory increment of cnt[key] for the active lanes
// (every lane must call it; inactive lanes pass any key).
__device__ __forceinline__ void warp_count(int32_t *cnt, unsigned key, bool active, int nbits)
{
    const unsigned act = __ballot_sync(kFullMask, active);
    const unsigned peers = peer_mask(key, nbits) & act;
    if (active && (threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1))
        atomicAdd(&cnt[key], __popc(peers));
}

struct GateParams {
    int E, k, G, Kg, kin, score_fn, normalize;
};

// Launchers (return the launch's cudaGetLastError()).
cudaError_t launch_gate(const float *scores, const float *bias, int T, const GateParams &p,
                        int32_t *topk_idx, float *topk_w, cudaStream_t st);

// Whether launch_gate takes the lane-segment kernel (gate_fast.cuh) for
// this configuration and these pointers; the warp-per-token kernel serves
// the rest.
bool gate_fast_supported(const GateParams &p, const float *scores, const float *bias);

// The dispatch layout (capacity mode when cap >= 0) by one thread-block
// cluster in one launch, with no workspace (layout_cluster.cu).  Launched
// with programmatic stream serialisation.  supported() says whether this
// device and these sizes fit it; the launch returns cudaErrorNotSupported
// otherwise.
bool layout_cluster_supported(int T, int k, int E, int epr);
cudaError_t launch_layout_cluster(const int32_t *topk_idx, int T, int k, int E, int epr, int cap,
                                  int32_t *expert_count, int32_t *expert_off, int32_t *rank_count,
                                  int32_t *rank_off, int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos,
                                  int32_t *src, int32_t *err_flag, cudaStream_t st);

int layout_tile_tokens(int k);
int layout_num_tiles(int T, int k);
size_t layout_workspace_bytes(int T, int k, int E, int epr);
cudaError_t launch_layout(const int32_t *topk_idx, int T, int k, int E, int epr, int32_t *expert_count,
                          int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                          int32_t *rank_tokens, int32_t *pos, int32_t *src, int32_t *err_flag,
                          void *workspace, cudaStream_t st);

cudaError_t launch_layout_capacity(const int32_t *topk_idx, int T, int k, int E, int epr, int cap,
                                   int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                                   int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos, int32_t *src,
                                   int32_t *err_flag, void *workspace, cudaStream_t st);

// rows: receive-buffer rows; a pos at or past it is skipped and flagged.
cudaError_t launch_dispatch_bf16(const uint16_t *x, int T, int H, int k, const int32_t *pos,
                                 uint16_t *recv, long long rows, int32_t *err_flag, cudaStream_t st);
cudaError_t launch_dispatch_fp8(const uint16_t *x, int T, int H, int k, const int32_t *pos,
                                uint8_t *recv_q, float *recv_s, long long rows, int32_t *err_flag, cudaStream_t st);

cudaError_t launch_dispatch_mxfp8(const uint16_t *x, int T, int H, int k, const int32_t *pos, uint8_t *recv_q,
                                  uint8_t *recv_e, long long rows, int32_t *err_flag, cudaStream_t st);

// w == NULL: unit weights (the backward of the BF16 dispatch).
cudaError_t launch_combine(const uint16_t *y, long long rows, const int32_t *pos, const float *w, int T, int H,
                           int k, uint16_t *out, int32_t *err_flag, cudaStream_t st);
cudaError_t launch_combine_fp8(const uint8_t *yq, const void *yscale, int mx, long long rows, const int32_t *pos,
                               const float *w, int T, int H, int k, uint16_t *out, int32_t *err_flag, cudaStream_t st);

cudaError_t launch_combine_backward(const uint16_t *grad_out, const uint16_t *y, long long rows, const int32_t *pos,
                                    const float *w, int T, int H, int k, uint16_t *grad_y, float *grad_w,
                                    int32_t *err_flag, cudaStream_t st);

size_t decode_max_entries();
cudaError_t launch_decode(const float *scores, const float *bias, int T, const GateParams &gp, int epr,
                          const uint16_t *x, int H, int dtype, int32_t *topk_idx, float *topk_w,
                          int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
                          int32_t *rank_tokens, int32_t *pos, int32_t *src, void *recv, void *recv_scales,
                          long long rows, int32_t *err_flag, void *barrier_word, cudaStream_t st);
cudaError_t launch_barrier_selftest(unsigned extra, long long spin_limit, int32_t *err_flag, void *barrier_word,
                                    cudaStream_t st);
// Gating and layout of a decode-sized batch (T <= 512, T*k <= 4096) in one
// clustered launch with no grid barrier (decode.cu): results equal
// launch_gate then launch_layout.
bool gate_layout_small_supported(int T, int k);
cudaError_t launch_gate_layout_small(const float *scores, const float *bias, int T, const GateParams &gp, int epr,
                                     int32_t *topk_idx, float *topk_w, int32_t *expert_count, int32_t *expert_off,
                                     int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens, int32_t *pos,
                                     int32_t *src, cudaStream_t st);

// Gating (gp != NULL: scores -> topk_idx, topk_w, with the lane-segment
// body) and the layout of the chosen experts, or the layout of topk_idx_in
// (gp == NULL; capacity mode when cap >= 0) -- one cooperative launch
// (route.cu).  workspace: at least route_workspace_bytes(E), 16-byte
// aligned; its first word (the grid barrier's arrival count) zero, and left
// zero by every call that completes.  route_supported says whether the
// sizes fit one grid of one CTA per SM (and, when gating, whether the
// lane-segment body serves the configuration).
size_t route_workspace_bytes(int E);
bool route_supported(int T, int k, int E, int epr, bool gate);
// The grid and cluster size the cooperative routing launch takes for T tokens.
void route_launch_shape(int T, int *grid, int *cluster);

// Layouts of at most this many entries (T*k) run as one kernel on one CTA.
constexpr int kSmallLayoutEntries = 4096;
// Layouts of at most this many entries take the one-cluster kernel.
constexpr long long kClusterLayoutEntries = 65536;
cudaError_t launch_route(const float *scores, const float *bias, const GateParams *gp, const int32_t *topk_idx_in,
                         int32_t *topk_idx, float *topk_w, int T, int k, int E, int epr, int32_t *expert_count,
                         int32_t *expert_off, int32_t *rank_count, int32_t *rank_off, int32_t *rank_tokens,
                         int32_t *pos, int32_t *src, int32_t *err_flag, void *workspace, cudaStream_t st,
                         int cap = -1, int32_t *expert_dropped = nullptr);

int device_sm_count();

// The current device, or -1 if it cannot be read.
int current_device();

constexpr int kMaxDevices = 64;

// Host-side values worth computing once per device: a kernel attribute that
// has been raised (cudaFuncSetAttribute acts per device), an occupancy
// figure, the SM count.  Slot [device][key] holds a positive value once
// computed.  The slots are atomics, so host threads may call concurrently; a
// first use on two threads at once computes the value twice, which is
// harmless because both get the same value.  A device past kMaxDevices is
// served by computing every time.
template <int kKeys = 1>
struct PerDeviceCache {
    std::atomic<int> v[kMaxDevices][kKeys];

    // The cached value for (current device, key), else f(): cached when > 0,
    // returned uncached otherwise (a failure is retried on the next call).
    template <class F>
    int get(F &&f, int key = 0)
    {
        const int d = current_device();
        if (d < 0 || d >= kMaxDevices || key < 0 || key >= kKeys)
            return f();
        int x = v[d][key].load(std::memory_order_acquire);
        if (x > 0)
            return x;
        x = f();
        if (x > 0)
            v[d][key].store(x, std::memory_order_release);
        return x;
    }
};

// Resident CTAs per SM of `kernel` at this block size and dynamic shared
// memory (at least 1), cached per device in slot `key` of `cache`.
template <int kKeys>
inline int occupancy_per_sm(PerDeviceCache<kKeys> &cache, const void *kernel, int threads, size_t smem, int key = 0)
{
    return cache.get(
        [&] {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            return per_sm;
        },
        key);
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device.  Returns the CUDA error of the first failing try.
inline cudaError_t raise_smem_limit(PerDeviceCache<1> &cache, const void *kernel, size_t bytes)
{
    cudaError_t err = cudaSuccess;
    cache.get([&] {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        return err == cudaSuccess ? 1 : 0;
    });
    return err;
}

// Launch shape of the CTA-per-row kernels (defined in combine.cu): a grid
// of every resident CTA (occupancy cached per device and block size in
// `cache`), at most one per row.
int chunk_threads(int c, int k);
int row_grid(const void *kern, int threads, int T, PerDeviceCache<33> &cache);

}  // namespace ep
