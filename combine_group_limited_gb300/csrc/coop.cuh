// coop.cuh -- helpers of the kernels whose CTAs work together: the bounded
// grid barrier of the cooperative kernels, and the thread-block cluster
// primitives (rank, barrier halves, distributed shared memory) of the
// clustered ones.  Not part of the public ABI.
#pragma once

#include "ep_internal.cuh"

namespace ep {
namespace {

// Polls of a grid barrier before it gives up (each poll sleeps ~32 ns
// plus the load; about a second of polling in all).
constexpr long long kGridSpinLimit = 1LL << 21;

// All CTAs of a cooperative grid arrive once; the wait is bounded.
// word[0] counts arrivals and is zero when the launch starts.  Each CTA adds
// one with acquire-release semantics (its writes, and those its threads made
// before the block barrier, become visible first) and learns its arrival
// number n.  The last to arrive (n == expected) puts the count back to zero
// with another read-modify-write, so the word is ready for the next launch
// with no clearing in between, and an acquire load of either value sees
// every CTA's writes.  The others poll the count with acquire loads until it
// equals `expected` or drops below n (the reset: every CTA has arrived; the
// count only grows until then, and the next launch cannot start before this
// one ends).  Returns false, with EP_FLAG_TIMEOUT set, if the limit ran out
// (the count is then left non-zero and must be cleared again; a count that
// was not zero at launch runs out the same way, unless it was below
// `expected`).
__device__ __forceinline__ bool grid_barrier(unsigned *word, unsigned expected, long long spin_limit,
                                             int32_t *err_flag)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned old;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(word) : "memory");
        const unsigned n = old + 1u;
        bool ok = true;
        if (n == expected) {
            atomicExch(word, 0u);  // a read-modify-write: it continues every arrival's release sequence
        } else {
            ok = false;
            for (long long it = 0; it < spin_limit; ++it) {
                unsigned c;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(word) : "memory");
                if (c == expected || c < n) {
                    ok = true;
                    break;
                }
                __nanosleep(32);
            }
        }
        s_ok = ok;
        if (!ok && err_flag)
            atomicOr(err_flag, 4);
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ unsigned cluster_ctarank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ unsigned cluster_nctarank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Index of this CTA's cluster in the (one-dimensional) grid of clusters.
__device__ __forceinline__ unsigned cluster_id_x()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Cluster-wide barrier halves: arrive releases this thread's prior writes
// (shared and global) to the cluster, wait acquires those of every thread
// that arrived.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Generic address of `local`'s counterpart in the shared memory of cluster
// CTA `rank`.
template <class V>
__device__ __forceinline__ const V *cluster_peer(const V *local, unsigned rank)
{
    uint64_t r;
    asm volatile("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
    return reinterpret_cast<const V *>(r);
}

// Stores v into `local`'s counterpart in the shared memory of cluster CTA
// `rank` (a 32-bit shared::cluster address; no reply is awaited).
__device__ __forceinline__ void cluster_store(int32_t *local, unsigned rank, int v)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// Programmatic dependent launch: wait for the grids this one depends on to
// complete (no-op without the launch attribute), and let dependent grids
// start their prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Inclusive warp scan.
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

}  // namespace
}  // namespace ep
