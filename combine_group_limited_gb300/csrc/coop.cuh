// coop.cuh -- helpers of the cooperative (grid-barrier) kernels: the fused
// decode path and the fused gating + layout.  Not part of the public ABI.
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
