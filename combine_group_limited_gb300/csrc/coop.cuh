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
// word[0] counts arrivals, word[1] is a generation number: the last CTA to
// arrive resets the count and advances the generation, which releases the
// others -- so the barrier leaves its two words ready for the next launch.
// Returns false, with EP_FLAG_TIMEOUT set, if the limit ran out (the words
// are then left mid-barrier and must be zeroed again).
__device__ __forceinline__ bool grid_barrier(unsigned *word, unsigned expected, long long spin_limit, int32_t *err_flag)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned *count = word, *gen = word + 1;
        unsigned g0;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g0) : "l"(gen) : "memory");
        __threadfence();  // this CTA's global writes before its arrival
        const unsigned arrived = atomicAdd(count, 1u) + 1u;
        bool ok = true;
        if (arrived == expected) {
            // release the others first; the count only has to be back at
            // zero before the next launch, which starts after this one ends
            atomicAdd(gen, 1u);
            atomicExch(count, 0u);
        } else {
            unsigned g = g0;
            long long it = 0;
            for (;;) {
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(gen) : "memory");
                if (g != g0 || ++it >= spin_limit)
                    break;
                __nanosleep(32);
            }
            ok = g != g0;
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
