// dispatch_impl.cuh -- per-item bodies of the permute-scatter, shared by the
// dispatch kernels and the fused low-latency decode kernel.
//
// "Expert Parallelism (Parallelisme d'experts)", section "Le pattern de
// communication all-to-all", Phase 1 Dispatch; FP8 modes from "DeepEP de
// DeepSeek ...", section "Support FP8 et MXFP8".  A warp item is one token's
// row segment: 32 lanes x 16 bytes (x kBf16Unroll for BF16) of x.  Lane j of
// the warp holds the token's j-th receive row in p0 (j + 32 in p1).
#pragma once

#include "ep_internal.cuh"

namespace ep {

constexpr int kBf16Unroll = 4;  // 16-byte chunks per lane per item (BF16)

// Receive rows of token t for the calling warp: slot `lane` in p0, slot
// `lane + 32` in p1; -1 where the slot does not exist, is empty, or names a
// row outside [0, rows) (flagged).
__device__ __forceinline__ void load_token_rows(const int32_t *__restrict__ pos, long long t, int k, int lane, int &p0,
                                                int &p1)
{
    p0 = -1;
    p1 = -1;
    if (lane < k)
        p0 = __ldg(pos + t * k + lane);
    if (lane + 32 < k)
        p1 = __ldg(pos + t * k + lane + 32);
}

__device__ __forceinline__ void check_token_rows(long long rows, int32_t *err_flag, int &p0, int &p1)
{
    if (p0 >= rows || p1 >= rows) {
        if (err_flag)
            atomicOr(err_flag, 2);
        if (p0 >= rows)
            p0 = -1;
        if (p1 >= rows)
            p1 = -1;
    }
}

__device__ __forceinline__ void token_rows(const int32_t *__restrict__ pos, long long t, int k, long long rows,
                                           int lane, int32_t *err_flag, int &p0, int &p1)
{
    load_token_rows(pos, t, k, lane, p0, p1);
    check_token_rows(rows, err_flag, p0, p1);
}

__device__ __forceinline__ int slot_row(int p0, int p1, int j)
{
    const int a = __shfl_sync(kFullMask, p0, j & 31);
    const int b = __shfl_sync(kFullMask, p1, j & 31);
    return j < 32 ? a : b;
}

// Walks warp items (token, segment) grid-stride without a division per item.
struct ItemWalk {
    long long t;
    int seg;
    int segs;
    long long T;
    int step_seg;
    long long step_t;

    __device__ ItemWalk(long long T_, int segs_)
    {
        T = T_;
        segs = segs_;
        // Items numbered across CTAs (balanced_warp) when there are few per
        // warp (small batches: spread over the SMs); CTA by CTA otherwise,
        // so that a CTA's warps take consecutive segments of the same tokens
        // (shared pos lines, contiguous rows).
        const long long nwarps = grid_warps();
        const long long warp = (long long)T * segs < 2 * nwarps
                                   ? balanced_warp()
                                   : (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
        t = warp / segs;
        seg = (int)(warp - t * segs);
        step_t = nwarps / segs;
        step_seg = (int)(nwarps - step_t * segs);
    }
    __device__ bool valid() const { return t < T; }
    __device__ void next()
    {
        t += step_t;
        seg += step_seg;
        if (seg >= segs) {
            seg -= segs;
            ++t;
        }
    }
};

// Items per token row.
__device__ __host__ __forceinline__ int bf16_segs(int H) { return (H / 8 + 32 * kBf16Unroll - 1) / (32 * kBf16Unroll); }
__device__ __host__ __forceinline__ int fp8_segs(int H) { return (H / 16 + 31) / 32; }

// BF16: recv[p_j, seg] = x[t, seg] for the token's k rows.  The load half
// and the store half are separate so that a kernel can issue the next item's
// loads before storing this one.
__device__ __forceinline__ void bf16_item_load(const uint16_t *__restrict__ x, int H, long long t, int seg,
                                               uint4 (&v)[kBf16Unroll])
{
    const int lane = threadIdx.x & 31;
    const int C = H / 8;  // 16-byte chunks per row
    const uint16_t *xrow = x + (size_t)t * H;
    const int c0 = seg * 32 * kBf16Unroll + lane;
#pragma unroll
    for (int u = 0; u < kBf16Unroll; ++u) {
        const int c = c0 + 32 * u;
        v[u] = c < C ? ld_stream16(xrow + (size_t)c * 8) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void bf16_item_store(int H, int k, int seg, int p0, int p1, const uint4 (&v)[kBf16Unroll],
                                                uint16_t *__restrict__ recv)
{
    const int lane = threadIdx.x & 31;
    const int C = H / 8;
    const int c0 = seg * 32 * kBf16Unroll + lane;
    for (int j = 0; j < k; ++j) {
        const int p = slot_row(p0, p1, j);
        if (p < 0)
            continue;
        uint16_t *dst = recv + (size_t)p * H;
#pragma unroll
        for (int u = 0; u < kBf16Unroll; ++u) {
            const int c = c0 + 32 * u;
            if (c < C)
                st_plain16(dst + (size_t)c * 8, v[u]);
        }
    }
}

__device__ __forceinline__ void dispatch_bf16_item(const uint16_t *__restrict__ x, int H, int k, long long t, int seg,
                                                   int p0, int p1, uint16_t *__restrict__ recv)
{
    uint4 v[kBf16Unroll];
    bf16_item_load(x, H, t, seg, v);
    bf16_item_store(H, k, seg, p0, p1, v, recv);
}

// FP8 e4m3 with one fp32 scale per 128 columns: the codes of the 16 columns
// [16c, 16c + 16) of row xrow and their block's scale s = amax / 448.  Eight
// consecutive lanes cover a block: every lane of the warp calls this (lanes
// with act == false contribute zeros).
// The 16 bf16 values [16c, 16c + 16) of row xrow as two 16-byte words
// (zeros where act is false).
__device__ __forceinline__ void load16(const uint16_t *__restrict__ xrow, int c, bool act, uint4 &a, uint4 &b)
{
    a = make_uint4(0, 0, 0, 0);
    b = make_uint4(0, 0, 0, 0);
    if (act) {
        a = ld_stream16(xrow + (size_t)c * 16);
        b = ld_stream16(xrow + (size_t)c * 16 + 8);
    }
}

// fp8_quant16's arithmetic on 16 values already loaded by load16.  The
// values are unpacked negated (one xor flips both signs of a bf16 pair) so
// that the quotient's three steps run as packed fp32x2 operations, whose
// operands cannot be negated in place: x*r is formed as (-x)*(-r), and the
// remainder and the correction take -x and -r; each product and sum is the
// same exact value as in the scalar form, so every rounding -- and the sign
// of a zero -- is the same.
__device__ __forceinline__ uint4 fp8_quant16_regs(const uint4 &a, const uint4 &b, float &s_out)
{
    const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float nf[16];  // -x
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t n = wv[i] ^ 0x80008000u;
        nf[2 * i] = bf16_lo(n);
        nf[2 * i + 1] = bf16_hi(n);
    }
    float amax = bf16x16_amax(a, b);
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
    } else if (s >= 0x1p-90f && s <= 0x1p125f) {
        // x / s without a division per element, by Markstein's correction
        // step (P. Markstein, "Computation of elementary functions on the IBM
        // RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
        // r the correctly rounded 1/s and q0 = x*r, the remainder e = s*q0 - x
        // is exact in one FMA, and q0 - e*r rounded once is the IEEE
        // quotient.  For bf16 x this holds for every pair of significands at
        // every exponent gap that gives a nonzero code (an exhaustive test
        // checks them all against IEEE division).  The scale range keeps r
        // normal and the remainder above fp32 underflow for every quotient
        // of 2^-11 or more; smaller quotients code to zero either way.  The
        // remainder's sign convention (s*q0 - x, then q0 - e*r) keeps the
        // sign of a zero x.
        const float r = __frcp_rn(s);
        const uint64_t s2 = f2_pack(s, s), nr2 = f2_pack(-r, -r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float d[4];
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                const uint64_t nx = f2_pack(nf[4 * i + j], nf[4 * i + j + 1]);
                const uint64_t q0 = f2_mul(nx, nr2);   // x * r
                const uint64_t e = f2_fma(q0, s2, nx);  // q0 * s - x, exact
                f2_unpack(f2_fma(e, nr2, q0), d[j], d[j + 1]);  // q0 - e * r
            }
            q[i] = pack_e4m3x2(d[0], d[1]) | (pack_e4m3x2(d[2], d[3]) << 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = pack_e4m3x2(__fdiv_rn(-nf[4 * i], s), __fdiv_rn(-nf[4 * i + 1], s));
            const uint32_t hi = pack_e4m3x2(__fdiv_rn(-nf[4 * i + 2], s), __fdiv_rn(-nf[4 * i + 3], s));
            q[i] = lo | (hi << 16);
        }
    }
    s_out = s;
    return make_uint4(q[0], q[1], q[2], q[3]);
}

__device__ __forceinline__ uint4 fp8_quant16(const uint16_t *__restrict__ xrow, int c, bool act, float &s_out)
{
    uint4 a, b;
    load16(xrow, c, act, a, b);
    return fp8_quant16_regs(a, b, s_out);
}

// The 16 columns a lane owns in item (t, seg) of an FP8 / MXFP8 dispatch.
__device__ __forceinline__ void q8_item_load(const uint16_t *__restrict__ x, int H, long long t, int seg, uint4 &a,
                                             uint4 &b)
{
    const int c = seg * 32 + (threadIdx.x & 31);
    load16(x + (size_t)t * H, c, c < H / 16, a, b);
}

// FP8 e4m3 with one fp32 scale per 128 columns: 8 lanes per block.  The
// store half takes the item's values from q8_item_load; fp8_item_put stores
// codes and scale already computed by fp8_quant16_regs.
__device__ __forceinline__ void fp8_item_put(int H, int k, int seg, int p0, int p1, const uint4 &qv, float s,
                                             uint8_t *__restrict__ recv_q, float *__restrict__ recv_s)
{
    const int lane = threadIdx.x & 31;
    const int C16 = H / 16;  // 16-column groups per row; 8 per 128-column block
    const int nb = H / 128;  // scales per row
    const int c = seg * 32 + lane;
    // C16 is a multiple of 8, so each 8-lane block is wholly in or out.
    const bool act = c < C16;
    for (int j = 0; j < k; ++j) {
        const int p = slot_row(p0, p1, j);
        if (p < 0 || !act)
            continue;
        st_plain16(recv_q + (size_t)p * H + (size_t)c * 16, qv);
        if ((c & 7) == 0)
            recv_s[(size_t)p * nb + (c >> 3)] = s;
    }
}

__device__ __forceinline__ void fp8_item_store(int H, int k, int seg, int p0, int p1, const uint4 &a, const uint4 &b,
                                               uint8_t *__restrict__ recv_q, float *__restrict__ recv_s)
{
    float s;
    const uint4 qv = fp8_quant16_regs(a, b, s);
    fp8_item_put(H, k, seg, p0, p1, qv, s, recv_q, recv_s);
}

__device__ __forceinline__ void dispatch_fp8_item(const uint16_t *__restrict__ x, int H, int k, long long t, int seg,
                                                  int p0, int p1, uint8_t *__restrict__ recv_q,
                                                  float *__restrict__ recv_s)
{
    uint4 a, b;
    q8_item_load(x, H, t, seg, a, b);
    fp8_item_store(H, k, seg, p0, p1, a, b, recv_q, recv_s);
}

// MXFP8 (E4M3 elements, E8M0 scale per 32 columns): the codes of the 16
// columns [16c, 16c + 16) and their block's scale byte.  Two consecutive
// lanes cover a block: every lane of the warp calls this.
// The products x * 2^-e run as packed fp32x2 multiplies (the same IEEE
// products, two per instruction).
__device__ __forceinline__ uint4 mx_quant16_regs(const uint4 &a, const uint4 &b, uint8_t &e_out)
{
    const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16_lo(wv[i]);
        f[2 * i + 1] = bf16_hi(wv[i]);
    }
    float amax = bf16x16_amax(a, b);
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    // floor(log2(amax)) from the exponent field; zero and fp32 subnormals
    // (below 2^-126) land on the clamp -127.
    const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
    int e = ef == 0 ? -127 : ef - 127 - 8;
    e = e < -127 ? -127 : e;
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, e in [-127, 119]
    const uint64_t inv2 = f2_pack(inv, inv);
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float d[4];
        f2_unpack(f2_mul(f2_pack(f[4 * i], f[4 * i + 1]), inv2), d[0], d[1]);
        f2_unpack(f2_mul(f2_pack(f[4 * i + 2], f[4 * i + 3]), inv2), d[2], d[3]);
        q[i] = pack_e4m3x2(d[0], d[1]) | (pack_e4m3x2(d[2], d[3]) << 16);
    }
    e_out = (uint8_t)(e + 127);
    return make_uint4(q[0], q[1], q[2], q[3]);
}

__device__ __forceinline__ uint4 mx_quant16(const uint16_t *__restrict__ xrow, int c, bool act, uint8_t &e_out)
{
    uint4 a, b;
    load16(xrow, c, act, a, b);
    return mx_quant16_regs(a, b, e_out);
}

// MXFP8: two lanes per 32-column block, E8M0 scale byte.  The store half
// takes the item's values from q8_item_load; mxfp8_item_put stores codes and
// scale byte already computed by mx_quant16_regs.
__device__ __forceinline__ void mxfp8_item_put(int H, int k, int seg, int p0, int p1, const uint4 &qv, uint8_t eb,
                                               uint8_t *__restrict__ recv_q, uint8_t *__restrict__ recv_e)
{
    const int lane = threadIdx.x & 31;
    const int nb = H / 32;  // scale bytes per row
    const int c = seg * 32 + lane;
    const bool act = c < H / 16;  // H / 16 is even: lane pairs are wholly in or out
    for (int j = 0; j < k; ++j) {
        const int p = slot_row(p0, p1, j);
        if (p < 0 || !act)
            continue;
        st_plain16(recv_q + (size_t)p * H + (size_t)c * 16, qv);
        if ((c & 1) == 0)
            recv_e[(size_t)p * nb + (c >> 1)] = eb;
    }
}

__device__ __forceinline__ void mxfp8_item_store(int H, int k, int seg, int p0, int p1, const uint4 &a,
                                                 const uint4 &b, uint8_t *__restrict__ recv_q,
                                                 uint8_t *__restrict__ recv_e)
{
    uint8_t eb;
    const uint4 qv = mx_quant16_regs(a, b, eb);
    mxfp8_item_put(H, k, seg, p0, p1, qv, eb, recv_q, recv_e);
}

__device__ __forceinline__ void dispatch_mxfp8_item(const uint16_t *__restrict__ x, int H, int k, long long t,
                                                    int seg, int p0, int p1, uint8_t *__restrict__ recv_q,
                                                    uint8_t *__restrict__ recv_e)
{
    uint4 a, b;
    q8_item_load(x, H, t, seg, a, b);
    mxfp8_item_store(H, k, seg, p0, p1, a, b, recv_q, recv_e);
}

}  // namespace ep
