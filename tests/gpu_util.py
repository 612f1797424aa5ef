"""Helpers shared by the GPU parity tests: host<->device marshalling of the
seeded inputs and the tolerances the floating-point outputs are held to.

Tolerances (u = 2^-24, the binary32 unit roundoff):
 * gate weights, raw scores: the kernel adds the k chosen scores in fp32
   (k-1 roundings of positive terms) and divides once, so its relative error
   against the exact quotient is at most k*u; the test allows (k+1)*u.
 * gate weights, softmax: each exp argument l - m is one fp32 subtraction
   (error <= u*|l - m|, amplified 1:1 by exp), expf adds at most 2 ulp
   (<= 4u), the sum adds (n-1)u and the division u, with n = k terms when
   normalised over the chosen k and n = E for the full softmax; so the
   relative error is below u*(2D + 8 + n) with D the spread of the logits
   involved; the test allows u*(2D + 10 + n).
 * combine: the stated bar is max(1 bf16 ulp, 1e-2 relative) against the
   exact (binary64) oracle, and the five workloads' full-size tests are held
   to it alone.  The kernel is specified to accumulate in fp32, whose fma
   chain can differ from the exact sum by k*u*sum_j|w_j y_j| before the final
   rounding; that only matters where the sum cancels, which the synthetic
   edge cases (signed weights, arbitrary expert outputs) provoke on purpose,
   so those tests add exactly that term (accumulation=True).
"""
import numpy as np
import torch

import synth

U = 2.0 ** -24


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gate_args(cfg):
    return (cfg["k"], cfg["n_groups"], cfg["topk_group"], cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])


def ep_cfg(ep, cfg):
    return ep.gate_cfg(cfg["E"], cfg["k"], cfg["n_groups"], cfg["topk_group"], cfg["topk_in_group"],
                       cfg["score_fn"], cfg["normalize"])


def weight_rtol(cfg, scores, idx):
    k = idx.shape[1]
    if cfg["score_fn"] == synth.SCORE_RAW:
        return np.full(idx.shape, (k + 1) * U)
    sel = np.take_along_axis(scores.astype(np.float64), idx.astype(np.int64), axis=1)
    if cfg["normalize"]:
        D = sel.max(axis=1) - sel.min(axis=1)
        n = k
    else:
        D = scores.max(axis=1).astype(np.float64) - scores.min(axis=1)
        n = scores.shape[1]
    return ((2 * D + 10 + n) * U)[:, None] * np.ones(idx.shape)


def assert_weights_close(w_gpu, w_ref, rtol):
    err = np.abs(w_gpu.astype(np.float64) - w_ref)
    bad = err > rtol * np.abs(w_ref)
    assert not bad.any(), "weights differ at %s: gpu %r ref %r" % (
        np.argwhere(bad)[:5].tolist(), w_gpu[bad][:5], w_ref[bad][:5])


def bf16_ulp(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.exp2(e - 7)


def assert_combine_close(out_gpu_bits, out_ref_bits, y_bits, pos, w, accumulation=True):
    """out_gpu vs out_ref (bf16 bit patterns, [T,H]) with the tolerance above:
    the stated bar, plus the fp32 accumulation term when accumulation=True."""
    g = synth.bf16_bits_to_f32(out_gpu_bits).astype(np.float64)
    r = synth.bf16_bits_to_f32(out_ref_bits).astype(np.float64)
    T, k = pos.shape
    yf = synth.bf16_bits_to_f32(y_bits)
    S = np.zeros_like(r)
    for j in range(k):
        p = pos[:, j]
        ok = p >= 0
        S[ok] += np.abs(w[ok, j].astype(np.float64))[:, None] * np.abs(yf[p[ok]].astype(np.float64))
    tol = np.maximum(bf16_ulp(r), 1e-2 * np.abs(r)) + (k * U * S if accumulation else 0.0)
    err = np.abs(g - r)
    bad = err > tol
    assert not bad.any(), "combine differs at %s: gpu %r ref %r tol %r" % (
        np.argwhere(bad)[:5].tolist(), g[bad][:5], r[bad][:5], tol[bad][:5])
