"""Seeded synthetic workloads for the MoE dispatch/combine path.

This module only draws random inputs: router scores or logits, the per-expert
selection bias, and the hidden rows.  It holds none of the method's
arithmetic, so both the CPU oracle and the CUDA library can be fed from it
without sharing any of the computation they are checked on.

Generator: a counter-based splitmix64 stream, value i of stream (seed, s) is
mix64(mix64(seed * 2^32 + s) + (i + 1) * 0x9E3779B97F4A7C15), with the
splitmix64 finaliser of Steele, Lea and Flood ("Fast splittable pseudorandom
number generators", OOPSLA 2014).  Uniforms are odd multiples of 2^-24 in
(0, 1), exact in binary32; normals use the Box-Muller transform in binary64.
Hidden rows are rounded to bfloat16 (nearest, ties to even) from binary32.
The normals go through the platform's libm, so a rare last bit may differ
between machines; every parity check feeds both sides from one process.

Workloads follow the shapes the pages talk about (DeepSeek-V3-style
256-expert group-limited routing, Mixtral-style 8-expert top-2, a 128-expert
top-8 family and a decode-sized batch); no dataset or trained router is
involved.
"""
import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

SCORE_RAW = 0
SCORE_SOFTMAX = 1


def _mix64_scalar(z):
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def _mix64(z):
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def u64(seed, stream, n, start=0):
    """n raw 64-bit values of stream (seed, stream), counters start..start+n-1."""
    key = _mix64_scalar((seed << 32) + stream)
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + i * np.uint64(GOLDEN))


def uniform_f32(seed, stream, shape):
    """U(0,1) binary32, odd multiples of 2^-24 (never 0, never 1)."""
    n = int(np.prod(shape))
    u = u64(seed, stream, n) >> np.uint64(41)               # 23 random bits
    return ((u.astype(np.float64) * 2.0 + 1.0) * 2.0 ** -24).astype(np.float32).reshape(shape)


def normal_f64(seed, stream, shape, chunk=1 << 22):
    """N(0,1) in binary64 by Box-Muller, generated in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float64)
    pairs = (n + 1) // 2
    for c0 in range(0, pairs, chunk):
        m = min(chunk, pairs - c0)
        a = u64(seed, stream, m, start=2 * c0)
        b = u64(seed, stream + 0x10000, m, start=2 * c0)
        u1 = ((a >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53   # (0, 1]
        u2 = (b >> np.uint64(11)).astype(np.float64) * 2.0 ** -53           # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        th = 2.0 * np.pi * u2
        lo = 2 * c0
        z = np.empty(2 * m)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        take = min(2 * m, n - lo)
        out[lo:lo + take] = z[:take]
    return out.reshape(shape)


def f32_to_bf16_bits(f):
    """binary32 -> bfloat16 bit patterns, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(f, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h):
    return (np.ascontiguousarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_bits(seed, stream, shape, sigma=1.0):
    return f32_to_bf16_bits((normal_f64(seed, stream, shape) * sigma).astype(np.float32))


def permutation(seed, stream, n):
    return np.argsort(u64(seed, stream, n), kind="stable").astype(np.int64)


# Streams of one workload.
_S_SCORES, _S_BIAS, _S_X, _S_PERM, _S_Y, _S_W = 1, 2, 3, 4, 5, 6

# Zipf exponent of the skewed workload and the bias strength that makes the
# hottest expert receive about 20x the mean count under group-limited top-8
# routing.  Calibrated with tests/golden/calibrate_skew.py against the CPU
# oracle's gating; tests/test_synth.py checks the ratio stays in [18, 22].
ZIPF_S = 1.2
SKEW_BETA = 0.1485

CONFIGS = {
    # 128 tokens, 8 experts on 4 logical ranks (2 each), raw U(0,1) scores.
    "tiny": dict(T=128, H=256, E=8, k=2, n_groups=1, topk_group=1, topk_in_group=1,
                 score_fn=SCORE_RAW, normalize=True, experts_per_rank=2,
                 scores="uniform", bias=None, dispatch=("bf16",), seed=1234),
    # Mixtral-style: 8 experts, top-2 over softmax of N(0,1) logits, renormalised.
    "mixtral": dict(T=4096, H=4096, E=8, k=2, n_groups=1, topk_group=1, topk_in_group=1,
                    score_fn=SCORE_SOFTMAX, normalize=True, experts_per_rank=1,
                    scores="normal", bias=None, dispatch=("bf16",), seed=1235),
    # DeepSeek-V3-style: 256 experts in 8 groups, top-4 groups then top-8,
    # U(0,1) affinities + N(0, 0.01) bias, 32 logical ranks x 8 experts.
    "dsv3": dict(T=8192, H=7168, E=256, k=8, n_groups=8, topk_group=4, topk_in_group=2,
                 score_fn=SCORE_RAW, normalize=True, experts_per_rank=8,
                 scores="uniform", bias="normal", dispatch=("fp8", "bf16"), seed=1236),
    # As dsv3 but with Zipf(1.2) expert popularity folded into the bias.
    "skewed": dict(T=8192, H=7168, E=256, k=8, n_groups=8, topk_group=4, topk_in_group=2,
                   score_fn=SCORE_RAW, normalize=True, experts_per_rank=8,
                   scores="uniform", bias="zipf", dispatch=("bf16", "fp8"), seed=1237),
    # 128 experts, top-8 over softmax of N(0,1) logits, 16 ranks x 8 experts.
    "qwen3": dict(T=16384, H=4096, E=128, k=8, n_groups=1, topk_group=1, topk_in_group=1,
                  score_fn=SCORE_SOFTMAX, normalize=True, experts_per_rank=8,
                  scores="normal", bias=None, dispatch=("bf16",), seed=1238),
    # Decode-sized batch: 128 tokens, 7168 hidden, 256 experts, softmax top-8.
    "decode": dict(T=128, H=7168, E=256, k=8, n_groups=1, topk_group=1, topk_in_group=1,
                   score_fn=SCORE_SOFTMAX, normalize=True, experts_per_rank=8,
                   scores="normal", bias=None, dispatch=("bf16", "fp8"), seed=1239),
}


def config(name, **over):
    """A copy of a named workload, optionally with fields overridden (e.g. T)."""
    c = dict(CONFIGS[name])
    c["name"] = name
    c.update(over)
    return c


def make_scores(cfg):
    T, E, seed = cfg["T"], cfg["E"], cfg["seed"]
    if cfg["scores"] == "uniform":
        return uniform_f32(seed, _S_SCORES, (T, E))
    return normal_f64(seed, _S_SCORES, (T, E)).astype(np.float32)


def make_bias(cfg, beta=None):
    E, seed = cfg["E"], cfg["seed"]
    kind = cfg["bias"]
    if kind is None:
        return None
    b = normal_f64(seed, _S_BIAS, (E,)) * 0.01
    if kind == "zipf":
        beta = SKEW_BETA if beta is None else beta
        perm = permutation(seed, _S_PERM, E)                # expert e has popularity rank perm[e]
        b = b + beta * (-ZIPF_S * np.log(perm + 1.0))
    return b.astype(np.float32)


def make_x(cfg):
    return normal_bf16_bits(cfg["seed"], _S_X, (cfg["T"], cfg["H"]))


def make_inputs(cfg):
    """dict(scores f32 [T,E], bias f32 [E] or None, x uint16 bf16 bits [T,H])."""
    return dict(scores=make_scores(cfg), bias=make_bias(cfg), x=make_x(cfg))


def make_expert_out(cfg, rows):
    """Stand-in expert outputs: bf16 N(0,1) rows [rows, H] (not the identity)."""
    return normal_bf16_bits(cfg["seed"], _S_Y, (rows, cfg["H"]))


def make_weights(cfg):
    """Random positive f32 weights [T,k] (not normalised), for combine-only checks."""
    return uniform_f32(cfg["seed"], _S_W, (cfg["T"], cfg["k"]))
