"""Pins for the oracle's combine (steps 4-5) and its bfloat16 rounding.

Combine brings each expert output back to its token and sums them weighted
by the router scores ("Expert Parallelism (Parallelisme d'experts)", section
"Le pattern de communication all-to-all", Phase 2).  The pins: exact rational
arithmetic with a nearest-bf16 search on tiny inputs, torch's own
binary32->bfloat16 rounding, and the identity-expert round trip
combine(dispatch(x)) == x when the weights sum to one.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth


def _bf16_value(bits):
    return Fraction(float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0]))


def _nearest_bf16(v: Fraction):
    """Nearest bfloat16 to an exact rational, ties to the even pattern."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    approx = np.float32(float(a)).view(np.uint32) >> 16
    cands = [int(c) for c in range(max(int(approx) - 2, 0), int(approx) + 3)]
    best = min(cands, key=lambda c: (abs(_bf16_value(c) - a), c & 1))
    return sign | best


def test_bf16_rounding_matches_torch_for_binary32_inputs():
    rng = np.random.default_rng(2)
    f = np.concatenate([rng.normal(0, 1, 50000) * np.exp2(rng.integers(-140, 120, 50000)),
                        [0.0, -0.0, 1.00390625, 1.01171875, 3.3e38, -3.4e38, 1e-45]]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_from_double(f.astype(np.float64)), ref)


def test_bf16_rounding_exact_search_on_doubles():
    rng = np.random.default_rng(4)
    d = rng.normal(0, 1, 3000) * np.exp2(rng.integers(-30, 30, 3000))
    got = oracle.bf16_from_double(d)
    want = [_nearest_bf16(Fraction(float(v))) for v in d]
    assert got.tolist() == want
    # a tie between two bf16 values decides by the even pattern
    assert oracle.bf16_from_double(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]))[:].tolist() == [0x3F80, 0x3F82]


def test_combine_exact_small():
    rng = np.random.default_rng(6)
    T, H, k = 7, 24, 3
    rows = T * k
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (rows, H)).astype(np.float32))
    w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[2, 1] = -1                                          # an empty slot
    out = oracle.combine(y, pos, w)
    for t in range(T):
        for h in range(H):
            acc = Fraction(0)
            for j in range(k):
                if pos[t, j] >= 0:
                    acc += Fraction(float(w[t, j])) * _bf16_value(y[pos[t, j], h])
            assert out[t, h] == _nearest_bf16(acc), (t, h)


def test_identity_round_trip_reproduces_x():
    cfg = synth.config("dsv3", T=64)
    inp = synth.make_inputs(cfg)
    idx, w64 = oracle.gate(inp["scores"], inp["bias"], 8, 8, 4, 2, oracle.SCORE_RAW, True)
    lay = oracle.layout(idx, 256, 8)
    recv = oracle.dispatch_bf16(inp["x"], lay["pos"])
    w = w64.astype(np.float32)
    out = oracle.combine(recv, lay["pos"], w)
    x = synth.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    o = synth.bf16_bits_to_f32(out).astype(np.float64)
    # sum_j w_j x = x * (sum_j w_j), and sum_j w_j is 1 up to the binary32
    # rounding of the k weights
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 7)
    assert np.all(np.abs(o - x) <= ulp + 8 * 2.0 ** -24 * np.abs(x))
    # with weights that sum to exactly 1 the round trip is exact
    w_exact = np.full((64, 8), 0.125, np.float32)
    np.testing.assert_array_equal(oracle.combine(recv, lay["pos"], w_exact), inp["x"])
