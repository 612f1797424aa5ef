"""Pins for the oracle's E4M3 codec and FP8 1x128 dispatch (step 3, FP8 mode).

The FP8 payload is the pages' ("DeepEP de DeepSeek ...", section "Support FP8
et MXFP8"); the format is the OCP E4M3 definition.  The pins: code values
from that definition (tests/golden), every code's round trip, torch's own
float8_e4m3fn conversion, a brute-force nearest-code search with the
tie-to-even rule, the exact midpoints of every adjacent code pair, and error
bounds / invariants of the block-scaled dispatch.
"""
import json
import os

import numpy as np
import torch

import oracle
import synth


def _all_finite_positive_codes():
    """Every finite non-negative E4M3 value, enumerated from the format's
    fields (exponent field 0..15, mantissa 0..7, S.1111.111 excluded)."""
    vals = []
    for E in range(16):
        for m in range(8):
            if E == 15 and m == 7:
                continue
            v = m * 2.0 ** -9 if E == 0 else (1 + m / 8) * 2.0 ** (E - 7)
            vals.append(((E << 3) | m, v))
    return vals


def test_codes_golden(golden_dir):
    with open(os.path.join(golden_dir, "e4m3_codes.json")) as f:
        g = json.load(f)
    for code, val in g["decode"]:
        got = oracle.e4m3_decode(np.array([code], np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val), code
    for val, code in g["encode"]:
        assert int(oracle.e4m3_encode(np.array([val], np.float32))[0]) == code, val


def test_every_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254                       # 0x7F and 0xFF are NaN
    back = oracle.e4m3_encode(vals[finite].astype(np.float32))
    np.testing.assert_array_equal(back, codes[finite])
    table = dict(_all_finite_positive_codes())
    for c in range(127):
        assert vals[c] == table[c]


def _brute_nearest(v):
    """Nearest finite code by exhaustive search; ties to the even mantissa;
    magnitudes beyond 448 saturate."""
    table = _all_finite_positive_codes()
    a = min(abs(float(v)), 448.0)
    best = None
    for code, val in table:
        d = abs(val - a)
        if best is None or d < best[0] or (d == best[0] and (code & 1) == 0):
            best = (d, code)
    return best[1] | (0x80 if np.signbit(v) else 0)


def test_encode_brute_force_sample():
    rng = np.random.default_rng(5)
    e = rng.uniform(-13, 10, size=4000)
    v = (np.exp2(e) * rng.choice([-1, 1], size=e.size)).astype(np.float32)
    got = oracle.e4m3_encode(v)
    want = np.array([_brute_nearest(x) for x in v], np.uint8)
    np.testing.assert_array_equal(got, want)


def test_encode_midpoints_and_neighbours():
    table = sorted(_all_finite_positive_codes(), key=lambda cv: cv[1])
    pts, want = [], []
    for (c0, v0), (c1, v1) in zip(table, table[1:]):
        mid = np.float32((v0 + v1) / 2)                  # exact: a few significant bits
        assert float(mid) == (v0 + v1) / 2
        even = c0 if (c0 & 1) == 0 else c1
        pts += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
        want += [even, c0, c1]
    got = oracle.e4m3_encode(np.array(pts, np.float32))
    np.testing.assert_array_equal(got, np.array(want, np.uint8))
    neg = oracle.e4m3_encode(-np.array(pts, np.float32))
    np.testing.assert_array_equal(neg, np.array(want, np.uint8) | 0x80)


def test_encode_matches_torch_float8_e4m3fn():
    """torch's CPU conversion rounds to nearest-even and gives NaN past the
    rounding range; inside +-464 it must agree bit for bit."""
    rng = np.random.default_rng(9)
    v = np.concatenate([
        rng.normal(0, 1, 20000) * np.exp2(rng.integers(-12, 9, 20000)),
        rng.uniform(-463.9, 463.9, 20000),
        np.exp2(np.arange(-16, 9)).repeat(2) * np.tile([1, -1], 25),
    ]).astype(np.float32)
    v = v[np.abs(v) < 464]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_encode_saturates():
    v = np.array([448.0, 448.01, 464.0, 1e6, np.inf, -np.inf, -500.0], np.float32)
    assert oracle.e4m3_encode(v).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_fp8_block_golden(golden_dir):
    with open(os.path.join(golden_dir, "fp8_block_example.json")) as f:
        g = json.load(f)
    H = g["H"]
    row = np.zeros(H, np.float32)
    row[:4] = g["row_head"]
    row[128 + 5] = -0.0
    x = synth.f32_to_bf16_bits(row)[None, :]
    q, s = oracle.dispatch_fp8(x, np.array([[0]], np.int32))
    assert q[0, :4].tolist() == g["codes_head"]
    assert np.all(q[0, 4:128] == 0)
    assert q[0, 128] == 0 and q[0, 128 + 5] == 0x80
    assert s[0, 0] == np.float32(2.0) / np.float32(448.0)
    assert s[0, 1] == g["scale1"]


def test_fp8_dispatch_bounds_and_invariants():
    cfg = synth.config("dsv3", T=96)
    inp = synth.make_inputs(cfg)
    x = inp["x"].copy()
    x[3, 128:256] = 0                                  # an all-zero block
    x[4, 0:128] = 0x8000                               # an all -0.0 block
    idx, _ = oracle.gate(inp["scores"], inp["bias"], 8, 8, 4, 2, oracle.SCORE_RAW, True)
    lay = oracle.layout(idx, 256, 8)
    q, s = oracle.dispatch_fp8(x, lay["pos"])
    # every copy of a token carries identical codes and scales
    rows = lay["pos"]
    for t in range(cfg["T"]):
        assert np.all(q[rows[t]] == q[rows[t][0]]) and np.all(s[rows[t]] == s[rows[t][0]])
    qt, st = q[rows[:, 0]], s[rows[:, 0]]                # per-token payload [T, H], [T, H/128]
    xf = synth.bf16_bits_to_f32(x).reshape(cfg["T"], -1, 128)
    amax = np.abs(xf).max(axis=2)
    np.testing.assert_array_equal(st, (amax / np.float32(448)).astype(np.float32))
    codes = qt.reshape(cfg["T"], -1, 128)
    # a block with amax > 0 maps its largest magnitude to +-448
    has = amax > 0
    assert np.all((np.abs(codes.astype(np.int32) & 0x7F) == 0x7E).any(axis=2)[has])
    # zero blocks: scale 0, signed-zero codes
    assert st[3, 1] == 0 and np.all(codes[3, 1] == 0)
    assert st[4, 0] == 0 and np.all(codes[4, 0] == 0x80)
    # dequantised error: half a code step (2^-4 relative for normals, 2^-10 s
    # for subnormals) plus the binary32 rounding of x/s
    deq = oracle.e4m3_decode(codes.reshape(-1)).reshape(codes.shape) * st[:, :, None]
    err = np.abs(deq - xf)
    bound = 2.0 ** -10 * st[:, :, None] * (1 + 2.0 ** -20) + (2.0 ** -4 + 2.0 ** -22) * np.abs(xf)
    assert np.all(err <= bound)
