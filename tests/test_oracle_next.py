"""Pins for the oracle's next rows: MXFP8 dispatch, FP8-input combine,
capacity-limited layout, and the backward of dispatch and combine.

MXFP8 and FP8 payloads: "DeepEP de DeepSeek ...", section "Support FP8 et
MXFP8" (the format itself is the OCP Microscaling definition).  Capacity:
"Expert Parallelism (Parallelisme d'experts)", section "Defis et
optimisations" (load balancing by capacity factor).  Backward: training, the
pages' main setting.  Pins: hand-worked fixtures, torch's float8 conversion
and numpy's frexp for the shared exponent, exact rational arithmetic with a
nearest-bf16 search, the stable argsort, and round-trip identities.
"""
import json
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth
from test_oracle_combine import _bf16_value, _nearest_bf16


def _e4m3_value(code):
    """E4M3 value from its fields (an independent table for the pins)."""
    s = -1 if code & 0x80 else 1
    E, m = (code >> 3) & 0xF, code & 7
    mag = Fraction(m, 512) if E == 0 else Fraction(8 + m, 8) * Fraction(2) ** (E - 7)
    return s * mag


def test_mxfp8_golden(golden_dir):
    with open(os.path.join(golden_dir, "mxfp8_block_example.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        row = np.zeros(64, np.float32)
        row[:len(case["head"])] = case["head"]
        x = synth.f32_to_bf16_bits(row)[None, :]
        if case["head"] and case["head"][-1] == -0.0 and len(case["head"]) == 2:
            x[0, 1] = 0x8000
        q, e = oracle.dispatch_mxfp8(x, np.array([[0]], np.int32))
        assert q[0, :len(case["codes"])].tolist() == case["codes"], case["name"]
        assert e[0, 0] == case["e8m0"], case["name"]
        assert e[0, 1] == 0 and np.all(q[0, 32:] == 0)       # second block is all zeros


def test_mxfp8_matches_frexp_and_torch():
    rng = np.random.default_rng(12)
    T, H = 40, 256
    f = (rng.normal(0, 1, (T, H)) * np.exp2(rng.integers(-20, 20, (T, 1)))).astype(np.float32)
    x = synth.f32_to_bf16_bits(f)
    q, e = oracle.dispatch_mxfp8(x, np.arange(T, dtype=np.int32)[:, None])
    xf = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(T, H // 32, 32)
    amax = np.abs(xf).max(axis=2)
    _, ex = np.frexp(amax)                        # amax = m * 2^ex, m in [0.5, 1): floor(log2) = ex - 1
    want_e = np.clip(ex - 1 - 8, -127, 127)
    np.testing.assert_array_equal(e.astype(np.int64) - 127, want_e)
    scaled = xf / np.exp2(want_e)[:, :, None]
    assert np.all(np.abs(scaled) < 512)
    sat = np.abs(scaled) >= 464                   # torch gives NaN there; the format saturates
    ref = torch.from_numpy(np.where(sat, 0, scaled).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    ref = ref.numpy().reshape(T, H)
    sat = sat.reshape(T, H)
    ref[sat] = np.where(np.signbit(scaled.reshape(T, H)[sat]), 0xFE, 0x7E)
    np.testing.assert_array_equal(q, ref)
    # the block maximum lands in the top binade [256, 448]
    top = np.abs(q.reshape(T, H // 32, 32).astype(np.int32) & 0x7F).max(axis=2)
    assert np.all(top >= 0x78)


def test_combine_fp8_exact_small():
    rng = np.random.default_rng(21)
    T, k = 5, 3
    for kind, H in ((0, 256), (1, 64)):
        rows = T * k
        yq = rng.integers(0, 256, size=(rows, H)).astype(np.uint8)
        yq[(yq & 0x7F) == 0x7F] = 0x11                 # no NaN codes
        if kind == 0:
            ys = rng.uniform(0.001, 2.0, size=(rows, H // 128)).astype(np.float32)
        else:
            ys = rng.integers(100, 140, size=(rows, H // 32)).astype(np.uint8)
        pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
        pos[1, 2] = -1
        w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
        out = oracle.combine_fp8(yq, ys, pos, w)
        bs = 128 if kind == 0 else 32
        for t in range(T):
            for h in range(0, H, 7):
                acc = Fraction(0)
                for j in range(k):
                    p = pos[t, j]
                    if p < 0:
                        continue
                    s = Fraction(float(ys[p, h // bs])) if kind == 0 else Fraction(2) ** (int(ys[p, h // bs]) - 127)
                    acc += Fraction(float(w[t, j])) * _e4m3_value(int(yq[p, h])) * s
                assert out[t, h] == _nearest_bf16(acc), (kind, t, h)


def test_fp8_round_trip_through_combine():
    cfg = synth.config("dsv3", T=48)
    inp = synth.make_inputs(cfg)
    idx, w64 = oracle.gate(inp["scores"], inp["bias"], 8, 8, 4, 2, oracle.SCORE_RAW, True)
    pos = oracle.layout(idx, 256, 8)["pos"]
    x = synth.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    for disp, bs in ((oracle.dispatch_fp8, 128), (oracle.dispatch_mxfp8, 32)):
        q, s = disp(inp["x"], pos)
        out = synth.bf16_bits_to_f32(oracle.combine_fp8(q, s, pos, np.full((48, 8), 0.125, np.float32)))
        row0 = pos[:, 0]
        step = s[row0].astype(np.float64) if bs == 128 else np.exp2(s[row0].astype(np.float64) - 127)
        step = np.repeat(step, bs, axis=1)                  # the block's scale, per column
        # half an e4m3 step: 2^-4 relative for normals, 2^-10 * scale for
        # subnormals; MXFP8 also saturates |x|/X in (448, 512) to 448 (at most
        # 1/8 relative); then one bf16 rounding (2^-8 relative)
        rel = 2.0 ** -4 if bs == 128 else 2.0 ** -3
        bound = (rel + 2.0 ** -8 + 2.0 ** -12) * np.abs(x) + 2.0 ** -10 * step
        assert np.all(np.abs(out - x) <= bound), disp.__name__


def test_capacity_golden(golden_dir):
    with open(os.path.join(golden_dir, "layout_8experts_4ranks.json")) as f:
        g = json.load(f)
    c = g["capacity_case"]
    lay = oracle.layout_capacity(np.array(g["topk_idx"], np.int32), g["num_experts"], g["experts_per_rank"],
                                 c["capacity"])
    for key in ("pos", "expert_count", "expert_dropped", "expert_off", "rank_count", "rank_off", "rank_tokens",
                "src"):
        assert lay[key].tolist() == c[key], key


def test_capacity_matches_stable_argsort():
    rng = np.random.default_rng(17)
    for T, k, E, epr, cap in ((300, 4, 16, 4, 50), (500, 8, 64, 8, 40), (200, 2, 8, 2, 0), (100, 3, 12, 3, 1000)):
        idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
        idx[rng.random((T, k)) < 0.3] = 3                 # a hot expert
        lay = oracle.layout_capacity(idx, E, epr, cap)
        flat = idx.reshape(-1)
        valid = flat >= 0
        order = np.flatnonzero(valid)[np.argsort(flat[valid], kind="stable")]
        cnt = np.bincount(flat[valid], minlength=E)
        start = np.concatenate([[0], np.cumsum(cnt)])[:-1]
        rank = np.empty(order.size, np.int64)
        rank[:] = np.arange(order.size) - start[flat[order]]
        want = np.full(T * k, -1, np.int64)
        kept = rank < cap
        want[order[kept]] = flat[order[kept]] * cap + rank[kept]
        np.testing.assert_array_equal(lay["pos"].reshape(-1), want)
        np.testing.assert_array_equal(lay["expert_count"], np.minimum(cnt, cap))
        np.testing.assert_array_equal(lay["expert_dropped"], cnt - np.minimum(cnt, cap))
        rows = lay["src"]
        assert set(rows[rows >= 0].tolist()) == set(order[kept].tolist())


def test_backward_exact_small():
    rng = np.random.default_rng(33)
    T, H, k = 4, 16, 3
    rows = T * k
    g = synth.f32_to_bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (rows, H)).astype(np.float32))
    gr = synth.f32_to_bf16_bits(rng.normal(0, 1, (rows, H)).astype(np.float32))
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[2, 0] = -1
    w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
    gx = oracle.dispatch_backward(gr, pos)
    gy, gw = oracle.combine_backward(g, y, pos, w)
    for t in range(T):
        for h in range(H):
            acc = sum((_bf16_value(gr[pos[t, j], h]) for j in range(k) if pos[t, j] >= 0), Fraction(0))
            assert gx[t, h] == _nearest_bf16(acc)
        for j in range(k):
            p = pos[t, j]
            if p < 0:
                assert gw[t, j] == 0
                continue
            for h in range(H):
                assert gy[p, h] == _nearest_bf16(Fraction(float(w[t, j])) * _bf16_value(g[t, h]))
            dot = sum((_bf16_value(g[t, h]) * _bf16_value(y[p, h]) for h in range(H)), Fraction(0))
            assert abs(Fraction(gw[t, j]) - dot) <= abs(dot) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 60)
    # the row the empty slot would have named is never written
    untouched = set(range(rows)) - set(pos[pos >= 0].tolist())
    for r in untouched:
        assert np.all(gy[r] == 0)


def test_dispatch_backward_of_copies_is_k_times():
    cfg = synth.config("dsv3", T=32)
    inp = synth.make_inputs(cfg)
    idx, _ = oracle.gate(inp["scores"], inp["bias"], 8, 8, 4, 2, oracle.SCORE_RAW, True)
    pos = oracle.layout(idx, 256, 8)["pos"]
    recv = oracle.dispatch_bf16(inp["x"], pos)
    gx = synth.bf16_bits_to_f32(oracle.dispatch_backward(recv, pos))
    np.testing.assert_array_equal(gx, 8 * synth.bf16_bits_to_f32(inp["x"]))    # 8 = 2^3: exact in bf16


def test_capacity_rank_counts_brute_force():
    """rank_count counts the kept entries of a rank's experts; rank_tokens
    counts the tokens with at least one kept entry on the rank (a dropped
    slot does not count its token), by direct enumeration on small cases."""
    rng = np.random.default_rng(23)
    for T, k, E, epr, cap in ((60, 4, 8, 2, 5), (40, 6, 12, 4, 3), (30, 3, 6, 3, 0), (25, 2, 4, 1, 100)):
        idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
        idx[rng.random((T, k)) < 0.3] = 1
        lay = oracle.layout_capacity(idx, E, epr, cap)
        pos = lay["pos"].reshape(T, k)
        R = E // epr
        kept_by_rank = [0] * R
        tokens_by_rank = [0] * R
        for t in range(T):
            seen = set()
            for j in range(k):
                if pos[t, j] >= 0:
                    r = int(idx[t, j]) // epr
                    kept_by_rank[r] += 1
                    seen.add(r)
            for r in seen:
                tokens_by_rank[r] += 1
        assert lay["rank_count"].tolist() == kept_by_rank
        assert lay["rank_tokens"].tolist() == tokens_by_rank
        assert lay["rank_off"].tolist() == [r * epr * cap for r in range(R + 1)]


def test_every_invalid_index_value_is_flagged_and_skipped():
    """-1 is an empty slot; every other value outside [0, E) -- -2, INT_MIN,
    E, INT_MAX -- raises the bad-expert flag and is skipped, in both the
    plain and the capacity layout."""
    E, epr = 8, 2
    for bad in (-2, -3, -2 ** 31, E, 2 ** 31 - 1):
        idx = np.array([[0, bad], [bad, 5], [3, -1]], np.int32)
        clean = np.where(idx == bad, -1, idx).astype(np.int32)
        lay, ref = oracle.layout(idx, E, epr), oracle.layout(clean, E, epr)
        assert lay["err_flag"] & 1 and not ref["err_flag"]
        for key in ("pos", "src", "expert_count", "rank_count", "rank_tokens"):
            assert lay[key].tolist() == ref[key].tolist(), (bad, key)
        cl, cr = oracle.layout_capacity(idx, E, epr, 2), oracle.layout_capacity(clean, E, epr, 2)
        assert cl["err_flag"] & 1 and not cr["err_flag"]
        for key in ("pos", "src", "expert_count", "expert_dropped", "rank_count", "rank_tokens"):
            assert cl[key].tolist() == cr[key].tolist(), (bad, key)
    empty = oracle.layout(np.array([[-1, -1]], np.int32), E, epr)
    assert empty["err_flag"] == 0 and empty["pos"].tolist() == [[-1, -1]]
