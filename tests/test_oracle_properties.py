"""Property-based pins of the oracle (hypothesis; skipped where it is not
installed): random small shapes and routings, each checked against an
independent definition.
 - gating: the exhaustive-search selection of test_oracle_gate on random
   tiny configurations with forced ties;
 - layout: numpy's stable argsort and bincount on random index tensors with
   empty slots and repeats;
 - capacity layout: the stable argsort with the first `cap` entries of each
   expert kept;
 - FP8 dispatch: the largest element of every block codes to +-448 and
   dequantised codes stay within half a code step of the input.
"""
import numpy as np
import pytest

import oracle
import synth

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

from test_oracle_gate import _brute, _draw_tied  # noqa: E402


@st.composite
def gate_cases(draw):
    G = draw(st.sampled_from([1, 2, 3, 4]))
    gsize = draw(st.integers(1, 4))
    E = G * gsize
    Kg = draw(st.integers(1, G))
    kin = draw(st.integers(1, gsize))
    k = draw(st.integers(1, Kg * gsize))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    levels = draw(st.sampled_from([2, 4, 16]))
    with_bias = draw(st.booleans())
    return E, G, Kg, kin, k, seed, levels, with_bias


@settings(max_examples=150, deadline=None)
@given(gate_cases())
def test_gate_matches_exhaustive_search(case):
    E, G, Kg, kin, k, seed, levels, with_bias = case
    rng = np.random.default_rng(seed)
    T = 4
    s = _draw_tied(rng, (T, E), levels)
    b = (rng.integers(-2, 3, size=E) / 8).astype(np.float32) if with_bias else None
    idx, w = oracle.gate(s, b, k, G, Kg, kin, oracle.SCORE_RAW, 1)
    for t in range(T):
        assert list(idx[t]) == _brute(s[t], b, k, G, Kg, kin)
        assert abs(float(w[t].sum()) - 1.0) < 1e-6


@settings(max_examples=100, deadline=None)
@given(st.integers(1, 300), st.integers(1, 9), st.integers(1, 40), st.integers(0, 2 ** 31 - 1))
def test_layout_matches_stable_argsort(T, k, E, seed):
    rng = np.random.default_rng(seed)
    epr = [d for d in range(1, E + 1) if E % d == 0][rng.integers(0, sum(1 for d in range(1, E + 1) if E % d == 0))]
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    lay = oracle.layout(idx, E, epr)
    flat = idx.reshape(-1)
    valid = flat >= 0
    order = np.flatnonzero(valid)[np.argsort(flat[valid], kind="stable")]
    cnt = np.bincount(flat[valid], minlength=E)
    np.testing.assert_array_equal(lay["expert_count"], cnt)
    want = np.full(T * k, -1, np.int64)
    want[order] = np.arange(order.size)
    np.testing.assert_array_equal(lay["pos"].reshape(-1), want)
    R = E // epr
    np.testing.assert_array_equal(lay["rank_count"], cnt.reshape(R, epr).sum(axis=1))
    toks = [set() for _ in range(R)]
    for i in np.flatnonzero(valid):
        toks[flat[i] // epr].add(i // k)
    np.testing.assert_array_equal(lay["rank_tokens"], [len(x) for x in toks])


@settings(max_examples=80, deadline=None)
@given(st.integers(1, 200), st.integers(1, 6), st.integers(1, 24), st.integers(0, 60), st.integers(0, 2 ** 31 - 1))
def test_capacity_layout_keeps_the_first_cap_entries(T, k, E, cap, seed):
    rng = np.random.default_rng(seed)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    lay = oracle.layout_capacity(idx, E, 1, cap)
    flat = idx.reshape(-1)
    seen = np.zeros(E, np.int64)
    want = np.full(T * k, -1, np.int64)
    for i, e in enumerate(flat):
        if e < 0:
            continue
        if seen[e] < cap:
            want[i] = e * cap + seen[e]
        seen[e] += 1
    np.testing.assert_array_equal(lay["pos"].reshape(-1), want)
    np.testing.assert_array_equal(lay["expert_dropped"], seen - np.minimum(seen, cap))


@settings(max_examples=60, deadline=None)
@given(st.integers(1, 6), st.integers(1, 4), st.floats(-30, 30), st.integers(0, 2 ** 31 - 1))
def test_fp8_dispatch_block_properties(T, nblk, log2scale, seed):
    rng = np.random.default_rng(seed)
    H = 128 * nblk
    x = synth.f32_to_bf16_bits((rng.normal(0, 1, (T, H)) * 2.0 ** log2scale).astype(np.float32))
    q, s = oracle.dispatch_fp8(x, np.arange(T, dtype=np.int32).reshape(T, 1))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(T):
        for b in range(nblk):
            blk = xf[t, b * 128:(b + 1) * 128]
            codes = q[t, b * 128:(b + 1) * 128]
            amax = np.abs(blk).max()
            if amax == 0:
                continue
            assert np.any((codes & 0x7F) == 0x7E)                        # the largest element codes to +-448
            deq = oracle.e4m3_decode(codes).reshape(-1) * float(s[t, b])
            step = np.maximum(np.abs(blk) * 2.0 ** -3, float(s[t, b]) * 2.0 ** -9)   # one code step
            assert np.all(np.abs(deq - blk) <= 0.5 * step + np.abs(blk) * 2.0 ** -22)
