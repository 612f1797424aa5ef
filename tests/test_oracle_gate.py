"""Pins for the oracle's gating (step 1), independent of the oracle's own code.

Group-limited gating restricts each token's experts to a few groups ("DeepEP de
DeepSeek ...", section "Group-limited gating algorithm").  The pins:
hand-worked cases (tests/golden), brute force over every group subset and
every expert subset on tiny inputs with forced ties, the plain-top-k special
case against numpy's stable sort and torch.topk, and weight identities.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

RAW, SOFTMAX = oracle.SCORE_RAW, oracle.SCORE_SOFTMAX


def _keys(s, b):
    return s.astype(np.float32) if b is None else (s.astype(np.float32) + b.astype(np.float32)).astype(np.float32)


def _brute(s, b, k, G, Kg, kin):
    """Selection by exhaustive search: the kept group set is the one Kg-subset
    whose every member beats every non-member in (score desc, index asc);
    likewise for the expert set inside the kept groups."""
    E = s.shape[0]
    gsize = E // G
    key = _keys(s, b)
    gs = []
    for g in range(G):
        vals = sorted(key[g * gsize:(g + 1) * gsize].tolist(), reverse=True)[:kin]
        acc = np.float32(vals[0])
        for v in vals[1:]:
            acc = np.float32(acc + np.float32(v))
        gs.append(acc)

    def beats(a, b_, score):
        return score[a] > score[b_] or (score[a] == score[b_] and a < b_)

    winners = [S for S in itertools.combinations(range(G), Kg)
               if all(beats(g, h, gs) for g in S for h in range(G) if h not in S)]
    assert len(winners) == 1
    kept = [e for e in range(E) if (e // gsize) in winners[0]]
    chosen = [S for S in itertools.combinations(kept, k)
              if all(beats(e, f, key) for e in S for f in kept if f not in S)]
    assert len(chosen) == 1
    return sorted(chosen[0], key=lambda e: (-float(key[e]), e))


def _draw_tied(rng, shape, levels=8):
    return (rng.integers(1, levels + 1, size=shape) / levels).astype(np.float32)


@pytest.mark.parametrize("E,G,Kg,k,kin", [
    (8, 4, 2, 2, 2), (8, 4, 2, 3, 1), (8, 2, 1, 2, 2), (12, 3, 2, 4, 2),
    (12, 4, 3, 3, 3), (16, 4, 2, 4, 2), (16, 8, 3, 5, 1), (16, 1, 1, 3, 1),
])
def test_gate_bruteforce_with_ties(E, G, Kg, k, kin):
    rng = np.random.default_rng(E * 1000 + G * 100 + Kg * 10 + k)
    T = 60
    s = _draw_tied(rng, (T, E))
    b = (rng.integers(-2, 3, size=E) / 16).astype(np.float32)
    idx, _ = oracle.gate(s, b, k, G, Kg, kin, RAW, True)
    for t in range(T):
        assert idx[t].tolist() == _brute(s[t], b, k, G, Kg, kin), t


def test_gate_plain_topk_is_stable_sort():
    """One group (or all groups kept) is plain top-k: numpy's stable sort on
    (-key) gives the same experts in the same slot order."""
    rng = np.random.default_rng(7)
    s = _draw_tied(rng, (200, 32), levels=16)
    b = (rng.integers(-3, 4, size=32) / 32).astype(np.float32)
    key = _keys(s, b)
    want = np.argsort(-key, axis=1, kind="stable")[:, :6]
    for G, Kg in ((1, 1), (4, 4), (8, 8)):
        idx, _ = oracle.gate(s, b, 6, G, Kg, 2 if G < 32 else 1, RAW, True)
        np.testing.assert_array_equal(idx, want)


def test_gate_softmax_indices_match_torch_topk():
    cfg = synth.config("qwen3", T=256)
    logits = synth.make_scores(cfg)
    idx, _ = oracle.gate(logits, None, 8, score_fn=SOFTMAX)
    ref = torch.topk(torch.from_numpy(logits), 8, dim=1, sorted=True).indices.numpy()
    np.testing.assert_array_equal(idx, ref)


def test_gate_softmax_weights_against_long_double():
    cfg = synth.config("mixtral", T=300, E=16)
    logits = synth.make_scores(cfg)
    for normalize in (True, False):
        idx, w = oracle.gate(logits, None, 4, score_fn=SOFTMAX, normalize=normalize)
        L = logits.astype(np.longdouble)
        p = np.exp(L - L.max(axis=1, keepdims=True))
        p = p / p.sum(axis=1, keepdims=True)
        sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        ref = sel / sel.sum(axis=1, keepdims=True) if normalize else sel
        np.testing.assert_allclose(w, ref.astype(np.float64), rtol=1e-13, atol=0)


def test_gate_raw_weights_normalised_and_proportional():
    cfg = synth.config("dsv3", T=400)
    inp = synth.make_inputs(cfg)
    idx, w = oracle.gate(inp["scores"], inp["bias"], 8, 8, 4, 2, RAW, True)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=8 * 2.0 ** -52)
    s_sel = np.take_along_axis(inp["scores"].astype(np.float64), idx.astype(np.int64), axis=1)
    # w is the unbiased score over the sum of the chosen unbiased scores
    np.testing.assert_allclose(w * s_sel.sum(axis=1, keepdims=True), s_sel, rtol=1e-14)
    _, w_raw = oracle.gate(inp["scores"], inp["bias"], 8, 8, 4, 2, RAW, False)
    np.testing.assert_array_equal(w_raw, s_sel)


def test_gate_group_limit_invariants_dsv3_shape():
    """On the 256-expert shape: chosen experts are distinct, span at most 4
    groups, every kept group outscores every dropped one, and inside the kept
    groups no unchosen expert has a larger key than a chosen one."""
    cfg = synth.config("dsv3", T=512)
    inp = synth.make_inputs(cfg)
    s, b = inp["scores"], inp["bias"]
    idx, _ = oracle.gate(s, b, 8, 8, 4, 2, RAW, True)
    key = _keys(s, b)
    for t in range(cfg["T"]):
        e = idx[t]
        assert len(set(e.tolist())) == 8
        groups = set((e // 32).tolist())
        assert len(groups) <= 4
        ks = key[t].reshape(8, 32)
        top2 = np.sort(ks, axis=1)[:, ::-1][:, :2]
        gsc = (top2[:, 0] + top2[:, 1]).astype(np.float32)
        order = sorted(range(8), key=lambda g: (-float(gsc[g]), g))
        kept = set(order[:4])
        assert groups <= kept
        in_kept = np.array([x for x in range(256) if x // 32 in kept])
        unchosen = np.setdiff1d(in_kept, e)
        assert key[t, e].min() >= key[t, unchosen].max()
        # slot order: descending key
        assert np.all(np.diff(key[t, e]) <= 0)


def test_gate_bias_only_selects():
    """A large bias on one expert makes it selected for every token, but the
    weight it gets is still its unbiased score's share."""
    rng = np.random.default_rng(3)
    s = rng.uniform(0.1, 1.0, size=(50, 16)).astype(np.float32)
    b = np.zeros(16, np.float32)
    b[11] = 10.0
    idx, w = oracle.gate(s, b, 2, score_fn=RAW, normalize=True)
    assert np.all(idx[:, 0] == 11)
    other = idx[:, 1]
    np.testing.assert_allclose(w[:, 0], s[:, 11] / (s[:, 11].astype(np.float64) + s[np.arange(50), other]), rtol=1e-15)


def test_gate_golden_hand_cases(golden_dir):
    with open(os.path.join(golden_dir, "gate_group_limited_e8.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        s = np.array([case["scores"]], np.float32)
        b = None if case["bias"] is None else np.array(case["bias"], np.float32)
        idx, w = oracle.gate(s, b, case["k"], case["n_groups"], case["topk_group"],
                             case["topk_in_group"], RAW, True)
        assert idx[0].tolist() == case["topk_idx"], case["name"]
        for got, num in zip(w[0], case["topk_w_num"]):
            assert Fraction(got).limit_denominator(1000) == Fraction(num, case["topk_w_den"]), case["name"]


def test_gate_rejects_bad_arguments():
    s = np.ones((2, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.gate(s, None, 9)                       # k > E
    with pytest.raises(ValueError):
        oracle.gate(s, None, 2, n_groups=3)           # E % G != 0
    with pytest.raises(ValueError):
        oracle.gate(s, None, 5, n_groups=4, topk_group=2)   # Kg * E/G < k
