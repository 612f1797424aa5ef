"""GPU parity of step 1 (gating) against the CPU oracle.

Indices must match bit for bit (the decisions are taken in fp32 on both
sides); weights within the derived tolerance (tests/gpu_util.py)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_weights_close, dev, ep_cfg, gate_args, weight_rtol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _run(ep, cfg, scores, bias):
    s_d = dev(scores)
    b_d = None if bias is None else dev(bias)
    idx, w = ep.ep_gate(s_d, b_d, ep_cfg(ep, cfg))
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def _check(ep, cfg, scores, bias):
    gi, gw = _run(ep, cfg, scores, bias)
    oi, ow = oracle.gate(scores, bias, *gate_args(cfg))
    np.testing.assert_array_equal(gi, oi)
    assert_weights_close(gw, ow, weight_rtol(cfg, scores, oi))


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_gate_full_size(ep, name):
    cfg = synth.config(name)
    _check(ep, cfg, synth.make_scores(cfg), synth.make_bias(cfg))


@pytest.mark.parametrize("E,G,Kg,kin,k", [
    (8, 1, 1, 1, 2), (8, 4, 2, 2, 2), (12, 3, 2, 3, 4), (40, 5, 2, 4, 7), (64, 8, 3, 2, 6),
    (96, 12, 5, 2, 9), (200, 8, 4, 2, 8), (256, 8, 4, 2, 8), (256, 32, 6, 4, 16), (320, 16, 3, 1, 5),
    (512, 16, 4, 2, 32), (33, 1, 1, 1, 32), (1, 1, 1, 1, 1),
])
def test_gate_shapes_with_ties(ep, E, G, Kg, kin, k):
    """Few distinct score levels force equal keys and equal group scores; a
    ragged token count leaves a partial CTA."""
    rng = np.random.default_rng(E * 7 + k)
    T = 37
    scores = (rng.integers(1, 9, size=(T, E)) / 8).astype(np.float32)
    bias = (rng.integers(-2, 3, size=E) / 16).astype(np.float32)
    cfg = dict(k=k, n_groups=G, topk_group=Kg, topk_in_group=kin, score_fn=synth.SCORE_RAW, normalize=True, E=E)
    _check(ep, cfg, scores, bias)
    _check(ep, cfg, scores, None)


def test_gate_signed_zero_keys_tie(ep):
    """-0.0 and +0.0 keys are equal: the lower index wins either way."""
    scores = np.zeros((4, 8), np.float32)
    scores[0, 3] = -0.0
    scores[1, :] = -0.0
    scores[2, 5] = 1.0
    scores[3, ::2] = -0.0
    cfg = dict(k=3, n_groups=1, topk_group=1, topk_in_group=1, score_fn=synth.SCORE_RAW, normalize=False, E=8)
    gi, gw = _run(ep, cfg, scores, None)
    oi, ow = oracle.gate(scores, None, *gate_args(cfg))
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gw, ow.astype(np.float32))


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("with_bias", [True, False])
def test_gate_softmax_modes(ep, normalize, with_bias):
    cfg = synth.config("decode", T=200, normalize=normalize)
    scores = synth.make_scores(cfg)
    bias = (synth.normal_f64(5, 9, (cfg["E"],)) * 0.5).astype(np.float32) if with_bias else None
    _check(ep, cfg, scores, bias)


def test_gate_raw_unnormalised_is_the_score(ep):
    cfg = synth.config("dsv3", T=300, normalize=False)
    scores, bias = synth.make_scores(cfg), synth.make_bias(cfg)
    gi, gw = _run(ep, cfg, scores, bias)
    oi, _ = oracle.gate(scores, bias, *gate_args(cfg))
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gw, np.take_along_axis(scores, oi.astype(np.int64), axis=1))


@pytest.mark.parametrize("T", [0, 1, 7, 9])
def test_gate_small_token_counts(ep, T):
    cfg = synth.config("dsv3", T=max(T, 1))
    scores = synth.make_scores(cfg)[:T]
    bias = synth.make_bias(cfg)
    gi, gw = _run(ep, cfg, scores, bias)
    assert gi.shape == (T, 8)
    if T:
        oi, ow = oracle.gate(scores, bias, *gate_args(cfg))
        np.testing.assert_array_equal(gi, oi)
        assert_weights_close(gw, ow, weight_rtol(cfg, scores, oi))


@pytest.mark.parametrize("E,G,Kg,kin,k", [(256, 1, 1, 1, 8), (256, 8, 4, 2, 8), (64, 1, 1, 1, 4), (8, 1, 1, 1, 2)])
def test_gate_planted_ties_at_and_inside_the_top_k(ep, E, G, Kg, kin, k):
    """Distinct random keys except where planted: one third of the tokens
    get a key equal to their k-th largest just outside the top k (the lower
    index must win the last slot), one third two equal keys inside the top
    k (lower index first), the rest none -- the warp's merged top-k path
    serves the last third, the round-by-round path the others."""
    rng = np.random.default_rng(E + k)
    T = 66
    scores = rng.normal(0, 1, size=(T, E)).astype(np.float32)
    for t in range(T):
        order = np.argsort(-scores[t], kind="stable")
        if t % 3 == 0 and k < E:
            a, b = sorted((order[k - 1], order[k]))
            scores[t, b] = scores[t, a]         # the k-th key, twice
        elif t % 3 == 1 and k > 1:
            scores[t, order[1]] = scores[t, order[0]]
    cfg = dict(k=k, n_groups=G, topk_group=Kg, topk_in_group=kin, score_fn=synth.SCORE_RAW, normalize=True, E=E)
    _check(ep, cfg, scores, None)
    cfg["score_fn"] = synth.SCORE_SOFTMAX
    _check(ep, cfg, scores, None)
