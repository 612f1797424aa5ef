"""GPU parity of the lane-segment gating kernel (a token served by L lanes of
E/L experts) against the CPU oracle, on the shapes it serves: every E it
takes, groups of one, two and four lanes, group scores of one to four keys,
bounds of one to four keys per lane, ties that overflow the candidate list,
signed zeros, the renormalised softmax; and on rows it hands to the
warp-per-token kernel (misaligned score rows), which must agree with it."""
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


def _cfg(E, k, G=1, Kg=1, kin=1, score_fn=synth.SCORE_RAW, normalize=True):
    return dict(E=E, k=k, n_groups=G, topk_group=Kg, topk_in_group=kin, score_fn=score_fn, normalize=normalize)


def _check(ep, cfg, scores, bias):
    s_d = dev(scores)
    b_d = None if bias is None else dev(bias)
    gi, gw = ep.ep_gate(s_d, b_d, ep_cfg(ep, cfg))
    torch.cuda.synchronize()
    oi, ow = oracle.gate(scores, bias, *gate_args(cfg))
    np.testing.assert_array_equal(gi.cpu().numpy(), oi)
    assert_weights_close(gw.cpu().numpy(), ow, weight_rtol(cfg, scores, oi))
    return gi, gw


# (E, k, G, Kg, kin): E = 8 .. 256 (1 .. 8 lanes per token); groups of 1, 2, 4
# lanes (E/G a multiple of the lane's experts); bounds of 1, 2, 4 keys a lane.
SHAPES = [
    (8, 2, 1, 1, 1), (8, 8, 1, 1, 1), (16, 3, 1, 1, 1), (16, 4, 2, 1, 2), (32, 5, 4, 2, 2), (32, 16, 1, 1, 1),
    (64, 6, 8, 3, 2), (64, 8, 4, 2, 4), (64, 9, 2, 1, 3), (128, 8, 1, 1, 1), (128, 8, 8, 4, 2), (128, 12, 4, 2, 4),
    (128, 32, 1, 1, 1), (256, 8, 8, 4, 2), (256, 8, 8, 4, 1), (256, 8, 8, 4, 4), (256, 6, 4, 1, 3),
    (256, 16, 8, 4, 2), (256, 32, 8, 2, 4), (256, 8, 2, 1, 2), (256, 1, 8, 1, 1), (256, 8, 1, 1, 1),
]


@pytest.mark.parametrize("E,k,G,Kg,kin", SHAPES)
def test_gate_fast_shapes_continuous(ep, E, k, G, Kg, kin):
    """Continuous scores (ties rare); a ragged token count leaves a partial CTA."""
    rng = np.random.default_rng(E * 131 + k * 7 + G)
    T = 301
    scores = rng.random((T, E), dtype=np.float32)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    cfg = _cfg(E, k, G, Kg, kin)
    _check(ep, cfg, scores, bias)
    _check(ep, cfg, scores, None)


@pytest.mark.parametrize("E,k,G,Kg,kin", SHAPES)
def test_gate_fast_shapes_with_ties(ep, E, k, G, Kg, kin):
    """Few distinct levels: equal keys, equal group scores, and (for E >= 128)
    more tied candidates than the list holds, which takes the exact
    threshold search."""
    rng = np.random.default_rng(E * 17 + k)
    T = 97
    scores = (rng.integers(1, 5, size=(T, E)) / 4).astype(np.float32)
    bias = (rng.integers(-1, 2, size=E) / 8).astype(np.float32)
    cfg = _cfg(E, k, G, Kg, kin)
    _check(ep, cfg, scores, bias)
    _check(ep, cfg, scores, None)


@pytest.mark.parametrize("E,k,G,Kg,kin", [(256, 8, 8, 4, 2), (256, 8, 1, 1, 1), (128, 32, 1, 1, 1),
                                          (64, 6, 8, 3, 2), (8, 2, 1, 1, 1)])
def test_gate_fast_all_equal_scores(ep, E, k, G, Kg, kin):
    """Every key equal: the lowest-index groups and experts win, in index
    order; every token overflows the candidate list at E >= 128."""
    T = 40
    scores = np.full((T, E), 0.5, np.float32)
    cfg = _cfg(E, k, G, Kg, kin)
    gi, _ = _check(ep, cfg, scores, None)
    if G == 1:
        np.testing.assert_array_equal(gi.cpu().numpy(), np.tile(np.arange(k, dtype=np.int32), (T, 1)))


def test_gate_fast_signed_zero_keys(ep):
    """-0.0 and +0.0 give equal keys on every lane width."""
    for E in (8, 64, 256):
        scores = np.zeros((6, E), np.float32)
        scores[0, 3] = -0.0
        scores[1, :] = -0.0
        scores[2, E // 2] = 1.0
        scores[3, ::2] = -0.0
        scores[4, 1::3] = -0.0
        scores[5, E - 1] = 1.0
        bias = np.zeros(E, np.float32)
        bias[::5] = -0.0
        cfg = _cfg(E, 3, normalize=False)
        for b in (None, bias):
            gi, gw = _check(ep, cfg, scores, b)


@pytest.mark.parametrize("E", [8, 128, 256])
def test_gate_fast_softmax_renormalised(ep, E):
    T = 515
    cfg = dict(_cfg(E, 8 if E > 8 else 2, score_fn=synth.SCORE_SOFTMAX, normalize=True))
    logits = synth.normal_f64(E, 3, (T, E)).astype(np.float32)
    bias = (synth.normal_f64(E, 4, (E,)) * 0.3).astype(np.float32)
    _check(ep, cfg, logits, None)
    _check(ep, cfg, logits, bias)


def test_gate_fast_and_warp_per_token_agree(ep):
    """A score tensor whose rows are not 16-byte aligned goes to the
    warp-per-token kernel; both kernels give the same bits."""
    cfg = synth.config("dsv3", T=999)
    scores, bias = synth.make_scores(cfg), synth.make_bias(cfg)
    gc = ep_cfg(ep, cfg)
    aligned = dev(scores)
    buf = torch.zeros(scores.size + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(aligned.reshape(-1))
    shifted = buf[1:].view(scores.shape)                 # base 4 bytes past a 16-byte boundary
    b = dev(bias)
    i1, w1 = ep.ep_gate(aligned, b, gc)
    i2, w2 = ep.ep_gate(shifted, b, gc)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(w1, w2)
