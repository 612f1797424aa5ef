"""GPU parity of step 2 (dispatch layout) against the CPU oracle: every
output array bit-exact, including the stable receive-row order."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, gate_args

pytestmark = pytest.mark.gpu

KEYS = ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "pos", "src")


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _gpu_layout(ep, idx, E, epr):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.ep_get_layout(dev(idx), E, epr, err_flag=flag)
    torch.cuda.synchronize()
    return {k: getattr(lay, k).cpu().numpy() for k in KEYS}, int(flag.item())


def _check(ep, idx, E, epr):
    g, gflag = _gpu_layout(ep, idx, E, epr)
    o = oracle.layout(idx, E, epr)
    for key in KEYS:
        np.testing.assert_array_equal(g[key].reshape(o[key].shape), o[key], err_msg=key)
    assert gflag == o["err_flag"]
    return g


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_layout_full_size(ep, name):
    cfg = synth.config(name)
    idx, _ = oracle.gate(synth.make_scores(cfg), synth.make_bias(cfg), *gate_args(cfg))
    _check(ep, idx, cfg["E"], cfg["experts_per_rank"])


@pytest.mark.parametrize("T,k,E,epr", [
    (1, 1, 1, 1), (1, 8, 256, 8), (5, 3, 12, 4), (255, 8, 256, 8), (257, 8, 256, 8), (1000, 2, 8, 1),
    (3000, 6, 1024, 32), (777, 16, 64, 64), (4097, 1, 16, 2), (300, 64, 1024, 16), (70, 64, 256, 8), (50, 64, 1024, 16),
])
def test_layout_random_with_skips_and_duplicates(ep, T, k, E, epr):
    """Arbitrary index tensors: -1 slots, repeated experts in one token,
    several tiles with a ragged last one."""
    rng = np.random.default_rng(T * 31 + k)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    _check(ep, idx, E, epr)


def test_layout_large_batch(ep):
    """Two million entries (4096 tiles): the multi-tile scan at a size well
    past any of the workloads, against the oracle."""
    rng = np.random.default_rng(11)
    idx = rng.integers(0, 256, size=(262144, 8)).astype(np.int32)
    _check(ep, idx, 256, 8)


def test_layout_every_token_on_the_same_experts(ep):
    """Maximum skew: all 8192 tokens pick experts 0..7 (one rank holds all)."""
    idx = np.tile(np.arange(8, dtype=np.int32), (8192, 1))
    g = _check(ep, idx, 256, 8)
    assert g["rank_count"][0] == 8192 * 8 and g["rank_tokens"][0] == 8192


def test_layout_out_of_range_flagged_and_skipped(ep):
    rng = np.random.default_rng(1)
    idx = rng.integers(0, 64, size=(500, 4)).astype(np.int32)
    idx[3, 1] = 64
    idx[200, 0] = -7
    idx[499, 3] = 1 << 30
    g = _check(ep, idx, 64, 8)
    assert g["pos"].reshape(500, 4)[3, 1] == -1


BAD_VALUES = np.array([-2, -3, -2**31, 2**31 - 1], np.int64)


@pytest.mark.parametrize("T,k,E,epr", [(300, 8, 64, 8), (4096, 1, 16, 2), (40, 64, 1024, 16),
                                       (3000, 6, 64, 8), (20000, 8, 256, 8)])
def test_every_invalid_index_value_is_flagged_and_skipped(ep, T, k, E, epr):
    """Any index outside [0, E) other than -1 -- including -2, INT_MIN and
    INT_MAX -- is flagged and becomes an empty slot, on the one-CTA layout
    (T*k <= 4096), the cooperative layout and the capacity layout."""
    rng = np.random.default_rng(T * k + E)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int64)
    m = rng.random((T, k))
    idx[m < 0.05] = rng.choice(np.append(BAD_VALUES, E), size=int((m < 0.05).sum()))
    idx[0, 0] = -2
    idx = idx.astype(np.int32)
    clean = idx.copy()
    clean[(clean < -1) | (clean >= E)] = -1
    g, gflag = _gpu_layout(ep, idx, E, epr)
    o = oracle.layout(clean, E, epr)
    for key in KEYS:
        np.testing.assert_array_equal(g[key].reshape(o[key].shape), o[key], err_msg=key)
    assert gflag == ep.EP_FLAG_BAD_EXPERT
    cap = max(1, (T * k) // E)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = ep.ep_get_layout_capacity(dev(idx), E, epr, cap, err_flag=flag)
    torch.cuda.synchronize()
    oc = oracle.layout_capacity(clean, E, epr, cap)
    for key in KEYS + ("expert_dropped",):
        got = getattr(c, key).cpu().numpy().reshape(-1)[: oc[key].size]
        np.testing.assert_array_equal(got, oc[key].reshape(-1), err_msg="capacity " + key)
    assert int(flag.item()) == ep.EP_FLAG_BAD_EXPERT


def test_layout_empty_batch(ep):
    idx = np.zeros((0, 8), np.int32)
    lay = ep.ep_get_layout(torch.zeros((0, 8), dtype=torch.int32, device="cuda"), 256, 8)
    torch.cuda.synchronize()
    assert lay.expert_off.cpu().tolist() == [0] * 257
    assert lay.rank_tokens.cpu().tolist() == [0] * 32
    del idx
