"""GPU parity of the one-cluster layout kernel (ep_get_layout from 4097 to
65536 entries, and capacity layouts up to 65536 entries) against the CPU
oracle: clusters of 1 to 16 CTAs, ranking blocks cut mid-CTA, repeated
experts within a token (the counting path), skipped and invalid entries,
capacities from 0 to past the batch, and the first batch past the cluster
(which takes the grid-wide kernel)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev

pytestmark = pytest.mark.gpu

KEYS = ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "pos", "src")
CAP_KEYS = KEYS + ("expert_dropped",)


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _indices(rng, T, k, E, distinct, p_skip=0.02, p_bad=0.0):
    if distinct:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int64)
    else:
        idx = rng.integers(0, E, size=(T, k)).astype(np.int64)
    idx[rng.random((T, k)) < p_skip] = -1
    if p_bad:
        idx[rng.random((T, k)) < p_bad] = E + 1
    return idx.astype(np.int32)


def _clean(idx, E):
    c = idx.copy()
    c[(c < -1) | (c >= E)] = -1
    return c


def _dropless(ep, idx, E, epr):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.ep_get_layout(dev(idx), E, epr, err_flag=flag)
    torch.cuda.synchronize()
    o = oracle.layout(_clean(idx, E), E, epr)
    for key in KEYS:
        np.testing.assert_array_equal(getattr(lay, key).cpu().numpy().reshape(o[key].shape), o[key], err_msg=key)
    return int(flag.item())


def _capacity(ep, idx, E, epr, cap):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.ep_get_layout_capacity(dev(idx), E, epr, cap, err_flag=flag)
    torch.cuda.synchronize()
    o = oracle.layout_capacity(_clean(idx, E), E, epr, cap)
    for key in CAP_KEYS:
        got = getattr(lay, key).cpu().numpy().reshape(-1)[: o[key].size]
        np.testing.assert_array_equal(got, o[key].reshape(-1), err_msg="capacity " + key)
    return int(flag.item())


# T: 513 tokens = 17 blocks (a 16-CTA cluster with one CTA of two blocks);
# 8192 and 16384: the DeepSeek-V3 and Qwen3 batch sizes; 1000 / 5000:
# ragged last blocks.
@pytest.mark.parametrize("T,k,E,epr", [(513, 8, 256, 8), (1000, 6, 64, 8), (5000, 2, 8, 1), (8192, 8, 256, 8),
                                       (16384, 8, 128, 8), (2049, 3, 1024, 32), (4097, 1, 16, 16)])
@pytest.mark.parametrize("distinct", [True, False])
def test_cluster_layout_dropless(ep, T, k, E, epr, distinct):
    rng = np.random.default_rng(T * 3 + k + E + distinct)
    idx = _indices(rng, T, k, E, distinct, p_bad=0.001)
    flag = _dropless(ep, idx, E, epr)
    assert flag == (ep.EP_FLAG_BAD_EXPERT if (idx >= E).any() else 0)


@pytest.mark.parametrize("T,k,E,epr", [(1, 8, 256, 8), (32, 8, 256, 8), (33, 4, 64, 8), (128, 8, 256, 8),
                                       (512, 2, 8, 4), (8192, 8, 256, 8), (3000, 5, 96, 12)])
@pytest.mark.parametrize("factor", [0.0, 0.5, 1.0, 3.0])
def test_cluster_layout_capacity(ep, T, k, E, epr, factor):
    rng = np.random.default_rng(T + k * 5 + int(factor * 10))
    idx = _indices(rng, T, k, E, distinct=(T % 2 == 0), p_bad=0.002)
    idx[: T // 3, 0] = 3                      # a hot expert that overflows
    cap = int(np.ceil(factor * T * k / E))
    _capacity(ep, idx, E, epr, cap)


def test_cluster_layout_one_token_many_repeats(ep):
    """Every slot of a token names the same expert, in every token."""
    T, k, E = 700, 8, 64
    idx = np.full((T, k), 5, np.int32)
    idx[::7, 3] = 9
    _dropless(ep, idx, E, 8)
    _capacity(ep, idx, E, 8, 100)


@pytest.mark.parametrize("T", [8192, 8193])
def test_cluster_layout_size_boundary(ep, T):
    """8192 tokens at k=8 (65536 entries) are the largest dropless batch the
    cluster kernel takes; one more token runs on the grid-wide kernel; both
    match the oracle."""
    rng = np.random.default_rng(T)
    idx = _indices(rng, T, 8, 256, distinct=True)
    _dropless(ep, idx, 256, 8)
    _capacity(ep, idx, 256, 8, T * 8 // 256)


def test_cluster_layout_repeated_calls_agree(ep):
    """Back-to-back launches on one stream (each may start its prologue
    while the previous one finishes) give the same bits."""
    rng = np.random.default_rng(5)
    idx = dev(_indices(rng, 8192, 8, 256, distinct=True))
    ref = ep.ep_get_layout(idx, 256, 8)
    outs = [ep.ep_get_layout(idx, 256, 8) for _ in range(6)]
    torch.cuda.synchronize()
    for o in outs:
        for key in KEYS:
            assert torch.equal(getattr(o, key), getattr(ref, key)), key
