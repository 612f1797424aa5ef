"""ep_get_layout_noalloc: the dispatch layout for callers that cannot
allocate device memory at call time (a plugin inside another runtime whose
pool owns the device memory, or a serving loop with a fixed memory budget).
Its scratch is a fixed array inside the library, shared by every call.

Checked through the C ABI against ep_get_layout (caller-provided workspace)
on two calls in a row with different routings, and on one call per layout
kernel back to back, so that whatever a call leaves in the shared array
cannot leak into the next.  The layout is
integer work, so the bar is bit-exact, as in the other layout tests.  This
file is collected last so that a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, gate_args

KEYS = ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "pos", "src")


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _routing(name, T=None):
    cfg = synth.config(name, **({} if T is None else {"T": T}))
    idx, _ = oracle.gate(synth.make_scores(cfg), synth.make_bias(cfg), *gate_args(cfg))
    return cfg, idx


@pytest.mark.gpu
def test_noalloc_layout_matches_workspace_layout_twice(ep):
    cases = [_routing("dsv3"), _routing("skewed")]
    outs = []
    for cfg, idx in cases:
        T, k, E, epr = cfg["T"], cfg["k"], cfg["E"], cfg["experts_per_rank"]
        d_idx = dev(idx)
        ref = ep.ep_get_layout(d_idx, E, epr)
        got = ep.alloc_layout(T, k, E, epr)
        for t in got:
            t.fill_(-12345)
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_get_layout_noalloc(d_idx, E, epr, got, err_flag=flag)
        torch.cuda.synchronize()
        for key in KEYS:
            np.testing.assert_array_equal(getattr(got, key).cpu().numpy(), getattr(ref, key).cpu().numpy(),
                                          err_msg=key)
        assert int(flag.item()) == 0
        outs.append(got.pos.cpu().numpy())
    assert not np.array_equal(outs[0], outs[1])     # the two calls really saw different routings


def _check_noalloc(ep, idx, E, epr):
    T, k = idx.shape
    d_idx = dev(idx)
    ref = ep.ep_get_layout(d_idx, E, epr)
    got = ep.alloc_layout(T, k, E, epr)
    for t in got:
        t.fill_(-12345)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_get_layout_noalloc(d_idx, E, epr, got, err_flag=flag)
    torch.cuda.synchronize()
    for key in KEYS:
        np.testing.assert_array_equal(getattr(got, key).cpu().numpy(), getattr(ref, key).cpu().numpy(),
                                      err_msg=key)
    assert int(flag.item()) == 0


@pytest.mark.gpu
def test_noalloc_layout_every_kernel_path_back_to_back(ep):
    """One call per layout kernel, back to back on the shared scratch, each
    checked bit for bit against ep_get_layout: the grid-wide kernel (which
    keeps its barrier count and per-cluster rows in the scratch), the three
    tile kernels (per-tile counts in the scratch), the one-CTA kernel, the
    one-cluster kernel (neither touches the scratch), and the grid-wide
    kernel again on a different routing, after the tile kernels have left
    their counts in the array."""
    rng = np.random.default_rng(3)
    cfg, idx = _routing("qwen3")                          # 131072 entries: the grid-wide kernel
    _check_noalloc(ep, idx, cfg["E"], cfg["experts_per_rank"])
    big = np.argsort(rng.random((30000, 256)), axis=1)[:, :8].astype(np.int32)
    assert ep.ep_layout_workspace_bytes(30000, 8, 256, 8) <= (1 << 20)
    _check_noalloc(ep, big, 256, 8)                       # more than 128 tokens a CTA: the tile kernels
    cfg, idx = _routing("tiny")                           # 256 entries: the one-CTA kernel
    _check_noalloc(ep, idx, cfg["E"], cfg["experts_per_rank"])
    cfg, idx = _routing("mixtral")                        # 8192 entries: the one-cluster kernel
    _check_noalloc(ep, idx, cfg["E"], cfg["experts_per_rank"])
    cfg, idx = _routing("dsv3", T=10000)                  # 80000 entries: the grid-wide kernel again
    _check_noalloc(ep, idx, cfg["E"], cfg["experts_per_rank"])


@pytest.mark.gpu
def test_noalloc_layout_rejects_sizes_beyond_its_scratch(ep):
    T, k, E, epr = 400000, 8, 256, 8                 # needs more than the fixed 1 MiB of scratch
    assert ep.ep_layout_workspace_bytes(T, k, E, epr) > (1 << 20)
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    out = ep.alloc_layout(T, k, E, epr)
    with pytest.raises(ep.EpError) as ei:
        ep.ep_get_layout_noalloc(idx, E, epr, out)
    assert ei.value.status == ep.EP_ERR_UNSUPPORTED
