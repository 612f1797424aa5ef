"""GPU parity of the routing call ep_gate_layout (one clustered launch for
batches of at most 4096 entries and 512 tokens; one grid-wide launch for
group-limited batches past 4096 entries and for batches past 65536 entries;
the gate kernel then the one-CTA or one-cluster layout otherwise) and of
ep_get_layout past 4096 entries (one cluster, the grid-wide launch, or three
launches for the largest batches), against the CPU oracle and against the
separate calls; the grid barrier's bounded wait reports a workspace whose
barrier words are not clear."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_weights_close, dev, ep_cfg, gate_args, weight_rtol

pytestmark = pytest.mark.gpu

KEYS = ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "pos", "src")


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _check_layout(lay, ol):
    for key in KEYS:
        np.testing.assert_array_equal(getattr(lay, key).cpu().numpy().reshape(ol[key].shape), ol[key], err_msg=key)


@pytest.mark.parametrize("name,T", [(n, None) for n in synth.CONFIGS] + [
    ("dsv3", 1), ("dsv3", 2), ("dsv3", 9), ("dsv3", 151), ("dsv3", 152), ("dsv3", 153), ("dsv3", 512),
    ("qwen3", 300), ("mixtral", 512), ("mixtral", 513), ("tiny", 1000), ("dsv3", 1000), ("skewed", 3001),
    ("qwen3", 40000), ("mixtral", 70001), ("dsv3", 100003),
])
def test_gate_layout_matches_oracle_and_separate_calls(ep, name, T):
    cfg = synth.config(name) if T is None else synth.config(name, T=T)
    scores = synth.make_scores(cfg)
    bias = synth.make_bias(cfg)
    s = dev(scores)
    b = None if bias is None else dev(bias)
    gc = ep_cfg(ep, cfg)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w, lay = ep.ep_gate_layout(s, b, gc, cfg["experts_per_rank"], err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    oi, ow = oracle.gate(scores, bias, *gate_args(cfg))
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    assert_weights_close(w.cpu().numpy(), ow, weight_rtol(cfg, scores, oi))
    _check_layout(lay, oracle.layout(oi, cfg["E"], cfg["experts_per_rank"]))
    # the separate calls give the same bits
    si, sw = ep.ep_gate(s, b, gc)
    slay = ep.ep_get_layout(si, cfg["E"], cfg["experts_per_rank"])
    torch.cuda.synchronize()
    assert torch.equal(si, idx) and torch.equal(sw, w)
    for key in KEYS:
        assert torch.equal(getattr(slay, key), getattr(lay, key)), key


def test_gate_layout_repeated_on_one_workspace(ep):
    """The barrier's arrival count is left clear, so a workspace is reused
    as is."""
    cfg = synth.config("dsv3")
    s, b = dev(synth.make_scores(cfg)), dev(synth.make_bias(cfg))
    gc = ep_cfg(ep, cfg)
    T, k, E, epr = cfg["T"], cfg["k"], cfg["E"], cfg["experts_per_rank"]
    ws = ep.alloc_layout_workspace(T, k, E, epr)
    ref = ep.ep_gate_layout(s, b, gc, epr, workspace=ws)
    for _ in range(3):
        got = ep.ep_gate_layout(s, b, gc, epr, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        for key in KEYS:
            assert torch.equal(getattr(got[2], key), getattr(ref[2], key)), key
    assert int(ws[:4].count_nonzero().item()) == 0


@pytest.mark.parametrize("T,k,E,epr", [(2000, 4, 64, 8), (4097, 1, 16, 2), (30000, 8, 256, 8), (600, 64, 1024, 16),
                                       (70000, 8, 160, 20)])
def test_cooperative_layout_random_with_skips_and_bad_indices(ep, T, k, E, epr):
    """More than 4096 entries (the one-cluster, grid-wide and three-launch
    layouts), on index tensors with -1 slots, repeated experts and
    out-of-range values."""
    rng = np.random.default_rng(T + k + E)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    idx[rng.random((T, k)) < 0.001] = E + 5
    idx[0, 0] = -7
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.ep_get_layout(dev(idx), E, epr, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == ep.EP_FLAG_BAD_EXPERT
    clean = idx.copy()
    clean[(clean < -1) | (clean >= E)] = -1
    _check_layout(lay, oracle.layout(clean, E, epr))


def test_uncleared_barrier_words_time_out_and_report(ep):
    """A workspace whose barrier count is not clear: no arrival completes the
    barrier, every CTA gives up after its bounded wait, sets EP_FLAG_TIMEOUT
    and returns; once cleared, the same workspace works."""
    cfg = synth.config("dsv3", T=2048)
    s, b = dev(synth.make_scores(cfg)), dev(synth.make_bias(cfg))
    gc = ep_cfg(ep, cfg)
    T, k, E, epr = cfg["T"], cfg["k"], cfg["E"], cfg["experts_per_rank"]
    ws = ep.alloc_layout_workspace(T, k, E, epr)
    ws[:4].view(torch.int32).fill_(1 << 30)          # an arrival count no grid reaches
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_gate_layout(s, b, gc, epr, workspace=ws, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & ep.EP_FLAG_TIMEOUT
    ws[:4].zero_()
    flag.zero_()
    idx, w, lay = ep.ep_gate_layout(s, b, gc, epr, workspace=ws, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    oi, _ = oracle.gate(synth.make_scores(cfg), synth.make_bias(cfg), *gate_args(cfg))
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    _check_layout(lay, oracle.layout(oi, E, epr))
