"""Pins for the oracle's dispatch layout (step 2) and BF16 dispatch (step 3).

Experts are placed whole on logical ranks, ``experts_per_rank`` contiguous
experts each ("Expert Parallelism (Parallelisme d'experts)", section "Le
principe de base"); dispatch sends each token to the holders of its experts
(section "Le pattern de communication all-to-all", Phase 1).  The pins: a
hand-worked example with 8 experts on 4 ranks, numpy's stable argsort and
bincount, and the bijection / stability invariants.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth


def _check_against_numpy(idx, E, epr):
    T, k = idx.shape
    R = E // epr
    lay = oracle.layout(idx, E, epr)
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    # counts and offsets
    cnt = np.bincount(flat[valid], minlength=E)
    np.testing.assert_array_equal(lay["expert_count"], cnt)
    np.testing.assert_array_equal(lay["expert_off"], np.concatenate([[0], np.cumsum(cnt)]))
    rc = cnt.reshape(R, epr).sum(axis=1)
    np.testing.assert_array_equal(lay["rank_count"], rc)
    np.testing.assert_array_equal(lay["rank_off"], np.concatenate([[0], np.cumsum(rc)]))
    # distinct tokens per rank
    rt = np.zeros(R, np.int64)
    for t in range(T):
        for r in {int(e) // epr for e in idx[t] if 0 <= e < E}:
            rt[r] += 1
    np.testing.assert_array_equal(lay["rank_tokens"], rt)
    # receive rows: stable sort of the valid entries by expert
    order = np.flatnonzero(valid)[np.argsort(flat[valid], kind="stable")]
    want_pos = np.full(T * k, -1, np.int64)
    want_pos[order] = np.arange(order.size)
    np.testing.assert_array_equal(lay["pos"].reshape(-1), want_pos)
    want_src = np.full(T * k, -1, np.int64)
    want_src[: order.size] = order
    np.testing.assert_array_equal(lay["src"], want_src)
    return lay


def test_layout_golden_8_experts_4_ranks(golden_dir):
    with open(os.path.join(golden_dir, "layout_8experts_4ranks.json")) as f:
        g = json.load(f)
    lay = oracle.layout(np.array(g["topk_idx"], np.int32), g["num_experts"], g["experts_per_rank"])
    for key in ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "pos", "src"):
        assert lay[key].tolist() == g[key], key
    assert lay["err_flag"] == 0


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "qwen3", "decode"])
def test_layout_matches_stable_argsort(name):
    cfg = synth.config(name, T=min(synth.CONFIGS[name]["T"], 1024))
    inp = synth.make_inputs(cfg)
    idx, _ = oracle.gate(inp["scores"], inp["bias"], cfg["k"], cfg["n_groups"], cfg["topk_group"],
                         cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])
    lay = _check_against_numpy(idx, cfg["E"], cfg["experts_per_rank"])
    N = cfg["T"] * cfg["k"]
    assert lay["expert_off"][-1] == N
    assert sorted(lay["pos"].reshape(-1).tolist()) == list(range(N))      # bijection
    assert sum(lay["rank_tokens"]) <= cfg["T"] * min(cfg["k"], cfg["E"] // cfg["experts_per_rank"])


def test_layout_arbitrary_indices_with_duplicates_and_skips():
    rng = np.random.default_rng(11)
    idx = rng.integers(-1, 12, size=(333, 5)).astype(np.int32)   # -1 = empty slot
    lay = _check_against_numpy(idx, 12, 3)
    assert lay["err_flag"] == 0
    assert lay["expert_off"][-1] == int((idx >= 0).sum())


def test_layout_out_of_range_sets_flag_and_is_skipped():
    idx = np.array([[0, 1], [2, 9], [-5, 3]], np.int32)
    lay = oracle.layout(idx, 4, 2)
    assert lay["err_flag"] & 1
    assert lay["pos"][1, 1] == -1 and lay["pos"][2, 0] == -1
    assert lay["expert_off"][-1] == 4


def test_layout_empty_batch():
    lay = oracle.layout(np.zeros((0, 4), np.int32), 8, 2)
    assert lay["expert_off"].tolist() == [0] * 9
    assert lay["rank_tokens"].tolist() == [0] * 4


def test_dispatch_bf16_is_the_permutation():
    cfg = synth.config("tiny")
    inp = synth.make_inputs(cfg)
    idx, _ = oracle.gate(inp["scores"], None, cfg["k"])
    lay = oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])
    recv = oracle.dispatch_bf16(inp["x"], lay["pos"])
    # every received row is the source row of the entry the layout put there
    np.testing.assert_array_equal(recv, inp["x"][lay["src"] // cfg["k"]])
    # and rank r's slice holds only tokens routed to rank r's experts
    for r in range(cfg["E"] // cfg["experts_per_rank"]):
        rows = lay["src"][lay["rank_off"][r]:lay["rank_off"][r + 1]]
        assert np.all(idx.reshape(-1)[rows] // cfg["experts_per_rank"] == r)
