"""The seeded generators: determinism, ranges, and the skewed workload's
hot-expert ratio (about 20x the mean receive count)."""
import numpy as np

import oracle
import synth


def test_streams_are_deterministic_and_distinct():
    a = synth.u64(1, 2, 1000)
    np.testing.assert_array_equal(a, synth.u64(1, 2, 1000))
    np.testing.assert_array_equal(a[10:20], synth.u64(1, 2, 10, start=10))
    assert not np.array_equal(a, synth.u64(1, 3, 1000))
    assert not np.array_equal(a, synth.u64(2, 2, 1000))


def test_uniform_open_interval_and_moments():
    u = synth.uniform_f32(7, 1, (200000,))
    assert u.dtype == np.float32 and u.min() > 0 and u.max() < 1
    assert abs(u.mean() - 0.5) < 0.005 and abs(u.var() - 1 / 12) < 0.002


def test_normal_moments_and_bf16():
    z = synth.normal_f64(7, 2, (400001,))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    b = synth.normal_bf16_bits(7, 2, (1000,))
    back = synth.bf16_bits_to_f32(b)
    zz = synth.normal_f64(7, 2, (1000,))
    assert np.all(np.abs(back - zz) <= np.abs(zz) * 2.0 ** -8 + 1e-30)


def test_skewed_workload_hot_expert_ratio():
    cfg = synth.config("skewed")
    inp = dict(scores=synth.make_scores(cfg), bias=synth.make_bias(cfg))
    idx, _ = oracle.gate(inp["scores"], inp["bias"], cfg["k"], cfg["n_groups"], cfg["topk_group"],
                         cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])
    cnt = oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])["expert_count"]
    ratio = cnt.max() / (cfg["T"] * cfg["k"] / cfg["E"])
    assert 18 <= ratio <= 22, ratio


def test_config_shapes():
    for name, c in synth.CONFIGS.items():
        assert c["E"] % c["experts_per_rank"] == 0
        assert c["E"] % c["n_groups"] == 0
        assert c["topk_group"] * (c["E"] // c["n_groups"]) >= c["k"]
        if "fp8" in c["dispatch"]:
            assert c["H"] % 128 == 0
