"""GPU parity of steps 4-5 (inverse gather + weighted combine) against the
CPU oracle: the five workloads with identity experts (y = the dispatched
rows) within the stated bar, max(1 bf16 ulp, 1e-2 relative); arbitrary
expert outputs and signed weights within that bar plus the fp32
accumulation term (tests/gpu_util.py)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_combine_close, dev, dev_bf16, ep_cfg, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _combine_both(ep, y_bits, pos, w, flag=None):
    T, k = pos.shape
    H = y_bits.shape[1]
    out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(dev_bf16(y_bits), dev(pos), dev(w), out=out, err_flag=flag)
    torch.cuda.synchronize()
    g = host_bits(out)
    ref_pos = np.where(pos >= T * k, -1, pos).astype(np.int32)
    r = oracle.combine(y_bits, ref_pos, w)
    assert_combine_close(g, r, y_bits, ref_pos, w)
    return g, r


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_combine_full_size_identity_experts(ep, name):
    """The path on device: gate -> layout -> BF16 dispatch -> combine with
    identity experts; the oracle combines the same rows with the same weights
    (the tolerance also covers the round trip back to x)."""
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    idx, w = ep.ep_gate(dev(inp["scores"]), None if inp["bias"] is None else dev(inp["bias"]), ep_cfg(ep, cfg))
    lay = ep.ep_get_layout(idx, cfg["E"], cfg["experts_per_rank"])
    recv = ep.ep_dispatch(dev_bf16(inp["x"]), lay.pos, "bf16")
    out = ep.ep_combine(recv, lay.pos, w)
    torch.cuda.synchronize()
    pos, wh, y = lay.pos.cpu().numpy(), w.cpu().numpy(), host_bits(recv)
    r = oracle.combine(y, pos, wh)
    g = host_bits(out)
    assert_combine_close(g, r, y, pos, wh, accumulation=False)   # the stated bar alone
    # weights sum to one: the round trip gives x back to within a bf16 ulp
    x = synth.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    o = synth.bf16_bits_to_f32(g).astype(np.float64)
    from gpu_util import bf16_ulp
    assert np.all(np.abs(o - x) <= bf16_ulp(x) + 16 * 2.0 ** -24 * np.abs(x))


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "qwen3", "decode"])
def test_combine_full_size_arbitrary_outputs(ep, name):
    cfg = synth.config(name)
    rows = cfg["T"] * cfg["k"]
    y = synth.make_expert_out(cfg, rows)
    pos = synth.permutation(cfg["seed"], 77, rows).reshape(cfg["T"], cfg["k"]).astype(np.int32)
    w = synth.make_weights(cfg)
    _combine_both(ep, y, pos, w)


@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (5, 16, 3), (33, 264, 8), (64, 7168, 9), (300, 512, 17), (7, 64, 40), (5, 16384, 64),
                                   (2100, 64, 1), (2500, 1032, 2)])   # the last two: one warp per token
def test_combine_small_shapes_signed_weights_empty_slots(ep, T, H, k):
    rng = np.random.default_rng(T + H + k)
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (T * k, H)).astype(np.float32))
    pos = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.25] = -1
    w = rng.uniform(-2, 2, (T, k)).astype(np.float32)
    _combine_both(ep, y, pos, w)


def test_combine_bad_rows_flagged_and_skipped(ep):
    rng = np.random.default_rng(2)
    T, H, k = 50, 128, 4
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (T * k, H)).astype(np.float32))
    pos = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    pos[0, 0] = T * k
    pos[49, 3] = 1 << 29
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    _combine_both(ep, y, pos, w, flag)
    assert int(flag.item()) == 2


def test_combine_all_slots_empty_gives_zero(ep):
    y = np.zeros((8, 64), np.uint16)
    pos = np.full((2, 4), -1, np.int32)
    g, _ = _combine_both(ep, synth.f32_to_bf16_bits(np.ones((8, 64), np.float32)), pos, np.ones((2, 4), np.float32))
    assert np.all(g == 0)
    del y


@pytest.mark.parametrize("k,unit", [(8, False), (2, False), (8, True)])
def test_combine_decode_sized_batch_equals_rows_of_a_large_batch(ep, k, unit):
    """A batch with fewer tokens than resident CTAs takes the thread-per-chunk
    kernel, a large one the CTA kernels: the same fp32 fma chain in slot
    order, so the small batch's rows equal the large batch's bit for bit
    (unit weights: the dispatch backward)."""
    rng = np.random.default_rng(40 + k)
    T, H = 3000, 1024
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (T * k, H)).astype(np.float32))
    pos = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.1] = -1
    w = None if unit else dev(rng.uniform(-1, 1, (T, k)).astype(np.float32))
    yd, pd = dev_bf16(y), dev(pos)
    big = ep.ep_combine(yd, pd, w) if not unit else ep.ep_dispatch_backward(yd, pd)
    n = 100
    small = (ep.ep_combine(yd, pd[:n].contiguous(), w[:n].contiguous()) if not unit
             else ep.ep_dispatch_backward(yd, pd[:n].contiguous()))
    torch.cuda.synchronize()
    assert torch.equal(small, big[:n])

