"""GPU parity of the fused low-latency decode path (gate + layout + dispatch
in one launch: the clustered kernel up to 512 tokens, the cooperative one
past that) against the CPU oracle and against the separate calls, and the
bounded grid barrier's timeout path."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_weights_close, dev, dev_bf16, ep_cfg, gate_args, host_bits, weight_rtol

pytestmark = pytest.mark.gpu

KEYS = ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "pos", "src")


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


@pytest.mark.parametrize("name,T,dtype", [
    ("decode", 128, "bf16"), ("decode", 128, "fp8"), ("decode", 128, "mxfp8"), ("decode", 1, "bf16"),
    ("decode", 77, "fp8"), ("dsv3", 256, "fp8"), ("dsv3", 512, "bf16"), ("skewed", 300, "mxfp8"),
    ("tiny", 128, "bf16"), ("mixtral", 2048, "bf16"), ("qwen3", 64, "bf16"),
    ("decode", 2, "fp8"), ("decode", 9, "mxfp8"), ("qwen3", 512, "bf16"), ("tiny", 600, "fp8"),
    ("mixtral", 513, "bf16"),
])
def test_decode_fused_matches_oracle(ep, name, T, dtype):
    cfg = synth.config(name, T=T)
    inp = synth.make_inputs(cfg)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w, lay, recv, scales = ep.ep_decode_dispatch(
        dev(inp["scores"]), None if inp["bias"] is None else dev(inp["bias"]), ep_cfg(ep, cfg),
        cfg["experts_per_rank"], dev_bf16(inp["x"]), dtype, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    oi, ow = oracle.gate(inp["scores"], inp["bias"], *gate_args(cfg))
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    assert_weights_close(w.cpu().numpy(), ow, weight_rtol(cfg, inp["scores"], oi))
    ol = oracle.layout(oi, cfg["E"], cfg["experts_per_rank"])
    for key in KEYS:
        np.testing.assert_array_equal(getattr(lay, key).cpu().numpy().reshape(ol[key].shape), ol[key], err_msg=key)
    if dtype == "bf16":
        np.testing.assert_array_equal(host_bits(recv), oracle.dispatch_bf16(inp["x"], ol["pos"]))
    elif dtype == "fp8":
        q, s = oracle.dispatch_fp8(inp["x"], ol["pos"])
        np.testing.assert_array_equal(recv.cpu().numpy(), q)
        np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), s.view(np.uint32))
    else:
        q, e = oracle.dispatch_mxfp8(inp["x"], ol["pos"])
        np.testing.assert_array_equal(recv.cpu().numpy(), q)
        np.testing.assert_array_equal(scales.cpu().numpy(), e)


def test_decode_fused_equals_separate_calls_repeatedly(ep):
    cfg = synth.config("decode")
    inp = synth.make_inputs(cfg)
    s, x = dev(inp["scores"]), dev_bf16(inp["x"])
    gc = ep_cfg(ep, cfg)
    idx, w = ep.ep_gate(s, None, gc)
    lay = ep.ep_get_layout(idx, cfg["E"], cfg["experts_per_rank"])
    q, sc = ep.ep_dispatch(x, lay.pos, "fp8")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    for _ in range(3):                      # the barrier counter is cleared by every call
        fi, fw, fl, fq, fs = ep.ep_decode_dispatch(s, None, gc, cfg["experts_per_rank"], x, "fp8", workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(fi, idx) and torch.equal(fw, w)
        for key in KEYS:
            assert torch.equal(getattr(fl, key), getattr(lay, key)), key
        assert torch.equal(fq, q) and torch.equal(fs, sc)


def test_grid_barrier_completes(ep):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_selftest_grid_barrier(0, 1 << 20, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0


def test_grid_barrier_times_out_and_reports(ep):
    """Arrivals that never come: every CTA gives up after its bounded wait,
    sets EP_FLAG_TIMEOUT and returns; the context stays usable."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_selftest_grid_barrier(1, 2048, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == ep.EP_FLAG_TIMEOUT
    # and the device still runs work afterwards
    flag.zero_()
    ep.ep_selftest_grid_barrier(0, 1 << 20, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
