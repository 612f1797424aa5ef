"""The benchmark's own step, in the launch configuration bench.py times, at
the full DeepSeek-V3-shaped size, checked end to end against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_combine_close, assert_weights_close, gate_args, host_bits, weight_rtol

pytestmark = pytest.mark.gpu


def test_bench_step_matches_oracle():
    import bench
    cfg = synth.config(bench.WORKLOAD)
    r = bench.PathRunner(cfg)
    for _ in range(2):                       # a repeated step must give the same answer
        r.step()
    torch.cuda.synchronize()
    assert int(r.err.item()) == 0
    inp = r.host
    oi, ow = oracle.gate(inp["scores"], inp["bias"], *gate_args(cfg))
    np.testing.assert_array_equal(r.topk_idx.cpu().numpy(), oi)
    w = r.topk_w.cpu().numpy()
    assert_weights_close(w, ow, weight_rtol(cfg, inp["scores"], oi))
    ol = oracle.layout(oi, cfg["E"], cfg["experts_per_rank"])
    for key in ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "src"):
        np.testing.assert_array_equal(getattr(r.lay, key).cpu().numpy(), ol[key], err_msg=key)
    pos = r.lay.pos.cpu().numpy()
    np.testing.assert_array_equal(pos, ol["pos"])
    oq, os_ = oracle.dispatch_fp8(inp["x"], pos)
    np.testing.assert_array_equal(r.recv_q.cpu().numpy(), oq)
    np.testing.assert_array_equal(r.recv_s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    y = host_bits(r.y)
    np.testing.assert_array_equal(y, oracle.dispatch_bf16(inp["x"], pos))
    assert_combine_close(host_bits(r.out), oracle.combine(y, pos, w), y, pos, w)


@pytest.mark.parametrize("T,bounds", [
    (1000, [0, 1, 130, 131, 517, 999, 1000]),
    # whole batch through the bulk-copy dispatch, slices through the warp-item kernel
    (4096, [0, 512, 1024, 1536, 2048, 2049, 3000, 4096]),
])
def test_token_chunked_calls_equal_whole_batch(T, bounds):
    """Dispatch and combine over token slices (as a pipelined caller issues
    them while rows stream in) give the whole-batch results bit for bit."""
    import combine_group_limited_gb300 as ep
    cfg = synth.config("dsv3", T=T)
    inp = synth.make_inputs(cfg)
    s = torch.from_numpy(inp["scores"]).cuda()
    b = torch.from_numpy(inp["bias"]).cuda()
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda().view(torch.bfloat16)
    gc = ep.gate_cfg(cfg["E"], cfg["k"], cfg["n_groups"], cfg["topk_group"], cfg["topk_in_group"], cfg["score_fn"],
                     cfg["normalize"])
    idx, w = ep.ep_gate(s, b, gc)
    lay = ep.ep_get_layout(idx, cfg["E"], cfg["experts_per_rank"])
    q, sc = ep.ep_dispatch(x, lay.pos, "fp8")
    y = ep.ep_dispatch(x, lay.pos, "bf16")
    out = ep.ep_combine(y, lay.pos, w)
    q2 = torch.zeros_like(q)
    sc2 = torch.zeros_like(sc)
    out2 = torch.zeros_like(out)
    for a, e in zip(bounds, bounds[1:]):
        ep.ep_dispatch(x[a:e], lay.pos[a:e], "fp8", recv=q2, recv_scales=sc2)
        ep.ep_combine(y, lay.pos[a:e], w[a:e], out=out2[a:e])
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(sc, sc2) and torch.equal(out, out2)


def test_step_replayed_from_a_cuda_graph_equals_direct_calls():
    """The step's C-ABI calls captured once in a CUDA graph (as the end-to-end
    leg of the bench does) and replayed give the results of direct calls."""
    import combine_group_limited_gb300 as ep
    cfg = synth.config("dsv3", T=2304)
    inp = synth.make_inputs(cfg)
    s = torch.from_numpy(inp["scores"]).cuda()
    b = torch.from_numpy(inp["bias"]).cuda()
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda().view(torch.bfloat16)
    gc = ep.gate_cfg(cfg["E"], cfg["k"], cfg["n_groups"], cfg["topk_group"], cfg["topk_in_group"], cfg["score_fn"],
                     cfg["normalize"])
    T, k, E, epr, H = cfg["T"], cfg["k"], cfg["E"], cfg["experts_per_rank"], cfg["H"]
    idx, w, lay = ep.ep_gate_layout(s, b, gc, epr)
    y = ep.ep_dispatch(x, lay.pos, "bf16")
    q, sc = ep.ep_dispatch(x, lay.pos, "fp8")
    out = ep.ep_combine(y, lay.pos, w)
    torch.cuda.synchronize()
    gidx, gw = torch.empty_like(idx), torch.empty_like(w)
    glay = ep.alloc_layout(T, k, E, epr, "cuda")
    ws = ep.alloc_layout_workspace(T, k, E, epr)
    gq, gsc, gout = torch.zeros_like(q), torch.zeros_like(sc), torch.zeros_like(out)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        ep.ep_gate_layout(s, b, gc, epr, topk_idx=gidx, topk_w=gw, out=glay, workspace=ws, err_flag=err)
        ep.ep_dispatch(x, glay.pos, "fp8", recv=gq, recv_scales=gsc, err_flag=err)
        ep.ep_combine(y, glay.pos, gw, out=gout, err_flag=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                    # first calls outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step()
        for t in (gq, gsc, gout):
            t.zero_()
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(gidx, idx) and torch.equal(gw, w) and torch.equal(glay.pos, lay.pos)
    assert torch.equal(gq, q) and torch.equal(gsc, sc) and torch.equal(gout, out)
