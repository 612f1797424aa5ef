"""The expert-parallel exchange with the library's CUDA kernels as its
local steps (layout, dispatch, the one-slot dispatch that permutes rows,
combine), on a one-rank NCCL group: the exchange degenerates to a local
copy, so the receive rows must equal the single-batch dispatch and the
combined rows the single-batch combine, bit for bit (the multi-rank
exchange itself is checked on CPU over gloo)."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
import synth
from gpu_util import dev, dev_bf16, gate_args, host_bits

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("name,T", [("dsv3", 1000), ("mixtral", 512)])
def test_expert_parallel_one_rank_with_cuda_ops(name, T):
    import combine_group_limited_gb300 as ep
    from combine_group_limited_gb300.expert_parallel import ExpertParallel, cuda_ops
    ep.load()
    cfg = synth.config(name, T=T)
    inp = synth.make_inputs(cfg)
    idx, w = oracle.gate(inp["scores"], inp["bias"], *gate_args(cfg))
    dist.init_process_group("nccl", rank=0, world_size=1, init_method="tcp://127.0.0.1:%d" % _free_port())
    try:
        xp = ExpertParallel(cfg["E"], cuda_ops())
        x = dev_bf16(inp["x"])
        rows, plan = xp.dispatch(x, dev(idx))
        out = xp.combine(rows, dev(w.astype(np.float32)), plan)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    lay = oracle.layout(idx, cfg["E"], cfg["E"])          # one rank holds every expert
    recv = oracle.dispatch_bf16(inp["x"], lay["pos"])
    np.testing.assert_array_equal(host_bits(rows), recv)
    want = oracle.combine(recv, lay["pos"], w.astype(np.float32))
    got = host_bits(out)
    gf = synth.bf16_bits_to_f32(got).astype(np.float64)
    wf = synth.bf16_bits_to_f32(want).astype(np.float64)
    # the kernel sums in fp32, the oracle in binary64: the combine bar
    assert np.all(np.abs(gf - wf) <= np.maximum(1e-2 * np.abs(wf), np.abs(wf) * 2.0 ** -7 + 1e-30))
