"""The expert-parallel split (combine_group_limited_gb300.expert_parallel)
on CPU, as world-size-2 and world-size-4 gloo process groups: tokens split
by rank, experts in contiguous blocks per rank, a count all-gather, a
dispatch all-to-all-v and a combine all-to-all-v back.

The rank-local steps are the CPU oracle's (layout, BF16 dispatch, combine)
and a numpy row permutation.  Each rank's receive rows must equal rows
rank_off[r] .. rank_off[r+1] of the oracle's single-batch layout of the
concatenated batch, and each rank's combined outputs (identity experts)
the oracle's combine of that batch for the rank's tokens, bit for bit."""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch(name, T_total):
    import oracle
    import synth
    cfg = synth.config(name, T=T_total)
    inp = synth.make_inputs(cfg)
    idx, w = oracle.gate(inp["scores"], inp["bias"], cfg["k"], cfg["n_groups"], cfg["topk_group"],
                         cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])
    return cfg, inp["x"], idx, w.astype(np.float32)


def _oracle_ops():
    import torch

    import oracle
    from combine_group_limited_gb300.expert_parallel import LocalOps

    def layout(idx, E, epr):
        lay = oracle.layout(idx.numpy(), E, epr)
        return {k: torch.from_numpy(lay[k]) for k in ("pos", "expert_count", "rank_count")}

    def dispatch(x, pos, rows):
        bits = x.numpy().view(np.uint16)
        recv = oracle.dispatch_bf16(bits, pos.numpy(), recv=np.zeros((rows, bits.shape[1]), np.uint16))
        return torch.from_numpy(recv.view(np.int16))

    def combine(y, pos, w):
        out = oracle.combine(y.numpy().view(np.uint16), pos.numpy(), w.numpy())
        return torch.from_numpy(out.view(np.int16))

    def permute(rows, target):
        out = torch.empty_like(rows)
        out[target] = rows
        return out

    return LocalOps(layout, dispatch, combine, permute)


def _rank_main(rank, world, port, out_dir, name, T_total):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from combine_group_limited_gb300.expert_parallel import ExpertParallel
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, x, idx, w = _batch(name, T_total)
        E = cfg["E"]
        lo, hi = T_total * rank // world, T_total * (rank + 1) // world   # this rank's tokens
        ep = ExpertParallel(E, _oracle_ops())
        x_r = torch.from_numpy(np.ascontiguousarray(x[lo:hi]).view(np.int16))
        idx_r = torch.from_numpy(np.ascontiguousarray(idx[lo:hi]))
        w_r = torch.from_numpy(np.ascontiguousarray(w[lo:hi]))
        rows, plan = ep.dispatch(x_r, idx_r)
        out = ep.combine(rows, w_r, plan)                 # identity experts

        # the single-batch reference, ranks as the logical ranks
        lay = oracle.layout(idx, E, E // world)
        recv_all = oracle.dispatch_bf16(x, lay["pos"])
        want_rows = recv_all[lay["rank_off"][rank]:lay["rank_off"][rank + 1]]
        want_out = oracle.combine(recv_all, lay["pos"], w)[lo:hi]
        res = {"rows_equal": bool(np.array_equal(rows.numpy().view(np.uint16), want_rows)),
               "rows": int(rows.shape[0]), "want_rows": int(want_rows.shape[0]),
               "out_equal": bool(np.array_equal(out.numpy().view(np.uint16), want_out)),
               "sent": sum(plan["send_splits"]), "received": sum(plan["recv_splits"])}
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,name,T_total", [(2, "tiny", 96), (4, "dsv3", 203), (2, "mixtral", 77)])
def test_expert_parallel_exchange_matches_the_single_batch_layout(tmp_path, world, name, T_total):
    import synth
    sys.path.insert(0, ROOT)
    cfg = synth.config(name, T=8)
    if cfg["E"] % world:
        pytest.skip("experts do not split over this world size")
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), name, T_total), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rows"] == d["want_rows"], (r, d)
        assert d["rows_equal"], (r, d)
        assert d["out_equal"], (r, d)
    k = synth.config(name, T=8)["k"]
    assert sum(d["sent"] for d in res) == sum(d["received"] for d in res) == T_total * k
