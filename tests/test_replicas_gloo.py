"""The multi-process host logic of bench.py on CPU: two ranks over gloo, as
torchrun launches them (one process per GPU on a real box).  Each rank is an
independent replica on its own seeded batch; the only collectives are the
barriers and the max over ranks of the measured times; rank 0 alone prints."""
import json
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import synth
    rep = bench.Replicas().init("gloo", "cpu")
    my_ms = 1.0 + 0.75 * rank                    # ranks finish at different times
    rep.barrier()
    worst = rep.max(my_ms)
    cfg = synth.config("tiny")
    cfg["seed"] += rep.seed_offset()
    x = synth.make_inputs(cfg)["x"]
    res = (worst, rep.is_printer(), rep.tokens_per_s(cfg["T"], worst), int(x[0, :8].astype(np.int64).sum()))
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump(res, f)
    rep.barrier()
    rep.close()


def test_two_replicas_over_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = {r: json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)}
    assert res[0][0] == res[1][0] == 1.75                 # the max over ranks, seen by every rank
    assert res[0][1] and not res[1][1]                    # rank 0 alone prints
    assert res[0][2] == world * 128 / 1.75e-3             # all ranks' tokens over the max time
    assert res[0][3] != res[1][3]                         # each replica draws its own batch


def test_single_process_needs_no_group():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    sys.path.insert(0, ROOT)
    import bench
    rep = bench.Replicas().init("gloo", "cpu")
    assert rep.world == 1 and rep.is_printer() and rep.seed_offset() == 0
    assert rep.max(2.5) == 2.5
    rep.barrier()
    rep.close()
