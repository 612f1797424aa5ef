"""Every finite bf16 value through the GPU's FP8 casts, bit-exact against
the oracle's encoder (itself pinned to the OCP E4M3 code table, every
rounding midpoint and a brute-force nearest-code search on the CPU).

Block construction: the positive finite bf16 patterns, in magnitude order,
are cut into runs of B-1 consecutive patterns; each run forms one block with
an anchor of magnitude (largest in the run) * 2^d, so the block's amax (and
hence its scale) puts the run's values d binades below the top code.  d runs
from 0 to 20, past the smallest E4M3 subnormal, so every code, every
rounding boundary between codes, saturation and underflow to zero are met.
Signs are random and each block is shuffled, so the anchor's lane varies.
This is the FP8 e4m3 1x128 dispatch of "DeepEP de DeepSeek ...", section
"Support FP8 et MXFP8", and its MXFP8 (1x32, power-of-two scale) variant."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu

D_MAX = 20


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _blocks(B, H, seed):
    pats = np.arange(0, 0x7F80, dtype=np.uint32)          # +0 .. largest finite bf16
    runs = [pats[i:i + B - 1] for i in range(0, len(pats), B - 1)]
    rng = np.random.default_rng(seed)
    blocks = []
    for d in range(D_MAX + 1):
        for r in runs:
            top = int(r[-1])
            anchor = top + (d << 7)                       # bf16: one binade = 128 patterns
            anchor = min(anchor, 0x7F7F)
            blk = np.concatenate([r, [anchor]]).astype(np.uint32)
            if len(blk) < B:
                blk = np.concatenate([blk, np.zeros(B - len(blk), np.uint32)])
            blk |= (rng.random(B) < 0.5).astype(np.uint32) << 15
            blocks.append(rng.permutation(blk))
    flat = np.concatenate(blocks).astype(np.uint16)
    rows = -(-len(flat) // H)
    x = np.zeros(rows * H, np.uint16)
    x[:len(flat)] = flat
    return x.reshape(rows, H)


@pytest.mark.parametrize("fmt,B,k,rep", [("fp8", 128, 2, 1), ("mxfp8", 32, 2, 1), ("fp8", 128, 5, 1),
                                          ("mxfp8", 32, 5, 1), ("fp8", 128, 4, 13), ("mxfp8", 32, 4, 13)])
def test_every_bf16_value_at_every_relative_scale(ep, fmt, B, k, rep):
    """rep > 1 repeats the rows up to a batch the bulk-copy kernel takes
    (T >= 2048, k >= 4); with rep = 1, k <= 4 runs the token-per-warp
    kernel and k = 5 the warp-item kernel."""
    H = 4096
    x = np.tile(_blocks(B, H, seed=77 + B), (rep, 1))
    T = x.shape[0]
    pos = np.random.default_rng(5).permutation(T * k).reshape(T, k).astype(np.int32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s = ep.ep_dispatch(dev_bf16(x), dev(pos), fmt, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    if fmt == "fp8":
        oq, os_ = oracle.dispatch_fp8(x, pos)
        np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    else:
        oq, os_ = oracle.dispatch_mxfp8(x, pos)
        np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    # coverage: every one of the 254 finite codes is produced, no NaN code is
    codes = np.unique(oq)
    assert len(codes) == 254 and not np.any((codes & 0x7F) == 0x7F)
