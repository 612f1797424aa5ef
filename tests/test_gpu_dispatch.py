"""GPU parity of step 3 (permute-scatter), BF16 and FP8 e4m3 1x128, against
the CPU oracle: receive rows, codes and scales bit-exact; rows the layout
does not name stay untouched; guard bytes around the buffers survive."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, dev_bf16, gate_args, host_bits

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of canary on each side of an output buffer


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _guarded(nbytes, fill=0xA5):
    buf = torch.full((nbytes + 2 * GUARD,), fill, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def _guards_ok(buf, fill=0xA5):
    h = buf.cpu().numpy()
    return bool(np.all(h[:GUARD] == fill) and np.all(h[-GUARD:] == fill))


def _dispatch_both(ep, x_bits, pos, dtype, flag=None):
    T, H = x_bits.shape
    k = pos.shape[1]
    rows = T * k
    xd = dev_bf16(x_bits)
    pd = dev(pos)
    if dtype == "bf16":
        buf, body = _guarded(rows * H * 2)
        recv = body.view(torch.bfloat16).view(rows, H)
        ep.ep_dispatch(xd, pd, "bf16", recv=recv, err_flag=flag)
        torch.cuda.synchronize()
        ref = np.full((rows, H), 0xA5A5, np.uint16)
        oracle.dispatch_bf16(x_bits, pos, recv=ref)
        np.testing.assert_array_equal(host_bits(recv), ref)
    else:
        buf, body = _guarded(rows * H)
        sbuf, sbody = _guarded(rows * (H // 128) * 4)
        q = body.view(rows, H)
        s = sbody.view(torch.float32).view(rows, H // 128)
        ep.ep_dispatch(xd, pd, "fp8", recv=q, recv_scales=s, err_flag=flag)
        torch.cuda.synchronize()
        rq = np.full((rows, H), 0xA5, np.uint8)
        rs = np.full((rows, H // 128), 0xA5A5A5A5, np.uint32).view(np.float32)
        oracle.dispatch_fp8(x_bits, pos, recv_q=rq, recv_s=rs)
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
        np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
        assert _guards_ok(sbuf)
    assert _guards_ok(buf)


def _layout_pos(cfg, inp):
    idx, _ = oracle.gate(inp["scores"], inp["bias"], *gate_args(cfg))
    return oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])["pos"]


@pytest.mark.parametrize("name,dtype", [(n, d) for n in synth.CONFIGS for d in ("bf16", "fp8")
                                         if d == "bf16" or synth.CONFIGS[n]["H"] % 128 == 0])
def test_dispatch_full_size(ep, name, dtype):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    _dispatch_both(ep, inp["x"], _layout_pos(cfg, inp), dtype)


@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (3, 24, 2), (17, 128, 3), (33, 384, 8), (9, 7168, 8), (130, 256, 5), (5, 16384, 64),
                                   (700, 1152, 2), (3000, 640, 1), (301, 384, 4), (500, 2176, 3), (2049, 4096, 2),
                                   (128, 7168, 2), (1000, 4608, 4)])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_dispatch_small_shapes_with_empty_slots(ep, T, H, k, dtype):
    if dtype == "fp8" and H % 128:
        pytest.skip("FP8 needs H % 128 == 0")
    rng = np.random.default_rng(T * H + k)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    pos = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.2] = -1        # empty slots: their rows must stay untouched
    _dispatch_both(ep, x, pos, dtype)


def test_fp8_special_blocks(ep):
    """Zero and -0 blocks, subnormal codes, exact code midpoints after
    scaling, huge and tiny magnitudes, a lone non-zero in a block."""
    H = 1024
    rows = []
    r = np.zeros(H, np.float32)
    r[128:256] = -0.0
    r[256:384] = np.linspace(-1, 1, 128) * 1e-3         # mostly subnormal codes against amax
    r[300] = 448.0
    r[384:512] = 3.0e38
    r[512:640] = 1e-38
    r[640] = -5.0                                       # lone value: -448 code
    r[768:896] = np.arange(128) / 16.0                  # multiples of 1/16 against amax 7.9375
    r[896:1024] = ((np.arange(128) % 9) - 4) * 2.0 ** -12
    rows.append(r)
    rows.append(np.full(H, -0.0, np.float32))
    rng = np.random.default_rng(3)
    rows.append((rng.normal(0, 1, H) * np.exp2(rng.integers(-30, 30, H))).astype(np.float32))
    x = synth.f32_to_bf16_bits(np.stack(rows))
    x[1, :] = 0x8000
    pos = np.arange(3 * 4, dtype=np.int32).reshape(3, 4)[:, ::-1].copy()
    _dispatch_both(ep, x, pos, "fp8")
    _dispatch_both(ep, x, pos, "bf16")


@pytest.mark.parametrize("dtype,k,H", [("bf16", 4, 256), ("fp8", 4, 256), ("fp8", 6, 256), ("fp8", 2, 2048)])
def test_dispatch_bad_rows_are_flagged_and_skipped(ep, dtype, k, H):
    """FP8 with k <= 4: the token-per-warp kernel; k = 6: the warp-item
    kernel."""
    rng = np.random.default_rng(8)
    T = 40
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    pos = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    pos[5, k - 1] = T * k             # one past the end
    pos[17, 0] = 1 << 30
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_pos = pos.copy()
    ref_pos[ref_pos >= T * k] = -1
    # the oracle skips negative rows; the kernel must skip out-of-range rows the same way
    T_, H_ = x.shape
    xd, pd = dev_bf16(x), dev(pos)
    if dtype == "bf16":
        buf, body = _guarded(T * k * H * 2)
        recv = body.view(torch.bfloat16).view(T * k, H)
        ep.ep_dispatch(xd, pd, "bf16", recv=recv, err_flag=flag)
        torch.cuda.synchronize()
        ref = np.full((T * k, H), 0xA5A5, np.uint16)
        oracle.dispatch_bf16(x, ref_pos, recv=ref)
        np.testing.assert_array_equal(host_bits(recv), ref)
    else:
        buf, body = _guarded(T * k * H)
        q = body.view(T * k, H)
        s = torch.empty((T * k, H // 128), dtype=torch.float32, device="cuda")
        ep.ep_dispatch(xd, pd, "fp8", recv=q, recv_scales=s, err_flag=flag)
        torch.cuda.synchronize()
        rq = np.full((T * k, H), 0xA5, np.uint8)
        oracle.dispatch_fp8(x, ref_pos, recv_q=rq)
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
    assert _guards_ok(buf)
    assert int(flag.item()) == 2


@pytest.mark.parametrize("T,H,k,dtype,scale_offset", [
    (2048, 384, 4, "fp8", 0),      # 12-byte scale rows: plain scale stores
    (2048, 7168, 8, "fp8", 4),     # scale buffer 4 bytes off a 16-byte boundary: plain scale stores
    (2500, 96, 5, "mxfp8", 0),     # 3-byte E8M0 rows
    (2049, 1024, 6, "mxfp8", 0),   # 32-byte E8M0 rows: bulk copies
    (3000, 256, 7, "bf16", 0),
])
def test_bulk_copy_dispatch_shapes(ep, T, H, k, dtype, scale_offset):
    """Batches the bulk-copy kernel takes (k >= 4, T >= 2048): each token's
    row staged in shared memory and written by cp.async.bulk copies, scale
    rows by bulk copies or, when short or unaligned, by plain stores; empty
    slots leave their rows untouched and guard bytes survive."""
    rng = np.random.default_rng(T * k + H)
    x = synth.f32_to_bf16_bits((rng.normal(0, 1, (T, H)) * np.exp2(rng.integers(-8, 8, (T, 1)))).astype(np.float32))
    rows = T * k
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.1] = -1
    xd, pd = dev_bf16(x), dev(pos)
    if dtype == "bf16":
        buf, body = _guarded(rows * H * 2)
        recv = body.view(torch.bfloat16).view(rows, H)
        ep.ep_dispatch(xd, pd, "bf16", recv=recv)
        torch.cuda.synchronize()
        ref = np.full((rows, H), 0xA5A5, np.uint16)
        oracle.dispatch_bf16(x, pos, recv=ref)
        np.testing.assert_array_equal(host_bits(recv), ref)
        assert _guards_ok(buf)
        return
    nsb = H // 128 * 4 if dtype == "fp8" else H // 32          # scale bytes per row
    buf, body = _guarded(rows * H)
    sbuf, sraw = _guarded(rows * nsb + 16)
    sbody = sraw[scale_offset:scale_offset + rows * nsb]
    q = body.view(rows, H)
    if dtype == "fp8":
        s = sbody.view(torch.float32).view(rows, H // 128)
        ep.ep_dispatch(xd, pd, "fp8", recv=q, recv_scales=s)
        torch.cuda.synchronize()
        rq = np.full((rows, H), 0xA5, np.uint8)
        rs = np.full((rows, H // 128), 0xA5A5A5A5, np.uint32).view(np.float32)
        oracle.dispatch_fp8(x, pos, recv_q=rq, recv_s=rs)
        np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    else:
        s = sbody.view(rows, H // 32)
        ep.ep_dispatch(xd, pd, "mxfp8", recv=q, recv_scales=s)
        torch.cuda.synchronize()
        rq = np.full((rows, H), 0xA5, np.uint8)
        rs = np.full((rows, H // 32), 0xA5, np.uint8)
        oracle.dispatch_mxfp8(x, pos, recv_q=rq, recv_e=rs)
        np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    assert _guards_ok(buf)
    h = sbuf.cpu().numpy()
    assert np.all(h[:GUARD + scale_offset] == 0xA5) and np.all(h[GUARD + scale_offset + rows * nsb:] == 0xA5)
