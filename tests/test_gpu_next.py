"""GPU parity of the next rows against the CPU oracle: MXFP8 dispatch (bit
exact), FP8-input combine (stated combine bar + the fp32 terms), capacity-
limited layout (bit exact), dispatch backward (combine bar) and combine
backward (grad_y bit exact, grad_w within the fp32 dot-product bound)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import U, assert_combine_close, bf16_ulp, dev, dev_bf16, ep_cfg, gate_args, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_group_limited_gb300 as m
    m.load()
    return m


def _pos(cfg, inp):
    idx, _ = oracle.gate(inp["scores"], inp["bias"], *gate_args(cfg))
    return idx, oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])["pos"]


# ---------------------------------------------------------------- MXFP8


@pytest.mark.parametrize("name", ["dsv3", "skewed", "qwen3", "decode", "tiny"])
def test_mxfp8_dispatch_full_size(ep, name):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    _, pos = _pos(cfg, inp)
    q, e = ep.ep_dispatch(dev_bf16(inp["x"]), dev(pos), "mxfp8")
    torch.cuda.synchronize()
    oq, oe = oracle.dispatch_mxfp8(inp["x"], pos)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    np.testing.assert_array_equal(e.cpu().numpy(), oe)


def test_mxfp8_special_blocks(ep):
    H = 512
    r = np.zeros((4, H), np.float32)
    r[0, 32:64] = -0.0
    r[0, 64:96] = np.linspace(-1, 1, 32) * 3.9           # saturating block (|x|/X up to ~500)
    r[0, 96:128] = 1e-38                                  # fp32-subnormal amax: clamped exponent
    r[0, 128:160] = 3.0e38
    r[0, 160] = 2.0 ** -17
    r[0, 161] = 1.0
    r[1] = np.arange(H) / 64.0
    rng = np.random.default_rng(4)
    r[2] = rng.normal(0, 1, H) * np.exp2(rng.integers(-40, 40, H))
    r[3] = -r[2]
    x = synth.f32_to_bf16_bits(r)
    x[0, 32:64] = 0x8000
    pos = np.array([[3, 1], [0, -1], [2, 6], [5, 4]], np.int32)
    q, e = ep.ep_dispatch(dev_bf16(x), dev(pos), "mxfp8")
    torch.cuda.synchronize()
    rq = np.zeros((8, H), np.uint8)
    re = np.zeros((8, H // 32), np.uint8)
    oracle.dispatch_mxfp8(x, pos, recv_q=rq, recv_e=re)
    rows = sorted(pos[pos >= 0].tolist())
    np.testing.assert_array_equal(q.cpu().numpy()[rows], rq[rows])
    np.testing.assert_array_equal(e.cpu().numpy()[rows], re[rows])


@pytest.mark.parametrize("T,H,k", [(40, 2048, 2), (301, 2176, 3), (2049, 4096, 1), (128, 7168, 2), (1000, 4608, 4)])
def test_mxfp8_small_k_rows_in_flight_with_bad_rows(ep, T, H, k):
    """k <= 4 with at least four row segments per token: the MXFP8 walk that
    keeps segments in flight through shared memory (a ragged last segment
    at H = 2176; tokens split into pieces of 4 and 5 segments at H = 7168
    and 4608); rows outside the buffer are flagged and skipped, rows no
    slot names stay untouched."""
    rng = np.random.default_rng(T + k)
    x = synth.f32_to_bf16_bits((rng.normal(0, 1, (T, H)) * np.exp2(rng.integers(-8, 8, (T, 1)))).astype(np.float32))
    pos = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.1] = -1
    pos[T // 2, k - 1] = T * k + 3
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = torch.full((T * k, H), 0xA5, dtype=torch.uint8, device="cuda")
    e = torch.full((T * k, H // 32), 0x5A, dtype=torch.uint8, device="cuda")
    ep.ep_dispatch(dev_bf16(x), dev(pos), "mxfp8", recv=q, recv_scales=e, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 2
    ref_pos = np.where(pos >= T * k, -1, pos).astype(np.int32)
    rq = np.full((T * k, H), 0xA5, np.uint8)
    re = np.full((T * k, H // 32), 0x5A, np.uint8)
    oracle.dispatch_mxfp8(x, ref_pos, recv_q=rq, recv_e=re)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(e.cpu().numpy(), re)


# ------------------------------------------------------- FP8-input combine


def _assert_fp8_combine_close(g_bits, r_bits, deq, pos, w, accumulation=True):
    """Stated bar max(1 bf16 ulp, 1e-2 rel), plus (accumulation=True) the
    fp32 terms: one rounding per dequantised product and one per fma,
    2k*u*sum|w*d| in all -- for the signed-weight edge cases, where sums
    cancel on purpose; the workloads' identity-expert runs take the stated
    bar alone."""
    g = synth.bf16_bits_to_f32(g_bits).astype(np.float64)
    r = synth.bf16_bits_to_f32(r_bits).astype(np.float64)
    T, k = pos.shape
    S = np.zeros_like(r)
    for j in range(k):
        ok = pos[:, j] >= 0
        S[ok] += np.abs(w[ok, j].astype(np.float64))[:, None] * np.abs(deq[pos[ok, j]])
    tol = np.maximum(bf16_ulp(r), 1e-2 * np.abs(r)) + (2 * k * U * S if accumulation else 0.0)
    bad = np.abs(g - r) > tol
    assert not bad.any(), np.argwhere(bad)[:5]


def _dequant(q, s, bs):
    vals = oracle.e4m3_decode(q.reshape(-1)).reshape(q.shape)
    scale = s.astype(np.float64) if s.dtype == np.float32 else np.exp2(s.astype(np.float64) - 127)
    return vals * np.repeat(scale, bs, axis=1)


@pytest.mark.parametrize("name,fmt", [("dsv3", "fp8"), ("dsv3", "mxfp8"), ("decode", "fp8"), ("qwen3", "mxfp8"),
                                      ("mixtral", "fp8"), ("mixtral", "mxfp8")])
def test_combine_fp8_full_size_identity_experts(ep, name, fmt):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    idx, w = ep.ep_gate(dev(inp["scores"]), None if inp["bias"] is None else dev(inp["bias"]), ep_cfg(ep, cfg))
    lay = ep.ep_get_layout(idx, cfg["E"], cfg["experts_per_rank"])
    q, s = ep.ep_dispatch(dev_bf16(inp["x"]), lay.pos, fmt)
    out = ep.ep_combine_fp8(q, s, lay.pos, w)
    torch.cuda.synchronize()
    pos, wh, qh, sh = lay.pos.cpu().numpy(), w.cpu().numpy(), q.cpu().numpy(), s.cpu().numpy()
    r = oracle.combine_fp8(qh, sh, pos, wh)
    _assert_fp8_combine_close(host_bits(out), r, _dequant(qh, sh, 128 if fmt == "fp8" else 32), pos, wh,
                              accumulation=False)


@pytest.mark.parametrize("fmt,T,H,k,scale_offset", [
    ("fp8", 77, 1024, 6, 0), ("mxfp8", 77, 1024, 6, 0),
    # larger batches; short scale rows (H = 384 FP8: 12 bytes, H = 96 MXFP8: 3
    # bytes); a scale buffer 4 bytes off a 16-byte boundary
    ("fp8", 2048, 1024, 6, 0), ("mxfp8", 2100, 512, 8, 0), ("fp8", 2048, 384, 4, 0), ("mxfp8", 2049, 96, 5, 0),
    ("fp8", 2048, 1024, 6, 4),
    # k <= 2 on large batches: one warp per token
    ("fp8", 2048, 1024, 2, 0), ("mxfp8", 2100, 96, 1, 0), ("fp8", 2500, 384, 2, 4),
    # k <= 2 with rows of several rounds of chunks per lane (the next round's
    # codes copied ahead), the last one ragged
    ("fp8", 600, 4224, 2, 4), ("mxfp8", 333, 7168, 1, 0), ("mxfp8", 700, 2560, 2, 0),
    # fewer tokens than resident CTAs but more than the thread-per-chunk
    # kernel takes: the CTA kernel with each row split over two CTAs
    ("fp8", 500, 4096, 6, 4), ("mxfp8", 400, 7168, 8, 0),
])
def test_combine_fp8_random_codes_signed_weights(ep, fmt, T, H, k, scale_offset):
    rng = np.random.default_rng(9 + T + H)
    rows = T * k
    q = rng.integers(0, 256, size=(rows, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C
    s = (rng.uniform(0.01, 3, (rows, H // 128)).astype(np.float32) if fmt == "fp8"
         else rng.integers(110, 140, (rows, H // 32)).astype(np.uint8))
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.2] = -1
    w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
    sb = s.view(np.uint8).reshape(-1)
    sraw = torch.zeros(sb.size + 16, dtype=torch.uint8, device="cuda")
    sraw[scale_offset:scale_offset + sb.size] = dev(sb)
    sd = sraw[scale_offset:scale_offset + sb.size]
    sd = sd.view(torch.float32).view(s.shape) if fmt == "fp8" else sd.view(s.shape)
    out = ep.ep_combine_fp8(dev(q), sd, dev(pos), dev(w))
    torch.cuda.synchronize()
    r = oracle.combine_fp8(q, s, pos, w)
    _assert_fp8_combine_close(host_bits(out), r, _dequant(q, s, 128 if fmt == "fp8" else 32), pos, w)


@pytest.mark.parametrize("fmt,H,k", [("fp8", 2176, 3), ("mxfp8", 2048, 8), ("fp8", 7168, 3), ("mxfp8", 2176, 5)])
def test_combine_fp8_large_batch_ragged_rows_with_bad_rows(ep, fmt, H, k):
    """2 < k <= 8 on 2048+ tokens, the CTA kernel: rows of 136, 128 and 448
    chunks of 16 codes (one pass and a partial second pass of the CTA's
    threads at 136 and 448); a row outside the buffer is flagged and
    skipped, empty slots add nothing."""
    rng = np.random.default_rng(H + k)
    T = 2100
    rows = T * k
    q = rng.integers(0, 256, size=(rows, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C
    s = (rng.uniform(0.01, 3, (rows, H // 128)).astype(np.float32) if fmt == "fp8"
         else rng.integers(110, 140, (rows, H // 32)).astype(np.uint8))
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.15] = -1
    pos[T // 3, k - 1] = rows + 7
    w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ep.ep_combine_fp8(dev(q), dev(s), dev(pos), dev(w), err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 2
    ref_pos = np.where(pos >= rows, -1, pos).astype(np.int32)
    r = oracle.combine_fp8(q, s, ref_pos, w)
    _assert_fp8_combine_close(host_bits(out), r, _dequant(q, s, 128 if fmt == "fp8" else 32), ref_pos, w)


@pytest.mark.parametrize("fmt", ["fp8", "mxfp8"])
def test_combine_fp8_decode_sized_batch_equals_rows_of_a_large_batch(ep, fmt):
    """Fewer tokens than resident CTAs: the thread-per-chunk kernel; its rows
    equal the CTA kernel's on the same expert outputs bit for bit; a row
    outside the buffer is flagged and skipped."""
    rng = np.random.default_rng(71)
    T, H, k = 3000, 1024, 8
    rows = T * k
    q = rng.integers(0, 256, size=(rows, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C
    s = (rng.uniform(0.01, 3, (rows, H // 128)).astype(np.float32) if fmt == "fp8"
         else rng.integers(110, 140, (rows, H // 32)).astype(np.uint8))
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.1] = -1
    w = rng.uniform(-1, 1, (T, k)).astype(np.float32)
    qd, sd, pd, wd = dev(q), dev(s), dev(pos), dev(w)
    big = ep.ep_combine_fp8(qd, sd, pd, wd)
    n = 100
    small = ep.ep_combine_fp8(qd, sd, pd[:n].contiguous(), wd[:n].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(small, big[:n])
    bad = pos[:n].copy()
    bad[3, 2] = rows + 5
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ep.ep_combine_fp8(qd, sd, dev(bad), wd[:n].contiguous(), err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 2
    skip = pos[:n].copy()
    skip[3, 2] = -1
    want = ep.ep_combine_fp8(qd, sd, dev(skip), wd[:n].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(got, want)


# -------------------------------------------------------- capacity layout

CAP_KEYS = ("expert_count", "expert_off", "rank_count", "rank_off", "rank_tokens", "expert_dropped", "pos", "src")


@pytest.mark.parametrize("name,factor", [("skewed", 1.0), ("skewed", 1.25), ("dsv3", 1.0), ("dsv3", 0.5),
                                         ("qwen3", 1.0), ("mixtral", 1.1), ("decode", 2.0)])
def test_capacity_layout_full_size(ep, name, factor):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    idx, _ = oracle.gate(inp["scores"], inp["bias"], *gate_args(cfg))
    cap = int(np.ceil(factor * cfg["T"] * cfg["k"] / cfg["E"]))
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = ep.ep_get_layout_capacity(dev(idx), cfg["E"], cfg["experts_per_rank"], cap, err_flag=flag)
    torch.cuda.synchronize()
    o = oracle.layout_capacity(idx, cfg["E"], cfg["experts_per_rank"], cap)
    for key in CAP_KEYS:
        got = getattr(g, key).cpu().numpy().reshape(-1)[: o[key].size]
        np.testing.assert_array_equal(got, o[key].reshape(-1), err_msg=key)
    assert int(flag.item()) == 0


@pytest.mark.parametrize("cap", [0, 1, 3, 10000])
def test_capacity_layout_extremes_with_skips(ep, cap):
    rng = np.random.default_rng(cap + 5)
    T, k, E, epr = 700, 5, 24, 4
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    idx[rng.random((T, k)) < 0.4] = 7
    g = ep.ep_get_layout_capacity(dev(idx), E, epr, cap)
    torch.cuda.synchronize()
    o = oracle.layout_capacity(idx, E, epr, cap)
    for key in CAP_KEYS:
        got = getattr(g, key).cpu().numpy().reshape(-1)[: o[key].size]
        np.testing.assert_array_equal(got, o[key].reshape(-1), err_msg=key)


@pytest.mark.parametrize("T,k,E,epr,cap", [(3000, 6, 64, 8, 200), (100000, 8, 256, 8, 2900)])
def test_capacity_layout_bad_indices_and_large_batches(ep, T, k, E, epr, cap):
    """Out-of-range indices are flagged and skipped in capacity mode too;
    100000 tokens run the three-launch kernels (a grid of one CTA per SM would
    hold more than 128 tokens per CTA), 3000 the one-cluster kernel."""
    rng = np.random.default_rng(T + cap)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    idx[rng.random((T, k)) < 0.002] = E + 3
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = ep.ep_get_layout_capacity(dev(idx), E, epr, cap, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == ep.EP_FLAG_BAD_EXPERT
    clean = idx.copy()
    clean[clean >= E] = -1
    o = oracle.layout_capacity(clean, E, epr, cap)
    for key in CAP_KEYS:
        got = getattr(g, key).cpu().numpy().reshape(-1)[: o[key].size]
        np.testing.assert_array_equal(got, o[key].reshape(-1), err_msg=key)


def test_capacity_path_end_to_end(ep):
    """Gate -> capacity layout -> dispatch into E*capacity rows -> combine:
    dropped entries (pos -1) contribute nothing; the rest match the oracle."""
    cfg = synth.config("skewed", T=2048)
    inp = synth.make_inputs(cfg)
    idx, w = ep.ep_gate(dev(inp["scores"]), dev(inp["bias"]), ep_cfg(ep, cfg))
    cap = int(np.ceil(1.25 * cfg["T"] * cfg["k"] / cfg["E"]))
    lay = ep.ep_get_layout_capacity(idx, cfg["E"], cfg["experts_per_rank"], cap)
    rows = cfg["E"] * cap
    recv = torch.zeros((rows, cfg["H"]), dtype=torch.bfloat16, device="cuda")
    ep.ep_dispatch(dev_bf16(inp["x"]), lay.pos, "bf16", recv=recv)
    q = torch.zeros((rows, cfg["H"]), dtype=torch.uint8, device="cuda")
    s8 = torch.zeros((rows, cfg["H"] // 32), dtype=torch.uint8, device="cuda")
    ep.ep_dispatch(dev_bf16(inp["x"]), lay.pos, "mxfp8", recv=q, recv_scales=s8)
    out = ep.ep_combine(recv, lay.pos, w)
    torch.cuda.synchronize()
    pos, wh = lay.pos.cpu().numpy(), w.cpu().numpy()
    assert (pos < 0).any()                                  # the hot experts overflow
    ref_recv = oracle.dispatch_bf16(inp["x"], pos, recv=np.zeros((rows, cfg["H"]), np.uint16))
    np.testing.assert_array_equal(host_bits(recv), ref_recv)
    oq, oe = oracle.dispatch_mxfp8(inp["x"], pos, recv_q=np.zeros((rows, cfg["H"]), np.uint8),
                                   recv_e=np.zeros((rows, cfg["H"] // 32), np.uint8))
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    np.testing.assert_array_equal(s8.cpu().numpy(), oe)
    r = oracle.combine(ref_recv, pos, wh)
    assert_combine_close(host_bits(out), r, ref_recv, pos, wh)


# ---------------------------------------------------------------- backward


@pytest.mark.parametrize("name", ["dsv3", "qwen3", "decode", "mixtral"])
def test_dispatch_backward_full_size(ep, name):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    _, pos = _pos(cfg, inp)
    rows = cfg["T"] * cfg["k"]
    gr = synth.make_expert_out(cfg, rows)
    gx = ep.ep_dispatch_backward(dev_bf16(gr), dev(pos))
    torch.cuda.synchronize()
    r = oracle.dispatch_backward(gr, pos)
    assert_combine_close(host_bits(gx), r, gr, pos, np.ones(pos.shape, np.float32))


@pytest.mark.parametrize("name", ["dsv3", "decode", "mixtral"])
def test_combine_backward_full_size(ep, name):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg)
    idx, pos = _pos(cfg, inp)
    rows = cfg["T"] * cfg["k"]
    y = synth.make_expert_out(cfg, rows)
    g = inp["x"]                                       # an N(0,1) bf16 gradient of the layer output
    w = synth.make_weights(cfg)
    gy_d = torch.zeros((rows, cfg["H"]), dtype=torch.bfloat16, device="cuda")
    gy, gw = ep.ep_combine_backward(dev_bf16(g), dev_bf16(y), dev(pos), dev(w), grad_y=gy_d)
    torch.cuda.synchronize()
    ogy, ogw = oracle.combine_backward(g, y, pos, w)
    np.testing.assert_array_equal(host_bits(gy), ogy)
    gf = synth.bf16_bits_to_f32(g).astype(np.float64)
    yf = synth.bf16_bits_to_f32(y).astype(np.float64)
    S = np.einsum("th,tkh->tk", np.abs(gf), np.abs(yf[pos]))
    assert np.all(np.abs(gw.cpu().numpy() - ogw) <= cfg["H"] * U * S + 1e-30)


def test_combine_backward_empty_slots_and_midpoints(ep):
    """Empty slots give grad_w 0 and leave their rows untouched; products
    that land on a bf16 midpoint in fp32 still round like the exact product."""
    rng = np.random.default_rng(6)
    T, H, k = 50, 256, 4
    rows = T * k
    # weights 1 + 2^-8 + 2^-20 and bf16 g: w*g sits next to bf16 midpoints
    w = np.full((T, k), 1 + 2.0 ** -8 + 2.0 ** -20, np.float32)
    w[::3] = 1 + 2.0 ** -8 - 2.0 ** -20
    g = synth.f32_to_bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (rows, H)).astype(np.float32))
    pos = rng.permutation(rows).reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.2] = -1
    gy_d = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device="cuda")
    gy, gw = ep.ep_combine_backward(dev_bf16(g), dev_bf16(y), dev(pos), dev(w), grad_y=gy_d)
    torch.cuda.synchronize()
    ref_gy = np.full((rows, H), 0x4040, np.uint16)    # bf16 3.0 where nothing is written
    _, ogw = oracle.combine_backward(g, y, pos, w, grad_y=ref_gy)
    np.testing.assert_array_equal(host_bits(gy), ref_gy)
    assert np.all(gw.cpu().numpy()[pos < 0] == 0)


@pytest.mark.parametrize("T,H,k", [(2048, 256, 1), (2100, 1032, 2), (2500, 136, 2), (3001, 4096, 1)])
def test_combine_backward_warp_per_token(ep, T, H, k):
    """k <= 2 on 2048+ tokens (one warp per token): ragged rows (H/8 not a
    multiple of the warp's chunk step), empty slots, and products next to
    bf16 midpoints; grad_y bit exact, untouched rows left alone, grad_w 0 on
    empty slots and within the fp32 dot-product bound elsewhere."""
    rng = np.random.default_rng(T + H + k)
    rows = T * k + 7
    w = np.full((T, k), 1 + 2.0 ** -8 + 2.0 ** -20, np.float32)
    w[::3] = 1 + 2.0 ** -8 - 2.0 ** -20
    w[1::3] = rng.random((len(w[1::3]), k)).astype(np.float32)
    g = synth.f32_to_bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    y = synth.f32_to_bf16_bits(rng.normal(0, 1, (rows, H)).astype(np.float32))
    pos = rng.permutation(rows)[:T * k].reshape(T, k).astype(np.int32)
    pos[rng.random((T, k)) < 0.1] = -1
    gy_d = torch.full((rows, H), 3.0, dtype=torch.bfloat16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    gy, gw = ep.ep_combine_backward(dev_bf16(g), dev_bf16(y), dev(pos), dev(w), grad_y=gy_d, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    ref_gy = np.full((rows, H), 0x4040, np.uint16)
    _, ogw = oracle.combine_backward(g, y, pos, w, grad_y=ref_gy)
    np.testing.assert_array_equal(host_bits(gy), ref_gy)
    gwn = gw.cpu().numpy()
    assert np.all(gwn[pos < 0] == 0)
    gf = synth.bf16_bits_to_f32(g).astype(np.float64)
    yf = synth.bf16_bits_to_f32(y).astype(np.float64)
    S = np.einsum("th,tkh->tk", np.abs(gf), np.abs(yf[np.maximum(pos, 0)]))
    ok = pos >= 0
    assert np.all(np.abs(gwn - ogw)[ok] <= H * U * S[ok] + 1e-30)
