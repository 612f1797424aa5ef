"""CPU oracle for the MoE dispatch/combine path -- TEST INFRASTRUCTURE ONLY.

A plain single-threaded C statement (``oracle.c``) of group-limited top-k
gating, the dispatch layout, the BF16/FP8 permute-scatter and the weighted
combine, wrapped here with numpy.  It shares no code with the CUDA library and
imports nothing from it.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may use it; the library itself never does.

The passages each function follows are cited in ``oracle.c``.  Parity pins
(brute force, invariants, library cross-checks) live in ``tests/``.

Array conventions: bf16 tensors travel as ``uint16`` bit patterns, FP8 e4m3
codes as ``uint8``; indices are ``int32``; weights out of the gate are
``float64``; the combine consumes the ``float32`` weights the GPU consumes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

SCORE_RAW = 0
SCORE_SOFTMAX = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        i64 = ctypes.c_int64
        lib.orc_gate.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, i32, P, P]
        lib.orc_gate.restype = ctypes.c_int
        lib.orc_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.orc_layout.restype = ctypes.c_int
        lib.orc_dispatch_bf16.argtypes = [P, i32, i32, i32, P, P]
        lib.orc_dispatch_bf16.restype = ctypes.c_int
        lib.orc_dispatch_fp8.argtypes = [P, i32, i32, i32, P, P, P]
        lib.orc_dispatch_fp8.restype = ctypes.c_int
        lib.orc_combine.argtypes = [P, P, P, i32, i32, i32, P]
        lib.orc_combine.restype = ctypes.c_int
        lib.orc_e4m3_encode_array.argtypes = [P, P, i64]
        lib.orc_e4m3_encode_array.restype = None
        lib.orc_e4m3_decode_array.argtypes = [P, P, i64]
        lib.orc_e4m3_decode_array.restype = None
        lib.orc_bf16_from_double_array.argtypes = [P, P, i64]
        lib.orc_bf16_from_double_array.restype = None
        lib.orc_dispatch_mxfp8.argtypes = [P, i32, i32, i32, P, P, P]
        lib.orc_combine_fp8.argtypes = [P, P, i32, P, P, i32, i32, i32, P]
        lib.orc_layout_capacity.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.orc_dispatch_backward.argtypes = [P, P, i32, i32, i32, P]
        lib.orc_combine_backward.argtypes = [P, P, P, P, i32, i32, i32, P, P]
        for f in ("orc_dispatch_mxfp8", "orc_combine_fp8", "orc_layout_capacity", "orc_dispatch_backward",
                  "orc_combine_backward"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def gate(scores, bias, k, n_groups=1, topk_group=1, topk_in_group=1, score_fn=SCORE_RAW, normalize=True):
    """Top-k (group-limited) gating.  Returns (topk_idx int32 [T,k], topk_w float64 [T,k])."""
    s = _c(scores, np.float32)
    T, E = s.shape
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = _load().orc_gate(_ptr(s), _ptr(b), T, E, k, n_groups, topk_group, topk_in_group,
                          score_fn, int(bool(normalize)), _ptr(idx), _ptr(w))
    if rc != 0:
        raise ValueError("oracle gate: invalid arguments")
    return idx, w


def layout(topk_idx, num_experts, experts_per_rank):
    """Dispatch layout.  Returns a dict of int32 arrays plus 'err_flag' (int)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    E = num_experts
    if experts_per_rank <= 0 or E % experts_per_rank:
        raise ValueError("oracle layout: invalid arguments")
    R = E // experts_per_rank
    out = dict(
        expert_count=np.empty(E, np.int32), expert_off=np.empty(E + 1, np.int32),
        rank_count=np.empty(R, np.int32), rank_off=np.empty(R + 1, np.int32),
        rank_tokens=np.empty(R, np.int32), pos=np.empty((T, k), np.int32),
        src=np.empty(T * k, np.int32))
    err = np.zeros(1, np.int32)
    rc = _load().orc_layout(_ptr(idx), T, k, E, experts_per_rank, _ptr(out["expert_count"]),
                            _ptr(out["expert_off"]), _ptr(out["rank_count"]), _ptr(out["rank_off"]),
                            _ptr(out["rank_tokens"]), _ptr(out["pos"]), _ptr(out["src"]), _ptr(err))
    if rc != 0:
        raise ValueError("oracle layout: invalid arguments")
    out["err_flag"] = int(err[0])
    return out


def dispatch_bf16(x_bits, pos, recv=None):
    """recv[pos[t,j]] = x[t].  x_bits uint16 [T,H]; returns uint16 [T*k, H]."""
    x = _c(x_bits, np.uint16)
    p = _c(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    if recv is None:
        recv = np.zeros((T * k, H), np.uint16)
    rc = _load().orc_dispatch_bf16(_ptr(x), T, H, k, _ptr(p), _ptr(recv))
    if rc != 0:
        raise ValueError("oracle dispatch_bf16: invalid arguments")
    return recv


def dispatch_fp8(x_bits, pos, recv_q=None, recv_s=None):
    """FP8 e4m3 1x128 dispatch.  Returns (codes uint8 [T*k,H], scales float32 [T*k,H/128])."""
    x = _c(x_bits, np.uint16)
    p = _c(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    if H % 128:
        raise ValueError("oracle dispatch_fp8: H must be a multiple of 128")
    if recv_q is None:
        recv_q = np.zeros((T * k, H), np.uint8)
    if recv_s is None:
        recv_s = np.zeros((T * k, H // 128), np.float32)
    rc = _load().orc_dispatch_fp8(_ptr(x), T, H, k, _ptr(p), _ptr(recv_q), _ptr(recv_s))
    if rc != 0:
        raise ValueError("oracle dispatch_fp8: invalid arguments")
    return recv_q, recv_s


def combine(y_bits, pos, w):
    """out[t] = bf16(sum_j w[t,j] * y[pos[t,j]]), binary64 sum.  Returns uint16 [T,H]."""
    y = _c(y_bits, np.uint16)
    p = _c(pos, np.int32)
    wf = _c(w, np.float32)
    T, k = p.shape
    H = y.shape[1]
    out = np.empty((T, H), np.uint16)
    rc = _load().orc_combine(_ptr(y), _ptr(p), _ptr(wf), T, H, k, _ptr(out))
    if rc != 0:
        raise ValueError("oracle combine: invalid arguments")
    return out


def e4m3_encode(v):
    a = _c(v, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().orc_e4m3_encode_array(_ptr(a), _ptr(out), a.size)
    return out


def e4m3_decode(c):
    a = _c(c, np.uint8)
    out = np.empty(a.shape, np.float64)
    _load().orc_e4m3_decode_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_from_double(v):
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().orc_bf16_from_double_array(_ptr(a), _ptr(out), a.size)
    return out


def dispatch_mxfp8(x_bits, pos, recv_q=None, recv_e=None):
    """MXFP8 (E4M3 elements, E8M0 scale per 32 columns) dispatch.
    Returns (codes uint8 [T*k,H], scale exponents uint8 [T*k,H/32])."""
    x = _c(x_bits, np.uint16)
    p = _c(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    if H % 32:
        raise ValueError("oracle dispatch_mxfp8: H must be a multiple of 32")
    if recv_q is None:
        recv_q = np.zeros((T * k, H), np.uint8)
    if recv_e is None:
        recv_e = np.zeros((T * k, H // 32), np.uint8)
    if _load().orc_dispatch_mxfp8(_ptr(x), T, H, k, _ptr(p), _ptr(recv_q), _ptr(recv_e)) != 0:
        raise ValueError("oracle dispatch_mxfp8: invalid arguments")
    return recv_q, recv_e


def combine_fp8(yq, yscale, pos, w):
    """Combine of FP8 expert outputs.  yscale float32 [rows, H/128] (1x128
    fp32 scales) or uint8 [rows, H/32] (E8M0).  Returns uint16 bf16 [T,H]."""
    q = _c(yq, np.uint8)
    p = _c(pos, np.int32)
    wf = _c(w, np.float32)
    kind = 0 if np.asarray(yscale).dtype == np.float32 else 1
    sc = _c(yscale, np.float32 if kind == 0 else np.uint8)
    T, k = p.shape
    H = q.shape[1]
    out = np.empty((T, H), np.uint16)
    if _load().orc_combine_fp8(_ptr(q), _ptr(sc), kind, _ptr(p), _ptr(wf), T, H, k, _ptr(out)) != 0:
        raise ValueError("oracle combine_fp8: invalid arguments")
    return out


def layout_capacity(topk_idx, num_experts, experts_per_rank, capacity):
    """Capacity-limited layout (fixed rows [e*capacity, (e+1)*capacity))."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    E = num_experts
    if experts_per_rank <= 0 or E % experts_per_rank or capacity < 0:
        raise ValueError("oracle layout_capacity: invalid arguments")
    R = E // experts_per_rank
    out = dict(
        expert_count=np.empty(E, np.int32), expert_off=np.empty(E + 1, np.int32),
        rank_count=np.empty(R, np.int32), rank_off=np.empty(R + 1, np.int32),
        rank_tokens=np.empty(R, np.int32), expert_dropped=np.empty(E, np.int32),
        pos=np.empty((T, k), np.int32), src=np.empty(E * capacity, np.int32))
    err = np.zeros(1, np.int32)
    rc = _load().orc_layout_capacity(_ptr(idx), T, k, E, experts_per_rank, capacity, _ptr(out["expert_count"]),
                                     _ptr(out["expert_off"]), _ptr(out["rank_count"]), _ptr(out["rank_off"]),
                                     _ptr(out["rank_tokens"]), _ptr(out["expert_dropped"]), _ptr(out["pos"]),
                                     _ptr(out["src"]), _ptr(err))
    if rc != 0:
        raise ValueError("oracle layout_capacity: invalid arguments")
    out["err_flag"] = int(err[0])
    return out


def dispatch_backward(grad_recv_bits, pos):
    """grad_x[t] = bf16(sum_j grad_recv[pos[t,j]]).  Returns uint16 [T,H]."""
    g = _c(grad_recv_bits, np.uint16)
    p = _c(pos, np.int32)
    T, k = p.shape
    H = g.shape[1]
    out = np.empty((T, H), np.uint16)
    if _load().orc_dispatch_backward(_ptr(g), _ptr(p), T, H, k, _ptr(out)) != 0:
        raise ValueError("oracle dispatch_backward: invalid arguments")
    return out


def combine_backward(grad_out_bits, y_bits, pos, w, grad_y=None):
    """Returns (grad_y uint16 [T*k,H], grad_w float64 [T,k])."""
    go = _c(grad_out_bits, np.uint16)
    y = _c(y_bits, np.uint16)
    p = _c(pos, np.int32)
    wf = _c(w, np.float32)
    T, k = p.shape
    H = go.shape[1]
    if grad_y is None:
        grad_y = np.zeros((y.shape[0], H), np.uint16)
    gw = np.empty((T, k), np.float64)
    if _load().orc_combine_backward(_ptr(go), _ptr(y), _ptr(p), _ptr(wf), T, H, k, _ptr(grad_y), _ptr(gw)) != 0:
        raise ValueError("oracle combine_backward: invalid arguments")
    return grad_y, gw
