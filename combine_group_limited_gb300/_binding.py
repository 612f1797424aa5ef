"""ctypes binding of ``libep_gb300.so`` (the C ABI of ``include/ep.h``).

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  Outputs may be
passed in (pre-allocated, as the pages' operators expect) or are allocated
here with ``torch.empty``.  There is no fallback: if the library is not built
the import of this module's functions fails with an error that says so.
"""
import ctypes
import os
from collections import namedtuple

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libep_gb300.so")

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED, EP_ERR_ALIGNMENT, EP_ERR_CUDA = range(5)
EP_FLAG_BAD_EXPERT, EP_FLAG_BAD_ROW, EP_FLAG_TIMEOUT = 1, 2, 4
EP_SCORE_RAW, EP_SCORE_SOFTMAX = 0, 1
EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_DTYPE_MXFP8_E4M3_B32 = 0, 1, 2

# Symbols include/ep.h declares (checked by the CPU test suite).
EXPORTS = ("ep_gate", "ep_layout_workspace_bytes", "ep_get_layout", "ep_get_layout_noalloc", "ep_gate_layout",
           "ep_dispatch",
           "ep_combine", "ep_combine_fp8", "ep_get_layout_capacity", "ep_dispatch_backward", "ep_combine_backward",
           "ep_decode_dispatch", "ep_selftest_grid_barrier", "ep_status_str")


class GateCfg(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("topk_in_group", ctypes.c_int32), ("score_fn", ctypes.c_int32),
                ("normalize", ctypes.c_int32)]


class EpError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, status_str(status), status))


_lib = None


def load():
    """Load libep_gb300.so (built by ``combine_group_limited_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libep_gb300.so is not built (expected at %s); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.ep_gate.argtypes = [P, P, i32, ctypes.POINTER(GateCfg), P, P, P]
    lib.ep_layout_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.ep_layout_workspace_bytes.restype = sz
    lib.ep_get_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, sz, P]
    lib.ep_get_layout_noalloc.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
    lib.ep_gate_layout.argtypes = [P, P, i32, ctypes.POINTER(GateCfg), i32, P, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.ep_dispatch.argtypes = [P, i32, i32, i32, P, i32, P, i32, P, P, P]
    lib.ep_combine.argtypes = [P, i32, P, P, i32, i32, i32, P, P, P]
    lib.ep_combine_fp8.argtypes = [P, P, i32, i32, P, P, i32, i32, i32, P, P, P]
    lib.ep_get_layout_capacity.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.ep_dispatch_backward.argtypes = [P, i32, P, i32, i32, i32, P, P, P]
    lib.ep_combine_backward.argtypes = [P, P, i32, P, P, i32, i32, i32, P, P, P, P]
    lib.ep_decode_dispatch.argtypes = [P, P, i32, ctypes.POINTER(GateCfg), i32, P, i32, i32, P, P, P, P, P, P, P, P,
                                       P, P, i32, P, P, P, sz, P]
    lib.ep_selftest_grid_barrier.argtypes = [i32, ctypes.c_int64, P, P, sz, P]
    for f in ("ep_gate", "ep_get_layout", "ep_get_layout_noalloc", "ep_dispatch", "ep_combine", "ep_combine_fp8",
              "ep_get_layout_capacity", "ep_dispatch_backward", "ep_combine_backward", "ep_decode_dispatch",
              "ep_selftest_grid_barrier"):
        getattr(lib, f).restype = ctypes.c_int
    lib.ep_status_str.argtypes = [ctypes.c_int]
    lib.ep_status_str.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_str(status):
    return load().ep_status_str(int(status)).decode()


def _check(fn, status):
    if status != EP_OK:
        raise EpError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def _dev(t, dtype, name, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _rows_of(t, H, name):
    if t.dim() != 2 or t.shape[1] != H:
        raise ValueError("%s must be [rows, %d]" % (name, H))
    return t.shape[0]


def gate_cfg(num_experts, top_k, n_groups=1, topk_group=1, topk_in_group=1, score_fn=EP_SCORE_RAW, normalize=True):
    return GateCfg(num_experts, top_k, n_groups, topk_group, topk_in_group, score_fn, int(bool(normalize)))


def ep_gate(scores, bias, cfg, topk_idx=None, topk_w=None, stream=None):
    """Step 1.  scores fp32 [T,E], bias fp32 [E] or None -> (topk_idx int32 [T,k], topk_w fp32 [T,k])."""
    lib = load()
    _dev(scores, torch.float32, "scores")
    T = scores.shape[0]
    k = cfg.top_k
    if bias is not None:
        _dev(bias, torch.float32, "bias", (cfg.num_experts,))
    if scores.dim() != 2 or scores.shape[1] != cfg.num_experts:
        raise ValueError("scores must be [T, num_experts]")
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=scores.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=scores.device)
    _dev(topk_idx, torch.int32, "topk_idx", (T, k))
    _dev(topk_w, torch.float32, "topk_w", (T, k))
    _check("ep_gate", lib.ep_gate(_ptr(scores), _ptr(bias), T, ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w),
                                  _stream(stream)))
    return topk_idx, topk_w


Layout = namedtuple("Layout", "expert_count expert_off rank_count rank_off rank_tokens pos src")


def ep_layout_workspace_bytes(T, k, E, experts_per_rank):
    return int(load().ep_layout_workspace_bytes(T, k, E, experts_per_rank))


def alloc_layout(T, k, E, experts_per_rank, device="cuda"):
    R = E // experts_per_rank
    z = lambda *s: torch.empty(s, dtype=torch.int32, device=device)  # noqa: E731
    return Layout(z(E), z(E + 1), z(R), z(R + 1), z(R), z(T, k), z(T * k))


def alloc_layout_workspace(T, k, E, experts_per_rank, device="cuda"):
    n = ep_layout_workspace_bytes(T, k, E, experts_per_rank)
    if n == 0:
        raise ValueError("invalid layout sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)  # ep_gate_layout wants its first 4 bytes zero


def ep_get_layout(topk_idx, num_experts, experts_per_rank, out=None, workspace=None, err_flag=None, stream=None):
    """Step 2.  topk_idx int32 [T,k] -> Layout of int32 device tensors."""
    lib = load()
    _dev(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    E, epr = num_experts, experts_per_rank
    if out is None:
        out = alloc_layout(T, k, E, epr, topk_idx.device) if epr > 0 and E % epr == 0 else None
    if out is None:
        raise ValueError("experts_per_rank must divide num_experts")
    if workspace is None:
        workspace = alloc_layout_workspace(T, k, E, epr, topk_idx.device)
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_get_layout", lib.ep_get_layout(
        _ptr(topk_idx), T, k, E, epr, _ptr(out.expert_count), _ptr(out.expert_off), _ptr(out.rank_count),
        _ptr(out.rank_off), _ptr(out.rank_tokens), _ptr(out.pos), _ptr(out.src), _ptr(err_flag),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def ep_gate_layout(scores, bias, cfg, experts_per_rank, topk_idx=None, topk_w=None, out=None, workspace=None,
                   err_flag=None, stream=None):
    """Steps 1 and 2 in one call (ep_gate, then ep_get_layout of its
    experts; the same results).  The workspace's first 4 bytes must be zero
    (alloc_layout_workspace gives such a buffer; calls leave them zero).
    Returns (topk_idx, topk_w, Layout)."""
    lib = load()
    _dev(scores, torch.float32, "scores")
    if scores.dim() != 2 or scores.shape[1] != cfg.num_experts:
        raise ValueError("scores must be [T, num_experts]")
    T, k, E, epr = scores.shape[0], cfg.top_k, cfg.num_experts, experts_per_rank
    if bias is not None:
        _dev(bias, torch.float32, "bias", (E,))
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=scores.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=scores.device)
    _dev(topk_idx, torch.int32, "topk_idx", (T, k))
    _dev(topk_w, torch.float32, "topk_w", (T, k))
    if out is None:
        if epr < 1 or E % epr:
            raise ValueError("experts_per_rank must divide num_experts")
        out = alloc_layout(T, k, E, epr, scores.device)
    if workspace is None:
        workspace = alloc_layout_workspace(T, k, E, epr, scores.device)
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_gate_layout", lib.ep_gate_layout(
        _ptr(scores), _ptr(bias), T, ctypes.byref(cfg), epr, _ptr(topk_idx), _ptr(topk_w), _ptr(out.expert_count),
        _ptr(out.expert_off), _ptr(out.rank_count), _ptr(out.rank_off), _ptr(out.rank_tokens), _ptr(out.pos),
        _ptr(out.src), _ptr(err_flag), _ptr(workspace), workspace.numel(), _stream(stream)))
    return topk_idx, topk_w, out


def ep_get_layout_noalloc(topk_idx, num_experts, experts_per_rank, out, err_flag=None, stream=None):
    """Step 2 without a workspace, for callers that cannot allocate device
    memory at call time (see include/ep.h): the scratch is a fixed array
    inside the library and ``out`` must be pre-allocated (alloc_layout).
    Calls that overlap on the GPU share that array and must not run
    concurrently."""
    lib = load()
    _dev(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_get_layout_noalloc", lib.ep_get_layout_noalloc(
        _ptr(topk_idx), T, k, num_experts, experts_per_rank, _ptr(out.expert_count), _ptr(out.expert_off),
        _ptr(out.rank_count), _ptr(out.rank_off), _ptr(out.rank_tokens), _ptr(out.pos), _ptr(out.src),
        _ptr(err_flag), _stream(stream)))
    return out


def ep_dispatch(x, pos, dtype="bf16", recv=None, recv_scales=None, err_flag=None, stream=None):
    """Step 3.  x bf16 [T,H], pos int32 [T,k].  recv defaults to T*k rows
    (any row count may be passed, e.g. E*capacity for a capacity layout).

    dtype "bf16"  -> recv bf16 [T*k, H];
    dtype "fp8"   -> (recv uint8 e4m3 codes [T*k, H], recv_scales fp32 [T*k, H/128]);
    dtype "mxfp8" -> (recv uint8 e4m3 codes [T*k, H], recv_scales uint8 E8M0 [T*k, H/32]).
    """
    lib = load()
    _dev(x, torch.bfloat16, "x")
    _dev(pos, torch.int32, "pos")
    T, H = x.shape
    k = pos.shape[1]
    if pos.shape[0] != T:
        raise ValueError("pos must be [T, k]")
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    if dtype == "bf16":
        if recv is None:
            recv = torch.empty((T * k, H), dtype=torch.bfloat16, device=x.device)
        _dev(recv, torch.bfloat16, "recv")
        _rows_of(recv, H, "recv")
        _check("ep_dispatch", lib.ep_dispatch(_ptr(x), T, H, k, _ptr(pos), EP_DTYPE_BF16, _ptr(recv), recv.shape[0],
                                              None, _ptr(err_flag), _stream(stream)))
        return recv
    if dtype not in ("fp8", "mxfp8"):
        raise ValueError("dtype must be 'bf16', 'fp8' or 'mxfp8'")
    mx = dtype == "mxfp8"
    if recv is None:
        recv = torch.empty((T * k, H), dtype=torch.uint8, device=x.device)
    if recv_scales is None:
        if mx:
            recv_scales = torch.empty((T * k, max(H // 32, 1)), dtype=torch.uint8, device=x.device)
        else:
            recv_scales = torch.empty((T * k, max(H // 128, 1)), dtype=torch.float32, device=x.device)
    _dev(recv, torch.uint8, "recv")
    _rows_of(recv, H, "recv")
    _dev(recv_scales, torch.uint8 if mx else torch.float32, "recv_scales",
         (recv.shape[0], H // (32 if mx else 128)))
    _check("ep_dispatch", lib.ep_dispatch(_ptr(x), T, H, k, _ptr(pos),
                                          EP_DTYPE_MXFP8_E4M3_B32 if mx else EP_DTYPE_FP8_E4M3_B128, _ptr(recv),
                                          recv.shape[0], _ptr(recv_scales), _ptr(err_flag), _stream(stream)))
    return recv, recv_scales


def ep_combine(y, pos, topk_w, out=None, err_flag=None, stream=None):
    """Steps 4-5.  y bf16 [T*k, H], pos int32 [T,k], topk_w fp32 [T,k] -> out bf16 [T,H]."""
    lib = load()
    _dev(y, torch.bfloat16, "y")
    _dev(pos, torch.int32, "pos")
    T, k = pos.shape
    _dev(topk_w, torch.float32, "topk_w", (T, k))
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _dev(out, torch.bfloat16, "out", (T, H))
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_combine", lib.ep_combine(_ptr(y), y.shape[0], _ptr(pos), _ptr(topk_w), T, H, k, _ptr(out),
                                        _ptr(err_flag), _stream(stream)))
    return out


def ep_combine_fp8(yq, yscales, pos, topk_w, out=None, err_flag=None, stream=None):
    """Steps 4-5 on FP8 expert outputs.  yq uint8 e4m3 [T*k, H]; yscales fp32
    [T*k, H/128] (1x128) or uint8 E8M0 [T*k, H/32] (MXFP8) -> out bf16 [T,H]."""
    lib = load()
    _dev(yq, torch.uint8, "yq")
    _dev(pos, torch.int32, "pos")
    T, k = pos.shape
    _dev(topk_w, torch.float32, "topk_w", (T, k))
    H = yq.shape[1]
    mx = yscales.dtype == torch.uint8
    _dev(yscales, torch.uint8 if mx else torch.float32, "yscales")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=yq.device)
    _dev(out, torch.bfloat16, "out", (T, H))
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _dev(yscales, torch.uint8 if mx else torch.float32, "yscales", (yq.shape[0], H // (32 if mx else 128)))
    _check("ep_combine_fp8", lib.ep_combine_fp8(
        _ptr(yq), _ptr(yscales), EP_DTYPE_MXFP8_E4M3_B32 if mx else EP_DTYPE_FP8_E4M3_B128, yq.shape[0], _ptr(pos),
        _ptr(topk_w), T, H, k, _ptr(out), _ptr(err_flag), _stream(stream)))
    return out


CapLayout = namedtuple("CapLayout", "expert_count expert_off rank_count rank_off rank_tokens expert_dropped pos src")


def ep_get_layout_capacity(topk_idx, num_experts, experts_per_rank, capacity, workspace=None, err_flag=None,
                           stream=None):
    """Capacity-limited layout: expert e owns rows [e*capacity, (e+1)*capacity)."""
    lib = load()
    _dev(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    E, epr = num_experts, experts_per_rank
    if epr <= 0 or E % epr:
        raise ValueError("experts_per_rank must divide num_experts")
    R = E // epr
    d = topk_idx.device
    z = lambda *s: torch.empty(s, dtype=torch.int32, device=d)  # noqa: E731
    out = CapLayout(z(E), z(E + 1), z(R), z(R + 1), z(R), z(E), z(T, k), z(max(E * capacity, 1)))
    if workspace is None:
        workspace = alloc_layout_workspace(T, k, E, epr, d)
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_get_layout_capacity", lib.ep_get_layout_capacity(
        _ptr(topk_idx), T, k, E, epr, int(capacity), _ptr(out.expert_count), _ptr(out.expert_off),
        _ptr(out.rank_count), _ptr(out.rank_off), _ptr(out.rank_tokens), _ptr(out.expert_dropped), _ptr(out.pos),
        _ptr(out.src), _ptr(err_flag), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def ep_dispatch_backward(grad_recv, pos, out=None, err_flag=None, stream=None):
    """grad_x[t] = bf16(sum_j grad_recv[pos[t,j]]).  grad_recv bf16 [T*k, H] -> bf16 [T, H]."""
    lib = load()
    _dev(grad_recv, torch.bfloat16, "grad_recv")
    _dev(pos, torch.int32, "pos")
    T, k = pos.shape
    H = grad_recv.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=grad_recv.device)
    _dev(out, torch.bfloat16, "grad_x", (T, H))
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_dispatch_backward", lib.ep_dispatch_backward(_ptr(grad_recv), grad_recv.shape[0], _ptr(pos), T, H, k,
                                                            _ptr(out), _ptr(err_flag), _stream(stream)))
    return out


def ep_combine_backward(grad_out, y, pos, topk_w, grad_y=None, grad_w=None, err_flag=None, stream=None):
    """Returns (grad_y bf16 [T*k, H], grad_w fp32 [T, k])."""
    lib = load()
    _dev(grad_out, torch.bfloat16, "grad_out")
    _dev(y, torch.bfloat16, "y")
    _dev(pos, torch.int32, "pos")
    T, k = pos.shape
    H = grad_out.shape[1]
    _dev(topk_w, torch.float32, "topk_w", (T, k))
    if grad_y is None:
        grad_y = torch.zeros((y.shape[0], H), dtype=torch.bfloat16, device=y.device)
    if grad_w is None:
        grad_w = torch.empty((T, k), dtype=torch.float32, device=y.device)
    _dev(grad_y, torch.bfloat16, "grad_y", (y.shape[0], H))
    _dev(grad_w, torch.float32, "grad_w", (T, k))
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_combine_backward", lib.ep_combine_backward(
        _ptr(grad_out), _ptr(y), y.shape[0], _ptr(pos), _ptr(topk_w), T, H, k, _ptr(grad_y), _ptr(grad_w),
        _ptr(err_flag), _stream(stream)))
    return grad_y, grad_w


_DTYPES = {"bf16": EP_DTYPE_BF16, "fp8": EP_DTYPE_FP8_E4M3_B128, "mxfp8": EP_DTYPE_MXFP8_E4M3_B32}


def ep_decode_dispatch(scores, bias, cfg, experts_per_rank, x, dtype="bf16", topk_idx=None, topk_w=None, out=None,
                       recv=None, recv_scales=None, err_flag=None, workspace=None, stream=None):
    """Fused gate + layout + dispatch for decode-sized batches (T*k <= 4096)
    in one launch.  Returns (topk_idx, topk_w, Layout, recv, recv_scales)."""
    lib = load()
    _dev(scores, torch.float32, "scores")
    _dev(x, torch.bfloat16, "x")
    T, E = scores.shape
    k, H = cfg.top_k, x.shape[1]
    d = scores.device
    if bias is not None:
        _dev(bias, torch.float32, "bias", (E,))
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=d)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=d)
    if out is None:
        out = alloc_layout(T, k, E, experts_per_rank, d)
    code = _DTYPES[dtype]
    if recv is None:
        recv = torch.empty((T * k, H), dtype=torch.bfloat16 if dtype == "bf16" else torch.uint8, device=d)
    if recv_scales is None and dtype != "bf16":
        recv_scales = (torch.empty((recv.shape[0], H // 128), dtype=torch.float32, device=d) if dtype == "fp8"
                       else torch.empty((recv.shape[0], H // 32), dtype=torch.uint8, device=d))
    if workspace is None:
        workspace = torch.zeros(64, dtype=torch.uint8, device=d)
    if err_flag is not None:
        _dev(err_flag, torch.int32, "err_flag")
    _check("ep_decode_dispatch", lib.ep_decode_dispatch(
        _ptr(scores), _ptr(bias), T, ctypes.byref(cfg), experts_per_rank, _ptr(x), H, code, _ptr(topk_idx),
        _ptr(topk_w), _ptr(out.expert_count), _ptr(out.expert_off), _ptr(out.rank_count), _ptr(out.rank_off),
        _ptr(out.rank_tokens), _ptr(out.pos), _ptr(out.src), _ptr(recv), recv.shape[0], _ptr(recv_scales),
        _ptr(err_flag), _ptr(workspace), workspace.numel(), _stream(stream)))
    return topk_idx, topk_w, out, recv, recv_scales


def ep_selftest_grid_barrier(missing_arrivals, spin_limit, err_flag, workspace=None, stream=None):
    """Runs the fused path's grid barrier alone (see include/ep.h)."""
    lib = load()
    _dev(err_flag, torch.int32, "err_flag")
    if workspace is None:
        workspace = torch.zeros(64, dtype=torch.uint8, device=err_flag.device)
    _check("ep_selftest_grid_barrier", lib.ep_selftest_grid_barrier(int(missing_arrivals), int(spin_limit),
                                                                    _ptr(err_flag), _ptr(workspace),
                                                                    workspace.numel(), _stream(stream)))
