"""CPU checks of the C ABI boundary: the library builds, loads and exports
every entry point include/ep.h declares, and the host-side argument checks
return their statuses before anything reaches the GPU (no CUDA call is made
on these paths, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


@pytest.fixture(scope="module")
def lib():
    from combine_group_limited_gb300 import build
    build.build()
    import combine_group_limited_gb300 as ep
    return ep.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "ep.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return set(re.findall(r"\b(ep_[a-z_0-9]+)\s*\(", src))


def test_every_declared_symbol_is_exported(lib):
    import combine_group_limited_gb300 as ep
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(ep.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    import combine_group_limited_gb300 as ep
    assert ep.status_str(ep.EP_OK) == "ok"
    assert "align" in ep.status_str(ep.EP_ERR_ALIGNMENT)
    assert ep.status_str(99) == "unknown status"


def _cfg(ep, **kw):
    base = dict(num_experts=256, top_k=8, n_groups=8, topk_group=4, topk_in_group=2, score_fn=0, normalize=1)
    base.update(kw)
    return ep.GateCfg(*[base[f] for f, _ in ep.GateCfg._fields_])


FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: every call below returns before a launch
ODD = ctypes.c_void_p(0x10004)


@pytest.mark.parametrize("kw,status", [
    (dict(top_k=0), 1), (dict(top_k=300), 1), (dict(n_groups=7), 1), (dict(topk_group=9), 1),
    (dict(topk_group=0), 1), (dict(topk_in_group=33), 1), (dict(topk_group=1, top_k=40), 1),
    (dict(score_fn=5), 1), (dict(normalize=2), 1), (dict(num_experts=1024, n_groups=8), 2),
    (dict(top_k=33, topk_group=8), 2), (dict(num_experts=512, n_groups=64, topk_group=64), 2),
    (dict(topk_in_group=5), 2),
])
def test_gate_rejects_configurations(lib, kw, status):
    import combine_group_limited_gb300 as ep
    cfg = _cfg(ep, **kw)
    assert lib.ep_gate(FAKE, None, 16, ctypes.byref(cfg), FAKE, FAKE, None) == status


def test_gate_host_checks(lib):
    import combine_group_limited_gb300 as ep
    cfg = _cfg(ep)
    assert lib.ep_gate(FAKE, None, 0, ctypes.byref(cfg), None, None, None) == 0      # empty batch: nothing to do
    assert lib.ep_gate(None, None, 16, ctypes.byref(cfg), FAKE, FAKE, None) == 1
    assert lib.ep_gate(FAKE, None, 16, None, FAKE, FAKE, None) == 1
    assert lib.ep_gate(FAKE, None, -1, ctypes.byref(cfg), FAKE, FAKE, None) == 1
    assert lib.ep_gate(ctypes.c_void_p(0x10002), None, 16, ctypes.byref(cfg), FAKE, FAKE, None) == 3


def test_layout_host_checks(lib):
    n = lib.ep_layout_workspace_bytes(8192, 8, 256, 8)
    assert n > 0 and n % 256 == 0
    assert lib.ep_layout_workspace_bytes(8192, 8, 256, 7) == 0
    assert lib.ep_layout_workspace_bytes(10, 8, 2048, 8) == 0
    args = lambda T, k, E, epr, ws=FAKE, wsb=n: (FAKE, T, k, E, epr, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,  # noqa
                                                 None, ws, wsb, None)
    assert lib.ep_get_layout(*args(8192, 8, 256, 7)) == 1
    assert lib.ep_get_layout(*args(-1, 8, 256, 8)) == 1
    assert lib.ep_get_layout(*args(8192, 0, 256, 8)) == 1
    assert lib.ep_get_layout(*args(100, 8, 2048, 8)) == 2
    assert lib.ep_get_layout(*args(8192, 8, 256, 8, wsb=n - 1)) == 1
    assert lib.ep_get_layout(*args(8192, 8, 256, 8, ws=None)) == 1
    assert lib.ep_get_layout(*args(8192, 8, 256, 8, ws=ctypes.c_void_p(0x10008))) == 3
    assert lib.ep_get_layout(*args(1 << 28, 16, 256, 8)) == 2


def test_dispatch_host_checks(lib):
    d = lib.ep_dispatch
    R = 128
    assert d(FAKE, 16, 7168, 8, FAKE, 3, FAKE, R, FAKE, None, None) == 1          # unknown dtype
    assert d(FAKE, 16, 7184, 8, FAKE, 2, FAKE, R, FAKE, None, None) == 2          # MXFP8 needs H % 32
    assert d(FAKE, 16, 7168, 8, FAKE, 2, FAKE, R, None, None, None) == 1          # MXFP8 without scales
    assert d(FAKE, 16, 7164, 8, FAKE, 0, FAKE, R, None, None, None) == 2          # H % 8
    assert d(FAKE, 16, 7232, 8, FAKE, 1, FAKE, R, FAKE, None, None) == 2          # FP8 needs H % 128
    assert d(FAKE, 16, 7168, 65, FAKE, 0, FAKE, R, None, None, None) == 2         # k > 64
    assert d(FAKE, 16, 7168, 8, FAKE, 1, FAKE, R, None, None, None) == 1          # FP8 without scales
    assert d(FAKE, 16, 7168, 8, FAKE, 0, FAKE, -1, None, None, None) == 1         # negative row count
    assert d(ctypes.c_void_p(0x10008), 16, 7168, 8, FAKE, 0, FAKE, R, None, None, None) == 3
    assert d(FAKE, 16, 7168, 8, FAKE, 0, ODD, R, None, None, None) == 3
    assert d(None, 0, 7168, 8, None, 0, None, 0, None, None, None) == 0           # empty batch
    assert d(FAKE, 16, 0, 8, FAKE, 0, FAKE, R, None, None, None) == 1


def test_combine_host_checks(lib):
    c = lib.ep_combine
    assert c(FAKE, 128, FAKE, FAKE, 16, 7164, 8, FAKE, None, None) == 2
    assert c(FAKE, 128, FAKE, FAKE, 16, 7168, 0, FAKE, None, None) == 1
    assert c(None, 128, FAKE, FAKE, 16, 7168, 8, FAKE, None, None) == 1
    assert c(FAKE, -3, FAKE, FAKE, 16, 7168, 8, FAKE, None, None) == 1
    assert c(FAKE, 128, FAKE, FAKE, 16, 7168, 8, ODD, None, None) == 3
    assert c(None, 0, None, None, 0, 7168, 8, None, None, None) == 0


def test_binding_fails_loudly_without_the_library(monkeypatch):
    from combine_group_limited_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", os.path.join(ROOT, "no_such_lib.so"))
    with pytest.raises(ImportError):
        _binding.load()


def test_next_row_entry_points_host_checks(lib):
    cf = lib.ep_combine_fp8
    assert cf(FAKE, FAKE, 0, 128, FAKE, FAKE, 16, 7168, 8, FAKE, None, None) == 1   # bf16 is no FP8 scale kind
    assert cf(FAKE, FAKE, 1, 128, FAKE, FAKE, 16, 7232, 8, FAKE, None, None) == 2   # 1x128 needs H % 128
    assert cf(FAKE, FAKE, 2, 128, FAKE, FAKE, 16, 7184, 8, FAKE, None, None) == 2   # MXFP8 needs H % 32
    assert cf(FAKE, None, 2, 128, FAKE, FAKE, 16, 7168, 8, FAKE, None, None) == 1
    assert cf(FAKE, FAKE, 2, 128, FAKE, FAKE, 16, 7168, 8, ODD, None, None) == 3
    assert cf(None, None, 2, 0, None, None, 0, 7168, 8, None, None, None) == 0
    n = lib.ep_layout_workspace_bytes(64, 8, 256, 8)
    lc = lambda T, cap, ws=FAKE, E=256: lib.ep_get_layout_capacity(  # noqa: E731
        FAKE, T, 8, E, 8, cap, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, ws, n, None)
    assert lc(64, -1) == 1
    assert lc(64, 1 << 24) == 2                                                     # E * capacity overflows
    assert lc(64, 16, ws=None) == 1
    assert lc(64, 16, E=2048) == 2
    db = lib.ep_dispatch_backward
    assert db(FAKE, 128, FAKE, 16, 7164, 8, FAKE, None, None) == 2
    assert db(FAKE, 128, FAKE, 16, 7168, 8, ODD, None, None) == 3
    assert db(None, 0, None, 0, 7168, 8, None, None, None) == 0
    cb = lib.ep_combine_backward
    assert cb(FAKE, FAKE, 128, FAKE, FAKE, 16, 7168, 0, FAKE, FAKE, None, None) == 1
    assert cb(FAKE, FAKE, 128, FAKE, FAKE, 16, 7168, 8, ODD, FAKE, None, None) == 3
    assert cb(FAKE, None, 128, FAKE, FAKE, 16, 7168, 8, FAKE, FAKE, None, None) == 1


def test_decode_entry_points_host_checks(lib):
    import combine_group_limited_gb300 as ep
    cfg = _cfg(ep)
    dd = lambda T, H=7168, dtype=1, ws=FAKE, wsb=64, c=cfg: lib.ep_decode_dispatch(  # noqa: E731
        FAKE, None, T, ctypes.byref(c), 8, FAKE, H, dtype, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
        FAKE, T * 8, FAKE, None, ws, wsb, None)
    assert dd(0) == 1                                  # the fused path needs a token
    assert dd(1000) == 2                               # T*k > 4096: use the separate calls
    assert dd(128, H=7232) == 2                        # FP8 needs H % 128
    assert dd(128, dtype=7) == 1
    assert dd(128, ws=None) == 1
    assert dd(128, wsb=4) == 1
    assert dd(128, c=_cfg(ep, top_k=0)) == 1
    sb = lib.ep_selftest_grid_barrier
    assert sb(-1, 100, FAKE, FAKE, 64, None) == 1
    assert sb(1, 0, FAKE, FAKE, 64, None) == 1
    assert sb(1, (1 << 24) + 1, FAKE, FAKE, 64, None) == 1
    assert sb(1, 100, None, FAKE, 64, None) == 1
    assert sb(1, 100, ODD, ctypes.c_void_p(0x10001), 64, None) == 3


def test_gate_layout_host_checks(lib):
    import combine_group_limited_gb300 as ep
    cfg = _cfg(ep)
    n = lib.ep_layout_workspace_bytes(8192, 8, 256, 8)
    gl = lambda T=8192, epr=8, c=cfg, ws=FAKE, wsb=n, s=FAKE: lib.ep_gate_layout(  # noqa: E731
        s, None, T, ctypes.byref(c), epr, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, ws, wsb, None)
    assert gl(T=-1) == 1
    assert gl(epr=7) == 1
    assert gl(c=_cfg(ep, top_k=0)) == 1
    assert gl(c=_cfg(ep, num_experts=1024, n_groups=8)) == 2
    assert gl(wsb=n - 1) == 1
    assert gl(ws=None) == 1
    assert gl(s=None) == 1
    assert gl(ws=ctypes.c_void_p(0x10008)) == 3
    assert gl(s=ctypes.c_void_p(0x10002)) == 3
