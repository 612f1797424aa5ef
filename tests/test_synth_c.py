"""The C generator (synth/synth.c) draws the arrays the Python one draws:
uniforms and the bf16 rounding bit for bit, normals to the last bits libm and
numpy may differ in, across a block boundary of the Box-Muller pairs; so a C
program checked against the oracle (tests/c_abi_check.c) sees the Python
tests' workloads."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("synthc") / "libsynth.so")
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall",
           os.path.join(ROOT, "synth", "synth.c"), "-o", out, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    L = ctypes.CDLL(out)
    u64, sz, vp = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
    L.synth_u64.restype = u64
    L.synth_u64.argtypes = [u64, u64, u64]
    for f in (L.synth_uniform_f32, L.synth_normal_f64):
        f.restype = None
        f.argtypes = [u64, u64, sz, vp]
    L.synth_normal_bf16.restype = None
    L.synth_normal_bf16.argtypes = [u64, u64, sz, ctypes.c_double, vp]
    return L


def test_raw_stream_values_match(lib):
    got = np.array([lib.synth_u64(1236, 3, i) for i in range(1000)], np.uint64)
    np.testing.assert_array_equal(got, synth.u64(1236, 3, 1000))


def test_uniforms_match_bit_for_bit(lib):
    n = 300001
    out = np.empty(n, np.float32)
    lib.synth_uniform_f32(1236, synth._S_SCORES, n, out.ctypes.data)
    np.testing.assert_array_equal(out.view(np.uint32), synth.uniform_f32(1236, synth._S_SCORES, (n,)).view(np.uint32))


def test_normals_match_across_a_block_boundary(lib):
    n = (1 << 23) + 11                          # more than one block of 2^22 Box-Muller pairs
    out = np.empty(n, np.float64)
    lib.synth_normal_f64(1239, synth._S_X, n, out.ctypes.data)
    ref = synth.normal_f64(1239, synth._S_X, (n,))
    exact = np.mean(out == ref)
    rel = np.abs(out - ref) / np.maximum(np.abs(ref), 1e-300)
    assert exact > 0.99, exact                  # libm and numpy agree on almost every value
    assert rel.max() <= 8 * 2.0 ** -52, rel.max()
    b = 1 << 23                                 # the block boundary, both sides of it
    np.testing.assert_allclose(out[b - 4:b + 4], ref[b - 4:b + 4], rtol=8 * 2.0 ** -52, atol=0)


def test_bf16_rows_match(lib):
    n = 1 << 20
    out = np.empty(n, np.uint16)
    lib.synth_normal_bf16(1236, synth._S_X, n, 1.0, out.ctypes.data)
    ref = synth.normal_bf16_bits(1236, synth._S_X, (n,))
    diff = out != ref
    assert diff.mean() < 1e-4, diff.mean()      # a last-bit normal difference can flip a bf16 rounding
    d = np.abs(synth.bf16_bits_to_f32(out).astype(np.float64) - synth.bf16_bits_to_f32(ref).astype(np.float64))
    ulp = np.abs(synth.bf16_bits_to_f32(ref).astype(np.float64)) * 2.0 ** -7
    assert np.all(d <= ulp + 1e-45)
