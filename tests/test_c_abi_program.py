"""The C ABI used from C alone: tests/c_abi_check.c includes include/ep.h,
the CUDA runtime and the C input generator (synth/synth.h), links
libep_gb300.so and the CPU oracle (liboracle.so), and checks a routed,
dispatched and combined batch against the oracle on the host (see the
program's header).  On CPU the program is compiled and linked; on a GPU it
also runs."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _build(tmp_path):
    from combine_group_limited_gb300 import build
    from oracle import build as obuild
    lib = build.build()
    olib = obuild.build()
    cuda = _cuda_home()
    exe = str(tmp_path / "c_abi_check")
    pkg, odir = os.path.dirname(lib), os.path.dirname(olib)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-Wall", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "synth"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), os.path.join(ROOT, "synth", "synth.c"), "-o", exe,
           "-L", pkg, "-lep_gb300", "-L", odir, "-loracle", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + pkg, "-Wl,-rpath," + odir, "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links_against_the_abi(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_program_runs_the_path(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c_abi_check ok" in r.stdout and "matches the oracle" in r.stdout
