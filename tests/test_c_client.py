"""The C ABI from a plain C program (tests/c/vc_from_c.c): the header
compiles as C11 with warnings as errors, the program links against
libvc.so, and the calls behave as from Python.  No torch involved."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

SRC = ROOT / "tests" / "c" / "vc_from_c.c"


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    from allreduce_reducescatter_allgather_gb300._binding import LIB_PATH
    return LIB_PATH


def _compile(tmp_path, with_cuda: bool):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib = _lib()
    exe = tmp_path / "vc_from_c"
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1", "-I", str(ROOT / "include"),
           str(SRC), "-o", str(exe), str(lib), f"-Wl,-rpath,{lib.parent}"]
    if with_cuda:
        cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
        cmd += ["-DVC_WITH_CUDA", "-I", f"{cuda}/include", f"-L{cuda}/lib64", "-lcudart",
                f"-Wl,-rpath,{cuda}/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_checks(tmp_path):
    exe = _compile(tmp_path, with_cuda=False)
    env = dict(os.environ, VC_TEST_FAIL_LAUNCH="1")
    r = subprocess.run([str(exe), "checks"], capture_output=True, text=True, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "checks ok" in r.stdout


@pytest.mark.gpu
def test_c_program_runs_the_worked_example(tmp_path):
    exe = _compile(tmp_path, with_cuda=True)
    env = {k: v for k, v in os.environ.items() if k != "VC_TEST_FAIL_LAUNCH"}
    r = subprocess.run([str(exe), "run"], capture_output=True, text=True, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "run ok" in r.stdout
