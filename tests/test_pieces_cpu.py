"""The library's misaligned 16-byte accesses (shards off the 16-byte grid),
checked on the CPU: tests/c/vc_pieces_host.cu includes the device header,
whose byte helpers also compile as host code, and compares every store and
load, for every element size, every offset and every element-aligned byte
range, with a byte-by-byte expectation (no byte outside the access written,
every byte inside it right)."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

SRC = ROOT / "tests" / "c" / "vc_pieces_host.cu"


def _nvcc():
    cand = shutil.which("nvcc") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"),
                                                "bin", "nvcc")
    if not os.path.exists(cand):
        pytest.skip("nvcc not found")
    return cand


def test_piece_accesses_byte_exact(tmp_path):
    exe = tmp_path / "vc_pieces_host"
    csrc = ROOT / "allreduce_reducescatter_allgather_gb300" / "csrc"
    cmd = [_nvcc(), "-std=c++17", "-O2", "-Werror", "all-warnings", "-I", str(csrc),
           "-I", str(ROOT / "include"), str(SRC), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-4000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
