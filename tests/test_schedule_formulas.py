"""The integer schedule formulas the kernels use (schedule.h, compiled for the
host here) against their definitions: worker c starts at floor(c T / G), and
the worker holding tile t is the largest c whose start is <= t."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mla_decode_attention_08_gb300", "csrc")


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    out = str(tmp_path_factory.mktemp("sched") / "libsched.so")
    subprocess.check_call([cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-I", CSRC,
                           os.path.join(HERE, "schedule_formulas.cpp"), "-o", out])
    so = ctypes.CDLL(out)
    for name in ("sched_worker_begin", "sched_worker_of_tile"):
        getattr(so, name).restype = ctypes.c_int32
        getattr(so, name).argtypes = [ctypes.c_int32] * 3
    return so


def cases():
    rng = np.random.default_rng(31)
    out = [(1, 1), (1, 7), (7, 1), (152, 16384), (152, 151), (1024, 3), (65535, 2**24),
           (65536, 2**24 - 1), (100000, 16777215), (2**31 - 1, 2**31 - 1), (3, 2**31 - 1)]
    for _ in range(60):
        g = int(rng.integers(1, 200000)) if rng.random() < 0.5 else int(rng.integers(1, 300))
        t = int(rng.integers(1, 2**31 - 1)) if rng.random() < 0.3 else int(rng.integers(1, 2**24))
        out.append((g, t))
    return out


@pytest.mark.parametrize("grid,total", cases())
def test_worker_begin_and_owner_match_their_definitions(lib, grid, total):
    rng = np.random.default_rng(grid * 7 + total % 1000)
    cs = sorted({0, 1, grid - 1, grid, grid // 2, *rng.integers(0, grid + 1, size=20).tolist()})
    for c in cs:
        if 0 <= c <= grid:
            assert lib.sched_worker_begin(c, total, grid) == (c * total) // grid, (c, total, grid)
    ts = sorted({0, total - 1, total // 2, *rng.integers(0, total, size=30).tolist()})
    for t in ts:
        want = ((t + 1) * grid - 1) // total
        assert lib.sched_worker_of_tile(t, total, grid) == want, (t, total, grid)
