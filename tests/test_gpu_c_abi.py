"""The C ABI from plain C: tests/c_abi_driver.c (no Python or torch in the
process) links libmla_decode, quantises the cache, plans, runs mla_decode_fwd
on device memory it allocated with the CUDA runtime, and returns the output,
which must match the float64 oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from mla_decode_attention_08_gb300.build import LIB
from mla_decode_attention_08_gb300.inputs import make_from_lengths

from .gpu_util import OracleCase, assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"


@pytest.fixture(scope="module")
def driver(built_library, tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_driver")
    libdir = os.path.dirname(LIB)
    cmd = [gcc, "-std=c11", "-O2", "-I", os.path.join(ROOT, "include"), "-I", f"{CUDA}/include",
           os.path.join(ROOT, "tests", "c_abi_driver.c"), "-L", libdir, "-lmla_decode",
           "-L", f"{CUDA}/lib64", "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{CUDA}/lib64",
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def run_driver(exe, inp, tmp_path):
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    paged = inp.kv_indices is not None
    n_tokens = int(inp.kv_indptr[-1])
    with open(src, "wb") as f:
        np.array([inp.batch, n_tokens, inp.max_kv_len, int(paged)], np.int32).tofile(f)
        inp.qo_indptr.astype(np.int32).tofile(f)
        inp.kv_indptr.astype(np.int32).tofile(f)
        if paged:
            inp.kv_indices.astype(np.int32).tofile(f)
        inp.q_bits.astype(np.uint16).tofile(f)
        inp.kv_bits.astype(np.uint16).tofile(f)
    r = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=300)
    raw = np.fromfile(dst, dtype=np.uint8)
    status, err = raw[:8].view(np.int32)
    out_bits = raw[8:].view(np.uint16).reshape(inp.batch, 16, 512)
    out = (out_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return r.returncode, int(status), int(err), out


@pytest.mark.parametrize("paged", [False, True])
def test_c_caller_matches_oracle(driver, tmp_path, paged):
    inp = make_from_lengths([1, 127, 128, 129, 700, 0, 3000, 5], seed=90, paged=paged)
    rc, status, err, out = run_driver(driver, inp, tmp_path)
    assert rc == 0 and status == 0 and err == 0, (rc, status, err)
    assert_close(out, OracleCase(inp).reference())
