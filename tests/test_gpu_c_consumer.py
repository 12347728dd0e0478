"""The C ABI used from plain C (tests/c_abi_consumer.c, built here with gcc
against the CUDA runtime and libtvfgp.so): the 32^3 and 128^3 workloads
through tvfgp_create_ex / tvfgp_run / tvfgp_primal, compared bit for bit
with the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from fgp_dual_stencil_gb300 import synth

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    from fgp_dual_stencil_gb300 import _build
    lib = _build.build()
    cuda = cuda_home()
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_consumer")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_abi_consumer.c"), "-o", exe,
           "-L", libdir, "-ltvfgp", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


@pytest.mark.parametrize("key,variant", [("c1", 0), ("c2", 0), ("c2", 3), ("c1", 2)])
def test_c_consumer_matches_oracle(consumer, tmp_path, key, variant):
    w = synth.WORKLOADS[key]
    b = synth.make_b(w, 0)
    bfile, ofile = tmp_path / "b.f32", tmp_path / "out.f32"
    b.tofile(bfile)
    out = subprocess.run([consumer, str(bfile), str(ofile), str(w.nx), str(w.ny), str(w.nz), repr(w.lam),
                          str(w.steps), str(variant)], check=True, capture_output=True, text=True)
    tf, ran = out.stdout.split()
    n = w.nvox
    got = np.fromfile(ofile, dtype=np.float32)
    assert got.size == 7 * n
    p = np.zeros((3,) + b.shape, np.float32)
    r = np.zeros_like(p)
    t_or = oracle.fgp_run(b, p, r, np.float32(w.lam), w.steps, 1.0)
    assert np.array_equal(got[:3 * n], p.ravel())
    assert np.array_equal(got[3 * n:6 * n], r.ravel())
    assert np.array_equal(got[6 * n:], oracle.primal(b, p, np.float32(w.lam)).ravel())
    assert float(tf) == t_or
    assert int(ran) in (0, 1, 2, 3, 4, 5, 6)
