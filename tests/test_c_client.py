"""The C ABI from plain C11 (tests/c_client/flce_client.c, no PyTorch): the
header compiles with -Wall -Wextra -Werror, the planner's plan reads the same
from C as through the Python binding (so both agree on the struct layout),
and on a GPU a C caller with cudaMalloc'd buffers gets the oracle's loss and
gradients."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from flce_testing import assert_parity
from linear_cross_entropy_token_gb300 import build as flce_build
from linear_cross_entropy_token_gb300 import flce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("needs gcc and the CUDA toolkit headers")
    lib = flce_build.build()
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(CUDA, "lib64")
    exe = str(tmp_path_factory.mktemp("c_client") / "flce_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c_client", "flce_client.c"), "-o", exe,
           "-L", libdir, "-lflce", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}:{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _plan_from_c(exe, N, H, V, chunk, budget, mode, cta):
    r = subprocess.run([exe, "plan", str(N), str(H), str(V), str(chunk), str(budget), str(mode), str(cta)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    f = r.stdout.split()
    return {f[i]: int(f[i + 1]) for i in range(0, len(f), 2)}


@pytest.mark.parametrize("N,H,V,chunk,budget,mode,cta", [
    (16384, 4096, 128256, 0, 0, "auto", "auto"),
    (16384, 4096, 151936, 0, 0, "slabs", "auto"),
    (131072, 4096, 128256, 0, 64 << 20, "slabs", "pair"),
    (1000, 64, 4099, 300, 0, "recompute", "single"),
])
def test_plan_reads_the_same_from_c(client, N, H, V, chunk, budget, mode, cta):
    c = _plan_from_c(client, N, H, V, chunk, budget, flce.DLOGITS[mode], flce.CTA[cta])
    py = flce.plan(N, H, V, "bf16", chunk=chunk, hbm_budget_bytes=budget, cta=cta, dlogits_mode=mode)
    py.pop("dlogits")   # the binding's name for the mode; C prints the number
    assert c == py


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["auto", "slabs"])
def test_c_caller_matches_the_oracle(client, tmp_path, mode):
    w = workloads.generate(workloads.custom(1000, 256, 20011, "bf16", ignore_frac=0.1, seed=21))
    w.x.tofile(tmp_path / "x.bin")
    w.W.tofile(tmp_path / "W.bin")
    w.t.astype(np.int64).tofile(tmp_path / "t.bin")
    r = subprocess.run([client, "run", str(tmp_path), str(w.N), str(w.H), str(w.V), "384",
                        str(flce.DLOGITS[mode])], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    loss = float(r.stdout.split()[1])
    dx = workloads.bf16_bits_to_f32(np.fromfile(tmp_path / "dx.bin", dtype=np.uint16)).reshape(w.N, w.H)
    dW = np.fromfile(tmp_path / "dW.bin", dtype=np.float32).reshape(w.V, w.H)
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
    assert_parity({"loss": loss, "dx": dx.astype(np.float64), "dW": dW.astype(np.float64)}, ref, "bf16")
