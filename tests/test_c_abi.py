"""The C ABI from plain C: tests/c_abi_main.c includes only include/fa_gb300.h
and the CUDA runtime header, links the shared library and cudart, and runs
the forward and the backward on buffers it allocates itself.  On the CPU the
program is only compiled and linked; on the GPU its outputs are checked
against the float64 oracle."""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    import exact_io_aware_15_gb300 as fa
    from exact_io_aware_15_gb300 import build as b
    if not os.path.exists(fa.LIB_PATH):
        if not os.path.exists(os.path.join(CUDA, "bin", "nvcc")):
            pytest.skip("library not built and nvcc unavailable")
        b.build()
    if shutil.which("gcc") is None:
        pytest.skip("gcc unavailable")
    libdir = os.path.dirname(fa.LIB_PATH)
    exe = os.path.join(out_dir, "c_abi_main")
    cuda_lib = next((d for d in ("lib64", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib")
                     if os.path.exists(os.path.join(CUDA, d, "libcudart.so"))), "lib64")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror",
           os.path.join(ROOT, "tests", "c_abi_main.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-lfa_gb300", "-Wl,-rpath," + libdir,
           "-L", os.path.join(CUDA, cuda_lib), "-lcudart",
           "-Wl,-rpath," + os.path.join(CUDA, cuda_lib), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links():
    with tempfile.TemporaryDirectory() as d:
        assert os.path.exists(_compile(d))


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,causal", [(1, 2, 300, 128, True), (2, 1, 257, 64, False)])
def test_c_program_matches_oracle(B, H, N, D, causal):
    case = inp.dense(B, H, N, D, seed=500 + N, causal=causal)
    do = inp.output_grad((B, H, N, D), seed=501 + N)
    with tempfile.TemporaryDirectory() as d:
        exe = _compile(d)
        for name, t in (("q", case.q), ("k", case.k), ("v", case.v), ("do", do)):
            t.contiguous().view(torch.int16).numpy().tofile(os.path.join(d, name + ".bin"))
        r = subprocess.run([exe, d, str(B), str(H), str(N), str(D), str(int(causal)),
                            repr(case.scale)], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stdout + r.stderr
        assert "c abi ok" in r.stdout

        def load_bf16(name):
            raw = np.fromfile(os.path.join(d, name + ".bin"), dtype=np.int16)
            return torch.from_numpy(raw).view(torch.bfloat16).to(torch.float64).numpy() \
                .reshape(B, H, N, D)
        o = load_bf16("o")
        lse = np.fromfile(os.path.join(d, "lse.bin"), dtype=np.float32).reshape(B, H, N)
        O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, causal)
        assert (np.abs(o - O) - 2.0 ** -8 * np.abs(O)).max() <= 1e-2
        assert np.abs(lse - L).max() <= 1e-3
        refs = ora.attention_bwd_ref(case.q, case.k, case.v, do, case.scale, causal)[:3]
        for name, ref in zip(("dq", "dk", "dv"), refs):
            g = load_bf16(name)
            assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 1e-2, name
