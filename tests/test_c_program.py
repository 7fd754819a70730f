"""The C ABI from a plain C program (tests/c/lce_c_abi_test.c), compiled
here with gcc against include/lce.h and linked to the built library, the
CUDA runtime and the float64 oracle (test infrastructure): without a GPU
it checks sizes, status strings and argument errors; on a GPU it runs a
small ragged problem through the recomputing, fused and loss-variant calls
and the sequence-tiled MLP on device buffers and compares every output with
the oracle."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "lce_c_abi_test.c")


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _cudart_dir(home: str) -> str:
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib",
                "targets/x86_64-linux/lib"):
        d = os.path.join(home, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    pytest.skip("libcudart.so not found")


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    import oracle
    from chunked_lm_head_gemm_gb300 import _binding as B
    from chunked_lm_head_gemm_gb300 import build as Bld
    B.load(build_if_missing=True)
    oracle_lib = oracle.build()
    home = _cuda_home()
    libdirs = [os.path.dirname(Bld.LIB_PATH), os.path.dirname(oracle_lib),
               _cudart_dir(home)]
    exe = str(tmp_path_factory.mktemp("cprog") / "lce_c_abi_test")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", SRC,
           "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(home, "include"), "-o", exe]
    for d in libdirs:
        cmd += ["-L", d, f"-Wl,-rpath,{d}"]
    cmd += ["-llce", "-llce_oracle", "-lcudart", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_without_gpu(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout


@pytest.mark.gpu
def test_c_program_on_gpu(program):
    from tests.gpu_util import require_gpu
    require_gpu()
    r = subprocess.run([program, "--gpu"], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok  ") >= 32 and "FAIL" not in r.stdout
