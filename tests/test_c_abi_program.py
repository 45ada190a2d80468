"""The C ABI from a C program: tests/c_abi/abi_check.c is compiled as C99
against include/decode_attn.h, linked to the built library and run (host-side
checks only, no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from split_kv_decode_attention_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_links_and_passes(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = cuda_build.build()
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "abi_check.c"),
                    "-L", os.path.dirname(lib), "-ldecode_attn",
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr


@pytest.mark.gpu
def test_c_program_runs_both_entries_on_the_gpu(tmp_path):
    """tests/c_abi/gpu_check.c: device buffers from the CUDA runtime, a paged
    cache with a shuffled block table; decode_attn() and decode_attn_host()
    give bit-identical, finite results with no status bit."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = cuda_build.build()
    exe = tmp_path / "gpu_check"
    nvcc = shutil.which("nvcc")
    if shutil.which("gcc") is None or nvcc is None:
        pytest.skip("no C compiler or CUDA toolkit")
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "gpu_check.c"),
                    "-L", os.path.dirname(lib), "-ldecode_attn",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
                    "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(cuda, "lib64"),
                    "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr
