"""The C ABI from plain C: tests/c_abi_check.c is compiled as C99 against include/moe_gb300.h,
linked to the built libmoe_gb300.so and run; it exercises the calls that need no GPU
(workspace sizing and validation, status strings, the host schedule).  tests/c_abi_gpu.c
(GPU only) runs the layer through the C ABI with cudaMalloc'd buffers against the oracle."""
import os
import shutil
import subprocess

import pytest

import mixture_experts_layer_top_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_dir():
    moe.build()
    return os.path.dirname(moe.LIB_PATH)


def test_plain_c_caller_compiles_links_and_runs(lib_dir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_check")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", lib_dir, "-lmoe_gb300",
           "-Wl,-rpath," + lib_dir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.gpu
def test_plain_c_caller_runs_the_layer_on_the_gpu(lib_dir, tmp_path):
    """tests/c_abi_gpu.c, a C99 program with cudaMalloc'd buffers, plans and runs the tiny layer
    through moe_plan / moe_forward / moe_get_status / moe_debug_routing, then as pipelined host
    forwards (moe_forward_host / moe_host_wait); its inputs and the oracle's expectations come
    from tests/golden/make_c_abi_case.py (oracle and synth only)."""
    import sys
    sys.path.insert(0, os.path.join(ROOT, "tests", "golden"))
    import make_c_abi_case
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    case = tmp_path / "case"
    make_c_abi_case.write_case(str(case))
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_gpu")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_gpu.c"), "-L", lib_dir,
           "-lmoe_gb300", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", "-Wl,-rpath," + lib_dir,
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe, str(case)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
    print(r.stdout.strip())
