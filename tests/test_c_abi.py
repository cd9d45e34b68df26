"""The boundary from C (no GPU): tests/c_abi/host_abi.c is compiled as C11
with warnings as errors against include/gdn.h, linked to the in-tree
libgdn.so and run; it exercises the host-side calls and returns 0 when every
check holds."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_dir():
    from gated_delta_net_02_gb300 import build
    return os.path.dirname(build.build())


def test_header_compiles_as_c_and_host_calls_work(lib_dir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "host_abi")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "host_abi.c"), "-o", exe, "-L", lib_dir,
           "-lgdn", f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "passed" in r.stdout


@pytest.mark.gpu
def test_forward_from_c_matches_the_oracle(lib_dir, tmp_path):
    # device buffers from the CUDA runtime, gdn_forward through the C ABI,
    # the fp64 oracle's C entry point as the reference
    import oracle.build as ob
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    olib = os.path.dirname(ob.build())
    exe = str(tmp_path / "gpu_decode")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi", "gpu_decode.c"), "-o", exe,
           "-L", lib_dir, "-lgdn", "-L", olib, "-lgdn_oracle",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{lib_dir}:{olib}:{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
