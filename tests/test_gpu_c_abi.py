"""The C ABI from plain C: tests/c_abi_roundtrip.c is compiled with gcc against
include/ep_gb300.h, linked with libep_gb300.so and the CUDA runtime, and run;
it checks a layout / dispatch / combine round trip on the host and prints "ok"."""
import glob
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def cuda_home():
    for c in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if c and os.path.isdir(os.path.join(c, "include")):
            return c
    pytest.skip("no CUDA toolkit headers")


def cudart_dir(home):
    for pat in ("lib64/libcudart.so*", "lib/libcudart.so*", "targets/*/lib/libcudart.so*"):
        hits = glob.glob(os.path.join(home, pat))
        if hits:
            return os.path.dirname(hits[0])
    pytest.skip("no shared CUDA runtime")


def test_c_program_round_trip(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    home = cuda_home()
    libdir = os.path.join(ROOT, "combine_ep_layout_gb300")
    rt = cudart_dir(home)
    exe = str(tmp_path / "c_abi_roundtrip")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(home, "include"),
                    os.path.join(ROOT, "tests", "c_abi_roundtrip.c"),
                    "-L", libdir, "-lep_gb300", "-L", rt, "-lcudart",
                    "-Wl,-rpath," + libdir, "-Wl,-rpath," + rt, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
