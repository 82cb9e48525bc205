"""A plain C program (tests/c/abi_example.c) built against include/vce.h and
libvce.so: the header compiles as C and links on any host; on a GB300 the
program runs the logits form on the hand-derived worked example."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_example(tmp_path):
    from vocabulary_cross_entropy_gb300 import build as vbuild
    lib = vbuild.build()
    libdir = os.path.dirname(lib)
    link = tmp_path / "libvce.so"
    if not link.exists():
        os.symlink(lib, link)
    exe = tmp_path / "abi_example"
    cc = shutil.which("gcc") or "cc"
    cmd = [cc, "-std=c11", "-O1", SRC, "-o", str(exe), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", str(tmp_path), "-lvce",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{tmp_path}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe, libdir


def test_c_program_compiles_and_links(tmp_path):
    exe, _ = build_example(tmp_path)
    assert exe.exists()


@pytest.mark.gpu
def test_c_program_runs_worked_example(tmp_path):
    exe, _ = build_example(tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_example ok" in r.stdout
