"""A plain C program (tests/c/abi_example.c) built against include/vce.h and
libvce.so: the header compiles as C and links on any host; on a GB300 the
program runs the logits form (separate and fused calls) on the hand-derived
worked example and the linear form on tests/golden/linear_case.json, whose
expected values tests/golden/make_linear_case.py computed with the oracle."""
import json
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
    cmd = [cc, "-std=c11", "-O1", "-Wall", "-Werror", SRC, "-o", str(exe), "-I", os.path.join(ROOT, "include"),
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


def write_linear_case(path):
    """The golden JSON as the whitespace-separated text the C program reads."""
    with open(os.path.join(ROOT, "tests", "golden", "linear_case.json")) as f:
        c = json.load(f)
    head = [c["n"], c["h"], c["v"], repr(c["label_smoothing"]), c["reduce_loss"], c["ignore_idx"],
            repr(c["grad_output"][0]), c["n_valid"], repr(c["loss"])]
    parts = [" ".join(str(x) for x in head)]
    parts += [" ".join(str(int(t)) for t in c["target"]), " ".join(str(b) for b in c["x_bf16_bits"]),
              " ".join(str(b) for b in c["w_bf16_bits"])]
    parts += [" ".join(repr(float(v)) for v in c[k]) for k in ("lse", "dX", "dW")]
    path.write_text("\n".join(parts) + "\n")
    return c


def test_golden_linear_case_is_the_oracles():
    # the stored expected values are what the oracle gives today on the stored inputs
    import numpy as np
    import oracle
    with open(os.path.join(ROOT, "tests", "golden", "linear_case.json")) as f:
        c = json.load(f)
    n, h, v = c["n"], c["h"], c["v"]
    x = np.array(c["x_bf16_bits"], dtype=np.uint16).reshape(n, h)
    w = np.array(c["w_bf16_bits"], dtype=np.uint16).reshape(v, h)
    y = np.array(c["target"], dtype=np.int64)
    f = oracle.lce_forward(x, w, y, c["label_smoothing"], c["reduce_loss"])
    dx, dw, _ = oracle.lce_backward(x, w, y, f["lse"], f["n_valid"], c["grad_output"], c["label_smoothing"],
                                    c["reduce_loss"], z=f["z"])
    assert f["n_valid"] == c["n_valid"] and abs(f["loss"] - c["loss"]) <= 1e-12
    np.testing.assert_allclose(f["lse"], c["lse"], rtol=1e-12)
    np.testing.assert_allclose(dx.ravel(), c["dX"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(dw.ravel(), c["dW"], rtol=1e-10, atol=1e-15)


@pytest.mark.gpu
def test_c_program_runs_linear_form(tmp_path):
    exe, _ = build_example(tmp_path)
    case = tmp_path / "linear_case.txt"
    write_linear_case(case)
    r = subprocess.run([str(exe), str(case)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_example ok" in r.stdout and "abi_example linear ok" in r.stdout
