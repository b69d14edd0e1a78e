"""The C ABI from a C program (examples/lmloss_c_example.c), with no Python in
the call path: it builds against include/lmloss.h and the library here, and on
a GPU its losses and gradient match the fp64 oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "examples", "lmloss_c_example.c")
CUDA = "/usr/local/cuda"


def _build(tmp_path):
    import lm_head_vocab_gb300._lib as L
    L.build()
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "lmloss_c_example")
    libdir = os.path.dirname(L.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), SRC, "-L", libdir, "-llmloss",
                    "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + libdir, "-o", exe],
                   check=True)
    return exe


def test_c_example_builds_and_links(tmp_path):
    exe = _build(tmp_path)
    assert os.access(exe, os.X_OK)
    # without arguments it prints its usage and exits 2, having touched no GPU
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 2 and "usage" in r.stderr


@pytest.mark.gpu
def test_c_example_matches_oracle(tmp_path):
    exe = _build(tmp_path)
    rng = np.random.default_rng(7)
    T, V = 40, 3001
    x = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    t = rng.integers(0, V, size=T).astype(np.int64)
    t[[3, 17]] = -100
    x.tofile(tmp_path / "x.f32")
    t.tofile(tmp_path / "t.i64")
    r = subprocess.run([exe, str(T), str(V), str(tmp_path / "x.f32"), str(tmp_path / "t.i64"),
                        str(tmp_path / "g.f32")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    loss = np.array([float(v) for v in r.stdout.split()])
    g = np.fromfile(tmp_path / "g.f32", dtype=np.float32).reshape(T, V).astype(np.float64)
    R, g_ref = oracle.forward_backward(oracle.Problem(logits=x, V=V, targets=t, z_alpha=1e-4))
    assert abs(loss[0] - R.total) <= 1e-5 * abs(R.total)
    assert abs(loss[1] - R.ce) <= 1e-5 * R.ce and abs(loss[2] - R.z) <= 1e-5 * R.z
    assert loss[3] == 0.0 and loss[4] == 0.0
    assert np.max(np.abs(g - g_ref)) <= 1e-6
    assert np.all(g[[3, 17]] == 0.0)
    # the logits left in host memory: lmloss_forward_backward_host, same bits
    r2 = subprocess.run([exe, str(T), str(V), str(tmp_path / "x.f32"), str(tmp_path / "t.i64"),
                         str(tmp_path / "g2.f32"), "host"], capture_output=True, text=True)
    assert r2.returncode == 0, r2.stderr
    assert r2.stdout == r.stdout
    assert (tmp_path / "g2.f32").read_bytes() == (tmp_path / "g.f32").read_bytes()
