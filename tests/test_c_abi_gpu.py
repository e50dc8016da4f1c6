"""The C ABI from a plain C program (tests/c_abi/softmax_xent_from_c.c): gcc
against include/fr.h, linked with libfr.so and the CUDA runtime, no Python
or PyTorch in the process.  Its fr_softmax and fr_xent outputs must match the
oracle like the binding's."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from compare import assert_close
from synth import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    import reduction_pointwise_row_gb300 as fr
    from reduction_pointwise_row_gb300 import buildlib
    lib = fr.library_path()
    assert os.path.exists(lib)
    cuda_lib = buildlib._cuda_lib_dir(buildlib._nvcc())
    cuda_inc = os.path.join(os.path.dirname(cuda_lib.rstrip("/")), "include")
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(
            buildlib._nvcc()))), "include")
    out = str(tmp_path_factory.mktemp("c_abi") / "softmax_xent_from_c")
    lib_dir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "c_abi", "softmax_xent_from_c.c"),
                    "-o", out, "-L", lib_dir, "-lfr", "-L", cuda_lib, "-lcudart",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}"], check=True)
    return out


def test_softmax_and_xent_from_a_c_program(c_program, tmp_path):
    rows, cols = 300, 1000
    x = workloads.make(1, rows=rows, cols=cols, seed=9100).arrays["x"]
    w = workloads.make(4, rows=rows, cols=cols, seed=9101)
    lg, t = w.arrays["logits"], w.arrays["target"]
    paths = {k: str(tmp_path / k) for k in ("x", "y", "lg", "t", "loss")}
    x.tofile(paths["x"])
    lg.tofile(paths["lg"])
    t.astype(np.int64).tofile(paths["t"])
    r = subprocess.run([c_program, str(rows), str(cols), paths["x"], paths["y"], paths["lg"],
                        paths["t"], paths["loss"]], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    o = oracle.get()
    y = np.fromfile(paths["y"], np.float32).reshape(rows, cols)
    assert_close(y, o.softmax(x), "f32", "softmax from C")
    loss = np.fromfile(paths["loss"], np.float32)
    ref = o.xent(lg, t, -100)
    assert_close(loss[:rows], ref["loss"], "loss", "xent loss from C")
    assert_close(loss[rows], ref["mean"], "loss", "xent mean from C")
