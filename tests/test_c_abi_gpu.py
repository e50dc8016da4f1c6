"""The C ABI from plain C programs (tests/c_abi/*.c): gcc against
include/fr.h, linked with libfr.so and the CUDA runtime, no Python or PyTorch
in the process.  softmax_xent_from_c calls fr_softmax and fr_xent;
reductions_from_c calls fr_reduce_relu_add_sum in its split form with a
workspace sized by fr_workspace_size, fr_layernorm, fr_reduce_sumsq with the
sqrt epilogue, and fr_check_device_error after a target outside the row.
Their outputs must match the oracle like the binding's."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from compare import assert_close
from synth import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def build_c_program(name, tmp_path_factory):
    import reduction_pointwise_row_gb300 as fr
    from reduction_pointwise_row_gb300 import buildlib
    lib = fr.library_path()
    assert os.path.exists(lib)
    cuda_lib = buildlib._cuda_lib_dir(buildlib._nvcc())
    cuda_inc = os.path.join(os.path.dirname(cuda_lib.rstrip("/")), "include")
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(
            buildlib._nvcc()))), "include")
    out = str(tmp_path_factory.mktemp("c_abi") / name)
    lib_dir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "c_abi", name + ".c"),
                    "-o", out, "-L", lib_dir, "-lfr", "-L", cuda_lib, "-lcudart",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}"], check=True)
    return out


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    return build_c_program("softmax_xent_from_c", tmp_path_factory)


@pytest.fixture(scope="module")
def c_reductions(tmp_path_factory):
    return build_c_program("reductions_from_c", tmp_path_factory)


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


def test_reductions_layernorm_and_device_error_from_a_c_program(c_reductions, tmp_path):
    ras_shape, ln_shape, l2_shape = (6, 300007), (300, 4096), (100, 5003)
    ras = workloads.make(3, rows=ras_shape[0], cols=ras_shape[1], seed=9200)
    ln = workloads.make(2, rows=ln_shape[0], cols=ln_shape[1], seed=9201)
    l2 = workloads.make_sumsq(l2_shape[0], l2_shape[1], seed=9202)
    files = {"a.bin": ras.arrays["a"], "b.bin": ras.arrays["b"], "x.bin": ln.arrays["x"],
             "gamma.bin": ln.arrays["gamma"], "beta.bin": ln.arrays["beta"],
             "s.bin": l2.arrays["x"]}
    for name, arr in files.items():
        np.ascontiguousarray(arr).tofile(str(tmp_path / name))
    r = subprocess.run([c_reductions, *map(str, ras_shape + ln_shape + l2_shape), str(tmp_path)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    info = dict(kv.split("=") for kv in r.stdout.split())
    assert info["ras_form"] == "3"  # FR_FORM_SPLIT, as requested
    assert info["ln_form"] == "2" and info["l2_form"] in ("1", "2")  # looped; AUTO's pick
    assert info["bad_target_status"] == "7" and info["bad_target_code"] == "1"  # BAD_TARGET
    assert info["clear_status"] == "0"
    o = oracle.get()
    got = np.fromfile(str(tmp_path / "ras.bin"), np.float32)
    assert_close(got, o.relu_add_sum(ras.arrays["a"], ras.arrays["b"], 2.0), "f32",
                 "split relu_add_sum from C")
    y_ref, mean_ref, rstd_ref = o.layernorm(ln.arrays["x"], ln.arrays["gamma"], ln.arrays["beta"],
                                            1e-5)
    y_bits = np.fromfile(str(tmp_path / "ln_y.bin"), np.uint16).reshape(ln_shape)
    assert_close((y_bits.astype(np.uint32) << 16).view(np.float32), y_ref, "bf16",
                 "layernorm y from C")
    assert_close(np.fromfile(str(tmp_path / "ln_mean.bin"), np.float32), mean_ref, "mean",
                 "layernorm mean from C")
    assert_close(np.fromfile(str(tmp_path / "ln_rstd.bin"), np.float32), rstd_ref, "f32",
                 "layernorm rstd from C")
    assert_close(np.fromfile(str(tmp_path / "l2.bin"), np.float32), o.row_l2norm(l2.arrays["x"]),
                 "f32", "row L2 norm from C")
