"""A bounded device wait that runs out records FR_DEVERR_TIMEOUT and returns.

Every wait of a kernel on an mbarrier is bounded by a clock budget (about one
second); when it runs out the kernel records FR_DEVERR_TIMEOUT in the device
error word, issues no further copy, waits (bounded) for the copies it issued
before, and finishes, so the context stays usable.  A real copy never takes a
second, so this test uses a test-only build of the library in which the first
wait of the LayerNorm bulk-copy ring (layernorm_ring with bulk staging) has a
budget of one clock and polls without blocking: it runs out while its copy is
still in flight.  Every other wait keeps its full budget, the final drain
included, so no CTA leaves while a copy still targets its shared memory.

The variant runs in a child process (it is a second copy of the library's
symbols); there, the shortened kernel must report the timeout, and then a
default-path LayerNorm from the same library must match the oracle, which shows
that the kernel returned and left the context usable.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FR_DEVERR_TIMEOUT = 2
ROWS, COLS, CHECK_ROWS = 2048, 32768, 256


def child(lib_path: str, out_path: str) -> None:
    import ctypes
    import torch
    sys.path.insert(0, ROOT)
    from synth import workloads
    lib = ctypes.CDLL(lib_path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.fr_layernorm.restype = ctypes.c_int
    lib.fr_layernorm.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                 ctypes.c_int, ctypes.c_int, vp]
    lib.fr_check_device_error.restype = ctypes.c_int
    lib.fr_check_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    w = workloads.make(2, rows=ROWS, cols=COLS)
    x = torch.from_numpy(w.arrays["x"].view(np.int16)).cuda()
    g = torch.from_numpy(w.arrays["gamma"]).cuda()
    b = torch.from_numpy(w.arrays["beta"]).cuda()
    y = torch.empty_like(x)
    mean = torch.empty(ROWS, device="cuda")
    rstd = torch.empty(ROWS, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def layernorm(rows):
        return lib.fr_layernorm(x.data_ptr(), g.data_ptr(), b.data_ptr(), y.data_ptr(),
                                mean.data_ptr(), rstd.data_ptr(), rows, COLS, COLS, COLS, 1e-5,
                                1, 2, stream)  # FR_BF16, FR_FORM_LOOPED

    def error_code():
        code = ctypes.c_int32(0)
        status = lib.fr_check_device_error(stream, ctypes.byref(code))
        return status, code.value

    res = {}
    os.environ["FR_LAYERNORM_KERNEL"] = "ring"
    os.environ["FR_LAYERNORM_STAGE"] = "bulk"
    res["ring_status"] = layernorm(ROWS)
    res["ring_check"] = error_code()
    del os.environ["FR_LAYERNORM_KERNEL"], os.environ["FR_LAYERNORM_STAGE"]
    res["default_status"] = layernorm(CHECK_ROWS)
    res["default_check"] = error_code()
    np.savez(out_path, y=y[:CHECK_ROWS].cpu().numpy().view(np.uint16),
             mean=mean[:CHECK_ROWS].cpu().numpy(), rstd=rstd[:CHECK_ROWS].cpu().numpy())
    print(json.dumps(res), flush=True)


def test_shortened_wait_times_out_and_the_kernel_returns(tmp_path):
    sys.path.insert(0, ROOT)
    import oracle
    from compare import assert_close
    from reduction_pointwise_row_gb300 import buildlib
    from synth import workloads
    lib = buildlib.build_variant("wait_test", ["-DFR_TEST_WAIT_BUDGET=1"])
    out = str(tmp_path / "after.npz")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), lib, out],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["ring_status"] == 0
    assert res["ring_check"] == [7, FR_DEVERR_TIMEOUT], res  # FR_ERR_DEVICE_DATA, timeout
    assert res["default_status"] == 0 and res["default_check"] == [0, 0], res
    w = workloads.make(2, rows=CHECK_ROWS, cols=COLS)
    y_ref, mean_ref, rstd_ref = oracle.get().layernorm(w.arrays["x"], w.arrays["gamma"],
                                                       w.arrays["beta"], 1e-5)
    got = np.load(out)
    assert_close(got["mean"], mean_ref, "mean", "mean after the timeout")
    assert_close(got["rstd"], rstd_ref, "f32", "rstd after the timeout")
    y = (got["y"].astype(np.uint32) << 16).view(np.float32)
    assert_close(y, y_ref, "bf16", "y after the timeout")


if __name__ == "__main__":
    child(sys.argv[1], sys.argv[2])
