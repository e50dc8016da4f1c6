"""The workspace-free split entry point against the regular one (GPU).

fr_reduce_relu_add_sum_split_static serves callers that cannot allocate device
memory where they launch -- code inside a host framework that owns every device
allocation, latency-critical paths where cudaMalloc/cudaFree may synchronise
the device, interfaces with no way to pass a workspace pointer.  Its partial
sums live in a fixed 64 KiB array inside the library instead of a caller
workspace.  These tests call it through the C ABI and check what its header
promises: the same bits as fr_reduce_relu_add_sum in its split form (the same
kernels with the same segment count), the oracle's values (bit for bit on
dyadic inputs, where every partial sum is exact), and no trace of an earlier
call's partials in a later call that uses fewer of them in another layout.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_bits_equal, assert_close
from synth import workloads

pytestmark = pytest.mark.gpu

F32, SPLIT, OP_RELU_ADD_SUM = 0, 3, 0


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def call_static(a, b, out, scale):
    rows, cols = a.shape
    return fr.lib().fr_reduce_relu_add_sum_split_static(
        _vp(a), _vp(b), _vp(out), rows, cols, a.stride(0), b.stride(0), F32, scale, _stream())


def call_with_workspace(a, b, out, scale):
    rows, cols = a.shape
    lib = fr.lib()
    n = lib.fr_workspace_size(OP_RELU_ADD_SUM, rows, cols, F32, SPLIT)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=a.device)
    status = lib.fr_reduce_relu_add_sum(_vp(a), _vp(b), _vp(out), rows, cols, a.stride(0),
                                        b.stride(0), F32, scale, SPLIT, _vp(ws), n, _stream())
    torch.cuda.synchronize()
    return status


def static_and_workspace(a_host, b_host, scale):
    """(static result, workspace result) on the same device inputs."""
    a = torch.from_numpy(a_host).cuda()
    b = torch.from_numpy(b_host).cuda()
    rows = a.shape[0]
    got = torch.full((rows,), float("nan"), device="cuda")
    ref = torch.full((rows,), float("nan"), device="cuda")
    assert call_static(a, b, got, scale) == fr.FR_OK
    torch.cuda.synchronize()
    assert fr.lib().fr_last_form() == SPLIT
    assert call_with_workspace(a, b, ref, scale) == fr.FR_OK
    return got.cpu().numpy(), ref.cpu().numpy()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def test_static_scratch_matches_the_workspace_split_form_twice_in_a_row(o):
    """Two calls in a row with different shapes and data: the same bits as the
    workspace split form and the oracle's values within the fp32 tolerance."""
    cases = [(8, 1 << 22, 2.0, 11), (5, (1 << 20) + 3, -0.5, 12)]
    for rows, cols, scale, seed in cases:
        w = workloads.make(3, rows=rows, cols=cols, seed=seed)
        got, ref = static_and_workspace(w.arrays["a"], w.arrays["b"], scale)
        what = f"static scratch {rows}x{cols}"
        assert_bits_equal(got, ref, what + " vs workspace")
        assert_close(got, o.relu_add_sum(w.arrays["a"], w.arrays["b"], scale), "f32",
                     what + " vs oracle")
        assert np.isfinite(got).all()


def test_static_scratch_is_bit_exact_on_dyadic_rows(o):
    """k/64 inputs below 65536 columns: every partial sum is exact, so the call
    equals the oracle bit for bit (14 segments per row here)."""
    rng = np.random.default_rng(7)
    rows, cols = 9, 60000
    a = (rng.integers(-64, 65, (rows, cols)) / 64).astype(np.float32)
    b = (rng.integers(-64, 65, (rows, cols)) / 64).astype(np.float32)
    got, ref = static_and_workspace(a, b, 2.0)
    exact = o.relu_add_sum(a, b, 2.0).astype(np.float32)
    assert_bits_equal(got, exact, "dyadic static vs oracle")
    assert_bits_equal(ref, exact, "dyadic workspace vs oracle")


def test_no_stale_partials_after_a_larger_call(o):
    """A call that fills the array's first slots with large partials (8 rows x
    76 segments on a 152-SM GB300), then one that uses fewer of them in another
    layout (2 rows x 128 segments): a slot the second call's first stage failed
    to write would add a stale large partial."""
    big = workloads.make(3, rows=8, cols=1 << 22, seed=21)
    got_big, ref_big = static_and_workspace(big.arrays["a"], big.arrays["b"], 1.0e6)
    assert_bits_equal(got_big, ref_big, "large partials")
    small = workloads.make(3, rows=2, cols=(1 << 19) + 5, seed=22)
    got, ref = static_and_workspace(small.arrays["a"], small.arrays["b"], 2.0)
    assert_bits_equal(got, ref, "after the larger call")
    assert_close(got, o.relu_add_sum(small.arrays["a"], small.arrays["b"], 2.0), "f32",
                 "after the larger call vs oracle")


def test_static_scratch_refuses_shapes_beyond_its_size():
    rows, cols = 8193, 16  # one partial per row: 8193 > 8192 slots
    a = torch.zeros(rows, cols, device="cuda")
    out = torch.full((rows,), 7.0, device="cuda")
    assert call_static(a, a, out, 2.0) == 5  # FR_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert (out == 7.0).all()  # nothing was enqueued
