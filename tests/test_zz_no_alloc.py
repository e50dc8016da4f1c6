"""The workspace-free split entry point against the regular one (GPU).

fr_reduce_relu_add_sum_split_static serves callers that cannot allocate device
memory where they launch -- code inside a host framework that owns every device
allocation, latency-critical paths where cudaMalloc/cudaFree may synchronise
the device, interfaces with no way to pass a workspace pointer.  Its partial
sums live in a fixed 64 KiB array inside the library instead of a caller
workspace.  These tests call it through the C ABI and compare it with
fr_reduce_relu_add_sum in its split form (the existing entry point, given a
workspace), on two calls in a row with different shapes and data, so the second
call runs on an array that still holds the first call's partials.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import reduction_pointwise_row_gb300 as fr
from compare import assert_close
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


def test_static_scratch_matches_the_workspace_split_form_twice_in_a_row():
    cases = [(8, 1 << 22, 2.0, 11), (5, (1 << 20) + 3, -0.5, 12)]
    for rows, cols, scale, seed in cases:
        w = workloads.make(3, rows=rows, cols=cols, seed=seed)
        a = torch.from_numpy(w.arrays["a"]).cuda()
        b = torch.from_numpy(w.arrays["b"]).cuda()
        got = torch.full((rows,), float("nan"), device="cuda")
        ref = torch.full((rows,), float("nan"), device="cuda")
        assert call_static(a, b, got, scale) == fr.FR_OK
        torch.cuda.synchronize()
        assert call_with_workspace(a, b, ref, scale) == fr.FR_OK
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), "f32",
                     f"static scratch vs workspace {rows}x{cols}")
        assert np.isfinite(got.cpu().numpy()).all()


def test_static_scratch_refuses_shapes_beyond_its_size():
    rows, cols = 8193, 16  # one partial per row: 8193 > 8192 slots
    a = torch.zeros(rows, cols, device="cuda")
    out = torch.full((rows,), 7.0, device="cuda")
    assert call_static(a, a, out, 2.0) == 5  # FR_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert (out == 7.0).all()  # nothing was enqueued
