"""fr_softmax_host: rows in page-locked host memory, read and written by the
kernel directly (chunk_rows 0) or through the library's chunked copy-in /
kernel / copy-out pipeline; results must be fr_softmax's, compared with the
oracle element by element (fp32) or in bf16 steps (bf16)."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_bf16_within_steps, assert_close
from synth import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("rows,cols,chunk", [(1000, 1000, 64), (7, 4097, 2), (300, 20000, 300),
                                             (513, 100, 1000), (64, 65537, 5), (1000, 1000, 0),
                                             (7, 4097, 0), (300, 20000, 0), (64, 65537, 0),
                                             (513, 100, 0)])
def test_host_pipeline_fp32(o, rows, cols, chunk):
    w = workloads.make(1, rows=rows, cols=cols, seed=8000 + rows + cols)
    x = torch.from_numpy(w.arrays["x"]).pin_memory()
    y = fr.fr_softmax_host(x, chunk_rows=chunk)
    torch.cuda.current_stream().synchronize()
    assert_close(y.numpy(), o.softmax(w.arrays["x"]), "f32", f"host {rows}x{cols}/{chunk}")


def test_host_pipeline_bf16_and_in_place(o):
    bits = workloads.make_softmax_bf16(300, 2048, seed=81).arrays["x"]
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    ref = o.softmax((bits.astype(np.uint32) << 16).view(np.float32))
    y = fr.fr_softmax_host(x, chunk_rows=50)
    torch.cuda.current_stream().synchronize()
    assert_bf16_within_steps(y.view(torch.int16).numpy().view(np.uint16), ref, 1, "host bf16")
    y0 = fr.fr_softmax_host(x, chunk_rows=0)
    torch.cuda.current_stream().synchronize()
    assert_bf16_within_steps(y0.view(torch.int16).numpy().view(np.uint16), ref, 1, "direct bf16")
    x2 = x.clone().pin_memory()
    fr.fr_softmax_host(x, out=x, chunk_rows=7)  # in place
    fr.fr_softmax_host(x2, out=x2, chunk_rows=0)  # in place, direct
    torch.cuda.current_stream().synchronize()
    assert_bf16_within_steps(x.view(torch.int16).numpy().view(np.uint16), ref, 1, "in place")
    assert_bf16_within_steps(x2.view(torch.int16).numpy().view(np.uint16), ref, 1, "in place direct")


@pytest.mark.parametrize("grid", [None, "1", "3", "1000"])
@pytest.mark.parametrize("dtype,cols", [("f32", 100), ("f32", 257), ("f32", 600), ("f32", 1024),
                                        ("bf16", 300), ("bf16", 513), ("bf16", 1500),
                                        ("bf16", 2048)])
def test_host_direct_small_grid(o, dtype, cols, grid, monkeypatch):
    """The direct form's persistent grid (warps taking rows in turn): the
    default (a quarter of the SMs), one CTA, three, and more CTAs than the
    rows need; rows not a multiple of the grid's warps."""
    if grid is not None:
        monkeypatch.setenv("FR_HOST_GRID", grid)
    rows = 1237
    if dtype == "f32":
        w = workloads.make(1, rows=rows, cols=cols, seed=8100 + cols)
        x = torch.from_numpy(w.arrays["x"]).pin_memory()
        y = fr.fr_softmax_host(x, chunk_rows=0)
        torch.cuda.current_stream().synchronize()
        assert_close(y.numpy(), o.softmax(w.arrays["x"]), "f32", f"direct {rows}x{cols} grid {grid}")
    else:
        bits = workloads.make_softmax_bf16(rows, cols, seed=8200 + cols).arrays["x"]
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        ref = o.softmax((bits.astype(np.uint32) << 16).view(np.float32))
        y = fr.fr_softmax_host(x, chunk_rows=0)
        torch.cuda.current_stream().synchronize()
        assert_bf16_within_steps(y.view(torch.int16).numpy().view(np.uint16), ref, 1,
                                 f"direct bf16 {rows}x{cols} grid {grid}")
    assert fr.fr_last_form() == "persistent"


def test_host_pipeline_orders_after_earlier_work_and_full_shape(o):
    """Work queued on the stream before the call (a copy into the pinned input)
    comes first; the softmax workload's shape, sampled rows against the oracle."""
    w = workloads.make(1)
    src = torch.from_numpy(w.arrays["x"]).cuda()
    x = torch.empty(src.shape, dtype=torch.float32).pin_memory()
    x.copy_(src, non_blocking=True)  # on the current stream, not yet done
    y = fr.fr_softmax_host(x, chunk_rows=2048)
    torch.cuda.current_stream().synchronize()
    rows = np.random.default_rng(5).choice(w.rows, 48, replace=False)
    rows.sort()
    ref = o.softmax(w.arrays["x"][rows])
    assert_close(y.numpy()[rows], ref, "f32", "sampled rows")
    x.zero_()
    x.copy_(src, non_blocking=True)
    y = fr.fr_softmax_host(x)  # direct
    torch.cuda.current_stream().synchronize()
    assert_close(y.numpy()[rows], ref, "f32", "sampled rows, direct")


def test_host_pipeline_refuses_pageable_memory():
    x = torch.zeros(4, 16)  # not page-locked
    with pytest.raises(fr.FRError, match="INVALID_ARG"):
        fr.fr_softmax_host(x, out=torch.zeros(4, 16).pin_memory())
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fr.FRError, match="WORKSPACE_TOO_SMALL"):
        fr.fr_softmax_host(torch.zeros(64, 1024).pin_memory(), chunk_rows=32, workspace=ws)


def test_host_direct_takes_no_workspace_and_rejects_negative_chunks(o):
    x = torch.from_numpy(workloads.make(1, rows=16, cols=64, seed=8101).arrays["x"]).pin_memory()
    lib = fr.lib()
    assert lib.fr_softmax_host_workspace(64, fr.DTYPES["f32"], 0) == 0
    y = torch.empty_like(x).pin_memory()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.fr_softmax_host(x.data_ptr(), y.data_ptr(), 16, 64, fr.DTYPES["f32"], 0, None, 0,
                               st) == 0
    assert lib.fr_softmax_host(x.data_ptr(), y.data_ptr(), 16, 64, fr.DTYPES["f32"], -1, None, 0,
                               st) == 1  # FR_ERR_INVALID_ARG
    torch.cuda.current_stream().synchronize()
    assert_close(y.numpy(), o.softmax(x.numpy()), "f32", "direct through the C ABI")
