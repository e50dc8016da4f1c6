"""CUDA Graph capture of the library's calls ("Stax (4): GPU Codegen and Dynamic
Shapes", section 9.9: a fixed sequence of launches recorded once and replayed
with one submission, valid while the shapes and the buffer addresses stay the
same).  The calls enqueue kernels on the caller's stream without allocating
or synchronising (the cross-entropy workspace is prepared once, before the
capture), so they can be captured; replays on new data written into the captured buffers must match
the oracle."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_close
from gpu_util import bf16_tensor, bf16_to_f32_host
from synth import workloads

pytestmark = pytest.mark.gpu


def capture(fn):
    """Warm up fn on a side stream, then capture it into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_graph_replays_every_op_on_new_data():
    o = oracle.get()
    dev = "cuda"
    # buffers fixed for the graph's lifetime
    a = torch.empty(8, 1 << 20, device=dev)
    b = torch.empty_like(a)
    ras_out = torch.empty(8, device=dev)
    ras_ws = torch.empty(fr.fr_workspace_size("relu_add_sum", 8, 1 << 20, "f32", "split"),
                         dtype=torch.uint8, device=dev)
    x = torch.empty(300, 1000, device=dev)
    y = torch.empty_like(x)
    lx = torch.empty(64, 4096, dtype=torch.bfloat16, device=dev)
    gam = torch.empty(4096, device=dev)
    bet = torch.empty(4096, device=dev)
    ly = torch.empty_like(lx)
    lm = torch.empty(64, device=dev)
    lr = torch.empty(64, device=dev)
    lg = torch.empty(33, 50257, dtype=torch.bfloat16, device=dev)
    tg = torch.empty(33, dtype=torch.int64, device=dev)
    xws = fr.fr_xent_workspace(33, 50257, "bf16")
    out = {}

    def step():
        fr.fr_reduce_relu_add_sum(a, b, 2.0, form="split", out=ras_out, workspace=ras_ws)
        fr.fr_softmax(x, out=y)
        fr.fr_layernorm(lx, gam, bet, 1e-5, out=ly, mean=lm, rstd=lr)
        out["xent"] = fr.fr_xent(lg, tg, -100, workspace=xws)

    def load(seed):
        w = workloads.make(3, rows=8, cols=1 << 20, seed=seed)
        a.copy_(torch.from_numpy(w.arrays["a"]))
        b.copy_(torch.from_numpy(w.arrays["b"]))
        w1 = workloads.make(1, rows=300, cols=1000, seed=seed)
        x.copy_(torch.from_numpy(w1.arrays["x"]))
        w2 = workloads.make(2, rows=64, cols=4096, seed=seed)
        lx.copy_(bf16_tensor(w2.arrays["x"]))
        gam.copy_(torch.from_numpy(w2.arrays["gamma"]))
        bet.copy_(torch.from_numpy(w2.arrays["beta"]))
        w4 = workloads.make(4, rows=33, cols=50257, seed=seed)
        lg.copy_(bf16_tensor(w4.arrays["logits"]))
        tg.copy_(torch.from_numpy(w4.arrays["target"]))
        return w, w1, w2, w4

    load(1)
    graph = capture(step)
    for seed in (2, 3):  # replays on data the graph has never seen
        w, w1, w2, w4 = load(seed)
        graph.replay()
        torch.cuda.synchronize()
        assert_close(ras_out.cpu().numpy(), o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0),
                     "f32", f"graph split {seed}")
        assert_close(y.cpu().numpy(), o.softmax(w1.arrays["x"]), "f32", f"graph softmax {seed}")
        ry, rm, rr = o.layernorm(w2.arrays["x"], w2.arrays["gamma"], w2.arrays["beta"],
                                 float(np.float32(1e-5)))
        assert_close(bf16_to_f32_host(ly), ry, "bf16", f"graph layernorm {seed}")
        assert_close(lm.cpu().numpy(), rm, "mean", f"graph layernorm mean {seed}")
        ref = o.xent(w4.arrays["logits"], w4.arrays["target"], -100)
        assert_close(out["xent"]["loss"].cpu().numpy(), ref["loss"], "loss", f"graph xent {seed}")
        assert_close(out["xent"]["mean"].cpu().numpy()[0], ref["mean"], "loss",
                     f"graph xent mean {seed}")
    assert fr.fr_check_device_error() == 0
