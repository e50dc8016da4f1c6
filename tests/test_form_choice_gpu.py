"""AUTO against every form, timed live on a few shapes whose forms differ
widely (the measured table's crossovers, Stax (4) section 9.6 Algorithm 9.1):
AUTO's time must be within the timing noise (8 %) of the fastest form's.
Calls run back to back on buffers larger than the L2, timed with CUDA events,
the median of five blocks."""
import os

import pytest
import torch

import reduction_pointwise_row_gb300 as fr

pytestmark = pytest.mark.gpu


def per_call_us(calls, steps=20, blocks=5):
    for c in calls[:3]:
        c()
    times = []
    for _ in range(blocks):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            calls[i % len(calls)]()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / steps)
    return sorted(times)[len(times) // 2]


def rotating(rows, cols, dtype, per_set_bytes):
    n = max(2, -(-(1 << 30) // per_set_bytes))
    buf = torch.empty(n * rows, cols, dtype=dtype, device="cuda").uniform_(-1, 1)
    return [buf[k * rows:(k + 1) * rows] for k in range(n)]


CASES = [("relu_add_sum", 8, 1 << 22), ("relu_add_sum", 4096, 16384), ("softmax", 2432, 32768),
         ("softmax", 304, 262144), ("softmax_bf16", 4864, 16384), ("layernorm", 174762, 768),
         ("layernorm", 4096, 32768)]


@pytest.mark.parametrize("op,rows,cols", CASES)
def test_auto_within_noise_of_the_fastest_form(op, rows, cols):
    if op == "relu_add_sum":
        A = rotating(rows, cols, torch.float32, 8 * rows * cols)
        B = rotating(rows, cols, torch.float32, 8 * rows * cols)
        out = torch.empty(rows, device="cuda")
        ws = torch.empty(max(16, fr.fr_workspace_size(op, rows, cols, "f32", "split")),
                         dtype=torch.uint8, device="cuda")

        def make(form):
            return [lambda a=a, b=b: fr.fr_reduce_relu_add_sum(a, b, 2.0, form=form, out=out,
                                                                workspace=ws)
                    for a, b in zip(A, B)]
        forms = ["looped", "split"]
    elif op.startswith("softmax"):
        dt = torch.bfloat16 if op.endswith("bf16") else torch.float32
        X = rotating(rows, cols, dt, 2 * rows * cols * X_SIZE[dt])
        Y = rotating(rows, cols, dt, 2 * rows * cols * X_SIZE[dt])

        def make(form):
            return [lambda x=x, y=y: fr.fr_softmax(x, form=form, out=y) for x, y in zip(X, Y)]
        forms = ["persistent", "looped", "split"]
    else:
        X = rotating(rows, cols, torch.bfloat16, 4 * rows * cols)
        Y = rotating(rows, cols, torch.bfloat16, 4 * rows * cols)
        g = torch.ones(cols, device="cuda")
        b = torch.zeros(cols, device="cuda")
        mean = torch.empty(rows, device="cuda")
        rstd = torch.empty(rows, device="cuda")

        def make(form):
            return [lambda x=x, y=y: fr.fr_layernorm(x, g, b, 1e-5, form=form, out=y, mean=mean,
                                                     rstd=rstd) for x, y in zip(X, Y)]
        forms = ["persistent", "looped"]
    times = {}
    for form in forms:
        try:
            times[form] = per_call_us(make(form))
        except fr.FRError:
            continue
    auto = per_call_us(make("auto"))
    best = min(times.values())
    assert auto <= 1.08 * best, (op, rows, cols, fr.fr_last_form(), auto, times)


X_SIZE = {torch.float32: 4, torch.bfloat16: 2}
