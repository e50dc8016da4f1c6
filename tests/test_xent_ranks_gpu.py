"""The cross entropy's batch mean over row shards (the path's one exchange
step): each fr_xent call leaves (sum of the losses it averaged, rows averaged)
in its workspace; shards' parts summed element-wise -- what an all-reduce with
sum gives the ranks -- then fr_xent_mean_from_parts must give the oracle's
mean over the whole batch.  The shards run one after another on one GPU; the
sum stands in for the collective, which the gloo test covers on the CPU."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_close
from gpu_util import bf16_tensor
from synth import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def shard_call(logits_bits, target, argmax):
    lg = bf16_tensor(logits_bits)
    t = torch.from_numpy(target).cuda()
    rows, cols = logits_bits.shape
    ws = fr.fr_xent_workspace(rows, cols, "bf16")
    r = fr.fr_xent(lg, t, want_argmax=argmax, workspace=ws)
    return r, ws


@pytest.mark.parametrize("cuts", [(0, 37, 80), (0, 1, 79, 80), (0, 40, 40, 80)])
@pytest.mark.parametrize("argmax", [False, True])
def test_mean_from_summed_parts_is_the_batch_mean(o, cuts, argmax):
    w = workloads.make(4, rows=80, cols=5003, seed=4242)
    lg, t = w.arrays["logits"], w.arrays["target"].copy()
    t[40:45] = -100
    ref = o.xent(lg, t, -100)
    total, first_ws = None, None
    for a, b in zip(cuts[:-1], cuts[1:]):
        if a == b:  # an empty shard adds nothing: parts (0, 0)
            continue
        r, ws = shard_call(lg[a:b], t[a:b], argmax)
        parts = fr.xent_mean_parts(ws)
        torch.cuda.synchronize()
        # one call's own parts: count exact, sum / count is its mean
        n = int(np.count_nonzero(t[a:b] != -100))
        assert parts[1].item() == n
        s = parts[0].item()
        assert np.float32(s / n) == r["mean"].cpu().numpy()[0]
        local = o.xent(lg[a:b], t[a:b], -100)
        assert abs(s - float(np.sum(local["loss"][t[a:b] != -100]))) <= 1e-5 * abs(s)
        if total is None:
            total, first_ws = parts.clone(), ws
        else:
            total += parts
    fr.xent_mean_parts(first_ws).copy_(total)
    mean = fr.fr_xent_mean_from_parts(first_ws)
    torch.cuda.synchronize()
    assert_close(mean.cpu().numpy()[0], ref["mean"], "loss", f"batch mean over shards {cuts}")


def test_mean_from_parts_no_counted_row_is_nan():
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    assert torch.isnan(fr.fr_xent_mean_from_parts(ws)).all()
    with pytest.raises(fr.FRError, match="MISALIGNED"):
        fr.fr_xent_mean_from_parts(ws[4:])


def test_unprepared_workspace_is_reported_and_preparing_fixes_it(o):
    """A workspace fr_xent_workspace_init never prepared (here all ones) makes
    the call record FR_DEVERR_BAD_WORKSPACE and leave the mean unwritten (the
    per-row losses are still right); once prepared, every later call works
    without another preparation."""
    w = workloads.make(4, rows=50, cols=3001, seed=4343)
    lg, t = bf16_tensor(w.arrays["logits"]), torch.from_numpy(w.arrays["target"]).cuda()
    ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
    n = fr.fr_workspace_size("xent", 50, 3001, "bf16")
    ws = torch.full((n,), 255, dtype=torch.uint8, device="cuda")
    mean = torch.full((1,), 7.0, device="cuda")
    lib = fr.lib()
    loss = torch.empty(50, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.fr_xent(lg.data_ptr(), t.data_ptr(), loss.data_ptr(), mean.data_ptr(), None, None,
                       50, 3001, 3001, -100, fr.DTYPES["bf16"], 0, ws.data_ptr(), n, st) == 0
    torch.cuda.synchronize()
    assert fr.fr_check_device_error() == 3  # FR_DEVERR_BAD_WORKSPACE
    assert mean.item() == 7.0
    assert_close(loss.cpu().numpy(), ref["loss"], "loss", "losses with a bad workspace")
    assert lib.fr_xent_workspace_init(ws.data_ptr(), n, st) == 0
    for _ in range(3):
        r = fr.fr_xent(lg, t, workspace=ws)
        torch.cuda.synchronize()
        assert fr.fr_check_device_error() == 0
        assert_close(r["mean"].cpu().numpy()[0], ref["mean"], "loss", "mean once prepared")
