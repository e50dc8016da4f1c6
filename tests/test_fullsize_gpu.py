"""Full-size parity: the five workloads at their real sizes, in the launch
configuration the benchmark times (FR_FORM_AUTO), compared element by element
with the oracle over every output (the oracle finishes each in seconds)."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_bits_equal, assert_close
from gpu_util import bf16_tensor, bf16_to_f32_host
from synth import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("nan", [False, True], ids=["plain", "4nan"])
def test_config0_example_1_1(o, nan):
    w = workloads.make(0, nan_variant=nan)
    a, b = (torch.from_numpy(w.arrays[k]).cuda() for k in ("a", "b"))
    got = fr.fr_reduce_relu_add_sum(a, b, 2.0).cpu().numpy()
    assert fr.fr_last_form() == "persistent"
    assert_close(got, o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0), "f32", "config 0")


def test_config1_softmax(o):
    w = workloads.make(1)
    y = fr.fr_softmax(torch.from_numpy(w.arrays["x"]).cuda())
    assert fr.fr_last_form() == "persistent"
    got = y.cpu().numpy()
    del y
    assert_close(got, o.softmax(w.arrays["x"]), "f32", "config 1")


def test_config2_layernorm(o):
    w = workloads.make(2)
    x = bf16_tensor(w.arrays["x"])
    g, b = (torch.from_numpy(w.arrays[k]).cuda() for k in ("gamma", "beta"))
    eps = float(np.float32(w.params["eps"]))
    y, mean, rstd = fr.fr_layernorm(x, g, b, eps)
    yh, mh, rh = bf16_to_f32_host(y), mean.cpu().numpy(), rstd.cpu().numpy()
    del x, y
    ry, rm, rr = o.layernorm(w.arrays["x"], w.arrays["gamma"], w.arrays["beta"], eps)
    assert_close(mh, rm, "mean", "config 2 mean")
    assert_close(rh, rr, "f32", "config 2 rstd")
    assert_close(yh, ry, "bf16", "config 2 y")


def test_config3_split_deterministic(o):
    w = workloads.make(3)
    a, b = (torch.from_numpy(w.arrays[k]).cuda() for k in ("a", "b"))
    first = fr.fr_reduce_relu_add_sum(a, b, 2.0).cpu().numpy()
    assert fr.fr_last_form() == "split"
    for _ in range(10):
        assert_bits_equal(fr.fr_reduce_relu_add_sum(a, b, 2.0).cpu().numpy(), first, "config 3 rerun")
    del a, b
    assert_close(first, o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0), "f32", "config 3")


def test_config4_cross_entropy(o):
    w = workloads.make(4)
    lg = bf16_tensor(w.arrays["logits"])
    t = torch.from_numpy(w.arrays["target"]).cuda()
    r = fr.fr_xent(lg, t, -100, want_target_logit=True, want_argmax=True)
    got = {k: v.cpu().numpy() for k, v in r.items()}
    first_mean = got["mean"].copy()
    for _ in range(5):  # the mean is summed in a fixed order
        again = fr.fr_xent(lg, t, -100)["mean"].cpu().numpy()
        assert_bits_equal(again, first_mean, "config 4 mean rerun")
    del lg
    assert fr.fr_check_device_error() == 0
    ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
    assert ref["n_counted"] == 8192 - 410
    assert_close(got["loss"], ref["loss"], "loss", "config 4 loss")
    assert_close(got["mean"][0], ref["mean"], "loss", "config 4 mean")
    assert_bits_equal(got["target_logit"], ref["target_logit"].astype(np.float32), "target logit")
    assert_bits_equal(got["argmax"], ref["argmax"], "argmax")
