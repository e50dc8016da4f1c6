"""GPU side of the launch-configuration search ("Stax (4): GPU Codegen and
Dynamic Shapes", section 9.6): every compiled point of the cross-entropy
kernels' configuration space (the ring kernel's box and the warp-per-row
points) gives the oracle's results, configurations that
cannot run are refused, and the tuner (Algorithm 9.1 then 9.2) records a
configuration that fr_xent then uses."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_bits_equal, assert_close
from gpu_util import bf16_tensor
from synth import workloads

pytestmark = pytest.mark.gpu

BOX = [(t, u, s) for t in (128, 256, 512, 1024) for u in (1, 2, 4, 8) for s in (2, 4, 8)]
WARP = [(32, 4, 1), (32, 8, 1)]  # the warp-per-row family


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def test_every_runnable_configuration_matches_the_oracle(o):
    rows, cols = 37, 50257  # unaligned rows (100514-byte pitch), several rows per CTA
    w = workloads.make(4, rows=rows, cols=cols, seed=4242)
    ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
    lg = bf16_tensor(w.arrays["logits"])
    t = torch.from_numpy(w.arrays["target"]).cuda()
    ran = 0
    try:
        for (th, u, s) in BOX + WARP:
            for g in (1, 2, 4):
                try:
                    fr.fr_xent_set_config(rows, cols, (th, u, s, g))
                except fr.FRError as e:  # cannot run here: shared memory, residency, spills
                    assert "UNSUPPORTED_FORM" in str(e)
                    continue
                assert fr.fr_xent_get_config(rows, cols) == (th, u, s, g)
                r = fr.fr_xent(lg, t, -100, want_target_logit=True)
                what = f"config {(th, u, s, g)}"
                assert_close(r["loss"].cpu().numpy(), ref["loss"], "loss", what)
                assert_close(r["mean"].cpu().numpy()[0], ref["mean"], "loss", what)
                assert_bits_equal(r["target_logit"].cpu().numpy(),
                                  ref["target_logit"].astype(np.float32), what)
                ran += 1
    finally:
        fr.fr_xent_set_config(rows, cols, None)
    assert ran >= 63
    assert fr.fr_xent_get_config(rows, cols) == (32, 8, 1, 2)  # the default again
    assert fr.fr_check_device_error() == 0


def test_configurations_outside_the_box_or_unrunnable_are_refused():
    for bad in [(100, 4, 4, 1), (256, 3, 4, 1), (256, 4, 1, 1), (256, 4, 4, 32), (2048, 4, 4, 1),
                (32, 4, 2, 1), (32, 2, 1, 1), (32, 4, 1, 32), (64, 4, 1, 1)]:
        with pytest.raises(fr.FRError, match="INVALID_ARG"):
            fr.fr_xent_set_config(64, 1000, bad)
    for cannot in [(1024, 8, 2, 1),    # not compiled: spills at 1024 threads x 8 vectors
                   (1024, 4, 8, 1),    # 512 KiB of ring
                   (512, 4, 4, 16),    # 16 CTAs of 128 KiB cannot be resident
                   (32, 8, 1, 4)]:     # 8 vectors a lane: two CTAs per SM at most
        with pytest.raises(fr.FRError, match="UNSUPPORTED_FORM"):
            fr.fr_xent_set_config(64, 1000, cannot)


def test_tune_records_a_configuration_that_fr_xent_uses(o):
    rows, cols = 1024, 50257
    w = workloads.make(4, rows=rows, cols=cols, seed=77)
    lg = bf16_tensor(w.arrays["logits"])
    t = torch.from_numpy(w.arrays["target"]).cuda()
    fr.fr_xent_set_config(rows, cols, None)
    try:
        res = fr.fr_xent_tune(lg, t, -100, eps=0.02, reps=3)
        th, u, s, g = res["config"]
        assert (th, u, s) in BOX + WARP and g in (1, 2, 4, 8, 16)
        assert res["evaluations"] >= 8 and res["ms"] > 0
        assert fr.fr_xent_get_config(rows, cols) == res["config"]
        again = fr.fr_xent_tune(lg, t, -100)  # Algorithm 9.1, line 1: the record, unmeasured
        assert again["config"] == res["config"] and again["evaluations"] == 0
        r = fr.fr_xent(lg, t, -100)
        ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
        assert_close(r["loss"].cpu().numpy(), ref["loss"], "loss", f"tuned {res['config']}")
        assert_close(r["mean"].cpu().numpy()[0], ref["mean"], "loss", "tuned mean")
    finally:
        fr.fr_xent_set_config(rows, cols, None)
