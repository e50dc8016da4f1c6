"""The same results from independent processes: three fresh processes compute
the split-form row sums, the cross-entropy loss and mean, the LayerNorm
statistics and the softmax of one seeded input; their bytes must be identical
(the fixed-order reductions do not depend on timing, placement or the order in
which CTAs finish), and the first process's values must match the oracle."""
import hashlib
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from compare import assert_close
from synth import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import hashlib, json, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import reduction_pointwise_row_gb300 as fr
from synth import workloads
from gpu_util import bf16_tensor
dev = torch.device("cuda")
out = {}
w = workloads.make(3, rows=4, cols=(1 << 20) + 3)
a, b = (torch.from_numpy(w.arrays[k]).to(dev) for k in ("a", "b"))
out["split"] = fr.fr_reduce_relu_add_sum(a, b, 2.0, form="split").cpu().numpy()
w = workloads.make(4, rows=700, cols=50257)
r = fr.fr_xent(bf16_tensor(w.arrays["logits"]), torch.from_numpy(w.arrays["target"]).to(dev))
out["loss"], out["mean"] = r["loss"].cpu().numpy(), r["mean"].cpu().numpy()
w = workloads.make(2, rows=64, cols=32768)
x = bf16_tensor(w.arrays["x"])
g, bt = (torch.from_numpy(w.arrays[k]).to(dev) for k in ("gamma", "beta"))
y, mean, rstd = fr.fr_layernorm(x, g, bt, 1e-5)
out["ln_mean"], out["ln_rstd"] = mean.cpu().numpy(), rstd.cpu().numpy()
out["ln_y"] = y.view(torch.int16).cpu().numpy()
w = workloads.make(1, rows=511, cols=65537)
out["softmax"] = fr.fr_softmax(torch.from_numpy(w.arrays["x"]).to(dev)).cpu().numpy()
np.savez(sys.argv[2], **out)
print(json.dumps({k: hashlib.sha256(v.tobytes()).hexdigest() for k, v in out.items()}))
"""


def test_three_processes_give_the_same_bits(tmp_path):
    digests = []
    for i in range(3):
        r = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(tmp_path / f"p{i}.npz")],
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        digests.append(json.loads(r.stdout.strip().splitlines()[-1]))
    assert digests[0] == digests[1] == digests[2], digests
    got = np.load(tmp_path / "p0.npz")
    o = oracle.get()
    w = workloads.make(3, rows=4, cols=(1 << 20) + 3)
    assert_close(got["split"], o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0), "f32", "split")
    w = workloads.make(4, rows=700, cols=50257)
    ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
    assert_close(got["loss"], ref["loss"], "loss", "loss")
    assert_close(got["mean"][0], ref["mean"], "loss", "mean")
    w = workloads.make(1, rows=511, cols=65537)
    assert_close(got["softmax"], o.softmax(w.arrays["x"]), "f32", "softmax")
    assert hashlib.sha256(got["ln_y"].tobytes()).hexdigest() == digests[0]["ln_y"]
