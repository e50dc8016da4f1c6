"""The programmatic overlap of consecutive kernels changes when CTAs are
placed, never what they compute: every op gives the same bits with it
(the default) and without it (FR_PDL=0, read once per process, so the second
run is a child process), also when the output of one call is the input of
the next one on the same stream."""
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import reduction_pointwise_row_gb300 as fr
from synth import workloads
out = {}
w = workloads.make(1, rows=4096, cols=1000, seed=11)
x = torch.from_numpy(w.arrays["x"]).cuda()
y = fr.fr_softmax(x)
z = fr.fr_softmax(y)          # reads what the previous kernel wrote
out["softmax2"] = z.cpu().numpy()
w = workloads.make(2, rows=300, cols=32768, seed=12)
xl = torch.from_numpy(w.arrays["x"].view(np.int16)).cuda().view(torch.bfloat16)
g, b = (torch.from_numpy(w.arrays[k]).cuda() for k in ("gamma", "beta"))
yl, m, r = fr.fr_layernorm(xl, g, b, 1e-5)
yl2, m2, r2 = fr.fr_layernorm(yl, g, b, 1e-5)  # chained
out["ln2"] = yl2.view(torch.int16).cpu().numpy(); out["ln_mean"] = m.cpu().numpy()
w = workloads.make(4, rows=500, cols=50257, seed=13)
lg = torch.from_numpy(w.arrays["logits"].view(np.int16)).cuda().view(torch.bfloat16)
t = torch.from_numpy(w.arrays["target"]).cuda()
res = fr.fr_xent(lg, t, -100, want_argmax=True)
out["xent_loss"] = res["loss"].cpu().numpy(); out["xent_mean"] = res["mean"].cpu().numpy()
out["xent_argmax"] = res["argmax"].cpu().numpy()
w = workloads.make(0, rows=300, cols=3000, seed=14)
a, bb = (torch.from_numpy(w.arrays[k]).cuda() for k in ("a", "b"))
out["ras"] = fr.fr_reduce_relu_add_sum(a, bb, 2.0).cpu().numpy()
torch.cuda.synchronize()
np.savez(sys.argv[2], **out)
'''


def run_child(path, pdl: str):
    env = dict(os.environ, FR_PDL=pdl)
    subprocess.run([sys.executable, "-c", CHILD, ROOT, str(path)], env=env, check=True,
                   timeout=600)
    return np.load(path)


def test_same_bits_with_and_without_the_overlap(tmp_path):
    on = run_child(tmp_path / "on.npz", "1")
    off = run_child(tmp_path / "off.npz", "0")
    for k in on.files:
        assert on[k].tobytes() == off[k].tobytes(), k
