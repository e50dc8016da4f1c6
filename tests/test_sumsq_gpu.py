"""GPU parity of the row sum of squares (Example 6.2 of "Stax (4): GPU Codegen
and Dynamic Shapes", Listing 9.4) and the row L2 norm (Exercise 1 of "CMU
15-779 Lecture 8", section 12) against the oracle, in every reduction form,
on ragged and unaligned rows, plus the full Example 6.2 shape and the
determinism of the split form."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_bits_equal, assert_close
from gpu_util import empty_like_placed, place
from synth import workloads

pytestmark = pytest.mark.gpu

COLS = [1, 2, 7, 31, 33, 129, 781, 1000, 1024, 1025, 4097, 16384, 65537]
LAYOUTS = [(0, 0), (1, 5), (3, 0), (7, 1)]  # (offset of x in elements, row padding)


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def forms(cols):
    return (["persistent"] if cols <= 1024 else []) + ["looped", "split", "auto"]


def run(x, form, epilogue, layout=(0, 0)):
    rows, cols = x.shape
    off, pad = layout
    px = place(x, off, cols + pad)
    po = empty_like_placed(1, rows, torch.float32)
    fr.fr_reduce_sumsq(px.t, epilogue, form=form, out=po.t[0])
    torch.cuda.synchronize()
    assert po.canaries_intact(), "write outside out[]"
    return po.t[0].cpu().numpy()


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [1, 9, 70])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["aligned", "off1_pad5", "off3", "off7_pad1"])
def test_sumsq_and_l2norm_forms(o, rows, cols, layout):
    x = workloads.make_sumsq(rows, cols, seed=5000 + rows * 13 + cols).arrays["x"]
    ref_s, ref_n = o.row_sumsq(x), o.row_l2norm(x)
    for form in forms(cols):
        assert_close(run(x, form, "sum", layout), ref_s, "f32", f"sumsq {form} {rows}x{cols}")
        assert_close(run(x, form, "sqrt", layout), ref_n, "f32", f"l2norm {form} {rows}x{cols}")


@pytest.mark.parametrize("cols", [100, 1024, 4097, 65535])
def test_dyadic_rows_are_bit_exact(o, cols):
    """k/64 inputs: every square and partial sum is exact, so each form equals the
    oracle bitwise (sum of squares) and the root is the correctly rounded one."""
    rng = np.random.default_rng(cols)
    x = (rng.integers(-64, 65, (5, cols)) / 64).astype(np.float32)
    ref = o.row_sumsq(x)
    for form in forms(cols):
        assert_bits_equal(run(x, form, "sum"), ref.astype(np.float32), f"dyadic {form}")
        assert_bits_equal(run(x, form, "sqrt"), np.sqrt(ref).astype(np.float32),
                          f"dyadic root {form}")


def test_example_6_2_shape_split_and_deterministic(o):
    w = workloads.make_sumsq()
    x = torch.from_numpy(w.arrays["x"]).cuda()
    first = fr.fr_reduce_sumsq(x).cpu().numpy()
    assert fr.fr_last_form() == "split"  # 64 outputs cannot fill the GPU one warp per row
    for _ in range(20):
        assert_bits_equal(fr.fr_reduce_sumsq(x).cpu().numpy(), first, "split rerun")
    assert_close(first, o.row_sumsq(w.arrays["x"]), "f32", "Example 6.2")
    assert_close(fr.fr_reduce_sumsq(x, "sqrt").cpu().numpy(), o.row_l2norm(w.arrays["x"]),
                 "f32", "Example 6.2 L2 norm")


def test_special_values(o):
    """NaN rows stay NaN, an inf makes the row inf, and a zero row has norm 0."""
    x = workloads.make_sumsq(6, 3000, seed=77).arrays["x"].copy()
    x[1, 2999] = np.nan
    x[2, 0] = -np.inf
    x[3, :] = 0.0
    x[4, :] = 1e20  # squares overflow fp32 to inf, as in the listing's fp32 multiply
    ref_s, ref_n = o.row_sumsq(x), o.row_l2norm(x)
    for form in forms(3000):
        got = run(x, form, "sum")
        assert_close(got, ref_s, "f32", f"special {form}")
        assert np.isnan(got[1]) and got[2] == np.inf and got[3] == 0.0 and got[4] == np.inf
        assert_close(run(x, form, "sqrt"), ref_n, "f32", f"special root {form}")


def test_errors_on_device():
    x = torch.zeros(4, 8, device="cuda")
    with pytest.raises(fr.FRError, match="UNSUPPORTED_FORM"):
        fr.fr_reduce_sumsq(torch.zeros(4, 2000, device="cuda"), form="persistent")
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    big = torch.zeros(2, 1 << 20, device="cuda")
    with pytest.raises(fr.FRError, match="WORKSPACE_TOO_SMALL"):
        fr.fr_reduce_sumsq(big, form="split", workspace=ws)
    assert fr.fr_reduce_sumsq(x).cpu().numpy().tolist() == [0.0] * 4
