"""GPU parity: every op, every form, against the CPU oracle, element by element.

Shapes span several tiles with ragged tails (row lengths that are not powers of
two, rows that are not 32-byte aligned, padded row strides); outputs live in
canary-filled buffers so a write outside the logical block fails the test.
Tolerances are those of tests/compare.py.
"""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
import synth
from compare import assert_bits_equal, assert_close
from gpu_util import bf16_to_f32_host, empty_like_placed, place
from synth import workloads

pytestmark = pytest.mark.gpu

COLS = [1, 2, 3, 7, 13, 31, 33, 127, 128, 129, 781, 1000, 1023, 1024, 1025, 4097]
# (offset of input a/x, offset of b/y, extra row padding)
LAYOUTS = [(0, 0, 0), (1, 1, 5), (0, 3, 0)]


STAGE_SPLIT_MAX_F32 = 409496  # the staged split's longest fp32 row


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def forms_for(op, cols, in_phase=True):
    if op == "relu_add_sum":
        return (["persistent"] if cols <= 1024 else []) + ["looped", "split"]
    if op == "softmax":  # rows past 1024 stay persistent (a CTA per row) up to 32768
        # columns; they also split over a cluster of CTAs (in phase: the
        # slices in registers up to 262144 columns, streamed twice beyond;
        # out of phase: staged in shared memory, up to 409496)
        split = cols > 1024 and (in_phase or cols <= STAGE_SPLIT_MAX_F32)
        return ((["persistent"] if cols <= 32768 else []) + (["split"] if split else []) +
                ["looped"])
    raise ValueError(op)


# ---------------------------------------------------------------- Example 1.1

def run_ras(a, b, form, la=(0, 0, 0), scale=2.0):
    rows, cols = a.shape
    oa, ob, pad = la
    pa = place(a, oa, cols + pad)
    pb = place(b, ob, cols + pad)
    po = empty_like_placed(1, rows, torch.float32)
    fr.fr_reduce_relu_add_sum(pa.t, pb.t, scale, form=form, out=po.t[0])
    torch.cuda.synchronize()
    assert po.canaries_intact(), "write outside out[]"
    return po.t[0].cpu().numpy()


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [1, 7, 65])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["aligned", "offset_same_phase", "offset_scalar"])
def test_relu_add_sum_forms(o, rows, cols, layout):
    w = workloads.make(0, rows=rows, cols=cols, seed=1000 + rows * 7 + cols)
    ref = o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0)
    for form in forms_for("relu_add_sum", cols):
        got = run_ras(w.arrays["a"], w.arrays["b"], form, layout)
        assert_close(got, ref, "f32", f"{form} {rows}x{cols} {layout}")


def test_relu_add_sum_example_1_1_and_nan_variant(o):
    for nan in (False, True):
        w = workloads.make(0, nan_variant=nan)
        ref = o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0)
        for form in ("auto", "persistent", "looped", "split"):
            got = run_ras(w.arrays["a"], w.arrays["b"], form)
            assert_close(got, ref, "f32", f"Example 1.1 {form} nan={nan}")
        if nan:
            rows_with_nan = {r for _, r, _ in w.params["nan_positions"]}
            assert set(np.flatnonzero(np.isnan(got)).tolist()) == rows_with_nan


@pytest.mark.parametrize("cols", [128, 1000, 4097, 65535])
def test_relu_add_sum_dyadic_is_bit_exact(o, cols):
    """k/64 inputs: every partial sum is exact, so all forms equal the oracle bitwise."""
    rng = np.random.default_rng(cols)
    a = (rng.integers(-64, 65, (9, cols)) / 64).astype(np.float32)
    b = (rng.integers(-64, 65, (9, cols)) / 64).astype(np.float32)
    ref = o.relu_add_sum(a, b, 2.0).astype(np.float32)
    for form in forms_for("relu_add_sum", cols):
        assert_bits_equal(run_ras(a, b, form), ref, f"{form} {cols}")


def test_relu_add_sum_split_long_rows_deterministic(o):
    rows, cols = 3, (1 << 20) + 3
    w = workloads.make(3, rows=rows, cols=cols)
    ref = o.relu_add_sum(w.arrays["a"], w.arrays["b"], 2.0)
    pa, pb = place(w.arrays["a"], 1), place(w.arrays["b"], 1)
    first = None
    for _ in range(50):
        got = fr.fr_reduce_relu_add_sum(pa.t, pb.t, 2.0, form="split").cpu().numpy()
        if first is None:
            first = got
            assert_close(got, ref, "f32", "split long rows")
        assert_bits_equal(got, first, "split run-to-run")


def test_relu_add_sum_scale_and_infinities(o):
    a = np.array([[np.inf, 1.0, -2.0], [-np.inf, 0.5, 0.25], [np.inf, 0.0, 0.0]], np.float32)
    b = np.array([[1.0, 1.0, 1.0], [1.0, 0.5, 0.25], [-np.inf, 0.0, 0.0]], np.float32)
    for scale in (2.0, -3.0, 0.5):
        ref = o.relu_add_sum(a, b, scale)
        for form in forms_for("relu_add_sum", 3):
            assert_close(run_ras(a, b, form, scale=scale), ref, "f32", f"{form} scale {scale}")


def _widen(bits):
    return synth.bf16_bits_to_f32(bits)


@pytest.mark.parametrize("cols", [1, 3, 7, 13, 31, 33, 129, 1000, 1024, 2047, 2048, 2049, 4097])
@pytest.mark.parametrize("rows", [1, 7, 65])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["aligned", "offset_same_phase", "offset_scalar"])
def test_relu_add_sum_bf16_forms(o, rows, cols, layout):
    """bf16 inputs: the oracle on the exactly widened values (the sum a + b in
    fp32, as for fp32 inputs); persistent up to 2048 columns."""
    seed = 1500 + rows * 7 + cols
    a = synth.normal_bf16((rows, cols), seed, 0, 0.0, 1.0)
    b = synth.normal_bf16((rows, cols), seed, 1, 0.0, 1.0)
    ref = o.relu_add_sum(_widen(a), _widen(b), 2.0)
    forms = (["persistent"] if cols <= 2048 else []) + ["looped", "split", "auto"]
    for form in forms:
        got = run_ras(a, b, form, layout)
        assert_close(got, ref, "f32", f"bf16 {form} {rows}x{cols} {layout}")


@pytest.mark.parametrize("cols", [128, 2048, 4097, 65535])
def test_relu_add_sum_bf16_dyadic_is_bit_exact(o, cols):
    """k/64 values are bf16 numbers: every partial sum is exact, as for fp32."""
    rng = np.random.default_rng(cols + 1)
    af = (rng.integers(-64, 65, (9, cols)) / 64).astype(np.float32)
    bf = (rng.integers(-64, 65, (9, cols)) / 64).astype(np.float32)
    a, b = (af.view(np.uint32) >> 16).astype(np.uint16), (bf.view(np.uint32) >> 16).astype(np.uint16)
    assert (_widen(a) == af).all()
    ref = o.relu_add_sum(af, bf, 2.0).astype(np.float32)
    for form in (["persistent"] if cols <= 2048 else []) + ["looped", "split"]:
        assert_bits_equal(run_ras(a, b, form), ref, f"bf16 {form} {cols}")


# ---------------------------------------------------------------- softmax

def run_softmax(x, form, layout=(0, 0, 0), kernel=None):
    """kernel pins the persistent kernel: "async" (cp.async ring) or "plain"."""
    import os
    rows, cols = x.shape
    ox, oy, pad = layout
    px = place(x, ox, cols + pad)
    py = empty_like_placed(rows, cols, torch.float32, oy, cols + pad)
    if kernel:
        os.environ["FR_SOFTMAX_KERNEL"] = kernel
    try:
        fr.fr_softmax(px.t, form=form, out=py.t)
    finally:
        os.environ.pop("FR_SOFTMAX_KERNEL", None)
    torch.cuda.synchronize()
    assert py.canaries_intact(), "softmax wrote outside y"
    return py.t.cpu().numpy()


# out of phase the persistent form holds rows of up to 4608 columns in
# registers and stages longer ones (up to 32768) in shared memory
@pytest.mark.parametrize("cols", COLS + [2048, 2055, 2056, 4608, 4609, 8193, 16385, 32768, 32769,
                                         65537])
@pytest.mark.parametrize("rows", [1, 7, 33])
@pytest.mark.parametrize("layout", LAYOUTS + [(1, 0, 3), (2, 7, 1), (3, 1, 0), (4, 0, 1)],
                         ids=["aligned", "offset_same_phase", "offset_scalar", "out_of_phase_1",
                              "out_of_phase_2", "out_of_phase_3", "out_of_phase_16B"])
def test_softmax_forms(o, rows, cols, layout):
    w = workloads.make(1, rows=rows, cols=cols, seed=2000 + rows * 7 + cols)
    ref = o.softmax(w.arrays["x"])
    in_phase = layout[0] == layout[1]
    for form in forms_for("softmax", cols, in_phase):
        for kernel in (("async", "plain") if form == "persistent" else (None,)):
            assert_close(run_softmax(w.arrays["x"], form, layout, kernel), ref, "f32",
                         f"{form}/{kernel} {rows}x{cols} {layout}")


@pytest.mark.parametrize("kernel,cols", [("stage", 1025), ("stage", 2055), ("stage", 4097),
                                         ("shift", 8192), ("shift", 12289), ("shift", 16374)])
@pytest.mark.parametrize("layout", [(1, 0, 3), (2, 7, 1), (4, 0, 1)])
def test_softmax_out_of_phase_pinned(o, kernel, cols, layout):
    """The out-of-phase kernels where AUTO does not take them, pinned by
    FR_SOFTMAX_OOP: x staged in shared memory for short rows, the row in
    registers with 8 chunks a thread up to 16 warps (16374 columns at any
    offset) for long ones."""
    import os
    w = workloads.make(1, rows=7, cols=cols, seed=2700 + cols)
    os.environ["FR_SOFTMAX_OOP"] = kernel
    try:
        got = run_softmax(w.arrays["x"], "persistent", layout)
    finally:
        os.environ.pop("FR_SOFTMAX_OOP", None)
    assert_close(got, o.softmax(w.arrays["x"]), "f32", f"{kernel} 7x{cols} {layout}")


@pytest.mark.parametrize("cols", [c for c in COLS if c <= 1024])
@pytest.mark.parametrize("rows", [1, 9, 300, 2500])
def test_softmax_persistent_aligned_rows_with_tails(o, rows, cols):
    """16-byte aligned rows whose length is not a multiple of 4 (row stride
    padded to a multiple of 4): the cp.async persistent kernel's tail path,
    and more rows than the persistent grid has warps."""
    w = workloads.make(1, rows=rows, cols=cols, seed=2500 + rows + cols)
    ref = o.softmax(w.arrays["x"])
    pad = (-cols) % 4 + 4
    for kernel in ("async", "plain"):
        assert_close(run_softmax(w.arrays["x"], "persistent", (0, 0, pad), kernel), ref, "f32",
                     f"{kernel} {rows}x{cols}")


@pytest.mark.parametrize("cols", [5, 1000, 4097])
def test_softmax_special_values(o, cols):
    x = workloads.make(1, rows=6, cols=cols, seed=7).arrays["x"].copy()
    x[1, cols // 2] = np.nan                 # NaN row
    x[2, : cols // 2] = -np.inf              # partly -inf
    x[3, :] = -np.inf                        # all -inf: 0/0
    x[4, cols - 1] = np.inf                  # +inf: inf - inf
    ref = o.softmax(x)
    for form in forms_for("softmax", cols):
        got = run_softmax(x, form)
        assert_close(got, ref, "f32", f"{form} special {cols}")
        assert np.isnan(got[[1, 3, 4]]).all() and np.isfinite(got[[0, 2, 5]]).all()
    for layout in ((1, 0, 3), (2, 7, 1)):  # out of phase (rows staggered by the padding)
        for form in forms_for("softmax", cols, in_phase=False):
            got = run_softmax(x, form, layout)
            assert_close(got, ref, "f32", f"{form} special {cols} {layout}")
            assert np.isnan(got[[1, 3, 4]]).all() and np.isfinite(got[[0, 2, 5]]).all()


@pytest.mark.parametrize("cols", [1025, 8193, 40000, 65537, 262145, 409496])
@pytest.mark.parametrize("layout", [(0, 0, 0), (1, 0, 3), (2, 7, 1), (4, 0, 1)])
@pytest.mark.parametrize("pin", [None, "stage"])
def test_softmax_split_staged(o, cols, layout, pin, monkeypatch):
    """The split form with the slices staged in shared memory: rows out of
    phase, rows past the register cluster's reach (262144), and with
    FR_SOFTMAX_SPLIT=stage rows in phase too; 2-8 CTAs a cluster by length."""
    if pin:
        monkeypatch.setenv("FR_SOFTMAX_SPLIT", pin)
    rows = 3 if cols > 100000 else 7
    w = workloads.make(1, rows=rows, cols=cols, seed=2950 + cols)
    ref = o.softmax(w.arrays["x"])
    assert_close(run_softmax(w.arrays["x"], "split", layout), ref, "f32",
                 f"staged split {rows}x{cols} {layout} {pin}")
    assert fr.fr_check_device_error() == 0


@pytest.mark.parametrize("cols", [1025, 40000, 65537])
def test_softmax_split_staged_special_values(o, cols):
    x = workloads.make(1, rows=6, cols=cols, seed=71).arrays["x"].copy()
    x[1, cols // 2] = np.nan                 # NaN row
    x[2, : cols // 2] = -np.inf              # partly -inf (whole slices of it)
    x[3, :] = -np.inf                        # all -inf: 0/0
    x[4, cols - 1] = np.inf                  # +inf: inf - inf
    ref = o.softmax(x)
    for layout in ((0, 0, 0), (1, 0, 3)):
        got = run_softmax(x, "split", layout)
        assert_close(got, ref, "f32", f"staged split special {cols} {layout}")
        assert np.isnan(got[[1, 3, 4]]).all() and np.isfinite(got[[0, 2, 5]]).all()


@pytest.mark.parametrize("cols", [1025, 8193, 40000, 65537, 131073, 262145, 409497, 1000003])
@pytest.mark.parametrize("layout", [(0, 0, 0), (1, 1, 5), (3, 3, 0)])
def test_softmax_split_loop(o, cols, layout, monkeypatch):
    """The split form's streaming cluster (FR_SOFTMAX_SPLIT=loop pins it for
    every row in phase): each CTA of the row's cluster folds its run into
    (m, d), the pairs are exchanged, and the run is read again to write y;
    rows staggered so that every CTA 0 and CTA C-1 has a ragged head or tail."""
    monkeypatch.setenv("FR_SOFTMAX_SPLIT", "loop")
    rows = 3 if cols > 100000 else 7
    w = workloads.make(1, rows=rows, cols=cols, seed=3050 + cols)
    ref = o.softmax(w.arrays["x"])
    assert_close(run_softmax(w.arrays["x"], "split", layout), ref, "f32",
                 f"loop split {rows}x{cols} {layout}")
    assert fr.fr_check_device_error() == 0


@pytest.mark.parametrize("shape", [{"FR_LOOP_K": "1"}, {"FR_LOOP_K": "2"},
                                   {"FR_LOOP_K": "4", "FR_LOOP_C": "4"},
                                   {"FR_LOOP_K": "2", "FR_LOOP_C": "16"},
                                   {"FR_LOOP_K": "4", "FR_LOOP_C": "16"}],
                         ids=["k1", "k2", "k4c4", "k2c16", "k4c16"])
@pytest.mark.parametrize("cols", [8193, 262145])
def test_softmax_split_loop_shapes(o, cols, shape, monkeypatch):
    """Every CTA size (1024, 512 or 256 threads: one, two or four CTAs an SM)
    and every cluster size (4, 8, and 16 CTAs past the portable limit) of the
    streaming cluster."""
    monkeypatch.setenv("FR_SOFTMAX_SPLIT", "loop")
    for k, v in shape.items():
        monkeypatch.setenv(k, v)
    w = workloads.make(1, rows=5, cols=cols, seed=3150 + cols)
    ref = o.softmax(w.arrays["x"])
    assert_close(run_softmax(w.arrays["x"], "split", (1, 1, 5)), ref, "f32",
                 f"loop split 5x{cols} {shape}")


@pytest.mark.parametrize("cols", [1025, 40000, 65537, 409497])
def test_softmax_split_loop_special_values(o, cols, monkeypatch):
    monkeypatch.setenv("FR_SOFTMAX_SPLIT", "loop")
    x = workloads.make(1, rows=6, cols=cols, seed=73).arrays["x"].copy()
    x[1, cols // 2] = np.nan                 # NaN row
    x[2, : cols // 2] = -np.inf              # partly -inf (whole runs of it)
    x[3, :] = -np.inf                        # all -inf: 0/0
    x[4, cols - 1] = np.inf                  # +inf: inf - inf
    ref = o.softmax(x)
    for layout in ((0, 0, 0), (1, 1, 5)):
        got = run_softmax(x, "split", layout)
        assert_close(got, ref, "f32", f"loop split special {cols} {layout}")
        assert np.isnan(got[[1, 3, 4]]).all() and np.isfinite(got[[0, 2, 5]]).all()


@pytest.mark.parametrize("rows,cols", [(200, 262145), (40, 1048577)])
def test_softmax_split_loop_many_rows(o, rows, cols):
    """AUTO on many long rows in phase: many waves of clusters (16 CTAs a row
    at these lengths); the first, middle and last rows against the oracle."""
    w = workloads.make(1, rows=rows, cols=cols, seed=3400 + rows)
    got = run_softmax(w.arrays["x"], "auto")
    assert fr.fr_last_form() == "split"
    for r in (0, 1, rows // 2, rows - 2, rows - 1):
        assert_close(got[r:r + 1], o.softmax(w.arrays["x"][r:r + 1]), "f32",
                     f"loop split row {r} of {rows}x{cols}")
    assert fr.fr_check_device_error() == 0


def test_softmax_split_loop_in_place_and_unpinned(o, monkeypatch):
    """In place through the streaming cluster, and rows in phase past the
    staged cluster's reach take it unpinned."""
    monkeypatch.setenv("FR_SOFTMAX_SPLIT", "loop")
    w = workloads.make(1, rows=5, cols=70001, seed=3300)
    ref = o.softmax(w.arrays["x"])
    t = torch.from_numpy(w.arrays["x"]).cuda()
    fr.fr_softmax(t, form="split", out=t)
    got = t.cpu().numpy()
    assert_close(got, ref, "f32", "loop split in place")
    assert np.abs(got.astype(np.float64).sum(1) - 1).max() < 1e-5
    monkeypatch.delenv("FR_SOFTMAX_SPLIT")
    w = workloads.make(1, rows=2, cols=STAGE_SPLIT_MAX_F32 + 1, seed=3301)
    assert_close(run_softmax(w.arrays["x"], "split"), o.softmax(w.arrays["x"]), "f32",
                 "split past the staged reach")
    assert fr.fr_last_form() == "split"


@pytest.mark.parametrize("cols", [1025, 8193, 32769, 65537, 131071, 262144])
def test_softmax_split_long_rows(o, cols):
    """The cluster split form on few long rows, row by row against the oracle,
    and AUTO on them picks the form fr_auto_form names."""
    w = workloads.make(1, rows=3, cols=cols, seed=2900 + cols)
    ref = o.softmax(w.arrays["x"])
    assert_close(run_softmax(w.arrays["x"], "split"), ref, "f32", f"split 3x{cols}")
    assert_close(run_softmax(w.arrays["x"], "auto"), ref, "f32", f"auto 3x{cols}")
    assert fr.fr_last_form() == fr.fr_auto_form("softmax", 3, cols, "f32", fr.sm_count())


def test_softmax_in_place_and_rows_sum_to_one(o):
    for form, cols in (("persistent", 1000), ("looped", 1000), ("persistent", 5000),
                       ("split", 5000)):
        w = workloads.make(1, rows=65, cols=cols)
        ref = o.softmax(w.arrays["x"])
        t = torch.from_numpy(w.arrays["x"]).cuda()
        fr.fr_softmax(t, form=form, out=t)
        got = t.cpu().numpy()
        assert_close(got, ref, "f32", f"in place {form} {cols}")
        assert np.abs(got.astype(np.float64).sum(1) - 1).max() < 1e-5


# ---------------------------------------------------------------- LayerNorm

def run_layernorm(x_bits, gamma, beta, eps, form, offset=0, kernel=None):
    """kernel pins the looped form's kernel: cluster, ring, ring-bulk (rows
    staged by bulk copies) or scalar."""
    import os
    os.environ.pop("FR_LAYERNORM_STAGE", None)
    if kernel == "ring-bulk":
        kernel = "ring"
        os.environ["FR_LAYERNORM_STAGE"] = "bulk"
    if kernel:
        os.environ["FR_LAYERNORM_KERNEL"] = kernel
    else:
        os.environ.pop("FR_LAYERNORM_KERNEL", None)
    rows, cols = x_bits.shape
    px = place(x_bits, offset)
    py = empty_like_placed(rows, cols, torch.bfloat16, offset)
    g, b = torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda()
    mean = torch.full((rows,), float("nan"), device="cuda")
    rstd = torch.full((rows,), float("nan"), device="cuda")
    try:
        fr.fr_layernorm(px.t, g, b, eps, form=form, out=py.t, mean=mean, rstd=rstd)
    finally:
        os.environ.pop("FR_LAYERNORM_KERNEL", None)
        os.environ.pop("FR_LAYERNORM_STAGE", None)
    torch.cuda.synchronize()
    assert py.canaries_intact(), "layernorm wrote outside y"
    return bf16_to_f32_host(py.t), mean.cpu().numpy(), rstd.cpu().numpy()


@pytest.mark.parametrize("cols", [1, 3, 8, 16, 32, 48, 776, 781, 1000, 1024, 4096, 4112, 8200,
                                  16384, 32768, 40000, 65537, 106496])
@pytest.mark.parametrize("rows", [1, 7, 33, 301])
@pytest.mark.parametrize("offset", [0, 1])
def test_layernorm_forms(o, rows, cols, offset):
    w = workloads.make(2, rows=rows, cols=cols, seed=3000 + rows * 7 + cols)
    eps = float(np.float32(w.params["eps"]))
    ry, rm, rr = o.layernorm(w.arrays["x"], w.arrays["gamma"], w.arrays["beta"], eps)
    vec_ok = offset == 0 and cols % 16 == 0 and cols <= 32768
    rows_ok = offset == 0 and cols % 8 == 0 and cols <= 16384  # row-group kernel
    runs = ([("persistent", None)] if vec_ok or rows_ok else []) + \
        ([("persistent", "cta")] if vec_ok else []) + \
        [("looped", k) for k in ("cluster", "ring", "ring-bulk", "scalar")]
    for form, kernel in runs:
        y, m, r = run_layernorm(w.arrays["x"], w.arrays["gamma"], w.arrays["beta"], eps, form,
                                offset, kernel)
        what = f"{form}/{kernel} {rows}x{cols} offset {offset}"
        assert_close(y, ry, "bf16", f"{what} y")
        assert_close(m, rm, "mean", f"{what} mean")
        assert_close(r, rr, "f32", f"{what} rstd")
    if not vec_ok and not rows_ok:
        with pytest.raises(fr.FRError) as e:
            run_layernorm(w.arrays["x"], w.arrays["gamma"], w.arrays["beta"], eps, "persistent",
                          offset)
        assert e.value.status == 3


@pytest.mark.parametrize("cols", [8, 16, 256, 264, 768, 1000, 1024, 1032, 2048, 3072, 4104, 5120,
                                  8192, 12288, 16384])
@pytest.mark.parametrize("layout", ["chunk", "planar"])
def test_layernorm_row_groups(o, cols, layout):
    """The row-group kernel (gamma/beta in shared memory, chunk by chunk or as
    four float4 planes; a row in the registers of 1, 2, 4 or 8 warps): more
    rows than the persistent grid has groups, ragged chunk counts, a constant
    row and a large-mean row."""
    import os
    os.environ["FR_LAYERNORM_ROWS_GB"] = layout
    try:
        _row_groups(o, cols)
    finally:
        os.environ.pop("FR_LAYERNORM_ROWS_GB", None)


def _row_groups(o, cols):
    for rows in (1, 7, 301, 2500):
        w = workloads.make(2, rows=rows, cols=cols, seed=3900 + rows + cols)
        x = w.arrays["x"].copy()
        if rows >= 7:
            x[2, :] = 0x3F80   # 1.0: var 0
            x[5, :] = 0x4780   # 65536: large mean, var 0
        eps = float(np.float32(w.params["eps"]))
        ry, rm, rr = o.layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps)
        y, m, r = run_layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps, "persistent",
                                kernel="rows")
        what = f"rows kernel {rows}x{cols}"
        assert_close(y, ry, "bf16", f"{what} y")
        assert_close(m, rm, "mean", f"{what} mean")
        assert_close(r, rr, "f32", f"{what} rstd")


@pytest.mark.parametrize("cta", ["256", "512", "128"])
@pytest.mark.parametrize("variant", ["r1a2", "r1a1", "r1a3", "r1a4", "r1a5", "r2a2", "classic"])
@pytest.mark.parametrize("cols", [16384, 32768])
def test_layernorm_cluster_variants(o, variant, cols, cta):
    """The cluster kernels where every thread holds 32 columns (one CTA per
    16384 columns), every ring depth and rows per step, on row counts that
    leave clusters with different numbers of rows (and with none), plus a
    constant row and a row of one repeated large value."""
    import os
    for rows in (1, 5, 77, 301):
        w = workloads.make(2, rows=rows, cols=cols, seed=3500 + rows + cols)
        x = w.arrays["x"].copy()
        if rows >= 5:
            x[1, :] = 0x4060   # 3.5: var 0, y = beta
            x[3, :] = 0x4780   # 65536: large mean, var 0
        eps = float(np.float32(w.params["eps"]))
        ry, rm, rr = o.layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps)
        os.environ["FR_LAYERNORM_CLUSTER"] = variant
        os.environ["FR_LAYERNORM_CTA"] = cta  # largest CTA of the equal-count kernel
        try:
            y, m, r = run_layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps, "looped",
                                    kernel="cluster")
        finally:
            os.environ.pop("FR_LAYERNORM_CLUSTER", None)
            os.environ.pop("FR_LAYERNORM_CTA", None)
        what = f"{variant}/{cta} {rows}x{cols}"
        assert_close(y, ry, "bf16", f"{what} y")
        assert_close(m, rm, "mean", f"{what} mean")
        assert_close(r, rr, "f32", f"{what} rstd")
    assert fr.fr_check_device_error() == 0


@pytest.mark.parametrize("variant", ["r1a2", "r2a2", "r1a3"])
@pytest.mark.parametrize("cols", [2048, 4096, 8192, 65536, 131072])
def test_layernorm_equal_count_shapes(o, variant, cols):
    """The equal-count cluster kernel at every CTA size (64 .. 512 threads) and
    cluster size (1 .. 8 CTAs per row): cols = C x T x 32."""
    import os
    for rows in ((1, 5, 77, 301) if cols <= 8192 else (1, 5, 40)):
        w = workloads.make(2, rows=rows, cols=cols, seed=3700 + rows + cols)
        x = w.arrays["x"].copy()
        if rows >= 5:
            x[2, :] = 0x3F80  # 1.0: var 0
        eps = float(np.float32(w.params["eps"]))
        ry, rm, rr = o.layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps)
        os.environ["FR_LAYERNORM_CLUSTER"] = variant
        try:
            y, m, r = run_layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps, "looped",
                                    kernel="cluster")
        finally:
            os.environ.pop("FR_LAYERNORM_CLUSTER", None)
        what = f"{variant} {rows}x{cols}"
        assert_close(y, ry, "bf16", f"{what} y")
        assert_close(m, rm, "mean", f"{what} mean")
        assert_close(r, rr, "f32", f"{what} rstd")
    assert fr.fr_check_device_error() == 0


@pytest.mark.parametrize("cta", ["256", "128", "512"])
@pytest.mark.parametrize("cols", [3072, 5120, 6144, 7168, 10240, 12288, 14336, 20480, 24576])
def test_layernorm_equal_count_odd_warps(o, cols, cta):
    """The equal-count cluster kernel with CTAs of 3, 5, 6 or 7 warps (the
    CTA-level merge carries counts through a tree over the next power of two):
    every row length a multiple of 1024 that such CTAs tile, with the CTA-size
    cap moving some of them to other (C, T) pairs (12288: 2 x 192 by default,
    4 x 96 under a cap of 128)."""
    import os
    for rows in (1, 5, 77, 301):
        w = workloads.make(2, rows=rows, cols=cols, seed=3800 + rows + cols)
        x = w.arrays["x"].copy()
        if rows >= 5:
            x[2, :] = 0x3F80  # 1.0: var 0
            x[4, :] = 0x4780  # 65536: large mean, var 0
        eps = float(np.float32(w.params["eps"]))
        ry, rm, rr = o.layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps)
        os.environ["FR_LAYERNORM_CTA"] = cta
        try:
            y, m, r = run_layernorm(x, w.arrays["gamma"], w.arrays["beta"], eps, "looped",
                                    kernel="cluster")
        finally:
            os.environ.pop("FR_LAYERNORM_CTA", None)
        what = f"cap {cta} {rows}x{cols}"
        assert_close(y, ry, "bf16", f"{what} y")
        assert_close(m, rm, "mean", f"{what} mean")
        assert_close(r, rr, "f32", f"{what} rstd")
    assert fr.fr_check_device_error() == 0


def test_layernorm_constant_rows(o):
    cols = 4096
    x = np.full((4, cols), 0x4060, np.uint16)  # 3.5 in bf16
    gamma = np.ones(cols, np.float32)
    beta = np.linspace(-1, 1, cols).astype(np.float32)
    eps = float(np.float32(1e-5))
    ry, rm, rr = o.layernorm(x, gamma, beta, eps)
    for form, kernel in (("persistent", None), ("looped", "cluster"), ("looped", "ring"),
                         ("looped", "ring-bulk"), ("looped", "scalar")):
        y, m, r = run_layernorm(x, gamma, beta, eps, form, kernel=kernel)
        assert_close(y, ry, "bf16", f"{form}/{kernel}")
        assert (m == 3.5).all()
        assert_close(r, rr, "f32", f"{form}/{kernel}")


# ---------------------------------------------------------------- cross entropy

# the default point (None: the warp-per-row kernel), its 4-vector point, and
# runnable points of the ring kernel's box: CTA sizes 128 .. 1024, 1 .. 8
# vectors per ring item, 2 .. 8 stages, 1 .. 4 CTAs per SM (the argmax
# kernel always runs at the default point; every runnable point is also
# checked in test_tune_gpu.py)
XENT_KERNELS = [None, (32, 4, 1, 4), (128, 8, 2, 4), (256, 4, 4, 2), (512, 2, 8, 1),
                (1024, 1, 2, 1), (128, 1, 2, 4), (256, 8, 2, 2)]


def run_xent(bits, target, ignore=-100, offset=0, pad=0, kernel=None, argmax=True):
    """kernel: None (the default configuration) or a configuration recorded for
    this shape for the call."""
    rows, cols = bits.shape
    px = place(bits, offset, cols + pad)
    t = torch.from_numpy(target).cuda()
    if kernel is not None:
        fr.fr_xent_set_config(rows, cols, kernel, ld=cols + pad)
    try:
        r = fr.fr_xent(px.t, t, ignore, want_target_logit=True, want_argmax=argmax)
    finally:
        if kernel is not None:
            fr.fr_xent_set_config(rows, cols, None, ld=cols + pad)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def check_xent(got, ref, what):
    assert_close(got["loss"], ref["loss"], "loss", f"{what} loss")
    assert_close(got["mean"][0], ref["mean"], "loss", f"{what} mean")
    assert_bits_equal(got["target_logit"], ref["target_logit"].astype(np.float32),
                      f"{what} target logit")
    if "argmax" in got:
        assert_bits_equal(got["argmax"], ref["argmax"], f"{what} argmax")


@pytest.mark.parametrize("cols", [1, 2, 3, 7, 13, 31, 33, 127, 128, 129, 1000, 4097, 50257])
@pytest.mark.parametrize("rows", [1, 7, 65])
@pytest.mark.parametrize("layout", [(0, 0), (1, 0), (3, 5)], ids=["base0", "base1", "base3_pad5"])
def test_xent(o, rows, cols, layout):
    w = workloads.make(4, rows=rows, cols=cols, seed=4000 + rows * 7 + cols)
    ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
    for kernel in XENT_KERNELS:
        for argmax in ((True, False) if kernel is None else (False,)):
            got = run_xent(w.arrays["logits"], w.arrays["target"], -100, *layout, kernel=kernel,
                           argmax=argmax)
            check_xent(got, ref, f"{kernel} argmax={argmax} {rows}x{cols} {layout}")
    assert fr.fr_check_device_error() == 0


@pytest.mark.parametrize("cols", [1, 2, 3, 5, 7, 13, 33, 128, 129, 1000, 4097, 50257])
@pytest.mark.parametrize("rows", [1, 7, 65])
@pytest.mark.parametrize("layout", [(0, 0), (1, 0), (3, 5)], ids=["base0", "base1", "base3_pad5"])
def test_xent_f32_logits(o, rows, cols, layout):
    """fp32 logits: every output against the oracle on the same fp32 values."""
    w = workloads.make_xent_f32(rows, cols, seed=4500 + rows * 7 + cols)
    ref = o.xent(w.arrays["logits"], w.arrays["target"], -100)
    for argmax in (True, False):
        got = run_xent(w.arrays["logits"], w.arrays["target"], -100, *layout, argmax=argmax)
        check_xent(got, ref, f"f32 argmax={argmax} {rows}x{cols} {layout}")
    assert fr.fr_check_device_error() == 0


def test_xent_f32_ties_nan_and_bad_targets(o):
    rng = np.random.default_rng(6)
    rows, cols = 40, 3001
    x = rng.integers(-3, 4, (rows, cols)).astype(np.float32)  # many ties
    one_up = np.nextafter(np.float32(3.0), np.float32(4.0))
    x[4, 2000] = one_up             # one fp32 step above the ties: the maximum
    x[5, 17] = np.nan
    x[6, [3, 2999]] = np.nan        # two NaNs: first wins
    x[7, :] = -np.inf
    t = rng.integers(0, cols, rows)
    t[[1, 2, 3]] = -100
    t[9] = cols                     # out of range
    ref = o.xent(x, t, -100)
    for offset in (0, 1):
        got = run_xent(x, t, -100, offset=offset)
        check_xent(got, ref, f"f32 ties/nan offset {offset}")
        assert got["argmax"][4] == 2000 and got["argmax"][5] == 17 and got["argmax"][6] == 3
        assert np.isnan(got["loss"][9])
        assert fr.fr_check_device_error() == 1


def test_xent_ties_nan_and_ignore(o):
    rng = np.random.default_rng(5)
    rows, cols = 40, 3001
    vals = rng.integers(-3, 4, (rows, cols)).astype(np.float32)  # many ties
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    bits[5, 17] = 0x7FC0            # NaN
    bits[6, [3, 2999]] = 0x7FC0     # two NaNs: first wins
    bits[7, :] = 0xFF80             # all -inf
    t = rng.integers(0, cols, rows)
    t[[1, 2, 3]] = -100
    ref = o.xent(bits, t, -100)
    for kernel in XENT_KERNELS:
        for offset in (0, 1):
            got = run_xent(bits, t, -100, offset=offset, kernel=kernel, argmax=kernel is None)
            check_xent(got, ref, f"ties/nan {kernel} offset {offset}")
            if kernel is None:
                assert got["argmax"][5] == 17 and got["argmax"][6] == 3
        # every row ignored: mean is 0/0
        allign = np.full(rows, -100, np.int64)
        got = run_xent(bits, allign, kernel=kernel, argmax=kernel is None)
        assert np.isnan(got["mean"][0]) and (got["loss"] == 0).all()
    assert fr.fr_check_device_error() == 0


def test_xent_bad_target_sets_device_error(o):
    w = workloads.make(4, rows=9, cols=777)
    t = w.arrays["target"].copy()
    t[4] = 777          # == cols: out of range
    t[6] = -5           # negative, not ignore_index
    ref = o.xent(w.arrays["logits"], t, -100)
    for kernel in XENT_KERNELS:
        got = run_xent(w.arrays["logits"], t, kernel=kernel, argmax=kernel is None)
        check_xent(got, ref, f"bad target {kernel}")
        assert np.isnan(got["loss"][[4, 6]]).all()
        assert fr.fr_check_device_error() == 1
        assert fr.fr_check_device_error() == 0   # read clears it


# ---------------------------------------------------------------- boundary

def test_error_statuses_on_device():
    x = torch.zeros(4, 40000, device="cuda")  # longer than a CTA holds
    with pytest.raises(fr.FRError) as e:
        fr.fr_softmax(x, form="persistent")
    assert e.value.status == 3
    with pytest.raises(fr.FRError) as e:  # short enough for one warp: no split
        fr.fr_softmax(torch.zeros(4, 1000, device="cuda"), form="split")
    assert e.value.status == 3
    with pytest.raises(fr.FRError) as e:  # out of phase and longer than a staged cluster holds
        n = STAGE_SPLIT_MAX_F32 + 1
        fr.fr_softmax(torch.zeros(2 * n + 1, device="cuda")[1:].view(2, n), form="split",
                      out=torch.empty(2, n, device="cuda"))
    assert e.value.status == 3
    buf = torch.zeros(4 * 2001 + 3, device="cuda")  # x and y rows out of 32-byte phase
    xs = buf[:4 * 2001].view(4, 2001)[:, :2000]
    ys = torch.empty(4 * 2000 + 3, device="cuda")[3:].view(4, 2000)
    fr.fr_softmax(xs, form="split", out=ys)  # a cluster per row, staged
    assert fr.fr_last_form() == "split"
    torch.cuda.synchronize()
    assert torch.allclose(ys, torch.full_like(ys, 1.0 / 2000))
    fr.fr_softmax(xs, form="persistent", out=ys)  # the row in registers, shifted
    assert fr.fr_last_form() == "persistent"
    torch.cuda.synchronize()
    assert torch.allclose(ys, torch.full_like(ys, 1.0 / 2000))
    with pytest.raises(fr.FRError) as e:  # out of phase and past 32768 columns
        big = torch.zeros(2 * 40001, device="cuda")
        fr.fr_softmax(big.view(2, 40001)[:, 1:], form="persistent",
                      out=torch.empty(2, 40000, device="cuda"))
    assert e.value.status == 3
    a = torch.zeros(2, 1 << 20, device="cuda")
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(fr.FRError) as e:
        fr.fr_reduce_relu_add_sum(a, a, 2.0, form="split", workspace=ws)
    assert e.value.status == 5
    lg = torch.zeros(3, 10, dtype=torch.bfloat16, device="cuda")
    tg = torch.zeros(3, dtype=torch.int64, device="cuda")
    with pytest.raises(fr.FRError) as e:
        fr.fr_xent(lg, tg, form="persistent")
    assert e.value.status == 3
    assert fr.fr_last_form() in ("persistent", "looped", "split")


def test_auto_form_choices():
    a = torch.zeros(64, 128, device="cuda")
    fr.fr_reduce_relu_add_sum(a, a)
    assert fr.fr_last_form() == "persistent"
    a = torch.zeros(8, 1 << 20, device="cuda")
    fr.fr_reduce_relu_add_sum(a, a)
    assert fr.fr_last_form() == "split"
    x = torch.zeros(16, 1024, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "persistent"
    x = torch.zeros(1024, 4097, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "persistent"  # one CTA per row, enough rows
    x = torch.zeros(16, 4097, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "persistent"  # up to 8192 columns at any row count
    x = torch.zeros(16, 16384, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "split"  # a cluster per row from 16384 columns
    x = torch.zeros(4, 32769, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "split"
    x = torch.zeros(2, 300000, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "split"  # past the registers' reach: a cluster, staged
    x = torch.zeros(2, STAGE_SPLIT_MAX_F32 + 1, device="cuda")
    fr.fr_softmax(x)
    assert fr.fr_last_form() == "split"  # a cluster streaming its runs twice, at any length
    n = STAGE_SPLIT_MAX_F32 + 1
    fr.fr_softmax(torch.zeros(2 * n + 1, device="cuda")[1:].view(2, n),
                  out=torch.empty(2, n, device="cuda"))
    assert fr.fr_last_form() == "looped"  # out of phase and longer than a staged cluster holds
