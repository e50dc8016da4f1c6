"""GPU parity of the bf16 softmax (bf16 rows in and out, fp32 arithmetic;
"Stax (4): GPU Codegen and Dynamic Shapes", section 9.5, Listing 9.5) against
the oracle's fp64 softmax of the same (exactly widened) values: every output
within one bf16 step of the nearest bf16 to the oracle's value."""
import numpy as np
import pytest
import torch

import oracle
import reduction_pointwise_row_gb300 as fr
from compare import assert_bf16_within_steps
from gpu_util import empty_like_placed, place
from synth import workloads

pytestmark = pytest.mark.gpu

COLS = [1, 2, 15, 16, 17, 31, 129, 511, 512, 513, 1000, 1024, 1536, 2047, 2048, 2049, 4097,
        8192, 16385, 32768, 32769, 65537, 131073, 262144]
# (offset of x, offset of y, extra row padding), in elements
LAYOUTS = [(0, 0, 0), (3, 3, 7), (0, 5, 0)]


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def widen(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def forms(cols, layout=(0, 0, 0)):
    """persistent: one warp per row up to 2048 columns, one CTA per row up to
    32768 (the row in registers in phase, staged in shared memory out of
    phase)"""
    in_phase = (layout[0] - layout[1]) * 2 % 32 == 0
    persistent = cols <= 32768
    # a cluster of CTAs per row (in phase at any length; out of phase staged,
    # up to 818992 columns)
    split = cols > 2048 and (in_phase or cols <= 818992)
    return (["persistent"] if persistent else []) + (["split"] if split else []) + ["looped", "auto"]


def run(bits, form, layout=(0, 0, 0)):
    rows, cols = bits.shape
    ox, oy, pad = layout
    px = place(bits, ox, cols + pad)
    py = empty_like_placed(rows, cols, torch.bfloat16, oy, cols + pad)
    fr.fr_softmax(px.t, form=form, out=py.t)
    torch.cuda.synchronize()
    assert py.canaries_intact(), "softmax wrote outside y"
    return py.t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [1, 9, 40])
@pytest.mark.parametrize("layout", LAYOUTS, ids=["aligned", "offset_same_phase", "offset_scalar"])
def test_softmax_bf16_forms(o, rows, cols, layout):
    bits = workloads.make_softmax_bf16(rows, cols, seed=6000 + rows * 11 + cols).arrays["x"]
    ref = o.softmax(widen(bits))
    for form in forms(cols, layout):
        assert_bf16_within_steps(run(bits, form, layout), ref, 1, f"{form} {rows}x{cols} {layout}")


# x past y by 1 .. 8 elements (shift 0 at 16 bytes: in 16-byte, not 32-byte
# phase), rows staggered by the padding
OOP_LAYOUTS = [(1, 0, 3), (2, 0, 1), (0, 5, 0), (4, 0, 2), (5, 0, 0), (6, 0, 1), (7, 0, 5),
               (8, 0, 0)]


@pytest.mark.parametrize("cols", [2049, 2055, 4096, 4097, 8192, 16369, 16385, 32768, 32769])
@pytest.mark.parametrize("rows", [1, 9, 40])
@pytest.mark.parametrize("layout", OOP_LAYOUTS)
def test_softmax_bf16_out_of_phase(o, rows, cols, layout):
    bits = workloads.make_softmax_bf16(rows, cols, seed=6500 + rows * 11 + cols).arrays["x"]
    ref = o.softmax(widen(bits))
    for form in forms(cols, layout):
        assert_bf16_within_steps(run(bits, form, layout), ref, 1, f"{form} {rows}x{cols} {layout}")


@pytest.mark.parametrize("kernel", ["stage", "warp"])
@pytest.mark.parametrize("cols", [1025, 1536, 2047, 2048])
@pytest.mark.parametrize("layout", [(1, 0, 3), (0, 5, 0), (8, 0, 0)])
def test_softmax_bf16_out_of_phase_short_rows(o, kernel, cols, layout, monkeypatch):
    """Rows of 1025 .. 2048 columns out of phase: staged in shared memory (the
    default from 32 x SMs rows) or a warp per row, pinned by FR_SOFTMAX_OOP."""
    monkeypatch.setenv("FR_SOFTMAX_OOP", kernel)
    bits = workloads.make_softmax_bf16(40, cols, seed=6700 + cols).arrays["x"]
    ref = o.softmax(widen(bits))
    assert_bf16_within_steps(run(bits, "persistent", layout), ref, 1, f"{kernel} 40x{cols} {layout}")


@pytest.mark.parametrize("cols", [8193, 12000, 16384])
@pytest.mark.parametrize("layout", [(0, 0, 0), (3, 3, 7)])
def test_softmax_bf16_long_rows_staged_in_phase(o, cols, layout, monkeypatch):
    """Rows in phase of 8193 .. 16384 columns through the staged kernel
    (AUTO's persistent kernel there from 8 x SMs rows; pinned here)."""
    monkeypatch.setenv("FR_SOFTMAX_BF16_CTA", "stage")
    bits = workloads.make_softmax_bf16(9, cols, seed=6800 + cols).arrays["x"]
    ref = o.softmax(widen(bits))
    assert_bf16_within_steps(run(bits, "persistent", layout), ref, 1, f"stage 9x{cols} {layout}")


def test_softmax_bf16_many_long_rows_auto(o):
    """8 x 152 rows of 16384 columns in phase: AUTO's persistent form stages
    them; the first and last 32 rows against the oracle."""
    rows, cols = 8 * 152, 16384
    bits = workloads.make_softmax_bf16(rows, cols, seed=6900).arrays["x"]
    got = run(bits, "auto")
    assert fr.fr_last_form() == fr.fr_auto_form("softmax", rows, cols, "bf16", fr.sm_count())
    for sl in (slice(0, 32), slice(rows - 32, rows)):
        assert_bf16_within_steps(got[sl], o.softmax(widen(bits[sl])), 1, f"auto {rows}x{cols}")


@pytest.mark.parametrize("cols", [2049, 65537, 300001, 818992])
@pytest.mark.parametrize("layout", [(0, 0, 0), (1, 0, 3), (0, 5, 0), (8, 0, 0)])
def test_softmax_bf16_split_staged(o, cols, layout, monkeypatch):
    """The split form with bf16 slices staged in shared memory (pinned in
    phase; out of phase and past 262144 columns it is the split form)."""
    monkeypatch.setenv("FR_SOFTMAX_SPLIT", "stage")
    rows = 2 if cols > 100000 else 7
    bits = workloads.make_softmax_bf16(rows, cols, seed=7000 + cols).arrays["x"]
    ref = o.softmax(widen(bits))
    assert_bf16_within_steps(run(bits, "split", layout), ref, 1, f"staged {rows}x{cols} {layout}")


@pytest.mark.parametrize("cols", [2049, 65537, 300001, 818993, 1000003])
@pytest.mark.parametrize("layout", [(0, 0, 0), (3, 3, 7), (16, 16, 0)])
def test_softmax_bf16_split_loop(o, cols, layout, monkeypatch):
    """The split form's streaming cluster on bf16 rows in phase (pinned below
    the staged cluster's reach, unpinned past it)."""
    if cols <= 818992:
        monkeypatch.setenv("FR_SOFTMAX_SPLIT", "loop")
    rows = 2 if cols > 100000 else 7
    bits = workloads.make_softmax_bf16(rows, cols, seed=7100 + cols).arrays["x"]
    ref = o.softmax(widen(bits))
    assert_bf16_within_steps(run(bits, "split", layout), ref, 1, f"loop {rows}x{cols} {layout}")
    assert fr.fr_check_device_error() == 0


def test_softmax_bf16_split_loop_many_rows(o):
    """AUTO on 320 bf16 rows of 300001 in phase (many waves of clusters);
    the first, middle and last rows against the oracle."""
    rows, cols = 320, 300001
    bits = workloads.make_softmax_bf16(rows, cols, seed=7300).arrays["x"]
    got = run(bits, "auto")
    assert fr.fr_last_form() == "split"
    for r in (0, 1, rows // 2, rows - 2, rows - 1):
        assert_bf16_within_steps(got[r:r + 1], o.softmax(widen(bits[r:r + 1])), 1,
                                 f"loop row {r} of {rows}x{cols}")


@pytest.mark.parametrize("cols", [4097, 300001])
def test_softmax_bf16_split_loop_special_values(o, cols, monkeypatch):
    monkeypatch.setenv("FR_SOFTMAX_SPLIT", "loop")
    bits = workloads.make_softmax_bf16(6, cols, seed=62).arrays["x"].copy()
    bits[1, cols // 2] = 0x7FC0               # NaN row
    bits[2, : cols // 2] = 0xFF80             # partly -inf
    bits[3, :] = 0xFF80                       # all -inf: 0/0
    bits[4, cols - 1] = 0x7F80                # +inf: inf - inf
    ref = o.softmax(widen(bits))
    for layout in ((0, 0, 0), (3, 3, 7)):
        assert_bf16_within_steps(run(bits, "split", layout), ref, 1, f"loop special {cols} {layout}")


@pytest.mark.parametrize("cols", [7, 1000, 2048, 4097, 20000])
def test_softmax_bf16_special_values(o, cols):
    bits = workloads.make_softmax_bf16(6, cols, seed=61).arrays["x"].copy()
    bits[1, cols // 2] = 0x7FC0               # NaN row
    bits[2, : cols // 2] = 0xFF80             # partly -inf
    bits[3, :] = 0xFF80                       # all -inf: 0/0
    bits[4, cols - 1] = 0x7F80                # +inf: inf - inf
    ref = o.softmax(widen(bits))
    for layout in ((0, 0, 0), (1, 0, 3), (0, 5, 0)):
        for form in forms(cols, layout):
            got = run(bits, form, layout)
            assert_bf16_within_steps(got, ref, 1, f"{form} special {cols} {layout}")


def test_softmax_bf16_in_place_and_full_headline_shape(o):
    """In place (x and y the same buffer), and the softmax workload's shape
    [32768, 1024] in bf16 checked on sampled rows."""
    bits = workloads.make_softmax_bf16(65, 1000).arrays["x"]
    ref = o.softmax(widen(bits))
    for form in ("persistent", "looped"):
        t = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        fr.fr_softmax(t, form=form, out=t)
        got = t.view(torch.int16).cpu().numpy().view(np.uint16)
        assert_bf16_within_steps(got, ref, 1, f"in place {form}")
    full = workloads.make_softmax_bf16(32768, 1024).arrays["x"]
    x = torch.from_numpy(full.view(np.int16)).cuda().view(torch.bfloat16)
    y = fr.fr_softmax(x)
    assert fr.fr_last_form() == "persistent"
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    rows = np.random.default_rng(3).choice(32768, 64, replace=False)
    rows.sort()
    assert_bf16_within_steps(got[rows], o.softmax(widen(full[rows])), 1, "sampled rows")


@pytest.mark.parametrize("cta", ["128", "256", "512"])
def test_softmax_bf16_looped_every_cta_size(o, cta, monkeypatch):
    """The looped form at each CTA size its rule can pick (FR_SOFTMAX_LOOP pins
    it), rows in and out of phase, short and long."""
    monkeypatch.setenv("FR_SOFTMAX_LOOP", cta)
    for rows, cols, layout in ((700, 4097, (0, 0, 0)), (9, 65537, (3, 3, 7)), (40, 3000, (0, 5, 0)),
                               (5, 17, (0, 0, 0))):
        bits = workloads.make_softmax_bf16(rows, cols, seed=6500 + cols).arrays["x"]
        ref = o.softmax(widen(bits))
        assert_bf16_within_steps(run(bits, "looped", layout), ref, 1,
                                 f"looped T={cta} {rows}x{cols} {layout}")
