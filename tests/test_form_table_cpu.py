"""The form selection against the committed measurements (no GPU).

profiles/form_table_gb300.md holds, for a grid of shapes, the time of every
reduction form (for LayerNorm, every kernel) measured on GB300 and the form
AUTO took with its own time (bench.py --only form_sweep).  Algorithm 9.1 of
"Stax (4): GPU Codegen and Dynamic Shapes", section 9.6, picks the fastest
measured candidate per shape; here the rules of fr_auto_form must (1) still
name the form AUTO took in that measurement -- a changed rule needs a new
measurement -- and (2) have cost no more than the timing noise over the
fastest candidate: AUTO's time within 6 % + 0.6 us of the fastest (two timings
of one kernel in one sweep differed by up to 6 %, and launch-bound shapes
take 6-8 us give or take 0.6).
"""
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "profiles", "form_table_gb300.md")


def table_rows():
    rows = []
    sms = None
    for line in open(TABLE):
        if line.startswith("device:"):
            sms = int(line.split("(")[1].split()[0])
        if not line.startswith("| ") or line.startswith("| op ") or line.startswith("|---"):
            continue
        f = [c.strip() for c in line.strip().strip("|").split("|")]
        times = {k: float(v) for k, v in (t.split() for t in f[4].split(";"))}
        rows.append(dict(op=f[0], dtype=f[1], rows=int(f[2]), cols=int(f[3]), times=times,
                         fastest=f[5], auto=f[6], auto_us=float(f[7])))
    assert sms and rows
    return sms, rows


OUT_OF_PHASE = "softmax, x out of phase"


def test_table_covers_every_op_and_the_forms():
    _, rows = table_rows()
    ops = {(r["op"], r["dtype"]) for r in rows}
    assert ops == {("relu_add_sum", "f32"), ("softmax", "f32"), ("softmax", "bf16"),
                   (OUT_OF_PHASE, "f32"), (OUT_OF_PHASE, "bf16"), ("layernorm", "bf16")}
    assert len(rows) >= 150


def test_rules_name_the_form_auto_took():
    """fr_auto_form answers for rows in phase; rows out of phase take the
    persistent form up to 32768 columns (fp32 rows past 16384 columns, fewer
    than SMs / 4 or at least 4 x SMs of them: the split form), then the split
    form (a cluster per row, staged) up to 409496 fp32 / 818992 bf16 columns,
    looped beyond."""
    import reduction_pointwise_row_gb300 as fr
    sms, rows = table_rows()
    for r in rows:
        if r["op"] == OUT_OF_PHASE:
            reach = 409496 if r["dtype"] == "f32" else 818992
            few = (r["dtype"] == "f32" and r["cols"] > 16384 and
                   (r["rows"] * 4 < sms or r["rows"] >= 4 * sms))
            want = ("split" if few and r["cols"] <= 32768 else
                    "persistent" if r["cols"] <= 32768 else
                    "split" if r["cols"] <= reach else "looped")
        else:
            want = fr.fr_auto_form(r["op"], r["rows"], r["cols"], r["dtype"], sms)
        assert want == r["auto"], r


def auto_kernel_time(r):
    """The candidate time of what AUTO ran: its form, or for LayerNorm the
    kernel that form launches first (persistent: row groups, else a CTA per
    row; looped: cluster, else ring, else scalar)."""
    t = r["times"]
    if r["op"] != "layernorm":
        return t[r["auto"]]
    order = ("rows", "cta") if r["auto"] == "persistent" else ("cluster", "ring", "scalar")
    return next(t[k] for k in order if k in t)


@pytest.mark.parametrize("tol,abs_us", [(0.06, 0.6)])
def test_auto_is_within_noise_of_the_fastest(tol, abs_us):
    """The form AUTO took against the fastest candidate.  The table holds two
    timings of AUTO's kernel: as a candidate and as AUTO, taken separately;
    the smaller is compared, since on launch-bound shapes (under about 10 us)
    one timing of a kernel has run up to 1.2 us over another of the same
    kernel in the same sweep (fp32 out of phase 304 x 8192: 9.04 and 7.94)."""
    _, rows = table_rows()
    slow = [(r["op"], r["dtype"], r["rows"], r["cols"], r["auto"], auto_kernel_time(r),
             r["auto_us"], r["fastest"], r["times"][r["fastest"]]) for r in rows
            if min(auto_kernel_time(r), r["auto_us"]) > (1 + tol) * r["times"][r["fastest"]] + abs_us]
    assert not slow, slow


def test_auto_times_track_the_candidates():
    """AUTO's separate timing is no slower than its form's timing by more than
    10 % + 0.6 us on all but the launch-bound shapes (fastest under 15 us): a
    slower AUTO would mean it ran something other than the form it names.
    (The other way round is no selection fault: bf16 rows of 65537 columns
    out of phase, 304 of them, timed 33-34 us under AUTO and 39-40 us as the
    looped candidate just before it in three sweeps, the same kernel.)"""
    _, rows = table_rows()
    off = [(r["op"], r["rows"], r["cols"], r["auto_us"], auto_kernel_time(r)) for r in rows
           if r["times"][r["fastest"]] >= 15.0
           and r["auto_us"] - auto_kernel_time(r) > 0.10 * auto_kernel_time(r) + 0.6]
    assert not off, off
