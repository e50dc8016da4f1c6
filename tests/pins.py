"""Pins of the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with what the pages or the mathematics fix: worked values the
pages print (``tests/golden/``), closed forms, exact rationals on dyadic inputs,
invariants (Proposition 9.1 of "Stax (4): GPU Codegen and Dynamic Shapes"), and
independent library routines (scipy, torch CPU in fp64).  The same list is run
against copies of the oracle with a planted mistake to show each mistake is
caught.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol=0.0):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    ok = np.isclose(a, b, rtol=rtol, atol=atol, equal_nan=True)
    if not ok.all():
        bad = np.argwhere(~ok)[:5].tolist()
        raise AssertionError(f"{int((~ok).sum())} mismatches, first at {bad}: "
                             f"{a[~ok][:5].tolist()} vs {b[~ok][:5].tolist()}")


def _bf16_bits(vals):
    """fp32 values that are exactly bf16 -> their bit patterns."""
    f = np.asarray(vals, dtype=np.float32)
    u = f.view(np.uint32)
    assert (u & 0xFFFF).max(initial=0) == 0, "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Example 1.1: out[x] = sum_r 2 * relu(a + b)
# ---------------------------------------------------------------------------

def pin_ras_dyadic_exact(o):
    """Inputs k/64 with |k| <= 64: every partial sum is exact, so the oracle must
    equal the exact rational sum bit for bit (Example 1.1 shape and a long row)."""
    rng = _rng(1)
    for rows, cols in ((64, 128), (3, 4099)):
        ka = rng.integers(-64, 65, size=(rows, cols))
        kb = rng.integers(-64, 65, size=(rows, cols))
        a = (ka / 64).astype(np.float32)
        b = (kb / 64).astype(np.float32)
        got = o.relu_add_sum(a, b, 2.0)
        for x in range(rows):
            exact = Fraction(int(np.maximum(ka[x] + kb[x], 0).sum()) * 2, 64)
            assert got[x] == float(exact), (x, got[x], exact)


def pin_ras_constant_row(o):
    """a + b == c everywhere gives out = 2 * cols * relu(c)."""
    a = np.full((4, 128), 0.25, np.float32)
    b = np.full((4, 128), 0.5, np.float32)
    assert (o.relu_add_sum(a, b, 2.0) == 2 * 128 * 0.75).all()
    assert (o.relu_add_sum(-a, -b, 2.0) == 0.0).all()


def pin_ras_nan_propagates(o):
    """relu keeps NaN (PropagateNan.ALL): exactly the rows holding a NaN are NaN
    and every other row is bit-identical to the NaN-free result."""
    rng = _rng(2)
    a = rng.uniform(-1, 1, (16, 200)).astype(np.float32)
    b = rng.uniform(-1, 1, (16, 200)).astype(np.float32)
    clean = o.relu_add_sum(a, b, 2.0)
    a2 = a.copy()
    b2 = b.copy()
    a2[3, 7] = np.nan
    b2[11, 0] = np.nan
    b2[3, 199] = np.nan
    got = o.relu_add_sum(a2, b2, 2.0)
    nan_rows = set(np.flatnonzero(np.isnan(got)).tolist())
    assert nan_rows == {3, 11}, nan_rows
    keep = [i for i in range(16) if i not in nan_rows]
    assert (got[keep] == clean[keep]).all()
    # a NaN whose partner would make a + b negative must still give NaN
    one = o.relu_add_sum(np.array([[np.nan]], np.float32), np.array([[-5.0]], np.float32))
    assert np.isnan(one[0])


def pin_ras_add_in_fp32(o):
    """Listing 9.1 adds the loaded fp32 values in fp32: 1 + 2^-30 rounds to 1."""
    a = np.array([[1.0]], np.float32)
    b = np.array([[2.0 ** -30]], np.float32)
    assert o.relu_add_sum(a, b, 2.0)[0] == 2.0


def pin_ras_infinities(o):
    f = np.float32
    r = o.relu_add_sum(np.array([[np.inf], [-np.inf], [np.inf]], f),
                       np.array([[1.0], [1.0], [-np.inf]], f), 2.0)
    assert r[0] == np.inf and r[1] == 0.0 and np.isnan(r[2])


def pin_ras_scale_sign(o):
    """scale = -1 negates the scale = 1 result exactly; scale = 4 quadruples it."""
    rng = _rng(3)
    a = rng.uniform(-1, 1, (5, 300)).astype(np.float32)
    b = rng.uniform(-1, 1, (5, 300)).astype(np.float32)
    p = o.relu_add_sum(a, b, 1.0)
    assert (o.relu_add_sum(a, b, -1.0) == -p).all()
    assert (o.relu_add_sum(a, b, 4.0) == 4.0 * p).all()


def pin_ras_row_stride(o):
    """A padded row stride reads only the first cols entries of each row."""
    rng = _rng(4)
    big_a = rng.uniform(-1, 1, (6, 40)).astype(np.float32)
    big_b = rng.uniform(-1, 1, (6, 40)).astype(np.float32)
    got = o.relu_add_sum(big_a[:, :33], big_b[:, :33], 2.0)
    ref = o.relu_add_sum(np.ascontiguousarray(big_a[:, :33]),
                         np.ascontiguousarray(big_b[:, :33]), 2.0)
    assert (got == ref).all()


def pin_sumsq_dyadic(o):
    """Sum of squares (Example 6.2) and the row L2 norm: exact on k/64 inputs;
    the row [3, 4] has norm 5."""
    rng = _rng(5)
    k = rng.integers(-64, 65, size=(4, 1000))
    x = (k / 64).astype(np.float32)
    got = o.row_sumsq(x)
    for i in range(4):
        assert got[i] == float(Fraction(int((k[i] ** 2).sum()), 4096))
    assert math.sqrt(o.row_sumsq(np.array([[3.0, 4.0]], np.float32))[0]) == 5.0


def pin_l2norm_pythagorean_rows(o):
    """Row L2 norm (Lecture 8, exercise 1) on integer rows whose norm is an
    integer: [3, 4] -> 5, [5, 12] -> 13, [1, 2, 2] -> 3, [2, 3, 6] -> 7,
    [1, 4, 8] -> 9; a one-hot row gives |value|; a power-of-two scale c gives
    |c| times the norm exactly."""
    rows = [([3, 4], 5), ([5, 12], 13), ([1, 2, 2], 3), ([2, 3, 6], 7), ([1, 4, 8], 9),
            ([0, 0, 0, -7.5, 0], 7.5)]
    x = np.zeros((len(rows), 5), np.float32)
    for i, (vals, _) in enumerate(rows):
        x[i, :len(vals)] = vals
    got = o.row_l2norm(x)
    assert got.tolist() == [float(n) for _, n in rows]
    rng = _rng(6)
    y = rng.standard_normal((3, 777)).astype(np.float32)
    base = o.row_l2norm(y)
    assert (o.row_l2norm(y * np.float32(-0.25)) == 0.25 * base).all()
    assert (o.row_l2norm(y * np.float32(8.0)) == 8.0 * base).all()


# ---------------------------------------------------------------------------
# softmax and the (m, d) monoid
# ---------------------------------------------------------------------------

def pin_softmax_hand_example(o):
    g = _golden("online_softmax_hand_example.json")
    y = o.softmax(np.array([g["scores"]], np.float32))[0]
    _close(y, g["p"], rtol=0, atol=g["tolerance_abs"])


def pin_softmax_rows_sum_to_one(o):
    x = (4 * _rng(6).standard_normal((50, 1000))).astype(np.float32)
    y = o.softmax(x)
    assert np.abs(y.sum(axis=1) - 1.0).max() < 1e-12
    assert (y > 0).all()


def pin_softmax_constant_row(o):
    """A constant row of length 2^k gives exactly 2^-k everywhere."""
    y = o.softmax(np.full((3, 1024), -7.25, np.float32))
    assert (y == 1.0 / 1024).all()


def pin_softmax_two_valued_closed_form(o):
    """n0 zeros and n1 entries equal to c: y = 1/(n0 + n1 e^c), e^c/(n0 + n1 e^c)."""
    for c, n0, n1 in ((3.0, 5, 2), (-2.5, 1, 7), (1000.0, 3, 1)):
        x = np.array([[0.0] * n0 + [c] * n1], np.float32)
        y = o.softmax(x)[0]
        if c > 700:  # e^c overflows fp64: the limit form
            want0, want1 = 0.0, 1.0 / n1
        else:
            den = n0 + n1 * math.exp(c)
            want0, want1 = 1.0 / den, math.exp(c) / den
        _close(y[:n0], [want0] * n0, rtol=1e-14, atol=1e-300)
        _close(y[n0:], [want1] * n1, rtol=1e-14)


def pin_softmax_one_hot(o):
    n = 781
    x = np.zeros((1, n), np.float32)
    x[0, -1] = 100.0
    y = o.softmax(x)[0]
    den = 1.0 + (n - 1) * math.exp(-100.0)
    _close(y[-1], 1.0 / den, rtol=1e-15)
    _close(y[:-1], np.full(n - 1, math.exp(-100.0) / den), rtol=1e-13)


def pin_softmax_shift_invariance(o):
    k = _rng(7).integers(-64, 65, size=(4, 333))
    x = (k / 16).astype(np.float32)
    _close(o.softmax(x), o.softmax(x + np.float32(8.0)), rtol=1e-12)


def pin_softmax_vs_scipy(o):
    from scipy.special import softmax as sp_softmax
    x = (4 * _rng(8).standard_normal((20, 777))).astype(np.float32)
    _close(o.softmax(x), sp_softmax(x.astype(np.float64), axis=1), rtol=1e-12)


def pin_softmax_nan_row(o):
    x = _rng(9).standard_normal((4, 64)).astype(np.float32)
    x[2, 5] = np.nan
    y = o.softmax(x)
    assert np.isnan(y[2]).all() and np.isfinite(y[[0, 1, 3]]).all()


def pin_md_fold_is_max_and_sum(o):
    """Folding (x, 1) elements with (+) gives (max, sum exp(x - max))."""
    x = 3 * _rng(10).standard_normal(513)
    m, d = o.md_fold(x)
    mx = float(x.max())
    assert m == mx
    _close(d, math.fsum(math.exp(v - mx) for v in x), rtol=1e-13)


def pin_md_any_order_any_segmentation(o):
    """Proposition 9.1: any segmentation and merge order gives the same (m, d)."""
    rng = _rng(11)
    x = 5 * rng.standard_normal(1000)
    m0, d0 = o.md_fold(x)
    for trial in range(20):
        cuts = np.sort(rng.choice(np.arange(1, 1000), size=rng.integers(1, 30), replace=False))
        segs = [o.md_fold(s) for s in np.split(rng.permutation(x), cuts)]
        order = rng.permutation(len(segs))
        m, d = -math.inf, 0.0
        for i in order:
            m, d = o.md_merge(m, d, *segs[i])
        assert m == m0
        _close(d, d0, rtol=1e-12)


def pin_md_identity(o):
    assert o.md_merge(-math.inf, 0.0, 1.5, 1.0) == (1.5, 1.0)
    assert o.md_merge(2.0, 3.0, -math.inf, 0.0) == (2.0, 3.0)
    assert o.md_merge(-math.inf, 0.0, -math.inf, 0.0) == (-math.inf, 0.0)
    m, d = o.md_merge(1.0, 1.0, 1.0, 1.0)
    assert (m, d) == (1.0, 2.0)


def pin_online_hand_example(o):
    """The worked row of hello-gpu section 12.1 and the frames of Figure 12.3."""
    g = _golden("online_softmax_hand_example.json")
    r = o.online_attn_row(g["scores"], g["values"])
    tol = g["tolerance_abs"]
    _close(r["p"], g["p"], rtol=0, atol=tol)
    _close(r["O"], g["O"], rtol=0, atol=tol)
    for j, fr in enumerate(g["frames"]):
        _close(r["m"][j], fr["m"], 0, tol)
        _close(r["l"][j], fr["l"], 0, tol)
        _close(r["alpha"][j], fr["alpha"], 0, tol)
        _close(r["beta"][j], fr["beta"], 0, tol)
        _close(r["a"][j], fr["a"], 0, tol)


def pin_online_equals_materialised(o):
    """O = sum_j softmax(s)_j V_j (scipy softmax), in any key order (exercise 2)."""
    from scipy.special import softmax as sp_softmax
    rng = _rng(12)
    s = 2 * rng.standard_normal(37)
    V = rng.standard_normal((37, 5))
    r = o.online_attn_row(s, V)
    _close(r["O"], sp_softmax(s) @ V, rtol=1e-12)
    _close(r["p"], sp_softmax(s), rtol=1e-12)
    perm = rng.permutation(37)
    r2 = o.online_attn_row(s[perm], V[perm])
    _close(r2["O"], r["O"], rtol=1e-12)


# ---------------------------------------------------------------------------
# LayerNorm
# ---------------------------------------------------------------------------

def pin_ln_integer_row(o):
    """x = [1, 2, 3, 4]: mean 5/2 and biased variance 5/4 exactly."""
    eps = 1e-5
    x = _bf16_bits([[1.0, 2.0, 3.0, 4.0]])
    y, mean, rstd = o.layernorm(x, np.ones(4, np.float32), np.zeros(4, np.float32), eps)
    assert mean[0] == 2.5
    _close(rstd[0], 1.0 / math.sqrt(1.25 + eps), rtol=1e-15)
    _close(y[0], (np.array([1, 2, 3, 4]) - 2.5) / math.sqrt(1.25 + eps), rtol=1e-15)


def pin_ln_constant_row(o):
    """A constant row has zero variance: rstd = 1/sqrt(eps) and y = beta."""
    eps = 1e-5
    x = _bf16_bits(np.full((2, 300), 3.5))
    beta = _rng(13).standard_normal(300).astype(np.float32)
    gamma = _rng(14).standard_normal(300).astype(np.float32)
    y, mean, rstd = o.layernorm(x, gamma, beta, eps)
    assert (mean == 3.5).all()
    _close(rstd, [1.0 / math.sqrt(eps)] * 2, rtol=1e-15)
    assert (y == beta.astype(np.float64)).all()


def pin_ln_normalised_moments(o):
    """gamma = 1, beta = 0: y has mean 0 and variance var / (var + eps)."""
    eps = 1e-2
    vals = (0.5 + 2 * _rng(15).standard_normal((3, 4096))).astype(np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y, mean, rstd = o.layernorm(bits, np.ones(4096, np.float32), np.zeros(4096, np.float32), eps)
    var = xv.var(axis=1)
    assert np.abs(y.mean(axis=1)).max() < 1e-12
    _close(y.var(axis=1), var / (var + eps), rtol=1e-12)
    _close(mean, xv.mean(axis=1), rtol=1e-13)


def pin_ln_vs_torch(o):
    import torch
    rng = _rng(16)
    vals = (0.5 + 2 * rng.standard_normal((8, 1000))).astype(np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gamma = (1 + 0.1 * rng.standard_normal(1000)).astype(np.float32)
    beta = (0.1 * rng.standard_normal(1000)).astype(np.float32)
    eps = 1e-5
    y, mean, rstd = o.layernorm(bits, gamma, beta, eps)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(xv), (1000,),
                                         torch.from_numpy(gamma.astype(np.float64)),
                                         torch.from_numpy(beta.astype(np.float64)), eps)
    _close(y, ref.numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# cross entropy
# ---------------------------------------------------------------------------

def pin_xent_uniform_row(o):
    """Equal logits: loss = ln V for any level c (V = 50257: 10.8249...)."""
    V = 50257
    x = _bf16_bits(np.full((2, V), 1.5))
    r = o.xent(x, np.array([7, V - 1]))
    _close(r["loss"], [math.log(V)] * 2, rtol=1e-13)
    assert abs(math.log(V) - 10.824905) < 1e-6


def pin_xent_vs_torch(o):
    """torch.nn.functional.cross_entropy in fp64, reduction none and mean."""
    import torch
    rng = _rng(17)
    rows, V = 64, 1000
    vals = (3 * rng.standard_normal((rows, V))).astype(np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    t = rng.integers(0, V, rows)
    t[[3, 10, 11, 40]] = -100
    r = o.xent(bits, t, -100)
    tx, tt = torch.from_numpy(xv), torch.from_numpy(t)
    none = torch.nn.functional.cross_entropy(tx, tt, ignore_index=-100, reduction="none")
    mean = torch.nn.functional.cross_entropy(tx, tt, ignore_index=-100, reduction="mean")
    _close(r["loss"], none.numpy(), rtol=1e-12, atol=1e-13)
    _close(r["mean"], float(mean), rtol=1e-12)
    assert r["n_counted"] == rows - 4
    _close(r["lse"], torch.logsumexp(tx, dim=1).numpy(), rtol=1e-13)


def pin_xent_brute_force_lse(o):
    """V <= 20 and small logits: log(sum e^x) taken directly, no max shift."""
    rng = _rng(18)
    for V in (1, 2, 3, 7, 20):
        k = rng.integers(-16, 17, size=(5, V))
        x = _bf16_bits(k / 4)
        t = rng.integers(0, V, 5)
        r = o.xent(x, t)
        for i in range(5):
            lse = math.log(math.fsum(math.exp(v / 4) for v in k[i]))
            _close(r["lse"][i], lse, rtol=1e-14)
            _close(r["loss"][i], lse - k[i, t[i]] / 4, rtol=1e-13, atol=1e-15)


def pin_xent_margin(o):
    """A target logit 100 above the rest gives a loss of about (V-1) e^-100."""
    x = np.zeros((1, 50), np.float32)
    x[0, 17] = 100.0
    r = o.xent(_bf16_bits(x), np.array([17]))
    assert 0.0 <= r["loss"][0] < 1e-40


def pin_xent_ignore_and_mean(o):
    """Ignored rows have loss 0 and leave the mean's denominator; all ignored -> NaN."""
    x = _bf16_bits([[0.0, 1.0, 2.0], [5.0, 0.0, 0.0], [1.0, 1.0, 1.0]])
    r = o.xent(x, np.array([2, -100, 0]))
    l0 = math.log(1 + math.e + math.e ** 2) - 2.0
    l2 = math.log(3.0)
    _close(r["loss"], [l0, 0.0, l2], rtol=1e-14)
    _close(r["mean"], (l0 + l2) / 2, rtol=1e-14)
    assert r["n_counted"] == 2 and r["target_logit"][1] == 0.0 and r["target_logit"][0] == 2.0
    assert math.isnan(o.xent(x, np.array([-100, -100, -100]))["mean"])


def pin_xent_argmax_ties_and_nan(o):
    x = _bf16_bits([[1.0, 3.0, 3.0, 2.0], [-1.0, np.nan, 5.0, np.nan], [0.0, 0.0, 0.0, 0.0]])
    r = o.xent(x, np.array([0, 0, 0]))
    assert r["argmax"].tolist() == [1, 1, 0]
    assert np.isnan(r["loss"][1]) and np.isfinite(r["loss"][[0, 2]]).all()


def pin_xent_bad_target(o):
    x = _bf16_bits([[0.0, 1.0], [0.0, 1.0]])
    r = o.xent(x, np.array([2, 1]))
    assert np.isnan(r["loss"][0]) and r["n_bad"] == 1 and np.isnan(r["mean"])


def pin_xent_shift_invariance(o):
    k = _rng(19).integers(-32, 33, size=(6, 257))
    t = _rng(20).integers(0, 257, 6)
    a = o.xent(_bf16_bits(k / 8), t)
    b = o.xent(_bf16_bits(k / 8 + 2.0), t)
    _close(a["loss"], b["loss"], rtol=1e-12)


def pin_xent_f32_vs_torch(o):
    """fp32 logits (not bf16-representable): torch cross_entropy in fp64 on the
    same values, reduction none and mean, and its logsumexp."""
    import torch
    rng = _rng(21)
    rows, V = 48, 777
    x = (3 * rng.standard_normal((rows, V))).astype(np.float32)
    t = rng.integers(0, V, rows)
    t[[0, 5]] = -100
    r = o.xent(x, t, -100)
    tx, tt = torch.from_numpy(x.astype(np.float64)), torch.from_numpy(t)
    none = torch.nn.functional.cross_entropy(tx, tt, ignore_index=-100, reduction="none")
    mean = torch.nn.functional.cross_entropy(tx, tt, ignore_index=-100, reduction="mean")
    _close(r["loss"], none.numpy(), rtol=1e-12, atol=1e-13)
    _close(r["mean"], float(mean), rtol=1e-12)
    _close(r["lse"], torch.logsumexp(tx, dim=1).numpy(), rtol=1e-13)
    _close(r["target_logit"][t >= 0], x[np.arange(rows), t][t >= 0].astype(np.float64), rtol=0)


def pin_xent_f32_keeps_every_bit(o):
    """fp32 logits are read as fp32: values one fp32 step apart (equal in bf16)
    keep their order for argmax and their difference in the loss; bf16 values
    given as fp32 give the bf16 results exactly."""
    one_up = np.nextafter(np.float32(1.0), np.float32(2.0))
    x = np.array([[1.0, one_up, 0.5]], np.float32)
    r = o.xent(x, np.array([0]))
    assert r["argmax"][0] == 1
    e = [math.exp(float(v)) for v in x[0]]
    _close(r["loss"][0], math.log(math.fsum(e)) - 1.0, rtol=1e-14)
    bits = _bf16_bits((_rng(22).integers(-64, 65, size=(4, 333)) / 16))
    as_f32 = (bits.astype(np.uint32) << 16).view(np.float32)
    t = np.array([1, 2, -100, 332])
    a, b = o.xent(bits, t), o.xent(as_f32, t)
    for k in ("loss", "lse", "target_logit", "argmax"):
        assert (np.asarray(a[k]) == np.asarray(b[k])).all(), k
    assert a["mean"] == b["mean"]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
