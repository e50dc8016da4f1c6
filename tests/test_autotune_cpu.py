"""The launch-configuration search of "Stax (4): GPU Codegen and Dynamic
Shapes", section 9.6, checked on the host against what Proposition 9.2 states:
termination within min(|box|, ceil(log(t0 / t_min) / -log(1 - eps)))
acceptances, and a result no single-coordinate neighbour of which is cheaper
by the factor (1 - eps).  The costs are synthetic functions on small boxes, so
t_min and every neighbourhood are found by brute force."""
import itertools
import math

import numpy as np
import pytest

import reduction_pointwise_row_gb300 as fr


def box_points(lo, hi):
    return list(itertools.product(*[range(a, b + 1) for a, b in zip(lo, hi)]))


def neighbours(c, lo, hi):
    for i in range(len(c)):
        for step in (1, -1):
            n = list(c)
            n[i] += step
            if lo[i] <= n[i] <= hi[i]:
                yield tuple(n)


def run(lo, hi, start, eps, t):
    seen = {}

    def cost(c):
        seen[c] = seen.get(c, 0) + 1
        return t(c)

    res, acc, ev = fr.fr_coordinate_descent(lo, hi, start, eps, cost)
    return res, acc, ev, seen


def check_prop_9_2(lo, hi, start, eps, t):
    res, acc, ev, seen = run(lo, hi, start, eps, t)
    pts = box_points(lo, hi)
    tmin = min(t(c) for c in pts)
    bound = min(len(pts), math.ceil(math.log(t(start) / tmin) / -math.log(1 - eps)))
    assert acc <= bound, (acc, bound)
    for n in neighbours(res, lo, hi):  # local optimality at termination
        assert t(n) >= (1 - eps) * t(res), (res, n)
    assert all(v == 1 for v in seen.values()), "a configuration was costed twice"
    assert ev == len(seen) <= len(pts)
    return res, acc


def test_separable_bowl_reaches_the_minimum():
    lo, hi = (7, 0, 1, 0), (10, 3, 3, 4)
    m = (8, 2, 2, 1)

    def t(c):
        return math.prod(1.0 + (a - b) ** 2 for a, b in zip(c, m))

    for start in [(7, 0, 1, 0), (10, 3, 3, 4), (10, 0, 3, 0)]:
        res, _ = check_prop_9_2(lo, hi, start, 0.02, t)
        assert res == m


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("eps", [0.01, 0.05, 0.3])
def test_random_costs_obey_the_bound_and_local_optimality(seed, eps):
    rng = np.random.default_rng(seed)
    lo, hi = (0, 0, 0), (3, 2, 4)
    table = {c: float(rng.uniform(1.0, 100.0)) for c in box_points(lo, hi)}
    start = tuple(int(rng.integers(a, b + 1)) for a, b in zip(lo, hi))
    check_prop_9_2(lo, hi, start, eps, table.__getitem__)


def test_two_basins_end_in_a_local_optimum():
    """A cost that is not unimodal: from the left the search stops in the
    shallow basin, which Proposition 9.2 allows."""
    lo, hi = (0,), (9,)
    vals = [5.0, 3.0, 2.0, 3.0, 6.0, 7.0, 4.0, 1.0, 1.5, 4.0]
    res, _ = check_prop_9_2(lo, hi, (0,), 0.05, lambda c: vals[c[0]])
    assert res == (2,)
    res, _ = check_prop_9_2(lo, hi, (9,), 0.05, lambda c: vals[c[0]])
    assert res == (7,)


def test_eps_stops_small_improvements():
    """A neighbour must be faster than (1 - eps) t to be accepted."""
    vals = [1.0, 0.99, 0.98]
    res, acc, _, _ = run((0,), (2,), (0,), 0.02, lambda c: vals[c[0]])
    assert res == (0,) and acc == 0
    res, acc, _, _ = run((0,), (2,), (0,), 0.005, lambda c: vals[c[0]])
    assert res == (2,) and acc == 2


def test_configurations_that_cannot_run_are_never_chosen():
    lo, hi = (0, 0), (4, 4)

    def t(c):
        if c[0] + c[1] > 5:  # e.g. too much shared memory: cost +inf
            return math.inf
        return 10.0 - c[0] - 0.5 * c[1]

    res, _ = check_prop_9_2(lo, hi, (0, 0), 0.01, t)
    assert math.isfinite(t(res)) and res[0] + res[1] == 5


def test_noisy_measurements_with_eps_above_the_noise_only_improve():
    """Measured t_hat = t (1 + eta), |eta| <= 0.01: with eps > 2 eta / (1 + eta)
    every acceptance lowers the true cost, so the true cost of the result is at
    most the start's (the reading of the noise remark after Proposition 9.2)."""
    eta_max = 0.01
    eps = 2 * eta_max / (1 + eta_max) + 1e-3
    rng = np.random.default_rng(7)
    lo, hi = (0, 0, 0), (3, 3, 3)
    for trial in range(20):
        true = {c: float(rng.uniform(1.0, 2.0)) for c in box_points(lo, hi)}
        eta = {c: float(rng.uniform(-eta_max, eta_max)) for c in true}
        start = (0, 0, 0)
        res, _, _, _ = run(lo, hi, start, eps, lambda c: true[c] * (1 + eta[c]))
        assert true[res] <= true[start]


def test_invalid_arguments():
    t = lambda c: 1.0  # noqa: E731
    with pytest.raises(fr.FRError, match="INVALID_ARG"):
        fr.fr_coordinate_descent((0,), (3,), (4,), 0.1, t)          # start outside the box
    with pytest.raises(fr.FRError, match="INVALID_ARG"):
        fr.fr_coordinate_descent((0,), (3,), (1,), 0.0, t)          # eps out of range
    with pytest.raises(fr.FRError, match="INVALID_ARG"):
        fr.fr_coordinate_descent((0,), (3,), (1,), 0.1, lambda c: math.inf)  # start cannot run
    with pytest.raises(fr.FRError, match="INVALID_ARG"):
        fr.fr_coordinate_descent((0,) * 9, (1,) * 9, (0,) * 9, 0.1, t)  # too many parameters
