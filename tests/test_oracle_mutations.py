"""Each planted mistake in the oracle must fail at least one pin (no GPU).

The mistakes are compiled into throw-away copies of the oracle
(``-DORACLE_PLANT=k``); the shipped oracle has none of them.
"""
import pytest

import oracle
from pins import ALL_PINS

PLANTS = {
    1: "relu by fmax (drops NaN)",
    2: "a + b added in fp64 instead of fp32",
    3: "softmax without the max subtraction",
    4: "online state: old accumulator not rescaled",
    5: "LayerNorm with the unbiased variance",
    6: "LayerNorm with eps outside the square root",
    7: "argmax: last index wins ties",
    8: "log-sum-exp without the max term",
    9: "ignored rows counted in the mean",
    10: "row L2 norm as the mean square instead of the root",
}


@pytest.mark.parametrize("k", sorted(PLANTS), ids=lambda k: f"plant{k}")
def test_planted_mistake_is_caught(k):
    o = oracle.planted(k)
    assert o.planted == k
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {k} ({PLANTS[k]}) passed every pin"
