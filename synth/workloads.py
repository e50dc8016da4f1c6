"""The five synthetic workloads: shapes, value distributions and seeds.

Each recipe states what one configuration feeds the path; the arrays come from
the counter-based generators in this package, seeded with 20261202 + index.
``rows``/``cols`` overrides keep the distribution but change the shape, which is
how the parity tests build small cases that still span several tiles and a
ragged tail.  No method arithmetic lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import indices, normal_bf16, normal_f32, targets, uniform_f32

SEED_BASE = 20261202
IGNORE_INDEX = -100


@dataclass
class Workload:
    name: str
    op: str
    rows: int
    cols: int
    arrays: dict = field(default_factory=dict)
    params: dict = field(default_factory=dict)


# (op, rows, cols) of each configuration at full size.
FULL_SHAPES = {
    0: ("relu_add_sum", 64, 128),
    1: ("softmax", 32768, 1024),
    2: ("layernorm", 4096, 32768),
    3: ("relu_add_sum", 8, 33554432),
    4: ("xent", 8192, 50257),
}

NAMES = {
    0: "relu_add_sum persistent fp32 [64,128] (Example 1.1)",
    1: "softmax persistent fp32 [32768,1024]",
    2: "layernorm looped Welford bf16 [4096,32768]",
    3: "relu_add_sum split fp32 [8,33554432]",
    4: "log-softmax+cross-entropy bf16 [8192,50257], int64 targets, 5% ignore_index=-100",
}


def seed_of(cfg: int) -> int:
    return SEED_BASE + cfg


def make(cfg: int, rows: int | None = None, cols: int | None = None, nan_variant: bool = False,
         seed: int | None = None, row0: int = 0, global_rows: int | None = None) -> Workload:
    """Host arrays for configuration ``cfg`` (optionally at another shape).

    ``row0``/``global_rows``: rows row0 .. row0 + rows - 1 of the same workload
    with ``global_rows`` rows (a data-parallel shard); the values are exactly
    those rows of the whole array (the generators are counter-based).
    """
    op, R, C = FULL_SHAPES[cfg]
    R = R if rows is None else rows
    C = C if cols is None else cols
    G = row0 + R if global_rows is None else global_rows
    assert 0 <= row0 and row0 + R <= G
    f = row0 * C  # first stream element of the shard
    s = seed_of(cfg) if seed is None else seed
    w = Workload(name=NAMES[cfg], op=op, rows=R, cols=C)
    w.params["row0"], w.params["global_rows"] = row0, G
    if op == "relu_add_sum":
        w.arrays["a"] = uniform_f32((R, C), s, 0, -1.0, 1.0, first=f)
        w.arrays["b"] = uniform_f32((R, C), s, 1, -1.0, 1.0, first=f)
        w.params["scale"] = 2.0
        if nan_variant:
            assert row0 == 0 and G == R, "the NaN variant is not sharded"
            # 4 NaNs at seeded (array, row, col) positions; positions may share rows.
            flat = indices(4, 2 * R * C, s, 2)
            pos = []
            for f in flat.tolist():
                arr, rem = divmod(f, R * C)
                r, c = divmod(rem, C)
                name = "a" if arr == 0 else "b"
                w.arrays[name][r, c] = np.float32("nan")
                pos.append((name, r, c))
            w.params["nan_positions"] = pos
    elif op == "softmax":
        w.arrays["x"] = normal_f32((R, C), s, 0, 0.0, 4.0, first=f)
    elif op == "layernorm":
        w.arrays["x"] = normal_bf16((R, C), s, 0, 0.5, 2.0, first=f)
        w.arrays["gamma"] = normal_f32((C,), s, 1, 1.0, 0.1)
        w.arrays["beta"] = normal_f32((C,), s, 2, 0.0, 0.1)
        w.params["eps"] = 1e-5
    elif op == "xent":
        w.arrays["logits"] = normal_bf16((R, C), s, 0, 0.0, 3.0, first=f)
        n_ignore = int(round(0.05 * G))  # 5 % of the whole batch
        w.arrays["target"] = targets(G, C, n_ignore, IGNORE_INDEX, s, 1)[row0:row0 + R].copy()
        w.params["ignore_index"] = IGNORE_INDEX
    else:
        raise ValueError(op)
    return w


# Example 6.2 of the Stax codegen chapter: x fp32 [64, 16384] reduced to its
# row sums of squares (the listing's wrapper asserts that shape); the pages
# give no value distribution, so x ~ N(0, 1) (torch.randn's).  Seeded with
# 20261202 + 5.
SUMSQ_SHAPE = (64, 16384)


def make_sumsq(rows: int | None = None, cols: int | None = None,
               seed: int | None = None) -> Workload:
    R = SUMSQ_SHAPE[0] if rows is None else rows
    C = SUMSQ_SHAPE[1] if cols is None else cols
    s = SEED_BASE + 5 if seed is None else seed
    w = Workload(name="row sum of squares / L2 norm fp32 (Example 6.2)", op="sumsq", rows=R,
                 cols=C)
    w.arrays["x"] = normal_f32((R, C), s, 0, 0.0, 1.0)
    return w


def make_softmax_bf16(rows: int, cols: int, seed: int | None = None) -> Workload:
    """The softmax workload's distribution, 4 * N(0, 1), rounded to bf16 (bit
    patterns), for the bf16 variant of the softmax row."""
    s = SEED_BASE + 6 if seed is None else seed
    w = Workload(name=f"softmax bf16 [{rows},{cols}]", op="softmax", rows=rows, cols=cols)
    w.arrays["x"] = normal_bf16((rows, cols), s, 0, 0.0, 4.0)
    return w


def make_xent_f32(rows: int, cols: int, seed: int | None = None) -> Workload:
    """The cross-entropy workload's recipe with fp32 logits: 3 * N(0, 1) in
    fp32 (not rounded to bf16), targets uniform with 5 % ignored."""
    s = SEED_BASE + 7 if seed is None else seed
    w = Workload(name=f"cross entropy fp32 logits [{rows},{cols}]", op="xent", rows=rows,
                 cols=cols)
    w.arrays["logits"] = normal_f32((rows, cols), s, 0, 0.0, 3.0)
    w.arrays["target"] = targets(rows, cols, int(round(0.05 * rows)), IGNORE_INDEX, s, 1)
    w.params["ignore_index"] = IGNORE_INDEX
    return w
