"""Algorithmic bytes: what each op must move between HBM and the SMs.

The count is the method's own: every input element read once, every output
element written once (the 2N bound of fused softmax, "Stax (4): GPU Codegen and
Dynamic Shapes", section 9.5), plus the small per-row vectors.  Achieved
bandwidth = these bytes / kernel time.

``naive_softmax_elements`` restates the five-kernel accounting of "CMU 15-779
Lecture 8", section 3 (amax, subtract, exp, sum, divide each reading and
writing HBM) so the tests can pin this model against the element counts that
page prints for a 1823 x 781 input.
"""
from __future__ import annotations


def naive_softmax_elements(rows: int, cols: int) -> tuple[int, int]:
    """(elements read, elements written) of the unfused 5-kernel softmax."""
    mn, m = rows * cols, rows
    reads = mn + (mn + m) + mn + mn + (mn + m)    # amax, sub, exp, sum, div
    writes = m + mn + mn + m + mn
    return reads, writes


def fused_softmax_elements(rows: int, cols: int) -> tuple[int, int]:
    return rows * cols, rows * cols


def algorithmic_bytes(op: str, rows: int, cols: int, **kw) -> int:
    if op == "relu_add_sum":          # a, b fp32 in; out fp32 [rows]
        return 2 * rows * cols * 4 + rows * 4
    if op == "relu_add_sum_bf16":     # a, b bf16 in; out fp32 [rows]
        return 2 * rows * cols * 2 + rows * 4
    if op == "sumsq":                 # x fp32 in; out fp32 [rows]
        return rows * cols * 4 + rows * 4
    if op == "softmax":               # x fp32 in; y fp32 out
        return 2 * rows * cols * 4
    if op == "softmax_offset":        # fp32 softmax, x and y out of phase: same bytes
        return 2 * rows * cols * 4
    if op == "softmax_bf16":          # x bf16 in; y bf16 out
        return 2 * rows * cols * 2
    if op == "softmax_bf16_offset":   # bf16 softmax, x and y out of phase: same bytes
        return 2 * rows * cols * 2
    if op == "layernorm":             # x bf16 in, y bf16 out, gamma/beta fp32, mean/rstd fp32
        return 2 * rows * cols * 2 + 2 * cols * 4 + 2 * rows * 4
    if op == "xent":                  # logits bf16, targets int64, loss fp32 [rows], mean fp32
        return rows * cols * 2 + rows * 8 + rows * 4 + 4
    if op == "xent_f32":              # the same with fp32 logits
        return rows * cols * 4 + rows * 8 + rows * 4 + 4
    raise ValueError(op)
