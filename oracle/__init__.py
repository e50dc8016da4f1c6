"""CPU oracle for the fused row-reduction path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp64); this file
only compiles it with gcc and marshals numpy arrays through ctypes.  Every
output is fp64; callers compare the GPU's fp32/bf16 results against it.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against worked values printed on the pages, closed forms, invariants and
independent library routines; ``tests/test_oracle_mutations.py`` shows that a
planted mistake in each function fails at least one pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(plant: int = 0, out_path: str | None = None, force: bool = False) -> str:
    """Compile the oracle (``plant`` > 0 builds a copy with one planted mistake)."""
    if out_path is None:
        out_path = _LIB if plant == 0 else os.path.join(
            tempfile.gettempdir(), f"liboracle_plant{plant}_{os.getpid()}.so")
    if force or plant or not os.path.exists(out_path) or \
            os.path.getmtime(out_path) < os.path.getmtime(_SRC):
        tmp = out_path + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fno-fast-math",
                        f"-DORACLE_PLANT={plant}", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out_path)
    return out_path


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, f32, f64, vp = ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
        lib.oracle_planted.restype = ctypes.c_int
        lib.oracle_relu_add_sum.argtypes = [vp, vp, i64, i64, i64, i64, f32, vp]
        lib.oracle_row_sumsq.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_row_l2norm.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_softmax.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_md_merge.argtypes = [f64, f64, f64, f64, vp, vp]
        lib.oracle_md_fold.argtypes = [vp, i64, vp, vp]
        lib.oracle_online_attn_row.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_layernorm.argtypes = [vp, i64, i64, i64, vp, vp, f64, vp, vp, vp]
        lib.oracle_xent.argtypes = [vp, i64, i64, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_xent_f32.argtypes = [vp, i64, i64, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp]
        for name in ("oracle_relu_add_sum", "oracle_row_sumsq", "oracle_row_l2norm",
                     "oracle_softmax",
                     "oracle_md_merge", "oracle_md_fold", "oracle_online_attn_row",
                     "oracle_layernorm", "oracle_xent", "oracle_xent_f32"):
            getattr(lib, name).restype = None
        self.lib = lib
        self.planted = lib.oracle_planted()

    # ---- Example 1.1 family -------------------------------------------------
    def relu_add_sum(self, a: np.ndarray, b: np.ndarray, scale: float = 2.0) -> np.ndarray:
        """out[x] = sum_r scale * relu(a[x,r] + b[x,r]); a, b fp32 2-D (row stride honoured)."""
        assert a.dtype == np.float32 and b.dtype == np.float32 and a.shape == b.shape
        assert a.strides[1] == 4 and b.strides[1] == 4
        rows, cols = a.shape
        out = np.empty(rows, dtype=np.float64)
        self.lib.oracle_relu_add_sum(a.ctypes.data, b.ctypes.data, rows, cols,
                                     a.strides[0] // 4, b.strides[0] // 4, scale,
                                     out.ctypes.data)
        return out

    def row_sumsq(self, x: np.ndarray) -> np.ndarray:
        assert x.dtype == np.float32 and x.strides[1] == 4
        out = np.empty(x.shape[0], dtype=np.float64)
        self.lib.oracle_row_sumsq(x.ctypes.data, x.shape[0], x.shape[1], x.strides[0] // 4,
                                  out.ctypes.data)
        return out

    def row_l2norm(self, x: np.ndarray) -> np.ndarray:
        """sqrt(sum_r x[x, r]^2) per row (fp32 squares, fp64 sum and root)."""
        assert x.dtype == np.float32 and x.strides[1] == 4
        out = np.empty(x.shape[0], dtype=np.float64)
        self.lib.oracle_row_l2norm(x.ctypes.data, x.shape[0], x.shape[1], x.strides[0] // 4,
                                   out.ctypes.data)
        return out

    # ---- softmax -----------------------------------------------------------
    def softmax(self, x: np.ndarray) -> np.ndarray:
        assert x.dtype == np.float32 and x.ndim == 2 and x.strides[1] == 4
        rows, cols = x.shape
        y = np.empty((rows, cols), dtype=np.float64)
        self.lib.oracle_softmax(x.ctypes.data, rows, cols, x.strides[0] // 4, y.ctypes.data)
        return y

    def md_merge(self, m1, d1, m2, d2):
        m, d = ctypes.c_double(), ctypes.c_double()
        self.lib.oracle_md_merge(m1, d1, m2, d2, ctypes.byref(m), ctypes.byref(d))
        return m.value, d.value

    def md_fold(self, x) -> tuple[float, float]:
        x = _f64(x)
        m, d = ctypes.c_double(), ctypes.c_double()
        self.lib.oracle_md_fold(x.ctypes.data, x.size, ctypes.byref(m), ctypes.byref(d))
        return m.value, d.value

    def online_attn_row(self, s, V):
        """Returns dict(p, O, m, l, a, alpha, beta) with the per-score trace."""
        s, V = _f64(s), _f64(V)
        n, D = V.shape
        assert s.shape == (n,) and D <= 64
        p, O = np.empty(n), np.empty(D)
        tm, tl, ta, tal, tbe = np.empty(n), np.empty(n), np.empty((n, D)), np.empty(n), \
            np.empty(n)
        self.lib.oracle_online_attn_row(s.ctypes.data, V.ctypes.data, n, D, p.ctypes.data,
                                        O.ctypes.data, tm.ctypes.data, tl.ctypes.data,
                                        ta.ctypes.data, tal.ctypes.data, tbe.ctypes.data)
        return dict(p=p, O=O, m=tm, l=tl, a=ta, alpha=tal, beta=tbe)

    # ---- LayerNorm ---------------------------------------------------------
    def layernorm(self, x_bits: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float):
        """x_bits: uint16 bf16 patterns [rows, cols]. Returns (y, mean, rstd) in fp64."""
        assert x_bits.dtype == np.uint16 and x_bits.strides[1] == 2
        rows, cols = x_bits.shape
        g = np.ascontiguousarray(gamma, dtype=np.float32)
        b = np.ascontiguousarray(beta, dtype=np.float32)
        y = np.empty((rows, cols), dtype=np.float64)
        mean, rstd = np.empty(rows), np.empty(rows)
        self.lib.oracle_layernorm(x_bits.ctypes.data, rows, cols, x_bits.strides[0] // 2,
                                  g.ctypes.data, b.ctypes.data, eps, y.ctypes.data,
                                  mean.ctypes.data, rstd.ctypes.data)
        return y, mean, rstd

    # ---- cross entropy -----------------------------------------------------
    def xent(self, logit_bits: np.ndarray, target: np.ndarray, ignore_index: int = -100):
        """logit_bits: uint16 bf16 patterns or float32 values [rows, cols];
        target int64 [rows]."""
        f32 = logit_bits.dtype == np.float32
        assert (f32 or logit_bits.dtype == np.uint16) and logit_bits.strides[1] == logit_bits.itemsize
        rows, cols = logit_bits.shape
        t = np.ascontiguousarray(target, dtype=np.int64)
        assert t.shape == (rows,)
        loss, lse, tl = np.empty(rows), np.empty(rows), np.empty(rows)
        am = np.empty(rows, dtype=np.int64)
        mean = ctypes.c_double()
        cnt, bad = ctypes.c_int64(), ctypes.c_int64()
        fn = self.lib.oracle_xent_f32 if f32 else self.lib.oracle_xent
        fn(logit_bits.ctypes.data, rows, cols, logit_bits.strides[0] // logit_bits.itemsize,
                             t.ctypes.data, ignore_index, loss.ctypes.data, lse.ctypes.data,
                             tl.ctypes.data, am.ctypes.data, ctypes.byref(mean),
                             ctypes.byref(cnt), ctypes.byref(bad))
        return dict(loss=loss, lse=lse, target_logit=tl, argmax=am, mean=mean.value,
                    n_counted=cnt.value, n_bad=bad.value)


_default: Oracle | None = None


def get() -> Oracle:
    """The shipped oracle (no planted mistake), compiled on first use."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def planted(k: int) -> Oracle:
    """A throw-away copy of the oracle with planted mistake k (tests only)."""
    return Oracle(build(plant=k))
