"""Seeded synthetic inputs, shared by the CPU oracle and the CUDA path.

Holds none of the method's arithmetic: counter-based SplitMix64 numbers,
Box-Muller normals and value casts only (see ``synth.c``).  Both sides of every
parity check are fed the same host bytes produced here.

The shared library is compiled from ``synth.c`` with gcc on first use (or by
``__graft_entry__.build()``) into this folder.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile libsynth.so with gcc (plain C11, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread", _SRC,
                        "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, u64, dbl, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        lib.synth_uniform_f32.argtypes = [vp, i64, u64, u64, dbl, dbl]
        lib.synth_normal_f32.argtypes = [vp, i64, u64, u64, dbl, dbl]
        lib.synth_normal_bf16.argtypes = [vp, i64, u64, u64, dbl, dbl]
        lib.synth_uniform_f32_at.argtypes = [vp, i64, u64, u64, u64, dbl, dbl]
        lib.synth_normal_f32_at.argtypes = [vp, i64, u64, u64, u64, dbl, dbl]
        lib.synth_normal_bf16_at.argtypes = [vp, i64, u64, u64, u64, dbl, dbl]
        lib.synth_targets.argtypes = [vp, i64, u64, u64, i64, i64, i64]
        lib.synth_targets.restype = ctypes.c_int
        lib.synth_indices.argtypes = [vp, i64, u64, u64, i64]
        lib.synth_u64.argtypes = [u64, u64, u64]
        lib.synth_u64.restype = u64
        for f in (lib.synth_uniform_f32, lib.synth_normal_f32, lib.synth_normal_bf16,
                  lib.synth_uniform_f32_at, lib.synth_normal_f32_at, lib.synth_normal_bf16_at,
                  lib.synth_indices):
            f.restype = None
        _lib = lib
    return _lib


def _empty(shape, dtype, out):
    if out is None:
        return np.empty(shape, dtype=dtype)
    assert out.dtype == dtype and out.flags.c_contiguous and out.shape == tuple(shape)
    return out


def u64(seed: int, stream: int, i: int) -> int:
    """The i-th raw SplitMix64 output of (seed, stream)."""
    return int(_load().synth_u64(seed, stream, i))


def uniform_f32(shape, seed: int, stream: int, lo: float = -1.0, hi: float = 1.0, out=None,
                first: int = 0):
    """fp32 array, each element uniform in [lo, hi) (24 random bits); elements
    first .. of the stream (a slice of a larger array when first > 0)."""
    a = _empty(shape, np.float32, out)
    _load().synth_uniform_f32_at(a.ctypes.data, a.size, seed, stream, first, lo, hi)
    return a


def normal_f32(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0, out=None,
               first: int = 0):
    """fp32 array of mean + std * N(0, 1) (Box-Muller in fp64, cast RNE)."""
    a = _empty(shape, np.float32, out)
    _load().synth_normal_f32_at(a.ctypes.data, a.size, seed, stream, first, mean, std)
    return a


def normal_bf16(shape, seed: int, stream: int, mean: float = 0.0, std: float = 1.0, out=None,
                first: int = 0):
    """uint16 array holding the bf16 bit patterns of mean + std * N(0, 1)."""
    a = _empty(shape, np.uint16, out)
    _load().synth_normal_bf16_at(a.ctypes.data, a.size, seed, stream, first, mean, std)
    return a


def targets(n: int, V: int, n_ignore: int, ignore_index: int, seed: int, stream: int):
    """int64 class indices uniform in [0, V), exactly n_ignore of them set to ignore_index."""
    a = np.empty(n, dtype=np.int64)
    rc = _load().synth_targets(a.ctypes.data, n, seed, stream, V, n_ignore, ignore_index)
    if rc != 0:
        raise ValueError("synth_targets: bad arguments")
    return a


def indices(count: int, bound: int, seed: int, stream: int):
    """count int64 values uniform in [0, bound)."""
    a = np.empty(count, dtype=np.int64)
    _load().synth_indices(a.ctypes.data, count, seed, stream, bound)
    return a


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
