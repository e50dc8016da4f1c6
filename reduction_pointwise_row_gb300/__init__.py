"""Fused pointwise + row-reduction kernels for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libfr.so`` (``include/fr.h``).  It only marshals
arguments -- device pointers, sizes, the current CUDA stream -- and every step of
the computation runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.  There is no fallback: if the library is missing or the
device is not an sm_103 GPU the calls raise.

Functions carry the C names:

    fr_reduce_relu_add_sum(a, b, scale=2.0, form="auto")     -> out [rows] fp32
    fr_softmax(x, form="auto")                                -> y fp32
    fr_layernorm(x, gamma, beta, eps=1e-5, form="auto")       -> (y bf16, mean, rstd)
    fr_xent(logits, target, ignore_index=-100, ...)           -> dict of outputs
    fr_workspace_size(op, rows, cols, dtype, form)
    fr_check_device_error()
"""
from __future__ import annotations

import ctypes
import os

from . import buildlib as _build

__all__ = [
    "FR_OK", "FRError", "lib", "fr_version", "fr_workspace_size", "fr_last_form", "fr_auto_form",
    "fr_reduce_relu_add_sum", "fr_reduce_sumsq", "fr_softmax", "fr_softmax_host", "fr_layernorm",
    "fr_xent", "fr_xent_workspace", "fr_xent_mean_from_parts", "xent_mean_parts",
    "allreduce_mean_parts", "XENT_PARTS_OFFSET",
    "fr_reduce_relu_add_sum_split_static", "fr_check_device_error", "FORMS", "OPS",
    "EPILOGUES", "fr_coordinate_descent", "fr_xent_get_config", "fr_xent_set_config",
    "fr_xent_tune",
]

FR_OK = 0
STATUS = {0: "FR_OK", 1: "FR_ERR_INVALID_ARG", 2: "FR_ERR_UNSUPPORTED_DTYPE",
          3: "FR_ERR_UNSUPPORTED_FORM", 4: "FR_ERR_MISALIGNED",
          5: "FR_ERR_WORKSPACE_TOO_SMALL", 6: "FR_ERR_CUDA", 7: "FR_ERR_DEVICE_DATA",
          8: "FR_ERR_NO_DEVICE"}
FORMS = {"auto": 0, "persistent": 1, "looped": 2, "split": 3}
FORM_NAMES = {v: k for k, v in FORMS.items()}
OPS = {"relu_add_sum": 0, "softmax": 1, "layernorm": 2, "xent": 3, "sumsq": 4}
EPILOGUES = {"sum": 0, "sqrt": 1}
DTYPES = {"f32": 0, "bf16": 1}

# name -> (restype, argtypes) of every symbol include/fr.h declares
_i64, _f32, _vp, _sz, _int = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, \
    ctypes.c_int
SIGNATURES = {
    "fr_version": (_int, []),
    "fr_status_string": (ctypes.c_char_p, [_int]),
    "fr_last_form": (_int, []),
    "fr_workspace_size": (_sz, [_int, _i64, _i64, _int, _int]),
    "fr_auto_form": (_int, [_int, _int, _i64, _i64, ctypes.c_int32]),
    "fr_reduce_relu_add_sum": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _f32, _int,
                                      _vp, _sz, _vp]),
    "fr_reduce_sumsq": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp, _sz, _vp]),
    "fr_softmax": (_int, [_vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _vp]),
    "fr_softmax_host_workspace": (_sz, [_i64, _int, _i64]),
    "fr_softmax_host": (_int, [_vp, _vp, _i64, _i64, _int, _i64, _vp, _sz, _vp]),
    "fr_layernorm": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _int,
                            _int, _vp]),
    "fr_xent": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _vp,
                       _sz, _vp]),
    "fr_xent_mean_from_parts": (_int, [_vp, _vp, _vp]),
    "fr_xent_workspace_init": (_int, [_vp, _sz, _vp]),
    "fr_check_device_error": (_int, [_vp, ctypes.POINTER(ctypes.c_int32)]),
    "fr_coordinate_descent": (_int, [ctypes.c_int32, _vp, _vp, _vp, ctypes.c_double, _vp, _vp,
                                     _vp, _vp]),
    "fr_xent_get_config": (_int, [_i64, _i64, _i64, _vp]),
    "fr_xent_set_config": (_int, [_i64, _i64, _i64, _vp]),
    "fr_xent_tune": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, ctypes.c_double,
                            ctypes.c_int32, _vp, _vp, _vp, _vp]),
    "fr_reduce_relu_add_sum_split_static": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _int,
                                                   _f32, _vp]),
}


class FRError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libfr.so (built in-tree by ``build()``; never a fallback)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: run reduction_pointwise_row_gb300.buildlib.build() "
                              "(nvcc for sm_103a) first")
        l = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def build(force: bool = False) -> str:
    return _build.build(force=force)


def _check(status: int, where: str):
    if status != FR_OK:
        raise FRError(status, where)


_current_raw_stream = None  # device index -> cudaStream_t of its current stream
_current_device = None


def _stream(stream=None, device_index=None):
    """The raw cudaStream_t (an int) to launch on: `stream`, else the current
    stream of the current (or given) device.  The lookups are resolved once:
    a call costs two C calls, no Stream object (launch-bound shapes feel it)."""
    global _current_raw_stream, _current_device
    if stream is not None:
        return stream.cuda_stream
    if _current_raw_stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _current_raw_stream = raw if raw is not None else (
            lambda i: torch.cuda.current_stream(i).cuda_stream)
        _current_device = getattr(torch._C, "_cuda_getDevice", torch.cuda.current_device)
    return _current_raw_stream(_current_device() if device_index is None else device_index)


def _on_current_device(*ts):
    """The library launches on the current CUDA device: refuse tensors that
    live on another one (their addresses mean nothing there)."""
    _stream()  # resolves the device lookup
    cur = _current_device()
    for t in ts:
        if t is not None and t.get_device() != cur:
            raise ValueError(f"tensor on cuda:{t.get_device()}, current device is cuda:{cur}: "
                             "call inside torch.cuda.device(...)")


def _ptr(t):
    """A tensor's device address as an int (ctypes passes it as void *), or None."""
    return t.data_ptr() if t is not None else None


def _ld(t) -> int:
    assert t.dim() == 2 and t.stride(1) == 1, "rows must be contiguous (stride(1) == 1)"
    return t.stride(0)


def fr_version() -> int:
    return lib().fr_version()


def fr_last_form() -> str:
    return FORM_NAMES[lib().fr_last_form()]


def fr_auto_form(op: str, rows: int, cols: int, dtype: str = "f32", sm_count: int = 152) -> str:
    """The form AUTO picks for this shape on a device with ``sm_count`` SMs
    (host-side; no device needed)."""
    return FORM_NAMES[lib().fr_auto_form(OPS[op], DTYPES[dtype], rows, cols, sm_count)]


def sm_count(device=None) -> int:
    """SMs of the current (or given) CUDA device."""
    import torch
    return torch.cuda.get_device_properties(
        torch.cuda.current_device() if device is None else device).multi_processor_count


def fr_workspace_size(op: str, rows: int, cols: int, dtype: str = "f32", form: str = "auto") -> int:
    return lib().fr_workspace_size(OPS[op], rows, cols, DTYPES[dtype], FORMS[form])


_WS_SIZES = {}  # (op, rows, cols, dtype, form, device index) -> bytes


def _workspace(op, rows, cols, dtype, form, device, given=None):
    import torch
    key = (op, rows, cols, dtype, form, device.index)
    n = _WS_SIZES.get(key)
    if n is None:  # depends only on the shape and the device model
        n = _WS_SIZES[key] = fr_workspace_size(op, rows, cols, dtype, form)
    if n == 0:
        return None, 0
    if given is not None:
        return given, given.numel() * given.element_size()
    return torch.empty(n, dtype=torch.uint8, device=device), n


def fr_reduce_relu_add_sum(a, b, scale: float = 2.0, form: str = "auto", out=None,
                           workspace=None, stream=None):
    """out[x] = sum_r scale * relu(a[x, r] + b[x, r]) (fp32 or bf16 in, fp32 out;
    bf16 inputs are widened exactly to fp32 before the sum)."""
    import torch
    assert a.is_cuda and b.is_cuda and a.dtype == b.dtype
    assert a.dtype in (torch.float32, torch.bfloat16)
    assert a.shape == b.shape and a.dim() == 2
    dt = "f32" if a.dtype == torch.float32 else "bf16"
    rows, cols = a.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=a.device)
    _on_current_device(a, b, out)
    ws, nws = _workspace("relu_add_sum", rows, cols, dt, form, a.device, workspace)
    _check(lib().fr_reduce_relu_add_sum(_ptr(a), _ptr(b), _ptr(out), rows, cols, _ld(a), _ld(b),
                                        DTYPES[dt], scale, FORMS[form], _ptr(ws), nws,
                                        _stream(stream)), "fr_reduce_relu_add_sum")
    return out


def fr_reduce_sumsq(x, epilogue: str = "sum", form: str = "auto", out=None, workspace=None,
                    stream=None):
    """out[x] = sum_r x[x, r]^2 (epilogue "sum") or its square root, the row L2
    norm (epilogue "sqrt"); fp32 in, fp32 out."""
    import torch
    assert x.is_cuda and x.dtype == torch.float32 and x.dim() == 2
    rows, cols = x.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=x.device)
    _on_current_device(x, out)
    ws, nws = _workspace("sumsq", rows, cols, "f32", form, x.device, workspace)
    _check(lib().fr_reduce_sumsq(_ptr(x), _ptr(out), rows, cols, _ld(x), DTYPES["f32"],
                                 EPILOGUES[epilogue], FORMS[form], _ptr(ws), nws,
                                 _stream(stream)), "fr_reduce_sumsq")
    return out


def fr_softmax(x, form: str = "auto", out=None, stream=None):
    """Row softmax of fp32 or bf16 x, y of the same dtype (returns a new tensor
    unless ``out`` is given)."""
    import torch
    assert x.is_cuda and x.dtype in (torch.float32, torch.bfloat16) and x.dim() == 2
    rows, cols = x.shape
    if out is None:
        out = torch.empty_like(x)
    assert out.dtype == x.dtype and out.shape == x.shape
    dt = DTYPES["f32"] if x.dtype == torch.float32 else DTYPES["bf16"]
    _on_current_device(x, out)
    _check(lib().fr_softmax(_ptr(x), _ptr(out), rows, cols, _ld(x), _ld(out), dt,
                            FORMS[form], _stream(stream)), "fr_softmax")
    return out


def fr_softmax_host(x_host, out=None, chunk_rows: int | None = None, workspace=None,
                    stream=None, device=None):
    """Row softmax of a page-locked host tensor (fp32 or bf16); ``out``
    (page-locked, same shape and dtype) receives y.  ``chunk_rows`` None or 0:
    the kernel reads and writes the host rows directly over the host link;
    ``chunk_rows`` >= 1: the library's chunked copy-in / kernel / copy-out
    pipeline through a device workspace.  Returns ``out``.  Ordered on
    ``stream`` (default: the current stream of ``device``) without
    synchronising."""
    import torch
    assert not x_host.is_cuda and x_host.dtype in (torch.float32, torch.bfloat16)
    assert x_host.dim() == 2 and x_host.is_contiguous()
    rows, cols = x_host.shape
    if out is None:
        out = torch.empty_like(x_host).pin_memory()
    assert out.shape == x_host.shape and out.dtype == x_host.dtype and out.is_contiguous()
    dt = DTYPES["f32"] if x_host.dtype == torch.float32 else DTYPES["bf16"]
    if chunk_rows is None:
        chunk_rows = 0
    if chunk_rows > 0 and workspace is None:
        n = lib().fr_softmax_host_workspace(cols, dt, min(chunk_rows, rows))
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    nws = 0 if workspace is None else workspace.numel()
    _check(lib().fr_softmax_host(_ptr(x_host), _ptr(out), rows, cols, dt, chunk_rows,
                                 _ptr(workspace), nws, _stream(stream)), "fr_softmax_host")
    return out


def fr_layernorm(x, gamma, beta, eps: float = 1e-5, form: str = "auto", out=None, mean=None,
                 rstd=None, stream=None):
    """LayerNorm of bf16 rows; returns (y bf16, mean fp32, rstd fp32)."""
    import torch
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2
    rows, cols = x.shape
    assert gamma.dtype == torch.float32 and beta.dtype == torch.float32
    assert gamma.numel() == cols and beta.numel() == cols
    if out is None:
        out = torch.empty_like(x)
    if mean is None:
        mean = torch.empty(rows, dtype=torch.float32, device=x.device)
    if rstd is None:
        rstd = torch.empty(rows, dtype=torch.float32, device=x.device)
    _on_current_device(x, gamma, beta, out, mean, rstd)
    _check(lib().fr_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(out), _ptr(mean), _ptr(rstd),
                              rows, cols, _ld(x), _ld(out), eps, DTYPES["bf16"], FORMS[form],
                              _stream(stream)), "fr_layernorm")
    return out, mean, rstd


XENT_PARTS_OFFSET = 16  # FR_XENT_PARTS_OFFSET


def fr_xent_workspace(rows: int, cols: int, dtype: str = "bf16", device=None, stream=None):
    """A prepared cross-entropy workspace for this shape (fr_workspace_size
    bytes, prepared by fr_xent_workspace_init on ``stream``).  Every fr_xent
    call leaves it prepared; one call at a time may use it."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    n = fr_workspace_size("xent", rows, cols, dtype)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    _check(lib().fr_xent_workspace_init(_ptr(ws), ws.numel(), _stream(stream, dev.index)),
           "fr_xent_workspace_init")
    return ws


_XENT_WS = {}  # (device, stream, bytes) -> a prepared workspace the binding reuses


def _xent_workspace_for(rows, cols, dtype, device, stream):
    """The binding's own prepared workspace for calls on this device and
    stream (calls on one stream are ordered, so they can share it)."""
    sid = _stream(stream, device.index)
    n = fr_workspace_size("xent", rows, cols, dtype)
    key = (device.index, sid)
    ws = _XENT_WS.get(key)
    if ws is None or ws.numel() < n:
        ws = fr_xent_workspace(rows, cols, dtype, device, stream)
        _XENT_WS[key] = ws
    return ws


def xent_mean_parts(workspace):
    """The two fp64 values an fr_xent call with the mean leaves in its
    workspace -- the sum of the losses it averaged and the number of rows it
    averaged -- as a view that an all-reduce can sum in place."""
    return workspace[XENT_PARTS_OFFSET:XENT_PARTS_OFFSET + 16].view(_torch().float64)


def allreduce_mean_parts(parts, group=None):
    """Sum mean parts element-wise over the ranks of ``group``
    (torch.distributed, in place): the path's one exchange step."""
    import torch.distributed as dist
    dist.all_reduce(parts, op=dist.ReduceOp.SUM, group=group)
    return parts


def fr_xent_mean_from_parts(workspace, mean=None, stream=None):
    """mean = sum / count from the (summed) parts in an fr_xent workspace."""
    import torch
    if mean is None:
        mean = torch.empty(1, dtype=torch.float32, device=workspace.device)
    _check(lib().fr_xent_mean_from_parts(_ptr(workspace), _ptr(mean), _stream(stream)),
           "fr_xent_mean_from_parts")
    return mean


def _torch():
    import torch
    return torch


def _nullcontext():
    import contextlib
    return contextlib.nullcontext()


def fr_xent(logits, target, ignore_index: int = -100, want_loss: bool = True,
            want_mean: bool = True, want_target_logit: bool = False, want_argmax: bool = False,
            form: str = "auto", workspace=None, stream=None, group=None):
    """Cross entropy of bf16 or fp32 logits rows against int64 targets.

    Returns a dict with the requested outputs: ``loss`` [rows], ``mean`` [1],
    ``target_logit`` [rows], ``argmax`` [rows] (int64).  ``workspace``, when
    given, must come from fr_xent_workspace (prepared once; each call keeps
    it prepared); by default the binding keeps one per device and stream.
    With ``group`` (a
    torch.distributed group whose ranks each pass their own rows of one
    batch), ``mean`` is the mean over the whole batch: the ranks' mean parts
    are all-reduced between this rank's kernel and the finishing kernel.
    """
    import torch
    assert logits.is_cuda and logits.dtype in (torch.bfloat16, torch.float32) and logits.dim() == 2
    dt = "bf16" if logits.dtype == torch.bfloat16 else "f32"
    assert target.dtype == torch.int64 and target.is_cuda
    rows, cols = logits.shape
    assert target.numel() == rows
    dev = logits.device
    res = {}
    loss = torch.empty(rows, dtype=torch.float32, device=dev) if want_loss else None
    mean = torch.empty(1, dtype=torch.float32, device=dev) if want_mean else None
    tl = torch.empty(rows, dtype=torch.float32, device=dev) if want_target_logit else None
    am = torch.empty(rows, dtype=torch.int64, device=dev) if want_argmax else None
    _on_current_device(logits, target)
    ws, nws = (None, 0)
    if want_mean:
        ws = workspace if workspace is not None else _xent_workspace_for(rows, cols, dt, dev,
                                                                         stream)
        nws = ws.numel() * ws.element_size()
    _check(lib().fr_xent(_ptr(logits), _ptr(target), _ptr(loss), _ptr(mean), _ptr(tl), _ptr(am),
                         rows, cols, _ld(logits), ignore_index, DTYPES[dt], FORMS[form],
                         _ptr(ws), nws, _stream(stream)), "fr_xent")
    if group is not None and want_mean:
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            allreduce_mean_parts(xent_mean_parts(ws), group)
            fr_xent_mean_from_parts(ws, mean, stream)
    for k, v in (("loss", loss), ("mean", mean), ("target_logit", tl), ("argmax", am)):
        if v is not None:
            res[k] = v
    return res


def fr_reduce_relu_add_sum_split_static(a, b, scale: float = 2.0, out=None, stream=None):
    """Split-form relu_add_sum with no workspace: the partial sums live in the
    library's fixed 64 KiB device array, so nothing is allocated for the call
    (for callers that cannot allocate device memory where they launch).  Calls
    on one device share that array: keep them ordered on one stream."""
    import torch
    assert a.is_cuda and b.is_cuda and a.dtype == torch.float32 and b.dtype == torch.float32
    assert a.shape == b.shape and a.dim() == 2
    rows, cols = a.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=a.device)
    _on_current_device(a, b, out)
    _check(lib().fr_reduce_relu_add_sum_split_static(_ptr(a), _ptr(b), _ptr(out), rows, cols,
                                                     _ld(a), _ld(b), DTYPES["f32"], scale,
                                                     _stream(stream)),
           "fr_reduce_relu_add_sum_split_static")
    return out


# ---- launch configurations ----------------------------------------------------

COST_FN = ctypes.CFUNCTYPE(ctypes.c_double, ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p)


class XentConfig(ctypes.Structure):
    _fields_ = [("threads", ctypes.c_int32), ("vectors", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32)]

    def as_tuple(self):
        return (self.threads, self.vectors, self.stages, self.ctas_per_sm)


def fr_coordinate_descent(lo, hi, start, eps: float, cost):
    """Coordinate descent (Algorithm 9.2) over log2 parameters in the box
    [lo, hi] from ``start``; ``cost(tuple)`` returns a time (inf: cannot run).
    Returns (result, acceptances, evaluations)."""
    p = len(start)
    arr = ctypes.c_int32 * p
    c_lo, c_hi, c = arr(*lo), arr(*hi), arr(*start)
    fn = COST_FN(lambda q, _ctx: float(cost(tuple(q[i] for i in range(p)))))
    acc, ev = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().fr_coordinate_descent(p, ctypes.byref(c_lo), ctypes.byref(c_hi),
                                       ctypes.byref(c), eps, ctypes.cast(fn, ctypes.c_void_p),
                                       None, ctypes.byref(acc), ctypes.byref(ev)),
           "fr_coordinate_descent")
    return tuple(c), acc.value, ev.value


def fr_xent_get_config(rows: int, cols: int, ld: int | None = None) -> tuple:
    out = XentConfig()
    _check(lib().fr_xent_get_config(rows, cols, cols if ld is None else ld, ctypes.byref(out)),
           "fr_xent_get_config")
    return out.as_tuple()


def fr_xent_set_config(rows: int, cols: int, cfg, ld: int | None = None):
    """Records (threads, vectors, stages, ctas_per_sm) for this shape; None forgets."""
    ptr = None if cfg is None else ctypes.byref(XentConfig(*cfg))
    _check(lib().fr_xent_set_config(rows, cols, cols if ld is None else ld, ptr),
           "fr_xent_set_config")


def fr_xent_tune(logits, target, ignore_index: int = -100, eps: float = 0.02, reps: int = 5,
                 loss=None, stream=None) -> dict:
    """Algorithm 9.1 + 9.2 on the caller's data; records and returns the chosen
    configuration with the number of configurations timed and its median ms."""
    import torch
    assert logits.is_cuda and logits.dtype == torch.bfloat16 and logits.dim() == 2
    rows, cols = logits.shape
    out, ev, ms = XentConfig(), ctypes.c_int32(0), ctypes.c_float(0)
    _check(lib().fr_xent_tune(_ptr(logits), _ptr(target), _ptr(loss), rows, cols, _ld(logits),
                              ignore_index, DTYPES["bf16"], eps, reps, _stream(stream),
                              ctypes.byref(out), ctypes.byref(ev), ctypes.byref(ms)),
           "fr_xent_tune")
    return {"config": out.as_tuple(), "evaluations": ev.value, "ms": ms.value}


def fr_check_device_error(stream=None) -> int:
    """Synchronises the stream; returns and clears the device error code (0 = none)."""
    code = ctypes.c_int32(0)
    st = lib().fr_check_device_error(_stream(stream), ctypes.byref(code))
    if st not in (FR_OK, 7):
        raise FRError(st, "fr_check_device_error")
    return code.value
