"""Benchmark of the fused row-reduction path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on stdout (rank 0).  The headline workload is the fused softmax in
its persistent form, fp32 [32768, 1024] (logits 4*N(0,1)); a step is one call
of fr_softmax over that batch, inputs resident in HBM, launched back to back
over rotating copies of the inputs and outputs (1 GiB in all, eight times the
L2, so no launch finds its operands cached), the K steps timed together
between two CUDA events on the stream they run on.  Consecutive kernels are
programmatic dependents of one another (a kernel's CTAs are placed while the
one before it finishes, and read nothing before it has).  ``value`` is
achieved HBM GB/s: algorithmic bytes (one read and one write of every element)
/ time per step, summed over ranks.
``per_config`` adds the other workloads of the path measured the same way.
``e2e`` is the same metric through the C-ABI's host-buffer call with the input copied
from pinned host memory and the result copied back inside the timed region.

``--impl reference`` times the CPU oracle (the plain fp64 C definition) on a
bounded sample of the same workload on the host cores; under torchrun only
rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = 1
# LayerNorm hidden sizes that --only layernorm_<cols> times alone (256 MiB of x)
LN_HIDDEN = (768, 1024, 1536, 2048, 2560, 3072, 4096, 8192, 5120, 6144, 7168, 10240, 12288, 14336, 20480, 24576)
METRIC = "fused row-reduction achieved HBM GB/s and % of GB300 peak; rows/s per config"
UNIT = "GB/s"
PROFILE = os.path.join(ROOT, "profiles", "softmax_persistent_32768x1024.md")
KERNEL_SRC = os.path.join(ROOT, "reduction_pointwise_row_gb300", "csrc", "softmax.cu")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extra", action="store_true", help="headline workload only")
    p.add_argument("--only", choices=["relu_add_sum", "softmax", "layernorm", "split", "xent",
                                      "sumsq", "l2norm", "softmax_4097", "softmax_4097_looped",
                                      "softmax_65537", "softmax_65537_looped",
                                      "looped", "looped_bf16", "softmax_bf16", "xent_f32",
                                      "softmax_bf16_4097", "softmax_bf16_4097_looped",
                                      "softmax_bf16_65537", "xent_box", "form_sweep",
                                      "softmax_4097_offset", "softmax_bf16_8192_offset",
                                      "softmax_65537_offset", "softmax_8192_offset",
                                      "softmax_262144", "softmax_bf16_262144",
                                      *[f"layernorm_{c}" for c in LN_HIDDEN]],
                   help="time one workload alone (for profiler captures) and exit")
    p.add_argument("--form", default="auto", choices=["auto", "persistent", "looped", "split"],
                   help="with --only: force a reduction form")
    p.add_argument("--sweep-ops", default="relu_add_sum,softmax,softmax_bf16,softmax_offset,"
                   "softmax_bf16_offset,layernorm",
                   help="with --only form_sweep: the ops to sweep")
    p.add_argument("--sweep-md", metavar="JSONL",
                   help="print the form table (markdown) of a form_sweep output and exit")
    p.add_argument("--launches-md", metavar="CSV",
                   help="print the per-kernel summary (markdown) of an ncu launch list "
                        "(--metrics gpu__time_duration.sum --csv) and exit")
    return p.parse_args()


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) kept only while a timed loop runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.windows = []
        self.t0 = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.lines = []

    def window(self, start, end):
        self.windows.append((start, end))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        t_end = time.time()
        rows = [l.split(", ") for l in out.strip().splitlines() if l.count(",") >= 8]
        if not rows:
            return None
        # nvidia-smi -lms prints at a fixed period: spread timestamps evenly
        dt = (t_end - self.t0) / max(len(rows), 1)
        keep, all_mhz = [], []
        for i, r in enumerate(rows):
            ts = self.t0 + (i + 0.5) * dt
            try:
                mhz, mx = float(r[1]), float(r[2])
            except ValueError:
                continue
            all_mhz.append(mhz)
            if any(a - 0.05 <= ts <= b + 0.05 for a, b in self.windows):
                keep.append((mhz, mx, r))
        if not keep:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, _, r in keep:
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(k[0] for k in keep),
                "sm_max_mhz": max(k[1] for k in keep),
                "reasons": sorted(reasons), "samples": len(keep)}


# ---------------------------------------------------------------- profile

def kernel_source_hash():
    """sha256[:16] of the headline kernel's own source text (its template
    line through the closing brace at column 0) and of csrc/common.cuh, whose
    helpers it inlines: other kernels of the same file may change without
    invalidating its counters."""
    text = open(KERNEL_SRC).read()
    name = text.find("\nsoftmax_warp_vec(")
    if name < 0:
        return None
    start = text.rfind("\ntemplate <", 0, name) + 1
    end = text.index("\n}\n", name) + 3
    h = hashlib.sha256(text[start:end].encode())
    with open(os.path.join(ROOT, "reduction_pointwise_row_gb300", "csrc", "common.cuh"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the capture."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != kernel_source_hash():
        return None
    return int(t.group(1))


# ---------------------------------------------------------------- our arm

def to_device(arr, dev):
    """Host array -> device tensor (uint16 arrays hold bf16 bit patterns)."""
    import numpy as np
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(arr).to(dev)


def run_ours(args):
    import torch

    import reduction_pointwise_row_gb300 as fr
    from reduction_pointwise_row_gb300 import traffic
    from synth import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    fr.lib()
    peak, peak_kind = measured_peak()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local) if not args.only else None

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    global SHARD
    SHARD = (rank, world)

    def max_ranks(x: float) -> float:
        return max_over_ranks(x, world, dev)

    def timed(calls, steps, warmup, launches_per_call, blocks=BLOCKS):
        """Device time (s) per step: `steps` calls back to back, cycling over the
        rotating input sets, between two CUDA events on the launching stream
        (a barrier and a synchronize on both sides); the slowest rank's.  The
        first block of `steps` calls gives the time; `blocks` - 1 more blocks
        of the same calls give the spread.  Returns (time per step of the
        first block, launches in all blocks, times per step of every block)."""
        for i in range(warmup):
            calls[i % len(calls)]()
        per_block = []
        for _ in range(blocks):
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            w0 = time.time()
            e0.record(stream)
            for i in range(steps):
                calls[i % len(calls)]()
            e1.record(stream)
            barrier()
            if clocks:
                clocks.window(w0, time.time())
            per_block.append(max_ranks(e0.elapsed_time(e1) / 1e3 / steps))
        return per_block[0], launches_per_call * steps * blocks, per_block

    if args.only == "form_sweep":
        form_sweep(fr, dev, timed, args, peak, rank)
        return
    if args.only == "xent_box":
        if rank == 0:
            print(json.dumps(xent_box(fr, workloads, dev, timed, args, peak)), flush=True)
        return
    if args.only:
        res = extra_configs(fr, traffic, workloads, timed, dev, peak, args, world, [args.only],
                            args.form)
        if rank == 0:
            print(json.dumps({"only": args.only, **next(iter(res.values()))}), flush=True)
        return

    # ---- headline: softmax persistent fp32 [32768, 1024]
    w = make_shard(workloads, HEADLINE)
    rows, cols = w.rows, w.cols
    calls, _, _, _, _ = setup_workload("softmax", fr, workloads, dev)
    calls[0]()
    form = fr.fr_last_form()
    nbytes = traffic.algorithmic_bytes("softmax", rows, cols)
    t_launch, launches, blocks_h = timed(calls, args.steps, args.warmup, 1)
    value = world * nbytes / t_launch / 1e9
    nsets = len(calls)
    del calls
    x_host = torch.from_numpy(w.arrays["x"]).pin_memory()

    # ---- context: a plain device copy moving the same bytes (128 MiB in,
    # 128 MiB out) over the same rotating buffers -- what HBM gives a
    # streaming kernel of this size on this GPU
    srcs = [torch.empty(rows, cols, device=dev) for _ in range(nsets)]
    dsts = [torch.empty(rows, cols, device=dev) for _ in range(nsets)]
    copies = [lambda a=a, b=b: b.copy_(a) for a, b in zip(srcs, dsts)]
    t_copy, _, _ = timed(copies, args.steps, args.warmup, 0, blocks=1)
    del srcs, dsts, copies

    # ---- e2e: the library's host-buffer entry point (fr_softmax_host) on the
    # same rows in page-locked host memory, every byte crossing the host link
    # inside the timed region.  Direct form: the kernel reads x and writes y
    # in host memory over NVLink-C2C (790 us per step on GB300 from a grid of a
    # quarter of the SMs' CTAs, against 950 for the staged form with 4096-row
    # chunks, the best of 512 .. 32768).
    y_host = torch.empty_like(x_host).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    E2E_CHUNK = 0  # direct
    ws_host = None

    def e2e_call():
        fr.fr_softmax_host(x_host, out=y_host, chunk_rows=E2E_CHUNK, workspace=ws_host)

    for _ in range(args.warmup):
        e2e_call()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_call()
    e1.record(stream)
    barrier()
    clocks.window(w0, time.time())
    t_e2e = max_ranks(e0.elapsed_time(e1) / 1e3 / e2e_steps)
    e2e = {"value": round(world * nbytes / t_e2e / 1e9, 2), "unit": UNIT,
           "h2d_bytes_per_step": x_host.numel() * 4, "d2h_bytes_per_step": y_host.numel() * 4,
           "ms_per_step": round(t_e2e * 1e3, 4), "api": "fr_softmax_host",
           "chunk_rows": E2E_CHUNK, "path": "direct: the kernel reads and writes page-locked "
           "host memory over NVLink-C2C"}
    launches += e2e_steps * (-(-rows // E2E_CHUNK) if E2E_CHUNK else 1)  # a kernel per chunk
    del x_host, y_host, ws_host

    # ---- the other workloads of the path, same method
    per_config = {}
    if not args.no_extra:
        per_config = extra_configs(fr, traffic, workloads, timed, dev, peak, args, world)
        launches += sum(v.pop("_launches") for v in per_config.values())

    head_key = "softmax_32768x1024" if world == 1 else f"softmax_{rows}x{cols}"
    head_entry = {"op": "softmax", "rows": rows, "cols": cols, "form": form,
                  "us": round(t_launch * 1e6, 3), "gbs": round(nbytes / t_launch / 1e9, 2),
                  "frac": round(nbytes / t_launch / 1e9 / peak, 4),
                  "rows_per_s": round(world * rows / t_launch, 1), **spread_us(blocks_h),
                  "rotating_sets": nsets}
    per_config = {head_key: head_entry, **per_config}
    clk = clocks.stop()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_launch * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 / Box-Muller, 4*N(0,1))",
        "config": {"workload": "fused softmax, persistent form, fp32 [32768,1024]",
                   "rows": rows, "cols": cols, "form": form,
                   "rows_per_s": round(world * rows / t_launch, 1),
                   "l2": f"inputs larger than L2: {nsets} rotating x/y sets (1 GiB), launches back to back",
                   "timing": "CUDA events around the K back-to-back steps on the launching stream",
                   "parallelism": f"rows sharded over {world} ranks, no collective on the "
                                  "softmax path"},
        "roofline": {"bound": "hbm", "achieved": round(nbytes / t_launch / 1e9, 2),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(nbytes / t_launch / 1e9 / peak, 4),
                     "traffic": profiled_traffic(),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy burst)",
                     "same_bytes_device_copy_gbs": round(nbytes / t_copy / 1e9, 2)},
        "e2e": e2e,
        "gpu_launches": launches,
        "per_config": per_config,
        "clocks": clk,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(w)
        if not args.no_extra:
            line["cpu_baseline"]["per_config"] = cpu_baselines(w)
        # last, so that a reader keeping only the end of the line has every
        # configuration: the five workloads in one compact block
        line["configs"] = compact_configs(per_config, line["cpu_baseline"])
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


ROTATE_BYTES = 1 << 30  # footprint of the rotating input/output sets (8x the L2)

# This rank's shard of every workload: with N ranks the global batch has N
# times the rows and rank r holds rows r*R .. r*R + R - 1 (the generators are
# counter-based, so a shard is exactly those rows of the global array).  Rows
# are independent, so no rank exchanges anything (weak scaling).
SHARD = (0, 1)


def shard_rows(rows: int, rank: int, world: int) -> tuple[int, int]:
    """(first row, global rows) of rank's shard when every rank holds `rows`."""
    return rank * rows, world * rows


def make_shard(workloads, cfg: int, rows: int | None = None, cols: int | None = None, **kw):
    rank, world = SHARD
    R = workloads.FULL_SHAPES[cfg][1] if rows is None else rows
    row0, g = shard_rows(R, rank, world)
    return workloads.make(cfg, rows=R, cols=cols, row0=row0, global_rows=g, **kw)


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (every rank gets it)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def setup_workload(name, fr, workloads, dev, form="auto"):
    """Device inputs and calls of one workload: (calls, op, rows, cols,
    launches per call).  ``calls`` cycles over enough copies of the inputs
    and outputs that their footprint is >= 1 GiB, so no launch finds its
    operands in the 126 MB L2.  Inputs are generated on the host once."""
    import torch
    from reduction_pointwise_row_gb300 import traffic

    def nsets(op, rows, cols):
        return max(1, -(-ROTATE_BYTES // traffic.algorithmic_bytes(op, rows, cols)))

    calls = []
    if name == "relu_add_sum":
        w = make_shard(workloads, 0)
        a, b = to_device(w.arrays["a"], dev), to_device(w.arrays["b"], dev)
        out = torch.empty(w.rows, device=dev)
        calls.append(lambda: fr.fr_reduce_relu_add_sum(a, b, 2.0, out=out, form=form))
        return calls, "relu_add_sum", w.rows, w.cols, 1
    if name == "softmax":
        w = make_shard(workloads, 1)
        for _ in range(nsets("softmax", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            calls.append(lambda x=x, y=y: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax", w.rows, w.cols, 1
    if name in ("softmax_4097", "softmax_65537", "softmax_4097_looped", "softmax_65537_looped"):
        # the two long-row sweep lengths, 256 MiB each: the form AUTO picks
        # (one CTA per row at 4097, a cluster per row at 65537) and the looped
        # online form
        cols = int(name.split("_")[1])
        f = "looped" if name.endswith("_looped") else form
        w = make_shard(workloads, 1, rows=(1 << 25) // cols, cols=cols)
        for _ in range(nsets("softmax", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            calls.append(lambda x=x, y=y: fr.fr_softmax(x, out=y, form=f))
        return calls, "softmax", w.rows, w.cols, 1
    if name in ("softmax_262144", "softmax_bf16_262144"):
        # rows of 262144 in phase (fp32 304 rows, bf16 608: 304 MiB of x):
        # the split form, a cluster per row whose CTAs stream their runs twice
        bf16 = "bf16" in name
        rows = 608 if bf16 else 304
        op = "softmax_bf16" if bf16 else "softmax"
        w = (workloads.make_softmax_bf16(rows, 262144, seed=20261202 + 7 + 1000 * SHARD[0])
             if bf16 else make_shard(workloads, 1, rows=rows, cols=262144))
        for _ in range(nsets(op, w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            calls.append(lambda x=x, y=y: fr.fr_softmax(x, out=y, form=form))
        return calls, op, w.rows, w.cols, 1
    if name == "softmax_8192_offset":
        # rows of 8192 with x one element past y's phase (4096 rows, 128 MiB
        # of x): the persistent form stages each row in shared memory
        w = make_shard(workloads, 1, rows=(1 << 25) // 8192, cols=8192)
        n = w.rows * w.cols
        for _ in range(nsets("softmax", w.rows, w.cols)):
            flat = torch.empty(n + 8, device=dev)
            flat[1:n + 1].copy_(torch.from_numpy(w.arrays["x"].reshape(-1)))
            x = flat[1:n + 1].view(w.rows, w.cols)
            y = torch.empty(w.rows, w.cols, device=dev)
            calls.append(lambda x=x, y=y, flat=flat: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax", w.rows, w.cols, 1
    if name == "softmax_65537_offset":
        # rows of 65537 with x one element past y's phase (511 rows, 128 MiB
        # of x): the split form stages each CTA's run in shared memory
        w = make_shard(workloads, 1, rows=(1 << 25) // 65537, cols=65537)
        n = w.rows * w.cols
        for _ in range(nsets("softmax", w.rows, w.cols)):
            flat = torch.empty(n + 8, device=dev)
            flat[1:n + 1].copy_(torch.from_numpy(w.arrays["x"].reshape(-1)))
            x = flat[1:n + 1].view(w.rows, w.cols)
            y = torch.empty(w.rows, w.cols, device=dev)
            calls.append(lambda x=x, y=y, flat=flat: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax", w.rows, w.cols, 1
    if name == "softmax_4097_offset":
        # rows of 4097 with x one element past y's 32-byte phase (8190 rows,
        # 256 MiB): the persistent form stages each row in shared memory
        w = make_shard(workloads, 1, rows=(1 << 25) // 4097, cols=4097)
        n = w.rows * w.cols
        for _ in range(nsets("softmax", w.rows, w.cols)):
            flat = torch.empty(n + 8, device=dev)
            flat[1:n + 1].copy_(torch.from_numpy(w.arrays["x"].reshape(-1)))
            x = flat[1:n + 1].view(w.rows, w.cols)
            y = torch.empty(w.rows, w.cols, device=dev)
            calls.append(lambda x=x, y=y, flat=flat: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax", w.rows, w.cols, 1
    if name == "softmax_bf16_8192_offset":
        # bf16 rows of 8192 with x one element past y's phase (8192 rows,
        # 256 MiB): the persistent form stages each row in shared memory
        w = workloads.make_softmax_bf16(8192, 8192, seed=1)
        n = w.rows * w.cols
        for _ in range(nsets("softmax_bf16", w.rows, w.cols)):
            flat = torch.empty(n + 16, dtype=torch.bfloat16, device=dev)
            flat[1:n + 1].copy_(to_device(w.arrays["x"], dev).reshape(-1))
            x = flat[1:n + 1].view(w.rows, w.cols)
            y = torch.empty(w.rows, w.cols, dtype=torch.bfloat16, device=dev)
            calls.append(lambda x=x, y=y, flat=flat: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax_bf16", w.rows, w.cols, 1
    if name == "softmax_bf16":
        # the bf16 softmax on [65536, 1024] (the fp32 workload's 256 MiB)
        w = workloads.make_softmax_bf16(65536, 1024, seed=20261202 + 6 + 1000 * SHARD[0])
        for _ in range(nsets("softmax_bf16", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            calls.append(lambda x=x, y=y: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax_bf16", w.rows, w.cols, 1
    if name == "softmax_bf16_65537":
        # bf16 rows of 65537 (the fp32 sweep's bytes: 1022 rows): AUTO takes
        # a cluster of CTAs per row
        w = workloads.make_softmax_bf16(1022, 65537, seed=20261202 + 6 + 1000 * SHARD[0])
        for _ in range(nsets("softmax_bf16", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            calls.append(lambda x=x, y=y: fr.fr_softmax(x, out=y, form=form))
        return calls, "softmax_bf16", w.rows, w.cols, 1
    if name in ("softmax_bf16_4097", "softmax_bf16_4097_looped"):
        # bf16 rows of 4097 (the fp32 sweep's bytes: 16380 rows): one CTA per
        # row (AUTO) or the looped online form
        f = "looped" if name.endswith("looped") else form
        w = workloads.make_softmax_bf16(16380, 4097, seed=20261202 + 6 + 1000 * SHARD[0])
        for _ in range(nsets("softmax_bf16", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            calls.append(lambda x=x, y=y: fr.fr_softmax(x, out=y, form=f))
        return calls, "softmax_bf16", w.rows, w.cols, 1
    if name == "looped":
        # Example 1.1's looped form on 16384 rows of 8192 (1 GiB of a and b)
        w = make_shard(workloads, 0, rows=16384, cols=8192)
        a, b = to_device(w.arrays["a"], dev), to_device(w.arrays["b"], dev)
        out = torch.empty(w.rows, device=dev)
        calls.append(lambda: fr.fr_reduce_relu_add_sum(a, b, 2.0, out=out, form=form))
        return calls, "relu_add_sum", w.rows, w.cols, 1
    if name == "looped_bf16":
        # the same in bf16: 16384 x 16384 (1 GiB of a and b), rounded from
        # Example 1.1's U(-1, 1) inputs
        w = make_shard(workloads, 0, rows=16384, cols=16384)
        a = torch.from_numpy(w.arrays["a"]).to(dev).to(torch.bfloat16)
        b = torch.from_numpy(w.arrays["b"]).to(dev).to(torch.bfloat16)
        out = torch.empty(w.rows, device=dev)
        calls.append(lambda: fr.fr_reduce_relu_add_sum(a, b, 2.0, out=out, form=form))
        return calls, "relu_add_sum_bf16", w.rows, w.cols, 1
    if name == "layernorm":
        w = make_shard(workloads, 2)
        g, bt = to_device(w.arrays["gamma"], dev), to_device(w.arrays["beta"], dev)
        for _ in range(nsets("layernorm", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            mean = torch.empty(w.rows, device=dev)
            rstd = torch.empty(w.rows, device=dev)
            calls.append(lambda x=x, y=y, mean=mean, rstd=rstd:
                         fr.fr_layernorm(x, g, bt, 1e-5, out=y, mean=mean, rstd=rstd,
                                         form=form))
        return calls, "layernorm", w.rows, w.cols, 1
    if name.startswith("layernorm_"):
        # LayerNorm at another hidden size, 256 MiB of x (the workload's
        # distribution, gamma/beta of that length)
        cols = int(name.split("_")[1])
        w = make_shard(workloads, 2, rows=(1 << 27) // cols, cols=cols)
        g, bt = to_device(w.arrays["gamma"], dev), to_device(w.arrays["beta"], dev)
        for _ in range(nsets("layernorm", w.rows, w.cols)):
            x = to_device(w.arrays["x"], dev)
            y = torch.empty_like(x)
            mean = torch.empty(w.rows, device=dev)
            rstd = torch.empty(w.rows, device=dev)
            calls.append(lambda x=x, y=y, mean=mean, rstd=rstd:
                         fr.fr_layernorm(x, g, bt, 1e-5, out=y, mean=mean, rstd=rstd,
                                         form=form))
        return calls, "layernorm", w.rows, w.cols, 1
    if name == "split":
        w = make_shard(workloads, 3)
        rows, cols = w.rows, w.cols
        for _ in range(nsets("relu_add_sum", rows, cols)):
            a, b = to_device(w.arrays["a"], dev), to_device(w.arrays["b"], dev)
            out = torch.empty(rows, device=dev)
            f = "split" if form == "auto" else form
            ws = torch.empty(max(16, fr.fr_workspace_size("relu_add_sum", rows, cols, "f32", f)),
                             dtype=torch.uint8, device=dev)
            calls.append(lambda a=a, b=b, out=out, ws=ws:
                         fr.fr_reduce_relu_add_sum(a, b, 2.0, out=out, workspace=ws, form=form))
        return calls, "relu_add_sum", rows, cols, 2
    if name in ("sumsq", "l2norm"):
        # Example 6.2's [64, 16384] sum of squares (split form), and the row L2
        # norm over 1 GiB of [16384, 16384] rows (looped form)
        sd = 20261202 + 5 + 1000 * SHARD[0]  # rank r: its own batch of rows
        w = (workloads.make_sumsq(seed=sd) if name == "sumsq"
             else workloads.make_sumsq(16384, 16384, seed=sd))
        rows, cols = w.rows, w.cols
        epi = "sum" if name == "sumsq" else "sqrt"
        for _ in range(nsets("sumsq", rows, cols)):
            x = to_device(w.arrays["x"], dev)
            out = torch.empty(rows, device=dev)
            ws = torch.empty(max(16, fr.fr_workspace_size("sumsq", rows, cols, "f32", form)),
                             dtype=torch.uint8, device=dev)
            calls.append(lambda x=x, out=out, ws=ws:
                         fr.fr_reduce_sumsq(x, epi, out=out, workspace=ws, form=form))
        split = fr.fr_workspace_size("sumsq", rows, cols, "f32", form) > 0
        return calls, "sumsq", rows, cols, 2 if split else 1
    if name == "xent":
        group = None
        if SHARD[1] > 1:
            import torch.distributed as dist
            group = dist.group.WORLD
        w = make_shard(workloads, 4)
        rows, cols = w.rows, w.cols
        tg = torch.from_numpy(w.arrays["target"]).to(dev)
        for _ in range(nsets("xent", rows, cols)):
            lg = to_device(w.arrays["logits"], dev)
            wsx = fr.fr_xent_workspace(rows, cols, "bf16", dev)
            # ranks > 1: the batch mean over every rank's rows (all-reduce of
            # the mean parts, then the finishing kernel)
            calls.append(lambda lg=lg, wsx=wsx: fr.fr_xent(lg, tg, -100, workspace=wsx,
                                                           group=group))
        return calls, "xent", rows, cols, 1 if group is None else 2
    if name == "xent_f32":  # the cross-entropy shape with fp32 logits
        rows, cols = 8192, 50257
        w = workloads.make_xent_f32(rows, cols)
        tg = torch.from_numpy(w.arrays["target"]).to(dev)
        for _ in range(nsets("xent_f32", rows, cols)):
            lg = to_device(w.arrays["logits"], dev)
            wsx = fr.fr_xent_workspace(rows, cols, "f32", dev)
            calls.append(lambda lg=lg, wsx=wsx: fr.fr_xent(lg, tg, -100, workspace=wsx))
        return calls, "xent_f32", rows, cols, 1
    raise ValueError(name)


EXTRA = {"relu_add_sum": "relu_add_sum_64x128", "layernorm": "layernorm_4096x32768",
         "split": "relu_add_sum_split_8x33554432", "xent": "xent_8192x50257",
         "sumsq": "sumsq_split_64x16384", "l2norm": "l2norm_looped_16384x16384",
         "softmax_4097": "softmax_8190x4097", "softmax_4097_looped": "softmax_looped_8190x4097",
         "softmax_65537": "softmax_511x65537", "softmax_65537_looped": "softmax_looped_511x65537",
         "looped": "relu_add_sum_looped_16384x8192", "softmax_bf16": "softmax_bf16_65536x1024",
         "xent_f32": "xent_f32_8192x50257", "looped_bf16": "relu_add_sum_bf16_looped_16384x16384",
         "softmax_bf16_4097": "softmax_bf16_16380x4097",
         "softmax_bf16_4097_looped": "softmax_bf16_looped_16380x4097",
         "softmax_bf16_65537": "softmax_bf16_1022x65537",
         "softmax_262144": "softmax_304x262144", "softmax_bf16_262144": "softmax_bf16_608x262144",
         "softmax_4097_offset": "softmax_offset_8190x4097",
         "softmax_8192_offset": "softmax_offset_4096x8192",
         "softmax_65537_offset": "softmax_offset_511x65537",
         "softmax_bf16_8192_offset": "softmax_bf16_offset_8192x8192",
         "layernorm_768": "layernorm_174762x768", "layernorm_6144": "layernorm_21845x6144"}


def extra_configs(fr, traffic, workloads, timed, dev, peak, args, world, names=None,
                  form="auto"):
    steps = max(3, min(args.steps, 50))
    res = {}
    for name in (names or EXTRA):
        calls, op, rows, cols, lpc = setup_workload(name, fr, workloads, dev, form)
        calls[0]()
        t, n, per_block = timed(calls, steps, args.warmup, lpc)
        nb = traffic.algorithmic_bytes(op, rows, cols)
        res[EXTRA.get(name, name)] = {
            "op": op, "rows": rows, "cols": cols, "form": fr.fr_last_form(),
            "us": round(t * 1e6, 3), "gbs": round(nb / t / 1e9, 2),
            "frac": round(nb / t / 1e9 / peak, 4), "rows_per_s": round(world * rows / t, 1),
            **spread_us(per_block), "_launches": n, "rotating_sets": len(calls)}
        if name in ("relu_add_sum", "sumsq"):
            res[EXTRA[name]].update(graph_replay(calls[0], steps, args.warmup))
            res[EXTRA[name]]["_launches"] += GRAPH_CALLS * steps * lpc
        if name == "xent":
            tuned = tune_xent(fr, workloads, dev, calls, timed, steps, args, nb, peak)
            res[EXTRA[name]]["_launches"] += tuned.pop("_launches")
            res[EXTRA[name]].update(tuned)
        del calls
        if op == "layernorm" and not args.only:
            # context: a device copy of the same bytes (x in, y out)
            import torch
            srcs = [torch.empty(rows * cols, dtype=torch.bfloat16, device=dev) for _ in range(2)]
            dsts = [torch.empty_like(srcs[0]) for _ in range(2)]
            cps = [lambda a=a, b=b: b.copy_(a) for a, b in zip(srcs, dsts)]
            tc, _, _ = timed(cps, steps, args.warmup, 0, blocks=1)
            res[EXTRA.get(name, name)]["same_bytes_device_copy_gbs"] = round(nb / tc / 1e9, 2)
            del srcs, dsts, cps
    return res


def xent_box(fr, workloads, dev, timed, args, peak):
    """Every runnable point of the cross-entropy kernels' configuration space
    (the ring kernel's box threads x vectors x stages x CTAs per SM, and the
    warp-per-row points), timed like the bench's other lines: the
    measurements behind the default configuration."""
    from reduction_pointwise_row_gb300 import traffic
    calls, op, rows, cols, _ = setup_workload("xent", fr, workloads, dev)
    nb = traffic.algorithmic_bytes(op, rows, cols)
    steps = max(3, min(args.steps, 30))
    out = []
    points = [(t, u, s, g) for t in (128, 256, 512, 1024) for u in (1, 2, 4, 8)
              for s in (2, 4, 8) for g in (1, 2, 4, 8, 16)]
    points += [(32, u, 1, g) for u in (4, 8) for g in (1, 2, 4, 8, 16)]  # warp per row
    for cfg in points:
        try:
            fr.fr_xent_set_config(rows, cols, cfg)
        except fr.FRError:
            continue
        sec, _, _ = timed(calls, steps, args.warmup, 1, blocks=1)
        out.append({"config": list(cfg), "us": round(sec * 1e6, 2),
                    "frac": round(nb / sec / 1e9 / peak, 4)})
    fr.fr_xent_set_config(rows, cols, None)
    out.sort(key=lambda r: r["us"])
    return {"only": "xent_box", "rows": rows, "cols": cols, "runnable": len(out),
            "default_config": list(fr.fr_xent_get_config(rows, cols)), "points": out}


# Shapes of the form sweep (rows x cols per op; every form that can run is
# timed).  Around the selection rules: warp-per-row rows (<= 1024 fp32), the
# split form's few-long-rows corner, one CTA or one cluster per row.
SWEEP_RAS_ROWS = (8, 32, 128, 512, 1024, 2048, 4096, 8192)
SWEEP_RAS_COLS = (1024, 4096, 16384, 65536, 262144, 1048576, 4194304)
SWEEP_SM_ROWS = (16, 64, 152, 304, 608, 1216, 2432, 4864, 16384)
SWEEP_SM_COLS = (1025, 2048, 4097, 8192, 16384, 32768, 65537, 131072, 262144, 393216, 1048576)
SWEEP_OFFSET_COLS = (1025, 2048, 4097, 8192, 16384, 32768, 65537, 131072)
SWEEP_LN_COLS = (768, 1024, 1536, 2048, 2560, 3072, 4096, 5120, 6144, 7168, 8192, 10240, 12288,
                 14336, 16384, 20480, 24576, 32768, 65536)
SWEEP_BYTES_MAX = 1 << 30  # largest input footprint of one call


def form_sweep(fr, dev, timed, args, peak, rank):
    """Every reduction form (and LayerNorm kernel) that can run, timed on a
    grid of shapes the way the bench times its workloads: back-to-back calls
    over rotating views of buffers that together exceed the L2 (1 GiB),
    inputs filled on the device (uniform(-1, 1); the times do not depend on
    the values).  Prints one JSON line per shape: the time per call of each
    form (median of three K-step blocks), the fastest, and AUTO's pick."""
    import torch
    from reduction_pointwise_row_gb300 import traffic
    steps = max(5, min(args.steps, 20))
    name = torch.cuda.get_device_name(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    ops = set(args.sweep_ops.split(","))

    def rotating(rows, cols, dtype, bytes_per_set, fill=True):
        """Views of one buffer, set k at element offset k*rows*cols (so two
        such lists of one shape pair up in the same 32-byte phase)."""
        n = max(2, -(-ROTATE_BYTES // max(bytes_per_set, 1)))
        buf = torch.empty(n * rows, cols, dtype=dtype, device=dev)
        if fill:
            buf.uniform_(-1.0, 1.0)
        return [buf[k * rows:(k + 1) * rows] for k in range(n)]

    def measure(make_calls, forms, op, rows, cols):
        res, auto_form, auto_us = {}, None, None
        for f in forms:
            calls = make_calls(f)
            try:
                calls[0]()
            except fr.FRError:
                continue
            _, _, per = timed(calls, steps, 3, 1, blocks=3)
            t = round(sorted(per)[1] * 1e6, 3)
            if f == "auto":
                auto_form, auto_us = fr.fr_last_form(), t
            else:
                res[f] = t
        best = min(res, key=res.get) if res else None
        nb = traffic.algorithmic_bytes(op, rows, cols)
        line = {"op": op, "rows": rows, "cols": cols, "device": name, "sms": sms, "us": res,
                "fastest": best, "auto": auto_form, "auto_us": auto_us,
                "best_frac": round(nb / (res[best] * 1e-6) / 1e9 / peak, 4) if best else None}
        if rank == 0:
            print(json.dumps(line), flush=True)

    forms3 = ["persistent", "looped", "split", "auto"]  # AUTO last: every form warmed alike
    # Example 1.1, fp32
    for rows in SWEEP_RAS_ROWS:
        for cols in SWEEP_RAS_COLS:
            if "relu_add_sum" not in ops or rows * cols * 8 > SWEEP_BYTES_MAX:
                continue
            As = rotating(rows, cols, torch.float32, rows * cols * 8)
            Bs = rotating(rows, cols, torch.float32, rows * cols * 8)
            out = torch.empty(rows, device=dev)
            ws = torch.empty(max(16, fr.fr_workspace_size("relu_add_sum", rows, cols, "f32",
                                                          "split")), dtype=torch.uint8, device=dev)

            def mk(f, As=As, Bs=Bs, out=out, ws=ws):
                return [lambda a=a, b=b: fr.fr_reduce_relu_add_sum(a, b, 2.0, out=out, form=f,
                                                                  workspace=ws)
                        for a, b in zip(As, Bs)]
            measure(mk, forms3, "relu_add_sum", rows, cols)
            del As, Bs
    # softmax, fp32 and bf16
    for dtype, op in ((torch.float32, "softmax"), (torch.bfloat16, "softmax_bf16")):
        es = 4 if dtype == torch.float32 else 2
        for rows in SWEEP_SM_ROWS:
            for cols in SWEEP_SM_COLS:
                if (op not in ops or rows * cols * es * 2 > SWEEP_BYTES_MAX or
                        rows * cols * es < (1 << 20)):
                    continue
                Xs = rotating(rows, cols, dtype, 2 * rows * cols * es)
                Ys = rotating(rows, cols, dtype, 2 * rows * cols * es, fill=False)

                def mk(f, Xs=Xs, Ys=Ys):
                    return [lambda x=x, y=y: fr.fr_softmax(x, out=y, form=f) for x, y in zip(Xs, Ys)]
                measure(mk, forms3, op, rows, cols)
                del Xs, Ys
    # softmax with x one element past y's phase (every row out of 32-byte
    # phase: no vector pairing of x and y), fp32 and bf16
    for dtype, op in ((torch.float32, "softmax_offset"), (torch.bfloat16, "softmax_bf16_offset")):
        es = 4 if dtype == torch.float32 else 2
        for rows in SWEEP_SM_ROWS:
            for cols in SWEEP_OFFSET_COLS:
                if (op not in ops or rows * cols * es * 2 > SWEEP_BYTES_MAX or
                        rows * cols * es < (1 << 20)):
                    continue
                nset = max(2, -(-ROTATE_BYTES // (2 * es * rows * cols)))
                flat = torch.empty(nset * rows * cols + 16, device=dev,
                                   dtype=dtype).uniform_(-1.0, 1.0)
                Xs = [flat[1 + k * rows * cols:1 + (k + 1) * rows * cols].view(rows, cols)
                      for k in range(nset)]
                Ys = rotating(rows, cols, dtype, 2 * es * rows * cols, fill=False)

                def mk(f, Xs=Xs, Ys=Ys):
                    return [lambda x=x, y=y: fr.fr_softmax(x, out=y, form=f)
                            for x, y in zip(Xs, Ys)]
                measure(mk, forms3, op, rows, cols)
                del Xs, Ys, flat
    # LayerNorm: its kernels (the looped form's cluster, ring and scalar
    # kernels, and the persistent form), 256 MiB of x per call
    for cols in SWEEP_LN_COLS if "layernorm" in ops else ():
        rows = (1 << 27) // cols
        Xs = rotating(rows, cols, torch.bfloat16, 4 * rows * cols)
        Ys = rotating(rows, cols, torch.bfloat16, 4 * rows * cols, fill=False)
        g = torch.ones(cols, device=dev)
        bt = torch.zeros(cols, device=dev)
        mean = torch.empty(rows, device=dev)
        rstd = torch.empty(rows, device=dev)
        res, auto_form, auto_us = {}, None, None
        for kname, f in (("cluster", "looped"), ("ring", "looped"), ("scalar", "looped"),
                         ("rows", "persistent"), ("cta", "persistent"), ("auto", "auto")):
            os.environ["FR_LAYERNORM_KERNEL"] = "" if kname == "auto" else kname
            calls = [lambda x=x, y=y, f=f: fr.fr_layernorm(x, g, bt, 1e-5, form=f, out=y, mean=mean,
                                                          rstd=rstd) for x, y in zip(Xs, Ys)]
            try:
                calls[0]()
            except fr.FRError:
                continue
            _, _, per = timed(calls, steps, 3, 1, blocks=3)
            t = round(sorted(per)[1] * 1e6, 3)
            if kname == "auto":
                auto_form, auto_us = fr.fr_last_form(), t
            else:
                res[kname] = t
        os.environ.pop("FR_LAYERNORM_KERNEL", None)
        best = min(res, key=res.get)
        nb = traffic.algorithmic_bytes("layernorm", rows, cols)
        if rank == 0:
            print(json.dumps({"op": "layernorm", "rows": rows, "cols": cols, "device": name,
                              "sms": sms, "us": res, "fastest": best, "auto": auto_form,
                              "auto_us": auto_us,
                              "best_frac": round(nb / (res[best] * 1e-6) / 1e9 / peak, 4)}),
                  flush=True)
        del Xs, Ys


def tune_xent(fr, workloads, dev, calls, timed, steps, args, nb, peak):
    """Launch-configuration search for the cross-entropy kernel on this
    workload (candidate set, then coordinate descent, eps = 0.02), followed by
    the same back-to-back timing with the chosen configuration."""
    import torch
    w = make_shard(workloads, 4)
    lg = to_device(w.arrays["logits"], dev)
    tg = torch.from_numpy(w.arrays["target"]).to(dev)
    fr.fr_xent_set_config(w.rows, w.cols, None)
    default = fr.fr_xent_get_config(w.rows, w.cols)
    r = fr.fr_xent_tune(lg, tg, -100, eps=0.02, reps=5)
    del lg
    t, n, _ = timed(calls, steps, args.warmup, 1, blocks=1)
    fr.fr_xent_set_config(w.rows, w.cols, None)
    return {"default_config": list(default), "tuned_config": list(r["config"]),
            "tune_evaluations": r["evaluations"], "tuned_us": round(t * 1e6, 3),
            "tuned_gbs": round(nb / t / 1e9, 2), "tuned_frac": round(nb / t / 1e9 / peak, 4),
            "_launches": n}


CPU_BASELINE_SECONDS = 1.0  # wall time of repeated oracle passes per CPU measurement
BLOCKS = 7  # K-step blocks per workload: the first gives the time, all give the spread


def spread_us(per_block):
    """p10 / median / p90 of the per-step times of the K-step blocks (us)."""
    import numpy as np
    q = np.percentile(np.asarray(per_block) * 1e6, [10, 50, 90])
    return {"p10_us": round(float(q[0]), 3), "p50_us": round(float(q[1]), 3),
            "p90_us": round(float(q[2]), 3), "blocks": len(per_block)}
GRAPH_CALLS = 64  # calls recorded in one CUDA graph for the launch-bound case


def graph_replay(call, steps, warmup):
    """The launch-bound small case replayed from a CUDA graph holding
    GRAPH_CALLS back-to-back calls: one submission per replay, so the time per
    call is the device's, not the host's launch path."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(GRAPH_CALLS):
            call()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (steps * GRAPH_CALLS)
    return {"graph_us_per_call": round(us, 3), "graph_calls_per_replay": GRAPH_CALLS}


# ---------------------------------------------------------------- oracle arms

def cpu_baseline(w):
    """The oracle as it stands on the whole headline workload: single-threaded,
    and row-partitioned over every host core (threads calling the C oracle on
    disjoint row blocks; rows are independent, so the results are the same).
    After one untimed pass, each is repeated until CPU_BASELINE_SECONDS of
    wall time have passed (at least once) and timed as the mean pass."""
    import concurrent.futures as cf
    import os
    import oracle
    from reduction_pointwise_row_gb300 import traffic
    o = oracle.get()
    rows = w.rows  # the whole workload: one pass takes well under a second
    x = w.arrays["x"]
    nb = traffic.algorithmic_bytes("softmax", rows, w.cols)

    def mean_pass(fn):
        fn()  # untimed: first touch of the input and output pages
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= CPU_BASELINE_SECONDS:
                return el / n, n

    dt1, n1 = mean_pass(lambda: o.softmax(x))
    cores = os.cpu_count() or 1
    blocks = [x[i * rows // cores:(i + 1) * rows // cores] for i in range(cores)]
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        dtn, nn = mean_pass(lambda: list(ex.map(o.softmax, blocks)))
    return {"value": round(nb / dtn / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": round(dtn, 4), "passes": nn, "single_thread_value": round(nb / dt1 / 1e9, 4),
            "single_thread_seconds": round(dt1, 4), "single_thread_passes": n1,
            "sample": f"{rows} of {w.rows} rows x {w.cols} per pass (fp64 C oracle, rows split "
                      f"over {cores} threads, {nn} passes in {round(nn * dtn, 2)} s; single-threaded "
                      f"alongside, {n1} passes)"}


# The five workloads' entries in per_config (configuration index -> key).
CONFIG_KEYS = {0: "relu_add_sum_64x128", 1: "softmax_32768x1024", 2: "layernorm_4096x32768",
               3: "relu_add_sum_split_8x33554432", 4: "xent_8192x50257"}
CONFIG_NAMES = {0: "relu_add_sum f32 64x128 (Example 1.1)", 1: "softmax f32 32768x1024",
                2: "layernorm bf16 4096x32768", 3: "relu_add_sum split f32 8x33554432",
                4: "xent bf16 8192x50257"}


def compact_configs(per_config, cpu):
    """configs 0-4 in a few keys each: us per step (first K-step block), GB/s,
    fraction of the measured peak, rows/s, the p10/p90 over the blocks, the
    form, and the oracle's GB/s on the host cores."""
    out = {}
    cpu_pc = cpu.get("per_config", {})
    for i, key in CONFIG_KEYS.items():
        e = per_config.get(key)
        if e is None:
            continue
        c = {"w": CONFIG_NAMES[i], "form": e["form"], "us": e["us"], "gbs": e["gbs"],
             "frac": e["frac"], "rows_s": e["rows_per_s"], "p10_us": e["p10_us"],
             "p90_us": e["p90_us"]}
        if "graph_us_per_call" in e:
            c["graph_us"] = e["graph_us_per_call"]
        if str(i) in cpu_pc:
            c["cpu_gbs"] = cpu_pc[str(i)]["gbs"]
        out[str(i)] = c
    return out


def _mean_pass(fn):
    """Mean wall time of fn over CPU_BASELINE_SECONDS (after one untimed call)."""
    fn()
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= CPU_BASELINE_SECONDS:
            return el / n, n


def cpu_baselines(w_softmax):
    """The oracle as it stands on every configuration's workload (or a stated
    sample of it), rows -- or, for the split workload's eight rows, column
    blocks -- spread over the host cores by threads calling the C oracle.
    Returns {config index: {gbs, rows_per_s, seconds, cores, sample}}."""
    import concurrent.futures as cf
    import numpy as np
    import oracle
    from reduction_pointwise_row_gb300 import traffic
    from synth import workloads
    o = oracle.get()
    cores = os.cpu_count() or 1
    res = {}

    def blocks_of(arr, n):
        return [arr[i * len(arr) // n:(i + 1) * len(arr) // n] for i in range(n)]

    def record(cfg, nbytes, rows_equiv, fn, threads, sample):
        dt, n = _mean_pass(fn)
        res[str(cfg)] = {"gbs": round(nbytes / dt / 1e9, 4), "rows_per_s": round(rows_equiv / dt, 1),
                         "seconds": round(dt, 5), "passes": n, "cores": threads, "sample": sample}

    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        # 0: Example 1.1, the whole [64, 128] on one thread (too small to split)
        w = workloads.make(0)
        a, b = w.arrays["a"], w.arrays["b"]
        record(0, traffic.algorithmic_bytes("relu_add_sum", 64, 128), 64,
               lambda: o.relu_add_sum(a, b, 2.0), 1, "all 64 rows x 128")
        # 1: the headline softmax, every row
        x = w_softmax.arrays["x"]
        xb = blocks_of(x, cores)
        record(1, traffic.algorithmic_bytes("softmax", *x.shape), x.shape[0],
               lambda: list(ex.map(o.softmax, xb)), cores, f"all {x.shape[0]} rows x {x.shape[1]}")
        # 2: LayerNorm, every row
        w = workloads.make(2)
        xs, g, bt = w.arrays["x"], w.arrays["gamma"], w.arrays["beta"]
        xsb = blocks_of(xs, cores)
        record(2, traffic.algorithmic_bytes("layernorm", w.rows, w.cols), w.rows,
               lambda: list(ex.map(lambda blk: o.layernorm(blk, g, bt, 1e-5), xsb)), cores,
               f"all {w.rows} rows x {w.cols}")
        # 3: the split workload's 8 rows, the first 2^22 columns of each, in
        # `cores` column blocks (each block a contiguous copy)
        cols3 = 1 << 22
        w = workloads.make(3, cols=cols3)
        ab = [(np.ascontiguousarray(w.arrays["a"][:, i * cols3 // cores:(i + 1) * cols3 // cores]),
               np.ascontiguousarray(w.arrays["b"][:, i * cols3 // cores:(i + 1) * cols3 // cores]))
              for i in range(cores)]
        record(3, traffic.algorithmic_bytes("relu_add_sum", 8, cols3), 8 * cols3 / 33554432,
               lambda: list(ex.map(lambda p: o.relu_add_sum(p[0], p[1], 2.0), ab)), cores,
               f"8 rows x the first {cols3} of 33554432 columns, in {cores} column blocks")
        # 4: cross entropy on the first 2048 of 8192 rows
        w = workloads.make(4, rows=2048)
        lg, tg = w.arrays["logits"], w.arrays["target"]
        parts = list(zip(blocks_of(lg, cores), blocks_of(tg, cores)))
        record(4, traffic.algorithmic_bytes("xent", w.rows, w.cols), w.rows,
               lambda: list(ex.map(lambda p: o.xent(p[0], p[1], -100), parts)), cores,
               f"the first {w.rows} of 8192 rows x {w.cols}")
    return res


def run_reference(args):
    """The oracle as it stands, on the host cores: each step is the whole
    headline workload with its rows split over every core (threads calling the
    C oracle on disjoint row blocks)."""
    import concurrent.futures as cf
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from reduction_pointwise_row_gb300 import traffic
    from synth import workloads
    w = make_shard(workloads, HEADLINE)
    o = oracle.get()
    rows = w.rows
    x = w.arrays["x"]
    cores = os.cpu_count() or 1
    blocks = [x[i * rows // cores:(i + 1) * rows // cores] for i in range(cores)]
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        def step():
            list(ex.map(o.softmax, blocks))
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        dt = (time.perf_counter() - t0) / args.steps
    nb = traffic.algorithmic_bytes("softmax", rows, w.cols)
    v = round(nb / dt / 1e9, 4)
    sample = f"all {rows} rows x {w.cols} per step, split over {cores} threads"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64 / Box-Muller, 4*N(0,1))",
            "config": {"workload": "fused softmax, persistent form, fp32 [32768,1024]",
                       "rows": w.rows, "cols": w.cols, "sample": sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


SWEEP_DTYPE = {"relu_add_sum": "f32", "softmax": "f32", "softmax_bf16": "bf16",
               "softmax_offset": "f32", "softmax_bf16_offset": "bf16", "layernorm": "bf16"}


def sweep_markdown(path: str) -> str:
    """The form table: one line per shape with every form's (for LayerNorm,
    every kernel's) time, the fastest, the form AUTO took and its time."""
    lines = [json.loads(ln) for ln in open(path) if ln.startswith("{")]
    dev = {(d["device"], d["sms"]) for d in lines}
    out = ["| op | dtype | rows | cols | us per call by form (kernel) | fastest | AUTO form | "
           "AUTO us | AUTO / fastest | fastest, % of peak |",
           "|---|---|---|---|---|---|---|---|---|---|"]
    for d in lines:
        op = d["op"]
        times = "; ".join(f"{k} {v:.2f}" for k, v in d["us"].items())
        best = d["us"][d["fastest"]]
        name = op.replace('_bf16', '').replace('softmax_offset', 'softmax, x out of phase')
        out.append(f"| {name} | {SWEEP_DTYPE[op]} | {d['rows']} | {d['cols']} | "
                   f"{times} | {d['fastest']} | {d['auto']} | {d['auto_us']:.2f} | "
                   f"{d['auto_us'] / best:.3f} | {100 * d['best_frac']:.1f} |")
    head = [f"device: {', '.join(f'{n} ({m} SMs)' for n, m in sorted(dev))}", ""]
    return "\n".join(head + out)


HOST_ROWS_NS = 300_000  # softmax launches longer than this read and write host memory (e2e)


def launches_markdown(path: str) -> str:
    """Launches, total time and share per kernel of an ncu launch list.  The
    softmax kernel's end-to-end launches (rows in page-locked host memory,
    fr_softmax_host's direct form, about 790 us each) are listed apart from
    its device-resident launches (under 300 us)."""
    import csv
    import re as _re
    rows = [r for r in csv.reader(ln for ln in open(path) if ln.startswith('"'))]
    head, rows = rows[0], rows[1:]
    ki, ui, vi = head.index("Kernel Name"), head.index("Metric Unit"), head.index("Metric Value")
    scale = {"ns": 1.0, "nsecond": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}
    groups = {}
    for r in rows:
        ns = float(r[vi].replace(",", "")) * scale[r[ui]]
        name = _re.sub(r"^void ", "", r[ki])
        name = name.replace("fr::<unnamed>::", "")
        name = _re.sub(r"\(.*$", "", name)
        if name.startswith("softmax_warp_vec") and ns > HOST_ROWS_NS:
            name += " (rows in host memory, e2e)"
        g = groups.setdefault(name, [0, 0.0])
        g[0] += 1
        g[1] += ns
    total = sum(g[1] for g in groups.values())
    out = [f"{len(rows)} launches, {total / 1e3:.1f} us in all.", "",
           "| kernel | launches | total us | mean us | share |", "|---|---|---|---|---|"]
    for name, (n, t) in sorted(groups.items(), key=lambda kv: -kv[1][1]):
        out.append(f"| `{name}` | {n} | {t / 1e3:.1f} | {t / n / 1e3:.2f} | {100 * t / total:.1f} % |")
    return "\n".join(out)


def main():
    args = parse()
    if args.launches_md:
        print(launches_markdown(args.launches_md))
        return
    if args.sweep_md:
        print(sweep_markdown(args.sweep_md))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
