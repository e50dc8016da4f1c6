"""Host-side checks that need no GPU: the library builds for sm_103a, loads,
and exports every entry point include/fr.h declares; the traffic model is
pinned to the element counts printed for the fused-softmax demo."""
import json
import os
import re


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fr_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for must in ("fr_reduce_relu_add_sum", "fr_reduce_sumsq", "fr_softmax", "fr_layernorm",
                 "fr_xent",
                 "fr_workspace_size", "fr_check_device_error", "fr_status_string"):
        assert must in names


def test_library_builds_loads_and_exports_every_symbol():
    import reduction_pointwise_row_gb300 as fr
    fr.build()
    lib = fr.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in fr.SIGNATURES, f"binding lacks a signature for {name}"
    assert fr.fr_version() >= 100


def test_status_strings():
    import reduction_pointwise_row_gb300 as fr
    lib = fr.lib()
    for code, name in fr.STATUS.items():
        assert lib.fr_status_string(code).decode() == name


def test_built_for_sm103a_only():
    log = open(os.path.join(ROOT, "reduction_pointwise_row_gb300", "_lib", "ptxas.log")).read()
    assert "sm_103a" in log and "sm_100" not in log.replace("sm_100-class", "")


def test_no_register_spills():
    """No kernel spills a register (-Xptxas -v): a spilling configuration
    counts as one that exceeds the resources (Definition 9.2 of Stax (4),
    section 9.6) and is not built."""
    log = open(os.path.join(ROOT, "reduction_pointwise_row_gb300", "_lib", "ptxas.log")).read()
    blocks = re.split(r"Compiling entry function '", log)[1:]
    assert blocks
    spilling = []
    for b in blocks:
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", b)
        if m and (int(m.group(1)) or int(m.group(2))):
            spilling.append((b.split("'")[0], int(m.group(1)), int(m.group(2))))
    assert not spilling, spilling


def test_traffic_model_matches_lecture_counts():
    from reduction_pointwise_row_gb300 import traffic
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "softmax_traffic_1823x781.json")))
    r, w = traffic.naive_softmax_elements(g["rows"], g["cols"])
    assert (r, w) == (g["naive_five_kernel"]["elements_read"],
                      g["naive_five_kernel"]["elements_written"])
    fr_, fw = traffic.fused_softmax_elements(g["rows"], g["cols"])
    assert (fr_, fw) == (g["fused"]["elements_read"], g["fused"]["elements_written"])
    assert round((r + w) / (fr_ + fw), 2) == g["ratio_printed"]


def test_algorithmic_bytes_of_the_five_workloads():
    from reduction_pointwise_row_gb300 import traffic
    assert traffic.algorithmic_bytes("relu_add_sum", 64, 128) == 65792
    assert traffic.algorithmic_bytes("softmax", 32768, 1024) == 268435456
    assert traffic.algorithmic_bytes("layernorm", 4096, 32768) == 537165824
    assert traffic.algorithmic_bytes("relu_add_sum", 8, 33554432) == 2147483680
    assert traffic.algorithmic_bytes("xent", 8192, 50257) == 823508996


def test_no_cpu_fallback_in_product():
    """The product package never imports the oracle or the generators."""
    pkg = os.path.join(ROOT, "reduction_pointwise_row_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "oracle.c" not in src, f


def test_argument_validation_needs_no_device():
    """Null pointers, bad shapes, dtypes and misaligned pointers are rejected on
    the host before any CUDA call, so these run without a GPU."""
    import ctypes
    import reduction_pointwise_row_gb300 as fr
    lib = fr.lib()
    P = ctypes.c_void_p
    good, odd = P(0x10000), P(0x10001)
    # relu_add_sum
    assert lib.fr_reduce_relu_add_sum(None, good, good, 4, 8, 8, 8, 0, 2.0, 0, None, 0, None) == 1
    assert lib.fr_reduce_relu_add_sum(good, good, good, 0, 8, 8, 8, 0, 2.0, 0, None, 0, None) == 1
    assert lib.fr_reduce_relu_add_sum(good, good, good, 4, 8, 7, 8, 0, 2.0, 0, None, 0, None) == 1
    assert lib.fr_reduce_relu_add_sum(good, good, good, 4, 8, 8, 8, 2, 2.0, 0, None, 0, None) == 2
    # bf16 inputs must be 2-byte aligned
    assert lib.fr_reduce_relu_add_sum(odd, good, good, 4, 8, 8, 8, 1, 2.0, 0, None, 0, None) == 4
    assert lib.fr_reduce_relu_add_sum(odd, good, good, 4, 8, 8, 8, 0, 2.0, 0, None, 0, None) == 4
    big = 1 << 40
    assert lib.fr_reduce_relu_add_sum(good, good, good, big, big, big, big, 0, 2.0, 0, None, 0,
                                      None) == 1
    # sum of squares / row L2 norm
    assert lib.fr_reduce_sumsq(None, good, 4, 8, 8, 0, 0, 0, None, 0, None) == 1
    assert lib.fr_reduce_sumsq(good, good, 4, 8, 7, 0, 0, 0, None, 0, None) == 1
    assert lib.fr_reduce_sumsq(good, good, 4, 8, 8, 1, 0, 0, None, 0, None) == 2
    assert lib.fr_reduce_sumsq(good, good, 4, 8, 8, 0, 2, 0, None, 0, None) == 1  # epilogue
    assert lib.fr_reduce_sumsq(odd, good, 4, 8, 8, 0, 1, 0, None, 0, None) == 4
    # softmax
    assert lib.fr_softmax(good, good, 4, 0, 8, 8, 0, 0, None) == 1
    assert lib.fr_softmax(good, good, 4, 8, 8, 8, 2, 0, None) == 2      # no such dtype
    assert lib.fr_softmax(odd, good, 4, 8, 8, 8, 1, 0, None) == 4       # bf16, odd address
    assert lib.fr_softmax(good, good, 4, 8, 8, 16, 0, 0, None) == 1   # in place, ldx != ldy
    assert lib.fr_softmax(good, odd, 4, 8, 8, 8, 0, 0, None) == 4
    # layernorm
    assert lib.fr_layernorm(good, good, good, good, None, None, 4, 8, 8, 8, 1e-5, 0, 0, None) == 2
    assert lib.fr_layernorm(good, None, good, good, None, None, 4, 8, 8, 8, 1e-5, 1, 0, None) == 1
    assert lib.fr_layernorm(good, good, good, good, None, None, 4, 8, 8, 8, -1.0, 1, 0, None) == 1
    assert lib.fr_layernorm(odd, good, good, good, None, None, 4, 8, 8, 8, 1e-5, 1, 0, None) == 4
    # xent
    assert lib.fr_xent(good, None, None, None, None, None, 4, 8, 8, -100, 1, 0, None, 0, None) == 1
    assert lib.fr_xent(good, good, None, None, None, None, 4, 8, 8, -100, 2, 0, None, 0, None) == 2
    # fp32 logits must be 4-byte aligned (bf16 ones 2-byte)
    assert lib.fr_xent(P(0x10002), good, None, None, None, None, 4, 8, 8, -100, 0, 0, None, 0,
                       None) == 4
    assert lib.fr_xent(good, P(0x10004), None, None, None, None, 4, 8, 8, -100, 1, 0, None, 0,
                       None) == 4
    assert lib.fr_xent(good, good, None, None, None, None, 4, 8, 8, -100, 1, 3, None, 0, None) == 3


def test_every_overlapped_kernel_waits_for_its_predecessor():
    """Launches with the programmatic-overlap attribute (launch_k, launch_pdl)
    may start a kernel while the one before it still runs; such a kernel must
    begin with pdl_enter() (griddepcontrol.wait) before touching memory.  Every
    kernel does, except those launched only without the attribute, listed here."""
    import glob
    import re
    plain_only = {"layernorm_persistent", "layernorm_looped_scalar", "layernorm_ring",
                  "layernorm_cluster", "softmax_warp_scalar", "softmax_warp_async",
                  "softmax_bf16_warp_scalar"}
    seen = set()
    for f in glob.glob(os.path.join(ROOT, "reduction_pointwise_row_gb300", "csrc", "*.cu")):
        s = open(f).read()
        for m in re.finditer(r"__global__", s):
            brace = s.index("{", m.end())
            head = re.sub(r"__launch_bounds__\([^)]*\)", "", s[m.end():brace])
            name = re.findall(r"\b([A-Za-z_]\w*)\s*\(", head)[0]
            seen.add(name)
            body = s[brace + 1:brace + 600]
            statements = [t.strip() for t in body.split(";")]
            waits = any(t.startswith("pdl_enter()") for t in statements[:2])
            if name in plain_only:
                # launched only with <<<>>>, cudaLaunchKernel or without the attribute
                assert not re.search(r"launch_(k|pdl)\(\s*(&)?" + name + r"\b", s), name
            else:
                assert waits, f"{name} ({os.path.basename(f)}) does not begin with pdl_enter()"
    assert plain_only <= seen


def test_xent_workspace_init_validates_before_any_device_call():
    import ctypes
    import reduction_pointwise_row_gb300 as fr
    lib = fr.lib()
    P = ctypes.c_void_p
    assert lib.fr_xent_workspace_init(None, 64, None) == 1          # NULL
    assert lib.fr_xent_workspace_init(P(0x10000), 8, None) == 5     # smaller than the ticket
    assert lib.fr_xent_workspace_init(P(0x10008), 64, None) == 4    # not 16-byte aligned


def test_traffic_model_counts_each_dtype_by_its_width():
    """Each op's algorithmic bytes: inputs read once and outputs written once,
    at the width of their dtype (bf16 rows move half the bytes of fp32 rows;
    the per-row vectors are the same)."""
    from reduction_pointwise_row_gb300 import traffic as t
    R, C = 300, 1000
    assert t.algorithmic_bytes("relu_add_sum", R, C) == 2 * R * C * 4 + 4 * R
    assert t.algorithmic_bytes("relu_add_sum_bf16", R, C) == 2 * R * C * 2 + 4 * R
    assert t.algorithmic_bytes("softmax", R, C) == 2 * t.algorithmic_bytes("softmax_bf16", R, C)
    assert (t.algorithmic_bytes("xent_f32", R, C) - t.algorithmic_bytes("xent", R, C)
            == R * C * 2)
    assert t.algorithmic_bytes("sumsq", R, C) == R * C * 4 + 4 * R
    assert t.algorithmic_bytes("layernorm", R, C) == 4 * R * C + 8 * C + 8 * R
