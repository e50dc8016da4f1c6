// C ABI of the fused row-reduction library: argument validation, reduction
// form selection and dispatch to the kernels.  Mirrors the generated wrapper
// of "Stax (4): GPU Codegen and Dynamic Shapes", section 9.7 (Listing 9.6):
// sizes and strides are checked before anything is enqueued, buffers are
// owned by the caller, every kernel goes onto the caller's stream in program
// order and nothing synchronises.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <mutex>
#include <vector>

#include "../../include/fr.h"
#include "launch.h"

namespace fr {

cudaError_t current_device_info(DevInfo *out) {
  constexpr int kMaxDev = 64;
  static DevInfo cache[kMaxDev];
  static bool have[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev) {
    std::lock_guard<std::mutex> lock(mu);
    if (have[dev]) {
      *out = cache[dev];
      return cudaSuccess;
    }
  }
  DevInfo d{};
  d.device = dev;
  if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev) {
    std::lock_guard<std::mutex> lock(mu);
    cache[dev] = d;
    have[dev] = true;
  }
  *out = d;
  return cudaSuccess;
}

}  // namespace fr

namespace {
thread_local fr_form g_last_form = FR_FORM_AUTO;
}  // namespace

namespace fr {
void set_last_form(int form) { g_last_form = static_cast<fr_form>(form); }
}  // namespace fr

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// rows >= 1, cols >= 1, ld >= cols and rows*ld*esize representable.
bool shape_ok(int64_t rows, int64_t cols, int64_t ld, int64_t esize) {
  if (rows < 1 || cols < 1 || ld < cols) return false;
  const int64_t lim = (INT64_C(1) << 62) / esize;
  return ld <= lim / rows;
}

// Rows of p and q (element size esize, leading dimensions lp, lq) share their
// offset modulo 32 bytes on every row.
bool same_phase(const void *p, int64_t lp, const void *q, int64_t lq, int64_t esize) {
  const int64_t d = static_cast<int64_t>(reinterpret_cast<uintptr_t>(p)) -
                    static_cast<int64_t>(reinterpret_cast<uintptr_t>(q));
  return (d % 32 == 0) && (((lp - lq) * esize) % 32 == 0);
}

fr_status device_ok(fr::DevInfo *info) {
  if (fr::current_device_info(info) != cudaSuccess) return FR_ERR_NO_DEVICE;
  if (info->cc_major != 10 || info->cc_minor != 3) return FR_ERR_NO_DEVICE;  // built for sm_103a
  return FR_OK;
}

// The split form of the softmax: a cluster of CTAs per row.  Rows in phase
// (x and y at the same offset within a 32-byte sector): the slices in
// registers, or for rows longer than split_loops allows the cluster whose
// CTAs stream their runs twice; rows out of phase: the cluster that stages
// its runs in shared memory.  FR_SOFTMAX_SPLIT=stage pins the staged cluster
// for every row, FR_SOFTMAX_SPLIT=loop the streaming one for every row in
// phase.
bool split_pinned(const char *v) {
  const char *e = getenv("FR_SOFTMAX_SPLIT");
  return e != nullptr && strcmp(e, v) == 0;
}
bool split_staged_pinned() { return split_pinned("stage"); }

// Rows in phase longer than 384 KiB: the streaming cluster.  Measured on
// GB300 (us per call, back to back; register cluster / streaming cluster):
// 256 KiB rows -- fp32 65537 columns: 608 rows 53.0 / 56.2, 1216 rows 99.2 /
// 106.2; bf16 131072: 304 rows 30.5 / 32.4, 1216 rows 102.1 / 112.2; 512 KiB
// rows -- fp32 131072: 152 rows 32.7 / 31.1, 608 rows 111.8 / 101.9; bf16
// 262144: 152 rows 35.5 / 32.3, 608 rows 119.9 / 104.2; 1 MiB rows -- fp32
// 262144: 152 rows 80.8 / 61.4, 304 rows 156.6 / 109.0.  The crossover lies
// between 256 and 512 KiB; the rule takes the middle.
bool split_loops(int64_t cols, int es) { return cols * es > (384 << 10); }

fr_status launched(cudaError_t e, fr_form form) {
  if (e != cudaSuccess) return FR_ERR_CUDA;
  g_last_form = form;
  return FR_OK;
}

// ---- form selection ---------------------------------------------------------
// Algorithm 9.1 of "Stax (4): GPU Codegen and Dynamic Shapes", section 9.6:
// every form that can run was timed on GB300 (152 SMs) over a grid of shapes
// (bench.py --only form_sweep; the table with every time is
// profiles/form_table_gb300.md), and each rule below puts its threshold at a
// measured crossover.  Thresholds on rows scale with the SM count.

// Shared memory one CTA may opt in to on sm_103 (227 KiB).
constexpr int kSm103SmemOptin = 232448;

// Example 1.1 and the sum of squares.  A row within one warp's registers:
// persistent.  Otherwise one warp per row streams the row (looped); that warp
// takes one dependent round trip per 32-byte vector a lane, so few long rows
// leave the GPU waiting on latency, and the split form (every SM on every
// row, plus a second small launch) wins.  Crossovers per input row of
// row_bytes: 64 KiB rows split up to 128 rows and loop from 512 (at 512 x
// 16384 fp32: looped 21.1 us, split 22.9; at 128: split 12.6, looped 18.3);
// 256 KiB rows split up to 1024 rows and tie at 2048 (1024 x 65536: split
// 84.3, looped 89.5; 2048: looped 153.3, split 154.9).
fr_form pick_ras(int64_t rows, int64_t cols, int sm_count, bool bf16 = false) {
  if (cols <= fr::ras_persistent_max_cols(bf16)) return FR_FORM_PERSISTENT;
  const int64_t row_bytes = cols * (bf16 ? 2 : 4);
  const int64_t sms = sm_count;
  if ((rows < 2 * sms && row_bytes >= (64 << 10)) || (rows < 12 * sms && row_bytes >= (256 << 10)))
    return FR_FORM_SPLIT;
  return FR_FORM_LOOPED;
}

// fp32 softmax, rows in phase.  Up to 1024 columns a warp per row; up to 8192
// a CTA per row at every row count (at fewer than 4 x SMs rows every form
// takes the launch time, 6.2-7 us; at 2432 x 8192: CTA per row 25.4 us,
// cluster 32.8); from 16384 a cluster of CTAs per row (16384: within 2 % of a
// CTA per row; 32768: 94.6 us against 105.9 at 2432 rows), its CTAs streaming
// their runs twice past 384 KiB rows (see split_loops), which beats the
// looped form at every row count measured (152 x 262144: 61.4 us, looped
// 76.0; 304 x 393216: 174.8 against 219.8; 64 x 1048576: 116.2 against
// 233.3; 16 x 4194304: 143.1 against 672.9).  Below 4 x SMs rows of
// 8192-16384 columns the two forms are within launch noise of each other
// (five sweeps, means: 304 x 16384 CTA per row 12.2 us, looped 11.3; 152 x
// 16384 8.8 against 9.5; 608 x 16384 16.7 against 20.3).  Rows out of phase
// (x and y at different offsets within a 32-byte sector): a CTA per row up to
// 32768 columns (the row in registers up to 4608, staged in shared memory
// beyond), then a cluster per row with its runs staged in shared memory (608
// x 65537: 62.6 us, looped 96.2; 608 x 131072: 148.0 against 191.4), looped
// past its reach.
fr_form pick_softmax(int64_t rows, int64_t cols, bool vec, int sm_count) {
  if (cols <= 1024) return FR_FORM_PERSISTENT;
  if (!vec) {  // rows of 16385 .. 32768 columns: a staged cluster per row under SMs / 4
              // rows (16 x 32768: 6.5 us, a CTA per row 7.6) and from 4 x SMs rows (its
              // 32 KiB runs against the CTA's 128 KiB, one an SM: 2432 x 32768 121.4
              // against 126.1), a CTA per row between (304 x 32768: 20.2 against 21.1)
    const int64_t sms = sm_count;
    if (cols <= fr::softmax_persistent_max_cols(false))
      return cols > 16384 && (rows * 4 < sms || rows >= 4 * sms) ? FR_FORM_SPLIT
                                                                 : FR_FORM_PERSISTENT;
    return cols <= fr::softmax_stage_split_max_cols(4) ? FR_FORM_SPLIT : FR_FORM_LOOPED;
  }
  return cols <= 8192 ? FR_FORM_PERSISTENT : FR_FORM_SPLIT;
}

// bf16 softmax.  Rows out of phase: up to 32768 columns a CTA per row, the row
// staged in shared memory (16384 x 4097: 48.3 us, looped 87.8; 4864 x 32768:
// 95.1 against 183.5), then a cluster per row with staged runs (608 x 65537:
// 32.9 us, looped 67.7; 2432 x 65537: 108.3 against 206.9), looped past its
// reach.  Rows in phase: up to 2048 columns a warp per row, up to 8192 a CTA
// per row; at 16384 the looped form from 4 x SMs rows (608: looped 9.4 us, CTA
// per row 10.5), a CTA per row below, and a CTA per row again from 8 x SMs
// rows, where the persistent form stages the row in shared memory (1216: 15.2
// us, looped 15.8; 16384: 153.2 against 165.6); at 32768 a CTA per row while
// the rows are no more than the SMs (152: 6.7 us against 7.7 for a cluster per
// row), else a cluster per row (2432 x 32768: 50.2 us, looped 55.3, CTA per
// row 73.9), its CTAs streaming their runs twice past 384 KiB rows (see
// split_loops; 304 x 393216: 90.7 us, looped 108.5; 64 x 1048576: 56.5
// against 138.5; 16 x 4194304: 80.8 against 424.3).
fr_form pick_softmax_bf16(int64_t rows, int64_t cols, bool vec, int sm_count) {
  if (cols <= 2048) return FR_FORM_PERSISTENT;
  if (!vec)
    return cols <= 32768                                 ? FR_FORM_PERSISTENT
           : cols <= fr::softmax_stage_split_max_cols(2) ? FR_FORM_SPLIT
                                                         : FR_FORM_LOOPED;
  if (cols <= 8192) return FR_FORM_PERSISTENT;
  if (cols <= 16384) {  // from 8 x SMs rows the persistent form stages rows in shared memory
    const int64_t sms = sm_count;
    return rows >= 8 * sms || rows < 4 * sms ? FR_FORM_PERSISTENT : FR_FORM_LOOPED;
  }
  return cols <= 32768 && rows <= sm_count ? FR_FORM_PERSISTENT : FR_FORM_SPLIT;
}

// LayerNorm (bf16 rows of 256 MiB, back to back).  Rows of C x T x 32
// columns whose CTAs have 4, 5, 7, 8 or 16 warps: the looped cluster kernel,
// gamma/beta in registers (4096: 84.7 us, 5120: 84.5, 10240: 84.5, 32768:
// 86.6); CTAs of 2, 3 or 6 warps (2048, 3072, 6144, 12288 columns: 86.5, 89.2,
// 88.9, 88.9 us) lose to the persistent row-group kernel (82.7, 88.6, 86.5,
// 85.2), which also takes the other rows whose gamma/beta fit in shared memory
// (768: 84.0 us, 1536: 84.1, 2560: 86.8); else the looped general cluster,
// ring or scalar kernel.
fr_form pick_layernorm(int64_t, int64_t cols, bool vec, bool aligned16, bool rows16,
                       int max_smem_optin) {
  const int t = fr::layernorm_cluster_full_threads(cols, aligned16);
  if (t != 0 && t != 64 && t != 96 && t != 192) return FR_FORM_LOOPED;
  if (fr::layernorm_rows_ok(cols, rows16, max_smem_optin)) return FR_FORM_PERSISTENT;
  if (fr::layernorm_cluster_ok(cols, aligned16) || fr::layernorm_ring_ok(cols, vec, max_smem_optin))
    return FR_FORM_LOOPED;
  return fr::layernorm_persistent_ok(cols, vec) ? FR_FORM_PERSISTENT : FR_FORM_LOOPED;
}

}  // namespace

extern "C" {

int fr_version(void) { return 100; }

const char *fr_status_string(fr_status s) {
  switch (s) {
    case FR_OK: return "FR_OK";
    case FR_ERR_INVALID_ARG: return "FR_ERR_INVALID_ARG";
    case FR_ERR_UNSUPPORTED_DTYPE: return "FR_ERR_UNSUPPORTED_DTYPE";
    case FR_ERR_UNSUPPORTED_FORM: return "FR_ERR_UNSUPPORTED_FORM";
    case FR_ERR_MISALIGNED: return "FR_ERR_MISALIGNED";
    case FR_ERR_WORKSPACE_TOO_SMALL: return "FR_ERR_WORKSPACE_TOO_SMALL";
    case FR_ERR_CUDA: return "FR_ERR_CUDA";
    case FR_ERR_DEVICE_DATA: return "FR_ERR_DEVICE_DATA";
    case FR_ERR_NO_DEVICE: return "FR_ERR_NO_DEVICE";
  }
  return "FR_ERR_UNKNOWN";
}

fr_form fr_last_form(void) { return g_last_form; }

fr_form fr_auto_form(fr_op op, fr_dtype dtype, int64_t rows, int64_t cols, int32_t sm_count) {
  if (rows < 1 || cols < 1 || sm_count < 1) return FR_FORM_AUTO;
  if (dtype != FR_F32 && dtype != FR_BF16) return FR_FORM_AUTO;
  switch (op) {
    case FR_OP_RELU_ADD_SUM: return pick_ras(rows, cols, sm_count, dtype == FR_BF16);
    case FR_OP_SUMSQ: return dtype == FR_F32 ? pick_ras(rows, cols, sm_count) : FR_FORM_AUTO;
    case FR_OP_SOFTMAX:
      return dtype == FR_F32 ? pick_softmax(rows, cols, true, sm_count)
                             : pick_softmax_bf16(rows, cols, true, sm_count);
    case FR_OP_LAYERNORM:
      return dtype == FR_BF16
                 ? pick_layernorm(rows, cols, cols % 16 == 0, true, cols % 8 == 0, kSm103SmemOptin)
                 : FR_FORM_AUTO;
    case FR_OP_XENT: return FR_FORM_LOOPED;
  }
  return FR_FORM_AUTO;
}

size_t fr_workspace_size(fr_op op, int64_t rows, int64_t cols, fr_dtype dtype, fr_form form) {
  if (rows < 1 || cols < 1) return 0;
  fr::DevInfo info;
  if (fr::current_device_info(&info) != cudaSuccess) return 0;
  switch (op) {
    case FR_OP_RELU_ADD_SUM: {
      const fr_form f =
          form == FR_FORM_AUTO ? pick_ras(rows, cols, info.sm_count, dtype == FR_BF16) : form;
      return f == FR_FORM_SPLIT ? fr::ras_split_workspace(rows, cols, info.sm_count) : 0;
    }
    case FR_OP_SUMSQ: {
      const fr_form f = form == FR_FORM_AUTO ? pick_ras(rows, cols, info.sm_count) : form;
      return f == FR_FORM_SPLIT ? fr::ras_split_workspace(rows, cols, info.sm_count) : 0;
    }
    case FR_OP_XENT: return fr::xent_workspace(rows, info.sm_count);
    default: return 0;
  }
}

fr_status fr_reduce_relu_add_sum(const void *a, const void *b, float *out, int64_t rows,
                                 int64_t cols, int64_t lda, int64_t ldb, fr_dtype dtype,
                                 float scale, fr_form form, void *workspace,
                                 size_t workspace_bytes, fr_stream_t stream) {
  if (dtype != FR_F32 && dtype != FR_BF16) return FR_ERR_UNSUPPORTED_DTYPE;
  const bool bf16 = dtype == FR_BF16;
  const int64_t es = bf16 ? 2 : 4;
  if (!a || !b || !out) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, lda, es) || !shape_ok(rows, cols, ldb, es)) return FR_ERR_INVALID_ARG;
  if (!aligned(a, es) || !aligned(b, es) || !aligned(out, 4)) return FR_ERR_MISALIGNED;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  const fr_form f = form == FR_FORM_AUTO ? pick_ras(rows, cols, info.sm_count, bf16) : form;
  const bool vec = same_phase(a, lda, b, ldb, es);
  const void *fa = a, *fb = b;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (f) {
    case FR_FORM_PERSISTENT:
      if (cols > fr::ras_persistent_max_cols(bf16)) return FR_ERR_UNSUPPORTED_FORM;
      return launched(fr::launch_ras_persistent(fa, fb, out, rows, cols, lda, ldb, scale, bf16,
                                                vec, s), f);
    case FR_FORM_LOOPED:
      return launched(fr::launch_ras_looped(fa, fb, out, rows, cols, lda, ldb, scale, bf16, vec,
                                            s), f);
    case FR_FORM_SPLIT: {
      if (rows > 65535) return FR_ERR_UNSUPPORTED_FORM;
      const size_t need = fr::ras_split_workspace(rows, cols, info.sm_count);
      if (!workspace || workspace_bytes < need) return FR_ERR_WORKSPACE_TOO_SMALL;
      if (!aligned(workspace, 16)) return FR_ERR_MISALIGNED;
      const int segs = fr::ras_split_segments(rows, cols, info.sm_count);
      return launched(fr::launch_ras_split(fa, fb, out, rows, cols, lda, ldb, scale, bf16, vec,
                                           static_cast<double *>(workspace), segs, s), f);
    }
    default: return FR_ERR_UNSUPPORTED_FORM;
  }
}

fr_status fr_reduce_sumsq(const void *x, float *out, int64_t rows, int64_t cols, int64_t ldx,
                          fr_dtype dtype, fr_epilogue epilogue, fr_form form, void *workspace,
                          size_t workspace_bytes, fr_stream_t stream) {
  if (dtype != FR_F32) return FR_ERR_UNSUPPORTED_DTYPE;
  if (!x || !out) return FR_ERR_INVALID_ARG;
  if (epilogue != FR_EPI_SUM && epilogue != FR_EPI_SQRT) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, ldx, 4)) return FR_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(out, 4)) return FR_ERR_MISALIGNED;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  // Same rule as Example 1.1: the kernels are the same with one input.
  const fr_form f = form == FR_FORM_AUTO ? pick_ras(rows, cols, info.sm_count) : form;
  const bool root = epilogue == FR_EPI_SQRT;
  const float *fx = static_cast<const float *>(x);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (f) {
    case FR_FORM_PERSISTENT:
      if (cols > fr::ras_persistent_max_cols()) return FR_ERR_UNSUPPORTED_FORM;
      return launched(fr::launch_sumsq_persistent(fx, out, rows, cols, ldx, root, s), f);
    case FR_FORM_LOOPED:
      return launched(fr::launch_sumsq_looped(fx, out, rows, cols, ldx, root, s), f);
    case FR_FORM_SPLIT: {
      if (rows > 65535) return FR_ERR_UNSUPPORTED_FORM;
      const size_t need = fr::ras_split_workspace(rows, cols, info.sm_count);
      if (!workspace || workspace_bytes < need) return FR_ERR_WORKSPACE_TOO_SMALL;
      if (!aligned(workspace, 16)) return FR_ERR_MISALIGNED;
      const int segs = fr::ras_split_segments(rows, cols, info.sm_count);
      return launched(fr::launch_sumsq_split(fx, out, rows, cols, ldx, root,
                                             static_cast<double *>(workspace), segs, s), f);
    }
    default: return FR_ERR_UNSUPPORTED_FORM;
  }
}

fr_status fr_softmax(const void *x, void *y, int64_t rows, int64_t cols, int64_t ldx,
                     int64_t ldy, fr_dtype dtype, fr_form form, fr_stream_t stream) {
  if (dtype != FR_F32 && dtype != FR_BF16) return FR_ERR_UNSUPPORTED_DTYPE;
  const int64_t esize = dtype == FR_F32 ? 4 : 2;
  if (!x || !y) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, ldx, esize) || !shape_ok(rows, cols, ldy, esize))
    return FR_ERR_INVALID_ARG;
  if (!aligned(x, esize) || !aligned(y, esize)) return FR_ERR_MISALIGNED;
  if (x == y && ldx != ldy) return FR_ERR_INVALID_ARG;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  const bool vec = same_phase(x, ldx, y, ldy, esize);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == FR_BF16) {
    const int64_t max_p = fr::softmax_bf16_persistent_max_cols(vec);
    const fr_form f =
        form == FR_FORM_AUTO ? pick_softmax_bf16(rows, cols, vec, info.sm_count) : form;
    const uint16_t *bx = static_cast<const uint16_t *>(x);
    uint16_t *by = static_cast<uint16_t *>(y);
    switch (f) {
      case FR_FORM_PERSISTENT:
        if (cols > max_p) return FR_ERR_UNSUPPORTED_FORM;
        return launched(fr::launch_softmax_bf16_persistent(bx, by, rows, cols, ldx, ldy, vec,
                                                                   info.sm_count, s), f);
      case FR_FORM_LOOPED:
        return launched(fr::launch_softmax_bf16_looped(bx, by, rows, cols, ldx, ldy, vec,
                                                       info.sm_count, s), f);
      case FR_FORM_SPLIT:
        if (cols <= 2048 || rows > 0x7fffffff / 8) return FR_ERR_UNSUPPORTED_FORM;
        if (vec && !split_staged_pinned() &&
            (split_pinned("loop") || split_loops(cols, 2) ||
             cols > fr::softmax_bf16_split_max_cols()))
          return launched(fr::launch_softmax_split_looped(bx, by, rows, cols, ldx, ldy, 2,
                                                          info.sm_count, s), f);
        if (vec && !split_staged_pinned())
          return launched(fr::launch_softmax_bf16_split(bx, by, rows, cols, ldx, ldy, s), f);
        if (cols > fr::softmax_stage_split_max_cols(2)) return FR_ERR_UNSUPPORTED_FORM;
        return launched(fr::launch_softmax_split_staged(bx, by, rows, cols, ldx, ldy, 2, s), f);
      default: return FR_ERR_UNSUPPORTED_FORM;
    }
  }
  const fr_form f = form == FR_FORM_AUTO ? pick_softmax(rows, cols, vec, info.sm_count) : form;
  const float *fx = static_cast<const float *>(x);
  float *fy = static_cast<float *>(y);
  switch (f) {
    case FR_FORM_PERSISTENT: {
      if (cols > fr::softmax_persistent_max_cols(vec)) return FR_ERR_UNSUPPORTED_FORM;
      // FR_SOFTMAX_KERNEL=async|plain pins the persistent kernel.  Default:
      // plain (measured on GB300, fp32 [32768, 1024] back to back: 40.2-41.2
      // us as programmatic dependents, 43.0 us without; the per-warp cp.async
      // ring runs half the warps per SM and took 49.0 us against 45.2 for
      // plain when both were ordinary launches).
      const char *pin = getenv("FR_SOFTMAX_KERNEL");
      const bool use_async = pin != nullptr && strcmp(pin, "async") == 0;
      const bool aligned16 = aligned(x, 16) && aligned(y, 16) && ldx % 4 == 0 && ldy % 4 == 0;
      if (use_async && fr::softmax_async_ok(cols, aligned16))
        return launched(fr::launch_softmax_async(fx, fy, rows, cols, ldx, ldy, info.sm_count, s), f);
      return launched(fr::launch_softmax_persistent(fx, fy, rows, cols, ldx, ldy, vec, s), f);
    }
    case FR_FORM_LOOPED:
      return launched(fr::launch_softmax_looped(fx, fy, rows, cols, ldx, ldy, vec, info.sm_count, s), f);
    case FR_FORM_SPLIT:
      if (cols <= 1024 || rows > 0x7fffffff / 8) return FR_ERR_UNSUPPORTED_FORM;
      if (vec && !split_staged_pinned() &&
          (split_pinned("loop") || split_loops(cols, 4) || cols > fr::softmax_split_max_cols()))
        return launched(fr::launch_softmax_split_looped(fx, fy, rows, cols, ldx, ldy, 4,
                                                        info.sm_count, s), f);
      if (vec && !split_staged_pinned())
        return launched(fr::launch_softmax_split(fx, fy, rows, cols, ldx, ldy, s), f);
      if (cols > fr::softmax_stage_split_max_cols(4)) return FR_ERR_UNSUPPORTED_FORM;
      return launched(fr::launch_softmax_split_staged(fx, fy, rows, cols, ldx, ldy, 4, s), f);
    default: return FR_ERR_UNSUPPORTED_FORM;
  }
}

size_t fr_softmax_host_workspace(int64_t cols, fr_dtype dtype, int64_t chunk_rows) {
  if (cols < 1 || chunk_rows < 1 || (dtype != FR_F32 && dtype != FR_BF16)) return 0;  // 0: direct
  const int64_t es = dtype == FR_F32 ? 4 : 2;
  return fr::host_pipeline_workspace(cols, es, es, chunk_rows);
}

namespace {
// The address at which the current device reaches page-locked host memory p
// (p itself under unified addressing), or nullptr when p is not page-locked.
void *host_device_ptr(const void *p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
bool page_locked(const void *p) { return host_device_ptr(p) != nullptr; }
}  // namespace

fr_status fr_softmax_host(const void *x_host, void *y_host, int64_t rows, int64_t cols,
                          fr_dtype dtype, int64_t chunk_rows, void *workspace,
                          size_t workspace_bytes, fr_stream_t stream) {
  if (dtype != FR_F32 && dtype != FR_BF16) return FR_ERR_UNSUPPORTED_DTYPE;
  const int64_t es = dtype == FR_F32 ? 4 : 2;
  if (!x_host || !y_host || chunk_rows < 0) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, cols, es)) return FR_ERR_INVALID_ARG;
  if (!aligned(x_host, es) || !aligned(y_host, es)) return FR_ERR_MISALIGNED;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  if (!page_locked(x_host) || !page_locked(y_host)) return FR_ERR_INVALID_ARG;
  if (chunk_rows == 0) {  // direct: the kernel reads and writes host memory over the host link
    const void *dx = host_device_ptr(x_host);
    void *dy = host_device_ptr(y_host);
    if (dtype == FR_F32 && cols <= 1024 && same_phase(dx, cols, dy, cols, 4) &&
        rows <= 0x7fffffffLL * 8)
      return launched(fr::launch_softmax_host_rows(static_cast<const float *>(dx),
                                                   static_cast<float *>(dy), rows, cols,
                                                   info.sm_count,
                                                   reinterpret_cast<cudaStream_t>(stream)),
                      FR_FORM_PERSISTENT);
    if (dtype == FR_BF16 && cols <= 2048 && same_phase(dx, cols, dy, cols, 2) &&
        rows <= 0x7fffffffLL * 8)
      return launched(fr::launch_softmax_bf16_host_rows(static_cast<const uint16_t *>(dx),
                                                        static_cast<uint16_t *>(dy), rows, cols,
                                                        info.sm_count,
                                                        reinterpret_cast<cudaStream_t>(stream)),
                      FR_FORM_PERSISTENT);
    return fr_softmax(dx, dy, rows, cols, cols, cols, dtype, FR_FORM_AUTO, stream);
  }
  if (chunk_rows > rows) chunk_rows = rows;
  if (!workspace || workspace_bytes < fr::host_pipeline_workspace(cols, es, es, chunk_rows))
    return FR_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 256)) return FR_ERR_MISALIGNED;
  fr_status kst = FR_OK;
  const fr::RowKernel kernel = [&](const void *x, void *y, int64_t nr, cudaStream_t s) {
    kst = fr_softmax(x, y, nr, cols, cols, cols, dtype, FR_FORM_AUTO,
                     reinterpret_cast<fr_stream_t>(s));
    return kst == FR_OK ? cudaSuccess : cudaErrorInvalidValue;
  };
  const cudaError_t e =
      fr::host_pipeline_run(x_host, y_host, rows, cols, es, es, chunk_rows, workspace,
                            reinterpret_cast<cudaStream_t>(stream), kernel);
  if (kst != FR_OK) return kst;
  return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

fr_status fr_layernorm(const void *x, const float *gamma, const float *beta, void *y,
                       float *mean, float *rstd, int64_t rows, int64_t cols, int64_t ldx,
                       int64_t ldy, float eps, fr_dtype dtype, fr_form form,
                       fr_stream_t stream) {
  if (dtype != FR_BF16) return FR_ERR_UNSUPPORTED_DTYPE;
  if (!x || !gamma || !beta || !y) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, ldx, 2) || !shape_ok(rows, cols, ldy, 2)) return FR_ERR_INVALID_ARG;
  if (!(eps >= 0.0f)) return FR_ERR_INVALID_ARG;
  if (!aligned(x, 2) || !aligned(y, 2) || !aligned(gamma, 4) || !aligned(beta, 4) ||
      (mean && !aligned(mean, 4)) || (rstd && !aligned(rstd, 4)))
    return FR_ERR_MISALIGNED;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  const bool vec = aligned(x, 32) && aligned(y, 32) && aligned(gamma, 32) && aligned(beta, 32) &&
                   ldx % 16 == 0 && ldy % 16 == 0 && cols % 16 == 0;
  const bool aligned16 = aligned(x, 32) && aligned(y, 32) && aligned(gamma, 16) &&
                         aligned(beta, 16) && ldx % 16 == 0 && ldy % 16 == 0;
  // row groups: 16-byte aligned rows (every row start: ld % 8 == 0) and gamma/beta
  const bool rows16 = aligned(x, 16) && aligned(y, 16) && aligned(gamma, 16) &&
                      aligned(beta, 16) && ldx % 8 == 0 && ldy % 8 == 0;
  const fr_form f = form == FR_FORM_AUTO
                       ? pick_layernorm(rows, cols, vec, aligned16, rows16, info.max_smem_optin)
                       : form;
  const uint16_t *bx = static_cast<const uint16_t *>(x);
  uint16_t *by = static_cast<uint16_t *>(y);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (f) {
    case FR_FORM_PERSISTENT: {
      // A row held on chip in one pass: by a group of warps, gamma/beta in
      // shared memory (default), or by one CTA with gamma/beta re-read from
      // L2 (FR_LAYERNORM_KERNEL=cta pins it).
      const char *pin = getenv("FR_LAYERNORM_KERNEL");
      const bool cta = pin != nullptr && strcmp(pin, "cta") == 0;
      if (!cta && fr::layernorm_rows_ok(cols, rows16, info.max_smem_optin))
        return launched(fr::launch_layernorm_rows(bx, gamma, beta, by, mean, rstd, rows, cols, ldx,
                                                  ldy, eps, info.sm_count, s), f);
      if (!fr::layernorm_persistent_ok(cols, vec)) return FR_ERR_UNSUPPORTED_FORM;
      return launched(fr::launch_layernorm_persistent(bx, gamma, beta, by, mean, rstd, rows, cols,
                                                      ldx, ldy, eps, s), f);
    }
    case FR_FORM_LOOPED: {
      // FR_LAYERNORM_KERNEL=cluster|ring|scalar pins one looped kernel (for
      // re-measuring the choice and for tests); unset = the first that fits.
      // Preference (measured): cluster, then staged ring, then scalar.
      const char *pin = getenv("FR_LAYERNORM_KERNEL");
      const bool any = pin == nullptr || pin[0] == 0;
      if ((any || strcmp(pin, "cluster") == 0) && fr::layernorm_cluster_ok(cols, aligned16))
        return launched(fr::launch_layernorm_cluster(bx, gamma, beta, by, mean, rstd, rows, cols,
                                                     ldx, ldy, eps, s), f);
      if ((any || strcmp(pin, "ring") == 0) && fr::layernorm_ring_ok(cols, vec, info.max_smem_optin))
        return launched(fr::launch_layernorm_ring(bx, gamma, beta, by, mean, rstd, rows, cols,
                                                  ldx, ldy, eps, info.sm_count,
                                                  info.max_smem_optin, s), f);
      return launched(fr::launch_layernorm_looped(bx, gamma, beta, by, mean, rstd, rows, cols, ldx,
                                                  ldy, eps, vec, info.sm_count,
                                                  info.max_smem_optin, s), f);
    }
    default: return FR_ERR_UNSUPPORTED_FORM;
  }
}

fr_status fr_xent(const void *logits, const int64_t *target, float *loss, float *loss_mean,
                  float *target_logit, int64_t *argmax, int64_t rows, int64_t cols, int64_t ld,
                  int64_t ignore_index, fr_dtype dtype, fr_form form, void *workspace,
                  size_t workspace_bytes, fr_stream_t stream) {
  if (dtype != FR_BF16 && dtype != FR_F32) return FR_ERR_UNSUPPORTED_DTYPE;
  const int64_t es = dtype == FR_F32 ? 4 : 2;
  if (!logits || !target) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, ld, es)) return FR_ERR_INVALID_ARG;
  if (!aligned(logits, es) || !aligned(target, 8) || (loss && !aligned(loss, 4)) ||
      (loss_mean && !aligned(loss_mean, 4)) || (target_logit && !aligned(target_logit, 4)) ||
      (argmax && !aligned(argmax, 8)))
    return FR_ERR_MISALIGNED;
  if (form != FR_FORM_AUTO && form != FR_FORM_LOOPED) return FR_ERR_UNSUPPORTED_FORM;
  if (cols >= (INT64_C(1) << 31)) return FR_ERR_UNSUPPORTED_FORM;  // 32-bit in-row indices
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  if (loss_mean) {
    if (!workspace || workspace_bytes < fr::xent_workspace(rows, info.sm_count))
      return FR_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return FR_ERR_MISALIGNED;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return launched(fr::launch_xent(logits, dtype == FR_F32, target, loss, loss_mean, target_logit,
                                  argmax, rows, cols, ld, ignore_index, workspace, info.sm_count,
                                  info.max_smem_optin, s),
                  FR_FORM_LOOPED);
}

fr_status fr_xent_workspace_init(void *workspace, size_t workspace_bytes, fr_stream_t stream) {
  if (!workspace) return FR_ERR_INVALID_ARG;
  if (workspace_bytes < 16) return FR_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 16)) return FR_ERR_MISALIGNED;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  return fr::launch_xent_workspace_init(workspace, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FR_OK
             : FR_ERR_CUDA;
}

fr_status fr_xent_mean_from_parts(const void *workspace, float *loss_mean, fr_stream_t stream) {
  if (!workspace || !loss_mean) return FR_ERR_INVALID_ARG;
  if (!aligned(workspace, 16) || !aligned(loss_mean, 4)) return FR_ERR_MISALIGNED;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  return fr::launch_xent_mean_from_parts(workspace, loss_mean,
                                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FR_OK
             : FR_ERR_CUDA;
}

namespace {

fr::XentConfig from_c(const fr_xent_config &c) {
  return fr::XentConfig{c.threads, c.vectors, c.stages, c.ctas_per_sm};
}
fr_xent_config to_c(const fr::XentConfig &c) {
  return fr_xent_config{c.threads, c.vectors, c.stages, c.ctas_per_sm};
}

// Median time (ms) of `reps` launches of configuration cfg after one warm-up
// launch; +inf when the configuration cannot run.
double time_xent_config(const fr::XentConfig &cfg, const uint16_t *logits, const int64_t *target,
                        float *loss, int64_t rows, int64_t cols, int64_t ld,
                        int64_t ignore_index, int reps, const fr::DevInfo &info,
                        cudaStream_t s) {
  const double inf = std::numeric_limits<double>::infinity();
  if (fr::xent_config_check(cfg, info.max_smem_optin) != cudaSuccess) {
    cudaGetLastError();
    return inf;
  }
  auto launch = [&]() {
    return fr::launch_xent_config(cfg, logits, target, loss, nullptr, nullptr, rows, cols, ld,
                                  ignore_index, nullptr, info.sm_count, info.max_smem_optin, s);
  };
  if (launch() != cudaSuccess) {
    cudaGetLastError();
    return inf;
  }
  std::vector<cudaEvent_t> ev(2 * static_cast<size_t>(reps));
  for (auto &e : ev)
    if (cudaEventCreate(&e) != cudaSuccess) return inf;
  bool ok = true;
  for (int r = 0; r < reps && ok; ++r) {
    ok = cudaEventRecord(ev[2 * r], s) == cudaSuccess && launch() == cudaSuccess &&
         cudaEventRecord(ev[2 * r + 1], s) == cudaSuccess;
  }
  std::vector<double> ms;
  if (ok && cudaStreamSynchronize(s) == cudaSuccess) {
    for (int r = 0; r < reps; ++r) {
      float t = 0.0f;
      if (cudaEventElapsedTime(&t, ev[2 * r], ev[2 * r + 1]) != cudaSuccess) {
        ok = false;
        break;
      }
      ms.push_back(t);
    }
  } else {
    ok = false;
  }
  for (auto &e : ev) cudaEventDestroy(e);
  if (!ok) {
    cudaGetLastError();
    return inf;
  }
  std::sort(ms.begin(), ms.end());
  return ms[ms.size() / 2];
}

int ilog2(int v) {
  int k = 0;
  while ((1 << (k + 1)) <= v) ++k;
  return k;
}

}  // namespace

fr_status fr_xent_get_config(int64_t rows, int64_t cols, int64_t ld, fr_xent_config *out) {
  if (!out || !shape_ok(rows, cols, ld, 2)) return FR_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FR_ERR_NO_DEVICE;
  }
  fr::XentConfig c = fr::xent_default_config();
  fr::xent_recorded_config(dev, rows, cols, ld, &c);
  *out = to_c(c);
  return FR_OK;
}

fr_status fr_xent_set_config(int64_t rows, int64_t cols, int64_t ld, const fr_xent_config *cfg) {
  if (!shape_ok(rows, cols, ld, 2)) return FR_ERR_INVALID_ARG;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  if (cfg == nullptr) {
    fr::xent_record_config(info.device, rows, cols, ld, nullptr);
    return FR_OK;
  }
  const fr::XentConfig c = from_c(*cfg);
  const cudaError_t e = fr::xent_config_check(c, info.max_smem_optin);
  if (e == cudaErrorInvalidValue) return FR_ERR_INVALID_ARG;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FR_ERR_UNSUPPORTED_FORM;
  }
  fr::xent_record_config(info.device, rows, cols, ld, &c);
  return FR_OK;
}

fr_status fr_xent_tune(const void *logits, const int64_t *target, float *loss, int64_t rows,
                       int64_t cols, int64_t ld, int64_t ignore_index, fr_dtype dtype,
                       double eps, int32_t reps, fr_stream_t stream, fr_xent_config *out,
                       int32_t *evaluations, float *best_ms) {
  if (dtype != FR_BF16) return FR_ERR_UNSUPPORTED_DTYPE;
  if (!logits || !target) return FR_ERR_INVALID_ARG;
  if (!shape_ok(rows, cols, ld, 2)) return FR_ERR_INVALID_ARG;
  if (!(eps > 0.0 && eps < 1.0) || reps < 1 || reps > 1000) return FR_ERR_INVALID_ARG;
  if (!aligned(logits, 2) || !aligned(target, 8) || (loss && !aligned(loss, 4)))
    return FR_ERR_MISALIGNED;
  if (cols >= (INT64_C(1) << 31)) return FR_ERR_UNSUPPORTED_FORM;
  fr::DevInfo info;
  if (fr_status st = device_ok(&info)) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t *lg = static_cast<const uint16_t *>(logits);
  if (evaluations) *evaluations = 0;
  if (best_ms) *best_ms = 0.0f;

  fr::XentConfig best{};
  if (fr::xent_recorded_config(info.device, rows, cols, ld, &best)) {  // Algorithm 9.1, line 1
    if (out) *out = to_c(best);
    return FR_OK;
  }
  int evals = 0;
  auto cost = [&](const fr::XentConfig &c) {
    ++evals;
    return time_xent_config(c, lg, target, loss, rows, cols, ld, ignore_index, reps, info, s);
  };
  // Algorithm 9.1: the fastest of a small candidate set -- the default (the
  // warp-per-row kernel), its 4-vector point, and the ring points the kernel
  // was developed with.
  const fr::XentConfig cands[] = {fr::xent_default_config(), {32, 4, 1, 4},   {128, 8, 2, 4},
                                  {256, 4, 4, 2},            {512, 4, 4, 1},  {128, 4, 4, 4},
                                  {256, 2, 8, 2},            {256, 8, 2, 2}};
  double t_best = std::numeric_limits<double>::infinity(), t_ring = t_best;
  fr::XentConfig ring{};
  for (const fr::XentConfig &c : cands) {
    const double t = cost(c);
    if (t < t_best) {
      t_best = t;
      best = c;
    }
    if (c.threads >= 128 && t < t_ring) {
      t_ring = t;
      ring = c;
    }
  }
  if (!std::isfinite(t_best)) return FR_ERR_CUDA;  // nothing could run
  double t_final = t_best;
  if (std::isfinite(t_ring)) {
    // Algorithm 9.2 from the fastest ring point over the ring's box of log2
    // parameters (the warp-per-row points lie outside it)
    const int lo[4] = {7, 0, 1, 0}, hi[4] = {10, 3, 3, 4};
    int c[4] = {ilog2(ring.threads), ilog2(ring.vectors), ilog2(ring.stages),
                ilog2(ring.ctas_per_sm)};
    const fr::CdResult r = fr::coordinate_descent(4, lo, hi, c, eps, [&](const int *q) {
      const fr::XentConfig x{1 << q[0], 1 << q[1], 1 << q[2], 1 << q[3]};
      if (x.threads == ring.threads && x.vectors == ring.vectors && x.stages == ring.stages &&
          x.ctas_per_sm == ring.ctas_per_sm)
        return t_ring;  // already timed
      return cost(x);
    });
    if (r.t < t_best) {
      best = fr::XentConfig{1 << c[0], 1 << c[1], 1 << c[2], 1 << c[3]};
      t_final = r.t;
    }
  }
  fr::xent_record_config(info.device, rows, cols, ld, &best);
  if (out) *out = to_c(best);
  if (evaluations) *evaluations = evals;
  if (best_ms) *best_ms = static_cast<float>(t_final);
  return cudaGetLastError() == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

fr_status fr_check_device_error(fr_stream_t stream, int32_t *code) {
  int v = 0;
  if (fr::device_error_read_and_clear(reinterpret_cast<cudaStream_t>(stream), &v) != cudaSuccess)
    return FR_ERR_CUDA;
  if (code) *code = v;
  return v == 0 ? FR_OK : FR_ERR_DEVICE_DATA;
}

}  // extern "C"
