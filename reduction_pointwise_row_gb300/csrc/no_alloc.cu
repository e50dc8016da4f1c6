// A split-form relu_add_sum that needs no caller workspace and allocates
// nothing.
//
// fr_reduce_relu_add_sum's split form writes its per-segment partial sums to
// a workspace the caller allocates.  Some callers cannot allocate device memory
// at the point where they launch: code that runs inside a host framework which
// owns every device allocation (its own pool and accounting) and forbids raw
// cudaMalloc in an operator callback, latency-critical paths where cudaMalloc /
// cudaFree may synchronise the whole device, and interfaces that simply have no
// way to hand a workspace pointer through.  For them this file keeps the
// partials in a fixed array in the library's own device memory.
//
// The array is a file-scope static __device__ variable, so every GPU that loads
// the library holds FR_STATIC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in); the device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on it, and passed to the kernels.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fr.h"
#include "launch.h"

namespace {

constexpr int64_t kScratchDoubles = FR_STATIC_SCRATCH_BYTES / sizeof(double);

// Shared by every call on a device; holds the last call's partials.
static __device__ __align__(256) double g_split_scratch[kScratchDoubles];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
double *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_split_scratch on `dev` (the current device), resolved
// once per device.  Returns nullptr if the lookup fails.
double *scratch_on(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // reset the runtime's last-error so it does not leak into later calls
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<double *>(p);
  }
  return g_scratch_ptr[dev];
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" fr_status fr_reduce_relu_add_sum_split_static(const void *a, const void *b,
                                                         float *out, int64_t rows, int64_t cols,
                                                         int64_t lda, int64_t ldb, fr_dtype dtype,
                                                         float scale, fr_stream_t stream) {
  if (dtype != FR_F32) return FR_ERR_UNSUPPORTED_DTYPE;
  if (!a || !b || !out) return FR_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1 || lda < cols || ldb < cols) return FR_ERR_INVALID_ARG;
  const int64_t lim = (INT64_C(1) << 62) / 4;
  if (lda > lim / rows || ldb > lim / rows) return FR_ERR_INVALID_ARG;
  if (!aligned4(a) || !aligned4(b) || !aligned4(out)) return FR_ERR_MISALIGNED;
  if (rows > 65535) return FR_ERR_UNSUPPORTED_FORM;
  fr::DevInfo info;
  if (fr::current_device_info(&info) != cudaSuccess) return FR_ERR_NO_DEVICE;
  if (info.cc_major != 10 || info.cc_minor != 3) return FR_ERR_NO_DEVICE;
  const int segments = fr::ras_split_segments(rows, cols, info.sm_count);
  // Beyond the fixed array: refuse before touching the device.
  if (rows * static_cast<int64_t>(segments) > kScratchDoubles) return FR_ERR_WORKSPACE_TOO_SMALL;
  double *scratch = scratch_on(info.device);
  if (scratch == nullptr) return FR_ERR_CUDA;
  // Stage 1 writes every one of the rows*segments partials before stage 2
  // reads them, so nothing in the array has to be cleared first.
  const int64_t d = static_cast<int64_t>(reinterpret_cast<uintptr_t>(a)) -
                    static_cast<int64_t>(reinterpret_cast<uintptr_t>(b));
  const bool vec = (d % 32 == 0) && (((lda - ldb) * 4) % 32 == 0);
  cudaError_t e = fr::launch_ras_split(a, b, out, rows, cols, lda, ldb, scale, false, vec,
                                       scratch, segments, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FR_ERR_CUDA;
  fr::set_last_form(FR_FORM_SPLIT);
  return FR_OK;
}
