// Example 1.1 of "Stax (4): GPU Codegen and Dynamic Shapes" (section 9.2,
// Listing 9.1):  out[x] = sum_r scale * relu(a[x, r] + b[x, r])  in its three
// reduction forms (section 9.4):
//
//   persistent  one warp per row, the whole row loaded in one pass (all of a
//               lane's loads in flight before any arithmetic), cols <= 1024;
//   looped      one warp per row streaming 32-byte vectors with a register
//               accumulator (the r0_offset loop of Listing 9.4);
//   split       (few, long rows) stage 1: grid (segments x rows), each CTA sums
//               one fixed segment of a row into an fp64 partial; stage 2: one
//               warp per row adds the partials in a fixed order.  Section 9.4 (3)
//               splits the reduction when there are too few outputs to fill the
//               GPU; here the segment count fills every SM of the device.
//
// Arithmetic: a + b in fp32 (Listing 9.1 tmp2), relu keeping NaN (tmp4,
// PropagateNan.ALL), times scale in fp32 (tmp6).  Runs of at most 8*U terms
// are summed in fp32 and then added into an fp64 accumulator; the warp/CTA
// combine and the cross-CTA combine are fp64 in a fixed tree order, so a given
// shape on a given device model always gives the same bits.
#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

constexpr int kRowThreads = 256;  // warp-per-row forms: 8 rows per CTA
constexpr int kPersistNV = 4;     // 32-byte vectors per lane in the persistent form
constexpr int kSplitThreads = 256;
constexpr int kSplitU = 2;        // vector pairs in flight per thread per iteration

__device__ __forceinline__ float term(float a, float b, float scale) {
  return relu_nan(a + b) * scale;
}

__device__ __forceinline__ float terms_v8(const V8 &va, const V8 &vb, float scale) {
  float t = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) t += term(__uint_as_float(va.w[j]), __uint_as_float(vb.w[j]), scale);
  return t;
}

// Warp-per-row form.  VEC: a and b rows share their offset modulo 32 bytes, so
// one head/body/tail split serves both; otherwise every element is a scalar
// (still coalesced: lane-strided).
template <bool VEC, bool LOOP>
__global__ void __launch_bounds__(kRowThreads)
ras_warp_row(const float *__restrict__ a, const float *__restrict__ b, float *__restrict__ out,
             int64_t rows, int64_t cols, int64_t lda, int64_t ldb, float scale) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float *pa = a + row * lda;
  const float *pb = b + row * ldb;
  double acc = 0.0;
  if constexpr (VEC) {
    const RowSplit sp = row_split(pa, cols, 4);
    float s = 0.0f;  // head and tail: at most 7 + 7 scalars, one per lane
    if (lane < sp.head) {
      s = term(ld_stream_f32(pa + lane), ld_stream_f32(pb + lane), scale);
    } else if (lane < sp.head + sp.tail) {
      const int64_t i = sp.head + sp.nvec * 8 + (lane - sp.head);
      s = term(ld_stream_f32(pa + i), ld_stream_f32(pb + i), scale);
    }
    acc = s;
    const float *va = pa + sp.head;
    const float *vb = pb + sp.head;
    for (int64_t base = 0; base < sp.nvec; base += 32 * kPersistNV) {
      V8 xa[kPersistNV], xb[kPersistNV];
#pragma unroll
      for (int k = 0; k < kPersistNV; ++k) {
        const int64_t vi = base + lane + 32 * k;
        if (vi < sp.nvec) {
          xa[k] = ld_stream_v8(va + vi * 8);
          xb[k] = ld_stream_v8(vb + vi * 8);
        }
      }
      float t = 0.0f;
#pragma unroll
      for (int k = 0; k < kPersistNV; ++k)
        if (base + lane + 32 * k < sp.nvec) t += terms_v8(xa[k], xb[k], scale);
      acc += static_cast<double>(t);
      if constexpr (!LOOP) break;
    }
  } else {
    for (int64_t base = 0; base < cols; base += 32 * 8) {
      float t = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t i = base + lane + 32 * k;
        if (i < cols) t += term(ld_stream_f32(pa + i), ld_stream_f32(pb + i), scale);
      }
      acc += static_cast<double>(t);
      if constexpr (!LOOP) {
        if (base + 32 * 8 >= 1024) break;
      }
    }
  }
  acc = warp_sum_f64(acc);
  if (lane == 0) out[row] = static_cast<float>(acc);
}

// Split form, stage 1: CTA (seg, row) sums its segment of the row's body
// vectors (segment 0 also takes the head scalars, the last segment the tail).
template <bool VEC>
__global__ void __launch_bounds__(kSplitThreads)
ras_split_stage1(const float *__restrict__ a, const float *__restrict__ b, int64_t cols,
                 int64_t lda, int64_t ldb, float scale, double *__restrict__ partials, int S) {
  const int seg = blockIdx.x;
  const int64_t row = blockIdx.y;
  const int tid = threadIdx.x;
  const float *pa = a + row * lda;
  const float *pb = b + row * ldb;
  const RowSplit sp = VEC ? row_split(pa, cols, 4) : RowSplit{0, cols, 0};
  const int64_t per = (sp.nvec + S - 1) / S;
  const int64_t lo = seg * per;
  const int64_t hi = lo + per < sp.nvec ? lo + per : sp.nvec;
  double acc = 0.0;
  if constexpr (VEC) {
    const float *va = pa + sp.head;
    const float *vb = pb + sp.head;
    for (int64_t base = lo; base < hi; base += kSplitThreads * kSplitU) {
      V8 xa[kSplitU], xb[kSplitU];
#pragma unroll
      for (int u = 0; u < kSplitU; ++u) {
        const int64_t vi = base + tid + kSplitThreads * u;
        if (vi < hi) {
          xa[u] = ld_stream_v8(va + vi * 8);
          xb[u] = ld_stream_v8(vb + vi * 8);
        }
      }
      float t = 0.0f;
#pragma unroll
      for (int u = 0; u < kSplitU; ++u)
        if (base + tid + kSplitThreads * u < hi) t += terms_v8(xa[u], xb[u], scale);
      acc += static_cast<double>(t);
    }
    if (seg == 0 && tid < sp.head)
      acc += static_cast<double>(term(ld_stream_f32(pa + tid), ld_stream_f32(pb + tid), scale));
    if (seg == S - 1 && tid < sp.tail) {
      const int64_t i = sp.head + sp.nvec * 8 + tid;
      acc += static_cast<double>(term(ld_stream_f32(pa + i), ld_stream_f32(pb + i), scale));
    }
  } else {
    for (int64_t base = lo; base < hi; base += kSplitThreads * 8) {
      float t = 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = base + tid + kSplitThreads * u;
        if (i < hi) t += term(ld_stream_f32(pa + i), ld_stream_f32(pb + i), scale);
      }
      acc += static_cast<double>(t);
    }
  }
  acc = warp_sum_f64(acc);
  __shared__ double warp_part[kSplitThreads / 32];
  if ((tid & 31) == 0) warp_part[tid >> 5] = acc;
  __syncthreads();
  if (tid == 0) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kSplitThreads / 32; ++w) t += warp_part[w];
    partials[row * S + seg] = t;
  }
}

// Split form, stage 2: one warp per row adds its S partials in a fixed order.
__global__ void __launch_bounds__(kRowThreads)
ras_split_stage2(const double *__restrict__ partials, float *__restrict__ out, int64_t rows,
                 int S) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  double t = 0.0;
  for (int k = lane; k < S; k += 32) t += partials[row * S + k];
  t = warp_sum_f64(t);
  if (lane == 0) out[row] = static_cast<float>(t);
}

unsigned warp_row_grid(int64_t rows) {
  return static_cast<unsigned>((rows + kRowThreads / 32 - 1) / (kRowThreads / 32));
}

}  // namespace

int64_t ras_persistent_max_cols() { return 32 * 8 * kPersistNV; }

int ras_split_segments(int64_t rows, int64_t cols, int sm_count) {
  // Enough CTAs for four per SM (one wave at the kernel's occupancy), but no
  // segment shorter than 512 vectors (16 KiB of each input).
  int64_t want = (4LL * sm_count + rows - 1) / rows;
  int64_t units = cols / 8;
  int64_t cap = units / 512;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  if (want > 65535) want = 65535;
  return static_cast<int>(want);
}

size_t ras_split_workspace(int64_t rows, int64_t cols, int sm_count) {
  return static_cast<size_t>(rows) * ras_split_segments(rows, cols, sm_count) * sizeof(double);
}

cudaError_t launch_ras_persistent(const float *a, const float *b, float *out, int64_t rows,
                                  int64_t cols, int64_t lda, int64_t ldb, float scale,
                                  bool vec, cudaStream_t s) {
  if (vec)
    ras_warp_row<true, false><<<warp_row_grid(rows), kRowThreads, 0, s>>>(a, b, out, rows, cols,
                                                                         lda, ldb, scale);
  else
    ras_warp_row<false, false><<<warp_row_grid(rows), kRowThreads, 0, s>>>(a, b, out, rows,
                                                                          cols, lda, ldb, scale);
  return cudaGetLastError();
}

cudaError_t launch_ras_looped(const float *a, const float *b, float *out, int64_t rows,
                              int64_t cols, int64_t lda, int64_t ldb, float scale, bool vec,
                              cudaStream_t s) {
  if (vec)
    ras_warp_row<true, true><<<warp_row_grid(rows), kRowThreads, 0, s>>>(a, b, out, rows, cols,
                                                                        lda, ldb, scale);
  else
    ras_warp_row<false, true><<<warp_row_grid(rows), kRowThreads, 0, s>>>(a, b, out, rows, cols,
                                                                         lda, ldb, scale);
  return cudaGetLastError();
}

cudaError_t launch_ras_split(const float *a, const float *b, float *out, int64_t rows,
                             int64_t cols, int64_t lda, int64_t ldb, float scale, bool vec,
                             double *partials, int segments, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(segments), static_cast<unsigned>(rows));
  if (vec)
    ras_split_stage1<true><<<grid, kSplitThreads, 0, s>>>(a, b, cols, lda, ldb, scale, partials,
                                                         segments);
  else
    ras_split_stage1<false><<<grid, kSplitThreads, 0, s>>>(a, b, cols, lda, ldb, scale, partials,
                                                          segments);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ras_split_stage2<<<warp_row_grid(rows), kRowThreads, 0, s>>>(partials, out, rows, segments);
  return cudaGetLastError();
}

}  // namespace fr
