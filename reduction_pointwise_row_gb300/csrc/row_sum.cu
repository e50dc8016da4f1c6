// Row sums with a fused pointwise prologue and an optional epilogue, in the
// three reduction forms of "Stax (4): GPU Codegen and Dynamic Shapes",
// section 9.4:
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
// Prologues:
//   ReluAdd  Example 1.1 (section 9.2, Listing 9.1): scale * relu(a + b), a + b
//            in fp32 (tmp2), relu keeping NaN (tmp4, PropagateNan.ALL), times
//            scale in fp32 (tmp6);
//   Square   Example 6.2 (Listing 9.4): x * x in fp32 (tmp1 = tmp0 * tmp0).
// Epilogue: the plain sum, or its square root (the row L2 norm of Exercise 1
// of "CMU 15-779 Lecture 8: ML Compilers Part 1, Tile-based DSLs", section 12),
// taken in fp64 on the fp64 sum and rounded once to fp32.
//
// Runs of at most 8*U terms are summed in fp32 and then added into an fp64
// accumulator; the warp/CTA combine and the cross-CTA combine are fp64 in a
// fixed tree order, so a given shape on a given device model always gives the
// same bits.
#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

constexpr int kRowThreads = 256;  // warp-per-row forms: 8 rows per CTA
constexpr int kPersistNV = 4;     // 32-byte vectors per lane in the persistent form
constexpr int kSplitThreads = 256;
constexpr int kSplitU = 2;        // vector pairs in flight per thread per iteration

struct ReluAdd {
  static constexpr bool kTwoInputs = true;
  float scale;
  __device__ __forceinline__ float operator()(float a, float b) const {
    return relu_nan(a + b) * scale;
  }
};

struct Square {
  static constexpr bool kTwoInputs = false;
  __device__ __forceinline__ float operator()(float x, float) const { return x * x; }
};

// Input element types: fp32, or bf16 widened exactly to fp32 before the
// prologue (Listing 9.1 loads then computes in fp32).
struct F32In {
  using T = float;
  static constexpr int kES = 4;
  static constexpr int kN = 8;  // elements per 32-byte vector
  __device__ __forceinline__ static float at(const T *p, int64_t i) { return ld_stream_f32(p + i); }
  // value j (0 .. kN - 1) of a 32-byte vector
  __device__ __forceinline__ static float lane(const V8 &v, int j) { return __uint_as_float(v.w[j]); }
};
struct Bf16In {
  using T = uint16_t;
  static constexpr int kES = 2;
  static constexpr int kN = 16;
  __device__ __forceinline__ static float at(const T *p, int64_t i) { return bf16_to_f32(ld_stream_u16(p + i)); }
  __device__ __forceinline__ static float lane(const V8 &v, int j) {
    return (j & 1) ? bf16_hi(v.w[j >> 1]) : bf16_lo(v.w[j >> 1]);
  }
};

template <class Op, class In>
__device__ __forceinline__ float term_at(const Op &op, const typename In::T *pa,
                                         const typename In::T *pb, int64_t i) {
  if constexpr (Op::kTwoInputs) return op(In::at(pa, i), In::at(pb, i));
  else return op(In::at(pa, i), 0.0f);
}

// N 32-byte vectors of each input in flight per thread (one-input prologues
// hold no second array).
template <class Op, class In, int N>
struct VecBuf {
  V8 a[N];
  V8 b[Op::kTwoInputs ? N : 1];

  __device__ __forceinline__ void load(int k, const typename In::T *pa,
                                       const typename In::T *pb, int64_t off) {
    a[k] = ld_stream_v8(pa + off);
    if constexpr (Op::kTwoInputs) b[k] = ld_stream_v8(pb + off);
  }

  __device__ __forceinline__ float terms(int k, const Op &op) const {
    float t = 0.0f;
    if constexpr (Op::kTwoInputs) {
#pragma unroll
      for (int j = 0; j < In::kN; ++j) t += op(In::lane(a[k], j), In::lane(b[k], j));
    } else {
#pragma unroll
      for (int j = 0; j < In::kN; ++j) t += op(In::lane(a[k], j), 0.0f);
    }
    return t;
  }
};

template <bool SQRT>
__device__ __forceinline__ float finish(double acc) {
  if constexpr (SQRT) return static_cast<float>(sqrt(acc));
  else return static_cast<float>(acc);
}

// Warp-per-row form.  VEC: the input rows share their offset modulo 32 bytes,
// so one head/body/tail split serves both; otherwise every element is a
// scalar (still coalesced: lane-strided).  b is unused by one-input prologues.
template <class Op, class In, bool VEC, bool LOOP, bool SQRT>
__global__ void __launch_bounds__(kRowThreads)
rowsum_warp(const typename In::T *__restrict__ a, const typename In::T *__restrict__ b,
            float *__restrict__ out, int64_t rows, int64_t cols, int64_t lda, int64_t ldb, Op op) {
  pdl_enter();
  using E = typename In::T;
  constexpr int EPV = In::kN;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const E *pa = a + row * lda;
  const E *pb = Op::kTwoInputs ? b + row * ldb : nullptr;
  double acc = 0.0;
  if constexpr (VEC) {
    const RowSplit sp = row_split(pa, cols, In::kES);
    float s = 0.0f;  // head and tail: fewer than 16 scalars each, one per lane
    if (lane < sp.head) {
      s = term_at<Op, In>(op, pa, pb, lane);
    } else if (lane < sp.head + sp.tail) {
      s = term_at<Op, In>(op, pa, pb, sp.head + sp.nvec * EPV + (lane - sp.head));
    }
    acc = s;
    const E *va = pa + sp.head;
    const E *vb = Op::kTwoInputs ? pb + sp.head : nullptr;
    // persistent: the row's vectors fit one pass (base 0 only)
    for (int64_t base = 0; base < (LOOP ? sp.nvec : 1); base += 32 * kPersistNV) {
      VecBuf<Op, In, kPersistNV> buf;
#pragma unroll
      for (int k = 0; k < kPersistNV; ++k) {
        const int64_t vi = base + lane + 32 * k;
        if (vi < sp.nvec) buf.load(k, va, vb, vi * EPV);
      }
      float t = 0.0f;
#pragma unroll
      for (int k = 0; k < kPersistNV; ++k)
        if (base + lane + 32 * k < sp.nvec) t += buf.terms(k, op);
      acc += static_cast<double>(t);
    }
  } else {
    for (int64_t base = 0; base < cols; base += 32 * 8) {
      float t = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t i = base + lane + 32 * k;
        if (i < cols) t += term_at<Op, In>(op, pa, pb, i);
      }
      acc += static_cast<double>(t);
      if constexpr (!LOOP) {
        if (base + 32 * 8 >= 32 * EPV * kPersistNV) break;  // the persistent form's row cap
      }
    }
  }
  acc = warp_sum_f64(acc);
  if (lane == 0) out[row] = finish<SQRT>(acc);
}

// Split form, stage 1: CTA (seg, row) sums its segment of the row's body
// vectors (segment 0 also takes the head scalars, the last segment the tail).
template <class Op, class In, bool VEC>
__global__ void __launch_bounds__(kSplitThreads)
rowsum_split_stage1(const typename In::T *__restrict__ a, const typename In::T *__restrict__ b,
                    int64_t cols, int64_t lda, int64_t ldb, Op op, double *__restrict__ partials,
                    int S) {
  pdl_enter();
  using E = typename In::T;
  constexpr int EPV = In::kN;
  const int seg = blockIdx.x;
  const int64_t row = blockIdx.y;
  const int tid = threadIdx.x;
  const E *pa = a + row * lda;
  const E *pb = Op::kTwoInputs ? b + row * ldb : nullptr;
  const RowSplit sp = VEC ? row_split(pa, cols, In::kES) : RowSplit{0, cols, 0};
  const int64_t per = (sp.nvec + S - 1) / S;
  const int64_t lo = seg * per;
  const int64_t hi = lo + per < sp.nvec ? lo + per : sp.nvec;
  double acc = 0.0;
  if constexpr (VEC) {
    const E *va = pa + sp.head;
    const E *vb = Op::kTwoInputs ? pb + sp.head : nullptr;
    for (int64_t base = lo; base < hi; base += kSplitThreads * kSplitU) {
      VecBuf<Op, In, kSplitU> buf;
#pragma unroll
      for (int u = 0; u < kSplitU; ++u) {
        const int64_t vi = base + tid + kSplitThreads * u;
        if (vi < hi) buf.load(u, va, vb, vi * EPV);
      }
      float t = 0.0f;
#pragma unroll
      for (int u = 0; u < kSplitU; ++u)
        if (base + tid + kSplitThreads * u < hi) t += buf.terms(u, op);
      acc += static_cast<double>(t);
    }
    if (seg == 0 && tid < sp.head) acc += static_cast<double>(term_at<Op, In>(op, pa, pb, tid));
    if (seg == S - 1 && tid < sp.tail)
      acc += static_cast<double>(term_at<Op, In>(op, pa, pb, sp.head + sp.nvec * EPV + tid));
  } else {
    for (int64_t base = lo; base < hi; base += kSplitThreads * 8) {
      float t = 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = base + tid + kSplitThreads * u;
        if (i < hi) t += term_at<Op, In>(op, pa, pb, i);
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
template <bool SQRT>
__global__ void __launch_bounds__(kRowThreads)
rowsum_split_stage2(const double *__restrict__ partials, float *__restrict__ out, int64_t rows,
                    int S) {
  pdl_enter();  // the partials are stage 1's: read only after it has completed
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  double t = 0.0;
  for (int k = lane; k < S; k += 32) t += partials[row * S + k];
  t = warp_sum_f64(t);
  if (lane == 0) out[row] = finish<SQRT>(t);
}

unsigned warp_row_grid(int64_t rows) {
  return static_cast<unsigned>((rows + kRowThreads / 32 - 1) / (kRowThreads / 32));
}

template <class Op, class In, bool LOOP, bool SQRT>
cudaError_t launch_warp(const void *a, const void *b, float *out, int64_t rows, int64_t cols,
                        int64_t lda, int64_t ldb, Op op, bool vec, cudaStream_t s) {
  using E = typename In::T;
  const E *ea = static_cast<const E *>(a), *eb = static_cast<const E *>(b);
  const dim3 grid(warp_row_grid(rows)), block(kRowThreads);
  if (vec)
    return launch_k(rowsum_warp<Op, In, true, LOOP, SQRT>, grid, block, 0, s, 0, ea, eb, out, rows,
                    cols, lda, ldb, op);
  return launch_k(rowsum_warp<Op, In, false, LOOP, SQRT>, grid, block, 0, s, 0, ea, eb, out, rows,
                  cols, lda, ldb, op);
}

template <class Op, class In, bool SQRT>
cudaError_t launch_split(const void *a, const void *b, float *out, int64_t rows, int64_t cols,
                         int64_t lda, int64_t ldb, Op op, bool vec, double *partials,
                         int segments, cudaStream_t s) {
  // Stage 1 an ordinary launch: as a programmatic dependent of the call
  // before, the split form measured slower on GB300 (fp32 [8, 33554432]: 323
  // us against 309 us), its one-wave stage 1 sharing the SMs with the next
  // call's early-placed CTAs.  Stage 2 a programmatic dependent of stage 1:
  // placed as stage 1's CTAs exit, it saves 1.5-2 us a call (8 x 1048576:
  // 19.1 us against 21.0; 32 x 1048576: 46.5 against 48.3; 8 x 33554432:
  // 307.6 against 309.5).
  using E = typename In::T;
  const E *ea = static_cast<const E *>(a), *eb = static_cast<const E *>(b);
  const dim3 grid(static_cast<unsigned>(segments), static_cast<unsigned>(rows));
  if (vec)
    rowsum_split_stage1<Op, In, true><<<grid, kSplitThreads, 0, s>>>(ea, eb, cols, lda, ldb, op,
                                                                    partials, segments);
  else
    rowsum_split_stage1<Op, In, false><<<grid, kSplitThreads, 0, s>>>(ea, eb, cols, lda, ldb, op,
                                                                     partials, segments);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_k(rowsum_split_stage2<SQRT>, dim3(warp_row_grid(rows)), dim3(kRowThreads), 0, s, 0,
                  static_cast<const double *>(partials), out, rows, segments);
}

}  // namespace

int64_t ras_persistent_max_cols(bool bf16) {
  return 32 * static_cast<int64_t>(kPersistNV) * (bf16 ? Bf16In::kN : F32In::kN);
}

int ras_split_segments(int64_t rows, int64_t cols, int sm_count) {
  // Enough CTAs for four per SM (one wave at the kernel's occupancy), but no
  // segment shorter than 512 vectors (16 KiB of each fp32 input).
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

cudaError_t launch_ras_persistent(const void *a, const void *b, float *out, int64_t rows,
                                  int64_t cols, int64_t lda, int64_t ldb, float scale, bool bf16,
                                  bool vec, cudaStream_t s) {
  return bf16 ? launch_warp<ReluAdd, Bf16In, false, false>(a, b, out, rows, cols, lda, ldb,
                                                           ReluAdd{scale}, vec, s)
              : launch_warp<ReluAdd, F32In, false, false>(a, b, out, rows, cols, lda, ldb,
                                                          ReluAdd{scale}, vec, s);
}

cudaError_t launch_ras_looped(const void *a, const void *b, float *out, int64_t rows,
                              int64_t cols, int64_t lda, int64_t ldb, float scale, bool bf16,
                              bool vec, cudaStream_t s) {
  return bf16 ? launch_warp<ReluAdd, Bf16In, true, false>(a, b, out, rows, cols, lda, ldb,
                                                          ReluAdd{scale}, vec, s)
              : launch_warp<ReluAdd, F32In, true, false>(a, b, out, rows, cols, lda, ldb,
                                                         ReluAdd{scale}, vec, s);
}

cudaError_t launch_ras_split(const void *a, const void *b, float *out, int64_t rows,
                             int64_t cols, int64_t lda, int64_t ldb, float scale, bool bf16,
                             bool vec, double *partials, int segments, cudaStream_t s) {
  return bf16 ? launch_split<ReluAdd, Bf16In, false>(a, b, out, rows, cols, lda, ldb,
                                                     ReluAdd{scale}, vec, partials, segments, s)
              : launch_split<ReluAdd, F32In, false>(a, b, out, rows, cols, lda, ldb,
                                                    ReluAdd{scale}, vec, partials, segments, s);
}

// One-input rows need no common phase with a second input: every row takes
// the vector path with its own head/body/tail split.  The L2 norm's persistent
// form runs the looped instance: a row within the persistent limit is exactly
// one pass of its loop, with the same loads in flight, while the separate
// persistent instance kept three registers on the stack around the fp64
// square root (12 bytes of spill per thread under -Xptxas -v).
cudaError_t launch_sumsq_persistent(const float *x, float *out, int64_t rows, int64_t cols,
                                    int64_t ldx, bool sqrt_out, cudaStream_t s) {
  return sqrt_out ? launch_warp<Square, F32In, true, true>(x, nullptr, out, rows, cols, ldx, 0,
                                                           Square{}, true, s)
                  : launch_warp<Square, F32In, false, false>(x, nullptr, out, rows, cols, ldx, 0,
                                                             Square{}, true, s);
}

cudaError_t launch_sumsq_looped(const float *x, float *out, int64_t rows, int64_t cols,
                                int64_t ldx, bool sqrt_out, cudaStream_t s) {
  return sqrt_out ? launch_warp<Square, F32In, true, true>(x, nullptr, out, rows, cols, ldx, 0,
                                                           Square{}, true, s)
                  : launch_warp<Square, F32In, true, false>(x, nullptr, out, rows, cols, ldx, 0,
                                                            Square{}, true, s);
}

cudaError_t launch_sumsq_split(const float *x, float *out, int64_t rows, int64_t cols,
                               int64_t ldx, bool sqrt_out, double *partials, int segments,
                               cudaStream_t s) {
  return sqrt_out ? launch_split<Square, F32In, true>(x, nullptr, out, rows, cols, ldx, 0,
                                                      Square{}, true, partials, segments, s)
                  : launch_split<Square, F32In, false>(x, nullptr, out, rows, cols, ldx, 0,
                                                       Square{}, true, partials, segments, s);
}

}  // namespace fr
