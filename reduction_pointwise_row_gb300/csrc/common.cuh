// Device helpers shared by the fused row-reduction kernels (sm_103a).
//
// Memory access follows the rules the pages give for this kind of kernel:
// read-once inputs are loaded with an evict-first L2 hint and without L1
// allocation ("eviction_policy='evict_first'" in Listing 9.1 of "Stax (4): GPU
// Codegen and Dynamic Shapes", section 9.2), adjacent threads read adjacent
// vectors so every warp access is coalesced ("CMU 15-779 Lecture 8",
// section 6.2), and masked lanes hold the reduction's identity (-inf for max,
// 0 for sum; Stax (4) section 9.5).  On sm_100-class parts a thread can move 32
// bytes per instruction (ld/st .v8.b32), so the vector unit here is 32 bytes.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fr.h"

namespace fr {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kVecBytes = 32;

struct alignas(32) V8 {
  uint32_t w[8];
};

// ---- global memory -------------------------------------------------------

// 32-byte read-once load: no L1 allocation, first in line for L2 eviction.
__device__ __forceinline__ V8 ld_stream_v8(const void *p) {
  V8 v;
  asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
        "=r"(v.w[6]), "=r"(v.w[7])
      : "l"(p));
  return v;
}

// 32-byte load of data that many CTAs re-read (kept in L2 normally).
__device__ __forceinline__ V8 ld_keep_v8(const void *p) {
  V8 v;
  asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
        "=r"(v.w[6]), "=r"(v.w[7])
      : "l"(p));
  return v;
}

// 16-byte load of data that many CTAs re-read.
__device__ __forceinline__ float4 ld_keep_f4(const float *p) {
  float4 v;
  asm("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_stream_f32(const float *p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void *p) {
  uint16_t v;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// 32-byte streaming store (written once, not re-read by this kernel).
__device__ __forceinline__ void st_stream_v8(void *p, const V8 &v) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

__device__ __forceinline__ void st_stream_f32(float *p, float v) {
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void st_stream_u16(void *p, uint16_t v) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

// ---- arithmetic ----------------------------------------------------------

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN when either operand is NaN (the PropagateNan.ALL rule).
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// relu(v) = max(0, v) keeping NaN: the comparison is false for NaN, so v passes.
__device__ __forceinline__ float relu_nan(float v) { return v < 0.0f ? 0.0f : v; }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Two fp32 values -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint16_t to_bf16(float v) {
  uint16_t d;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(d) : "f"(v));
  return d;
}

// ---- reductions ----------------------------------------------------------

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Online-softmax pair (m, d): d = sum exp(x - m) over the elements merged so
// far.  The merge is the operator of Stax (4) section 9.5; M = -inf (both
// sides empty) returns the identity (-inf, 0) instead of exp(-inf + inf) = NaN.
struct MD {
  float m, d;
};

__device__ __forceinline__ MD md_merge(MD a, MD b) {
  float M = max_nan(a.m, b.m);
  if (M == -INFINITY) return MD{-INFINITY, 0.0f};
  float sa = ex2((a.m - M) * kLog2e);
  float sb = ex2((b.m - M) * kLog2e);
  return MD{M, a.d * sa + b.d * sb};
}

__device__ __forceinline__ MD warp_md(MD v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MD w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.d, o)};
    v = md_merge(v, w);
  }
  return v;
}

// ---- row geometry --------------------------------------------------------

// Split a row of `cols` elements of size `esize` starting at `p` into a head
// of scalars up to the first 32-byte boundary, a body of whole 32-byte
// vectors and a tail of scalars.
struct RowSplit {
  int head;      // elements before the first aligned vector
  int64_t nvec;  // whole 32-byte vectors
  int tail;      // elements after the last whole vector
};

__device__ __forceinline__ RowSplit row_split(const void *p, int64_t cols, int esize) {
  const int per = kVecBytes / esize;
  int64_t head = ((kVecBytes - (reinterpret_cast<uintptr_t>(p) & (kVecBytes - 1))) &
                  (kVecBytes - 1)) / esize;
  if (head > cols) head = cols;
  int64_t nvec = (cols - head) / per;
  RowSplit s;
  s.head = static_cast<int>(head);
  s.nvec = nvec;
  s.tail = static_cast<int>(cols - head - nvec * per);
  return s;
}

}  // namespace fr
