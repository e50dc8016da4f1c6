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
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
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

// 16-byte read-once load: no L1 allocation, and `policy` (an L2 policy from
// createpolicy, e.g. l2_evict_first_policy()) as the L2 hint.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p, uint64_t policy) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(policy));
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

__device__ __forceinline__ void st_stream_u4(void *p, uint4 v) {
  asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
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

// Element-wise max of two bf16x2 words; NaN in either lane gives NaN there.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Paired fp32 arithmetic (one instruction for two lanes on sm_100-class SMs).
// A pair is a 64-bit value: low 32 bits = first lane, high 32 bits = second.
// (register-pair moves: ptxas allocates the pair, no arithmetic is emitted)
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo;
}
__device__ __forceinline__ float f32x2_hi(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

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

// ---- bulk asynchronous copies into shared memory --------------------------
// cp.async.bulk moves a contiguous global range (16-byte aligned, a multiple
// of 16 bytes) into shared memory without registers; completion is counted in
// bytes on an mbarrier (the tensor-memory-accelerator path that "CMU 15-779
// Lecture 8", section 5 describes as one instruction moving a whole tile).

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes the initialised barriers visible to the async proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the barrier for at most `budget` SM clocks.
// Returns false on timeout (the caller records an error and stops waiting).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}

// An L2 policy that evicts the copied lines first (read-once data).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy ones (a bulk copy overwriting data the CTA has read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Per-thread asynchronous 16-byte global -> shared copy (no registers; the
// L1 is bypassed).  Copies are grouped with commit and waited for with
// wait_group<N>: at most N of the thread's most recent groups still pending.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
// The same with an L2 policy (createpolicy) as the hint.
__device__ __forceinline__ void cp_async_16_hint(void *dst, const void *src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)),
               "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 32 bytes from shared memory (two 16-byte loads).
__device__ __forceinline__ V8 lds_v8(const void *p) {
  V8 v;
  const uint32_t a = smem_addr(p);
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
               : "r"(a));
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
               : "r"(a + 16));
  return v;
}

// ---- thread-block clusters ------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Split cluster barrier: arrive releases this thread's earlier writes (shared
// memory included) to the cluster; wait acquires everyone's.  Every thread of
// every CTA in the cluster calls them in the same alternating order.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive without releasing this thread's writes (for signalling that this
// CTA's mbarriers are initialised, after fence.mbarrier_init).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// 16 bytes from the shared memory of CTA `rank` of this cluster, at the
// offset that `local` has in this CTA's shared memory.
__device__ __forceinline__ float4 ld_dsmem_f4(const void *local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}
// Writes 16 bytes into the shared memory of CTA `rank` of this cluster (at
// the offset `local_dst` has here) and counts them on that CTA's mbarrier at
// the offset of `local_bar`: the receiver waits on its own barrier, so the
// writer needs no release fence (which would also wait for its global stores).
__device__ __forceinline__ void st_async_f4(const void *local_dst, const uint64_t *local_bar,
                                            uint32_t rank, float4 v) {
  uint32_t rd, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rd) : "r"(smem_addr(local_dst)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(local_bar)), "r"(rank));
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(rd),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rb)
      : "memory");
}

// Writes 8 bytes into the shared memory of CTA `rank` of this cluster (at the
// address `local` has in this CTA); made visible by the next cluster barrier.
__device__ __forceinline__ void st_cluster_f2(void *local, uint32_t rank, float a, float b) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(a), "f"(b) : "memory");
}

__device__ __forceinline__ uint4 lds_u4(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
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

// The 16 bytes from 2-byte half S (0 .. 7) of the 32 bytes a[0..3], b[0..3]:
// a 16-byte chunk at one alignment cut from two chunks at another.
template <int S>
__device__ __forceinline__ uint4 cut_halves(const uint32_t (&a)[4], const uint32_t (&b)[4]) {
  uint32_t c[8] = {a[0], a[1], a[2], a[3], b[0], b[1], b[2], b[3]};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = (S & 1) ? __byte_perm(c[i + S / 2], c[i + S / 2 + 1], 0x5432) : c[i + S / 2];
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with launch_k may be placed on the SMs while the kernel
// before it on the stream is finishing (its CTAs take the slots that kernel's
// exiting CTAs free).  It starts with pdl_enter(): let the next grid be
// placed the same way, then wait until the previous grid has completed and
// its memory writes are visible -- so nothing is read early, whatever the
// previous kernel wrote.  Both instructions do nothing in an ordinary launch.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// FR_PDL=0 turns the overlap off (every kernel then waits for the one before
// it to finish before any of its CTAs is placed).
inline bool pdl_enabled() {
  static const bool on = [] {
    const char *e = getenv("FR_PDL");
    return !(e != nullptr && strcmp(e, "0") == 0);
  }();
  return on;
}

// Launches kern<<<grid, block, smem, s>>>(args...) as a programmatic
// dependent of the previous kernel on s (unless FR_PDL=0).  cluster > 0: a
// cluster launch of `cluster` CTAs along x (kernels that use cluster
// barriers, mapa or shared::cluster stores are always launched as clusters,
// also of one CTA); cluster = 0: an ordinary grid.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The same for a kernel held as an untyped pointer with packed arguments.
inline cudaError_t launch_pdl(const void *kern, dim3 grid, dim3 block, void **args, size_t smem,
                              cudaStream_t s) {
  if (!pdl_enabled()) return cudaLaunchKernel(kern, grid, block, args, smem, s);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

// ---- launch properties, looked up once ---------------------------------------
// The dynamic shared memory a kernel may use and its occupancy depend only on
// the kernel, the device and the launch shape, so each is asked of the runtime
// once and remembered (a launch-bound call otherwise pays for the driver calls
// on every launch).

// Raises kern's dynamic shared-memory limit on the current device to at least
// `bytes` (a limit, so a larger earlier setting serves).
inline cudaError_t set_smem_limit(const void *kern, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t &have = done[{dev, kern}];
  if (have >= bytes && (have > 0 || bytes == 0)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess) have = bytes > have ? bytes : have;
  return e;
}

// CTAs of `threads` threads and `smem` dynamic bytes that one SM holds.
inline cudaError_t blocks_per_sm(int *out, const void *kern, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void *, int, size_t>, int> known;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, kern, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(key);
    if (it != known.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kern, threads, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  known[key] = *out;
  return cudaSuccess;
}

// Clusters of cfg's shape (clusterDim.x CTAs of blockDim.x threads,
// dynamicSmemBytes each) resident on the device at once.
inline cudaError_t resident_clusters(int *out, const void *kern, const cudaLaunchConfig_t &cfg,
                                     unsigned cluster) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void *, unsigned, size_t, unsigned>, int> known;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, kern, cfg.blockDim.x, cfg.dynamicSmemBytes, cluster);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(key);
    if (it != known.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  e = cudaOccupancyMaxActiveClusters(out, kern, &cfg);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  known[key] = *out;
  return cudaSuccess;
}

}  // namespace fr
