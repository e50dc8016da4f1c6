// Row softmax, split form with the row staged in shared memory ("Stax (4):
// GPU Codegen and Dynamic Shapes", sections 9.4 and 9.5; "CMU 15-779
// Lecture 8", section 3):
//     m = max_r x,   y = exp(x - m) / sum_r exp(x - m),
// for rows that neither a CTA nor a cluster holds in registers and whose x
// and y sit at different offsets within a 32-byte sector (and for any row
// with FR_SOFTMAX_SPLIT=stage).  A thread-block cluster of C CTAs takes a
// row; CTA q owns a run of y's 16-byte chunks and stages the x elements of
// those chunks in its shared memory by 16-byte asynchronous copies at x's
// alignment (the run's ragged ends element by element).  Each CTA reduces its
// run to the pair (m_q, d_q) over shared memory and pushes it into every CTA
// of the cluster with st.async (counted on the receiver's mbarrier); once all
// C pairs are in, a CTA merges them in rank order with the merge of section
// 9.5 (the same (M, D) in every CTA) and writes its run of y: each 16-byte
// chunk cut from two aligned chunks of shared memory by a shift the CTA
// shares, its exponentials taken again (none kept).  One read of x and one
// write of y.  The wait is bounded; on expiry the kernel records
// FR_DEVERR_TIMEOUT and goes on.  fp32 and bf16 rows (fp32 arithmetic).
//
// Rows in phase (x and y at the same offset within a 32-byte sector) longer
// than 384 KiB, at any length, take softmax_cluster_loop: the same kind of
// cluster and exchange, but each CTA streams its run of x twice -- once
// folding the chunks into (m_q, d_q) with the merge of section 9.5, once after
// the exchange to write y -- the looped form of section 9.4 (2) within a
// cluster.  A run is 1/C of the row (C = 8, or 16 for fp32 rows of 1-4 MiB),
// so the second read follows the first within a few microseconds and finds x
// in L2; the CTAs an SM are set so that the runs read once and not yet again
// fit in half of L2, and the second pass goes through the run backwards, so
// that a run too long for L2 still finds its last-read part there.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

constexpr int kScMaxCluster = 8;
constexpr long long kScWaitBudget = 1LL << 31;  // SM clocks (about one second)
constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;

// Element type traits: a 16-byte chunk's max, its sum of 2^(x log2 e - mb),
// and y's chunk for it; one element as fp32 and back.
template <typename E>
struct Chunk;

template <>
struct Chunk<float> {
  static constexpr int kV = 4;
  static __device__ __forceinline__ float max(uint4 r) {
    return max_nan(max_nan(__uint_as_float(r.x), __uint_as_float(r.y)),
                   max_nan(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  static __device__ __forceinline__ float sum(uint4 r, float mb) {
    return (ex2(fmaf(__uint_as_float(r.x), kLog2e, -mb)) +
            ex2(fmaf(__uint_as_float(r.y), kLog2e, -mb))) +
           (ex2(fmaf(__uint_as_float(r.z), kLog2e, -mb)) +
            ex2(fmaf(__uint_as_float(r.w), kLog2e, -mb)));
  }
  static __device__ __forceinline__ uint32_t out1(uint32_t w, float mb, float inv) {
    return __float_as_uint(ex2(fmaf(__uint_as_float(w), kLog2e, -mb)) * inv);
  }
  static __device__ __forceinline__ uint4 out(uint4 r, float mb, float inv) {
    return make_uint4(out1(r.x, mb, inv), out1(r.y, mb, inv), out1(r.z, mb, inv),
                      out1(r.w, mb, inv));
  }
  static __device__ __forceinline__ float get(float v) { return v; }
  static __device__ __forceinline__ float put(float v) { return v; }
  static __device__ __forceinline__ float load1(const float *p) { return ld_stream_f32(p); }
  static __device__ __forceinline__ void store1(float *p, float v) { st_stream_f32(p, v); }
};

template <>
struct Chunk<uint16_t> {
  static constexpr int kV = 8;
  static __device__ __forceinline__ float max(uint4 r) {
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(r.x, r.y), max_nan_bf16x2(r.z, r.w));
    return max_nan(bf16_lo(m), bf16_hi(m));
  }
  static __device__ __forceinline__ float sum2(uint32_t w, float mb) {
    return ex2(fmaf(bf16_lo(w), kLog2e, -mb)) + ex2(fmaf(bf16_hi(w), kLog2e, -mb));
  }
  static __device__ __forceinline__ float sum(uint4 r, float mb) {
    return (sum2(r.x, mb) + sum2(r.y, mb)) + (sum2(r.z, mb) + sum2(r.w, mb));
  }
  static __device__ __forceinline__ uint32_t out2(uint32_t w, float mb, float inv) {
    return pack_bf16x2(ex2(fmaf(bf16_lo(w), kLog2e, -mb)) * inv,
                       ex2(fmaf(bf16_hi(w), kLog2e, -mb)) * inv);
  }
  static __device__ __forceinline__ uint4 out(uint4 r, float mb, float inv) {
    return make_uint4(out2(r.x, mb, inv), out2(r.y, mb, inv), out2(r.z, mb, inv),
                      out2(r.w, mb, inv));
  }
  static __device__ __forceinline__ float get(uint16_t v) { return bf16_to_f32(v); }
  static __device__ __forceinline__ uint16_t put(float v) { return to_bf16(v); }
  static __device__ __forceinline__ uint16_t load1(const uint16_t *p) { return ld_stream_u16(p); }
  static __device__ __forceinline__ void store1(uint16_t *p, uint16_t v) { st_stream_u16(p, v); }
};

// y's full chunks [cf, cl) of this CTA's run, chunk c at element V c - oy,
// staged at srow[V c - oy - e_lo + ox]: sh (in 2-byte halves) past a 16-byte
// boundary for every chunk.
template <typename E, int SH>
__device__ __forceinline__ void put_run(const E *srow, E *py, int cf, int cl, int oy, int e_lo,
                                        int ox, float mb, float inv, int tid, int T) {
  using K = Chunk<E>;
  constexpr int V = K::kV, SE = SH * 2 / static_cast<int>(sizeof(E));  // shift in elements
  for (int c = cf + tid; c < cl; c += T) {
    const int p = V * c - oy - e_lo + ox - SE;  // 16-byte aligned
    const uint4 *al = reinterpret_cast<const uint4 *>(srow + p);
    uint4 r = al[0];
    if constexpr (SH > 0) {
      const uint4 ra = al[0], rb = al[1];
      const uint32_t a[4] = {ra.x, ra.y, ra.z, ra.w}, b[4] = {rb.x, rb.y, rb.z, rb.w};
      r = cut_halves<SH>(a, b);
    }
    st_stream_u4(py + (V * c - oy), K::out(r, mb, inv));
  }
}

template <typename E, int T>
__global__ void __launch_bounds__(T)
softmax_cluster_stage(const E *__restrict__ x, E *__restrict__ y, int64_t cols, int64_t ldx,
                      int64_t ldy, int *__restrict__ err) {
  pdl_enter();
  using K = Chunk<E>;
  constexpr int V = K::kV, ES = static_cast<int>(sizeof(E)), W = T / 32;
  extern __shared__ __align__(16) unsigned char sraw[];
  E *srow = reinterpret_cast<E *>(sraw);
  __shared__ float red[2][W];
  __shared__ __align__(16) float4 pairs[kScMaxCluster];
  __shared__ __align__(8) uint64_t xbar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_nctarank(), q = cluster_ctarank();
  if (tid == 0) {
    mbar_init(&xbar, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(&xbar, 16u * C);
  }
  __syncthreads();
  cluster_arrive_relaxed();  // this CTA's mbarrier is ready for the peers' pairs
  const int64_t row = cluster_id_x();
  const E *px = x + row * ldx;
  E *py = y + row * ldy;
  const int n = static_cast<int>(cols);
  // y's chunks: chunk c holds elements V c - oy .. V c - oy + V - 1 (those in
  // the row); CTA q owns chunks [c0, c1) and so elements [e_lo, e_hi)
  const int oy = static_cast<int>((reinterpret_cast<uintptr_t>(py) & 15) / ES);
  const int ny = (n + oy + V - 1) / V;
  const int kc = (ny + static_cast<int>(C) - 1) / static_cast<int>(C);
  const int c0 = min(ny, static_cast<int>(q) * kc), c1 = min(ny, c0 + kc);
  const int e_lo = c0 < c1 ? max(0, V * c0 - oy) : 0;
  const int e_hi = c0 < c1 ? min(n, V * c1 - oy) : 0;
  const int nl = e_hi - e_lo;
  // stage x[e_lo, e_hi): hx elements up to x's 16-byte boundary, whole
  // chunks, the rest; element e at srow[e - e_lo + ox], x's chunks 16-byte
  // aligned in shared memory
  const E *pl = px + e_lo;
  const int hx = min(nl, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(pl) & 15)) & 15) / ES));
  const int ox = (V - hx % V) % V;
  const int ncx = (nl - hx) / V;
  const uint64_t policy = l2_evict_first_policy();
  for (int c = tid; c < ncx; c += T) cp_async_16_hint(srow + ox + hx + V * c, pl + hx + V * c, policy);
  cp_async_commit();
  const int tx0 = hx + V * ncx;
  if (tid < hx) srow[ox + tid] = K::load1(pl + tid);
  if (tid < nl - tx0) srow[ox + tx0 + tid] = K::load1(pl + tx0 + tid);
  cp_async_wait<0>();
  __syncthreads();

  // the run's (m, d).  fp32: one pass over shared memory, each thread folding
  // its chunks in with the merge of section 9.5 (a chunk's max, then its
  // exponentials against the running max) before the CTA merges the pairs;
  // bf16: the max, then the sum, two passes (measured on GB300, one pass /
  // two: fp32 out of phase 608 x 65537 58.1 / 62.6 us, 2432 x 32769 104.8 /
  // 114.1; bf16 2432 x 65537 112.8 / 108.3, its chunks of 8 pay a rescale
  // each for fewer shared-memory reads)
  const uint4 *body = reinterpret_cast<const uint4 *>(srow + ox + hx);
  float m, d;
  if constexpr (ES == 4) {
    MD st{-INFINITY, 0.0f};
    for (int c = tid; c < ncx; c += T) {
      const uint4 r = body[c];
      const float M = max_nan(st.m, K::max(r));
      if (M == -INFINITY) continue;  // nothing but -inf so far: adds 0
      st.d = st.m == -INFINITY ? 0.0f : st.d * ex2((st.m - M) * kLog2e);
      st.m = M;
      st.d += K::sum(r, M * kLog2e);
    }
    if (tid < hx) st = md_merge(st, MD{K::get(srow[ox + tid]), 1.0f});
    if (tid < nl - tx0) st = md_merge(st, MD{K::get(srow[ox + tx0 + tid]), 1.0f});
    st = warp_md(st);
    if (lane == 0) {
      red[0][warp] = st.m;
      red[1][warp] = st.d;
    }
    __syncthreads();
    const MD cta = warp_md(lane < W ? MD{red[0][lane], red[1][lane]} : MD{-INFINITY, 0.0f});
    m = cta.m;
    d = cta.d;
  } else {
    m = -INFINITY;
    for (int c = tid; c < ncx; c += T) m = max_nan(m, K::max(body[c]));
    if (tid < hx) m = max_nan(m, K::get(srow[ox + tid]));
    if (tid < nl - tx0) m = max_nan(m, K::get(srow[ox + tx0 + tid]));
    m = warp_max_nan(m);
    if (lane == 0) red[0][warp] = m;
    __syncthreads();
    m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
    // a run of nothing but -inf (or of nothing) contributes d = 0
    const float mq = m == -INFINITY ? 0.0f : m * kLog2e;
    d = 0.0f;
    for (int c = tid; c < ncx; c += T) d += K::sum(body[c], mq);
    if (tid < hx) d += ex2(fmaf(K::get(srow[ox + tid]), kLog2e, -mq));
    if (tid < nl - tx0) d += ex2(fmaf(K::get(srow[ox + tx0 + tid]), kLog2e, -mq));
    d = warp_sum(d);
    if (lane == 0) red[1][warp] = d;
    __syncthreads();
    d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  }
  cluster_wait();  // every peer's mbarrier is initialised
  if (tid < static_cast<int>(C))
    st_async_f4(&pairs[q], &xbar, static_cast<uint32_t>(tid), make_float4(m, d, 0.0f, 0.0f));
  if (!mbar_wait_bounded(&xbar, 0, kScWaitBudget) && tid == 0) atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
  // the C pairs merged in rank order: the same (M, D) in every CTA
  float M = -INFINITY;
  for (uint32_t r = 0; r < C; ++r) M = max_nan(M, pairs[r].x);
  float D = 0.0f;
  if (M != -INFINITY)
    for (uint32_t r = 0; r < C; ++r) D += pairs[r].y * ex2((pairs[r].x - M) * kLog2e);
  const float mb = M * kLog2e, inv = __frcp_rn(D);

  // y: the run's full 16-byte chunks, then its ragged ends element by element
  const int cf = c0 + ((c0 == 0 && oy > 0) ? 1 : 0);
  const int cl = (c1 > c0 && V * c1 - oy > n) ? c1 - 1 : c1;
  int fl = e_hi, fh = e_hi;  // the full chunks' elements
  if (cl > cf) {
    fl = V * cf - oy;
    fh = V * cl - oy;
    const int sh = ((V * cf - oy - e_lo + ox) % V) * ES / 2;  // in 2-byte halves
    switch (sh) {  // uniform: one branch for the whole CTA
      case 0: put_run<E, 0>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      case 1: put_run<E, 1>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      case 2: put_run<E, 2>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      case 3: put_run<E, 3>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      case 4: put_run<E, 4>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      case 5: put_run<E, 5>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      case 6: put_run<E, 6>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
      default: put_run<E, 7>(srow, py, cf, cl, oy, e_lo, ox, mb, inv, tid, T); break;
    }
  }
  const int nfront = min(fl, e_hi) - e_lo, nback = e_hi - max(fh, e_lo);
  auto scalar_y = [&](int e) {
    K::store1(py + e, K::put(ex2(fmaf(K::get(srow[e - e_lo + ox]), kLog2e, -mb)) * inv));
  };
  if (tid < nfront) scalar_y(e_lo + tid);
  else if (tid >= 32 && tid - 32 < nback && fh < e_hi) scalar_y(max(fh, e_lo) + tid - 32);
}

template <typename E, int T>
cudaError_t launch_stage_t(const E *x, E *y, int64_t rows, int64_t cols, int64_t ldx,
                           int64_t ldy, int C, size_t smem, cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  e = set_smem_limit(reinterpret_cast<const void *>(softmax_cluster_stage<E, T>), smem);
  if (e != cudaSuccess) return e;
  return launch_k(softmax_cluster_stage<E, T>, dim3(static_cast<unsigned>(rows * C)), dim3(T),
                  smem, s, static_cast<unsigned>(C), x, y, cols, ldx, ldy, err);
}

// The cluster for a row: the fewest CTAs (2, 4 or 8) whose runs take at most
// 48 KiB of shared memory each, else 8 CTAs with runs of up to 200 KiB; 512
// threads for runs past 64 KiB, 256 below.  Measured on GB300 (us per call,
// runs of at most 96 / 48 / 32 KiB): fp32 out of phase 608 x 32769 38.8 /
// 33.6 / 42.1, 608 x 65537 73.1 / 62.6 / 83.2, 2432 x 32769 132.0 / 114.1 /
// 152.1; bf16 2432 x 65537 119.5 / 108.3 / 136.4 -- runs of about 32 KiB,
// four to seven CTAs an SM.  FR_STAGE_RUN_KB=<KiB> sets the bound.
bool stage_shape(int64_t cols, int es, int *C, size_t *smem, int *T) {
  const int v = 16 / es;
  size_t target = 48u << 10;
  if (const char *e = getenv("FR_STAGE_RUN_KB")) {
    const int kb = atoi(e);
    if (kb >= 4 && kb <= 200) target = static_cast<size_t>(kb) << 10;
  }
  const int64_t ny = (cols + v - 1) / v + 1;  // y's chunks at the largest offset
  for (int c = 2; c <= kScMaxCluster; c <<= 1) {
    const int64_t kc = (ny + c - 1) / c;
    const size_t bytes = static_cast<size_t>((kc + 3) * v) * es;  // run + shift + padding
    if (bytes <= target || (c == kScMaxCluster && bytes <= (200u << 10))) {
      *C = c;
      *smem = (bytes + 15) / 16 * 16;
      *T = bytes > (64u << 10) ? 512 : 256;
      return true;
    }
  }
  return false;
}

}  // namespace

int64_t softmax_stage_split_max_cols(int es) {
  // the longest row stage_shape takes (200 KiB runs over 8 CTAs, less the
  // chunks of shift and padding)
  const int v = 16 / es;
  return (static_cast<int64_t>((200u << 10) / es / v) - 3) * kScMaxCluster * v - 2 * v;
}

cudaError_t launch_softmax_split_staged(const void *x, void *y, int64_t rows, int64_t cols,
                                        int64_t ldx, int64_t ldy, int es, cudaStream_t s) {
  int C = 0, T = 0;
  size_t smem = 0;
  if (!stage_shape(cols, es, &C, &smem, &T) || rows * C > 0x7fffffff || cols > 0x7fffffff)
    return cudaErrorInvalidValue;
  if (es == 4) {
    const float *fx = static_cast<const float *>(x);
    float *fy = static_cast<float *>(y);
    return T == 512 ? launch_stage_t<float, 512>(fx, fy, rows, cols, ldx, ldy, C, smem, s)
                    : launch_stage_t<float, 256>(fx, fy, rows, cols, ldx, ldy, C, smem, s);
  }
  const uint16_t *bx = static_cast<const uint16_t *>(x);
  uint16_t *by = static_cast<uint16_t *>(y);
  return T == 512 ? launch_stage_t<uint16_t, 512>(bx, by, rows, cols, ldx, ldy, C, smem, s)
                  : launch_stage_t<uint16_t, 256>(bx, by, rows, cols, ldx, ldy, C, smem, s);
}


namespace {

// L2 policies for the first pass's loads (the second pass reads them again).
__device__ __forceinline__ uint64_t l2_policy(bool keep) {
  uint64_t pol;
  if (keep)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

constexpr int kLoopU = 8;  // 16-byte chunks a thread has in flight per pass
constexpr int kLoopMaxCluster = 16;  // beyond the portable 8: opted in per kernel

// One cluster of C CTAs per row, x and y rows in phase; CTA q takes the whole
// 16-byte chunks [c0, c1) of the row (the chunks of y and of x coincide),
// CTA 0 the ragged head, CTA C - 1 the ragged tail.
template <typename E, int T>
__global__ void __launch_bounds__(T, 1024 / T)
softmax_cluster_loop(const E *__restrict__ x, E *__restrict__ y, int cols, int64_t ldx,
                     int64_t ldy, int keep, int *__restrict__ err) {
  pdl_enter();
  using K = Chunk<E>;
  constexpr int V = K::kV, ES = static_cast<int>(sizeof(E)), W = T / 32, U = kLoopU;
  __shared__ float red[2][W];
  __shared__ __align__(16) float4 pairs[kLoopMaxCluster];
  __shared__ __align__(8) uint64_t xbar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_nctarank(), q = cluster_ctarank();
  if (tid == 0) {
    mbar_init(&xbar, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(&xbar, 16u * C);
  }
  __syncthreads();
  cluster_arrive_relaxed();  // this CTA's mbarrier is ready for the peers' pairs
  const int64_t row = cluster_id_x();
  const E *px = x + row * ldx;
  E *py = y + row * ldy;
  const int n = cols;
  // h elements before the first whole chunk, nf whole chunks, then the tail
  const int h = min(n, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(px) & 15)) & 15) / ES));
  const int nf = (n - h) / V, t0 = h + V * nf, tail = n - t0;
  const int kc = (nf + static_cast<int>(C) - 1) / static_cast<int>(C);
  const int c0 = min(nf, static_cast<int>(q) * kc), c1 = min(nf, c0 + kc);
  const uint4 *xv = reinterpret_cast<const uint4 *>(px + h);
  uint4 *yv = reinterpret_cast<uint4 *>(py + h);
  const bool head_here = q == 0 && tid < h;
  const bool tail_here = q == C - 1 && tid >= 32 && tid - 32 < tail;
  const int se = head_here ? tid : t0 + tid - 32;  // this thread's ragged element

  // pass 1: (m, d) of the run, U chunks at a time: their max, one rescale of
  // d to it, then their exponentials against it
  MD st{-INFINITY, 0.0f};
  const uint64_t first_pol = l2_policy(keep != 0);
  for (int base = c0 + tid; base < c1; base += T * U) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + T * u < c1) r[u] = ld_stream_u4(xv + base + T * u, first_pol);
    float gm = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + T * u < c1) gm = max_nan(gm, K::max(r[u]));
    const float M = max_nan(st.m, gm);
    if (M == -INFINITY) continue;  // nothing but -inf so far: adds 0
    if (M != st.m) st.d *= ex2((st.m - M) * kLog2e);  // 0 while st.m is -inf
    st.m = M;
    const float mb = M * kLog2e;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + T * u < c1) st.d += K::sum(r[u], mb);
  }
  if (head_here || tail_here) st = md_merge(st, MD{K::get(K::load1(px + se)), 1.0f});
  st = warp_md(st);
  if (lane == 0) {
    red[0][warp] = st.m;
    red[1][warp] = st.d;
  }
  __syncthreads();
  const MD cta = warp_md(lane < W ? MD{red[0][lane], red[1][lane]} : MD{-INFINITY, 0.0f});

  cluster_wait();  // every peer's mbarrier is initialised
  if (tid < static_cast<int>(C))
    st_async_f4(&pairs[q], &xbar, static_cast<uint32_t>(tid), make_float4(cta.m, cta.d, 0.0f, 0.0f));
  if (!mbar_wait_bounded(&xbar, 0, kScWaitBudget) && tid == 0) atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
  // the C pairs merged in rank order: the same (M, D) in every CTA
  float M = -INFINITY;
  for (uint32_t r = 0; r < C; ++r) M = max_nan(M, pairs[r].x);
  float D = 0.0f;
  if (M != -INFINITY)
    for (uint32_t r = 0; r < C; ++r) D += pairs[r].y * ex2((pairs[r].x - M) * kLog2e);
  const float mb = M * kLog2e, inv = __frcp_rn(D);

  // pass 2: the run again, its blocks of T U chunks in reverse order (the
  // ones read last in pass 1 first: what of a run too long for L2 is still
  // there), each chunk's last read (first out of L2), y written out
  const uint64_t policy = l2_evict_first_policy();
  for (int it = (c1 - c0 + T * U - 1) / (T * U) - 1; it >= 0; --it) {
    const int base = c0 + it * T * U + tid;
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + T * u < c1) r[u] = ld_stream_u4(xv + base + T * u, policy);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + T * u < c1) st_stream_u4(yv + base + T * u, K::out(r[u], mb, inv));
  }
  if (head_here || tail_here)
    K::store1(py + se, K::put(ex2(fmaf(K::get(K::load1(px + se)), kLog2e, -mb)) * inv));
}

template <typename E, int T>
cudaError_t launch_loop_t(const E *x, E *y, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t ldy, int C, int per_sm, cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const void *kern = reinterpret_cast<const void *>(softmax_cluster_loop<E, T>);
  if (C > 8) {  // clusters past the portable size are opted in to once per device
    static std::mutex mu;
    static std::set<std::pair<int, const void *>> done;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (!done.count({dev, kern})) {
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
          cudaSuccess)
        return e;
      done.insert({dev, kern});
    }
  }
  if ((e = set_smem_limit(kern, 0)) != cudaSuccess) return e;
  if (C > 8) {  // a device (or partition) that holds no cluster of C: 8
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(T);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((e = resident_clusters(&clusters, kern, cfg, static_cast<unsigned>(C))) != cudaSuccess)
      return e;
    if (clusters < 1) C = 8;
  }
  // CTAs an SM: what the registers allow, held to per_sm by padding the
  // dynamic shared memory ((per_sm + 1) padded CTAs do not fit an SM)
  int resident = 0;
  if ((e = blocks_per_sm(&resident, kern, T, 0)) != cudaSuccess) return e;
  size_t smem = 0;
  if (resident > per_sm) {
    int dev = 0, per_sm_smem = 0, reserved = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
            cudaSuccess)
      return e;
    smem = static_cast<size_t>((per_sm_smem / (per_sm + 1) - reserved + 1023) / 1024 * 1024);
    if ((e = set_smem_limit(kern, smem)) != cudaSuccess) return e;
  }
  // The first pass's loads marked evict-last (FR_LOOP_KEEP=0: evict-normal).
  // Measured on GB300, back to back, evict-last / evict-normal: fp32 304 x
  // 262144 107.4 / 110.1 us, 152 x 393216 87.8 / 88.5; bf16 608 x 262144
  // 102.8 / 105.0, 304 x 393216 81.9 / 82.7; rows of 1048576 alike (their
  // runs do not stay in L2 either way).
  const char *kp = getenv("FR_LOOP_KEEP");
  const int keep = !(kp != nullptr && kp[0] == '0');
  return launch_k(softmax_cluster_loop<E, T>, dim3(static_cast<unsigned>(rows * C)), dim3(T),
                  smem, s, static_cast<unsigned>(C), x, y, static_cast<int>(cols), ldx, ldy, keep,
                  err);
}

// The loop cluster's shape: C = 8 CTAs a row, 16 for fp32 rows of 1 to 4 MiB;
// four CTAs of 256 threads an SM while the runs read once and not yet again
// -- every resident CTA's run -- fit in 64 MB (half of L2), else two of 512.
// Measured on GB300 (us per call, back to back).  CTAs an SM 1 / 2 / 4 with C
// = 8: fp32 152 x 262144 84.7 / 60.6 / 70.5, 304 x 393216 234.4 / 174.8 /
// 207.3, 16 x 4194304 172.3 / 143.1 / 197.7; bf16 304 x 262144 120.6 / 66.0 /
// 56.5, 152 x 393216 76.3 / 51.7 / 48.3, 64 x 1048576 71.3 / 57.0 / 64.7.
// Clusters of 16 (shorter runs: each cluster lives half as long, so the last
// rows leave the GPU idle for less time), against 8 at the rule's CTAs an SM:
// fp32 304 x 262144 106.8 / 109.5, 152 x 393216 86.5 / 90.7, 64 x 1048576
// 107.6 / 116.5, but 16 x 4194304 150.2 / 143.6 and 608 x 131072 116.1 /
// 102.0; bf16 slower at every length but 4194304 (608 x 262144 122.1 / 104.3,
// 64 x 1048576 61.3 / 56.6, 16 x 4194304 74.2 / 80.6).  Clusters of 4 were
// slower than of 8 but at bf16 64 x 393216 (22.8 against 25.6 at two CTAs an
// SM, 22.5 at four).
// FR_LOOP_C=4|8|16, FR_LOOP_K=1|2|4 and FR_LOOP_L2_MB=<MB> pin them.
void loop_shape(int64_t rows, int64_t cols, int es, int sm_count, int *C, int *per_sm) {
  *C = kScMaxCluster;
  if (es == 4 && cols * es >= (1 << 20) && cols * es <= (4 << 20) && rows * 16 <= 0x7fffffff)
    *C = 16;
  if (const char *e = getenv("FR_LOOP_C")) {
    const int c = atoi(e);
    if (c == 4 || (c == 16 && rows * 16 <= 0x7fffffff)) *C = c;
  }
  int64_t budget = 64ll << 20;
  if (const char *e = getenv("FR_LOOP_L2_MB")) {
    const int mb = atoi(e);
    if (mb >= 1 && mb <= 1024) budget = static_cast<int64_t>(mb) << 20;
  }
  const int64_t run = cols * es / *C;
  *per_sm = static_cast<int64_t>(sm_count) * 4 * run <= budget ? 4 : 2;
  if (const char *e = getenv("FR_LOOP_K")) {
    const int k = atoi(e);
    if (k == 1 || k == 2 || k == 4) *per_sm = k;
  }
}

}  // namespace

cudaError_t launch_softmax_split_looped(const void *x, void *y, int64_t rows, int64_t cols,
                                        int64_t ldx, int64_t ldy, int es, int sm_count,
                                        cudaStream_t s) {
  if (rows < 1 || cols < 1 || cols > 0x7fffffff || rows * kScMaxCluster > 0x7fffffff)
    return cudaErrorInvalidValue;
  int C = 0, per_sm = 0;
  loop_shape(rows, cols, es, sm_count, &C, &per_sm);
  if (es == 4) {
    const float *fx = static_cast<const float *>(x);
    float *fy = static_cast<float *>(y);
    switch (per_sm) {
      case 4: return launch_loop_t<float, 256>(fx, fy, rows, cols, ldx, ldy, C, 4, s);
      case 2: return launch_loop_t<float, 512>(fx, fy, rows, cols, ldx, ldy, C, 2, s);
      default: return launch_loop_t<float, 1024>(fx, fy, rows, cols, ldx, ldy, C, 1, s);
    }
  }
  const uint16_t *bx = static_cast<const uint16_t *>(x);
  uint16_t *by = static_cast<uint16_t *>(y);
  switch (per_sm) {
    case 4: return launch_loop_t<uint16_t, 256>(bx, by, rows, cols, ldx, ldy, C, 4, s);
    case 2: return launch_loop_t<uint16_t, 512>(bx, by, rows, cols, ldx, ldy, C, 2, s);
    default: return launch_loop_t<uint16_t, 1024>(bx, by, rows, cols, ldx, ldy, C, 1, s);
  }
}

}  // namespace fr
