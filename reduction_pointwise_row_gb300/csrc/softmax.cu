// Row softmax, "Stax (4): GPU Codegen and Dynamic Shapes", section 9.5
// (Listing 9.5) and "CMU 15-779 Lecture 8", section 3:
//     m = max_r x,   y = exp(x - m) / sum_r exp(x - m).
//
// persistent  one warp per row, the row held in registers (up to 1024 fp32 per
//             warp), the max and the sum taken in two passes over registers:
//             one read and one write of each element (the 2N lower bound);
//             longer rows one CTA per row the same way.  Rows whose x and y
//             sit at different offsets within a 32-byte sector: a CTA per row
//             with the row in registers and y's chunks shifted by shuffles
//             (up to 4608 columns) or the row staged in shared memory.
// split       a thread-block cluster per row, each CTA a slice in registers,
//             the slices' (m, d) exchanged through distributed shared memory.
// looped      one CTA per row (grid-stride over rows) for rows longer than a
//             warp can hold.  Pass 1 keeps a per-thread online pair (m, d) and
//             folds each chunk in with the merge of section 9.5 (a chunk's max
//             first, then one exponential per element and one rescale per
//             chunk); the CTA combines the pairs with the same merge
//             (Proposition 9.1 makes the order irrelevant).  Pass 2 streams the
//             row again (an L2 hit when the row was just read) and writes y.
//
// exp(x - m) is computed as 2^(x*log2(e) - m*log2(e)) with one FMA and one
// SFU instruction; masked lanes are -inf for the max and contribute 0 to the
// sum.  A NaN makes the row's max NaN (max.NaN), hence the whole row NaN.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

constexpr int kWarpRowThreads = 256;

__device__ __forceinline__ float fbits(uint32_t w) { return __uint_as_float(w); }

// Persistent form, 32-byte vectors: NV vectors per lane (cols <= 256*NV).
// x and y rows share their offset modulo 32 bytes (checked by the host).
// HOST: rows in host memory, read and written over the host link by a grid
// of a few CTAs an SM whose warps take rows row, row + W, row + 2W, ... (W
// the grid's warps), which bounds the requests in flight on the link; a warp
// for every row at once oversubscribes it.
template <int NV, bool HOST = false>
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_warp_vec(const float *__restrict__ x, float *__restrict__ y, int64_t rows, int64_t cols,
                 int64_t ldx, int64_t ldy) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t first =
      static_cast<int64_t>(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
  auto one_row = [&](int64_t row) {
    const float *px = x + row * ldx;
    float *py = y + row * ldy;
    const RowSplit sp = row_split(px, cols, 4);
    // head and tail scalars (at most 7 + 7): one per lane
    int64_t si = -1;
    if (lane < sp.head) si = lane;
    else if (lane < sp.head + sp.tail) si = sp.head + sp.nvec * 8 + (lane - sp.head);
    const float *vx = px + sp.head;
    V8 v[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t vi = lane + 32 * k;
      if (vi < sp.nvec) v[k] = ld_stream_v8(vx + vi * 8);
    }
    float sv = -INFINITY;
    if (si >= 0) sv = ld_stream_f32(px + si);

    float m = sv;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (lane + 32 * k < sp.nvec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) m = max_nan(m, fbits(v[k].w[j]));
      }
    m = warp_max_nan(m);
    const float mb = m * kLog2e;

    float se = si >= 0 ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
    float d = se;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (lane + 32 * k < sp.nvec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float e = ex2(fmaf(fbits(v[k].w[j]), kLog2e, -mb));
          v[k].w[j] = __float_as_uint(e);
          d += e;
        }
      }
    d = warp_sum(d);
    const float inv = __frcp_rn(d);

    float *vy = py + sp.head;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t vi = lane + 32 * k;
      if (vi < sp.nvec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[k].w[j] = __float_as_uint(fbits(v[k].w[j]) * inv);
        st_stream_v8(vy + vi * 8, v[k]);
      }
    }
    if (si >= 0) st_stream_f32(py + si, se * inv);
  };
  if constexpr (HOST) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * (kWarpRowThreads / 32);
    for (int64_t row = first; row < rows; row += step) one_row(row);
  } else {
    if (first < rows) one_row(first);
  }
}

// Persistent form, scalar lane-strided elements (rows without a shared 32-byte
// alignment): NS elements per lane, cols <= 32*NS.
template <int NS>
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_warp_scalar(const float *__restrict__ x, float *__restrict__ y, int64_t rows,
                    int64_t cols, int64_t ldx, int64_t ldy) {
  const int lane = threadIdx.x & 31;
  const int64_t row =
      static_cast<int64_t>(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float *px = x + row * ldx;
  float *py = y + row * ldy;
  float v[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int64_t i = lane + 32 * k;
    v[k] = i < cols ? ld_stream_f32(px + i) : -INFINITY;
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < NS; ++k)
    if (lane + 32 * k < cols) m = max_nan(m, v[k]);
  m = warp_max_nan(m);
  const float mb = m * kLog2e;
  float d = 0.0f;
#pragma unroll
  for (int k = 0; k < NS; ++k)
    if (lane + 32 * k < cols) {
      v[k] = ex2(fmaf(v[k], kLog2e, -mb));
      d += v[k];
    }
  d = warp_sum(d);
  const float inv = __frcp_rn(d);
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int64_t i = lane + 32 * k;
    if (i < cols) st_stream_f32(py + i, v[k] * inv);
  }
}

// Persistent form for rows longer than a warp holds: one CTA of T threads per
// row, NV 32-byte vectors per thread in registers (body <= 8 * T * NV
// elements; the head and tail scalars, at most 7 + 7, one per thread).  The max
// and the sum are CTA reductions (one barrier each); each element is read once
// and written once.  x and y rows share their offset modulo 32 bytes.
template <int T, int NV>
__global__ void __launch_bounds__(T)
softmax_cta_vec(const float *__restrict__ x, float *__restrict__ y, int64_t cols, int64_t ldx,
                int64_t ldy) {
  pdl_enter();
  constexpr int W = T / 32;
  __shared__ float red[2][W];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float *px = x + row * ldx;
  float *py = y + row * ldy;
  const RowSplit sp = row_split(px, cols, 4);
  int64_t si = -1;
  if (tid < sp.head) si = tid;
  else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * 8 + (tid - sp.head);
  const float *vx = px + sp.head;
  V8 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = tid + static_cast<int64_t>(T) * k;
    if (vi < sp.nvec) v[k] = ld_stream_v8(vx + vi * 8);
  }
  const float sv = si >= 0 ? ld_stream_f32(px + si) : -INFINITY;

  float m = sv;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (tid + T * k < sp.nvec) {
#pragma unroll
      for (int j = 0; j < 8; ++j) m = max_nan(m, fbits(v[k].w[j]));
    }
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
  const float mb = m * kLog2e;

  const float se = si >= 0 ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
  float d = se;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (tid + T * k < sp.nvec) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float e = ex2(fmaf(fbits(v[k].w[j]), kLog2e, -mb));
        v[k].w[j] = __float_as_uint(e);
        d += e;
      }
    }
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();
  d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  const float inv = __frcp_rn(d);

  float *vy = py + sp.head;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = tid + static_cast<int64_t>(T) * k;
    if (vi < sp.nvec) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[k].w[j] = __float_as_uint(fbits(v[k].w[j]) * inv);
      st_stream_v8(vy + vi * 8, v[k]);
    }
  }
  if (si >= 0) st_stream_f32(py + si, se * inv);
}

// Split form for long rows: a thread-block cluster of C CTAs holds one row,
// CTA rank q its slice of the row's body vectors in registers (rank 0 also the
// head scalars, rank C - 1 the tail).  Each CTA reduces its slice to the pair
// (m_q, d_q) (two passes over registers) and pushes the pair into every CTA of
// the cluster with st.async, which counts the bytes on the receiver's
// mbarrier; once its own mbarrier has seen all C pairs, a CTA merges them in
// rank order with the merge of section 9.5 -- the same (M, D) in every CTA
// (Proposition 9.1 makes it the row's) -- and writes its exponentials scaled
// by 2^((m_q - M) log2 e) / D.  One read and one write per element; the
// exchange is 16 bytes per CTA pair and needs no release fence.  The only
// cluster barrier tells the peers that this CTA's mbarrier is initialised;
// it is arrived at before the loads and waited for after them.  A CTA leaves
// only after receiving every pair sent to it.  The wait is bounded; on expiry
// the kernel records FR_DEVERR_TIMEOUT and goes on.
constexpr int kSmClusterMax = 8;
constexpr long long kSmWaitBudget = 1LL << 31;  // SM clocks (about one second)

template <int T, int NV>
__global__ void __launch_bounds__(T)
softmax_cluster(const float *__restrict__ x, float *__restrict__ y, int64_t cols, int64_t ldx,
                int64_t ldy, int *__restrict__ err) {
  pdl_enter();
  constexpr int W = T / 32;
  __shared__ float red[2][W];
  __shared__ __align__(16) float4 pairs[kSmClusterMax];
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
  const float *px = x + row * ldx;
  float *py = y + row * ldy;
  const RowSplit sp = row_split(px, cols, 4);
  const int64_t per = (sp.nvec + C - 1) / C;
  const int64_t lo = per * q;
  const int64_t hi = lo + per < sp.nvec ? lo + per : sp.nvec;
  int64_t si = -1;  // head scalars: rank 0, threads 0..6; tail: rank C - 1, threads 32..38
  if (q == 0 && tid < sp.head) si = tid;
  else if (q == C - 1 && tid >= 32 && tid - 32 < sp.tail) si = sp.head + sp.nvec * 8 + (tid - 32);
  const float *vx = px + sp.head;
  V8 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = lo + tid + static_cast<int64_t>(T) * k;
    if (vi < hi) v[k] = ld_stream_v8(vx + vi * 8);
  }
  const float sv = si >= 0 ? ld_stream_f32(px + si) : -INFINITY;

  float m = sv;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (lo + tid + T * k < hi) {
#pragma unroll
      for (int j = 0; j < 8; ++j) m = max_nan(m, fbits(v[k].w[j]));
    }
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
  // a slice of nothing but -inf contributes d = 0 (and scales to 0 below)
  const float mb = m == -INFINITY ? 0.0f : m * kLog2e;

  const float se = si >= 0 ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
  float d = se;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (lo + tid + T * k < hi) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float e = ex2(fmaf(fbits(v[k].w[j]), kLog2e, -mb));
        v[k].w[j] = __float_as_uint(e);
        d += e;
      }
    }
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();
  d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  cluster_wait();  // every peer's mbarrier is initialised
  if (tid < static_cast<int>(C))
    st_async_f4(&pairs[q], &xbar, static_cast<uint32_t>(tid), make_float4(m, d, 0.0f, 0.0f));
  if (!mbar_wait_bounded(&xbar, 0, kSmWaitBudget) && tid == 0) atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
  float M = -INFINITY;
  for (uint32_t r = 0; r < C; ++r) M = max_nan(M, pairs[r].x);
  float D = 0.0f;
  if (M != -INFINITY)
    for (uint32_t r = 0; r < C; ++r) D += pairs[r].y * ex2((pairs[r].x - M) * kLog2e);
  const float scale = (M == -INFINITY ? 1.0f : ex2((m - M) * kLog2e)) * __frcp_rn(D);

  float *vy = py + sp.head;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = lo + tid + static_cast<int64_t>(T) * k;
    if (vi < hi) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[k].w[j] = __float_as_uint(fbits(v[k].w[j]) * scale);
      st_stream_v8(vy + vi * 8, v[k]);
    }
  }
  if (si >= 0) st_stream_f32(py + si, se * scale);
}

// Persistent form for rows whose x and y do not share their offset within a
// 32-byte sector (the kernels above pair x's vectors with y's): one CTA per
// row stages x in shared memory with 16-byte asynchronous copies at x's
// alignment (element i at srow[i + ox], ox putting x's 16-byte chunks on
// 16-byte boundaries), takes the max and the exponentials there (written back
// in place, one ex2 per element), and writes y in 16-byte chunks at y's
// alignment: each chunk is cut from two aligned float4 of shared memory by a
// shift the whole CTA shares.  One read of x and one write of y, for rows of
// up to kStageMaxCols elements.
constexpr int kStageMaxCols = 32768;

template <int T>
__global__ void __launch_bounds__(T)
softmax_cta_stage(const float *__restrict__ x, float *__restrict__ y, int64_t cols, int64_t ldx,
                  int64_t ldy) {
  pdl_enter();
  constexpr int W = T / 32;
  extern __shared__ __align__(16) float srow[];  // cols + 8 floats
  __shared__ float red[2][W];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float *px = x + row * ldx;
  float *py = y + row * ldy;
  const int n = static_cast<int>(cols);
  const int hx = min(n, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(px) & 15)) & 15) >> 2));
  const int ox = (4 - (hx & 3)) & 3;
  const int ncx = (n - hx) >> 2;  // x's whole 16-byte chunks
  const uint64_t policy = l2_evict_first_policy();
  for (int c = tid; c < ncx; c += T) cp_async_16_hint(srow + ox + hx + 4 * c, px + hx + 4 * c, policy);
  cp_async_commit();
  const int tx0 = hx + 4 * ncx;
  if (tid < hx) srow[ox + tid] = ld_stream_f32(px + tid);
  if (tid < n - tx0) srow[ox + tx0 + tid] = ld_stream_f32(px + tx0 + tid);
  cp_async_wait<0>();
  __syncthreads();

  const float4 *body = reinterpret_cast<const float4 *>(srow + ox + hx);  // x's chunks
  float m = -INFINITY;
  for (int c = tid; c < ncx; c += T) {
    const float4 v = body[c];
    m = max_nan(max_nan(m, v.x), max_nan(v.y, max_nan(v.z, v.w)));
  }
  if (tid < hx) m = max_nan(m, srow[ox + tid]);
  if (tid < n - tx0) m = max_nan(m, srow[ox + tx0 + tid]);
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
  const float mb = m * kLog2e;

  float d = 0.0f;
  float4 *wbody = reinterpret_cast<float4 *>(srow + ox + hx);
  for (int c = tid; c < ncx; c += T) {
    float4 v = wbody[c];
    v.x = ex2(fmaf(v.x, kLog2e, -mb));
    v.y = ex2(fmaf(v.y, kLog2e, -mb));
    v.z = ex2(fmaf(v.z, kLog2e, -mb));
    v.w = ex2(fmaf(v.w, kLog2e, -mb));
    wbody[c] = v;
    d += (v.x + v.y) + (v.z + v.w);
  }
  if (tid < hx) {
    const float e = ex2(fmaf(srow[ox + tid], kLog2e, -mb));
    srow[ox + tid] = e;
    d += e;
  }
  if (tid < n - tx0) {
    const float e = ex2(fmaf(srow[ox + tx0 + tid], kLog2e, -mb));
    srow[ox + tx0 + tid] = e;
    d += e;
  }
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();  // also: every exponential is in shared memory
  d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  const float inv = __frcp_rn(d);

  // y: hy scalars up to its 16-byte boundary, then 16-byte chunks; y's chunk
  // c holds elements hy + 4c .. + 3, at srow[ox + hy + 4c ...], sh floats past
  // a 16-byte boundary (sh the same for every chunk)
  const int hy = min(n, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(py) & 15)) & 15) >> 2));
  const int ncy = (n - hy) >> 2;
  const int base = ox + hy, sh = base & 3;
  const float4 *al = reinterpret_cast<const float4 *>(srow + (base - sh));
  float *vy = py + hy;
  auto put = [&](int c, float4 o) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(vy + 4 * c), "f"(o.x * inv),
                 "f"(o.y * inv), "f"(o.z * inv), "f"(o.w * inv)
                 : "memory");
  };
  switch (sh) {  // uniform: one branch for the whole CTA
    case 0:
      for (int c = tid; c < ncy; c += T) put(c, al[c]);
      break;
    case 1:
      for (int c = tid; c < ncy; c += T) {
        const float4 a = al[c], b = al[c + 1];
        put(c, make_float4(a.y, a.z, a.w, b.x));
      }
      break;
    case 2:
      for (int c = tid; c < ncy; c += T) {
        const float4 a = al[c], b = al[c + 1];
        put(c, make_float4(a.z, a.w, b.x, b.y));
      }
      break;
    default:
      for (int c = tid; c < ncy; c += T) {
        const float4 a = al[c], b = al[c + 1];
        put(c, make_float4(a.w, b.x, b.y, b.z));
      }
      break;
  }
  const int ty0 = hy + 4 * ncy;
  if (tid < hy) st_stream_f32(py + tid, srow[ox + tid] * inv);
  if (tid < n - ty0) st_stream_f32(py + ty0 + tid, srow[ox + ty0 + tid] * inv);
}

// Persistent form for rows out of phase, held in registers: one CTA of T
// threads (a multiple of 32, blockDim) per row, NV 16-byte chunks of x a
// thread, loaded at x's alignment (chunk c = tid + T k, the row's first and
// last chunks element by element).  With x's chunk 0 starting ox elements
// before the row and y's oy before it (ox >= oy, one chunk before the row
// added when x's offset is the smaller), y's chunk c holds the last 4 - s
// values of x's chunk c and the first s of chunk c + 1, s = ox - oy the same
// for the whole row: a thread gets them from the next lane with s shuffles,
// and the last lane of a warp from the chunks lane 0 of the next warp left in
// shared memory before the second barrier.  One read of x and one write of y,
// nothing staged.
template <int S, int NV>
__device__ __forceinline__ void write_shifted(float4 (&v)[NV], const float4 (*first)[NV],
                                              float *py, float *ya, int n, int oy, int ny,
                                              float inv, int tid, int T) {
  const int lane = tid & 31, warp = tid >> 5, nw = T >> 5;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    float4 nb = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if constexpr (S > 0) {
      nb.x = __shfl_down_sync(0xffffffffu, v[k].x, 1);
      if constexpr (S > 1) nb.y = __shfl_down_sync(0xffffffffu, v[k].y, 1);
      if constexpr (S > 2) nb.z = __shfl_down_sync(0xffffffffu, v[k].z, 1);
      if (lane == 31) {
        if (warp + 1 < nw) nb = first[warp + 1][k];
        else if (k + 1 < NV) nb = first[0][k + 1];
      }
    }
    const float4 a = v[k];
    float4 o = S == 0 ? a
             : S == 1 ? make_float4(a.y, a.z, a.w, nb.x)
             : S == 2 ? make_float4(a.z, a.w, nb.x, nb.y)
                      : make_float4(a.w, nb.x, nb.y, nb.z);
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
    const int c = tid + T * k;
    if (c < ny) {
      const int e0 = 4 * c - oy;
      if (e0 >= 0 && e0 + 4 <= n) {
        st_stream_u4(ya + 4 * c, make_uint4(__float_as_uint(o.x), __float_as_uint(o.y),
                                            __float_as_uint(o.z), __float_as_uint(o.w)));
      } else {
        const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j >= 0 && e0 + j < n) st_stream_f32(py + e0 + j, ov[j]);
      }
    }
  }
}

constexpr int kShiftMaxThreads = 512;
constexpr int kShiftChunks = 8;

template <int NV>
__global__ void __launch_bounds__(kShiftMaxThreads)
softmax_cta_shift(const float *__restrict__ x, float *__restrict__ y, int64_t cols, int64_t ldx,
                  int64_t ldy) {
  pdl_enter();
  constexpr int kMaxW = kShiftMaxThreads / 32;
  __shared__ float red[2][kMaxW];
  __shared__ float4 first[kMaxW][NV];  // lane 0's chunks (exponentials) per warp
  const int T = blockDim.x, nw = T >> 5;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float *px = x + row * ldx;
  float *py = y + row * ldy;
  const int n = static_cast<int>(cols);
  const int ox0 = static_cast<int>((reinterpret_cast<uintptr_t>(px) & 15) >> 2);
  const int oy = static_cast<int>((reinterpret_cast<uintptr_t>(py) & 15) >> 2);
  const int ox = ox0 < oy ? ox0 + 4 : ox0;
  const int nx = (n + ox + 3) >> 2, ny = (n + oy + 3) >> 2;
  const float *xa = px - ox;  // x's chunk c at xa + 4c, 16-byte aligned
  float *ya = py - oy;
  const uint64_t policy = l2_evict_first_policy();
  float4 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = tid + T * k;
    const int e0 = 4 * c - ox;
    v[k] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (c < nx) {
      if (e0 >= 0 && e0 + 4 <= n) {
        const uint4 u = ld_stream_u4(xa + 4 * c, policy);
        v[k] = make_float4(fbits(u.x), fbits(u.y), fbits(u.z), fbits(u.w));
      } else {
        float t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          t[j] = e0 + j >= 0 && e0 + j < n ? ld_stream_f32(px + e0 + j) : -INFINITY;
        v[k] = make_float4(t[0], t[1], t[2], t[3]);
      }
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    m = max_nan(m, max_nan(max_nan(v[k].x, v[k].y), max_nan(v[k].z, v[k].w)));
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < nw ? red[0][lane] : -INFINITY);
  const float mb = m * kLog2e;
  float d = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {  // masked slots: ex2(-inf) = 0
    v[k].x = ex2(fmaf(v[k].x, kLog2e, -mb));
    v[k].y = ex2(fmaf(v[k].y, kLog2e, -mb));
    v[k].z = ex2(fmaf(v[k].z, kLog2e, -mb));
    v[k].w = ex2(fmaf(v[k].w, kLog2e, -mb));
    d += (v[k].x + v[k].y) + (v[k].z + v[k].w);
  }
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < NV; ++k) first[warp][k] = v[k];
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();  // also: every warp's first chunks are in shared memory
  d = warp_sum(lane < nw ? red[1][lane] : 0.0f);
  const float inv = __frcp_rn(d);
  switch (ox - oy) {  // uniform: one branch for the whole CTA
    case 0: write_shifted<0, NV>(v, first, py, ya, n, oy, ny, inv, tid, T); break;
    case 1: write_shifted<1, NV>(v, first, py, ya, n, oy, ny, inv, tid, T); break;
    case 2: write_shifted<2, NV>(v, first, py, ya, n, oy, ny, inv, tid, T); break;
    default: write_shifted<3, NV>(v, first, py, ya, n, oy, ny, inv, tid, T); break;
  }
}

// Fold `n` values (already max-reduced to cm) into the online pair st.
__device__ __forceinline__ MD fold_chunk(MD st, float cm) {
  const float M = max_nan(st.m, cm);
  if (M == -INFINITY) return st;  // nothing but masked values so far
  st.d = st.d * ex2((st.m - M) * kLog2e);
  st.m = M;
  return st;
}

// CTA-wide merge of the per-thread pairs; every thread gets the row's (m, d).
template <int T>
__device__ __forceinline__ MD block_md(MD st, MD *smem) {
  constexpr int NW = T / 32;
  st = warp_md(st);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) smem[warp] = st;
  __syncthreads();
  MD r = lane < NW ? smem[lane] : MD{-INFINITY, 0.0f};
  r = warp_md(r);
  __syncthreads();  // smem free for the next row
  return r;
}

template <bool VEC, int T, int U, bool PF>
__global__ void __launch_bounds__(T)
softmax_block_looped(const float *__restrict__ x, float *__restrict__ y, int64_t rows,
                     int64_t cols, int64_t ldx, int64_t ldy) {
  pdl_enter();
  __shared__ MD red[T / 32];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float *px = x + row * ldx;
    float *py = y + row * ldy;
    const RowSplit sp = VEC ? row_split(px, cols, 4) : RowSplit{0, 0, static_cast<int>(0)};
    MD st{-INFINITY, 0.0f};
    if constexpr (VEC) {
      // PF: chunk base + T*U is loaded while chunk base is reduced (two
      // register buffers), so a thread always has a chunk of loads in flight.
      // Loads keep the row in L2 for pass 2.
      const float *vx = px + sp.head;
      V8 nx[U];
      if constexpr (PF) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (tid + T * u < sp.nvec) nx[u] = ld_keep_v8(vx + (tid + T * u) * 8);
      }
      for (int64_t base = 0; base < sp.nvec; base += T * U) {
        V8 v[U];
        const int64_t lb = PF ? base + T * U : base;  // the chunk loaded now
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if constexpr (PF) v[u] = nx[u];
          const int64_t vi = lb + tid + T * u;
          if (vi < sp.nvec) (PF ? nx[u] : v[u]) = ld_keep_v8(vx + vi * 8);
        }
        float cm = -INFINITY;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t vi = base + tid + T * u;
          if (vi < sp.nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j) cm = max_nan(cm, fbits(v[u].w[j]));
          }
        }
        st = fold_chunk(st, cm);
        if (st.m == -INFINITY) continue;  // every value so far is -inf: adds 0
        const float mb = st.m * kLog2e;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (base + tid + T * u < sp.nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j) st.d += ex2(fmaf(fbits(v[u].w[j]), kLog2e, -mb));
          }
      }
      int64_t si = -1;
      if (tid < sp.head) si = tid;
      else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * 8 + (tid - sp.head);
      if (si >= 0) st = md_merge(st, MD{ld_stream_f32(px + si), 1.0f});
    } else {
      for (int64_t base = 0; base < cols; base += T * 8) {
        float v[8];
        float cm = -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int64_t i = base + tid + T * u;
          v[u] = i < cols ? px[i] : -INFINITY;
          cm = max_nan(cm, v[u]);
        }
        st = fold_chunk(st, cm);
        if (st.m == -INFINITY) continue;
        const float mb = st.m * kLog2e;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (base + tid + T * u < cols) st.d += ex2(fmaf(v[u], kLog2e, -mb));
      }
    }
    const MD r = block_md<T>(st, red);
    const float mb = r.m * kLog2e;
    const float inv = __frcp_rn(r.d);
    if constexpr (VEC) {
      // Pass 2 walks the chunks last to first: pass 1 read them first to
      // last, so the chunks L2 still holds when a row is longer than its
      // share of L2 are the ones read again first (measured on GB300: 1216 x
      // 65537 140.2 us against 147.1 first to last, 2432 x 32768 128.1
      // against 134.7).
      const float *vx = px + sp.head;
      float *vy = py + sp.head;
      const int64_t nck = (sp.nvec + T * U - 1) / (T * U);
      V8 nx[U];
      if constexpr (PF) {
        if (nck > 0) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int64_t vi = (nck - 1) * T * U + tid + T * u;
            if (vi < sp.nvec) nx[u] = ld_stream_v8(vx + vi * 8);
          }
        }
      }
      for (int64_t ck = nck - 1; ck >= 0; --ck) {
        const int64_t base = ck * T * U;
        V8 v[U];
        const int64_t lb = PF ? base - T * U : base;  // the chunk loaded now
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if constexpr (PF) v[u] = nx[u];
          const int64_t vi = lb + tid + T * u;
          if (lb >= 0 && vi < sp.nvec) (PF ? nx[u] : v[u]) = ld_stream_v8(vx + vi * 8);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t vi = base + tid + T * u;
          if (vi < sp.nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              v[u].w[j] = __float_as_uint(ex2(fmaf(fbits(v[u].w[j]), kLog2e, -mb)) * inv);
            st_stream_v8(vy + vi * 8, v[u]);
          }
        }
      }
      int64_t si = -1;
      if (tid < sp.head) si = tid;
      else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * 8 + (tid - sp.head);
      if (si >= 0) st_stream_f32(py + si, ex2(fmaf(ld_stream_f32(px + si), kLog2e, -mb)) * inv);
    } else {  // first to last (last to first measured slower here: 1216 x 65537
              // out of phase 200.1 us against 180.6)
      for (int64_t i = tid; i < cols; i += T)
        st_stream_f32(py + i, ex2(fmaf(ld_stream_f32(px + i), kLog2e, -mb)) * inv);
    }
  }
}

// Persistent form with asynchronous-copy staging: warp w of the grid owns rows
// w, w + W, w + 2W, ... (W = warps in the grid) and keeps its next NS - 1 rows
// in flight in a per-warp shared-memory ring filled with cp.async (16 bytes per
// lane per copy, one commit group per row), so loads never stop while a row is
// reduced from registers and stored.  Rows of at most 128 * VPL fp32 with
// 16-byte aligned starts (x and y); the last cols % 4 elements are scalars.
constexpr int kAsyncThreads = 256;
constexpr int kAsyncStages = 3;

template <int VPL>
__global__ void __launch_bounds__(kAsyncThreads)
softmax_warp_async(const float *__restrict__ x, float *__restrict__ y, int64_t rows, int64_t cols,
                   int64_t ldx, int64_t ldy) {
  extern __shared__ __align__(128) unsigned char smem[];  // [warps][stages][VPL*32] x 16 B
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kAsyncThreads / 32;
  const int64_t W = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t wg = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nk = wg < rows ? (rows - wg + W - 1) / W : 0;
  const int nvec = static_cast<int>(cols >> 2);  // whole 16-byte vectors
  const int tail = static_cast<int>(cols & 3);
  unsigned char *wbuf = smem + static_cast<size_t>(warp) * kAsyncStages * VPL * 32 * 16;
  auto slot = [&](int st, int j) { return wbuf + (static_cast<size_t>(st) * VPL * 32 + j * 32 + lane) * 16; };
  auto stage = [&](int64_t k) {
    if (k < nk) {
      const float *src = x + (wg + k * W) * ldx;
      const int st = static_cast<int>(k % kAsyncStages);
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int v = j * 32 + lane;
        if (v < nvec) cp_async_16(slot(st, j), src + 4 * v);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < kAsyncStages - 1; ++i) stage(i);
  for (int64_t k = 0; k < nk; ++k) {
    stage(k + kAsyncStages - 1);
    cp_async_wait<kAsyncStages - 1>();
    const int64_t row = wg + k * W;
    const int st = static_cast<int>(k % kAsyncStages);
    float v[VPL][4];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (j * 32 + lane < nvec) {
        const uint4 q = lds_u4(slot(st, j));
        v[j][0] = __uint_as_float(q.x); v[j][1] = __uint_as_float(q.y);
        v[j][2] = __uint_as_float(q.z); v[j][3] = __uint_as_float(q.w);
      } else {
        v[j][0] = v[j][1] = v[j][2] = v[j][3] = -INFINITY;
      }
    }
    float sv = -INFINITY;  // tail scalar (at most 3, one per lane)
    if (lane < tail) sv = ld_stream_f32(x + row * ldx + 4 * nvec + lane);
    float m = sv;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) m = max_nan(m, v[j][e]);
    m = warp_max_nan(m);
    const float mb = m * kLog2e;
    float d = 0.0f;
    float se = lane < tail ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (j * 32 + lane < nvec) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[j][e] = ex2(fmaf(v[j][e], kLog2e, -mb));
          d += v[j][e];
        }
      }
    d = warp_sum(d + se);
    const float inv = __frcp_rn(d);
    float *py = y + row * ldy;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int vv = j * 32 + lane;
      if (vv < nvec)
        asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(py + 4 * vv),
                     "f"(v[j][0] * inv), "f"(v[j][1] * inv), "f"(v[j][2] * inv), "f"(v[j][3] * inv)
                     : "memory");
    }
    if (lane < tail) st_stream_f32(py + 4 * nvec + lane, se * inv);
  }
  cp_async_wait<0>();
}

unsigned warp_row_grid(int64_t rows) {
  return static_cast<unsigned>((rows + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32));
}

}  // namespace

// Rows up to 1024 take one warp; longer rows one CTA, holding the row in
// registers (x and y in phase: up to 1024 threads x 4 vectors, 128 KiB of
// registers) or in shared memory (out of phase), up to 32768 elements.
int64_t softmax_persistent_max_cols(bool) { return 32768; }

namespace {
template <int T, int NV>
cudaError_t launch_cta(const float *x, float *y, int64_t rows, int64_t cols, int64_t ldx,
                       int64_t ldy, cudaStream_t s) {
  return launch_k(softmax_cta_vec<T, NV>, dim3(static_cast<unsigned>(rows)), dim3(T), 0, s, 0, x,
                  y, cols, ldx, ldy);
}
}  // namespace

cudaError_t launch_softmax_persistent(const float *x, float *y, int64_t rows, int64_t cols,
                                      int64_t ldx, int64_t ldy, bool vec, cudaStream_t s) {
  const unsigned grid = warp_row_grid(rows);
  if (vec && cols > 1024) {
    if (rows > 0x7fffffff) return cudaErrorInvalidValue;
    const int64_t nvec = cols / 8;  // at least the body's vectors
    if (nvec <= 128 * 2) return launch_cta<128, 2>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 128 * 4) return launch_cta<128, 4>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 256 * 4) return launch_cta<256, 4>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 512 * 4) return launch_cta<512, 4>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 1024 * 4) return launch_cta<1024, 4>(x, y, rows, cols, ldx, ldy, s);
    return cudaErrorInvalidValue;
  }
  if (!vec && cols > 1024) {  // out of phase
    if (rows > 0x7fffffff || cols > kStageMaxCols) return cudaErrorInvalidValue;
    // Rows of up to 4608 columns: the row in registers, shifted by shuffles
    // (8 chunks a thread, the fewest warps that hold the row at any offset);
    // longer rows staged in shared memory.  Measured on GB300 (fp32, x one
    // element past y's phase, us per call, registers / staged): 16384 x 1536
    // 31.6 / 33.4, x 3072 59.4 / 60.0, x 4097 78.7 / 83.9, x 5120 96.7 /
    // 96.9, x 8192 157.7 / 153.6; 4864 x 16384 109.1 / 94.7.
    // FR_SOFTMAX_OOP=shift|stage pins one (shift: up to 16374 columns).
    const char *oop = getenv("FR_SOFTMAX_OOP");
    const bool pin_shift = oop != nullptr && strcmp(oop, "shift") == 0;
    const bool pin_stage = oop != nullptr && strcmp(oop, "stage") == 0;
    const int64_t nx = (cols + 7 + 3) / 4;  // chunks at the largest offset
    if (!pin_stage && (cols <= 4608 || pin_shift) && nx <= kShiftMaxThreads * kShiftChunks) {
      int64_t t = (nx + 32 * kShiftChunks - 1) / (32 * kShiftChunks) * 32;
      if (t < 64) t = 64;
      return launch_k(softmax_cta_shift<kShiftChunks>, dim3(static_cast<unsigned>(rows)),
                      dim3(static_cast<unsigned>(t)), 0, s, 0, x, y, cols, ldx, ldy);
    }
    // else the row staged in shared memory
    // four to twelve 16-byte chunks a thread (measured on GB300, us per call:
    // 16384 x 1025 with 64 threads 24.3, 128 27.2; x 2048 with 128 41.1, 64
    // 43.4; x 4097 with 256 84.1, 128 80.5, 512 117.5, and at 1216 rows 10.2
    // with 256, 12.5 with 128; x 8192 with 256 154.0, 512 164.1)
    const size_t smem = (static_cast<size_t>(cols) + 8) * 4;
    const int T = cols <= 1536 ? 64 : cols <= 3072 ? 128 : cols <= 12288 ? 256 : 512;
    auto kern = T == 64 ? softmax_cta_stage<64> : T == 128 ? softmax_cta_stage<128>
              : T == 256 ? softmax_cta_stage<256> : softmax_cta_stage<512>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_k(kern, dim3(static_cast<unsigned>(rows)), dim3(T), smem, s, 0, x, y, cols, ldx,
                    ldy);
  }
  if (vec) {
    const int64_t nv = (cols + 255) / 256;
    void (*kern)(const float *, float *, int64_t, int64_t, int64_t, int64_t) =
        nv == 1 ? softmax_warp_vec<1> : nv == 2 ? softmax_warp_vec<2>
                                      : nv == 3 ? softmax_warp_vec<3> : softmax_warp_vec<4>;
    if (nv < 1 || nv > 4) return cudaErrorInvalidValue;
    // a programmatic dependent of the previous kernel (measured on GB300,
    // fp32 [32768, 1024] back to back: 40.4 us against 43.0 us)
    return launch_k(kern, dim3(grid), dim3(kWarpRowThreads), 0, s, 0, x, y, rows, cols, ldx, ldy);
  } else {
    if (cols <= 128) softmax_warp_scalar<4><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else if (cols <= 256) softmax_warp_scalar<8><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else if (cols <= 512) softmax_warp_scalar<16><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else if (cols <= 1024) softmax_warp_scalar<32><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Rows in host memory (fp32, at most 1024 columns, x and y in phase): the
// warp-per-row kernel over a small grid whose warps take rows in turn, so
// that the host link sees a bounded number of requests in flight.  Measured
// on GB300 (fp32 [32768, 1024] in page-locked memory, x in and y out over
// NVLink-C2C, GB/s both ways): 19 CTAs of 8 warps 337.2, 38 340.4, 76 338.4,
// 152 334.3, 304 325.3, 608 298.1, a warp for every row (4096 CTAs) 304.2 --
// about 1.2 MB of loads in flight is what the link serves best.
// FR_HOST_GRID=<CTAs> pins the grid (default a quarter of the SMs).
cudaError_t launch_softmax_host_rows(const float *x, float *y, int64_t rows, int64_t cols,
                                     int sm_count, cudaStream_t s) {
  const int64_t nv = (cols + 255) / 256;
  if (nv < 1 || nv > 4) return cudaErrorInvalidValue;
  int64_t grid = sm_count / 4 > 0 ? sm_count / 4 : 1;
  if (const char *e = getenv("FR_HOST_GRID")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 65535) grid = v;
  }
  const int64_t need = (rows + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32);
  if (grid > need) grid = need;
  void (*kern)(const float *, float *, int64_t, int64_t, int64_t, int64_t) =
      nv == 1 ? softmax_warp_vec<1, true> : nv == 2 ? softmax_warp_vec<2, true>
                                          : nv == 3 ? softmax_warp_vec<3, true>
                                                    : softmax_warp_vec<4, true>;
  return launch_k(kern, dim3(static_cast<unsigned>(grid)), dim3(kWarpRowThreads), 0, s, 0, x, y,
                  rows, cols, cols, cols);
}

bool softmax_async_ok(int64_t cols, bool aligned16) { return aligned16 && cols <= 1024; }

cudaError_t launch_softmax_async(const float *x, float *y, int64_t rows, int64_t cols,
                                 int64_t ldx, int64_t ldy, int sm_count, cudaStream_t s) {
  const int vpl = static_cast<int>((cols / 4 + 31) / 32);
  const void *kern;
  switch (vpl) {
    case 0:
    case 1: kern = reinterpret_cast<const void *>(&softmax_warp_async<1>); break;
    case 2: kern = reinterpret_cast<const void *>(&softmax_warp_async<2>); break;
    case 3:
    case 4: kern = reinterpret_cast<const void *>(&softmax_warp_async<4>); break;
    case 5:
    case 6:
    case 7:
    case 8: kern = reinterpret_cast<const void *>(&softmax_warp_async<8>); break;
    default: return cudaErrorInvalidValue;
  }
  const int vp = vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : 8;
  const size_t smem = static_cast<size_t>(kAsyncThreads / 32) * kAsyncStages * vp * 32 * 16;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern), kAsyncThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = static_cast<int64_t>(sm_count) * per_sm;
  const int64_t need = (rows + kAsyncThreads / 32 - 1) / (kAsyncThreads / 32);
  if (grid > need) grid = need;
  void *args[] = {&x, &y, &rows, &cols, &ldx, &ldy};
  return cudaLaunchKernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kAsyncThreads), args, smem,
                          s);
}

// The split (cluster) form: C CTAs of T threads x 4 vectors per row, the
// smallest T in {256, 512, 1024} whose C-fold (C <= 8) holds the row's body;
// 0 when no cluster holds it.
namespace {
// The smallest CTA size, then the smallest cluster, whose registers hold the
// row (4 vectors of 8 per thread).  Measured on GB300, fp32 [511, 65537]:
// 8 CTAs of 256 threads 45.1 us, 4 of 512 48.2, 2 of 1024 56.5.
bool cluster_shape(int64_t cols, int *T, int *C) {
  const int64_t nvec = cols / 8;  // at least the body's vectors
  // FR_SOFTMAX_CLUSTER=<threads>x<ctas> pins a shape that holds the row.
  if (const char *e = getenv("FR_SOFTMAX_CLUSTER"); e != nullptr) {
    const int t = atoi(e);
    const char *xp = strchr(e, 'x');
    const int c = xp != nullptr ? atoi(xp + 1) : 0;
    if ((t == 256 || t == 512 || t == 1024) && (c == 2 || c == 4 || c == 8) && c <= kSmClusterMax &&
        nvec <= static_cast<int64_t>(c) * t * 4) {
      *T = t;
      *C = c;
      return true;
    }
  }
  for (int t = 256; t <= 1024; t <<= 1)
    for (int c = 2; c <= kSmClusterMax; c <<= 1)
      if (nvec <= static_cast<int64_t>(c) * t * 4) {
        *T = t;
        *C = c;
        return true;
      }
  return false;
}

template <int T, int NV>
cudaError_t launch_cluster_kernel(const float *x, float *y, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, int C, cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  return launch_k(softmax_cluster<T, NV>, dim3(static_cast<unsigned>(rows * C)), dim3(T), 0, s,
                  static_cast<unsigned>(C), x, y, cols, ldx, ldy, err);
}
}  // namespace

int64_t softmax_split_max_cols() { return static_cast<int64_t>(kSmClusterMax) * 1024 * 4 * 8; }

cudaError_t launch_softmax_split(const float *x, float *y, int64_t rows, int64_t cols,
                                 int64_t ldx, int64_t ldy, cudaStream_t s) {
  int T = 0, C = 0;
  if (!cluster_shape(cols, &T, &C) || rows * C > 0x7fffffff) return cudaErrorInvalidValue;
  switch (T) {
    case 256: return launch_cluster_kernel<256, 4>(x, y, rows, cols, ldx, ldy, C, s);
    case 512: return launch_cluster_kernel<512, 4>(x, y, rows, cols, ldx, ldy, C, s);
    default: return launch_cluster_kernel<1024, 4>(x, y, rows, cols, ldx, ldy, C, s);
  }
}

namespace {
template <int T, int U, bool PF>
cudaError_t launch_looped_t(const float *x, float *y, int64_t rows, int64_t cols, int64_t ldx,
                            int64_t ldy, bool vec, int sm_count, int per_sm_cap, cudaStream_t s) {
  auto kern = vec ? softmax_block_looped<true, T, U, PF> : softmax_block_looped<false, T, U, PF>;
  int per_sm = 0;
  cudaError_t e = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern), T, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if (per_sm > per_sm_cap) per_sm = per_sm_cap;
  int64_t grid = static_cast<int64_t>(sm_count) * per_sm;  // persistent: rows strided over CTAs
  if (grid > rows) grid = rows;
  return launch_k(kern, dim3(static_cast<unsigned>(grid)), dim3(T), 0, s, 0, x, y, rows, cols, ldx,
                  ldy);
}
}  // namespace

cudaError_t launch_softmax_looped(const float *x, float *y, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, bool vec, int sm_count,
                                  cudaStream_t s) {
  // Many rows: 256-thread CTAs, as many per SM as fit (more rows in flight);
  // few rows: 512 threads, two per SM, each thread loading its next chunk
  // while it reduces the current one.  Measured on GB300: fp32 [8190, 4097]
  // 48.8 us with 256 threads against 80.3 with 512 and 53.3 with 128 (56.7
  // with 256 and the next chunk in flight: 64 registers instead of 48 leave
  // room for four CTAs per SM instead of five); [511, 65537] 53.8 us with 512
  // and the next chunk in flight, 55.1 without, 63.9 with 256.
  // FR_SOFTMAX_LOOP=128|256|512 pins the CTA size.
  const char *e = getenv("FR_SOFTMAX_LOOP");
  const int t = e != nullptr ? atoi(e) : rows >= 4 * static_cast<int64_t>(sm_count) ? 256 : 512;
  if (t == 128) return launch_looped_t<128, 4, false>(x, y, rows, cols, ldx, ldy, vec, sm_count, 16, s);
  if (t == 256) return launch_looped_t<256, 2, false>(x, y, rows, cols, ldx, ldy, vec, sm_count, 16, s);
  return launch_looped_t<512, 2, true>(x, y, rows, cols, ldx, ldy, vec, sm_count, 2, s);
}

}  // namespace fr
