// Row softmax on bf16 rows ("Stax (4): GPU Codegen and Dynamic Shapes",
// section 9.5 and Listing 9.5, whose loads cast to fp32 before the max):
// x is read as bf16 and widened exactly to fp32, the max, the exponentials,
// the sum and the division are fp32, and y is rounded to bf16 (nearest even).
//
// persistent  one warp per row, the row's exponentials held in registers (up
//             to 2048 elements per warp, 32-byte vectors of 16 bf16 per lane),
//             the max and the sum in two passes over registers: one read and
//             one write of each element; rows of 2049 .. 32768 in phase take
//             one CTA per row the same way, with CTA reductions; rows out of
//             phase one CTA per row with the row staged in shared memory.
// looped      one CTA per row (grid-stride over rows) for longer rows: per-
//             thread online pairs (m, d) folded chunk by chunk with the merge
//             of section 9.5, combined across the CTA in any order
//             (Proposition 9.1), then a second streaming pass writes y.
//
// The max runs on packed bf16 pairs (max.NaN.bf16x2 is exact on bf16 values);
// NaN anywhere in the row makes the row NaN; masked lanes are -inf for the max
// and 0 for the sum.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

constexpr int kWarpRowThreads = 256;
constexpr int kLoopU = 2;
constexpr int kPer = 16;                    // bf16 per 32-byte vector
constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;

__device__ __forceinline__ float vec_max(const V8 &v) {
  uint32_t m = kNegInfBf16x2;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = max_nan_bf16x2(m, v.w[j]);
  return max_nan(bf16_lo(m), bf16_hi(m));
}

// Persistent form, 32-byte vectors: NV vectors of 16 elements per lane
// (cols <= 512 * NV).  x and y rows share their offset modulo 32 bytes.  The
// 16 * NV exponentials stay in registers (89 at NV = 4, no spill).
// HOST: rows in host memory over the host link, from a small grid whose
// warps take rows row, row + W, ... (W the grid's warps): a bounded number of
// requests in flight (the fp32 kernel's launch_softmax_host_rows has the
// measurements).
template <int NV, bool HOST = false>
__global__ void __launch_bounds__(kWarpRowThreads, 1)
softmax_bf16_warp_vec(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int64_t rows,
                      int64_t cols, int64_t ldx, int64_t ldy) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t first =
      static_cast<int64_t>(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
  auto one_row = [&](int64_t row) {
    const uint16_t *px = x + row * ldx;
    uint16_t *py = y + row * ldy;
    const RowSplit sp = row_split(px, cols, 2);
    // head and tail scalars (at most 15 + 15): one per lane
    int64_t si = -1;
    if (lane < sp.head) si = lane;
    else if (lane < sp.head + sp.tail) si = sp.head + sp.nvec * kPer + (lane - sp.head);
    const uint16_t *vx = px + sp.head;
    V8 v[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t vi = lane + 32 * k;
      if (vi < sp.nvec) v[k] = ld_stream_v8(vx + vi * kPer);
    }
    const float sv = si >= 0 ? bf16_to_f32(ld_stream_u16(px + si)) : -INFINITY;

    float m = sv;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (lane + 32 * k < sp.nvec) m = max_nan(m, vec_max(v[k]));
    m = warp_max_nan(m);
    const float mb = m * kLog2e;

    const float se = si >= 0 ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
    float e[NV][kPer];
    float d = se;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (lane + 32 * k < sp.nvec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          e[k][2 * j] = ex2(fmaf(bf16_lo(v[k].w[j]), kLog2e, -mb));
          e[k][2 * j + 1] = ex2(fmaf(bf16_hi(v[k].w[j]), kLog2e, -mb));
          d += e[k][2 * j] + e[k][2 * j + 1];
        }
      }
    d = warp_sum(d);
    const float inv = __frcp_rn(d);

    uint16_t *vy = py + sp.head;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t vi = lane + 32 * k;
      if (vi < sp.nvec) {
        V8 o;
#pragma unroll
        for (int j = 0; j < 8; ++j) o.w[j] = pack_bf16x2(e[k][2 * j] * inv, e[k][2 * j + 1] * inv);
        st_stream_v8(vy + vi * kPer, o);
      }
    }
    if (si >= 0) st_stream_u16(py + si, to_bf16(se * inv));
  };
  if constexpr (HOST) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * (kWarpRowThreads / 32);
    for (int64_t row = first; row < rows; row += step) one_row(row);
  } else {
    if (first < rows) one_row(first);
  }
}

// Persistent form for longer rows in phase: one CTA of T threads per row,
// NV vectors of 16 elements per thread (cols <= 16 * T * NV), the
// exponentials in registers as in the warp form; the max and the sum are CTA
// reductions (per-warp values through shared memory).
template <int T, int NV>
__global__ void __launch_bounds__(T)
softmax_bf16_cta_vec(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int64_t cols,
                     int64_t ldx, int64_t ldy) {
  pdl_enter();
  constexpr int W = T / 32;
  __shared__ float red[2][W];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const uint16_t *px = x + row * ldx;
  uint16_t *py = y + row * ldy;
  const RowSplit sp = row_split(px, cols, 2);
  int64_t si = -1;  // head and tail scalars (at most 15 + 15), one per thread
  if (tid < sp.head) si = tid;
  else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * kPer + (tid - sp.head);
  const uint16_t *vx = px + sp.head;
  V8 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = tid + static_cast<int64_t>(T) * k;
    if (vi < sp.nvec) v[k] = ld_stream_v8(vx + vi * kPer);
  }
  const float sv = si >= 0 ? bf16_to_f32(ld_stream_u16(px + si)) : -INFINITY;

  float m = sv;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (tid + T * k < sp.nvec) m = max_nan(m, vec_max(v[k]));
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
  const float mb = m * kLog2e;

  const float se = si >= 0 ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
  float e[NV][kPer];
  float d = se;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (tid + T * k < sp.nvec) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        e[k][2 * j] = ex2(fmaf(bf16_lo(v[k].w[j]), kLog2e, -mb));
        e[k][2 * j + 1] = ex2(fmaf(bf16_hi(v[k].w[j]), kLog2e, -mb));
        d += e[k][2 * j] + e[k][2 * j + 1];
      }
    }
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();
  d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  const float inv = __frcp_rn(d);

  uint16_t *vy = py + sp.head;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = tid + static_cast<int64_t>(T) * k;
    if (vi < sp.nvec) {
      V8 o;
#pragma unroll
      for (int j = 0; j < 8; ++j) o.w[j] = pack_bf16x2(e[k][2 * j] * inv, e[k][2 * j + 1] * inv);
      st_stream_v8(vy + vi * kPer, o);
    }
  }
  if (si >= 0) st_stream_u16(py + si, to_bf16(se * inv));
}

// y's value of a word of two raw x elements, packed to bf16
__device__ __forceinline__ uint32_t softmax_word(uint32_t w, float mb, float inv) {
  return pack_bf16x2(ex2(fmaf(bf16_lo(w), kLog2e, -mb)) * inv,
                     ex2(fmaf(bf16_hi(w), kLog2e, -mb)) * inv);
}

// The persistent form's other kernel for rows out of phase: one CTA of T
// threads per row stages x (raw bf16) in shared memory with 16-byte
// asynchronous copies at x's alignment (element i at srow[i + ox], ox putting
// x's 16-byte chunks on 16-byte boundaries); the max comes from packed pairs,
// the sum from one exponential per element, and y's 16-byte chunks are cut
// from two aligned chunks of shared memory by a shift the whole CTA shares,
// their exponentials taken again there (two per element in all: 2 bytes of
// shared memory a column instead of 4 of registers, so more rows in flight
// per SM).  One read of x and one write of y, up to kBfStageMaxCols columns.
constexpr int kBfStageMaxCols = 32768;

template <int S>
__device__ __forceinline__ void bf16_stage_put(const uint4 *al, uint16_t *vy, int ncy, float mb,
                                               float inv, int tid, int T) {
  for (int c = tid; c < ncy; c += T) {
    const uint4 ra = al[c];
    uint4 r = ra;
    if constexpr (S > 0) {
      const uint4 rb = al[c + 1];
      const uint32_t a[4] = {ra.x, ra.y, ra.z, ra.w}, b[4] = {rb.x, rb.y, rb.z, rb.w};
      r = cut_halves<S>(a, b);
    }
    st_stream_u4(vy + 8 * c, make_uint4(softmax_word(r.x, mb, inv), softmax_word(r.y, mb, inv),
                                        softmax_word(r.z, mb, inv), softmax_word(r.w, mb, inv)));
  }
}

template <int T>
__global__ void __launch_bounds__(T)
softmax_bf16_cta_stage(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int64_t cols,
                       int64_t ldx, int64_t ldy) {
  pdl_enter();
  constexpr int W = T / 32;
  extern __shared__ __align__(16) uint16_t srow16[];  // cols + 16 elements
  __shared__ float red[2][W];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const uint16_t *px = x + row * ldx;
  uint16_t *py = y + row * ldy;
  const int n = static_cast<int>(cols);
  const int hx = min(n, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(px) & 15)) & 15) >> 1));
  const int ox = (8 - (hx & 7)) & 7;
  const int ncx = (n - hx) >> 3;  // x's whole 16-byte chunks
  const uint64_t policy = l2_evict_first_policy();
  for (int c = tid; c < ncx; c += T)
    cp_async_16_hint(srow16 + ox + hx + 8 * c, px + hx + 8 * c, policy);
  cp_async_commit();
  const int tx0 = hx + 8 * ncx;
  if (tid < hx) srow16[ox + tid] = ld_stream_u16(px + tid);
  if (tid < n - tx0) srow16[ox + tx0 + tid] = ld_stream_u16(px + tx0 + tid);
  cp_async_wait<0>();
  __syncthreads();

  const uint4 *body = reinterpret_cast<const uint4 *>(srow16 + ox + hx);  // x's chunks
  uint32_t mw = kNegInfBf16x2;
  for (int c = tid; c < ncx; c += T) {
    const uint4 v = body[c];
    mw = max_nan_bf16x2(max_nan_bf16x2(mw, max_nan_bf16x2(v.x, v.y)), max_nan_bf16x2(v.z, v.w));
  }
  float m = max_nan(bf16_lo(mw), bf16_hi(mw));
  if (tid < hx) m = max_nan(m, bf16_to_f32(srow16[ox + tid]));
  if (tid < n - tx0) m = max_nan(m, bf16_to_f32(srow16[ox + tx0 + tid]));
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
  const float mb = m * kLog2e;

  float d = 0.0f;
  for (int c = tid; c < ncx; c += T) {
    const uint4 v = body[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      d += ex2(fmaf(bf16_lo(w[j]), kLog2e, -mb)) + ex2(fmaf(bf16_hi(w[j]), kLog2e, -mb));
  }
  if (tid < hx) d += ex2(fmaf(bf16_to_f32(srow16[ox + tid]), kLog2e, -mb));
  if (tid < n - tx0) d += ex2(fmaf(bf16_to_f32(srow16[ox + tx0 + tid]), kLog2e, -mb));
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();
  d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  const float inv = __frcp_rn(d);

  // y: hy scalars up to its 16-byte boundary, then 16-byte chunks; y's chunk
  // c holds elements hy + 8c .. + 7, at srow16[ox + hy + 8c ...], sh elements
  // past a 16-byte boundary (the same for every chunk)
  const int hy = min(n, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(py) & 15)) & 15) >> 1));
  const int ncy = (n - hy) >> 3;
  const int base = ox + hy, sh = base & 7;
  const uint4 *al = reinterpret_cast<const uint4 *>(srow16 + (base - sh));
  uint16_t *vy = py + hy;
  switch (sh) {  // uniform: one branch for the whole CTA
    case 0: bf16_stage_put<0>(al, vy, ncy, mb, inv, tid, T); break;
    case 1: bf16_stage_put<1>(al, vy, ncy, mb, inv, tid, T); break;
    case 2: bf16_stage_put<2>(al, vy, ncy, mb, inv, tid, T); break;
    case 3: bf16_stage_put<3>(al, vy, ncy, mb, inv, tid, T); break;
    case 4: bf16_stage_put<4>(al, vy, ncy, mb, inv, tid, T); break;
    case 5: bf16_stage_put<5>(al, vy, ncy, mb, inv, tid, T); break;
    case 6: bf16_stage_put<6>(al, vy, ncy, mb, inv, tid, T); break;
    default: bf16_stage_put<7>(al, vy, ncy, mb, inv, tid, T); break;
  }
  const int ty0 = hy + 8 * ncy;
  auto scalar_y = [&](int i) {
    st_stream_u16(py + i, to_bf16(ex2(fmaf(bf16_to_f32(srow16[ox + i]), kLog2e, -mb)) * inv));
  };
  if (tid < hy) scalar_y(tid);
  if (tid < n - ty0) scalar_y(ty0 + tid);
}

// Split form for long rows in phase: a thread-block cluster of C CTAs per
// row, CTA rank q holding its slice of the row's 16-element vectors and their
// exponentials in registers (rank 0 also the head scalars, rank C - 1 the
// tail).  Each CTA reduces its slice to (m_q, d_q), pushes the pair into every
// CTA of the cluster with st.async (counted on the receiver's mbarrier), and
// once all C pairs are in, merges them in rank order with the merge of
// section 9.5 -- the same (M, D) in every CTA -- and writes its values scaled
// by 2^((m_q - M) log2 e) / D.  One read and one write per element.  The wait
// is bounded; on expiry the kernel records FR_DEVERR_TIMEOUT and goes on.
constexpr int kBfClusterMax = 8;
constexpr long long kBfWaitBudget = 1LL << 31;  // SM clocks (about one second)

// RE: recompute the exponentials in the writing pass instead of holding
// them (registers for twice the vectors per thread; two ex2 per element).
template <int T, int NV, bool RE>
__global__ void __launch_bounds__(T)
softmax_bf16_cluster(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int64_t cols,
                     int64_t ldx, int64_t ldy, int *__restrict__ err) {
  pdl_enter();
  constexpr int W = T / 32;
  __shared__ float red[2][W];
  __shared__ __align__(16) float4 pairs[kBfClusterMax];
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
  const uint16_t *px = x + row * ldx;
  uint16_t *py = y + row * ldy;
  const RowSplit sp = row_split(px, cols, 2);
  const int64_t per = (sp.nvec + C - 1) / C;
  const int64_t lo = per * q;
  const int64_t hi = lo + per < sp.nvec ? lo + per : sp.nvec;
  int64_t si = -1;  // head scalars: rank 0, threads 0..14; tail: rank C - 1, threads 32..46
  if (q == 0 && tid < sp.head) si = tid;
  else if (q == C - 1 && tid >= 32 && tid - 32 < sp.tail) si = sp.head + sp.nvec * kPer + (tid - 32);
  const uint16_t *vx = px + sp.head;
  V8 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = lo + tid + static_cast<int64_t>(T) * k;
    if (vi < hi) v[k] = ld_stream_v8(vx + vi * kPer);
  }
  const float sv = si >= 0 ? bf16_to_f32(ld_stream_u16(px + si)) : -INFINITY;

  float m = sv;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (lo + tid + T * k < hi) m = max_nan(m, vec_max(v[k]));
  m = warp_max_nan(m);
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = warp_max_nan(lane < W ? red[0][lane] : -INFINITY);
  // a slice of nothing but -inf contributes d = 0 (and scales to 0 below)
  const float mb = m == -INFINITY ? 0.0f : m * kLog2e;

  const float se = si >= 0 ? ex2(fmaf(sv, kLog2e, -mb)) : 0.0f;
  float e[RE ? 1 : NV][kPer];
  float d = se;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (lo + tid + T * k < hi) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float e0 = ex2(fmaf(bf16_lo(v[k].w[j]), kLog2e, -mb));
        const float e1 = ex2(fmaf(bf16_hi(v[k].w[j]), kLog2e, -mb));
        if constexpr (!RE) {
          e[k][2 * j] = e0;
          e[k][2 * j + 1] = e1;
        }
        d += e0 + e1;
      }
    }
  d = warp_sum(d);
  if (lane == 0) red[1][warp] = d;
  __syncthreads();
  d = warp_sum(lane < W ? red[1][lane] : 0.0f);
  cluster_wait();  // every peer's mbarrier is initialised
  if (tid < static_cast<int>(C))
    st_async_f4(&pairs[q], &xbar, static_cast<uint32_t>(tid), make_float4(m, d, 0.0f, 0.0f));
  if (!mbar_wait_bounded(&xbar, 0, kBfWaitBudget) && tid == 0) atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
  float M = -INFINITY;
  for (uint32_t r = 0; r < C; ++r) M = max_nan(M, pairs[r].x);
  float D = 0.0f;
  if (M != -INFINITY)
    for (uint32_t r = 0; r < C; ++r) D += pairs[r].y * ex2((pairs[r].x - M) * kLog2e);
  const float scale = (M == -INFINITY ? 1.0f : ex2((m - M) * kLog2e)) * __frcp_rn(D);

  uint16_t *vy = py + sp.head;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t vi = lo + tid + static_cast<int64_t>(T) * k;
    if (vi < hi) {
      V8 o;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if constexpr (RE)
          o.w[j] = pack_bf16x2(ex2(fmaf(bf16_lo(v[k].w[j]), kLog2e, -mb)) * scale,
                               ex2(fmaf(bf16_hi(v[k].w[j]), kLog2e, -mb)) * scale);
        else
          o.w[j] = pack_bf16x2(e[k][2 * j] * scale, e[k][2 * j + 1] * scale);
      }
      st_stream_v8(vy + vi * kPer, o);
    }
  }
  if (si >= 0) st_stream_u16(py + si, to_bf16(se * scale));
}

// Persistent form, lane-strided scalars (x and y rows out of phase): NS
// elements per lane, cols <= 32 * NS.
template <int NS>
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_bf16_warp_scalar(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int64_t rows,
                         int64_t cols, int64_t ldx, int64_t ldy) {
  const int lane = threadIdx.x & 31;
  const int64_t row =
      static_cast<int64_t>(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint16_t *px = x + row * ldx;
  uint16_t *py = y + row * ldy;
  float v[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int64_t i = lane + 32 * k;
    v[k] = i < cols ? bf16_to_f32(ld_stream_u16(px + i)) : -INFINITY;
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
    if (i < cols) st_stream_u16(py + i, to_bf16(v[k] * inv));
  }
}

// Fold a chunk whose max is cm into the online pair: rescale d to the new max.
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

template <bool VEC, int T>
__global__ void __launch_bounds__(T)
softmax_bf16_block_looped(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int64_t rows,
                          int64_t cols, int64_t ldx, int64_t ldy) {
  pdl_enter();
  __shared__ MD red[T / 32];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint16_t *px = x + row * ldx;
    uint16_t *py = y + row * ldy;
    const RowSplit sp = VEC ? row_split(px, cols, 2) : RowSplit{0, 0, 0};
    MD st{-INFINITY, 0.0f};
    if constexpr (VEC) {
      const uint16_t *vx = px + sp.head;
      for (int64_t base = 0; base < sp.nvec; base += T * kLoopU) {
        V8 v[kLoopU];
        float cm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kLoopU; ++u) {
          const int64_t vi = base + tid + T * u;
          if (vi < sp.nvec) {
            v[u] = ld_keep_v8(vx + vi * kPer);  // pass 2 re-reads it from L2
            cm = max_nan(cm, vec_max(v[u]));
          }
        }
        st = fold_chunk(st, cm);
        if (st.m == -INFINITY) continue;  // every value so far is -inf: adds 0
        const float mb = st.m * kLog2e;
#pragma unroll
        for (int u = 0; u < kLoopU; ++u)
          if (base + tid + T * u < sp.nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st.d += ex2(fmaf(bf16_lo(v[u].w[j]), kLog2e, -mb)) +
                      ex2(fmaf(bf16_hi(v[u].w[j]), kLog2e, -mb));
          }
      }
      int64_t si = -1;
      if (tid < sp.head) si = tid;
      else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * kPer + (tid - sp.head);
      if (si >= 0) st = md_merge(st, MD{bf16_to_f32(ld_stream_u16(px + si)), 1.0f});
    } else {
      for (int64_t base = 0; base < cols; base += T * 8) {
        float v[8];
        float cm = -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int64_t i = base + tid + T * u;
          v[u] = i < cols ? bf16_to_f32(ld_stream_u16(px + i)) : -INFINITY;
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
      // 131072 134.8 us against 141.9 first to last).
      const uint16_t *vx = px + sp.head;
      uint16_t *vy = py + sp.head;
      for (int64_t base = (sp.nvec - 1) / (T * kLoopU) * (T * kLoopU); base >= 0;
           base -= T * kLoopU) {
        V8 v[kLoopU];
#pragma unroll
        for (int u = 0; u < kLoopU; ++u) {
          const int64_t vi = base + tid + T * u;
          if (vi < sp.nvec) v[u] = ld_stream_v8(vx + vi * kPer);
        }
#pragma unroll
        for (int u = 0; u < kLoopU; ++u) {
          const int64_t vi = base + tid + T * u;
          if (vi < sp.nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              v[u].w[j] = pack_bf16x2(ex2(fmaf(bf16_lo(v[u].w[j]), kLog2e, -mb)) * inv,
                                      ex2(fmaf(bf16_hi(v[u].w[j]), kLog2e, -mb)) * inv);
            st_stream_v8(vy + vi * kPer, v[u]);
          }
        }
      }
      int64_t si = -1;
      if (tid < sp.head) si = tid;
      else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * kPer + (tid - sp.head);
      if (si >= 0)
        st_stream_u16(py + si,
                      to_bf16(ex2(fmaf(bf16_to_f32(ld_stream_u16(px + si)), kLog2e, -mb)) * inv));
    } else {  // chunks of 8 a thread, last to first as above (out of phase,
              // measured on GB300: 152 x 65537 29.2 us against 33.5 first to
              // last, 608 x 65537 68.8 against 75.3)
      for (int64_t base = (cols - 1) / (T * 8) * (T * 8); base >= 0; base -= T * 8) {
        uint16_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int64_t i = base + tid + T * u;
          v[u] = i < cols ? ld_stream_u16(px + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int64_t i = base + tid + T * u;
          if (i < cols)
            st_stream_u16(py + i, to_bf16(ex2(fmaf(bf16_to_f32(v[u]), kLog2e, -mb)) * inv));
        }
      }
    }
  }
}

unsigned warp_row_grid(int64_t rows) {
  return static_cast<unsigned>((rows + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32));
}

}  // namespace

// bf16 rows of at most 2048 columns in host memory, x and y in phase, ld =
// cols: the warp kernel over a grid of a quarter of the SMs' CTAs
// (FR_HOST_GRID=<CTAs> pins it).  Measured on GB300 (bf16 [65536, 1024],
// GB/s both ways): 19 CTAs 258.5, 38 335.5, 76 336.9, 152 337.7, a warp for
// every row 335.6 -- rows half the bytes of fp32 ones oversubscribe the link
// less.
cudaError_t launch_softmax_bf16_host_rows(const uint16_t *x, uint16_t *y, int64_t rows,
                                          int64_t cols, int sm_count, cudaStream_t s) {
  const int64_t nv = (cols + 32 * kPer - 1) / (32 * kPer);
  if (nv < 1 || nv > 4) return cudaErrorInvalidValue;
  int64_t grid = sm_count / 4 > 0 ? sm_count / 4 : 1;
  if (const char *e = getenv("FR_HOST_GRID")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 65535) grid = v;
  }
  const int64_t need = (rows + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32);
  if (grid > need) grid = need;
  void (*kern)(const uint16_t *, uint16_t *, int64_t, int64_t, int64_t, int64_t) =
      nv == 1 ? softmax_bf16_warp_vec<1, true> : nv == 2 ? softmax_bf16_warp_vec<2, true>
                                               : nv == 3 ? softmax_bf16_warp_vec<3, true>
                                                         : softmax_bf16_warp_vec<4, true>;
  return launch_k(kern, dim3(static_cast<unsigned>(grid)), dim3(kWarpRowThreads), 0, s, 0, x, y,
                  rows, cols, cols, cols);
}

// Rows up to 2048 take one warp; longer rows in phase take one CTA of up to
// 1024 threads x 2 vectors (32768 elements).
int64_t softmax_bf16_persistent_max_cols(bool) { return 32768; }

namespace {
template <int T, int NV>
cudaError_t launch_bf16_cta(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                            int64_t ldx, int64_t ldy, cudaStream_t s) {
  return launch_k(softmax_bf16_cta_vec<T, NV>, dim3(static_cast<unsigned>(rows)), dim3(T), 0, s,
                  0, x, y, cols, ldx, ldy);
}
}  // namespace

namespace {
// The smallest CTA size, then the smallest cluster, whose registers hold the
// row (nv vectors of 16 per thread).
bool bf16_cluster_shape(int64_t cols, int nv, int *T, int *C) {
  const int64_t nvec = cols / kPer;  // at least the body's vectors
  for (int t = 256; t <= 1024; t <<= 1)
    for (int c = 2; c <= kBfClusterMax; c <<= 1)
      if (nvec <= static_cast<int64_t>(c) * t * nv) {
        *T = t;
        *C = c;
        return true;
      }
  return false;
}

template <int T, int NV, bool RE>
cudaError_t launch_bf16_cluster(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                                int64_t ldx, int64_t ldy, int C, cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  return launch_k(softmax_bf16_cluster<T, NV, RE>, dim3(static_cast<unsigned>(rows * C)), dim3(T),
                  0, s, static_cast<unsigned>(C), x, y, cols, ldx, ldy, err);
}
}  // namespace

int64_t softmax_bf16_split_max_cols() {
  return static_cast<int64_t>(kBfClusterMax) * 1024 * 2 * kPer;
}

cudaError_t launch_softmax_bf16_split(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                                      int64_t ldx, int64_t ldy, cudaStream_t s) {
  // Exponentials recomputed in the writing pass (4 vectors a thread, twice
  // the bytes in flight) unless the row needs 1024-thread CTAs; measured on
  // GB300, bf16 [1022, 65537]: 45.6 us recomputed, 60.1 held (2 vectors a
  // thread), 55.4 looped.  FR_SOFTMAX_BF16_SPLIT=hold pins the held form.
  const char *pin = getenv("FR_SOFTMAX_BF16_SPLIT");
  const bool re = pin == nullptr || strcmp(pin, "hold") != 0;
  int T = 0, C = 0;
  if (re && bf16_cluster_shape(cols, 4, &T, &C) && T <= 512 && rows * C <= 0x7fffffff) {
    if (T == 256) return launch_bf16_cluster<256, 4, true>(x, y, rows, cols, ldx, ldy, C, s);
    return launch_bf16_cluster<512, 4, true>(x, y, rows, cols, ldx, ldy, C, s);
  }
  if (!bf16_cluster_shape(cols, 2, &T, &C) || rows * C > 0x7fffffff) return cudaErrorInvalidValue;
  switch (T) {
    case 256: return launch_bf16_cluster<256, 2, false>(x, y, rows, cols, ldx, ldy, C, s);
    case 512: return launch_bf16_cluster<512, 2, false>(x, y, rows, cols, ldx, ldy, C, s);
    default: return launch_bf16_cluster<1024, 2, false>(x, y, rows, cols, ldx, ldy, C, s);
  }
}

cudaError_t launch_softmax_bf16_persistent(const uint16_t *x, uint16_t *y, int64_t rows,
                                           int64_t cols, int64_t ldx, int64_t ldy, bool vec,
                                           int sm_count, cudaStream_t s) {
  const unsigned grid = warp_row_grid(rows);
  // In phase, rows of 8193 .. 16384 columns from 8 x SMs rows take the
  // staged kernel below too: 32 KiB of shared memory a row fits seven rows an
  // SM, where the register kernel's 512-thread CTAs fit two (measured on
  // GB300, us per call, registers / staged / looped: 16384 x 16384 153.2 /
  // 153.2 / 165.6 -- above 24 x SMs rows the same kernel --, 2432 x 16384
  // 32.2 / 26.0 / 27.9, 1216 x 16384 18.4 / 15.2 / 15.8, 1216 x 12288 15.8 /
  // 12.6 / 13.3).  FR_SOFTMAX_BF16_CTA=regs|stage pins the kernel.
  const char *cta_pin = getenv("FR_SOFTMAX_BF16_CTA");
  const bool stage_long =
      vec && cols > 8192 && cols <= 16384 &&
      (cta_pin != nullptr ? strcmp(cta_pin, "stage") == 0
                          : rows >= 8 * static_cast<int64_t>(sm_count));
  if (vec && cols > 2048 && !stage_long) {
    if (rows > 0x7fffffff) return cudaErrorInvalidValue;
    const int64_t nvec = cols / kPer;  // at least the body's vectors
    if (nvec <= 128 * 2) return launch_bf16_cta<128, 2>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 256 * 2) return launch_bf16_cta<256, 2>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 512 * 2) return launch_bf16_cta<512, 2>(x, y, rows, cols, ldx, ldy, s);
    if (nvec <= 1024 * 2) return launch_bf16_cta<1024, 2>(x, y, rows, cols, ldx, ldy, s);
    return cudaErrorInvalidValue;
  }
  // Out of phase: rows of 2049 .. 32768 columns staged in shared memory, and
  // of 1025 .. 2048 too from 32 x SMs rows, a warp per row below (measured
  // on GB300, us per call, warp / staged: 4864 x 1025 12.7 / 8.2, 16384 x
  // 1536 35.3 / 22.1, 32768 x 2048 68.8 / 54.6; 1216 x 1025 7.3 / 8.2).
  // FR_SOFTMAX_OOP=stage|warp pins the choice for 1025 .. 2048 columns.
  const char *oop = getenv("FR_SOFTMAX_OOP");
  const bool stage_short = oop != nullptr ? strcmp(oop, "stage") == 0
                                          : rows >= 32 * static_cast<int64_t>(sm_count);
  if ((!vec && (cols > 2048 || (stage_short && cols > 1024))) || stage_long) {  // staged
    if (rows > 0x7fffffff || cols > kBfStageMaxCols) return cudaErrorInvalidValue;
    // four to eight 16-byte chunks a thread
    const size_t smem = (static_cast<size_t>(cols) + 16) * 2;
    const int T = cols <= 4096 ? 64 : cols <= 8192 ? 128 : cols <= 16384 ? 256 : 512;
    auto kern = T == 64 ? softmax_bf16_cta_stage<64> : T == 128 ? softmax_bf16_cta_stage<128>
              : T == 256 ? softmax_bf16_cta_stage<256> : softmax_bf16_cta_stage<512>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_k(kern, dim3(static_cast<unsigned>(rows)), dim3(T), smem, s, 0, x, y, cols, ldx,
                    ldy);
  }
  if (vec) {
    const int64_t nv = (cols + 32 * kPer - 1) / (32 * kPer);
    switch (nv) {
      case 1: return launch_k(softmax_bf16_warp_vec<1>, dim3(grid), dim3(kWarpRowThreads), 0, s, 0, x, y, rows, cols, ldx, ldy);
      case 2: return launch_k(softmax_bf16_warp_vec<2>, dim3(grid), dim3(kWarpRowThreads), 0, s, 0, x, y, rows, cols, ldx, ldy);
      case 3: return launch_k(softmax_bf16_warp_vec<3>, dim3(grid), dim3(kWarpRowThreads), 0, s, 0, x, y, rows, cols, ldx, ldy);
      case 4: return launch_k(softmax_bf16_warp_vec<4>, dim3(grid), dim3(kWarpRowThreads), 0, s, 0, x, y, rows, cols, ldx, ldy);
      default: return cudaErrorInvalidValue;
    }
  } else {
    if (cols <= 128) softmax_bf16_warp_scalar<4><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else if (cols <= 512) softmax_bf16_warp_scalar<16><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else if (cols <= 1024) softmax_bf16_warp_scalar<32><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else if (cols <= 2048) softmax_bf16_warp_scalar<64><<<grid, kWarpRowThreads, 0, s>>>(x, y, rows, cols, ldx, ldy);
    else return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

namespace {
template <int T>
cudaError_t launch_bf16_looped_t(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                                 int64_t ldx, int64_t ldy, bool vec, int sm_count, int per_sm_cap,
                                 cudaStream_t s) {
  auto kern = vec ? softmax_bf16_block_looped<true, T> : softmax_bf16_block_looped<false, T>;
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

cudaError_t launch_softmax_bf16_looped(const uint16_t *x, uint16_t *y, int64_t rows,
                                       int64_t cols, int64_t ldx, int64_t ldy, bool vec,
                                       int sm_count, cudaStream_t s) {
  // As for fp32: many rows take small CTAs, as many per SM as fit (the
  // smallest that covers a row's vectors in one chunk); few rows 512-thread
  // CTAs, two per SM.  Measured on GB300, bf16 [16380, 4097]: 54.2 us with
  // 128 threads, 84.5 with 256, 148.5 with 512.  FR_SOFTMAX_LOOP=128|256|512
  // pins the CTA size.
  const char *e = getenv("FR_SOFTMAX_LOOP");
  int t = 512;
  if (e != nullptr) t = atoi(e);
  else if (rows >= 4 * static_cast<int64_t>(sm_count)) t = cols / kPer <= 128 * kLoopU ? 128 : 256;
  if (t == 128) return launch_bf16_looped_t<128>(x, y, rows, cols, ldx, ldy, vec, sm_count, 16, s);
  if (t == 256) return launch_bf16_looped_t<256>(x, y, rows, cols, ldx, ldy, vec, sm_count, 16, s);
  return launch_bf16_looped_t<512>(x, y, rows, cols, ldx, ldy, vec, sm_count, 2, s);
}

}  // namespace fr
