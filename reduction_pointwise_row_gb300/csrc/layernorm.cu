// LayerNorm over rows of bf16 with Welford statistics.
//
// The pages name LayerNorm only as an example of an operator a tile DSL must
// express ("CMU 15-779 Lecture 8", section 1); the definition is the standard
// one: mean = sum x / n, var = sum (x - mean)^2 / n (biased),
// rstd = 1/sqrt(var + eps), y = (x - mean) * rstd * gamma + beta -> bf16 (RNE).
//
// Statistics: each thread turns a chunk of its elements into a Welford triple
// (count, mean, M2) by a two-pass over registers (no division per element),
// triples are combined with the parallel merge of Chan, Golub and LeVeque
// (1979):  n = na + nb,  delta = mb - ma,  mean = ma + delta * nb / n,
// M2 = M2a + M2b + delta^2 * na * nb / n.  All in fp32.
//
// Kernels, in the order the looped form prefers them:
// layernorm_cluster_full  rows of C*T*32 columns (C in 1, 2, 4, 8 CTAs of T in
//             64 .. 512 threads): a persistent grid of thread-block clusters,
//             each CTA owning a fixed column slice of every row (its gamma and
//             beta held in registers), each row slice staged in shared memory
//             by one bulk copy, the C slices' (mean, M2) pairs exchanged
//             through distributed shared memory and merged with equal counts;
//             the default for 2048 .. 131072 columns.
// layernorm_cluster  the same with 512 threads and C = 1 or 2 for other
//             lengths that are multiples of 32 * C (per-thread cp.async ring).
// layernorm_ring  one persistent CTA per SM, rows staged whole in a ring of
//             shared-memory buffers (per-thread cp.async or one bulk copy per
//             row), R rows normalised per gamma/beta pass.
// layernorm_looped_scalar  any alignment and length: lane-strided scalars,
//             pass 1 merges Welford triples over chunks, pass 2 re-reads the
//             row (from L2) to write y.
// layernorm_persistent  the persistent form: one CTA per row, the row held in
//             registers as packed bf16 (x read once, y written once).
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

struct Welford {
  float n, mean, m2;
};

// The merge weight nb / n uses the approximate reciprocal (within one ulp, and
// exact for the power-of-two counts the balanced merge trees produce): a
// correctly rounded division here costs more than the rest of the merge, and
// measured on GB300 it made the LayerNorm kernels 12-34 % slower.
__device__ __forceinline__ Welford chan_merge(Welford a, Welford b) {
  const float n = a.n + b.n;
  if (n == 0.0f) return Welford{0.0f, 0.0f, 0.0f};
  float rn;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rn) : "f"(n));
  const float delta = b.mean - a.mean;
  const float fb = b.n * rn;
  Welford r;
  r.n = n;
  r.mean = fmaf(delta, fb, a.mean);
  r.m2 = a.m2 + b.m2 + delta * delta * a.n * fb;
  return r;
}

// Chan's merge of two sides of equal count 2 half_n: weight 1/2, correction
// delta^2 * half_n (no reciprocal).
__device__ __forceinline__ void merge_equal(float &mean, float &m2, float mean_b, float m2_b,
                                            float half_n) {
  const float delta = mean_b - mean;
  mean = fmaf(delta, 0.5f, mean);
  m2 = fmaf(delta * delta, half_n, m2 + m2_b);
}

__device__ __forceinline__ Welford warp_welford(Welford w) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Welford v{__shfl_xor_sync(0xffffffffu, w.n, o), __shfl_xor_sync(0xffffffffu, w.mean, o),
              __shfl_xor_sync(0xffffffffu, w.m2, o)};
    w = chan_merge(w, v);
  }
  return w;
}

// CTA-wide merge; returns the row triple to every thread.  smem: >= 32 entries.
__device__ __forceinline__ Welford block_welford(Welford w, Welford *smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  w = warp_welford(w);
  if (lane == 0) smem[warp] = w;
  __syncthreads();
  Welford r = lane < nw ? smem[lane] : Welford{0.0f, 0.0f, 0.0f};
  r = warp_welford(r);
  __syncthreads();
  return r;
}

// Welford triple of 16 bf16 values packed in a V8 (two passes over registers).
__device__ __forceinline__ Welford welford16(const V8 &v) {
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += bf16_lo(v.w[j]) + bf16_hi(v.w[j]);
  const float mean = s * (1.0f / 16.0f);
  float q = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float a = bf16_lo(v.w[j]) - mean, b = bf16_hi(v.w[j]) - mean;
    q = fmaf(a, a, q);
    q = fmaf(b, b, q);
  }
  return Welford{16.0f, mean, q};
}

// Bound of every mbarrier wait, in SM clocks (about one second).  A wait that
// runs out records FR_DEVERR_TIMEOUT; its kernel then issues no further copy,
// skips its remaining waits on data (its outputs are garbage) and, before it
// exits, waits -- again bounded -- for the copies it issued before the timeout.
constexpr long long kWaitBudget = 1LL << 31;
// The first wait of layernorm_ring's bulk staging.  A test build
// (-DFR_TEST_WAIT_BUDGET=<clocks>) shortens its budget so that it runs out
// while its copy is still in flight, to exercise the path above; every other
// wait, the final drain included, keeps the full budget.
// The shortened wait polls without blocking (mbarrier.try_wait may suspend
// the thread for a while before it gives up; test_wait answers at once).
__device__ __forceinline__ bool first_wait(uint64_t *bar, uint32_t parity) {
#ifdef FR_TEST_WAIT_BUDGET
  const long long t0 = clock64();
  while (!mbar_test_wait(bar, parity))
    if (clock64() - t0 > FR_TEST_WAIT_BUDGET) return false;
  return true;
#else
  return mbar_wait_bounded(bar, parity, kWaitBudget);
#endif
}

// ---- row groups: gamma/beta in shared memory, rows in registers --------------
// For rows up to 16384 columns (cols % 8 == 0, 16-byte aligned rows and
// gamma/beta).  A persistent grid of 256-thread CTAs, each holding the whole
// of gamma and beta in shared memory (loaded once), works on rows with
// groups of WG warps: 8 / WG rows at a time per CTA.  Thread j of a group owns
// the 16-byte chunks j + 32 WG c (c < NC) of its row, 8 columns each, so a
// warp's loads and stores are 512 contiguous bytes.  Statistics: each thread's
// values two-pass in registers (sum, then squared deviations), triples merged
// with Chan's formula across the warp by shuffles and across the group's
// warps through shared memory (one named barrier per row, slots double
// buffered); when every thread holds the same number of chunks, every merge
// joins equal counts and takes no reciprocal.  One read of x, one write of y;
// gamma/beta come from shared memory for every row.
constexpr int kRgThreads = 256;

template <int WG>
__device__ __forceinline__ void group_sync(int group) {
  if constexpr (WG > 1)
    asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(WG * 32) : "memory");
}

// Chan merge that returns the other side exactly when one side is empty.
__device__ __forceinline__ Welford merge_or_keep(Welford a, Welford b) {
  if (b.n == 0.0f) return a;
  if (a.n == 0.0f) return b;
  return chan_merge(a, b);
}

// PF: the next row's chunks are loaded while the current row is worked on.
// PL: gamma/beta in shared memory as four float4 planes (below); otherwise
// chunk by chunk, gamma [cols] then beta [cols].
// EQ: every thread of a group holds the same number of chunks (the row's
// chunks are a multiple of the group's threads), so every merge joins two
// equal counts (weight 1/2, no reciprocal); otherwise Chan's general merge.
// Launch bounds: three CTAs an SM (at most 80 registers a thread) where a
// thread holds at most 8 chunks of rows, counting the prefetched one.
// Measured on GB300 (256 MiB of x, us per call, bounds of 1 / 3 / 4 CTAs):
// 768 columns 94.5 / 84.1 / 90.1, 1024 89.1 / 84.3 / 85.6, 2560 100.4 /
// 87.4 / 92.6, 4096 94.4 / 86.6 / 89.8, 8192 93.1 / 88.3 / 85.5: left to
// itself the compiler stopped at 64 registers with spills; at four CTAs it
// spills more.
template <int WG, int NC, bool PF, bool PL, bool EQ>
__global__ void __launch_bounds__(kRgThreads, NC * (PF ? 2 : 1) <= 8 ? 3 : 1)
layernorm_rows(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
               const float *__restrict__ beta, uint16_t *__restrict__ y,
               float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
               int64_t cols, int64_t ldx, int64_t ldy, float eps, float inv_n,
               float inv_nt_eq, float half_nt_eq) {
  pdl_enter();
  constexpr int kGroups = kRgThreads / 32 / WG;  // rows a CTA works on at once
  // gamma and beta of chunk j (its 8 columns) as four float4 planes:
  // gb[j] = gamma 8j..8j+3, gb[nch + j] = gamma 8j+4..8j+7, then beta the
  // same at 2 nch and 3 nch, so a warp reading one plane for 32 consecutive
  // chunks reads 512 contiguous bytes (one 32-byte chunk a lane would take
  // twice the shared-memory wavefronts)
  extern __shared__ __align__(16) float4 gb[];
  __shared__ Welford part[2][kRgThreads / 32];     // per-warp triples, by row parity
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = warp / WG, gt = (warp % WG) * 32 + lane;
  const int nch = static_cast<int>(cols >> 3);  // 16-byte chunks of a row
  if constexpr (PL) {
    for (int i = tid; i < nch * 4; i += kRgThreads) {
      const int plane = i / nch, j = i - plane * nch;
      gb[i] = ld_keep_f4((plane < 2 ? gamma : beta) + 8 * j + 4 * (plane & 1));
    }
  } else {
    for (int i = tid; i < nch * 4; i += kRgThreads)
      gb[i] = ld_keep_f4((i < 2 * nch ? gamma : beta - 8 * nch) + 4 * i);
  }
  __syncthreads();
  const uint64_t policy = l2_evict_first_policy();
  int nv = 0;  // this thread's chunks of a row
#pragma unroll
  for (int c = 0; c < NC; ++c) nv += gt + 32 * WG * c < nch;
  // 1 / cols, and with equal counts 1 / (values a thread) and half of that
  // count, come from the host as arguments
  const float n_t = static_cast<float>(8 * nv);
  const float inv_nt = EQ ? inv_nt_eq : nv > 0 ? 1.0f / n_t : 0.0f;
  const int64_t step = static_cast<int64_t>(gridDim.x) * kGroups;
  int64_t row = static_cast<int64_t>(blockIdx.x) * kGroups + group;
  uint4 nx[PF ? NC : 1];
  if constexpr (PF) {
    if (row < rows) {
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (c < nv) nx[c] = ld_stream_u4(x + row * ldx + 8 * (gt + 32 * WG * c), policy);
    }
  }
  int it = 0;
  for (; row < rows; row += step, ++it) {
    uint4 v[NC];
    if constexpr (PF) {
#pragma unroll
      for (int c = 0; c < NC; ++c) v[c] = nx[c];
      if (row + step < rows) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (c < nv) nx[c] = ld_stream_u4(x + (row + step) * ldx + 8 * (gt + 32 * WG * c), policy);
      }
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (c < nv) v[c] = ld_stream_u4(x + row * ldx + 8 * (gt + 32 * WG * c), policy);
    }
    // two passes over the thread's values: mean, then squared deviations
    uint64_t s2 = 0;
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (c < nv) {
        s2 = add_f32x2(s2, add_f32x2(pack_f32x2(bf16_lo(v[c].x), bf16_hi(v[c].x)),
                                     pack_f32x2(bf16_lo(v[c].y), bf16_hi(v[c].y))));
        s2 = add_f32x2(s2, add_f32x2(pack_f32x2(bf16_lo(v[c].z), bf16_hi(v[c].z)),
                                     pack_f32x2(bf16_lo(v[c].w), bf16_hi(v[c].w))));
      }
    const float mean_t = (f32x2_lo(s2) + f32x2_hi(s2)) * inv_nt;
    const uint64_t nm = pack_f32x2(-mean_t, -mean_t);
    uint64_t q2 = 0;
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (c < nv) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint64_t d = add_f32x2(pack_f32x2(bf16_lo(w[h]), bf16_hi(w[h])), nm);
          q2 = fma_f32x2(d, d, q2);
        }
      }
    float mean, m2;
    if constexpr (EQ) {
      mean = mean_t;
      m2 = f32x2_lo(q2) + f32x2_hi(q2);
      float hn = half_nt_eq;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1, hn *= 2.0f)
        merge_equal(mean, m2, __shfl_xor_sync(0xffffffffu, mean, o),
                    __shfl_xor_sync(0xffffffffu, m2, o), hn);
      if constexpr (WG > 1) {
        // the group's WG pairs (equal counts) on lanes 0 .. WG - 1, merged
        // by a fixed xor tree
        if (lane == 0) part[it & 1][warp] = Welford{0.0f, mean, m2};
        group_sync<WG>(group);
        const Welford u = part[it & 1][group * WG + (lane & (WG - 1))];
        mean = u.mean;
        m2 = u.m2;
#pragma unroll
        for (int o = WG / 2; o > 0; o >>= 1, hn *= 2.0f)
          merge_equal(mean, m2, __shfl_xor_sync(0xffffffffu, mean, o),
                      __shfl_xor_sync(0xffffffffu, m2, o), hn);
      }
      // lane 0's result in every lane (the xor tree's lanes may differ in
      // the last bit)
      mean = __shfl_sync(0xffffffffu, mean, 0);
      m2 = __shfl_sync(0xffffffffu, m2, 0);
    } else {
      Welford t = warp_welford(Welford{n_t, mean_t, f32x2_lo(q2) + f32x2_hi(q2)});
      if constexpr (WG > 1) {
        // the group's WG triples on lanes 0 .. WG - 1, merged by a fixed xor
        // tree (the same bits in every warp of the group)
        if (lane == 0) part[it & 1][warp] = t;
        group_sync<WG>(group);
        t = lane < WG ? part[it & 1][group * WG + lane] : Welford{0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int o = WG / 2; o > 0; o >>= 1)
          t = merge_or_keep(t, Welford{__shfl_xor_sync(0xffffffffu, t.n, o),
                                       __shfl_xor_sync(0xffffffffu, t.mean, o),
                                       __shfl_xor_sync(0xffffffffu, t.m2, o)});
      }
      mean = __shfl_sync(0xffffffffu, t.mean, 0);
      m2 = __shfl_sync(0xffffffffu, t.m2, 0);
    }
    const float rstd = rsqrtf(fmaf(m2, inv_n, eps));
    if (gt == 0) {
      if (mean_out) mean_out[row] = mean;
      if (rstd_out) rstd_out[row] = rstd;
    }
    uint16_t *yr = y + row * ldy;
    const uint64_t nmr = pack_f32x2(-mean, -mean), r2 = pack_f32x2(rstd, rstd);
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (c < nv) {
        const int j = gt + 32 * WG * c;
        const float4 g0 = PL ? gb[j] : gb[2 * j], g1 = PL ? gb[nch + j] : gb[2 * j + 1],
                     b0 = PL ? gb[2 * nch + j] : gb[2 * nch + 2 * j],
                     b1 = PL ? gb[3 * nch + j] : gb[2 * nch + 2 * j + 1];
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        const uint64_t gg[4] = {pack_f32x2(g0.x, g0.y), pack_f32x2(g0.z, g0.w),
                                pack_f32x2(g1.x, g1.y), pack_f32x2(g1.z, g1.w)};
        const uint64_t bb[4] = {pack_f32x2(b0.x, b0.y), pack_f32x2(b0.z, b0.w),
                                pack_f32x2(b1.x, b1.y), pack_f32x2(b1.z, b1.w)};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint64_t d = add_f32x2(pack_f32x2(bf16_lo(w[h]), bf16_hi(w[h])), nmr);
          const uint64_t yv = fma_f32x2(mul_f32x2(d, r2), gg[h], bb[h]);
          o[h] = pack_bf16x2(f32x2_lo(yv), f32x2_hi(yv));
        }
        st_stream_u4(yr + 8 * j, make_uint4(o[0], o[1], o[2], o[3]));
      }
  }
}

// Persistent form.  Requires 32-byte aligned x/y rows, gamma, beta and
// cols % 16 == 0 (checked by the host); NV vectors of 16 per thread.
constexpr int kPersistMaxThreads = 512;

template <int NV>  // four vectors a thread need more than the 64 registers two CTAs leave
__global__ void __launch_bounds__(kPersistMaxThreads, NV >= 4 ? 1 : 2)
layernorm_persistent(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
                     const float *__restrict__ beta, uint16_t *__restrict__ y,
                     float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t cols,
                     int64_t ldx, int64_t ldy, float eps) {
  __shared__ Welford red[32];
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  const int nvec = static_cast<int>(cols >> 4);  // <= 2048 here
  const uint16_t *px = x + row * ldx;
  V8 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int vi = tid + T * k;
    if (vi < nvec) v[k] = ld_stream_v8(px + vi * 16);
  }
  Welford w{0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (tid + T * k < nvec) w = chan_merge(w, welford16(v[k]));
  const Welford r = block_welford(w, red);
  const float mean = r.mean;
  const float rstd = rsqrtf(fmaf(r.m2, __frcp_rn(r.n), eps));
  if (tid == 0) {
    if (mean_out) mean_out[row] = mean;
    if (rstd_out) rstd_out[row] = rstd;
  }
  uint16_t *py = y + row * ldy;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int vi = tid + T * k;
    if (vi < nvec) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {  // 4 columns of gamma/beta at a time; y overwrites x
        const float4 g = ld_keep_f4(gamma + vi * 16 + 4 * h);
        const float4 b = ld_keep_f4(beta + vi * 16 + 4 * h);
        const uint32_t w0 = v[k].w[2 * h], w1 = v[k].w[2 * h + 1];
        v[k].w[2 * h] = pack_bf16x2(fmaf((bf16_lo(w0) - mean) * rstd, g.x, b.x),
                                    fmaf((bf16_hi(w0) - mean) * rstd, g.y, b.y));
        v[k].w[2 * h + 1] = pack_bf16x2(fmaf((bf16_lo(w1) - mean) * rstd, g.z, b.z),
                                        fmaf((bf16_hi(w1) - mean) * rstd, g.w, b.w));
      }
      st_stream_v8(py + vi * 16, v[k]);
    }
  }
}

constexpr int kLoopThreads = 512;

// Looped form, any alignment: lane-strided scalars, chunks of 8 per thread.
__global__ void __launch_bounds__(kLoopThreads)
layernorm_looped_scalar(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
                        const float *__restrict__ beta, uint16_t *__restrict__ y,
                        float *__restrict__ mean_out, float *__restrict__ rstd_out,
                        int64_t rows, int64_t cols, int64_t ldx, int64_t ldy, float eps) {
  __shared__ Welford red[32];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint16_t *px = x + row * ldx;
    Welford w{0.0f, 0.0f, 0.0f};
    for (int64_t base = 0; base < cols; base += kLoopThreads * 8) {
      float v[8];
      float s = 0.0f;
      int c = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = base + tid + kLoopThreads * u;
        v[u] = i < cols ? bf16_to_f32(px[i]) : 0.0f;
        s += v[u];
        c += i < cols;
      }
      if (c == 0) continue;
      const float cm = s * __frcp_rn(static_cast<float>(c));
      float q = 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (base + tid + kLoopThreads * u < cols) q = fmaf(v[u] - cm, v[u] - cm, q);
      w = chan_merge(w, Welford{static_cast<float>(c), cm, q});
    }
    const Welford r = block_welford(w, red);
    const float mean = r.mean;
    const float rstd = rsqrtf(fmaf(r.m2, __frcp_rn(r.n), eps));
    if (tid == 0) {
      if (mean_out) mean_out[row] = mean;
      if (rstd_out) rstd_out[row] = rstd;
    }
    uint16_t *py = y + row * ldy;
    for (int64_t i = tid; i < cols; i += kLoopThreads)
      py[i] = to_bf16(fmaf((bf16_to_f32(px[i]) - mean) * rstd, gamma[i], beta[i]));
  }
}

// ---- looped form with asynchronous-copy staging -----------------------------
// A persistent CTA per SM owns rows blockIdx.x + k * gridDim.x, stages them in
// a ring of kRingBufs shared-memory row buffers (row k in buffer k % kRingBufs)
// and works on R rows at a time.  Every thread copies its own 32-byte pieces
// of a row with cp.async (16 bytes per copy, one commit group per row) and
// later reads back exactly those pieces, so staging needs no barrier of its
// own.  Pass 1 lifts the R rows' pieces into registers (Welford triples per 16
// elements) and immediately refills their buffers with the next rows, so
// kRingBufs rows are always in flight; after one CTA merge of the R triples,
// pass 2 normalises all R rows from registers with one load of each
// gamma/beta value -- the fp32 gamma/beta re-reads, four times the bytes of
// x, are what limit a one-row-at-a-time LayerNorm.
constexpr int kRingThreads = 512;
constexpr int kRingBufs = 3;
constexpr int kRingPieces = 4;    // 32-byte pieces per thread per row: rows of
                                  // at most 512 * 4 * 16 = 32768 bf16

// CTA-wide merge of R triples at once (one pair of barriers for all R).
template <int R>
__device__ __forceinline__ void block_welford_n(Welford (&w)[R], Welford (*smem)[32]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    w[r] = warp_welford(w[r]);
    if (lane == 0) smem[r][warp] = w[r];
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    Welford t = lane < nw ? smem[r][lane] : Welford{0.0f, 0.0f, 0.0f};
    w[r] = warp_welford(t);
  }
  __syncthreads();
}

// BULK: stage each row with one bulk asynchronous copy completing on an
// mbarrier (the copy writes shared memory without the load/store path that
// per-thread copies occupy) instead of per-thread cp.async.
template <int R, bool BULK>
__global__ void __launch_bounds__(kRingThreads, 1)
layernorm_ring(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
               const float *__restrict__ beta, uint16_t *__restrict__ y,
               float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
               int64_t cols, int64_t ldx, int64_t ldy, float eps, int *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Welford red[R][32];
  __shared__ __align__(8) uint64_t full[kRingBufs];
  __shared__ int timed_out;
  const int tid = threadIdx.x;
  const int npieces = static_cast<int>(cols >> 4);  // cols % 16 == 0
  const size_t buf_bytes = static_cast<size_t>(npieces) * 32;
  const int64_t G = gridDim.x;
  // rows of this CTA: blockIdx.x + k * G for k < nk
  const int64_t nk = blockIdx.x < rows ? (rows - blockIdx.x + G - 1) / G : 0;
  const uint64_t policy = l2_evict_first_policy();
  int64_t last_issued = -1;  // thread 0: the last row whose bulk copy it issued

  auto stage_bulk = [&](int64_t k) {  // thread 0: row k into buffer k % kRingBufs
    if (k < nk) {
      const int b = static_cast<int>(k % kRingBufs);
      mbar_arrive_expect_tx(&full[b], static_cast<uint32_t>(buf_bytes));
      bulk_copy_g2s(smem + static_cast<size_t>(b) * buf_bytes, x + (blockIdx.x + k * G) * ldx,
                    static_cast<uint32_t>(buf_bytes), &full[b], policy);
      last_issued = k;
    }
  };
  auto stage = [&](int64_t k) {  // this thread's pieces of row k into buffer k % kRingBufs
    if constexpr (BULK) return;
    if (k < nk) {
      const unsigned char *src = reinterpret_cast<const unsigned char *>(x + (blockIdx.x + k * G) * ldx);
      unsigned char *dst = smem + static_cast<size_t>(k % kRingBufs) * buf_bytes;
#pragma unroll
      for (int j = 0; j < kRingPieces; ++j) {
        const int p = tid + j * kRingThreads;
        if (p < npieces) {
          cp_async_16(dst + static_cast<size_t>(p) * 32, src + static_cast<size_t>(p) * 32);
          cp_async_16(dst + static_cast<size_t>(p) * 32 + 16, src + static_cast<size_t>(p) * 32 + 16);
        }
      }
    }
    cp_async_commit();  // one group per row index, empty past the last row
  };

  if constexpr (BULK) {
    if (tid == 0) {
      timed_out = 0;
      for (int b = 0; b < kRingBufs; ++b) mbar_init(&full[b], 1);
      mbar_init_fence();
      for (int b = 0; b < kRingBufs; ++b) stage_bulk(b);
    }
    __syncthreads();
  } else {
    for (int b = 0; b < kRingBufs; ++b) stage(b);
  }
  int64_t next = kRingBufs;  // next row index to stage
  for (int64_t k0 = 0; k0 < nk; k0 += R) {
    V8 v[R][kRingPieces];
    Welford w[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if constexpr (BULK) {
        const int64_t kk = k0 + r;
        const uint32_t par = static_cast<uint32_t>((kk / kRingBufs) & 1);
        if (kk < nk && !timed_out &&
            !(kk == 0 ? first_wait(&full[0], par)
                      : mbar_wait_bounded(&full[kk % kRingBufs], par, kWaitBudget))) {
          timed_out = 1;
          atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
        }
      } else {
        // Groups committed so far: rows 0 .. next - 1 = k0 + r + kRingBufs - 1.
        // Row k0 + r has landed once at most the kRingBufs - 1 newer ones pend.
        cp_async_wait<kRingBufs - 1>();
      }
      w[r] = Welford{0.0f, 0.0f, 0.0f};
      const unsigned char *buf = smem + static_cast<size_t>((k0 + r) % kRingBufs) * buf_bytes;
#pragma unroll
      for (int j = 0; j < kRingPieces; ++j) {
        const int p = tid + j * kRingThreads;
        if (k0 + r < nk && p < npieces) {
          v[r][j] = lds_v8(buf + static_cast<size_t>(p) * 32);
          w[r] = chan_merge(w[r], welford16(v[r][j]));
        }
      }
      stage(next++);  // buffer of row k0 + r is in registers: refill it
    }
    block_welford_n<R>(w, red);
    if constexpr (BULK) {
      // every thread has read the R buffers (the reduction's barriers lie
      // between): refill them with the next rows
      if (tid == 0 && !timed_out) {
        fence_proxy_async_smem();
#pragma unroll
        for (int r = 0; r < R; ++r) stage_bulk(next - R + r);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t row = blockIdx.x + (k0 + r) * G;
      if (k0 + r < nk && tid == 0) {
        if (mean_out) mean_out[row] = w[r].mean;
        if (rstd_out) rstd_out[row] = rsqrtf(fmaf(w[r].m2, __frcp_rn(w[r].n), eps));
      }
    }
    float mean[R], rstd[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      mean[r] = w[r].mean;
      rstd[r] = rsqrtf(fmaf(w[r].m2, __frcp_rn(w[r].n), eps));
    }
#pragma unroll
    for (int j = 0; j < kRingPieces; ++j) {
      const int p = tid + j * kRingThreads;
      if (p >= npieces) continue;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float4 g = ld_keep_f4(gamma + p * 16 + 4 * h);
        const float4 bb = ld_keep_f4(beta + p * 16 + 4 * h);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t w0 = v[r][j].w[2 * h], w1 = v[r][j].w[2 * h + 1];
          v[r][j].w[2 * h] = pack_bf16x2(fmaf((bf16_lo(w0) - mean[r]) * rstd[r], g.x, bb.x),
                                         fmaf((bf16_hi(w0) - mean[r]) * rstd[r], g.y, bb.y));
          v[r][j].w[2 * h + 1] = pack_bf16x2(fmaf((bf16_lo(w1) - mean[r]) * rstd[r], g.z, bb.z),
                                             fmaf((bf16_hi(w1) - mean[r]) * rstd[r], g.w, bb.w));
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (k0 + r < nk)
          st_stream_v8(y + (blockIdx.x + (k0 + r) * G) * ldy + static_cast<int64_t>(p) * 16,
                       v[r][j]);
    }
  }
  cp_async_wait<0>();  // no copy may still target this CTA's shared memory
  if constexpr (BULK) {
    // After a timeout thread 0 issued no further copy.  A buffer is refilled
    // only once every thread's wait on its previous row succeeded, so at most
    // its latest copy can be in flight, and the latest copies of the
    // kRingBufs buffers are those of the last kRingBufs rows issued: wait for
    // each (a completed phase returns at once).
    __syncthreads();
    if (tid == 0 && timed_out)
      for (int64_t k = last_issued - kRingBufs + 1 < 0 ? 0 : last_issued - kRingBufs + 1;
           k <= last_issued; ++k)
        mbar_wait_bounded(&full[k % kRingBufs], static_cast<uint32_t>((k / kRingBufs) & 1),
                          kWaitBudget);
  }
}

// ---- cluster form: gamma/beta resident in registers -----------------------------
// (The general cluster kernel; the equal-count kernel below takes clusters of
// up to 8 CTAs.)  A cluster of C CTAs (C = 1 or 2) splits every row into C column slices of
// S = cols / C <= 16384; thread t of CTA rank q owns the 32 columns
// q*S + 32t .. + 31 for the whole kernel, so its 32 gamma and 32 beta values
// live in registers and per row only x comes in and y goes out -- no per-row
// re-read of the fp32 gamma/beta (4x the bytes of x).  Each thread streams its
// 64-byte pieces of the cluster's rows through a kClStages-deep cp.async ring
// (no barrier: every thread reads back exactly what it copied).  Per row:
// Welford triple of 32 elements -> warp -> CTA (warp 0) -> pushed into every
// CTA of the cluster (st.async, counted on the receiver's mbarrier).  Row k is
// published before row k - 1 is finalised (merge of the C triples in rank
// order, identical in every CTA, then normalisation of the x held in
// registers), so the exchange latency overlaps the next row's work.
constexpr int kClThreads = 512;
constexpr int kClCols = 32;      // columns per thread
constexpr int kClStages = 4;     // rows in the cp.async ring
constexpr int kClSlots = 4;      // triple slots: a peer writes row k + 4 only after
                                 // this CTA published row k + 2, i.e. after it
                                 // finalised row k
constexpr int kClMaxCluster = 2;
constexpr int64_t kClMaxSlice = static_cast<int64_t>(kClCols) * kClThreads;  // 16384

__global__ void __launch_bounds__(kClThreads, 1)
layernorm_cluster(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
                  const float *__restrict__ beta, uint16_t *__restrict__ y,
                  float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char smem[];  // [kClStages][T] x 64 bytes
  __shared__ __align__(16) float4 slot[kClSlots][kClMaxCluster];  // [row % 4][rank]
  __shared__ __align__(8) uint64_t pbar[kClSlots];
  __shared__ Welford red[2][32];  // per-warp triples, double-buffered by row
  __shared__ int timed_out;

  const uint32_t C = cluster_nctarank(), q = cluster_ctarank();
  const int64_t cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t S = cols / C;
  const bool own = static_cast<int64_t>(kClCols) * tid < S;
  const int64_t col0 = static_cast<int64_t>(q) * S + static_cast<int64_t>(kClCols) * tid;
  const int64_t nr = cid < rows ? (rows - cid + ncl - 1) / ncl : 0;  // rows of this cluster
  const uint32_t part_bytes = 16u * C;

  float g[kClCols], b[kClCols];
  if (own) {
#pragma unroll
    for (int h = 0; h < kClCols / 4; ++h) {
      const float4 gv = ld_keep_f4(gamma + col0 + 4 * h), bv = ld_keep_f4(beta + col0 + 4 * h);
      g[4 * h] = gv.x; g[4 * h + 1] = gv.y; g[4 * h + 2] = gv.z; g[4 * h + 3] = gv.w;
      b[4 * h] = bv.x; b[4 * h + 1] = bv.y; b[4 * h + 2] = bv.z; b[4 * h + 3] = bv.w;
    }
  }
  auto row_of = [&](int64_t k) { return cid + k * ncl; };
  auto piece = [&](int64_t k) {
    return smem + (static_cast<size_t>(k % kClStages) * kClThreads + tid) * 64;
  };
  auto stage = [&](int64_t k) {  // this thread's 64 bytes of row k
    if (k < nr && own) {
      const uint16_t *src = x + row_of(k) * ldx + col0;
      unsigned char *dst = piece(k);
#pragma unroll
      for (int c = 0; c < 4; ++c) cp_async_16(dst + 16 * c, src + 8 * c);
    }
    cp_async_commit();
  };

  if (tid == 0) {
    timed_out = 0;
    for (int i = 0; i < kClSlots; ++i) mbar_init(&pbar[i], 1);
    mbar_init_fence();
    for (int64_t k = 0; k < kClSlots && k < nr; ++k) mbar_arrive_expect_tx(&pbar[k], part_bytes);
  }
  for (int i = 0; i < kClStages - 1; ++i) stage(i);
  __syncthreads();
  cluster_arrive();  // every CTA's barriers are armed before anyone sends
  cluster_wait();

  V8 xa[2], xb[2];  // rows k (current) and k - 1 (being finalised): 32 bf16 each
  for (int64_t k = 0; k <= nr; ++k) {
    if (k < nr) {
      stage(k + kClStages - 1);
      cp_async_wait<kClStages - 1>();  // row k landed
      Welford w{0.0f, 0.0f, 0.0f};
      if (own) {
        xa[0] = lds_v8(piece(k));
        xa[1] = lds_v8(piece(k) + 32);
        w = chan_merge(welford16(xa[0]), welford16(xa[1]));
      }
      w = warp_welford(w);
      if (lane == 0) red[k & 1][warp] = w;
      __syncthreads();
      if (warp == 0) {  // only warp 0 needs the CTA's triple
        Welford m = lane < kClThreads / 32 ? red[k & 1][lane] : Welford{0.0f, 0.0f, 0.0f};
        m = warp_welford(m);
        if (lane < static_cast<int>(C)) {
          const int sl = static_cast<int>(k % kClSlots);
          st_async_f4(&slot[sl][q], &pbar[sl], static_cast<uint32_t>(lane),
                      make_float4(m.n, m.mean, m.m2, 0.0f));
        }
      }
    }
    if (k > 0) {  // finalise row k - 1 with the x held in xb
      const int64_t kp = k - 1;
      const int sl = static_cast<int>(kp % kClSlots);
      if (!timed_out &&
          !mbar_wait_bounded(&pbar[sl], static_cast<uint32_t>((kp / kClSlots) & 1), kWaitBudget)) {
        timed_out = 1;
        atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
      }
      const float4 u0 = slot[sl][0];
      Welford t{u0.x, u0.y, u0.z};
      if (C == 2) {  // rank order: identical in every CTA
        const float4 u1 = slot[sl][1];
        t = chan_merge(t, Welford{u1.x, u1.y, u1.z});
      }
      // Re-arm slot sl for row kp + 4 (peers send it only after this CTA
      // publishes row kp + 2, which comes after this point).
      if (tid == 0 && kp + kClSlots < nr) mbar_arrive_expect_tx(&pbar[sl], part_bytes);
      const int64_t row = row_of(kp);
      const float mean = t.mean;
      const float rstd = rsqrtf(fmaf(t.m2, __frcp_rn(t.n), eps));
      if (q == 0 && tid == 0) {
        if (mean_out) mean_out[row] = mean;
        if (rstd_out) rstd_out[row] = rstd;
      }
      if (own) {
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
          V8 o;
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const int c = 16 * hv + 2 * h;
            o.w[h] = pack_bf16x2(fmaf((bf16_lo(xb[hv].w[h]) - mean) * rstd, g[c], b[c]),
                                 fmaf((bf16_hi(xb[hv].w[h]) - mean) * rstd, g[c + 1], b[c + 1]));
          }
          st_stream_v8(y + row * ldy + col0 + 16 * hv, o);
        }
      }
    }
    xb[0] = xa[0];
    xb[1] = xa[1];
  }
  cp_async_wait<0>();
  // No CTA may leave while a peer can still write into its shared memory.
  cluster_arrive();
  cluster_wait();
}

// ---- the cluster form when every thread holds 32 columns ----------------------
// When cols = C * 512 * 32 (every thread of every CTA owns exactly 32
// columns) all the triples merged at one tree level have equal counts, and
// the Chan merge needs no reciprocal: with n_a = n_b = n the weight is 1/2 and
// the correction delta^2 * n_a * n_b / (n_a + n_b) is delta^2 * n / 2.  The
// per-element work uses paired fp32 instructions (two columns per
// instruction).  Each CTA's 32 KB slice of a row arrives in shared memory by
// one bulk asynchronous copy (the tensor-memory-accelerator path, which does
// not occupy the load/store pipe that per-thread copies and the shared-memory
// reads share), completing on the slot's mbarrier; the row being finalised is
// read again from its slot instead of being held in registers.  Otherwise the
// same design as layernorm_cluster.
// Ring geometry of layernorm_cluster_full<R, A>: A rows in flight ahead of
// the step being reduced, and 2R + A row slots (the previous step's R rows,
// this step's R and those ahead).
__host__ __device__ constexpr int full_slots(int R, int A) { return 2 * R + A; }
constexpr int kFullMaxCluster = 8;

// Two bf16 values of a word as a pair of fp32 (low half first).
__device__ __forceinline__ uint64_t unpack_pair(uint32_t w) {
  return pack_f32x2(bf16_lo(w), bf16_hi(w));
}

// (mean, M2) of the 32 bf16 values of two 32-byte vectors in one pass, by
// sums shifted by one of the values, c: S1 = sum (x - c), S2 = sum (x - c)^2,
// mean = c + S1 / 32, M2 = S2 - S1^2 / 32 (the shifted-data form of Chan,
// Golub and LeVeque, 1983).  Since c is one of the 32 values, M2 >= (c -
// mean)^2, so the cancellation in S2 - S1^2 / 32 loses at most a factor 33 of
// relative precision (about 2e-6 in fp32), and x - c is exact for bf16
// values.  Paired fp32 arithmetic, two columns an instruction.
__device__ __forceinline__ void stats32(const V8 &a, const V8 &b, float &mean, float &m2) {
  const float c = bf16_lo(a.w[0]);
  const uint64_t nc = pack_f32x2(-c, -c);
  uint64_t s0 = 0, s1 = 0, q0 = 0, q1 = 0;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const uint64_t da = add_f32x2(unpack_pair(a.w[h]), nc);
    const uint64_t db = add_f32x2(unpack_pair(b.w[h]), nc);
    s0 = add_f32x2(s0, da);
    s1 = add_f32x2(s1, db);
    q0 = fma_f32x2(da, da, q0);
    q1 = fma_f32x2(db, db, q1);
  }
  const uint64_t sv = add_f32x2(s0, s1), qv = add_f32x2(q0, q1);
  const float S1 = f32x2_lo(sv) + f32x2_hi(sv), S2 = f32x2_lo(qv) + f32x2_hi(qv);
  mean = fmaf(S1, 1.0f / 32.0f, c);
  m2 = fmaxf(fmaf(-S1, S1 * (1.0f / 32.0f), S2), 0.0f);
}

// T threads per CTA (a power of two, 64 .. 512, or 96, 160, 192, 224), a
// cluster of C CTAs (1, 2, 4 or 8) per row: cols = C * T * 32.  R rows per
// step, A rows ahead.
// Launch bounds: the CTAs of up to 512 threads that one SM holds at 128
// registers a thread (two CTAs of 256 threads: 16 warps); a register more and
// only one CTA of 256 fits, which halves the bytes in flight (measured on
// GB300, [4096, 32768]: 120.8 us at 132 registers against 85-90 us at 128).
template <int T, int R, int A>  // A >= R: the rows a step reduces were issued a step earlier
__global__ void __launch_bounds__(T, T >= 512 ? 1 : 512 / T)
layernorm_cluster_full(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
                       const float *__restrict__ beta, uint16_t *__restrict__ y,
                       float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
                       int64_t cols, int64_t ldx, int64_t ldy, float eps, int *__restrict__ err) {
  static_assert(A >= R, "a step's rows must be issued during the step before");
  pdl_enter();
  constexpr int kSlotsR = full_slots(R, A), kAhead = A;
  extern __shared__ __align__(128) unsigned char smem[];  // [kSlotsR] row slices
  __shared__ __align__(8) uint64_t landed[kSlotsR];       // bulk-copy completion per slot
  __shared__ __align__(16) float4 slot[kClSlots][kFullMaxCluster];  // [step % 4][rank]
  __shared__ __align__(8) uint64_t pbar[kClSlots];
  constexpr int W = T / 32;
  __shared__ float2 red[2][R][W];  // per-warp (mean, M2), double-buffered by step
  __shared__ int timed_out;

  const uint32_t C = cluster_nctarank(), q = cluster_ctarank();
  const int64_t cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t S = cols / C;  // = T * 32
  const uint32_t slice = static_cast<uint32_t>(S) * 2;  // bytes of a row slice
  // Thread t owns the 16-byte chunks j = t + T c (c = 0..3) of its CTA's
  // slice, columns 8j .. 8j + 7: a warp's shared-memory reads and global
  // stores of one chunk are 512 contiguous bytes (no bank conflicts).
  const int64_t cbase = static_cast<int64_t>(q) * S + 8 * static_cast<int64_t>(tid);
  constexpr int64_t kChunkStride = 8 * T;  // columns between a thread's chunks
  const int64_t nr = cid < rows ? (rows - cid + ncl - 1) / ncl : 0;  // rows of this cluster
  const int64_t ns = (nr + R - 1) / R;                                // steps of R rows
  const uint32_t part_bytes = 16u * C;
  const float inv_n = __frcp_rn(static_cast<float>(cols));

  auto row_of = [&](int64_t k) { return cid + k * ncl; };
  auto slot_of = [&](int64_t k) { return smem + static_cast<size_t>(k % kSlotsR) * slice; };
  // this thread's 32 values of a staged row: chunks 0, 1 in one V8, 2, 3 in another
  auto read_row = [&](int64_t k, V8 &c0, V8 &c1) {
    const unsigned char *p = slot_of(k) + static_cast<size_t>(tid) * 16;
    const uint4 a = lds_u4(p), b = lds_u4(p + 16 * T), c = lds_u4(p + 32 * T),
                d = lds_u4(p + 48 * T);
    c0.w[0] = a.x; c0.w[1] = a.y; c0.w[2] = a.z; c0.w[3] = a.w;
    c0.w[4] = b.x; c0.w[5] = b.y; c0.w[6] = b.z; c0.w[7] = b.w;
    c1.w[0] = c.x; c1.w[1] = c.y; c1.w[2] = c.z; c1.w[3] = c.w;
    c1.w[4] = d.x; c1.w[5] = d.y; c1.w[6] = d.z; c1.w[7] = d.w;
  };
  const uint64_t policy = l2_evict_first_policy();
  int last_issued = -1;  // thread 0: the last row whose slice it requested
  auto issue = [&](int64_t k) {  // thread 0: this CTA's slice of row k, one bulk copy
    if (k < nr && !timed_out) {
      uint64_t *b = &landed[k % kSlotsR];
      mbar_arrive_expect_tx(b, slice);
      bulk_copy_g2s(slot_of(k), x + row_of(k) * ldx + static_cast<int64_t>(q) * S, slice, b,
                    policy);
      last_issued = static_cast<int>(k);
    }
  };
  auto wait_row = [&](int64_t k) {
    if (!timed_out &&
        !mbar_wait_bounded(&landed[k % kSlotsR], static_cast<uint32_t>((k / kSlotsR) & 1),
                           kWaitBudget)) {
      timed_out = 1;
      atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
    }
  };

  // The first rows are requested before anything else: the gamma/beta loads
  // and the cluster barrier below overlap their flight (loading gamma/beta
  // first held the first copies back, about 1 us of a 4 us start).
  if (tid == 0) {
    timed_out = 0;
    for (int i = 0; i < kSlotsR; ++i) mbar_init(&landed[i], 1);
    for (int i = 0; i < kClSlots; ++i) mbar_init(&pbar[i], 1);
    mbar_init_fence();
    for (int i = 0; i < kAhead; ++i) issue(i);
    for (int64_t st = 0; st < kClSlots && st < ns; ++st) mbar_arrive_expect_tx(&pbar[st], part_bytes);
  }
  uint64_t g2[kClCols / 2], b2[kClCols / 2];  // gamma/beta pairs of this thread's columns
#pragma unroll
  for (int h = 0; h < kClCols / 4; ++h) {  // chunk h / 2, columns 4 (h % 2) .. + 3
    const int64_t col = cbase + kChunkStride * (h >> 1) + 4 * (h & 1);
    const float4 gv = ld_keep_f4(gamma + col), bv = ld_keep_f4(beta + col);
    g2[2 * h] = pack_f32x2(gv.x, gv.y);
    g2[2 * h + 1] = pack_f32x2(gv.z, gv.w);
    b2[2 * h] = pack_f32x2(bv.x, bv.y);
    b2[2 * h + 1] = pack_f32x2(bv.z, bv.w);
  }
  __syncthreads();
  cluster_arrive();  // every CTA's barriers are armed before anyone sends
  cluster_wait();

  // Step s: reduce rows sR .. sR + R - 1 (this thread's 32 values of each) and
  // publish the CTA's R (mean, M2) pairs in one 16-byte message; then finalise
  // the rows of step s - 1, reading their values again from their slots.
  // Slots hold the previous step's rows, this step's and kAhead rows ahead;
  // after this step's barrier every thread has finished with the rows of step
  // s - 2, whose slots thread 0 then refills with the next rows.
  for (int64_t s = 0; s <= ns; ++s) {
    if (s < ns) {
      float mean[R], m2[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t k = s * R + r;
        mean[r] = m2[r] = 0.0f;
        if (k < nr) {
          wait_row(k);
          V8 c0, c1;
          read_row(k, c0, c1);
          stats32(c0, c1, mean[r], m2[r]);
        }
      }
      float half_n = 16.0f;  // half of each side's count
#pragma unroll
      for (int o = 16; o > 0; o >>= 1, half_n *= 2.0f)
#pragma unroll
        for (int r = 0; r < R; ++r)
          merge_equal(mean[r], m2[r], __shfl_xor_sync(0xffffffffu, mean[r], o),
                      __shfl_xor_sync(0xffffffffu, m2[r], o), half_n);
      if (lane == 0)
#pragma unroll
        for (int r = 0; r < R; ++r) red[s & 1][r][warp] = make_float2(mean[r], m2[r]);
      __syncthreads();
      if (tid == 0) {  // refill the slots of step s - 2 with the rows kAhead ahead
        fence_proxy_async_smem();
#pragma unroll
        for (int r = 0; r < R; ++r) issue(s * R + r + kAhead);
      }
      if (warp == 0) {  // the CTA's W warp pairs (1024 values each) on lanes 0..W-1
        float wm[R], w2[R];
        if constexpr ((W & (W - 1)) == 0) {  // equal counts at every level of the tree
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float2 t = red[s & 1][r][lane & (W - 1)];
            wm[r] = t.x;
            w2[r] = t.y;
          }
          float hn = 512.0f;
#pragma unroll
          for (int o = W / 2; o > 0; o >>= 1, hn *= 2.0f)
#pragma unroll
            for (int r = 0; r < R; ++r)
              merge_equal(wm[r], w2[r], __shfl_xor_sync(0xffffffffu, wm[r], o),
                          __shfl_xor_sync(0xffffffffu, w2[r], o), hn);
        } else {  // W = 3, 5, 6, 7: the warps' pairs folded in warp order, in every lane
          // (pair k joins the first k: weight 1 / (k + 1), correction
          // delta^2 * 1024 k / (k + 1), constants of the fold)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float2 t = red[s & 1][r][0];
            wm[r] = t.x;
            w2[r] = t.y;
          }
#pragma unroll
          for (int k = 1; k < W; ++k)
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float2 t = red[s & 1][r][k];
              const float delta = t.x - wm[r];
              wm[r] = fmaf(delta, 1.0f / static_cast<float>(k + 1), wm[r]);
              w2[r] = fmaf(delta * delta, 1024.0f * static_cast<float>(k) / static_cast<float>(k + 1),
                           w2[r] + t.y);
            }
        }
        if (lane < static_cast<int>(C)) {
          const int sl = static_cast<int>(s % kClSlots);
          st_async_f4(&slot[sl][q], &pbar[sl], static_cast<uint32_t>(lane),
                      make_float4(wm[0], w2[0], R > 1 ? wm[R - 1] : 0.0f,
                                  R > 1 ? w2[R - 1] : 0.0f));
        }
      }
    }
    if (s > 0) {  // finalise the rows of step s - 1
      const int64_t sp = s - 1;
      const int sl = static_cast<int>(sp % kClSlots);
      if (!timed_out &&
          !mbar_wait_bounded(&pbar[sl], static_cast<uint32_t>((sp / kClSlots) & 1), kWaitBudget)) {
        timed_out = 1;
        atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
      }
      // Re-arm slot sl for step sp + 4 after reading it (peers send it only
      // after this CTA publishes step sp + 2, which comes after this point).
      float4 u[kFullMaxCluster];
#pragma unroll
      for (int rk = 0; rk < kFullMaxCluster; ++rk)
        u[rk] = rk < static_cast<int>(C) ? slot[sl][rk] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (tid == 0 && sp + kClSlots < ns && !timed_out) mbar_arrive_expect_tx(&pbar[sl], part_bytes);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t k = sp * R + r;
        if (k >= nr) break;
        // the C ranks' pairs merged by a fixed tree over rank order (equal
        // counts at every level): the same bits in every CTA of the cluster
        float cm[kFullMaxCluster], c2[kFullMaxCluster];
#pragma unroll
        for (int rk = 0; rk < kFullMaxCluster; ++rk) {
          cm[rk] = r == 0 ? u[rk].x : u[rk].z;
          c2[rk] = r == 0 ? u[rk].y : u[rk].w;
        }
        float hs = 0.5f * static_cast<float>(S);
#pragma unroll
        for (int w = 1; w < kFullMaxCluster; w <<= 1, hs *= 2.0f)
#pragma unroll
          for (int rk = 0; rk + w < kFullMaxCluster; rk += 2 * w)
            if (rk + w < static_cast<int>(C)) merge_equal(cm[rk], c2[rk], cm[rk + w], c2[rk + w], hs);
        const float mean = cm[0], m2 = c2[0];
        const int64_t row = row_of(k);
        const float rstd = rsqrtf(fmaf(m2, inv_n, eps));
        if (q == 0 && tid == 0) {
          if (mean_out) mean_out[row] = mean;
          if (rstd_out) rstd_out[row] = rstd;
        }
        const uint64_t nm = pack_f32x2(-mean, -mean), r2 = pack_f32x2(rstd, rstd);
        const unsigned char *p = slot_of(k) + static_cast<size_t>(tid) * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // chunk c: 8 columns, pairs 4c .. 4c + 3
          const uint4 v = lds_u4(p + 16 * T * c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint64_t d = add_f32x2(unpack_pair(w[h]), nm);
            const uint64_t yv = fma_f32x2(mul_f32x2(d, r2), g2[4 * c + h], b2[4 * c + h]);
            o[h] = pack_bf16x2(f32x2_lo(yv), f32x2_hi(yv));
          }
          st_stream_u4(y + row * ldy + cbase + kChunkStride * c,
                       make_uint4(o[0], o[1], o[2], o[3]));
        }
      }
    }
  }
  // After a timeout no slot was refilled; a slot is refilled only after every
  // thread's wait on its previous row succeeded, so at most its latest copy
  // is in flight, and the last kSlotsR rows issued hold the latest copy of
  // every slot: wait for those (a completed phase returns at once).
  if (timed_out && tid == 0)
    for (int k = last_issued - kSlotsR + 1 < 0 ? 0 : last_issued - kSlotsR + 1; k <= last_issued;
         ++k)
      mbar_wait_bounded(&landed[k % kSlotsR], static_cast<uint32_t>((k / kSlotsR) & 1), kWaitBudget);
  // No CTA may leave while a peer can still write into its shared memory.
  cluster_arrive();
  cluster_wait();
}

}  // namespace

// Cluster size: the smallest C in {1, 2} with slices of at most 16384
// columns (32 columns per thread), and only when the slices keep at least
// half the 512 threads busy (a slice of 8192 columns or more: at 768 columns
// the kernel took 1649 us, 24 of 512 threads working, against 90 us for row
// groups; at 5120, 278 against 240 for the ring; at 12288, 149).
int cluster_size_for(int64_t cols) {
  for (int c = 1; c <= kClMaxCluster; c <<= 1)
    if (cols % (kClCols * c) == 0 && cols / c <= kClMaxSlice && cols / c >= kClMaxSlice / 2)
      return c;
  return 0;
}

size_t cluster_smem(int64_t, int) {
  return static_cast<size_t>(kClStages) * kClThreads * 64;  // the cp.async ring
}


namespace {

using LnKern = void (*)(const uint16_t *, const float *, const float *, uint16_t *, float *,
                        float *, int64_t, int64_t, int64_t, int64_t, float, int *);

// One rows-per-step / rows-ahead choice of the equal-count kernel, for each
// CTA size.
struct FullShape {
  const char *name;
  int slots;
  LnKern kern[4];  // T = 64, 128, 256, 512
};

#define FR_LNF(R, A)                                                                       \
  {layernorm_cluster_full<64, R, A>, layernorm_cluster_full<128, R, A>,                      \
   layernorm_cluster_full<256, R, A>, layernorm_cluster_full<512, R, A>}
// CTAs of 3, 5, 6 and 7 warps (rows of 3, 5, 6, 7, 10, 12, 14, 20, 24 or 28
// times 1024 columns), in the default shape only.
constexpr int kOddT[] = {96, 160, 192, 224};
const LnKern kFullOdd[] = {layernorm_cluster_full<96, 1, 2>, layernorm_cluster_full<160, 1, 2>,
                           layernorm_cluster_full<192, 1, 2>, layernorm_cluster_full<224, 1, 2>};
const FullShape kFullShapes[] = {{"r1a2", full_slots(1, 2), FR_LNF(1, 2)},
                                 {"r1a1", full_slots(1, 1), FR_LNF(1, 1)},
                                 {"r1a3", full_slots(1, 3), FR_LNF(1, 3)},
                                 {"r1a4", full_slots(1, 4), FR_LNF(1, 4)},
                                 {"r1a5", full_slots(1, 5), FR_LNF(1, 5)},
                                 {"r2a2", full_slots(2, 2), FR_LNF(2, 2)}};
#undef FR_LNF

// The equal-count kernel's shape for a row length: cols = C * T * 32 with
// C in 1, 2, 4, 8 and T a power of two in 64 .. 512 or one of kOddT.  Measured on GB300
// (256 MiB of bf16 rows, launches back to back): 8192 columns 84.2 us with
// one CTA of 256 threads, 86.8 with 2 of 128; 16384 84.1 with 2 of 256,
// 86.1 with 4 of 128, 88.3 with 1 of 512; 32768 86.3 with 4 of 256, 88.8
// with 2 of 512, 96.0 with 8 of 128; 65536 93.1 with 4 of 512, 95.7-99.4
// with 8 of 256.  FR_LAYERNORM_CTA=64|128|256|512 caps T.
bool full_shape(int64_t cols, int *T, int *C) {
  const char *e = getenv("FR_LAYERNORM_CTA");
  const int v = e != nullptr ? atoi(e) : 256;
  const int tmax = v == 64 || v == 128 || v == 512 ? v : 256;
  // Clusters of up to 4 CTAs first (8 cost 5-10 %: [2048, 65536] 96.9 us
  // with 8 CTAs of 256 threads, 93.0 with 4 of 512), then CTAs of at most
  // tmax threads (the largest such), then larger ones.
  constexpr int kTs[] = {512, 256, 224, 192, 160, 128, 96, 64};
  for (int cmax = 4; cmax <= kFullMaxCluster; cmax <<= 1)
    for (int pass = 0; pass < 2; ++pass)
      for (int c = 1; c <= cmax; c <<= 1)
        for (int t : kTs) {
          if ((pass == 0) != (t <= tmax)) continue;
          if (cols == static_cast<int64_t>(c) * t * kClCols) {
            *T = t;
            *C = c;
            return true;
          }
        }
  return false;
}

// The equal-count kernel of a shape for T threads.  The odd CTA sizes exist
// in the default shape (r1a2) only, which a pinned shape falls back to there.
LnKern full_kernel(const FullShape &sh, int T) {
  switch (T) {
    case 64: return sh.kern[0];
    case 128: return sh.kern[1];
    case 256: return sh.kern[2];
    case 512: return sh.kern[3];
  }
  for (size_t i = 0; i < sizeof kOddT / sizeof kOddT[0]; ++i)
    if (kOddT[i] == T) return kFullOdd[i];
  return nullptr;
}

}  // namespace

bool layernorm_cluster_ok(int64_t cols, bool aligned) {
  int t = 0, c = 0;
  return aligned && (cluster_size_for(cols) > 0 || full_shape(cols, &t, &c));
}

int layernorm_cluster_full_threads(int64_t cols, bool aligned) {
  int t = 0, c = 0;
  return aligned && full_shape(cols, &t, &c) ? t : 0;
}

cudaError_t launch_layernorm_cluster(const uint16_t *x, const float *gamma, const float *beta,
                                     uint16_t *y, float *mean, float *rstd, int64_t rows,
                                     int64_t cols, int64_t ldx, int64_t ldy, float eps,
                                     cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  // Rows of C * T * 32 columns: the equal-count kernel (every thread 32
  // columns), R rows per step and A rows ahead (FR_LAYERNORM_CLUSTER=classic|
  // r1a1|...|r2a2 pins one; default r1a2).  Measured on GB300, bf16
  // [4096, 32768]: r1a2 91.4 us, r1a3 93.2, r2a2 95.8, r1a5 97.3, r1a4 98.2,
  // r1a1 113.9, classic 132.3.  Other rows: the general cluster kernel.
  const char *pin = getenv("FR_LAYERNORM_CLUSTER");
  auto pinned = [&](const char *v) { return pin != nullptr && strcmp(pin, v) == 0; };
  int T = kClThreads, C = 0;
  const bool full = !pinned("classic") && full_shape(cols, &T, &C);
  if (!full) {
    T = kClThreads;
    C = cluster_size_for(cols);
  }
  if (C == 0) return cudaErrorInvalidValue;
  const FullShape *sh = &kFullShapes[0];
  for (const FullShape &c : kFullShapes)
    if (pinned(c.name)) sh = &c;
  LnKern kern = full ? full_kernel(*sh, T) : layernorm_cluster;
  if (kern == nullptr) return cudaErrorInvalidValue;
  if (full && (T & (T - 1)) != 0) sh = &kFullShapes[0];
  const size_t smem = !full ? cluster_smem(cols, C)
                            : static_cast<size_t>(sh->slots) * static_cast<size_t>(cols / C) * 2;
  e = set_smem_limit(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  if (C > 8) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(static_cast<unsigned>(T));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  int clusters = 0;
  e = resident_clusters(&clusters, reinterpret_cast<const void *>(kern), cfg, cfg.attrs[0].val.clusterDim.x);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  int64_t ncl = clusters;  // persistent: every cluster that can be resident
  if (ncl > rows) ncl = rows;
  // Both kernels: a cluster launch without the programmatic overlap.  The
  // equal-count kernel is persistent (every resident cluster, one wave), and
  // as a programmatic dependent of its own previous call each launch's
  // clusters took the slots the previous call's clusters left, in the order
  // they left: measured on GB300, bf16 [4096, 32768] back to back, blocks of
  // 20 calls then fell into modes 2.65 us a call apart (86.2, 88.8, 91.4,
  // 94.1 us; block means over 9 blocks 88.2-89.8, the mode kept for a whole
  // block), with the dependents signalled at the kernel's start or at its
  // end alike; as ordinary launches every block took 88.4-89.2 (means
  // 88.7-88.9).
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * C));
  return cudaLaunchKernelEx(&cfg, kern, x, gamma, beta, y, mean, rstd, rows, cols, ldx, ldy, eps,
                            err);
}

size_t layernorm_ring_smem(int64_t cols, int nbuf) {
  return static_cast<size_t>(nbuf) * static_cast<size_t>(cols) * 2;
}

bool layernorm_ring_ok(int64_t cols, bool vec, int max_smem_optin) {
  return vec && cols % 16 == 0 && cols / 16 <= static_cast<int64_t>(kRingThreads) * kRingPieces &&
         layernorm_ring_smem(cols, kRingBufs) + 1024 <= static_cast<size_t>(max_smem_optin);
}

cudaError_t launch_layernorm_ring(const uint16_t *x, const float *gamma, const float *beta,
                                  uint16_t *y, float *mean, float *rstd, int64_t rows,
                                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int sm_count,
                                  int, cudaStream_t s) {
  const size_t smem = layernorm_ring_smem(cols, kRingBufs);
  // R rows per gamma/beta pass; FR_LAYERNORM_ROWS=1|2 pins it (default 2;
  // three rows need more than the 128 registers a thread can have).
  int R = 2;
  if (const char *e = getenv("FR_LAYERNORM_ROWS")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 2) R = v;
  }
  // FR_LAYERNORM_STAGE=bulk stages rows with one bulk copy each (default:
  // per-thread cp.async).
  const char *st = getenv("FR_LAYERNORM_STAGE");
  const bool bulk = st != nullptr && strcmp(st, "bulk") == 0;
  const void *kern =
      R == 1 ? (bulk ? reinterpret_cast<const void *>(&layernorm_ring<1, true>)
                     : reinterpret_cast<const void *>(&layernorm_ring<1, false>))
             : (bulk ? reinterpret_cast<const void *>(&layernorm_ring<2, true>)
                     : reinterpret_cast<const void *>(&layernorm_ring<2, false>));
  int *err = nullptr;
  if (cudaError_t ee = device_error_word(&err); ee != cudaSuccess) return ee;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern), kRingThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = static_cast<int64_t>(sm_count) * per_sm;
  if (grid > rows) grid = rows;
  void *args[] = {&x, &gamma, &beta, &y, &mean, &rstd, &rows, &cols, &ldx, &ldy, &eps, &err};
  return cudaLaunchKernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kRingThreads), args, smem,
                          s);
}

// Row groups: the fewest warps per row (1, 2, 4 or 8) that hold it in at most
// NMAX chunks of 8 columns a thread; NC rounded up to 2, 4, 6 or 8.
// FR_LAYERNORM_ROWS_NC=4|8 sets NMAX (default 8).
namespace {
bool rows_shape(int64_t cols, int *WG, int *NC) {
  const int64_t nch = cols / 8;
  const char *e = getenv("FR_LAYERNORM_ROWS_NC");
  const int nmax = e != nullptr && atoi(e) == 4 ? 4 : 8;
  for (int wg = 1; wg <= 8; wg <<= 1) {
    const int64_t need = (nch + 32 * wg - 1) / (32 * wg);
    if (need <= nmax) {
      *WG = wg;
      *NC = need <= 2 ? 2 : need <= 4 ? 4 : need <= 6 ? 6 : 8;
      return true;
    }
  }
  return false;
}
}  // namespace

using RowsKern = void (*)(const uint16_t *, const float *, const float *, uint16_t *, float *,
                         float *, int64_t, int64_t, int64_t, int64_t, float, float, float, float);

// The row-group kernel for WG warps a row and NC chunks a thread: the next
// row prefetched into registers with 2 or 4 chunks, and with 6 or 8 when pf8
// (8 warps a row); otherwise more rows in flight instead.
template <int W, bool P, bool E>
RowsKern rows_nc(int NC, bool pf8) {
  if constexpr (W == 1)
    if (NC == 2) return layernorm_rows<1, 2, true, P, E>;
  if (NC == 4) return layernorm_rows<W, 4, true, P, E>;
  if constexpr (W == 8)
    if (pf8) return NC == 6 ? layernorm_rows<8, 6, true, P, E> : layernorm_rows<8, 8, true, P, E>;
  return NC == 6 ? layernorm_rows<W, 6, false, P, E> : layernorm_rows<W, 8, false, P, E>;
}

template <bool P, bool E>
RowsKern rows_kernel(int WG, int NC, bool pf8) {
  switch (WG) {
    case 1: return rows_nc<1, P, E>(NC, pf8);
    case 2: return rows_nc<2, P, E>(NC, pf8);
    case 4: return rows_nc<4, P, E>(NC, pf8);
    default: return rows_nc<8, P, E>(NC, pf8);
  }
}

bool layernorm_rows_ok(int64_t cols, bool aligned16, int max_smem_optin) {
  int wg = 0, nc = 0;
  return aligned16 && cols % 8 == 0 && rows_shape(cols, &wg, &nc) &&
         static_cast<int64_t>(cols) * 8 + 1024 <= max_smem_optin;
}

cudaError_t launch_layernorm_rows(const uint16_t *x, const float *gamma, const float *beta,
                                  uint16_t *y, float *mean, float *rstd, int64_t rows,
                                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int sm_count,
                                  cudaStream_t s) {
  int WG = 0, NC = 0;
  if (!rows_shape(cols, &WG, &NC)) return cudaErrorInvalidValue;
  // gamma/beta layout, measured on GB300 (256 MiB of x, us per call, chunk
  // by chunk / planes): 768 columns 90.8 / 89.5, 1024 85.5 / 96.4, 1536
  // 84.2 / 96.0, 2560 92.4 / 85.0, 3072 88.9 / 93.7, 5120 100.9 / 88.6, 6144
  // 106.3 / 99.6, 12288 134.0 / 127.4.  The planes, though they halve the
  // shared-memory wavefronts (768: 20.6 M to 12.0 M), were slower where one
  // or two warps hold a row and every thread holds all NC chunks; the rule
  // below picks the faster layout at all eight sizes.
  // FR_LAYERNORM_ROWS_GB=planar|chunk pins one where every thread holds the
  // same number of chunks; rows with unequal counts always take the planes.
  const int64_t nch = cols / 8;
  const bool full_chunks = nch % (32 * static_cast<int64_t>(WG)) == 0 &&
                           nch / (32 * static_cast<int64_t>(WG)) == NC;
  bool pl = WG >= 4 || !full_chunks;
  if (const char *gl = getenv("FR_LAYERNORM_ROWS_GB"); gl != nullptr)
    pl = strcmp(gl, "planar") == 0;
  // Rows past 8192 columns (8 warps a row, 64 KiB and more of gamma/beta: at
  // most three CTAs an SM) prefetch the next row with 6 or 8 chunks a thread
  // too: fewer rows in flight otherwise.
  const bool pf8 = cols > 8192;
  const bool eq = nch % (32 * static_cast<int64_t>(WG)) == 0;
  RowsKern kern = !eq ? rows_kernel<true, false>(WG, NC, pf8)
               : pl ? rows_kernel<true, true>(WG, NC, pf8) : rows_kernel<false, true>(WG, NC, pf8);
  const float inv_n = 1.0f / static_cast<float>(cols);
  const float n_t = eq ? static_cast<float>(8 * (nch / (32 * WG))) : 1.0f;  // values a thread
  const float inv_nt = 1.0f / n_t, half_nt = 0.5f * n_t;
  const size_t smem = static_cast<size_t>(cols) * 8;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern), kRgThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int groups = kRgThreads / 32 / WG;
  int64_t grid = static_cast<int64_t>(sm_count) * per_sm;
  const int64_t need = (rows + groups - 1) / groups;
  if (grid > need) grid = need;
  return launch_k(kern, dim3(static_cast<unsigned>(grid)), dim3(kRgThreads), smem, s, 0, x, gamma,
                  beta, y, mean, rstd, rows, cols, ldx, ldy, eps, inv_n, inv_nt, half_nt);
}

bool layernorm_persistent_ok(int64_t cols, bool vec) {
  return vec && cols % 16 == 0 && cols / 16 <= kPersistMaxThreads * 4;
}

cudaError_t launch_layernorm_persistent(const uint16_t *x, const float *gamma,
                                        const float *beta, uint16_t *y, float *mean,
                                        float *rstd, int64_t rows, int64_t cols, int64_t ldx,
                                        int64_t ldy, float eps, cudaStream_t s) {
  const int64_t nvec = cols / 16;
  // Threads: the smallest warp multiple that holds the row in at most 4
  // vectors per thread, at least 128.
  int64_t t = (nvec + 3) / 4;
  t = (t + 31) / 32 * 32;
  if (t < 128) t = 128;
  if (t > kPersistMaxThreads) return cudaErrorInvalidValue;
  const int64_t nv = (nvec + t - 1) / t;
  const unsigned grid = static_cast<unsigned>(rows);
  const unsigned block = static_cast<unsigned>(t);
  switch (nv) {
    case 1: layernorm_persistent<1><<<grid, block, 0, s>>>(x, gamma, beta, y, mean, rstd, cols, ldx, ldy, eps); break;
    case 2: layernorm_persistent<2><<<grid, block, 0, s>>>(x, gamma, beta, y, mean, rstd, cols, ldx, ldy, eps); break;
    case 3:
    case 4: layernorm_persistent<4><<<grid, block, 0, s>>>(x, gamma, beta, y, mean, rstd, cols, ldx, ldy, eps); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_layernorm_looped(const uint16_t *x, const float *gamma, const float *beta,
                                    uint16_t *y, float *mean, float *rstd, int64_t rows,
                                    int64_t cols, int64_t ldx, int64_t ldy, float eps, bool,
                                    int sm_count, int, cudaStream_t s) {
  int64_t grid = static_cast<int64_t>(sm_count) * 2;
  if (grid > rows) grid = rows;
  layernorm_looped_scalar<<<static_cast<unsigned>(grid), kLoopThreads, 0, s>>>(
      x, gamma, beta, y, mean, rstd, rows, cols, ldx, ldy, eps);
  return cudaGetLastError();
}

}  // namespace fr
