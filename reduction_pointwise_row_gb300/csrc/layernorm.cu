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
// persistent  one CTA per row, the row held in registers as packed bf16
//             (x read once from HBM, y written once).
// looped      one CTA per row, grid-stride over rows: pass 1 streams the row
//             in chunks merging Welford triples, pass 2 streams it again
//             (from L2) to write y.  Any alignment (scalar lane-strided).
#include <cstdlib>

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

// Persistent form.  Requires 32-byte aligned x/y rows, gamma, beta and
// cols % 16 == 0 (checked by the host); NV vectors of 16 per thread.
constexpr int kPersistMaxThreads = 512;

template <int NV>
__global__ void __launch_bounds__(kPersistMaxThreads, 2)
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

template <int R>
__global__ void __launch_bounds__(kRingThreads, 1)
layernorm_ring(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
               const float *__restrict__ beta, uint16_t *__restrict__ y,
               float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
               int64_t cols, int64_t ldx, int64_t ldy, float eps) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Welford red[R][32];
  const int tid = threadIdx.x;
  const int npieces = static_cast<int>(cols >> 4);  // cols % 16 == 0
  const size_t buf_bytes = static_cast<size_t>(npieces) * 32;
  const int64_t G = gridDim.x;
  // rows of this CTA: blockIdx.x + k * G for k < nk
  const int64_t nk = blockIdx.x < rows ? (rows - blockIdx.x + G - 1) / G : 0;

  auto stage = [&](int64_t k) {  // this thread's pieces of row k into buffer k % kRingBufs
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

  for (int b = 0; b < kRingBufs; ++b) stage(b);
  int64_t next = kRingBufs;  // next row index to stage
  for (int64_t k0 = 0; k0 < nk; k0 += R) {
    V8 v[R][kRingPieces];
    Welford w[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      // Groups committed so far: rows 0 .. next - 1 = k0 + r + kRingBufs - 1.
      // Row k0 + r has landed once at most the kRingBufs - 1 newer ones pend.
      cp_async_wait<kRingBufs - 1>();
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
}

constexpr long long kWaitBudget = 1LL << 31;  // SM clocks (about one second) per wait

// ---- cluster form: gamma/beta resident in shared memory -----------------------
// A cluster of C CTAs (C = 1 or 2) splits every row into C column slices of
// S = cols / C <= 16384.  Each CTA keeps the gamma/beta of its slice in shared
// memory for the whole kernel (S * 8 <= 128 KiB) and streams x through a ring
// of kClBufs slice buffers filled with per-thread cp.async copies, kClBufs rows
// (a wave) at a time: pass 1 lifts the wave's x into registers (thread t owns
// the 16 columns 16t .. 16t + 15 of the slice) and refills the ring at once;
// one CTA merge reduces the wave's Welford triples; warp 0 pushes them into
// every CTA of the cluster (st.async, counted on the receiver's mbarrier); each
// CTA merges the C triples of a row in rank order (the same bits everywhere)
// and normalises the wave from registers, reading each gamma/beta value from
// shared memory once per wave.  HBM sees x once and y once; gamma/beta are
// read from HBM once per CTA.
constexpr int kClThreads = 1024;
constexpr int kClBufs = 3;        // rows per wave = slice buffers in the ring
constexpr int kClSlots = 4;       // published triples: wave w + 4 is written
                                  // only after this CTA published wave w + 1
constexpr int kClMaxCluster = 2;
constexpr int64_t kClMaxSlice = 16 * kClThreads;  // 16384 columns

__global__ void __launch_bounds__(kClThreads, 1)
layernorm_cluster(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
                  const float *__restrict__ beta, uint16_t *__restrict__ y,
                  float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(16) float4 slot[kClSlots][kClBufs][kClMaxCluster];  // [wave%4][row][rank]
  __shared__ __align__(8) uint64_t pbar[kClSlots];
  __shared__ Welford red[kClBufs][32];
  __shared__ int timed_out;

  const uint32_t C = cluster_nctarank(), q = cluster_ctarank();
  const int64_t cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t S = cols / C;
  const int npieces = static_cast<int>(S >> 4);        // 16 columns per piece, <= 1024
  const bool own = tid < npieces;
  const int64_t c0 = static_cast<int64_t>(q) * S;       // first column of the slice
  const int64_t col0 = c0 + 16 * static_cast<int64_t>(tid);
  float *sg = reinterpret_cast<float *>(smem);          // gamma[S], beta[S]
  float *sb = sg + S;
  unsigned char *ring = smem + static_cast<size_t>(S) * 8;
  const size_t buf_bytes = static_cast<size_t>(S) * 2;
  const int64_t nr = cid < rows ? (rows - cid + ncl - 1) / ncl : 0;  // rows of this cluster
  const int64_t nwaves = (nr + kClBufs - 1) / kClBufs;
  const uint32_t part_bytes = 16u * kClBufs * C;

  // gamma/beta of the slice into shared memory (once)
  for (int64_t i = tid; i < S / 4; i += kClThreads) {
    reinterpret_cast<float4 *>(sg)[i] = ld_keep_f4(gamma + c0 + 4 * i);
    reinterpret_cast<float4 *>(sb)[i] = ld_keep_f4(beta + c0 + 4 * i);
  }
  auto stage = [&](int64_t k) {  // row k of this cluster into buffer k % kClBufs
    if (k < nr && own) {
      const unsigned char *src =
          reinterpret_cast<const unsigned char *>(x + (cid + k * ncl) * ldx + col0);
      unsigned char *dst = ring + static_cast<size_t>(k % kClBufs) * buf_bytes + 32 * tid;
      cp_async_16(dst, src);
      cp_async_16(dst + 16, src + 16);
    }
    cp_async_commit();
  };
  if (tid == 0) {
    timed_out = 0;
    for (int i = 0; i < kClSlots; ++i) mbar_init(&pbar[i], 1);
    mbar_init_fence();
    for (int64_t w = 0; w < kClSlots && w < nwaves; ++w) mbar_arrive_expect_tx(&pbar[w], part_bytes);
  }
  for (int b = 0; b < kClBufs; ++b) stage(b);
  // gamma/beta and the barriers are ready in every CTA before anyone sends
  __syncthreads();
  cluster_arrive();
  cluster_wait();

  int64_t next = kClBufs;
  for (int64_t wv = 0; wv < nwaves; ++wv) {
    const int64_t k0 = wv * kClBufs;
    V8 v[kClBufs];
    Welford w[kClBufs];
#pragma unroll
    for (int r = 0; r < kClBufs; ++r) {
      cp_async_wait<kClBufs - 1>();  // row k0 + r landed (the newer rows may pend)
      w[r] = Welford{0.0f, 0.0f, 0.0f};
      if (own && k0 + r < nr) {
        v[r] = lds_v8(ring + static_cast<size_t>((k0 + r) % kClBufs) * buf_bytes + 32 * tid);
        w[r] = welford16(v[r]);
      }
      stage(next++);  // the row is in registers: refill its buffer
    }
    block_welford_n<kClBufs>(w, red);  // w[r] = this CTA's triple of row k0 + r
    const int sl = static_cast<int>(wv % kClSlots);
    if (tid < kClBufs * static_cast<int>(C)) {  // lanes of warp 0: (row, destination rank)
      const int r = tid / static_cast<int>(C), k = tid % static_cast<int>(C);
      Welford m = w[0];
      if (r == 1) m = w[1];
      if (r == 2) m = w[2];
      st_async_f4(&slot[sl][r][q], &pbar[sl], static_cast<uint32_t>(k),
                  make_float4(m.n, m.mean, m.m2, 0.0f));
    }
    if (!timed_out &&
        !mbar_wait_bounded(&pbar[sl], static_cast<uint32_t>((wv / kClSlots) & 1), 1LL << 31)) {
      timed_out = 1;
      atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
    }
    float mean[kClBufs], rstd[kClBufs];
#pragma unroll
    for (int r = 0; r < kClBufs; ++r) {
      Welford t{0.0f, 0.0f, 0.0f};
      for (uint32_t k = 0; k < C; ++k) {  // rank order: identical in every CTA
        const float4 u = slot[sl][r][k];
        t = chan_merge(t, Welford{u.x, u.y, u.z});
      }
      mean[r] = t.mean;
      rstd[r] = rsqrtf(fmaf(t.m2, __frcp_rn(t.n), eps));
      const int64_t row = cid + (k0 + r) * ncl;
      if (q == 0 && tid == 0 && k0 + r < nr) {
        if (mean_out) mean_out[row] = mean[r];
        if (rstd_out) rstd_out[row] = rstd[r];
      }
    }
    // Re-arm the slot for wave wv + 4: peers write it only after this CTA
    // publishes wave wv + 1, which every thread reaches after this point.
    if (tid == 0 && wv + kClSlots < nwaves) mbar_arrive_expect_tx(&pbar[sl], part_bytes);
    if (own) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {  // 4 columns of gamma/beta at a time, shared by the wave
        const float4 g = *reinterpret_cast<const float4 *>(sg + 16 * tid + 4 * h);
        const float4 bb = *reinterpret_cast<const float4 *>(sb + 16 * tid + 4 * h);
#pragma unroll
        for (int r = 0; r < kClBufs; ++r) {
          const uint32_t w0 = v[r].w[2 * h], w1 = v[r].w[2 * h + 1];
          v[r].w[2 * h] = pack_bf16x2(fmaf((bf16_lo(w0) - mean[r]) * rstd[r], g.x, bb.x),
                                      fmaf((bf16_hi(w0) - mean[r]) * rstd[r], g.y, bb.y));
          v[r].w[2 * h + 1] = pack_bf16x2(fmaf((bf16_lo(w1) - mean[r]) * rstd[r], g.z, bb.z),
                                          fmaf((bf16_hi(w1) - mean[r]) * rstd[r], g.w, bb.w));
        }
      }
#pragma unroll
      for (int r = 0; r < kClBufs; ++r)
        if (k0 + r < nr) st_stream_v8(y + (cid + (k0 + r) * ncl) * ldy + col0, v[r]);
    }
  }
  cp_async_wait<0>();
  // No CTA may leave while a peer can still write into its shared memory.
  cluster_arrive();
  cluster_wait();
}

}  // namespace

// Cluster size: 1 when gamma/beta of the whole row fit one CTA, else 2.
int cluster_size_for(int64_t cols) {
  for (int c = 1; c <= kClMaxCluster; c <<= 1)
    if (cols % (16 * c) == 0 && cols / c <= kClMaxSlice) return c;
  return 0;
}

size_t cluster_smem(int64_t cols, int c) {
  const int64_t S = cols / c;
  return static_cast<size_t>(S) * 8 + static_cast<size_t>(kClBufs) * S * 2;
}

bool layernorm_cluster_ok(int64_t cols, bool aligned) {
  const int c = cluster_size_for(cols);
  return aligned && c > 0;
}

cudaError_t launch_layernorm_cluster(const uint16_t *x, const float *gamma, const float *beta,
                                     uint16_t *y, float *mean, float *rstd, int64_t rows,
                                     int64_t cols, int64_t ldx, int64_t ldy, float eps,
                                     cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const int C = cluster_size_for(cols);
  if (C == 0) return cudaErrorInvalidValue;
  const size_t smem = cluster_smem(cols, C);
  e = cudaFuncSetAttribute(layernorm_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, layernorm_cluster, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  int64_t ncl = clusters;  // persistent: every cluster that can be resident
  if (ncl > rows) ncl = rows;
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * C));
  return cudaLaunchKernelEx(&cfg, layernorm_cluster, x, gamma, beta, y, mean, rstd, rows, cols,
                            ldx, ldy, eps, err);
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
  const void *kern = R == 1 ? reinterpret_cast<const void *>(&layernorm_ring<1>)
                            : reinterpret_cast<const void *>(&layernorm_ring<2>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRingThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = static_cast<int64_t>(sm_count) * per_sm;
  if (grid > rows) grid = rows;
  void *args[] = {&x, &gamma, &beta, &y, &mean, &rstd, &rows, &cols, &ldx, &ldy, &eps};
  return cudaLaunchKernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kRingThreads), args, smem,
                          s);
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
