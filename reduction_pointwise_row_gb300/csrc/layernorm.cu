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
#include "common.cuh"
#include "launch.h"

namespace fr {
namespace {

struct Welford {
  float n, mean, m2;
};

__device__ __forceinline__ Welford chan_merge(Welford a, Welford b) {
  const float n = a.n + b.n;
  if (n == 0.0f) return Welford{0.0f, 0.0f, 0.0f};
  const float delta = b.mean - a.mean;
  const float fb = b.n * __frcp_rn(n);
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

// ---- looped form with bulk-copy staging ------------------------------------
// A persistent CTA per SM owns rows blockIdx.x + k * gridDim.x and keeps NB
// row buffers in shared memory.  Row k is copied into buffer k % NB as
// kRingChunk-byte bulk copies, each completing on its own mbarrier; pass 1
// merges Welford triples of each chunk as it lands, pass 2 normalises from
// shared memory and streams y out, then buffer k % NB is refilled with row
// k + NB.  So NB - 1 rows are always in flight while one row is computed.
constexpr int kRingThreads = 1024;
constexpr int kRingChunk = 16384;     // bytes per bulk copy
constexpr int kRingMaxChunks = 13;    // rows of up to 208 KiB (106496 bf16)
constexpr int kRingMaxBuffers = 4;
constexpr int kRingHeader = 512;      // mbarriers (NB x chunks), then the buffers
constexpr long long kWaitBudget = 1LL << 31;  // SM clocks (about one second)

__global__ void __launch_bounds__(kRingThreads, 1)
layernorm_ring(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
               const float *__restrict__ beta, uint16_t *__restrict__ y,
               float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
               int64_t cols, int64_t ldx, int64_t ldy, float eps, int nbuf,
               int *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [nbuf][nch]
  __shared__ Welford red[32];
  __shared__ int timed_out;
  const int tid = threadIdx.x;
  const int64_t row_bytes = cols * 2;
  const size_t buf_bytes = static_cast<size_t>((row_bytes + 127) / 128 * 128);
  const int nch = static_cast<int>((row_bytes + kRingChunk - 1) / kRingChunk);
  const int npieces = static_cast<int>(cols >> 4);  // 32-byte pieces (cols % 16 == 0)
  constexpr int kPiecesPerChunk = kRingChunk / 32;
  const uint64_t policy = l2_evict_first_policy();
  auto buffer = [&](int b) { return smem + kRingHeader + static_cast<size_t>(b) * buf_bytes; };

  auto issue = [&](int64_t row, int b) {  // thread 0 only
    const unsigned char *src = reinterpret_cast<const unsigned char *>(x + row * ldx);
    unsigned char *dst = buffer(b);
    for (int c = 0; c < nch; ++c) {
      const int64_t off = static_cast<int64_t>(c) * kRingChunk;
      const uint32_t bytes =
          static_cast<uint32_t>(row_bytes - off < kRingChunk ? row_bytes - off : kRingChunk);
      mbar_arrive_expect_tx(&full[b * nch + c], bytes);
      bulk_copy_g2s(dst + off, src + off, bytes, &full[b * nch + c], policy);
    }
  };

  if (tid == 0) {
    timed_out = 0;
    for (int i = 0; i < nbuf * nch; ++i) mbar_init(&full[i], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (int b = 0; b < nbuf; ++b) {
      const int64_t r = blockIdx.x + static_cast<int64_t>(b) * gridDim.x;
      if (r < rows) issue(r, b);
    }
  int64_t k = 0;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++k) {
    const int b = static_cast<int>(k % nbuf);
    const uint32_t parity = static_cast<uint32_t>((k / nbuf) & 1);
    const unsigned char *buf = buffer(b);
    // pass 1: Welford over 16-element pieces, chunk by chunk as copies land
    Welford w{0.0f, 0.0f, 0.0f};
    for (int c = 0; c < nch; ++c) {
      if (!timed_out && !mbar_wait_bounded(&full[b * nch + c], parity, kWaitBudget)) {
        timed_out = 1;  // benign race: every writer stores 1
        atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
      }
      const int p_end = (c + 1) * kPiecesPerChunk < npieces ? (c + 1) * kPiecesPerChunk : npieces;
      for (int p = c * kPiecesPerChunk + tid; p < p_end; p += kRingThreads)
        w = chan_merge(w, welford16(lds_v8(buf + static_cast<size_t>(p) * 32)));
    }
    const Welford r = block_welford(w, red);
    const float mean = r.mean;
    const float rstd = rsqrtf(fmaf(r.m2, __frcp_rn(r.n), eps));
    if (tid == 0) {
      if (mean_out) mean_out[row] = mean;
      if (rstd_out) rstd_out[row] = rstd;
    }
    // pass 2: y = (x - mean) * rstd * gamma + beta from the staged row
    uint16_t *py = y + row * ldy;
    for (int p = tid; p < npieces; p += kRingThreads) {
      V8 v = lds_v8(buf + static_cast<size_t>(p) * 32);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float4 g = ld_keep_f4(gamma + p * 16 + 4 * h);
        const float4 bb = ld_keep_f4(beta + p * 16 + 4 * h);
        const uint32_t w0 = v.w[2 * h], w1 = v.w[2 * h + 1];
        v.w[2 * h] = pack_bf16x2(fmaf((bf16_lo(w0) - mean) * rstd, g.x, bb.x),
                                 fmaf((bf16_hi(w0) - mean) * rstd, g.y, bb.y));
        v.w[2 * h + 1] = pack_bf16x2(fmaf((bf16_lo(w1) - mean) * rstd, g.z, bb.z),
                                     fmaf((bf16_hi(w1) - mean) * rstd, g.w, bb.w));
      }
      st_stream_v8(py + static_cast<int64_t>(p) * 16, v);
    }
    __syncthreads();  // the whole CTA is done reading buffer b
    if (timed_out) {
      // Give every copy still in flight a last bounded wait, then stop.
      if (tid == 0)
        for (int j = 0; j < nbuf; ++j) {
          const int64_t kj = k + j;
          const int64_t rj = blockIdx.x + kj * gridDim.x;
          if (rj >= rows) break;
          const int bj = static_cast<int>(kj % nbuf);
          const uint32_t pj = static_cast<uint32_t>((kj / nbuf) & 1);
          for (int c = 0; c < nch; ++c) mbar_wait_bounded(&full[bj * nch + c], pj, kWaitBudget);
        }
      return;
    }
    const int64_t next = row + static_cast<int64_t>(nbuf) * gridDim.x;
    if (tid == 0 && next < rows) {
      fence_proxy_async_smem();
      issue(next, b);
    }
  }
}

// ---- cluster form: row slices across CTAs, gamma/beta in registers ---------
// A cluster of C CTAs splits every row into C column slices of S = cols / C;
// thread t of CTA rank q owns columns q*S + 8t .. q*S + 8t + 7 for the whole
// kernel, so its 8 gamma and 8 beta values are loaded once into registers and
// the only per-row traffic is x in and y out.  Each CTA streams its slices of
// kClRows rows at a time through a kClStages-deep ring of bulk copies.  Per
// row group: Welford triples of 8 elements per thread -> warp -> CTA; warp 0
// then pushes the CTA's triple of each row into every CTA of the cluster
// (st.async into the peer's shared memory, counted on the peer's mbarrier).
// Each CTA waits on its own barrier, merges the C triples in rank order (the
// same bits in every CTA) and normalises the x it still holds in registers.
// The merge of group g - 1 follows the publication of group g, so the
// exchange latency overlaps the next group's work.
constexpr int kClThreads = 512;
constexpr int kClRows = 2;     // rows per group
constexpr int kClStages = 4;   // groups in the bulk-copy ring
constexpr int kClSlots = 4;    // partial slots: a peer can write group g + 4 only
                               // after this CTA published g + 2, i.e. after it
                               // finished reading group g
constexpr int kClMaxCluster = 8;

__device__ __forceinline__ Welford welford8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) s += bf16_lo(w[j]) + bf16_hi(w[j]);
  const float mean = s * 0.125f;
  float q = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = bf16_lo(w[j]) - mean, b = bf16_hi(w[j]) - mean;
    q = fmaf(a, a, q);
    q = fmaf(b, b, q);
  }
  return Welford{8.0f, mean, q};
}

__global__ void __launch_bounds__(kClThreads, 2)
layernorm_cluster(const uint16_t *__restrict__ x, const float *__restrict__ gamma,
                  const float *__restrict__ beta, uint16_t *__restrict__ y,
                  float *__restrict__ mean_out, float *__restrict__ rstd_out, int64_t rows,
                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [kClStages] bulk-copy barriers
  uint64_t *pbar = full + kClStages;                    // [kClSlots] partial barriers
  unsigned char *stages = smem + 128;
  // slot[s][j][k]: rank k's triple of row j of the group using slot s
  __shared__ __align__(16) float4 slot[kClSlots][kClRows][kClMaxCluster];
  __shared__ Welford red[2][kClRows][kClThreads / 32];
  __shared__ int timed_out;

  const uint32_t C = cluster_nctarank(), q = cluster_ctarank();
  const int64_t cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t S = cols / C;  // columns of this CTA's slice
  const uint32_t slice_bytes = static_cast<uint32_t>(S * 2);
  const bool own = 8 * static_cast<int64_t>(tid) < S;
  const int64_t col0 = static_cast<int64_t>(q) * S + 8 * tid;
  const int64_t nrows_c = cid < rows ? (rows - cid + ncl - 1) / ncl : 0;
  const int64_t ngroups = (nrows_c + kClRows - 1) / kClRows;
  const uint32_t part_bytes = 16u * kClRows * C;  // triples arriving per group
  const uint64_t policy = l2_evict_first_policy();

  float g8[8], b8[8];
  if (own) {
    const float4 g0 = ld_keep_f4(gamma + col0), g1 = ld_keep_f4(gamma + col0 + 4);
    const float4 b0 = ld_keep_f4(beta + col0), b1 = ld_keep_f4(beta + col0 + 4);
    g8[0] = g0.x; g8[1] = g0.y; g8[2] = g0.z; g8[3] = g0.w;
    g8[4] = g1.x; g8[5] = g1.y; g8[6] = g1.z; g8[7] = g1.w;
    b8[0] = b0.x; b8[1] = b0.y; b8[2] = b0.z; b8[3] = b0.w;
    b8[4] = b1.x; b8[5] = b1.y; b8[6] = b1.z; b8[7] = b1.w;
  }
  auto row_of = [&](int64_t gi, int j) { return cid + (gi * kClRows + j) * ncl; };
  auto issue = [&](int64_t gi) {  // thread 0: group gi into stage gi % kClStages
    const int st = static_cast<int>(gi % kClStages);
    int nvalid = 0;
    for (int j = 0; j < kClRows; ++j) nvalid += row_of(gi, j) < rows;
    mbar_arrive_expect_tx(&full[st], nvalid * slice_bytes);
    for (int j = 0; j < kClRows; ++j) {
      const int64_t r = row_of(gi, j);
      if (r < rows)
        bulk_copy_g2s(stages + (static_cast<size_t>(st) * kClRows + j) * slice_bytes,
                      x + r * ldx + static_cast<int64_t>(q) * S, slice_bytes, &full[st], policy);
    }
  };

  if (tid == 0) {
    timed_out = 0;
    for (int i = 0; i < kClStages; ++i) mbar_init(&full[i], 1);
    for (int i = 0; i < kClSlots; ++i) mbar_init(&pbar[i], 1);
    mbar_init_fence();
    // arm the partial barriers of the first groups (peers may send at once
    // after the cluster barrier below)
    for (int64_t gi = 0; gi < kClSlots && gi < ngroups; ++gi)
      mbar_arrive_expect_tx(&pbar[gi], part_bytes);
    for (int64_t gi = 0; gi < kClStages && gi < ngroups; ++gi) issue(gi);
  }
  // every CTA's barriers are initialised and armed before anyone sends
  cluster_arrive();
  cluster_wait();

  uint4 xprev[kClRows], xcur[kClRows];
  for (int64_t gi = 0; gi <= ngroups; ++gi) {
    if (gi < ngroups) {
      const int st = static_cast<int>(gi % kClStages);
      const uint32_t parity = static_cast<uint32_t>((gi / kClStages) & 1);
      if (!timed_out && !mbar_wait_bounded(&full[st], parity, kWaitBudget)) {
        timed_out = 1;
        atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
      }
      Welford w[kClRows];
#pragma unroll
      for (int j = 0; j < kClRows; ++j) {
        w[j] = Welford{0.0f, 0.0f, 0.0f};
        xcur[j] = make_uint4(0, 0, 0, 0);
        if (own && row_of(gi, j) < rows) {
          xcur[j] = lds_u4(stages + (static_cast<size_t>(st) * kClRows + j) * slice_bytes +
                           16 * static_cast<size_t>(tid));
          w[j] = welford8(xcur[j]);
        }
        w[j] = warp_welford(w[j]);
        if (lane == 0) red[gi & 1][j][warp] = w[j];
      }
      __syncthreads();  // every thread has read stage st; red[gi & 1] complete
      if (tid == 0 && gi + kClStages < ngroups) {
        fence_proxy_async_smem();
        issue(gi + kClStages);
      }
      if (warp == 0) {
        // CTA triple of every row, then lane (j * C + k) sends row j's triple
        // to rank k.
        float4 mine = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < kClRows; ++j) {
          Welford r = lane < kClThreads / 32 ? red[gi & 1][j][lane] : Welford{0.0f, 0.0f, 0.0f};
          r = warp_welford(r);
          if (lane / static_cast<int>(C) == j) mine = make_float4(r.n, r.mean, r.m2, 0.0f);
        }
        if (lane < kClRows * static_cast<int>(C)) {
          const int j = lane / static_cast<int>(C), k = lane % static_cast<int>(C);
          const int sl = static_cast<int>(gi % kClSlots);
          st_async_f4(&slot[sl][j][q], &pbar[sl], static_cast<uint32_t>(k), mine);
        }
      }
    }
    if (gi > 0) {
      // finalise group gi - 1: wait for every rank's triples, merge in rank order
      const int64_t gp = gi - 1;
      const int sl = static_cast<int>(gp % kClSlots);
      const uint32_t pp = static_cast<uint32_t>((gp / kClSlots) & 1);
      if (!timed_out && !mbar_wait_bounded(&pbar[sl], pp, kWaitBudget)) {
        timed_out = 1;
        atomicCAS(err, 0, FR_DEVERR_TIMEOUT);
      }
      const int j_l = lane / static_cast<int>(C), k_l = lane % static_cast<int>(C);
      Welford pw{0.0f, 0.0f, 0.0f};
      if (j_l < kClRows) {
        const float4 v = slot[sl][j_l][k_l];
        pw = Welford{v.x, v.y, v.z};
      }
      // fixed butterfly inside each group of C lanes (lower rank first), so
      // every lane of the group and every CTA gets the same bits
      for (uint32_t o = 1; o < C; o <<= 1) {
        Welford v{__shfl_xor_sync(0xffffffffu, pw.n, o), __shfl_xor_sync(0xffffffffu, pw.mean, o),
                  __shfl_xor_sync(0xffffffffu, pw.m2, o)};
        pw = (k_l & o) ? chan_merge(v, pw) : chan_merge(pw, v);
      }
      // Re-arm slot sl for group gp + kClSlots.  Peers can send that group only
      // after this CTA publishes group gp + 2, which every thread reaches only
      // after finishing this finalisation, so the slot's data and the phase
      // every thread here waits on are both safe.
      if (tid == 0 && gp + kClSlots < ngroups) mbar_arrive_expect_tx(&pbar[sl], part_bytes);
#pragma unroll
      for (int j = 0; j < kClRows; ++j) {
        const int src = j * static_cast<int>(C);
        const float n = __shfl_sync(0xffffffffu, pw.n, src);
        const float mean = __shfl_sync(0xffffffffu, pw.mean, src);
        const float m2 = __shfl_sync(0xffffffffu, pw.m2, src);
        const int64_t r = row_of(gp, j);
        if (r >= rows) continue;
        const float rstd = rsqrtf(fmaf(m2, __frcp_rn(n), eps));
        if (q == 0 && tid == 0) {
          if (mean_out) mean_out[r] = mean;
          if (rstd_out) rstd_out[r] = rstd;
        }
        if (own) {
          const uint32_t wv[4] = {xprev[j].x, xprev[j].y, xprev[j].z, xprev[j].w};
          uint32_t o[4];
#pragma unroll
          for (int h = 0; h < 4; ++h)
            o[h] = pack_bf16x2(fmaf((bf16_lo(wv[h]) - mean) * rstd, g8[2 * h], b8[2 * h]),
                               fmaf((bf16_hi(wv[h]) - mean) * rstd, g8[2 * h + 1], b8[2 * h + 1]));
          uint16_t *dst = y + r * ldy + col0;
          asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(dst), "r"(o[0]), "r"(o[1]),
                       "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kClRows; ++j) xprev[j] = xcur[j];
  }
  // No CTA may leave while a peer can still write into or read its shared memory.
  cluster_arrive();
  cluster_wait();
  if (timed_out && tid == 0)  // last bounded wait on each stage's latest copy
    for (int64_t gl = ngroups - 1; gl >= 0 && gl >= ngroups - kClStages; --gl)
      mbar_wait_bounded(&full[gl % kClStages], static_cast<uint32_t>((gl / kClStages) & 1),
                        kWaitBudget);
}

// Buffers per CTA for a row of `cols` bf16 within `max_smem` bytes.
int ring_buffers(int64_t cols, int max_smem) {
  const size_t buf = static_cast<size_t>((cols * 2 + 127) / 128 * 128);
  const size_t avail = static_cast<size_t>(max_smem) - kRingHeader - 1024;  // static smem
  int nb = static_cast<int>(avail / buf);
  if (nb > kRingMaxBuffers) nb = kRingMaxBuffers;
  return nb;
}

}  // namespace

// Smallest cluster size whose slices fit one thread per 8 columns.
int cluster_size_for(int64_t cols) {
  for (int c = 1; c <= kClMaxCluster; c <<= 1)
    if (cols % (8 * c) == 0 && cols / c <= 8 * kClThreads) return c;
  return 0;
}

bool layernorm_cluster_ok(int64_t cols, bool aligned16) {
  return aligned16 && cluster_size_for(cols) > 0;
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
  const size_t smem = 128 + static_cast<size_t>(kClStages) * kClRows * (cols / C) * 2;
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
  // Persistent: every cluster that can be resident, no more than one per row.
  int64_t ncl = clusters;
  if (ncl > rows) ncl = rows;
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * C));
  return cudaLaunchKernelEx(&cfg, layernorm_cluster, x, gamma, beta, y, mean, rstd, rows, cols,
                            ldx, ldy, eps, err);
}

size_t layernorm_ring_smem(int64_t cols, int nbuf) {
  return static_cast<size_t>(kRingHeader) +
         static_cast<size_t>(nbuf) * static_cast<size_t>((cols * 2 + 127) / 128 * 128);
}

bool layernorm_ring_ok(int64_t cols, bool vec, int max_smem_optin) {
  return vec && cols % 16 == 0 && (cols * 2 + kRingChunk - 1) / kRingChunk <= kRingMaxChunks &&
         ring_buffers(cols, max_smem_optin) >= 1;
}

cudaError_t launch_layernorm_ring(const uint16_t *x, const float *gamma, const float *beta,
                                  uint16_t *y, float *mean, float *rstd, int64_t rows,
                                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int sm_count,
                                  int max_smem_optin, cudaStream_t s) {
  int *err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const int nbuf = ring_buffers(cols, max_smem_optin);
  if (nbuf < 1) return cudaErrorInvalidValue;
  const size_t smem = layernorm_ring_smem(cols, nbuf);
  e = cudaFuncSetAttribute(layernorm_ring, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layernorm_ring, kRingThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = static_cast<int64_t>(sm_count) * per_sm;
  if (grid > rows) grid = rows;
  layernorm_ring<<<static_cast<unsigned>(grid), kRingThreads, smem, s>>>(
      x, gamma, beta, y, mean, rstd, rows, cols, ldx, ldy, eps, nbuf, err);
  return cudaGetLastError();
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
