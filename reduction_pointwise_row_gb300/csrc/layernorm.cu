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

}  // namespace

bool layernorm_persistent_ok(int64_t cols, bool vec) {
  return vec && cols % 16 == 0 && cols / 16 <= kPersistMaxThreads * 4;
}

bool layernorm_looped_ring_ok(int64_t, bool, int) { return false; }

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
