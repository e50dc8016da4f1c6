// Fused log-softmax + cross entropy over bf16 logits, one pass per row.
//
// Per row, each thread keeps an online pair (m, l) -- the max so far and
// sum exp(x - m) -- and folds every chunk in with the merge of "Stax (4): GPU
// Codegen and Dynamic Shapes", section 9.5 (chunk max first, then one
// exponential per element and one rescale per chunk).  The CTA combines the
// pairs with the same merge (Proposition 9.1), and LSE = m + log l
// (section 9.10).  The loss follows PyTorch's cross_entropy: LSE - x[t] for a
// valid target, 0 for ignore_index; other targets give NaN and set the device
// error word (no trap).
//
// Rows need not be aligned (a row of 50257 bf16 is 100514 bytes): each row is
// split into a head of scalars up to the first 32-byte boundary, a body of
// 32-byte vectors and a tail of scalars; the masked lanes of the body never
// exist, so no -inf fill is needed except for the empty chunk.
//
// The grid is persistent (a fixed number of CTAs per SM, rows strided over
// CTAs).  The mean over counted rows is deterministic: each CTA adds its rows'
// losses in row order into an fp64 partial, writes it to the workspace, and
// the last CTA to finish (an atomic ticket; nobody waits) adds the partials in
// CTA order.
#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "launch.h"

namespace fr {

__device__ int g_fr_device_error;

namespace {

constexpr int kThreads = 512;
constexpr int kCtasPerSm = 2;

struct ArgBest {
  float v;
  int64_t i;
};

// The better of two (value, index) candidates: NaN beats numbers, larger
// beats smaller, equal values go to the lower index.
__device__ __forceinline__ ArgBest arg_better(ArgBest a, ArgBest b) {
  const bool an = a.v != a.v, bn = b.v != b.v;
  if (an || bn) {
    if (an && bn) return a.i <= b.i ? a : b;
    return an ? a : b;
  }
  if (a.v > b.v) return a;
  if (b.v > a.v) return b;
  return a.i <= b.i ? a : b;
}

__device__ __forceinline__ MD fold_chunk(MD st, float cm) {
  const float M = max_nan(st.m, cm);
  if (M == -INFINITY) return st;
  st.d = st.d * ex2((st.m - M) * kLog2e);
  st.m = M;
  return st;
}

struct Workspace {
  unsigned int *ticket;  // zeroed on the stream before each launch
  double *sums;          // [grid]
  long long *counts;     // [grid]
};

__device__ __forceinline__ Workspace carve(void *ws, int grid) {
  char *p = static_cast<char *>(ws);
  Workspace w;
  w.ticket = reinterpret_cast<unsigned int *>(p);
  w.sums = reinterpret_cast<double *>(p + 16);
  w.counts = reinterpret_cast<long long *>(p + 16 + 8 * static_cast<size_t>(grid));
  return w;
}

// U: 32-byte vectors (16 bf16 each) per thread per chunk.  DB: load the next
// chunk into a second register buffer while the current one is reduced.
template <bool ARGMAX, int U, bool DB>
__global__ void __launch_bounds__(kThreads, (ARGMAX || (DB && U > 1)) ? 1 : 2)
xent_rows(const uint16_t *__restrict__ logits, const int64_t *__restrict__ target,
          float *__restrict__ loss, float *__restrict__ target_logit, int64_t *__restrict__ argmax,
          float *__restrict__ loss_mean, void *__restrict__ ws, int64_t rows, int64_t cols,
          int64_t ld, int64_t ignore_index) {
  // Per-warp partials, double-buffered by row parity so one barrier per row
  // suffices (the next row writes the other half).
  __shared__ MD red_md[2][kThreads / 32];
  __shared__ ArgBest red_arg[2][kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  double cta_sum = 0.0;
  long long cta_cnt = 0;
  // Thread 0 fetches each row's target one row ahead, and gathers x[t] at the
  // start of the row, so neither load is waited for at the row's end.
  int64_t t_next = (tid == 0 && blockIdx.x < rows) ? target[blockIdx.x] : 0;
  int parity = 0;

  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
    const uint16_t *px = logits + row * ld;
    int64_t t = 0;
    uint16_t xt_bits = 0;
    if (tid == 0) {
      t = t_next;
      if (t >= 0 && t < cols) xt_bits = px[t];
      if (row + gridDim.x < rows) t_next = target[row + gridDim.x];
    }
    const RowSplit sp = row_split(px, cols, 2);
    const uint16_t *vx = px + sp.head;
    MD st{-INFINITY, 0.0f};
    ArgBest best{-INFINITY, INT64_MAX};
    // With DB the next chunk's loads are in flight while the current chunk is
    // reduced (register double buffering).
    const int nvec = static_cast<int>(sp.nvec);  // rows shorter than 2^31 (host check)
    constexpr int kU = U;
    V8 cur[kU], nxt[kU];
    if constexpr (DB) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int vi = tid + kThreads * u;
        if (vi < nvec) cur[u] = ld_stream_v8(vx + static_cast<size_t>(vi) * 16);
      }
    }
    for (int base = 0; base < nvec; base += kThreads * kU) {
      const int nbase = base + kThreads * kU;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if constexpr (DB) {
          const int vi = nbase + tid + kThreads * u;
          if (vi < nvec) nxt[u] = ld_stream_v8(vx + static_cast<size_t>(vi) * 16);
        } else {
          const int vi = base + tid + kThreads * u;
          if (vi < nvec) cur[u] = ld_stream_v8(vx + static_cast<size_t>(vi) * 16);
        }
      }
      // chunk max on packed bf16 pairs (exact: a max only selects)
      uint32_t m2 = 0xFF80FF80u;  // (-inf, -inf)
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (base + tid + kThreads * u < nvec) {
#pragma unroll
          for (int j = 0; j < 8; ++j) m2 = max_nan_bf16x2(m2, cur[u].w[j]);
        }
      const float cm = max_nan(bf16_lo(m2), bf16_hi(m2));
      if constexpr (ARGMAX) {
        // Only the first chunk and a chunk that beats the thread's best need a
        // scan for the first position of their max (elements are visited in
        // index order, so a later equal value never wins).
        if (best.i == INT64_MAX || (cm > best.v) || (cm != cm && best.v == best.v)) {
          bool found = false;
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int vi = base + tid + kThreads * u;
            if (vi < nvec) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float e = (j & 1) ? bf16_hi(cur[u].w[j >> 1]) : bf16_lo(cur[u].w[j >> 1]);
                const bool hit = (cm != cm) ? (e != e) : (e == cm);
                if (!found && hit) {
                  found = true;
                  best = ArgBest{cm, sp.head + static_cast<int64_t>(vi) * 16 + j};
                }
              }
            }
          }
        }
      }
      st = fold_chunk(st, cm);
      if (st.m != -INFINITY) {
        // exp(x - m) = 2^(x*log2e - m*log2e): one paired FMA and two SFU ops
        // per two elements, summed with a paired add.
        const float nmb = -st.m * kLog2e;
        const uint64_t l2e2 = pack_f32x2(kLog2e, kLog2e), nmb2 = pack_f32x2(nmb, nmb);
        uint64_t acc2 = 0;
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (base + tid + kThreads * u < nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t w = cur[u].w[j];
              const uint64_t t2 = fma_f32x2(pack_f32x2(bf16_lo(w), bf16_hi(w)), l2e2, nmb2);
              acc2 = add_f32x2(acc2, pack_f32x2(ex2(f32x2_lo(t2)), ex2(f32x2_hi(t2))));
            }
          }
        st.d += f32x2_lo(acc2) + f32x2_hi(acc2);
      }
      if constexpr (DB) {
#pragma unroll
        for (int u = 0; u < kU; ++u) cur[u] = nxt[u];
      }
    }
    // head and tail scalars (at most 15 + 15), one per thread
    int64_t si = -1;
    if (tid < sp.head) si = tid;
    else if (tid < sp.head + sp.tail) si = sp.head + sp.nvec * 16 + (tid - sp.head);
    if (si >= 0) {
      const float e = bf16_to_f32(ld_stream_u16(px + si));
      st = md_merge(st, MD{e, 1.0f});
      if constexpr (ARGMAX) best = arg_better(best, ArgBest{e, si});
    }

    // CTA combine
    st = warp_md(st);
    if constexpr (ARGMAX) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ArgBest other{__shfl_xor_sync(0xffffffffu, best.v, o),
                      static_cast<int64_t>(__shfl_xor_sync(0xffffffffu,
                                                           static_cast<long long>(best.i), o))};
        best = arg_better(best, other);
      }
    }
    if (lane == 0) {
      red_md[parity][warp] = st;
      if constexpr (ARGMAX) red_arg[parity][warp] = best;
    }
    __syncthreads();
    if (warp == 0) {
      MD r = red_md[parity][lane < kThreads / 32 ? lane : 0];
      if (lane >= kThreads / 32) r = MD{-INFINITY, 0.0f};
      r = warp_md(r);
      ArgBest b{-INFINITY, INT64_MAX};
      if constexpr (ARGMAX) {
        if (lane < kThreads / 32) b = red_arg[parity][lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ArgBest other{__shfl_xor_sync(0xffffffffu, b.v, o),
                        static_cast<int64_t>(__shfl_xor_sync(0xffffffffu,
                                                             static_cast<long long>(b.i), o))};
          b = arg_better(b, other);
        }
      }
      if (lane == 0) {  // thread 0: holds t and x[t]
        const float lse = r.m + logf(r.d);
        float l, xt;
        if (t == ignore_index) {
          l = 0.0f;
          xt = 0.0f;
        } else if (t < 0 || t >= cols) {
          l = __int_as_float(0x7fc00000);
          xt = l;
          atomicCAS(&g_fr_device_error, 0, FR_DEVERR_BAD_TARGET);
        } else {
          xt = bf16_to_f32(xt_bits);
          l = lse - xt;
        }
        if (loss) loss[row] = l;
        if (target_logit) target_logit[row] = xt;
        if constexpr (ARGMAX) argmax[row] = b.i;
        if (t != ignore_index) {
          cta_sum += static_cast<double>(l);
          ++cta_cnt;
        }
      }
    }
    // No trailing barrier: the next row uses the other half of red_*, and the
    // barrier of that row orders this row's reads before the half is reused.
  }

  if (loss_mean != nullptr && tid == 0) {
    Workspace w = carve(ws, gridDim.x);
    w.sums[blockIdx.x] = cta_sum;
    w.counts[blockIdx.x] = cta_cnt;
    __threadfence();
    const unsigned int ticket = atomicAdd(w.ticket, 1u);
    if (ticket == gridDim.x - 1) {
      __threadfence();
      double s = 0.0;
      long long c = 0;
      for (unsigned int k = 0; k < gridDim.x; ++k) {
        s += *reinterpret_cast<volatile double *>(&w.sums[k]);
        c += *reinterpret_cast<volatile long long *>(&w.counts[k]);
      }
      *loss_mean = static_cast<float>(s / static_cast<double>(c));
      *w.ticket = 0u;
    }
  }
}

// Launch-configuration candidates (Stax (4), section 9.6, Algorithm 9.1):
// a small set of compiled variants, the fastest chosen by measurement on
// GB300; FR_XENT_VARIANT=<index> forces one (for re-measuring the choice).
struct XentVariant {
  const void *kern;      // the non-argmax kernel
  const void *kern_arg;  // the argmax kernel
  int ctas_per_sm;
};

template <int U, bool DB>
XentVariant make_variant() {
  return XentVariant{reinterpret_cast<const void *>(&xent_rows<false, U, DB>),
                     reinterpret_cast<const void *>(&xent_rows<true, U, DB>), 0};
}

constexpr int kNumVariants = 4;
constexpr int kDefaultVariant = 0;

XentVariant *variants() {
  static XentVariant v[kNumVariants] = {make_variant<2, false>(), make_variant<1, true>(),
                                        make_variant<4, false>(), make_variant<2, true>()};
  return v;
}

int chosen_variant() {
  static int chosen = -1;
  if (chosen < 0) {
    chosen = kDefaultVariant;
    if (const char *e = getenv("FR_XENT_VARIANT")) {
      const int k = atoi(e);
      if (k >= 0 && k < kNumVariants) chosen = k;
    }
  }
  return chosen;
}

// CTAs per SM the chosen kernel keeps resident (registers decide it), so the
// persistent grid fills every SM whatever the compiler's register count.
int xent_ctas_per_sm(bool argmax) {
  XentVariant &v = variants()[chosen_variant()];
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, argmax ? v.kern_arg : v.kern, kThreads,
                                                    0) != cudaSuccess) {
    cudaGetLastError();
    return kCtasPerSm;
  }
  return n < 1 ? 1 : n;
}

// Persistent grid of one kernel: every CTA it can keep resident on every SM.
int xent_grid(int64_t rows, int sm_count, bool argmax) {
  int64_t g = static_cast<int64_t>(sm_count) * xent_ctas_per_sm(argmax);
  if (g > rows) g = rows;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

size_t xent_workspace(int64_t rows, int sm_count) {
  // One fp64 sum and one count per CTA of the larger of the two grids.
  const int g = std::max(xent_grid(rows, sm_count, false), xent_grid(rows, sm_count, true));
  return 16 + 16 * static_cast<size_t>(g);
}

cudaError_t launch_xent(const uint16_t *logits, const int64_t *target, float *loss,
                        float *loss_mean, float *target_logit, int64_t *argmax, int64_t rows,
                        int64_t cols, int64_t ld, int64_t ignore_index, void *workspace,
                        int sm_count, cudaStream_t s) {
  const int grid = xent_grid(rows, sm_count, argmax != nullptr);
  if (loss_mean != nullptr) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, 16, s);
    if (e != cudaSuccess) return e;
  }
  const XentVariant &v = variants()[chosen_variant()];
  void *args[] = {&logits, &target, &loss, &target_logit, &argmax, &loss_mean, &workspace,
                  &rows, &cols, &ld, &ignore_index};
  return cudaLaunchKernel(argmax != nullptr ? v.kern_arg : v.kern, dim3(grid), dim3(kThreads),
                          args, 0, s);
}

cudaError_t device_error_word(int **out) {
  constexpr int kMaxDev = 64;
  static int *cache[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && cache[dev] != nullptr) {
    *out = cache[dev];
    return cudaSuccess;
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_fr_device_error);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev) cache[dev] = static_cast<int *>(p);
  *out = static_cast<int *>(p);
  return cudaSuccess;
}

cudaError_t device_error_read_and_clear(cudaStream_t s, int *code) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_fr_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_fr_device_error, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *code = v;
  return cudaSuccess;
}

}  // namespace fr
