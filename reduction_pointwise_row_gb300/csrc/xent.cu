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
#include "common.cuh"
#include "launch.h"

namespace fr {

__device__ int g_fr_device_error;

namespace {

constexpr int kThreads = 512;
constexpr int kU = 2;  // 32-byte vectors (16 bf16 each) per thread per iteration
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

template <bool ARGMAX>
__global__ void __launch_bounds__(kThreads)
xent_rows(const uint16_t *__restrict__ logits, const int64_t *__restrict__ target,
          float *__restrict__ loss, float *__restrict__ target_logit, int64_t *__restrict__ argmax,
          float *__restrict__ loss_mean, void *__restrict__ ws, int64_t rows, int64_t cols,
          int64_t ld, int64_t ignore_index) {
  __shared__ MD red_md[kThreads / 32];
  __shared__ ArgBest red_arg[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  double cta_sum = 0.0;
  long long cta_cnt = 0;

  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint16_t *px = logits + row * ld;
    const RowSplit sp = row_split(px, cols, 2);
    const uint16_t *vx = px + sp.head;
    MD st{-INFINITY, 0.0f};
    ArgBest best{-INFINITY, INT64_MAX};
    for (int64_t base = 0; base < sp.nvec; base += kThreads * kU) {
      V8 v[kU];
      float cm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t vi = base + tid + kThreads * u;
        if (vi < sp.nvec) v[u] = ld_stream_v8(vx + vi * 16);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (base + tid + kThreads * u < sp.nvec) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            cm = max_nan(cm, max_nan(bf16_lo(v[u].w[j]), bf16_hi(v[u].w[j])));
        }
      if constexpr (ARGMAX) {
        // Only the first chunk and a chunk that beats the thread's best need a
        // scan for the first position of their max (elements are visited in
        // index order, so a later equal value never wins).
        if (best.i == INT64_MAX || (cm > best.v) || (cm != cm && best.v == best.v)) {
          bool found = false;
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int64_t vi = base + tid + kThreads * u;
            if (vi < sp.nvec) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float e = (j & 1) ? bf16_hi(v[u].w[j >> 1]) : bf16_lo(v[u].w[j >> 1]);
                const bool hit = (cm != cm) ? (e != e) : (e == cm);
                if (!found && hit) {
                  found = true;
                  best = ArgBest{cm, sp.head + vi * 16 + j};
                }
              }
            }
          }
        }
      }
      st = fold_chunk(st, cm);
      if (st.m == -INFINITY) continue;
      const float mb = st.m * kLog2e;
      float acc = 0.0f;
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (base + tid + kThreads * u < sp.nvec) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc += ex2(fmaf(bf16_lo(v[u].w[j]), kLog2e, -mb));
            acc += ex2(fmaf(bf16_hi(v[u].w[j]), kLog2e, -mb));
          }
        }
      st.d += acc;
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
      red_md[warp] = st;
      if constexpr (ARGMAX) red_arg[warp] = best;
    }
    __syncthreads();
    if (warp == 0) {
      MD r = red_md[lane < kThreads / 32 ? lane : 0];
      if (lane >= kThreads / 32) r = MD{-INFINITY, 0.0f};
      r = warp_md(r);
      ArgBest b{-INFINITY, INT64_MAX};
      if constexpr (ARGMAX) {
        if (lane < kThreads / 32) b = red_arg[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ArgBest other{__shfl_xor_sync(0xffffffffu, b.v, o),
                        static_cast<int64_t>(__shfl_xor_sync(0xffffffffu,
                                                             static_cast<long long>(b.i), o))};
          b = arg_better(b, other);
        }
      }
      if (lane == 0) {
        const float lse = r.m + logf(r.d);
        const int64_t t = target[row];
        float l, xt;
        if (t == ignore_index) {
          l = 0.0f;
          xt = 0.0f;
        } else if (t < 0 || t >= cols) {
          l = __int_as_float(0x7fc00000);
          xt = l;
          atomicCAS(&g_fr_device_error, 0, FR_DEVERR_BAD_TARGET);
        } else {
          xt = bf16_to_f32(px[t]);
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
    __syncthreads();  // red_* reused by the next row
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

int xent_grid(int64_t rows, int sm_count) {
  int64_t g = static_cast<int64_t>(sm_count) * kCtasPerSm;
  if (g > rows) g = rows;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

size_t xent_workspace(int64_t rows, int sm_count) {
  return 16 + 16 * static_cast<size_t>(xent_grid(rows, sm_count));
}

cudaError_t launch_xent(const uint16_t *logits, const int64_t *target, float *loss,
                        float *loss_mean, float *target_logit, int64_t *argmax, int64_t rows,
                        int64_t cols, int64_t ld, int64_t ignore_index, void *workspace,
                        int sm_count, cudaStream_t s) {
  const int grid = xent_grid(rows, sm_count);
  if (loss_mean != nullptr) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, 16, s);
    if (e != cudaSuccess) return e;
  }
  if (argmax != nullptr)
    xent_rows<true><<<grid, kThreads, 0, s>>>(logits, target, loss, target_logit, argmax,
                                              loss_mean, workspace, rows, cols, ld, ignore_index);
  else
    xent_rows<false><<<grid, kThreads, 0, s>>>(logits, target, loss, target_logit, argmax,
                                               loss_mean, workspace, rows, cols, ld,
                                               ignore_index);
  return cudaGetLastError();
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
