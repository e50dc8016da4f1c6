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
// split into a head of scalars up to the first 16-byte boundary, an interior
// of 16-byte vectors streamed through a per-thread cp.async ring, and a tail
// of scalars; vectors past the interior's end are filled with -inf (adding
// nothing to l).
//
// The launch configuration (threads, vectors per ring item, ring stages,
// CTAs per SM) is a point of a box searched by measurement ("Stax (4)",
// section 9.6); the default is the fastest point on GB300.  The grid is
// persistent (CTAs per SM x SMs, rows strided over CTAs).  The mean over counted rows is deterministic: each CTA adds its rows'
// losses in row order into an fp64 partial, writes it to the workspace, and
// the last CTA to finish (an atomic ticket; nobody waits) adds the partials in
// a fixed order.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace fr {

__device__ int g_fr_device_error;

namespace {

constexpr int kMaxCtasPerSm = 16;  // largest persistent grid: 16 CTAs per SM (workspace bound)

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

// Workspace layout: the ticket (bytes 0..7), the batch's mean parts at
// FR_XENT_PARTS_OFFSET (fp64 sum of the averaged losses, fp64 count of the
// rows averaged), then one fp64 partial sum and one count per CTA.
//
// The ticket holds a tag (high 32 bits) and the CTAs arrived so far (low 32
// bits).  fr_xent_workspace_init writes the tag with no arrivals; the last
// CTA of every launch writes it back, so a prepared workspace stays prepared
// and no launch needs a reset of its own.  A CTA that finds another tag (a
// workspace never prepared) records FR_DEVERR_BAD_WORKSPACE and the mean is
// not written.
constexpr size_t kPartsOffset = FR_XENT_PARTS_OFFSET;
constexpr size_t kCtaOffset = kPartsOffset + 16;
static_assert(kPartsOffset % 8 == 0 && kPartsOffset >= 8, "parts after the ticket, fp64 aligned");
constexpr unsigned long long kTicketTag = 0x4652584EULL << 32;  // "FRXN", no arrivals

struct Workspace {
  unsigned long long *ticket;  // tag | arrivals
  double *parts;               // [2]: sum of the averaged losses, rows averaged
  double *sums;                // [grid]
  long long *counts;           // [grid]
};

__device__ __forceinline__ Workspace carve(void *ws, int grid) {
  char *p = static_cast<char *>(ws);
  Workspace w;
  w.ticket = reinterpret_cast<unsigned long long *>(p);
  w.parts = reinterpret_cast<double *>(p + kPartsOffset);
  w.sums = reinterpret_cast<double *>(p + kCtaOffset);
  w.counts = reinterpret_cast<long long *>(p + kCtaOffset + 8 * static_cast<size_t>(grid));
  return w;
}

// The mean over counted rows, in a fixed order: every CTA stores its fp64
// partial and count; the last CTA to arrive (an atomic ticket, nobody waits)
// adds them up -- thread i the partials i, i + T, ... in order, then a fixed
// tree over the CTA -- writes the mean and resets the ticket to its tag.  Called by
// every thread of the CTA at the end of the kernel; cta_sum and cta_cnt are
// thread 0's.  (A single thread adding the partials one after another took
// 18 us for 304 CTAs on GB300, whose fp64 adds are slow.)
template <int T>
__device__ __forceinline__ void finish_mean(void *ws, float *loss_mean, double cta_sum,
                                            long long cta_cnt) {
  __shared__ int last;
  __shared__ double red_s[T / 32];
  __shared__ long long red_c[T / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Workspace w = carve(ws, gridDim.x);
  __syncthreads();
  if (tid == 0) {
    w.sums[blockIdx.x] = cta_sum;
    w.counts[blockIdx.x] = cta_cnt;
    __threadfence();
    const unsigned long long old = atomicAdd(w.ticket, 1ull);
    if ((old & ~0xFFFFFFFFull) != kTicketTag) {  // not a prepared workspace
      atomicCAS(&g_fr_device_error, 0, FR_DEVERR_BAD_WORKSPACE);
      last = 0;
    } else {
      last = (old & 0xFFFFFFFFull) == gridDim.x - 1;
    }
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  double s = 0.0;
  long long c = 0;
  for (unsigned int i = tid; i < gridDim.x; i += T) {
    s += *reinterpret_cast<volatile double *>(&w.sums[i]);
    c += *reinterpret_cast<volatile long long *>(&w.counts[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_down_sync(0xffffffffu, s, o);
    c += __shfl_down_sync(0xffffffffu, c, o);
  }
  if (lane == 0) {
    red_s[warp] = s;
    red_c[warp] = c;
  }
  __syncthreads();
  if (tid == 0) {
    double S = 0.0;
    long long n = 0;
    for (int i = 0; i < T / 32; ++i) {
      S += red_s[i];
      n += red_c[i];
    }
    w.parts[0] = S;
    w.parts[1] = static_cast<double>(n);
    *loss_mean = static_cast<float>(S / static_cast<double>(n));
    *w.ticket = kTicketTag;
  }
}

struct RowGeom {
  const unsigned char *row;  // row start
  uint64_t a0;               // first 16-byte boundary at or after the row start
  uint32_t ibytes;           // interior bytes (multiple of 16)
  int head;                  // elements before a0
  int tail;                  // elements after the interior
};

// ES: bytes per logit (2 for bf16, 4 for fp32)
template <int ES>
__device__ __forceinline__ RowGeom row_geom(const void *logits, int64_t row, int64_t ld,
                                            int64_t cols) {
  RowGeom g;
  g.row = static_cast<const unsigned char *>(logits) + row * ld * ES;
  const uint64_t s0 = reinterpret_cast<uint64_t>(g.row);
  const uint64_t s1 = s0 + ES * static_cast<uint64_t>(cols);
  const uint64_t a0 = (s0 + 15) & ~uint64_t(15), a1 = s1 & ~uint64_t(15);
  if (a1 <= a0) {  // a row too short to hold an aligned 16 bytes: all head
    g.a0 = s0;
    g.ibytes = 0;
    g.head = static_cast<int>(cols);
    g.tail = 0;
    return g;
  }
  g.a0 = a0;
  g.ibytes = static_cast<uint32_t>(a1 - a0);
  g.head = static_cast<int>((a0 - s0) / ES);
  g.tail = static_cast<int>((s1 - a1) / ES);
  return g;
}

// Logit i of a row as fp32 (bf16 widened exactly), plain or streaming load.
template <bool F32>
__device__ __forceinline__ float logit_at(const unsigned char *row, int64_t i) {
  if constexpr (F32) return reinterpret_cast<const float *>(row)[i];
  else return bf16_to_f32(reinterpret_cast<const uint16_t *>(row)[i]);
}
template <bool F32>
__device__ __forceinline__ float logit_stream(const unsigned char *row, int64_t i) {
  if constexpr (F32) return ld_stream_f32(reinterpret_cast<const float *>(row) + i);
  else return bf16_to_f32(ld_stream_u16(reinterpret_cast<const uint16_t *>(row) + i));
}

// ---- asynchronous-copy ring variant ---------------------------------------------
// Each thread streams its share of the CTA's rows as items of U 16-byte vectors
// (item c of row k covers vectors c*T*U + u*T + tid of the row's 16-byte
// aligned interior).  Items go through a per-thread ring of NS shared-memory
// stages filled with cp.async (no registers held, one commit group per item),
// continuing across row boundaries, so NS - 1 items per thread are always in
// flight -- also while the CTA combines a finished row.  The template covers
// argmax and fp32 logits; the library instantiates it over its configuration
// box for bf16 logits without argmax (the warp-per-row kernel serves the
// other cases).
template <bool ARGMAX, int T, int U, int NS, bool F32 = false>
__global__ void __launch_bounds__(T, 1)
xent_async(const void *__restrict__ logits, const int64_t *__restrict__ target,
           float *__restrict__ loss, float *__restrict__ target_logit,
           int64_t *__restrict__ argmax, float *__restrict__ loss_mean, void *__restrict__ ws,
           int64_t rows, int64_t cols, int64_t ld, int64_t ignore_index) {
  pdl_enter();
  constexpr int ES = F32 ? 4 : 2;  // bytes per logit
  constexpr int EPV = 16 / ES;     // logits per 16-byte vector
  extern __shared__ __align__(128) unsigned char smem[];  // [NS][U][T] x 16 bytes
  __shared__ MD red_md[2][T / 32];
  __shared__ ArgBest red_arg[2][T / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t G = gridDim.x;
  const int64_t nk = blockIdx.x < rows ? (rows - blockIdx.x + G - 1) / G : 0;
  auto slot = [&](int s, int u) {
    return smem + (static_cast<size_t>(s * U + u) * T + tid) * 16;
  };
  // Producer cursor: the next item to copy is item pc of row pk (pn items).
  // Rows without items (too short for an aligned interior) are skipped, as
  // the consumer skips them: the i-th item produced is the i-th consumed.
  int64_t pk = 0;
  int pc = 0, pn = 0, ps = 0;
  RowGeom pg{};
  auto load_row = [&]() {
    for (; pk < nk; ++pk) {
      pg = row_geom<ES>(logits, blockIdx.x + pk * G, ld, cols);
      pn = static_cast<int>((pg.ibytes / 16 + T * U - 1) / (T * U));
      if (pn > 0) return;
    }
  };
  load_row();
  auto produce = [&]() {
    if (pk < nk) {
      const int nv = static_cast<int>(pg.ibytes / 16);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = pc * T * U + u * T + tid;
        if (v < nv)
          cp_async_16(slot(ps, u),
                      reinterpret_cast<const unsigned char *>(pg.a0) + 16 * static_cast<size_t>(v));
      }
      if (++pc >= pn) {  // next row with items
        pc = 0;
        ++pk;
        load_row();
      }
    }
    cp_async_commit();  // one group per item, empty past the last item
    ps = ps + 1 == NS ? 0 : ps + 1;
  };
#pragma unroll
  for (int i = 0; i < NS - 1; ++i) produce();

  double cta_sum = 0.0;
  long long cta_cnt = 0;
  int64_t t_next = (tid == 0 && nk > 0) ? target[blockIdx.x] : 0;
  int cs = 0;  // consumer stage
  int parity = 0;
  for (int64_t k = 0; k < nk; ++k, parity ^= 1) {
    const int64_t row = blockIdx.x + k * G;
    const RowGeom g = row_geom<ES>(logits, row, ld, cols);
    int64_t t = 0;
    float xt_v = 0.0f;
    if (tid == 0) {
      t = t_next;
      if (t >= 0 && t < cols) xt_v = logit_at<F32>(g.row, t);
      if (k + 1 < nk) t_next = target[row + G];
    }
    const int nv = static_cast<int>(g.ibytes / 16);
    const int nitems = (nv + T * U - 1) / (T * U);
    MD st{-INFINITY, 0.0f};
    ArgBest best{-INFINITY, INT64_MAX};
    for (int c = 0; c < nitems; ++c) {
      produce();                 // keep NS - 1 items in flight
      cp_async_wait<NS - 1>();   // this thread's copies of item (k, c) landed
      // a vector past the interior holds -inf (adds nothing)
      constexpr uint32_t kNegInf = F32 ? 0xFF800000u : 0xFF80FF80u;
      uint32_t wv[U][4];
      uint32_t m2 = kNegInf;  // bf16: running max of bf16 pairs
      float mf = -INFINITY;   // fp32: running max
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = c * T * U + u * T + tid;
        if (v < nv) {
          const uint4 q = lds_u4(slot(cs, u));
          wv[u][0] = q.x; wv[u][1] = q.y; wv[u][2] = q.z; wv[u][3] = q.w;
          if constexpr (F32)
            mf = max_nan(max_nan(mf, max_nan(__uint_as_float(q.x), __uint_as_float(q.y))),
                         max_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
          else
            m2 = max_nan_bf16x2(m2, max_nan_bf16x2(max_nan_bf16x2(q.x, q.y), max_nan_bf16x2(q.z, q.w)));
        } else {
          wv[u][0] = wv[u][1] = wv[u][2] = wv[u][3] = kNegInf;
        }
      }
      cs = cs + 1 == NS ? 0 : cs + 1;
      const float cm = F32 ? mf : max_nan(bf16_lo(m2), bf16_hi(m2));
      // logit j (0 .. EPV - 1) of vector u
      auto elem = [&](int u, int j) {
        if constexpr (F32) return __uint_as_float(wv[u][j]);
        else return (j & 1) ? bf16_hi(wv[u][j >> 1]) : bf16_lo(wv[u][j >> 1]);
      };
      if constexpr (ARGMAX) {
        if (best.i == INT64_MAX || cm > best.v || (cm != cm && best.v == best.v)) {
          bool found = false;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = c * T * U + u * T + tid;
#pragma unroll
            for (int j = 0; j < EPV; ++j) {
              const float e = elem(u, j);
              const bool hit = (cm != cm) ? (e != e) : (e == cm);
              if (!found && hit && v < nv) {
                found = true;
                best = ArgBest{cm, g.head + EPV * static_cast<int64_t>(v) + j};
              }
            }
          }
        }
      }
      st = fold_chunk(st, cm);
      if (st.m != -INFINITY) {
        const float nmb = -st.m * kLog2e;
        const uint64_t l2e2 = pack_f32x2(kLog2e, kLog2e), nmb2 = pack_f32x2(nmb, nmb);
        uint64_t acc2 = 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int j = 0; j < EPV / 2; ++j) {  // a pair of logits per step
            const uint64_t t2 = fma_f32x2(pack_f32x2(elem(u, 2 * j), elem(u, 2 * j + 1)), l2e2, nmb2);
            acc2 = add_f32x2(acc2, pack_f32x2(ex2(f32x2_lo(t2)), ex2(f32x2_hi(t2))));
          }
        st.d += f32x2_lo(acc2) + f32x2_hi(acc2);
      }
    }
    int64_t si = -1;
    if (tid < g.head) si = tid;
    else if (tid < g.head + g.tail) si = g.head + g.ibytes / ES + (tid - g.head);
    if (si >= 0) {
      const float e = logit_stream<F32>(g.row, si);
      st = md_merge(st, MD{e, 1.0f});
      if constexpr (ARGMAX) best = arg_better(best, ArgBest{e, si});
    }
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
      MD r = lane < T / 32 ? red_md[parity][lane] : MD{-INFINITY, 0.0f};
      r = warp_md(r);
      ArgBest bb{-INFINITY, INT64_MAX};
      if constexpr (ARGMAX) {
        if (lane < T / 32) bb = red_arg[parity][lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ArgBest other{__shfl_xor_sync(0xffffffffu, bb.v, o),
                        static_cast<int64_t>(__shfl_xor_sync(0xffffffffu,
                                                             static_cast<long long>(bb.i), o))};
          bb = arg_better(bb, other);
        }
      }
      if (lane == 0) {
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
          xt = xt_v;
          l = lse - xt;
        }
        if (loss) loss[row] = l;
        if (target_logit) target_logit[row] = xt;
        if constexpr (ARGMAX) argmax[row] = bb.i;
        if (t != ignore_index) {
          cta_sum += static_cast<double>(l);
          ++cta_cnt;
        }
      }
    }
  }
  cp_async_wait<0>();
  if (loss_mean != nullptr) finish_mean<T>(ws, loss_mean, cta_sum, cta_cnt);
}

// ---- warp-per-row variant ------------------------------------------------------
// Each warp streams whole rows with 32-byte register loads (NV vectors of
// EPV logits per lane in flight, evict-first), folding every chunk into the
// lane's online pair (m, l); the lane pairs merge by shuffles (Proposition
// 9.1), so a row needs no CTA barrier.  The grid is persistent (warp w takes
// rows w, w + W, ...); each warp adds its rows' losses in row order, the CTA
// adds its warps' sums in warp order, and the last CTA adds the CTAs' sums
// in a fixed order (finish_mean).
constexpr int kWarpCta = 256;

template <bool ARGMAX, bool F32, int NV>
__global__ void __launch_bounds__(kWarpCta, ARGMAX || NV > 4 ? 2 : 4)
xent_warp(const void *__restrict__ logits, const int64_t *__restrict__ target,
          float *__restrict__ loss, float *__restrict__ target_logit, int64_t *__restrict__ argmax,
          float *__restrict__ loss_mean, void *__restrict__ ws, int64_t rows, int64_t cols,
          int64_t ld, int64_t ignore_index) {
  pdl_enter();
  constexpr int ES = F32 ? 4 : 2;  // bytes per logit
  constexpr int EPV = 32 / ES;     // logits per 32-byte vector
  constexpr int W = kWarpCta / 32;
  __shared__ double warp_s[W];
  __shared__ long long warp_c[W];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * W + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * W;
  const unsigned char *base = static_cast<const unsigned char *>(logits);
  double w_sum = 0.0;
  long long w_cnt = 0;
  for (int64_t row = gw; row < rows; row += nw) {
    const unsigned char *pr = base + row * ld * ES;
    const RowSplit sp = row_split(pr, cols, ES);
    const unsigned char *pv = pr + static_cast<int64_t>(sp.head) * ES;
    MD st{-INFINITY, 0.0f};
    ArgBest best{-INFINITY, INT64_MAX};
    for (int64_t b0 = 0; b0 < sp.nvec; b0 += 32 * NV) {
      V8 v[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int64_t vi = b0 + lane + 32 * k;
        if (vi < sp.nvec) v[k] = ld_stream_v8(pv + vi * 32);
        else
#pragma unroll
          for (int j = 0; j < 8; ++j) v[k].w[j] = F32 ? 0xFF800000u : 0xFF80FF80u;  // -inf
      }
      // logit j (0 .. EPV - 1) of vector k
      auto elem = [&](int k, int j) {
        if constexpr (F32) return __uint_as_float(v[k].w[j]);
        else return (j & 1) ? bf16_hi(v[k].w[j >> 1]) : bf16_lo(v[k].w[j >> 1]);
      };
      float cm;
      if constexpr (F32) {
        cm = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
          for (int j = 0; j < 8; ++j) cm = max_nan(cm, __uint_as_float(v[k].w[j]));
      } else {
        uint32_t m2 = 0xFF80FF80u;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
          for (int j = 0; j < 8; ++j) m2 = max_nan_bf16x2(m2, v[k].w[j]);
        cm = max_nan(bf16_lo(m2), bf16_hi(m2));
      }
      if constexpr (ARGMAX) {
        if (best.i == INT64_MAX || cm > best.v || (cm != cm && best.v == best.v)) {
          bool found = false;
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int64_t vi = b0 + lane + 32 * k;
#pragma unroll
            for (int j = 0; j < EPV; ++j) {
              const float e = elem(k, j);
              const bool hit = (cm != cm) ? (e != e) : (e == cm);
              if (!found && hit && vi < sp.nvec) {
                found = true;
                best = ArgBest{cm, sp.head + EPV * vi + j};
              }
            }
          }
        }
      }
      st = fold_chunk(st, cm);
      if (st.m != -INFINITY) {
        const float nmb = -st.m * kLog2e;
        const uint64_t l2e2 = pack_f32x2(kLog2e, kLog2e), nmb2 = pack_f32x2(nmb, nmb);
        uint64_t acc2 = 0;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
          for (int j = 0; j < EPV / 2; ++j) {
            const uint64_t t2 = fma_f32x2(pack_f32x2(elem(k, 2 * j), elem(k, 2 * j + 1)), l2e2, nmb2);
            acc2 = add_f32x2(acc2, pack_f32x2(ex2(f32x2_lo(t2)), ex2(f32x2_hi(t2))));
          }
        st.d += f32x2_lo(acc2) + f32x2_hi(acc2);
      }
    }
    // head and tail scalars, one per lane (fewer than EPV each)
    int64_t si = -1;
    if (lane < sp.head) si = lane;
    else if (lane < sp.head + sp.tail) si = sp.head + sp.nvec * EPV + (lane - sp.head);
    if (si >= 0) {
      const float e = logit_stream<F32>(pr, si);
      st = md_merge(st, MD{e, 1.0f});
      if constexpr (ARGMAX) best = arg_better(best, ArgBest{e, si});
    }
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
      const int64_t t = target[row];
      const float lse = st.m + logf(st.d);
      float l, xt;
      if (t == ignore_index) {
        l = 0.0f;
        xt = 0.0f;
      } else if (t < 0 || t >= cols) {
        l = __int_as_float(0x7fc00000);
        xt = l;
        atomicCAS(&g_fr_device_error, 0, FR_DEVERR_BAD_TARGET);
      } else {
        xt = logit_at<F32>(pr, t);
        l = lse - xt;
      }
      if (loss) loss[row] = l;
      if (target_logit) target_logit[row] = xt;
      if constexpr (ARGMAX) argmax[row] = best.i;
      if (t != ignore_index) {
        w_sum += static_cast<double>(l);
        ++w_cnt;
      }
    }
  }
  if (loss_mean == nullptr) return;
  if (lane == 0) {
    warp_s[warp] = w_sum;
    warp_c[warp] = w_cnt;
  }
  __syncthreads();
  double cta_sum = 0.0;
  long long cta_cnt = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < W; ++i) {  // the CTA's warps in order
      cta_sum += warp_s[i];
      cta_cnt += warp_c[i];
    }
  finish_mean<kWarpCta>(ws, loss_mean, cta_sum, cta_cnt);
}

}  // namespace

size_t xent_workspace(int64_t rows, int sm_count) {
  // A ticket, the mean's parts, then one fp64 sum and one count per CTA of
  // the largest grid.
  int64_t g = static_cast<int64_t>(sm_count) * kMaxCtasPerSm;
  if (g > rows) g = rows;
  if (g < 1) g = 1;
  return kCtaOffset + 16 * static_cast<size_t>(g);
}

namespace {

// ---- the configuration space of the asynchronous-copy kernel -----------------
// threads x vectors x stages (compiled) x CTAs per SM (at launch), each a
// power of two: the box the coordinate descent of section 9.6 walks.  Only the
// kernel without argmax is instantiated over the box, and not at 1024 threads x
// 8 vectors, which spills registers (Algorithm 9.1, line 4: cost +inf).
struct AsyncEntry {
  int T, U, NS;
  const void *kern;
};
#define FR_XA(T, U, NS) AsyncEntry{T, U, NS, reinterpret_cast<const void *>(&xent_async<false, T, U, NS>)}
#define FR_XA_T(T)                                                                           \
  FR_XA(T, 1, 2), FR_XA(T, 1, 4), FR_XA(T, 1, 8), FR_XA(T, 2, 2), FR_XA(T, 2, 4), FR_XA(T, 2, 8), \
      FR_XA(T, 4, 2), FR_XA(T, 4, 4), FR_XA(T, 4, 8), FR_XA(T, 8, 2), FR_XA(T, 8, 4), FR_XA(T, 8, 8)
const AsyncEntry kAsyncBox[] = {FR_XA_T(128), FR_XA_T(256), FR_XA_T(512), FR_XA(1024, 1, 2),
                                FR_XA(1024, 1, 4), FR_XA(1024, 1, 8), FR_XA(1024, 2, 2),
                                FR_XA(1024, 2, 4), FR_XA(1024, 2, 8), FR_XA(1024, 4, 2),
                                FR_XA(1024, 4, 4), FR_XA(1024, 4, 8)};
#undef FR_XA_T
#undef FR_XA

const AsyncEntry *async_entry(const XentConfig &c) {
  for (const AsyncEntry &e : kAsyncBox)
    if (e.T == c.threads && e.U == c.vectors && e.NS == c.stages) return &e;
  return nullptr;
}

struct Recorded {
  int device;
  int64_t rows, cols, ld;
  XentConfig cfg;
};
std::mutex g_rec_mu;
std::vector<Recorded> g_recorded;

}  // namespace

cudaError_t capped_smem(size_t need, int per_sm, size_t *out);
cudaError_t launch_warp_kernel(const void *kern, int per_sm_cap, const void *logits,
                               const int64_t *target, float *loss, float *loss_mean,
                               float *target_logit, int64_t *argmax, int64_t rows, int64_t cols,
                               int64_t ld, int64_t ignore_index, void *workspace, int sm_count,
                               cudaStream_t s);
template <bool ARGMAX, bool F32>
const void *warp_kernel(int nv);

// The default point: the warp-per-row kernel with 8 vectors a lane, two CTAs
// per SM.  Measured on GB300 for bf16 [8192, 50257] with the mean (back to
// back, rotating inputs; every runnable point of both families): (32, 8, 1, 2)
// 126.5 us, (32, 4, 1, 4) 127.5, the ring's fastest point (128, 8, 2, 4)
// 129.7, (128, 4, 4, 4) 131.7, (128, 2, 8, 4) 136.9 ... (32, 4, 1, 1) 189.2,
// (128, 1, 2, 1) 938.6.
XentConfig xent_default_config() { return XentConfig{32, 8, 1, 2}; }

namespace {
// The warp-per-row family: threads 32 (a warp per row), vectors 4 or 8,
// stages 1 (no ring), ctas_per_sm the cap on 256-thread CTAs per SM.
cudaError_t warp_config_check(const XentConfig &cfg) {
  auto pow2_in = [](int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; };
  if ((cfg.vectors != 4 && cfg.vectors != 8) || cfg.stages != 1 ||
      !pow2_in(cfg.ctas_per_sm, 1, kMaxCtasPerSm))
    return cudaErrorInvalidValue;
  const void *kern = warp_kernel<false, false>(cfg.vectors);
  cudaFuncAttributes fa{};
  cudaError_t err = cudaFuncGetAttributes(&fa, kern);
  if (err != cudaSuccess) return err;
  if (fa.localSizeBytes > 0) return cudaErrorInvalidConfiguration;  // spills: t = inf
  if ((err = set_smem_limit(reinterpret_cast<const void *>(kern), 0)) !=
      cudaSuccess)
    return err;
  int per_sm = 0;
  err = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern), kWarpCta, 0);
  if (err != cudaSuccess) return err;
  return per_sm >= cfg.ctas_per_sm ? cudaSuccess : cudaErrorInvalidConfiguration;
}
}  // namespace

cudaError_t xent_config_check(const XentConfig &cfg, int max_smem_optin) {
  auto pow2_in = [](int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; };
  if (cfg.threads == 32) return warp_config_check(cfg);
  if (!pow2_in(cfg.threads, 128, 1024) || !pow2_in(cfg.vectors, 1, 8) ||
      !pow2_in(cfg.stages, 2, 8) || !pow2_in(cfg.ctas_per_sm, 1, kMaxCtasPerSm))
    return cudaErrorInvalidValue;
  const AsyncEntry *e = async_entry(cfg);
  if (e == nullptr) return cudaErrorInvalidConfiguration;  // in the box, not compiled (spills)
  const size_t smem = static_cast<size_t>(e->NS) * e->U * e->T * 16;
  if (smem > static_cast<size_t>(max_smem_optin)) return cudaErrorInvalidConfiguration;
  cudaFuncAttributes fa{};
  cudaError_t err = cudaFuncGetAttributes(&fa, e->kern);
  if (err != cudaSuccess) return err;
  if (fa.localSizeBytes > 0) return cudaErrorInvalidConfiguration;  // spills: t = inf
  err = set_smem_limit(reinterpret_cast<const void *>(e->kern), smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(e->kern), e->T, smem);
  if (err != cudaSuccess) return err;
  return per_sm >= cfg.ctas_per_sm ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Dynamic shared memory for a launch that must keep at most `per_sm` CTAs on
// an SM: the kernel's own need, raised so that per_sm + 1 CTAs (each with the
// runtime's reserved shared memory) no longer fit.  The grid is per_sm CTAs
// per SM; without the cap the CTAs of a launch that overlaps the previous one
// (a programmatic dependent, or any concurrent kernel) fill the spare slot of
// the SMs that free up first and pile up there.  FR_XENT_PAD=0 launches with
// the kernel's own need only.
cudaError_t capped_smem(size_t need, int per_sm, size_t *out) {
  *out = need;
  if (const char *e = getenv("FR_XENT_PAD"); e != nullptr && e[0] == '0') return cudaSuccess;
  int dev = 0, per_sm_smem = 0, reserved = 0, max_smem_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  dev)) != cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                  dev)) != cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
      cudaSuccess)
    return e;
  // (per_sm + 1) * (pad + reserved) > per_sm_smem
  const int64_t pad = per_sm_smem / (per_sm + 1) - reserved + 1;
  if (pad > static_cast<int64_t>(need) && pad <= max_smem_optin &&
      static_cast<int64_t>(per_sm) * (pad + reserved) <= per_sm_smem)
    *out = static_cast<size_t>(pad);
  return cudaSuccess;
}

cudaError_t launch_xent_config(const XentConfig &cfg, const void *logits,
                               const int64_t *target, float *loss, float *loss_mean,
                               float *target_logit, int64_t rows, int64_t cols, int64_t ld,
                               int64_t ignore_index, void *workspace, int sm_count,
                               int max_smem_optin, cudaStream_t s) {
  cudaError_t e = xent_config_check(cfg, max_smem_optin);
  if (e != cudaSuccess) return e;
  if (cfg.threads == 32)
    return launch_warp_kernel(warp_kernel<false, false>(cfg.vectors), cfg.ctas_per_sm, logits,
                              target, loss, loss_mean, target_logit, nullptr, rows, cols, ld,
                              ignore_index, workspace, sm_count, s);
  const AsyncEntry *a = async_entry(cfg);
  size_t smem = 0;
  e = capped_smem(static_cast<size_t>(a->NS) * a->U * a->T * 16, cfg.ctas_per_sm, &smem);
  if (e != cudaSuccess) return e;
  if ((e = set_smem_limit(reinterpret_cast<const void *>(a->kern), smem)) != cudaSuccess)
    return e;
  int64_t grid = static_cast<int64_t>(sm_count) * cfg.ctas_per_sm;
  if (grid > rows) grid = rows;
  int64_t *no_argmax = nullptr;
  void *args[] = {&logits, &target, &loss, &target_logit, &no_argmax, &loss_mean, &workspace,
                  &rows, &cols, &ld, &ignore_index};
  return launch_pdl(a->kern, dim3(static_cast<unsigned>(grid)), dim3(a->T), args, smem, s);
}

bool xent_recorded_config(int device, int64_t rows, int64_t cols, int64_t ld, XentConfig *out) {
  std::lock_guard<std::mutex> lock(g_rec_mu);
  for (const Recorded &r : g_recorded)
    if (r.device == device && r.rows == rows && r.cols == cols && r.ld == ld) {
      *out = r.cfg;
      return true;
    }
  return false;
}

void xent_record_config(int device, int64_t rows, int64_t cols, int64_t ld,
                        const XentConfig *cfg) {
  std::lock_guard<std::mutex> lock(g_rec_mu);
  for (size_t i = 0; i < g_recorded.size(); ++i)
    if (g_recorded[i].device == device && g_recorded[i].rows == rows &&
        g_recorded[i].cols == cols && g_recorded[i].ld == ld) {
      if (cfg) g_recorded[i].cfg = *cfg;
      else g_recorded.erase(g_recorded.begin() + static_cast<std::ptrdiff_t>(i));
      return;
    }
  if (cfg) g_recorded.push_back(Recorded{device, rows, cols, ld, *cfg});
}

// The warp-per-row kernel: a persistent grid of at most per_sm_cap 256-thread
// CTAs per SM (and what stays resident), shrunk so that every warp takes the
// same number of rows (8192 rows on 152 SMs x 4 CTAs: 2 rows a warp on 512
// CTAs, 1.5 % faster than 1 or 2 rows on 608), its dynamic shared memory
// padded so that no more than that many CTAs share an SM.
cudaError_t launch_warp_kernel(const void *kern, int per_sm_cap, const void *logits,
                               const int64_t *target, float *loss, float *loss_mean,
                               float *target_logit, int64_t *argmax, int64_t rows, int64_t cols,
                               int64_t ld, int64_t ignore_index, void *workspace, int sm_count,
                               cudaStream_t s) {
  int per_sm = 0;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(kern), 0);
  if (e != cudaSuccess) return e;
  if ((e = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern), kWarpCta, 0)) !=
      cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int resident = per_sm;
  if (per_sm > per_sm_cap) per_sm = per_sm_cap;
  if (per_sm > kMaxCtasPerSm) per_sm = kMaxCtasPerSm;
  constexpr int64_t W = kWarpCta / 32;
  const int64_t warps = static_cast<int64_t>(sm_count) * per_sm * W;
  const int64_t per_warp = (rows + warps - 1) / warps;  // rows a warp takes
  const int64_t grid = (rows + per_warp * W - 1) / (per_warp * W);
  // pad only when the cap is below what the registers allow (the padding's
  // shared-memory carveout cost 3 % when it was not needed)
  size_t smem = 0;
  if (per_sm < resident && (e = capped_smem(0, per_sm, &smem)) != cudaSuccess) return e;
  if ((e = set_smem_limit(reinterpret_cast<const void *>(kern), smem)) != cudaSuccess)
    return e;
  void *args[] = {&logits, &target, &loss, &target_logit, &argmax, &loss_mean, &workspace,
                  &rows, &cols, &ld, &ignore_index};
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kWarpCta), args, smem, s);
}

template <bool ARGMAX, bool F32>
const void *warp_kernel(int nv) {
  if constexpr (ARGMAX) {
    (void)nv;
    return reinterpret_cast<const void *>(&xent_warp<true, F32, 4>);
  } else {
    return nv == 8 ? reinterpret_cast<const void *>(&xent_warp<false, F32, 8>)
                   : reinterpret_cast<const void *>(&xent_warp<false, F32, 4>);
  }
}

cudaError_t launch_xent(const void *logits, bool f32, const int64_t *target, float *loss,
                        float *loss_mean, float *target_logit, int64_t *argmax, int64_t rows,
                        int64_t cols, int64_t ld, int64_t ignore_index, void *workspace,
                        int sm_count, int max_smem_optin, cudaStream_t s) {
  const XentConfig d = xent_default_config();
  // fp32 logits: the warp-per-row kernel at the default point; argmax: the
  // same kernel with 4 vectors a lane (the argmax state leaves no registers
  // for 8), two CTAs per SM
  if (argmax != nullptr)
    return launch_warp_kernel(f32 ? warp_kernel<true, true>(4) : warp_kernel<true, false>(4), 2,
                              logits, target, loss, loss_mean, target_logit, argmax, rows, cols,
                              ld, ignore_index, workspace, sm_count, s);
  if (f32)
    return launch_warp_kernel(warp_kernel<false, true>(d.vectors), d.ctas_per_sm, logits, target,
                              loss, loss_mean, target_logit, argmax, rows, cols, ld, ignore_index,
                              workspace, sm_count, s);
  // the configuration recorded for this shape (fr_xent_tune / _set_config),
  // else the default point
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  XentConfig cfg = d;
  xent_recorded_config(dev, rows, cols, ld, &cfg);
  return launch_xent_config(cfg, logits, target, loss, loss_mean, target_logit, rows, cols, ld,
                            ignore_index, workspace, sm_count, max_smem_optin, s);
}

__global__ void xent_workspace_init_kernel(unsigned long long *ticket) {
  pdl_enter();
  *ticket = kTicketTag;
}

cudaError_t launch_xent_workspace_init(void *workspace, cudaStream_t s) {
  return launch_k(xent_workspace_init_kernel, dim3(1), dim3(1), 0, s, 0,
                  static_cast<unsigned long long *>(workspace));
}

// The mean from parts that ranks holding shards of one batch have summed
// (an all-reduce of the two fp64 values each call leaves in its workspace).
__global__ void xent_mean_from_parts_kernel(const double *__restrict__ parts,
                                            float *__restrict__ loss_mean) {
  pdl_enter();
  *loss_mean = static_cast<float>(parts[0] / parts[1]);
}

cudaError_t launch_xent_mean_from_parts(const void *workspace, float *loss_mean,
                                        cudaStream_t s) {
  const double *parts = reinterpret_cast<const double *>(
      static_cast<const unsigned char *>(workspace) + kPartsOffset);
  return launch_k(xent_mean_from_parts_kernel, dim3(1), dim3(1), 0, s, 0, parts, loss_mean);
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
