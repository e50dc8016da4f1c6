/*
 * Seeded synthetic inputs for the fused row-reduction workloads.
 *
 * This module is shared by the CPU oracle and the CUDA path: both sides are fed
 * the very same bytes.  It therefore holds none of the method's arithmetic --
 * only counter-based random numbers and value casts:
 *
 *   - SplitMix64 (S. Vigna, "Further scramblings of Marsaglia's xorshift
 *     generators", 2015; the public-domain splitmix64.c).  The i-th output of a
 *     stream whose state starts at s0 is mix(s0 + (i+1)*GAMMA), so every element
 *     is generated from its own index and the result does not depend on how the
 *     work is split over threads.
 *   - uniforms from the top 24 (fp32 use) or 53 (Box-Muller) bits of an output;
 *   - normals by the Box-Muller transform in fp64 (one pair of uniforms per
 *     element, the sine branch unused);
 *   - fp64 -> fp32 by the C cast (round to nearest even), fp32 -> bf16 by
 *     round to nearest even on the bit pattern.
 *
 * Plain C11, no architecture-specific code: it gives identical bytes on x86_64
 * and aarch64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* i-th output (0-based) of the SplitMix64 stream with initial state s0. */
static inline uint64_t sm64_at(uint64_t s0, uint64_t i) {
  return sm64_mix(s0 + (i + 1) * SM64_GAMMA);
}

/* Initial state of sub-stream `stream` of a seed: two scrambles keep streams of
 * nearby seeds and nearby stream ids unrelated. */
uint64_t synth_stream_state(uint64_t seed, uint64_t stream) {
  return sm64_mix(sm64_mix(seed ^ 0x5DEECE66DULL) + stream * SM64_GAMMA);
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i) {
  return sm64_at(synth_stream_state(seed, stream), i);
}

/* [0, 1) with 24 random bits: exactly representable in fp32. */
static inline double u24(uint64_t z) { return (double)(z >> 40) * (1.0 / 16777216.0); }
/* (0, 1] with 53 random bits: safe under log(). */
static inline double u53_open0(uint64_t z) {
  return (double)((z >> 11) + 1) * (1.0 / 9007199254740992.0);
}
/* [0, 1) with 53 random bits. */
static inline double u53(uint64_t z) { return (double)(z >> 11) * (1.0 / 9007199254740992.0); }

static inline double normal_at(uint64_t s0, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double r1 = u53_open0(sm64_at(s0, 2 * i));
  double r2 = u53(sm64_at(s0, 2 * i + 1));
  return sqrt(-2.0 * log(r1)) * cos(two_pi * r2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ---- threaded fill over [0, n) ---------------------------------------- */

enum { K_UNIFORM_F32, K_NORMAL_F32, K_NORMAL_BF16 };

typedef struct {
  int kind;
  void *out;
  int64_t begin, end;
  uint64_t s0, first; /* output i holds stream element first + i */
  double p0, p1;
} fill_job;

static void *fill_worker(void *arg) {
  fill_job *j = (fill_job *)arg;
  if (j->kind == K_UNIFORM_F32) {
    float *o = (float *)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = (float)(j->p0 + (j->p1 - j->p0) * u24(sm64_at(j->s0, j->first + (uint64_t)i)));
  } else if (j->kind == K_NORMAL_F32) {
    float *o = (float *)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = (float)(j->p0 + j->p1 * normal_at(j->s0, j->first + (uint64_t)i));
  } else {
    uint16_t *o = (uint16_t *)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = f32_to_bf16_rne((float)(j->p0 + j->p1 * normal_at(j->s0, j->first + (uint64_t)i)));
  }
  return NULL;
}

static void fill(int kind, void *out, int64_t n, uint64_t seed, uint64_t stream, uint64_t first,
                 double p0, double p1) {
  enum { MAX_T = 64 };
  long nc = sysconf(_SC_NPROCESSORS_ONLN);
  int t = (int)(nc < 1 ? 1 : (nc > MAX_T ? MAX_T : nc));
  if (n < (1 << 20)) t = 1;
  uint64_t s0 = synth_stream_state(seed, stream);
  fill_job jobs[MAX_T];
  pthread_t th[MAX_T];
  int64_t per = (n + t - 1) / t;
  for (int k = 0; k < t; ++k) {
    int64_t b = (int64_t)k * per, e = b + per;
    if (b > n) b = n;
    if (e > n) e = n;
    jobs[k] = (fill_job){kind, out, b, e, s0, first, p0, p1};
  }
  int started[MAX_T] = {0};
  for (int k = 1; k < t; ++k) {
    started[k] = pthread_create(&th[k], NULL, fill_worker, &jobs[k]) == 0;
    if (!started[k]) fill_worker(&jobs[k]); /* no thread: run it here */
  }
  fill_worker(&jobs[0]);
  for (int k = 1; k < t; ++k)
    if (started[k]) pthread_join(th[k], NULL);
}

/* n fp32 values uniform in [lo, hi): elements first .. first + n - 1 of the
 * stream (first = 0: the start; a later first gives a slice of a larger array). */
void synth_uniform_f32_at(float *out, int64_t n, uint64_t seed, uint64_t stream, uint64_t first,
                          double lo, double hi) {
  fill(K_UNIFORM_F32, out, n, seed, stream, first, lo, hi);
}
void synth_uniform_f32(float *out, int64_t n, uint64_t seed, uint64_t stream, double lo,
                       double hi) {
  synth_uniform_f32_at(out, n, seed, stream, 0, lo, hi);
}

/* n fp32 values mean + std * N(0,1) (elements first .. of the stream). */
void synth_normal_f32_at(float *out, int64_t n, uint64_t seed, uint64_t stream, uint64_t first,
                         double mean, double std) {
  fill(K_NORMAL_F32, out, n, seed, stream, first, mean, std);
}
void synth_normal_f32(float *out, int64_t n, uint64_t seed, uint64_t stream, double mean,
                      double std) {
  synth_normal_f32_at(out, n, seed, stream, 0, mean, std);
}

/* n bf16 bit patterns of mean + std * N(0,1) (fp64 -> fp32 -> bf16, each RNE). */
void synth_normal_bf16_at(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream,
                          uint64_t first, double mean, double std) {
  fill(K_NORMAL_BF16, out, n, seed, stream, first, mean, std);
}
void synth_normal_bf16(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream, double mean,
                       double std) {
  synth_normal_bf16_at(out, n, seed, stream, 0, mean, std);
}

/* n class indices uniform in [0, V) (Lemire's multiply-shift), then exactly
 * n_ignore distinct positions, chosen by a seeded partial Fisher-Yates shuffle,
 * are overwritten with ignore_index.  Returns 0, or -1 on bad arguments. */
int synth_targets(int64_t *out, int64_t n, uint64_t seed, uint64_t stream, int64_t V,
                  int64_t n_ignore, int64_t ignore_index) {
  if (n < 0 || V <= 0 || n_ignore < 0 || n_ignore > n) return -1;
  uint64_t s0 = synth_stream_state(seed, stream);
  for (int64_t i = 0; i < n; ++i) {
    unsigned __int128 p = (unsigned __int128)sm64_at(s0, (uint64_t)i) * (uint64_t)V;
    out[i] = (int64_t)(p >> 64);
  }
  if (n_ignore == 0) return 0;
  int64_t *idx = (int64_t *)malloc((size_t)n * sizeof(int64_t));
  if (!idx) return -1;
  for (int64_t i = 0; i < n; ++i) idx[i] = i;
  uint64_t s1 = synth_stream_state(seed, stream + 0x1000);
  for (int64_t k = 0; k < n_ignore; ++k) {
    unsigned __int128 p = (unsigned __int128)sm64_at(s1, (uint64_t)k) * (uint64_t)(n - k);
    int64_t j = k + (int64_t)(p >> 64);
    int64_t tmp = idx[k];
    idx[k] = idx[j];
    idx[j] = tmp;
    out[idx[k]] = ignore_index;
  }
  free(idx);
  return 0;
}

/* count integers, each uniform in [0, bound). */
void synth_indices(int64_t *out, int64_t count, uint64_t seed, uint64_t stream, int64_t bound) {
  uint64_t s0 = synth_stream_state(seed, stream);
  for (int64_t i = 0; i < count; ++i) {
    unsigned __int128 p = (unsigned __int128)sm64_at(s0, (uint64_t)i) * (uint64_t)bound;
    out[i] = (int64_t)(p >> 64);
  }
}
