/*
 * A plain C caller of the rest of libfr.so's compute entry points: no Python,
 * no PyTorch.  Device memory and the workspace come from the CUDA runtime and
 * are sized by fr_workspace_size, as a C program would size them.
 *
 * usage: reductions_from_c RAS_ROWS RAS_COLS LN_ROWS LN_COLS L2_ROWS L2_COLS DIR
 * Reads from DIR (raw little-endian files):
 *   a.bin, b.bin        RAS_ROWS*RAS_COLS fp32: fr_reduce_relu_add_sum, split form
 *   x.bin               LN_ROWS*LN_COLS bf16 bit patterns: fr_layernorm
 *   gamma.bin, beta.bin LN_COLS fp32
 *   s.bin               L2_ROWS*L2_COLS fp32: fr_reduce_sumsq with the sqrt epilogue
 * Writes to DIR: ras.bin (fp32 [RAS_ROWS]), ln_y.bin (bf16), ln_mean.bin,
 * ln_rstd.bin (fp32 [LN_ROWS]), l2.bin (fp32 [L2_ROWS]).
 * Then runs fr_xent on 4 rows whose third target lies outside [0, cols) and
 * reads the device error word.  Prints one line:
 *   ras_form=F ln_form=F l2_form=F bad_target_status=S bad_target_code=C clear_status=S
 * Exit status 0 on success; any unexpected library or CUDA error exits 1.
 */
#include <cuda_runtime_api.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fr.h"

static int fail(const char *what, int code) {
  fprintf(stderr, "%s failed: %d\n", what, code);
  return 1;
}

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  void *p = malloc(bytes);
  size_t got = p ? fread(p, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int write_file(const char *dir, const char *name, const void *p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : 1;
}

/* Host buffer -> new device buffer; NULL on failure. */
static void *to_device(const void *h, size_t bytes, cudaStream_t s) {
  void *d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  if (cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return NULL;
  return d;
}

static int from_device(const char *dir, const char *name, const void *d, size_t bytes,
                       cudaStream_t s) {
  void *h = malloc(bytes);
  if (!h) return 1;
  int bad = cudaMemcpyAsync(h, d, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess || write_file(dir, name, h, bytes);
  free(h);
  return bad;
}

int main(int argc, char **argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s RAS_ROWS RAS_COLS LN_ROWS LN_COLS L2_ROWS L2_COLS DIR\n", argv[0]);
    return 2;
  }
  const int64_t rr = atoll(argv[1]), rc = atoll(argv[2]), lr = atoll(argv[3]),
                lc = atoll(argv[4]), sr = atoll(argv[5]), sc = atoll(argv[6]);
  const char *dir = argv[7];
  const size_t nr = (size_t)rr * (size_t)rc, nl = (size_t)lr * (size_t)lc,
               ns = (size_t)sr * (size_t)sc;
  float *a = read_file(dir, "a.bin", nr * 4), *b = read_file(dir, "b.bin", nr * 4);
  uint16_t *x = read_file(dir, "x.bin", nl * 2);
  float *g = read_file(dir, "gamma.bin", (size_t)lc * 4), *be = read_file(dir, "beta.bin", (size_t)lc * 4);
  float *sq = read_file(dir, "s.bin", ns * 4);
  if (!a || !b || !x || !g || !be || !sq) return fail("reading the inputs", 0);

  cudaStream_t s;
  cudaError_t e;
  if ((e = cudaStreamCreate(&s))) return fail("cudaStreamCreate", (int)e);
  fr_status st;

  /* Example 1.1, split form: the caller sizes and owns the workspace. */
  void *da = to_device(a, nr * 4, s), *db = to_device(b, nr * 4, s), *dras = NULL, *dws = NULL;
  const size_t ws = fr_workspace_size(FR_OP_RELU_ADD_SUM, rr, rc, FR_F32, FR_FORM_SPLIT);
  if (!da || !db || ws == 0 || cudaMalloc(&dras, (size_t)rr * 4) || cudaMalloc(&dws, ws))
    return fail("relu_add_sum buffers", 0);
  st = fr_reduce_relu_add_sum(da, db, (float *)dras, rr, rc, rc, rc, FR_F32, 2.0f, FR_FORM_SPLIT,
                              dws, ws, (fr_stream_t)s);
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);
  const int ras_form = (int)fr_last_form();
  /* one byte short of the workspace: refused before anything is enqueued */
  st = fr_reduce_relu_add_sum(da, db, (float *)dras, rr, rc, rc, rc, FR_F32, 2.0f, FR_FORM_SPLIT,
                              dws, ws - 1, (fr_stream_t)s);
  if (st != FR_ERR_WORKSPACE_TOO_SMALL) return fail("short workspace not refused", (int)st);
  if (from_device(dir, "ras.bin", dras, (size_t)rr * 4, s)) return fail("ras out", 0);

  /* LayerNorm, bf16 rows with fp32 gamma/beta, mean and rstd. */
  void *dx = to_device(x, nl * 2, s), *dg = to_device(g, (size_t)lc * 4, s),
       *dbe = to_device(be, (size_t)lc * 4, s), *dy = NULL, *dm = NULL, *dr = NULL;
  if (!dx || !dg || !dbe || cudaMalloc(&dy, nl * 2) || cudaMalloc(&dm, (size_t)lr * 4) ||
      cudaMalloc(&dr, (size_t)lr * 4))
    return fail("layernorm buffers", 0);
  st = fr_layernorm(dx, (const float *)dg, (const float *)dbe, dy, (float *)dm, (float *)dr, lr,
                    lc, lc, lc, 1e-5f, FR_BF16, FR_FORM_AUTO, (fr_stream_t)s);
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);
  const int ln_form = (int)fr_last_form();
  if (from_device(dir, "ln_y.bin", dy, nl * 2, s) ||
      from_device(dir, "ln_mean.bin", dm, (size_t)lr * 4, s) ||
      from_device(dir, "ln_rstd.bin", dr, (size_t)lr * 4, s))
    return fail("layernorm out", 0);

  /* Row L2 norm (Example 6.2's sum of squares with the sqrt epilogue). */
  void *ds = to_device(sq, ns * 4, s), *dl2 = NULL, *dws2 = NULL;
  const size_t ws2 = fr_workspace_size(FR_OP_SUMSQ, sr, sc, FR_F32, FR_FORM_AUTO);
  if (!ds || cudaMalloc(&dl2, (size_t)sr * 4) || (ws2 && cudaMalloc(&dws2, ws2)))
    return fail("sumsq buffers", 0);
  st = fr_reduce_sumsq(ds, (float *)dl2, sr, sc, sc, FR_F32, FR_EPI_SQRT, FR_FORM_AUTO, dws2, ws2,
                       (fr_stream_t)s);
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);
  const int l2_form = (int)fr_last_form();
  if (from_device(dir, "l2.bin", dl2, (size_t)sr * 4, s)) return fail("l2 out", 0);

  /* A target outside [0, cols): the call succeeds, the device error word
   * records FR_DEVERR_BAD_TARGET, and reading it clears it. */
  const int64_t xr = 4, xc = 100;
  uint16_t zeros[4 * 100];
  memset(zeros, 0, sizeof zeros);
  const int64_t tg[4] = {0, 5, 100, -100};
  void *dlg = to_device(zeros, sizeof zeros, s), *dtg = to_device(tg, sizeof tg, s), *dloss = NULL;
  if (!dlg || !dtg || cudaMalloc(&dloss, (size_t)xr * 4)) return fail("xent buffers", 0);
  st = fr_xent(dlg, (const int64_t *)dtg, (float *)dloss, NULL, NULL, NULL, xr, xc, xc, -100,
               FR_BF16, FR_FORM_AUTO, NULL, 0, (fr_stream_t)s);
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);
  int32_t code = -1;
  const fr_status bad = fr_check_device_error((fr_stream_t)s, &code);
  int32_t code2 = -1;
  const fr_status clear = fr_check_device_error((fr_stream_t)s, &code2);
  if (code2 != 0) return fail("error word not cleared", code2);

  printf("ras_form=%d ln_form=%d l2_form=%d bad_target_status=%d bad_target_code=%d "
         "clear_status=%d\n",
         ras_form, ln_form, l2_form, (int)bad, (int)code, (int)clear);
  void *bufs[] = {da, db, dras, dws, dx, dg, dbe, dy, dm, dr, ds, dl2, dws2, dlg, dtg, dloss};
  for (size_t i = 0; i < sizeof bufs / sizeof bufs[0]; ++i) cudaFree(bufs[i]);
  cudaStreamDestroy(s);
  free(a);
  free(b);
  free(x);
  free(g);
  free(be);
  free(sq);
  return 0;
}
