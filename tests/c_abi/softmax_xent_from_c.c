/*
 * A plain C caller of libfr.so: no Python, no PyTorch.  Device memory comes
 * from the CUDA runtime, every argument is a pointer or an integer, results
 * come back to the host -- the boundary as a C program sees it.
 *
 * usage: softmax_xent_from_c ROWS COLS X_F32 Y_F32 LOGITS_BF16 TARGET_I64 LOSS_F32
 *   X_F32        rows*cols fp32 input of fr_softmax (raw little-endian file)
 *   Y_F32        written: fr_softmax's output
 *   LOGITS_BF16  rows*cols bf16 bit patterns for fr_xent
 *   TARGET_I64   rows int64 targets (ignore_index -100)
 *   LOSS_F32     written: rows per-row losses, then the mean
 * Exit status 0 on success; any library or CUDA error is printed and exits 1.
 */
#include <cuda_runtime_api.h>
#include <stdio.h>
#include <stdlib.h>

#include "fr.h"

static int fail(const char *what, int code) {
  fprintf(stderr, "%s failed: %d\n", what, code);
  return 1;
}

static void *read_file(const char *path, size_t bytes) {
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

static int write_file(const char *path, const void *p, size_t bytes) {
  FILE *f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : 1;
}

int main(int argc, char **argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s ROWS COLS X_F32 Y_F32 LOGITS_BF16 TARGET_I64 LOSS_F32\n", argv[0]);
    return 2;
  }
  const int64_t rows = atoll(argv[1]), cols = atoll(argv[2]);
  const size_t n = (size_t)rows * (size_t)cols;
  float *x = read_file(argv[3], n * 4);
  uint16_t *lg = read_file(argv[5], n * 2);
  int64_t *tg = read_file(argv[6], (size_t)rows * 8);
  if (!x || !lg || !tg) return fail("reading the inputs", 0);

  void *dx, *dy, *dlg, *dtg, *dloss, *dmean, *dws;
  const size_t ws = fr_workspace_size(FR_OP_XENT, rows, cols, FR_BF16, FR_FORM_AUTO);
  cudaError_t e;
  if ((e = cudaMalloc(&dx, n * 4)) || (e = cudaMalloc(&dy, n * 4)) ||
      (e = cudaMalloc(&dlg, n * 2)) || (e = cudaMalloc(&dtg, (size_t)rows * 8)) ||
      (e = cudaMalloc(&dloss, (size_t)rows * 4)) || (e = cudaMalloc(&dmean, 4)) ||
      (e = cudaMalloc(&dws, ws)))
    return fail("cudaMalloc", (int)e);
  cudaStream_t s;
  if ((e = cudaStreamCreate(&s))) return fail("cudaStreamCreate", (int)e);
  fr_status st = fr_xent_workspace_init(dws, ws, (fr_stream_t)s);  /* once per workspace */
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);
  if ((e = cudaMemcpyAsync(dx, x, n * 4, cudaMemcpyHostToDevice, s)) ||
      (e = cudaMemcpyAsync(dlg, lg, n * 2, cudaMemcpyHostToDevice, s)) ||
      (e = cudaMemcpyAsync(dtg, tg, (size_t)rows * 8, cudaMemcpyHostToDevice, s)))
    return fail("copy in", (int)e);

  st = fr_softmax(dx, dy, rows, cols, cols, cols, FR_F32, FR_FORM_AUTO, (fr_stream_t)s);
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);
  st = fr_xent(dlg, (const int64_t *)dtg, (float *)dloss, (float *)dmean, NULL, NULL, rows, cols,
               cols, -100, FR_BF16, FR_FORM_AUTO, dws, ws, (fr_stream_t)s);
  if (st != FR_OK) return fail(fr_status_string(st), (int)st);

  float *y = malloc(n * 4), *loss = malloc(((size_t)rows + 1) * 4);
  if (!y || !loss) return fail("malloc", 0);
  if ((e = cudaMemcpyAsync(y, dy, n * 4, cudaMemcpyDeviceToHost, s)) ||
      (e = cudaMemcpyAsync(loss, dloss, (size_t)rows * 4, cudaMemcpyDeviceToHost, s)) ||
      (e = cudaMemcpyAsync(loss + rows, dmean, 4, cudaMemcpyDeviceToHost, s)) ||
      (e = cudaStreamSynchronize(s)))
    return fail("copy out", (int)e);
  int32_t dev_err = 0;
  if ((st = fr_check_device_error((fr_stream_t)s, &dev_err)) != FR_OK || dev_err != 0)
    return fail("device error word", dev_err);
  if (write_file(argv[4], y, n * 4) || write_file(argv[7], loss, ((size_t)rows + 1) * 4))
    return fail("writing the outputs", 0);
  cudaFree(dx);
  cudaFree(dy);
  cudaFree(dlg);
  cudaFree(dtg);
  cudaFree(dloss);
  cudaFree(dmean);
  cudaFree(dws);
  cudaStreamDestroy(s);
  free(x);
  free(lg);
  free(tg);
  free(y);
  free(loss);
  return 0;
}
