// Host-side launchers of the row-reduction kernels.  Only fr_api.cu calls
// these; each returns the launch's cudaError_t and never synchronises.
#pragma once

#include <cstddef>
#include <cstdint>
#include <functional>
#include <cuda_runtime.h>

namespace fr {

// Properties of the current device the launch shapes depend on.
struct DevInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  int max_smem_optin;  // bytes of shared memory one CTA may opt in to
};
cudaError_t current_device_info(DevInfo *out);
// Records the form of a call that enqueued its kernels (what fr_last_form
// returns on this host thread).
void set_last_form(int form);

// ---- Example 1.1: out[x] = sum_r scale * relu(a + b) ------------------------

// Largest row (elements) the persistent form holds in one pass.
int64_t ras_persistent_max_cols(bool bf16 = false);
// Segments per row of the split form for this shape (fixed per device model).
int ras_split_segments(int64_t rows, int64_t cols, int sm_count);
size_t ras_split_workspace(int64_t rows, int64_t cols, int sm_count);

// a, b: fp32, or bf16 bit patterns when bf16 (widened exactly before the sum)
cudaError_t launch_ras_persistent(const void *a, const void *b, float *out, int64_t rows,
                                  int64_t cols, int64_t lda, int64_t ldb, float scale, bool bf16,
                                  bool vec, cudaStream_t s);
cudaError_t launch_ras_looped(const void *a, const void *b, float *out, int64_t rows,
                              int64_t cols, int64_t lda, int64_t ldb, float scale, bool bf16,
                              bool vec, cudaStream_t s);
cudaError_t launch_ras_split(const void *a, const void *b, float *out, int64_t rows,
                             int64_t cols, int64_t lda, int64_t ldb, float scale, bool bf16,
                             bool vec, double *partials, int segments, cudaStream_t s);

// ---- Example 6.2 and its L2-norm epilogue: out[x] = (sqrt) sum_r x^2 ------
// Same forms, segment rule and workspace as above.
cudaError_t launch_sumsq_persistent(const float *x, float *out, int64_t rows, int64_t cols,
                                    int64_t ldx, bool sqrt_out, cudaStream_t s);
cudaError_t launch_sumsq_looped(const float *x, float *out, int64_t rows, int64_t cols,
                                int64_t ldx, bool sqrt_out, cudaStream_t s);
cudaError_t launch_sumsq_split(const float *x, float *out, int64_t rows, int64_t cols,
                               int64_t ldx, bool sqrt_out, double *partials, int segments,
                               cudaStream_t s);

// ---- softmax ---------------------------------------------------------------

int64_t softmax_persistent_max_cols(bool vec);
// Split form, the row staged in shared memory: a cluster of 2-8 CTAs per row
// (any offsets of x and y; es = 4 for fp32, 2 for bf16 rows), up to
// softmax_stage_split_max_cols(es) columns.
int64_t softmax_stage_split_max_cols(int es);
cudaError_t launch_softmax_split_staged(const void *x, void *y, int64_t rows, int64_t cols,
                                        int64_t ldx, int64_t ldy, int es, cudaStream_t s);
// Split form for rows in phase (x and y at the same offset within a 32-byte
// sector), any length up to 2^31 - 1 columns: a cluster of 4, 8 or 16 CTAs
// per row, each streaming its run of the row twice (the second read from L2).
cudaError_t launch_softmax_split_looped(const void *x, void *y, int64_t rows, int64_t cols,
                                        int64_t ldx, int64_t ldy, int es, int sm_count,
                                        cudaStream_t s);
// fp32 rows of at most 1024 columns in host memory, x and y in phase, ld =
// cols: the persistent form over a small grid (a quarter of the SMs' CTAs).
cudaError_t launch_softmax_host_rows(const float *x, float *y, int64_t rows, int64_t cols,
                                     int sm_count, cudaStream_t s);
cudaError_t launch_softmax_persistent(const float *x, float *y, int64_t rows, int64_t cols,
                                      int64_t ldx, int64_t ldy, bool vec, cudaStream_t s);
// Persistent warp-per-row form with a per-warp cp.async ring (16-byte aligned
// x and y rows, cols <= 1024).
bool softmax_async_ok(int64_t cols, bool aligned16);
cudaError_t launch_softmax_async(const float *x, float *y, int64_t rows, int64_t cols,
                                 int64_t ldx, int64_t ldy, int sm_count, cudaStream_t s);
cudaError_t launch_softmax_looped(const float *x, float *y, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, bool vec, int sm_count,
                                  cudaStream_t s);
// Split form: a thread-block cluster of up to 8 CTAs per row exchanging the
// (m, d) pairs through distributed shared memory (x and y in phase, rows of
// 1025 .. 262144 elements).
int64_t softmax_split_max_cols();
cudaError_t launch_softmax_split(const float *x, float *y, int64_t rows, int64_t cols,
                                 int64_t ldx, int64_t ldy, cudaStream_t s);

// bf16 rows (x and y bf16, fp32 arithmetic): persistent up to 32768 columns
// (a warp per row up to 2048; then a CTA per row, in phase the row in
// registers, out of phase staged in shared memory).
int64_t softmax_bf16_persistent_max_cols(bool vec);
// bf16 rows of at most 2048 columns in host memory, x and y in phase, ld =
// cols: the persistent form over a small grid (a quarter of the SMs' CTAs).
cudaError_t launch_softmax_bf16_host_rows(const uint16_t *x, uint16_t *y, int64_t rows,
                                          int64_t cols, int sm_count, cudaStream_t s);
// Split form of the bf16 softmax: a thread-block cluster per row (rows in
// phase, 2049 .. softmax_bf16_split_max_cols() columns).
int64_t softmax_bf16_split_max_cols();
cudaError_t launch_softmax_bf16_split(const uint16_t *x, uint16_t *y, int64_t rows, int64_t cols,
                                      int64_t ldx, int64_t ldy, cudaStream_t s);
cudaError_t launch_softmax_bf16_persistent(const uint16_t *x, uint16_t *y, int64_t rows,
                                           int64_t cols, int64_t ldx, int64_t ldy, bool vec,
                                           int sm_count, cudaStream_t s);
cudaError_t launch_softmax_bf16_looped(const uint16_t *x, uint16_t *y, int64_t rows,
                                       int64_t cols, int64_t ldx, int64_t ldy, bool vec,
                                       int sm_count, cudaStream_t s);

// ---- LayerNorm -------------------------------------------------------------

// True when the persistent (register-resident) form can hold this row.
bool layernorm_persistent_ok(int64_t cols, bool vec);
// The looped form with bulk-copy staging: 32-byte aligned rows and
// gamma/beta, cols % 16 == 0, the row fits one CTA's shared memory.
// The cluster form: rows split over a thread-block cluster, gamma/beta held
// in registers; 32-byte aligned rows, 16-byte aligned gamma/beta,
// cols % (16 * cluster) == 0 and at most 32768 columns (8 CTAs x 256 threads
// x 16 columns).
bool layernorm_cluster_ok(int64_t cols, bool aligned);
// The equal-count cluster kernel: cols = C x T x 32 (T a power of two in
// 64 .. 512 threads, or 96, 160, 192, 224; C in 1, 2, 4, 8 CTAs), aligned as
// above.  Returns the CTA size T it takes for a row length (0: none).
int layernorm_cluster_full_threads(int64_t cols, bool aligned);
cudaError_t launch_layernorm_cluster(const uint16_t *x, const float *gamma, const float *beta,
                                     uint16_t *y, float *mean, float *rstd, int64_t rows,
                                     int64_t cols, int64_t ldx, int64_t ldy, float eps,
                                     cudaStream_t s);
// Row groups: gamma/beta in shared memory, each row in the registers of a
// group of warps (cols % 8 == 0 and at most 16384, 16-byte aligned rows and
// gamma/beta, 8 * cols bytes of shared memory).
bool layernorm_rows_ok(int64_t cols, bool aligned16, int max_smem_optin);
cudaError_t launch_layernorm_rows(const uint16_t *x, const float *gamma, const float *beta,
                                  uint16_t *y, float *mean, float *rstd, int64_t rows,
                                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int sm_count,
                                  cudaStream_t s);
bool layernorm_ring_ok(int64_t cols, bool vec, int max_smem_optin);
size_t layernorm_ring_smem(int64_t cols, int nbuf);
cudaError_t launch_layernorm_ring(const uint16_t *x, const float *gamma, const float *beta,
                                  uint16_t *y, float *mean, float *rstd, int64_t rows,
                                  int64_t cols, int64_t ldx, int64_t ldy, float eps, int sm_count,
                                  int max_smem_optin, cudaStream_t s);
cudaError_t launch_layernorm_persistent(const uint16_t *x, const float *gamma,
                                        const float *beta, uint16_t *y, float *mean,
                                        float *rstd, int64_t rows, int64_t cols, int64_t ldx,
                                        int64_t ldy, float eps, cudaStream_t s);
cudaError_t launch_layernorm_looped(const uint16_t *x, const float *gamma, const float *beta,
                                    uint16_t *y, float *mean, float *rstd, int64_t rows,
                                    int64_t cols, int64_t ldx, int64_t ldy, float eps,
                                    bool vec, int sm_count, int max_smem_optin,
                                    cudaStream_t s);

// ---- rows held in host memory ------------------------------------------------

// Computes chunk rows x [rows, cols] (contiguous, device) -> y on stream s.
using RowKernel = std::function<cudaError_t(const void *x, void *y, int64_t rows,
                                            cudaStream_t s)>;
// Device staging bytes for chunks of chunk_rows rows (three slots each way).
size_t host_pipeline_workspace(int64_t cols, int64_t esize_in, int64_t esize_out,
                               int64_t chunk_rows);
// Copies x_host in, runs `kernel` chunk by chunk and copies y out, copies and
// kernels overlapping on the device's internal streams; ordered after the
// caller's earlier work on `caller`, which resumes after the last copy out.
cudaError_t host_pipeline_run(const void *x_host, void *y_host, int64_t rows, int64_t cols,
                              int64_t esize_in, int64_t esize_out, int64_t chunk_rows,
                              void *workspace, cudaStream_t caller, const RowKernel &kernel);

// ---- launch-configuration search (Algorithm 9.2) -----------------------------

struct CdResult {
  int acceptances;  // moves accepted
  int evaluations;  // distinct configurations measured
  double t;         // cost of the returned configuration
};
// Coordinate descent over log2 parameters c[i] in [lo[i], hi[i]]; c is updated
// in place.  A start of infinite cost returns at once (t = inf).
CdResult coordinate_descent(int p, const int *lo, const int *hi, int *c, double eps,
                            const std::function<double(const int *)> &cost);

// ---- cross entropy ---------------------------------------------------------

// One point of the cross-entropy kernel's configuration space.
struct XentConfig {
  int threads;      // per CTA: 128 .. 1024
  int vectors;      // 16-byte copies per thread per item: 1 .. 8
  int stages;       // items in the per-thread ring: 2 .. 8
  int ctas_per_sm;  // CTAs per SM in the persistent grid: 1 .. 16
};
// The configuration used when none was recorded for a shape.
XentConfig xent_default_config();
// cudaSuccess when cfg is in the space and can run on this device (shared
// memory, residency of ctas_per_sm CTAs, no register spills);
// cudaErrorInvalidValue outside the space, cudaErrorInvalidConfiguration when
// it cannot run.
cudaError_t xent_config_check(const XentConfig &cfg, int max_smem_optin);
// The configuration recorded for (device, rows, cols, ld), if any; recording
// nullptr forgets it.
bool xent_recorded_config(int device, int64_t rows, int64_t cols, int64_t ld, XentConfig *out);
void xent_record_config(int device, int64_t rows, int64_t cols, int64_t ld,
                        const XentConfig *cfg);
// The non-argmax kernel with configuration cfg.
cudaError_t launch_xent_config(const XentConfig &cfg, const void *logits,
                               const int64_t *target, float *loss, float *loss_mean,
                               float *target_logit, int64_t rows, int64_t cols, int64_t ld,
                               int64_t ignore_index, void *workspace, int sm_count,
                               int max_smem_optin, cudaStream_t s);

size_t xent_workspace(int64_t rows, int sm_count);
cudaError_t launch_xent_mean_from_parts(const void *workspace, float *loss_mean, cudaStream_t s);
cudaError_t launch_xent_workspace_init(void *workspace, cudaStream_t s);
// f32: logits are fp32 (else bf16 bit patterns)
cudaError_t launch_xent(const void *logits, bool f32, const int64_t *target, float *loss,
                        float *loss_mean, float *target_logit, int64_t *argmax, int64_t rows,
                        int64_t cols, int64_t ld, int64_t ignore_index, void *workspace,
                        int sm_count, int max_smem_optin, cudaStream_t s);
// Device address of the current device's error word (kernels record
// FR_DEVERR_* codes there with atomicCAS; the first code wins).
cudaError_t device_error_word(int **out);
// Reads and clears the device error word of the current device (synchronises s).
cudaError_t device_error_read_and_clear(cudaStream_t s, int *code);

}  // namespace fr
