/*
 * fr.h -- C ABI of the GB300 (sm_103a) fused pointwise + row-reduction library.
 *
 * Every entry point takes plain pointers and sizes; no framework types cross
 * this boundary.  Conventions shared by all calls:
 *
 *   Layout.    A matrix is `rows` rows of `cols` elements, row-major, the
 *              reduction running along the contiguous dimension (the INNER
 *              reduction of "Stax (4): GPU Codegen and Dynamic Shapes", section
 *              9.4).  `ld*` is the distance between row starts in elements
 *              (ld >= cols).  Base pointers need only the element's natural
 *              alignment; 16-byte aligned rows take the vectorised path, others
 *              a scalar or head/tail-peeled path (same results).
 *   Memory.    Every pointer is DEVICE memory owned by the caller (inputs,
 *              outputs and workspace).  The library allocates nothing.
 *   Streams.   All work is enqueued on `stream` (a cudaStream_t; NULL = the
 *              legacy default stream) and the call returns without
 *              synchronising.  Kernels of one call are ordered by the stream
 *              alone, as the generated wrapper of section 9.7 orders its two
 *              launches.
 *   Errors.    The return value reports argument validation and launch errors
 *              only; on any non-FR_OK return nothing was enqueued.  Errors that
 *              depend on device data (an out-of-range target) are recorded in
 *              a device-side error word that fr_check_device_error() reads;
 *              kernels never trap.
 *   Forms.     `form` selects the reduction form of section 9.4: persistent
 *              (a row held on chip in one pass), looped (a row streamed in
 *              chunks), split (few long rows: two-stage cross-CTA reduction).
 *              FR_FORM_AUTO picks one from the shape using rules measured on
 *              GB300; a form that cannot handle the shape returns
 *              FR_ERR_UNSUPPORTED_FORM.  fr_last_form() reports the choice.
 *   Devices.   Calls run on the caller's current CUDA device.
 */
#ifndef FR_H_
#define FR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *fr_stream_t; /* == cudaStream_t */

typedef enum {
  FR_OK = 0,
  FR_ERR_INVALID_ARG = 1,        /* null pointer, rows/cols <= 0, ld < cols, size overflow */
  FR_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype not offered by this call */
  FR_ERR_UNSUPPORTED_FORM = 3,   /* forced form cannot handle this shape */
  FR_ERR_MISALIGNED = 4,         /* pointer not aligned to its element size */
  FR_ERR_WORKSPACE_TOO_SMALL = 5,/* workspace_bytes < fr_workspace_size(...) */
  FR_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
  FR_ERR_DEVICE_DATA = 7,        /* device data error recorded (see fr_check_device_error) */
  FR_ERR_NO_DEVICE = 8           /* no usable CUDA device / wrong architecture */
} fr_status;

typedef enum { FR_F32 = 0, FR_BF16 = 1 } fr_dtype;

typedef enum {
  FR_FORM_AUTO = 0,
  FR_FORM_PERSISTENT = 1,
  FR_FORM_LOOPED = 2,
  FR_FORM_SPLIT = 3
} fr_form;

typedef enum {
  FR_OP_RELU_ADD_SUM = 0,
  FR_OP_SOFTMAX = 1,
  FR_OP_LAYERNORM = 2,
  FR_OP_XENT = 3,
  FR_OP_SUMSQ = 4
} fr_op;

/* Epilogue applied to a row sum after the reduction. */
typedef enum {
  FR_EPI_SUM = 0, /* the sum itself */
  FR_EPI_SQRT = 1 /* its square root (taken in fp64, rounded once to fp32) */
} fr_epilogue;

/* Device error codes written by kernels (read by fr_check_device_error). */
#define FR_DEVERR_NONE 0
#define FR_DEVERR_BAD_TARGET 1 /* a target outside [0, cols) and != ignore_index */
#define FR_DEVERR_TIMEOUT 2    /* an asynchronous copy did not complete within its
                                  time budget; the kernel gave up and returned */
#define FR_DEVERR_BAD_WORKSPACE 3 /* fr_xent's workspace was not prepared by
                                    fr_xent_workspace_init (the mean is not written) */

/* Library version (major*10000 + minor*100 + patch). */
int fr_version(void);

/* Human-readable name of a status code (static storage). */
const char *fr_status_string(fr_status status);

/* The form chosen by the most recent successful call on this host thread. */
fr_form fr_last_form(void);

/*
 * The form FR_FORM_AUTO picks for `op` on rows x cols of `dtype` on a device
 * with `sm_count` SMs, for rows whose inputs and outputs share their offset
 * modulo 32 bytes (contiguous tensors of one shape do; other layouts may take
 * the looped form instead).  LayerNorm assumes sm_103's 227 KiB of opt-in
 * shared memory.  A host-side query: no device is touched.  FR_FORM_AUTO (0)
 * for arguments no call accepts.  The rules are measured crossovers of the
 * forms on GB300 (Stax (4), section 9.6, Algorithm 9.1: the fastest measured
 * candidate per shape, recorded).
 */
fr_form fr_auto_form(fr_op op, fr_dtype dtype, int64_t rows, int64_t cols, int32_t sm_count);

/*
 * Bytes of device workspace that `op` needs for this shape and form
 * (0 when none).  FR_FORM_AUTO reports the need of the form AUTO will pick.
 * The workspace must be 16-byte aligned; its contents on entry are ignored.
 */
size_t fr_workspace_size(fr_op op, int64_t rows, int64_t cols, fr_dtype dtype, fr_form form);

/*
 * out[x] = sum_{r < cols} scale * relu(a[x*lda + r] + b[x*ldb + r])
 *
 * Example 1.1 of "Stax (4): GPU Codegen and Dynamic Shapes", section 9.2,
 * Listing 9.1 (there with scale = 2): the two loads are added in fp32, relu is
 * maximum(0, v) with NaN propagation (a NaN input makes its row's sum NaN) and
 * the product is summed along the row with fp32 accumulators over short runs
 * and an fp64 combine across threads and CTAs.  Section 9.4 gives the forms:
 * persistent and looped (one warp or CTA per row), split (section 9.4 (3):
 * rows too few and too long -- stage 1 writes per-segment partials to the
 * workspace, stage 2 sums them in a fixed order; results are bitwise
 * run-to-run deterministic for a given shape).
 *
 *   a, b       [rows, lda] / [rows, ldb] device inputs of `dtype` (read only)
 *   out        fp32 [rows] device output
 *   dtype      FR_F32, or FR_BF16 (bit patterns, widened exactly to fp32
 *              before the sum; the persistent form then holds rows of up
 *              to 2048 columns instead of 1024)
 *   workspace  device scratch of fr_workspace_size(FR_OP_RELU_ADD_SUM, ...)
 *              bytes (only the split form uses it; may be NULL otherwise)
 */
fr_status fr_reduce_relu_add_sum(const void *a, const void *b, float *out, int64_t rows,
                                 int64_t cols, int64_t lda, int64_t ldb, fr_dtype dtype,
                                 float scale, fr_form form, void *workspace,
                                 size_t workspace_bytes, fr_stream_t stream);

/*
 * out[x] = sum_{r < cols} x[x*ldx + r]^2            (epilogue FR_EPI_SUM)
 * out[x] = sqrt(sum_{r < cols} x[x*ldx + r]^2)      (epilogue FR_EPI_SQRT)
 *
 * The sum of squares is Example 6.2 of "Stax (4): GPU Codegen and Dynamic
 * Shapes" (Listing 9.4: each element squared in fp32, summed along the row;
 * there [64, 16384] split into two segments per row); the square-root epilogue
 * is the row-wise L2 norm of Exercise 1 in "CMU 15-779 Lecture 8: ML Compilers
 * Part 1, Tile-based DSLs", section 12 (masked lanes contribute 0).  The same
 * kernels and forms as fr_reduce_relu_add_sum with a one-input prologue: fp32
 * accumulators over short runs, fp64 combine, the split form's partials in
 * the workspace summed in a fixed order (bitwise run-to-run deterministic);
 * the square root is taken in fp64 on the fp64 sum.
 *
 *   x          fp32 [rows, ldx] device input (read only)
 *   out        fp32 [rows] device output
 *   dtype      FR_F32 (the only dtype offered)
 *   epilogue   FR_EPI_SUM or FR_EPI_SQRT; anything else is FR_ERR_INVALID_ARG
 *   workspace  device scratch of fr_workspace_size(FR_OP_SUMSQ, ...) bytes
 *              (only the split form uses it; may be NULL otherwise)
 */
fr_status fr_reduce_sumsq(const void *x, float *out, int64_t rows, int64_t cols, int64_t ldx,
                          fr_dtype dtype, fr_epilogue epilogue, fr_form form, void *workspace,
                          size_t workspace_bytes, fr_stream_t stream);

/*
 * y[x, :] = softmax(x[x, :]):  m = max_r x,  y = exp(x - m) / sum_r exp(x - m)
 *
 * "Stax (4)", section 9.5 (the softmax equation and Listing 9.5: one read and
 * one write per row, masked lanes filled with -inf for the max and 0 for the
 * sum) and "CMU 15-779 Lecture 8", section 3.  The persistent form keeps the
 * row on chip and takes the max and the sum in two passes over registers; the
 * looped form merges per-chunk (m, d) pairs with the online-softmax operator
 * of section 9.5 (Proposition 9.1) and then streams the row again to write y.
 * NaN anywhere in a row makes that row NaN.  Arithmetic is fp32 for both
 * dtypes: FR_F32 reads and writes fp32; FR_BF16 reads bf16, widens it exactly
 * to fp32 (the listing's load-then-cast) and rounds y to bf16 (nearest even).
 *
 *   x          [rows, ldx] device input; y [rows, ldy] device output, both of
 *              `dtype` (bf16 as uint16 bit patterns); x and y may be the same
 *              buffer when ldx == ldy
 *   dtype      FR_F32 or FR_BF16; persistent up to 1024 (fp32) or 2048 (bf16)
 *              columns with one warp per row, up to 32768 with one CTA per
 *              row (the row in registers; for x and y rows at different
 *              offsets within a 32-byte sector, fp32 rows of up to 4608
 *              columns in registers with y's chunks shifted, longer ones
 *              and bf16 rows staged in shared memory); longer rows (or few
 *              rows) take the split form (a cluster of CTAs per row).  Rows
 *              in phase: the slices in registers up to 384 KiB rows, past
 *              that (any length) each CTA streams its run twice, the second
 *              time from L2.  Rows out of phase: the runs staged in shared
 *              memory, up to 409496 fp32 or 818992 bf16 columns, the looped
 *              form beyond
 */
fr_status fr_softmax(const void *x, void *y, int64_t rows, int64_t cols, int64_t ldx,
                     int64_t ldy, fr_dtype dtype, fr_form form, fr_stream_t stream);

/*
 * fr_softmax over rows held in HOST memory, in one of two ways.
 *   direct (chunk_rows = 0): the softmax kernel itself reads x_host and writes
 *     y_host where they are, over the host link (NVLink-C2C on GB300, which
 *     keeps the GPU coherent with host memory); no staging, no workspace.
 *     fp32 rows of up to 1024 columns and bf16 rows of up to 2048 take a
 *     small grid (a quarter of the SMs' CTAs, warps taking rows in turn): the
 *     link serves a bounded number of requests in flight best (fp32: 340 GB/s
 *     both ways against 304 with a warp for every row at once).
 *   staged (chunk_rows >= 1): the rows go to the device in chunks of
 *     `chunk_rows`, through three device staging slots each way (the caller's
 *     workspace), and come back the same way, with a chunk's copy in, the
 *     previous chunk's kernel and the copy out of the one before running at
 *     the same time on the library's own streams (created once per device).
 * The results are those of fr_softmax on the same rows.  The call returns
 * without synchronising; `stream` resumes after the last write of y_host,
 * and work queued on `stream` before the call runs first.  The pages have no
 * counterpart: this is the end-to-end path from host memory.  Measured on
 * GB300 with fp32 [32768, 1024]: direct 790 us, staged (4096-row chunks) 950.
 *
 *   x_host, y_host  [rows, cols] contiguous, of `dtype`, in page-locked host
 *                   memory (cudaHostAlloc or cudaHostRegister); anything else
 *                   is FR_ERR_INVALID_ARG.  They may be the same buffer.
 *   chunk_rows      0 (direct) or rows per chunk (staged)
 *   workspace       staged: device memory of fr_softmax_host_workspace(...)
 *                   bytes, 256-byte aligned, one call at a time may use it;
 *                   direct: ignored (may be NULL)
 *   dtype           FR_F32 or FR_BF16
 * Arguments are checked before anything is enqueued; a CUDA error while the
 * chunks are being enqueued (FR_ERR_CUDA) may leave part of the work queued.
 */
size_t fr_softmax_host_workspace(int64_t cols, fr_dtype dtype, int64_t chunk_rows);
fr_status fr_softmax_host(const void *x_host, void *y_host, int64_t rows, int64_t cols,
                          fr_dtype dtype, int64_t chunk_rows, void *workspace,
                          size_t workspace_bytes, fr_stream_t stream);

/*
 * LayerNorm over each row (not defined on the pages; standard definition):
 *   mean = sum x / n,  var = sum (x - mean)^2 / n,  rstd = 1 / sqrt(var + eps),
 *   y = (x - mean) * rstd * gamma + beta      (rounded to bf16, nearest even)
 * The statistics are Welford (count, mean, M2) triples per thread chunk,
 * combined with the Chan et al. parallel merge, in fp32.  The looped form
 * streams each row through a shared-memory ring filled by bulk asynchronous
 * copies (the multi-stage staging of "Stax (4)", section 9.8, and the tensor
 * descriptors of "CMU 15-779 Lecture 8", section 5) and normalises from the
 * staged copy; the persistent form keeps the row in registers.  FR_FORM_AUTO
 * takes the looped form where cols = C x T x 32 with CTAs of T = 128, 160,
 * 224, 256 or 512 threads (a cluster of C CTAs a row, 32 columns a thread),
 * else the persistent form up to 16384 columns (cols % 8 == 0, 16-byte
 * aligned rows), else the looped form.
 *
 *   x          bf16 [rows, ldx] device input (uint16 bit patterns)
 *   gamma,beta fp32 [cols] device inputs
 *   y          bf16 [rows, ldy] device output
 *   mean, rstd fp32 [rows] device outputs (either may be NULL)
 *   dtype      FR_BF16
 */
fr_status fr_layernorm(const void *x, const float *gamma, const float *beta, void *y,
                       float *mean, float *rstd, int64_t rows, int64_t cols, int64_t ldx,
                       int64_t ldy, float eps, fr_dtype dtype, fr_form form,
                       fr_stream_t stream);

/*
 * Fused log-softmax + cross entropy, one pass over each row:
 *   (m, l) = (max_r x, sum_r exp(x - m)) by the online-softmax merge of
 *   "Stax (4)", section 9.5;  LSE = m + log l (section 9.10);
 *   loss[x] = LSE - x[x, t]  for 0 <= t < cols,   0 for t == ignore_index;
 *   *loss_mean = sum of loss over rows with t != ignore_index / their count
 *               (NaN when every row is ignored), summed in a fixed order.
 * Cross entropy and ignore_index are not on the pages; the semantics follow
 * PyTorch's cross_entropy(reduction='mean').  A target outside [0, cols) other
 * than ignore_index gives that row NaN and sets FR_DEVERR_BAD_TARGET.
 *
 *   logits       bf16 (or fp32) [rows, ld] device input; any ld >= cols (rows
 *                need not be 16-byte aligned: heads and tails are peeled)
 *   target       int64 [rows] device input
 *   loss         fp32 [rows] device output (may be NULL)
 *   loss_mean    fp32 [1] device output (may be NULL)
 *   target_logit fp32 [rows] device output x[x, t] exactly (0 for ignored rows,
 *                NaN for bad targets); may be NULL
 *   argmax       int64 [rows] device output, first index of the row maximum,
 *                NaN counting as the maximum; may be NULL
 *   dtype        FR_BF16 (logits as bf16 bit patterns, widened exactly) or
 *                FR_F32; fp32 logits always run at the default launch
 *                configuration (fr_xent_tune and recorded configurations
 *                are for bf16 logits)
 *   workspace    fr_workspace_size(FR_OP_XENT, ...) bytes when loss_mean is
 *                requested (a ticket, the mean's parts and per-CTA partial
 *                sums), prepared once by fr_xent_workspace_init; every call
 *                leaves it prepared for the next (the last CTA resets the
 *                ticket), so no call spends a launch on a reset.  A workspace
 *                that was not prepared makes the call record
 *                FR_DEVERR_BAD_WORKSPACE and leave loss_mean unwritten.  After
 *                the call it holds the mean's parts at FR_XENT_PARTS_OFFSET.
 *                One call at a time may use a workspace.
 */
fr_status fr_xent(const void *logits, const int64_t *target, float *loss, float *loss_mean,
                  float *target_logit, int64_t *argmax, int64_t rows, int64_t cols,
                  int64_t ld, int64_t ignore_index, fr_dtype dtype, fr_form form,
                  void *workspace, size_t workspace_bytes, fr_stream_t stream);

/*
 * Prepares an fr_xent workspace (writes its ticket; one single-thread kernel on
 * `stream`).  Needed once after the workspace is allocated; fr_xent keeps it
 * prepared.  FR_ERR_INVALID_ARG for NULL, FR_ERR_WORKSPACE_TOO_SMALL under 16
 * bytes, FR_ERR_MISALIGNED unless 16-byte aligned.
 */
fr_status fr_xent_workspace_init(void *workspace, size_t workspace_bytes, fr_stream_t stream);

/*
 * The mean over a batch whose rows are sharded across ranks (one process per
 * GPU, each calling fr_xent on its own rows with loss_mean requested).  Each
 * call leaves two fp64 values in its workspace at byte FR_XENT_PARTS_OFFSET:
 * the sum of the losses it averaged and the number of rows it averaged (those
 * whose target is not ignore_index).  The ranks add their pairs element-wise
 * (an all-reduce with sum, e.g. NCCL over the 16 bytes in place), then each
 * calls fr_xent_mean_from_parts, which writes sum / count rounded to fp32
 * (NaN when no row of the batch counts) -- the mean fr_xent gives on the
 * whole batch, up to the order of the fp64 additions.  This is the path's one
 * exchange step; every other step of every op is independent per row.
 *
 *   workspace    the workspace of the rank's fr_xent call, parts summed over
 *                the ranks; read only
 *   loss_mean    fp32 [1] device output
 * One single-thread kernel on `stream`.
 */
#define FR_XENT_PARTS_OFFSET 16
fr_status fr_xent_mean_from_parts(const void *workspace, float *loss_mean, fr_stream_t stream);

/* ---- launch configurations ----------------------------------------------
 *
 * "Stax (4)", section 9.6: a kernel's launch configuration is a point of a
 * box of parameters (Definition 9.2), chosen by measuring a small candidate
 * set (Algorithm 9.1) and refined by coordinate descent (Algorithm 9.2).
 */

/* Largest number of parameters fr_coordinate_descent takes. */
#define FR_CD_MAX_PARAMS 8

/* Measured cost of a configuration given as log2 of each parameter; return
 * +inf (or NaN) for a configuration that cannot run. */
typedef double (*fr_cost_fn)(const int32_t *log2_params, void *ctx);

/*
 * Algorithm 9.2 over the box lo[i] <= c[i] <= hi[i] of log2 parameters: the
 * neighbours of c are c with one coordinate +1 or -1 (that parameter times or
 * divided by 2); a neighbour is accepted when its cost is below (1 - eps)
 * times the current one; the search ends after a full pass without an
 * acceptance.  Each configuration is costed at most once (the result is
 * remembered), so by Proposition 9.2 the number of acceptances is at most
 * min(|box|, ceil(log(t(c0) / t_min) / -log(1 - eps))) and no neighbour of
 * the result is cheaper by the factor (1 - eps).  Host code only; runs on the
 * calling thread.
 *
 *   p            number of parameters, 1 .. FR_CD_MAX_PARAMS
 *   lo, hi       the box, per parameter (lo[i] <= hi[i])
 *   c            in: the start (inside the box, finite cost); out: the result
 *   eps          acceptance threshold, 0 < eps < 1
 *   acceptances  moves accepted (may be NULL)
 *   evaluations  distinct configurations costed (may be NULL)
 * FR_ERR_INVALID_ARG for a bad argument or a start of infinite cost (c is
 * then left unchanged).
 */
fr_status fr_coordinate_descent(int32_t p, const int32_t *lo, const int32_t *hi, int32_t *c,
                                double eps, fr_cost_fn cost, void *ctx, int32_t *acceptances,
                                int32_t *evaluations);

/* A launch configuration of the cross-entropy kernels (fr_xent without
 * argmax): each field a power of two.  Two families:
 *   the ring kernel (a CTA per row, each thread streaming its 16-byte pieces
 *   through a cp.async ring): threads 128 .. 1024, vectors 1 .. 8 (16-byte
 *   copies per thread per ring item), stages 2 .. 8, ctas_per_sm 1 .. 16;
 *   the warp-per-row kernel (a warp streams a row with 32-byte register
 *   loads, 256-thread CTAs): threads 32, vectors 4 or 8 (32-byte vectors a
 *   lane holds), stages 1, ctas_per_sm 1 .. 16 (a cap).
 * The default is the warp-per-row point (32, 8, 1, 2). */
typedef struct {
  int32_t threads;     /* threads per CTA (32: a warp per row) */
  int32_t vectors;     /* copies or vectors per thread, see above */
  int32_t stages;      /* items in each thread's copy ring (1: no ring) */
  int32_t ctas_per_sm; /* CTAs per SM of the persistent grid, 1 .. 16 */
} fr_xent_config;

/*
 * The configuration fr_xent uses (without argmax) for this shape on the
 * current device: the one recorded by fr_xent_tune or fr_xent_set_config,
 * else the default.  FR_ERR_INVALID_ARG for a bad shape or a NULL out.
 */
fr_status fr_xent_get_config(int64_t rows, int64_t cols, int64_t ld, fr_xent_config *out);

/*
 * Records `cfg` for this shape on the current device (NULL forgets the
 * record).  FR_ERR_INVALID_ARG when cfg is outside the box,
 * FR_ERR_UNSUPPORTED_FORM when it cannot run on this device (shared memory,
 * residency of ctas_per_sm CTAs, register spills).  Records live until the
 * process exits.
 */
fr_status fr_xent_set_config(int64_t rows, int64_t cols, int64_t ld, const fr_xent_config *cfg);

/*
 * Chooses and records the configuration for this shape by measurement on the
 * caller's data (Algorithm 9.1 then Algorithm 9.2).  If a configuration is
 * already recorded for the shape it is returned unmeasured (Algorithm 9.1,
 * line 1).  Otherwise a candidate set of eight configurations (two warp-per-
 * row points, six ring points) is timed (those that cannot run cost +inf),
 * coordinate descent with threshold `eps` walks the ring's box threads x
 * vectors x stages x ctas_per_sm from the fastest ring point, and the faster
 * of its result and the best candidate is recorded.
 * Each configuration is timed over `reps` launches after one warm-up launch
 * (CUDA events on `stream`, the median).  The launches write `loss` (which
 * may be NULL); the call synchronises `stream` and must not be captured into
 * a CUDA graph.  Inputs larger than the L2 cache give cold-cache times.
 *
 *   logits, target, rows, cols, ld, ignore_index, dtype   as for fr_xent
 *   eps          0 < eps < 1; above twice the relative timing noise
 *   reps         1 .. 1000
 *   out          the chosen configuration (may be NULL)
 *   evaluations  configurations timed (may be NULL)
 *   best_ms      median time of the chosen configuration (may be NULL; 0
 *                when the record was returned unmeasured)
 */
fr_status fr_xent_tune(const void *logits, const int64_t *target, float *loss, int64_t rows,
                       int64_t cols, int64_t ld, int64_t ignore_index, fr_dtype dtype,
                       double eps, int32_t reps, fr_stream_t stream, fr_xent_config *out,
                       int32_t *evaluations, float *best_ms);

/*
 * Size of the library's built-in scratch array used by
 * fr_reduce_relu_add_sum_split_static (64 KiB = 8192 fp64 partial sums).
 */
#define FR_STATIC_SCRATCH_BYTES 65536

/*
 * The split form of fr_reduce_relu_add_sum without a caller workspace: same
 * arguments minus form/workspace, same result bit for bit (the same kernels
 * with the same segment count).  The pages have no counterpart of this call;
 * it exists for callers that cannot allocate device memory where they launch
 * -- code inside a host framework that owns every device allocation and
 * forbids raw cudaMalloc in its operator callbacks, latency-critical paths
 * where cudaMalloc/cudaFree may synchronise the device, and interfaces with no
 * way to pass a workspace pointer.
 *
 * The stage-1 partial sums go to a fixed FR_STATIC_SCRATCH_BYTES array in the
 * library's device memory (a static __device__ variable: every GPU that loads
 * the library keeps it until the process exits).  No cudaMalloc, cudaFree or
 * other allocating call is made.
 *
 *   Limit.     rows * segments partials must fit the array (8192 of them; on a
 *              152-SM GB300 every shape with rows <= 8192 fits).  Larger shapes
 *              return FR_ERR_WORKSPACE_TOO_SMALL and nothing is enqueued;
 *              rows > 65535 return FR_ERR_UNSUPPORTED_FORM as for the split form.
 *   First use. The first call on each device looks up the array's device
 *              address (cudaGetSymbolAddress, with that device current) and
 *              caches it; make that first call before any stream capture.
 *   Sharing.   All calls on a device share the one array and it keeps the last
 *              call's partials.  Stage 1 overwrites every partial it uses, so
 *              nothing needs clearing, but calls that overlap on the GPU (on
 *              different streams, or from several host threads without
 *              ordering) race on the array: order them on one stream.
 */
fr_status fr_reduce_relu_add_sum_split_static(const void *a, const void *b, float *out,
                                              int64_t rows, int64_t cols, int64_t lda,
                                              int64_t ldb, fr_dtype dtype, float scale,
                                              fr_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns FR_OK when no device data error was recorded, otherwise
 * FR_ERR_DEVICE_DATA with the FR_DEVERR_* code in *code (if non-NULL).
 */
fr_status fr_check_device_error(fr_stream_t stream, int32_t *code);

#ifdef __cplusplus
}
#endif

#endif /* FR_H_ */
