/*
 * lopt.h -- C ABI of the GB300 learned-optimizer step library (liblopt.so).
 *
 * One call, lopt_step(), performs one step of a small_fc_lopt-style learned
 * optimizer over a whole list of parameter tensors on one GPU:
 *
 *   for every element of every tensor
 *     - update three momenta, one RMS accumulator and the Adafactor-factored
 *       row/column accumulators from the gradient,
 *     - build the 39-wide feature vector (28 per-element features + 11
 *       time features),
 *     - divide each per-element feature by its root-mean-square over the
 *       whole tensor,
 *     - run the per-element MLP 39 -> H -> H -> 2 (ReLU, ReLU, linear),
 *     - update = direction * exp(magnitude * 1e-3) * 1e-3,
 *       param -= lr * update.
 *
 * Method: "PyLO: Towards Accessible Learned Optimizers in PyTorch" (MLSys 2026
 * talk notes), sections "融合カーネル戦略" (kernel 1 = features + per-feature
 * sum of squares, kernel 2 = features + normalisation + MLP + update),
 * "メモリ階層の活用" (features in registers, statistics in shared memory,
 * d_feat ~ 39, d_hidden ~ 32) and "PyLO のライブラリ設計" (per-parameter
 * accumulators kept by the optimiser).
 *
 * Conventions for every entry point
 *   - Return 0 (LOPT_OK) on success, a negative LOPT_E_* code otherwise;
 *     lopt_strerror() names the code.
 *   - Device pointers are CUDA global-memory addresses on the device that was
 *     current when the handle was created; host pointers are ordinary CPU
 *     memory.  No pointer is retained past the call that receives it, except
 *     that lopt_step() enqueues GPU work that reads and writes the tensor
 *     buffers until that work has completed on the given stream.
 *   - Nothing in this ABI uses C++ or PyTorch types.
 */
#ifndef LOPT_H
#define LOPT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ------------------------------------------------------- */
#define LOPT_OK             0
#define LOPT_E_ARG         -1  /* null / out-of-range argument            */
#define LOPT_E_SHAPE       -2  /* rows*cols < 1 or too large               */
#define LOPT_E_ALIGN       -3  /* a tensor pointer is not 4-byte aligned   */
#define LOPT_E_CUDA        -4  /* a CUDA runtime call failed               */
#define LOPT_E_OOM         -5  /* device workspace allocation failed       */
#define LOPT_E_UNSUPPORTED -6  /* hidden width / MLP path not available    */
#define LOPT_E_TIMEOUT     -7  /* a bounded device-side wait gave up       */
#define LOPT_E_ALIAS       -8  /* two tensor buffers overlap               */
#define LOPT_E_TOO_LARGE   -9  /* needs more than the fixed static scratch */

/* ---- fixed sizes ------------------------------------------------------- */
#define LOPT_D_FEAT        39  /* 28 per-element + 11 time features        */
#define LOPT_N_STATS       28  /* normalised (per-element) features        */
#define LOPT_MAX_HIDDEN    64

/* ---- MLP evaluation paths (lopt_set_mlp_path) -------------------------- */
#define LOPT_MLP_FP32       0  /* FP32 FMA on CUDA cores (default)          */
#define LOPT_MLP_TC         1  /* tcgen05 tensor cores for the two hidden   */
                               /* layers (FP16 operands, FP32 accumulation);*/
                               /* output layer in FP32 on CUDA cores        */

typedef struct lopt_ctx* lopt_handle;

/*
 * One parameter tensor.  All pointers are DEVICE pointers to contiguous fp32
 * arrays, owned by the caller; lopt_step() updates them in place.
 *
 *   param   [rows*cols]  read, then overwritten with the stepped values
 *   grad    [rows*cols]  read only
 *   mom[k]  [rows*cols]  momentum with decay 0.1, 0.5, 0.9 (k = 0, 1, 2)
 *   rms     [rows*cols]  second moment, decay 0.999
 *   row[k]  [rows]       Adafactor row accumulator, decay 0.1, 0.5, 0.9
 *   col[k]  [cols]       Adafactor column accumulator, decay 0.1, 0.5, 0.9
 *
 * Layout: element (i, j) of the [rows x cols] view sits at i*cols + j.  A
 * rank-1 tensor of n elements is passed as rows = 1, cols = n; a rank-0
 * tensor as 1 x 1; rank >= 3 as prod(leading dims) x last dim.
 * Accumulators must be zero before the first step.  No buffer may overlap
 * another buffer of the same call.
 * weight_set selects one of the MLP weight sets given to lopt_create().
 */
typedef struct {
  float*       param;
  const float* grad;
  float*       mom[3];
  float*       rms;
  float*       row[3];
  float*       col[3];
  int64_t      rows;
  int64_t      cols;
  int32_t      weight_set;
  int32_t      reserved;   /* must be 0 */
} lopt_tensor;

/*
 * Number of floats in one MLP weight set for the given widths:
 * d_feat*H + H + H*H + H + 2*H + 2.
 */
int lopt_weight_set_size(int d_feat, int hidden);

/*
 * Create a handle on the current CUDA device.
 *   mlp_weights  HOST pointer, n_sets consecutive weight sets, each laid out
 *                row-major as W1[d_feat][H], b1[H], W2[H][H], b2[H],
 *                W3[H][2], b3[2]  (h1 = ReLU(x W1 + b1), h2 = ReLU(h1 W2 + b2),
 *                (direction, magnitude) = h2 W3 + b3).  Copied to the device;
 *                the caller may free it after the call returns.
 *   d_feat       must be LOPT_D_FEAT (39).
 *   hidden       1 .. LOPT_MAX_HIDDEN.
 *   n_sets       >= 1.
 *   out          receives the handle.
 * Errors: LOPT_E_ARG (bad pointer / size), LOPT_E_UNSUPPORTED (hidden out of
 * range), LOPT_E_CUDA / LOPT_E_OOM (device failure; *out is left NULL).
 * Synchronous.
 */
int lopt_create(const float* mlp_weights, int d_feat, int hidden, int n_sets,
                lopt_handle* out);

/*
 * Choose how the MLP is evaluated by later lopt_step() calls:
 * LOPT_MLP_FP32 (exact FP32 arithmetic) or LOPT_MLP_TC (tensor cores for
 * the two hidden layers: the 28 normalised features, W1, b1 + sum_s tau_s
 * W1[28 + s], ReLU(h1) and W2 in FP16 with FP32 accumulation, b2 in FP32;
 * the output layer in FP32 on CUDA cores).  The FP16 operands cost about
 * 1e-3 of the update's RMS on average and up to a few 1e-2 of it on outlier
 * elements (as an exact FP16-operand MLP does); an updated parameter of a
 * tensor that is not all update (weights, LayerNorm scales) stays within
 * 2e-3 of the exact value.  LOPT_E_UNSUPPORTED if the path cannot run this
 * handle's hidden width (it covers widths up to 32).
 */
int lopt_set_mlp_path(lopt_handle h, int path);

/*
 * Decoupled weight decay for later lopt_step() calls: every element becomes
 *   param <- param - lr * (update + weight_decay * param)
 * with the parameter before the step (0 by default: param -= lr * update).
 * The pages on PyLO report that learning-rate schedules and weight decay
 * change what a learned optimiser reaches (section "学習率スケジュールと重み
 * 減衰の効果"); the schedule is the caller's per-step lr.  Applied in the
 * apply pass at no extra memory traffic.  LOPT_E_ARG if weight_decay is
 * negative or not finite.
 */
int lopt_set_weight_decay(lopt_handle h, float weight_decay);

/*
 * Single sweep through L2 for later lopt_step() calls.  With group_bytes >
 * 0 the list is cut into groups of consecutive tensors whose state (p, g,
 * m0..2, v: 24 bytes per element) is at most group_bytes, a larger tensor
 * forming a group of its own, and each group runs the three kernels before
 * the next group starts.  The statistics pass then reads g just after the
 * row/column pass read it, and the apply pass reads p, g, m, v just after
 * the statistics pass read them, so that with groups well inside the L2
 * (129 MB on GB300) most of those re-reads come from L2 instead of DRAM.
 * This is the pages' direction of keeping a tensor's state on chip between
 * the two passes ("PyLO: Towards Accessible Learned Optimizers in PyTorch",
 * sections "メモリ階層の活用" and "制約と今後の展望"), done by launch
 * order.  Every statistic still covers a whole tensor, so results are the
 * same bits as without groups.  Each group adds three launches and their
 * start and end.  0 (the default) turns it off: one launch of each kernel
 * over the whole list.  Row-sharded steps and host-buffer steps always use
 * one group.  Kernel timing (lopt_kernel_times) sums each kernel over the
 * groups.  Errors: LOPT_E_ARG (NULL handle or a negative size).
 */
int lopt_set_sweep_bytes(lopt_handle h, int64_t group_bytes);

/*
 * One learned-optimizer step over n_tensors tensors (HOST array of
 * descriptors; it is read during the call only).
 *   t       1-based step count (drives the 11 time features tanh(t / x_s)).
 *   lr      multiplies the update (param -= lr * update, plus the decay set
 *           by lopt_set_weight_decay()).
 *   stream  cudaStream_t to enqueue on (NULL = legacy default stream).
 * The whole list is processed by three kernel launches (row/column moments,
 * feature statistics, normalise + MLP + apply), or three per group of
 * tensors after lopt_set_sweep_bytes().  Asynchronous: returns once
 * the work is enqueued.  Validation happens before anything is enqueued and
 * a failed validation leaves every buffer untouched.  Calls on one handle
 * are ordered with each other even across streams; a handle must not be
 * used from two host threads at once.
 * Errors: LOPT_E_ARG, LOPT_E_SHAPE, LOPT_E_ALIGN, LOPT_E_ALIAS (validation);
 * LOPT_E_OOM (workspace growth); LOPT_E_CUDA (launch failure).
 */
int lopt_step(lopt_handle h, const lopt_tensor* tensors, int n_tensors,
              int64_t t, float lr, void* stream);

/*
 * The same step for a training loop that holds gradients and parameters in
 * HOST memory: for each tensor i, grad_host[i] (rows * cols floats) is the
 * gradient, and the updated parameters are copied into param_host[i]
 * (rows * cols floats).  tensors[i].grad is not used (it may be NULL): the
 * gradients go through two device staging buffers of the handle, used by
 * alternate calls.  The accumulators (mom, rms, row, col) and the device
 * parameters are updated as by lopt_step().
 *
 * Per tensor the step is the same computation as lopt_step() (every
 * normalisation statistic belongs to one tensor), so results are
 * identical.  The list is cut into up to 2 groups (lopt_set_host_groups)
 * of consecutive tensors of about equal size (at least 4 Mi elements
 * each), each stepped by its own three launches on `stream`; the copies
 * run on two streams of the handle, so that gradient and parameter copies
 * overlap the kernels of other groups, also across consecutive calls.  Adjacent tensors whose buffers
 * follow each other on both sides move in one copy.
 *
 * Ordering.  The kernels are ordered with other work on `stream`.  The
 * parameter copies are not: they may still run after `stream` has passed
 * the call.  Before reading param_host, writing new gradients into the
 * same grad_host buffers, or touching the device parameters with other
 * work, call lopt_host_sync() on the stream that does so (or lopt_check(),
 * which waits on the host).  lopt_step() and the sharded calls of the
 * handle wait for these copies by themselves.
 *
 * grad_host, param_host: HOST arrays of n_tensors HOST pointers, read during
 * the call only.  The buffers must not overlap one another; page-locked
 * memory (cudaHostAlloc, or pinned) lets the copies overlap the kernels,
 * pageable memory works without that.  The staging buffers take 2 x 4 bytes
 * per element of device memory, allocated on the first call with a new
 * list.  Kernel timing (lopt_set_kernel_timing) and lopt_feature_stats()
 * cover lopt_step() calls only.
 * Errors: as lopt_step() (validation covers the list with its staging
 * gradients); LOPT_E_ARG also for a NULL host pointer of a non-empty tensor
 * and during a row-sharded step; LOPT_E_OOM if the staging buffers cannot
 * be allocated.
 */
int lopt_step_host(lopt_handle h, const lopt_tensor* tensors, int n_tensors,
                   const float* const* grad_host, float* const* param_host,
                   int64_t t, float lr, void* stream);

/*
 * Makes `stream` wait (without blocking the host) until every parameter
 * copy of the handle's host-buffer steps enqueued so far is done: after it,
 * work on `stream` may read param_host, and the host may use param_host and
 * refill grad_host once `stream` has reached this point.
 * Errors: LOPT_E_ARG (NULL handle), LOPT_E_CUDA.
 */
int lopt_host_sync(lopt_handle h, void* stream);

/*
 * Most groups of tensors a host-buffer step of this handle uses (1..16;
 * default 2).  One group runs the copies and the kernels one after the
 * other; with more, the copies of one group overlap the kernels of
 * another, but each group adds three launches and their start and end.
 * Takes effect on the next lopt_step_host() call.  Errors: LOPT_E_ARG (NULL handle or a
 * value out of range).
 */
int lopt_set_host_groups(lopt_handle h, int max_groups);

/*
 * ---- Row-sharded step (data parallel over ranks) --------------------------
 * The step of the PyLO pages' distributed optimiser (section "分散最適化
 * ステップ": each rank owns a slice of the optimiser state, as after a
 * reduce-scatter of the gradients).  Every rank owns whole rows of each
 * tensor; the only quantities that need all rows are the column means of
 * g^2, the mean of the row accumulators (rho) and the 28 feature square
 * sums, so a step is three calls with two sums over the ranks in between:
 *
 *   lopt_shard_begin   row moments of the local rows; writes this rank's
 *                      column sums of g^2 and row-accumulator sums to x1
 *   (caller: x1 <- sum of x1 over the ranks, e.g. an all-reduce)
 *   lopt_shard_middle  column accumulators and rho from x1; writes this
 *                      rank's feature square sums to x2
 *   (caller: x2 <- sum of x2 over the ranks)
 *   lopt_shard_end     normalisation from x2, MLP, update of the local rows
 *
 * Every rank passes the same list: same tensors, order, cols and weight
 * sets; tensors[i].rows is the number of rows this rank owns (0 allowed:
 * then only col[k] is read, the other pointers may be NULL) and
 * global_rows[i] the rows of the whole tensor.  The column accumulators are
 * replicated: every rank passes its own copy and all copies stay equal.
 * The ranks' rows of a tensor must add up to global_rows[i]; rows are in
 * any order.  With one rank owning everything the results equal
 * lopt_step() up to the rounding of the sums.
 *
 * x1, x2: caller-owned DEVICE buffers of n_x1, n_x2 doubles
 * (lopt_shard_sizes), read and written by the kernels of this step only;
 * lopt_shard_begin zeroes them.  All three calls are asynchronous on their
 * stream and ordered with each other; no other step of the handle may run
 * between them (LOPT_E_ARG).  Errors as lopt_step().
 */
int lopt_shard_sizes(const lopt_tensor* tensors, int n_tensors, int64_t* n_x1, int64_t* n_x2);
int lopt_shard_begin(lopt_handle h, const lopt_tensor* tensors, const int64_t* global_rows,
                     int n_tensors, int64_t t, float lr, double* x1, double* x2, void* stream);
int lopt_shard_middle(lopt_handle h, void* stream);
int lopt_shard_end(lopt_handle h, void* stream);

/*
 * The launch schedule that lopt_step() builds for a tensor list, computed on
 * the host alone (no device call, no handle; thread-safe).  The step's work
 * is split into units ("PyLO: Towards Accessible Learned Optimizers in
 * PyTorch", section "融合カーネル戦略": statistics over every element of a
 * tensor before its apply pass):
 *   K0  row strips of a tensor (row/column second moments; its last strip
 *       sums the strips' column partials);
 *   K1  chunks of 16,384 elements (feature square sums);
 *   K2  chunks of 4,096 elements (normalise, MLP, update).
 *   tensors, n_tensors  as for lopt_step(); only rows, cols, reserved and
 *               the 16-byte alignment of the pointers are read (the
 *               pointers are never dereferenced).
 *   sweep_bytes as lopt_set_sweep_bytes() (0: one launch per kernel).
 *   n_units     out, 3 ints: the units of K0, K1, K2.
 *   units       out or NULL: 2 ints per unit, (tensor index, index of the
 *               unit within its tensor), K0's units in launch order, then
 *               K1's, then K2's.
 *   strip_rows  out or NULL: n_tensors ints, the rows of each K0 strip (the
 *               last strip of a tensor may have fewer).
 *   n_groups    out: the groups of the single sweep (0 when sweep_bytes is 0).
 *   groups      out or NULL: 6 ints per group: the first unit and the unit
 *               count of K0, K1 and K2.
 * Call with NULL units / strip_rows / groups for the counts, then again
 * with arrays of that size.  Errors: LOPT_E_ARG (n_tensors < 0, NULL
 * tensors with n_tensors > 0, NULL n_units or n_groups, a negative
 * sweep_bytes, reserved != 0); LOPT_E_SHAPE (lopt_step()'s shape rules).
 */
int lopt_schedule_info(const lopt_tensor* tensors, int n_tensors, int64_t sweep_bytes,
                       int32_t* n_units, int32_t* units, int32_t* strip_rows,
                       int32_t* n_groups, int32_t* groups);

/*
 * Wait for the handle's last step and report device-side status:
 * LOPT_OK, LOPT_E_TIMEOUT (a bounded wait inside a kernel gave up; that
 * step's results are invalid) or LOPT_E_CUDA.  Clears the status.
 */
int lopt_check(lopt_handle h);

/*
 * Per-feature sums of squares S_d (d = 0..27) that the last step computed
 * for tensor `index` of its list: S_d = sum over elements of feature_d^2,
 * the statistic the normalisation divides by (as sqrt(S_d / N + 1e-30)).
 * out: HOST array of at least LOPT_N_STATS doubles.  Synchronous.
 */
int lopt_feature_stats(lopt_handle h, int index, double* out);

/*
 * Per-kernel device timing of later steps.  enable = 1 makes lopt_step()
 * record CUDA events on its stream around each of its three launches
 * (enable = 0, the default, records none).
 */
int lopt_set_kernel_timing(lopt_handle h, int enable);

/*
 * Device time summed over the steps timed since timing was enabled or since
 * the last call: ms[0] row/column kernel, ms[1] statistics kernel, ms[2]
 * apply kernel (milliseconds, CUDA-event resolution); launches[k] = number of
 * launches summed.  ms and launches: HOST arrays of 3.  Waits for the last
 * timed step; resets the sums.
 */
int lopt_kernel_times(lopt_handle h, double* ms, int64_t* launches);

/*
 * Row/column second-moment update of ONE tensor without any device
 * allocation.  The paper has no counterpart to this entry point; it exists
 * for callers that cannot call cudaMalloc: code running inside a runtime or
 * framework that owns every device allocation, or under a fixed device-memory
 * budget, or on a path where cudaMalloc's implicit device-wide
 * synchronisation is not acceptable.  It runs the same row/column kernel as
 * lopt_step() over the same strips, but takes its scratch from a fixed array
 * of LOPT_STATIC_SCRATCH_BYTES bytes that the library reserves in device
 * memory of every GPU on which it is loaded, held until the process exits.
 * When grad, the column accumulators and every other array lopt_step() is
 * given for the tensor are 16-byte aligned (as torch allocations are), both
 * calls take the same 128-bit route and their results are the same bits;
 * otherwise they agree to rounding.  The descriptor and unit table are
 * written into the scratch by a small kernel from its launch parameters (no
 * host-to-device copy).  No handle is needed.
 *   grad     DEVICE [rows*cols] fp32, read.
 *   row      HOST array of 3 DEVICE pointers, [rows] fp32 each: the row
 *            accumulators (decays 0.1, 0.5, 0.9), updated in place.
 *   col      HOST array of 3 DEVICE pointers, [cols] fp32 each: the column
 *            accumulators, updated in place.
 *   rows, cols  the [rows x cols] view, as in lopt_tensor.
 *   inv_rho  DEVICE [3] fp32, written: 1 / mean_i row[k][i] after the
 *            update, or 0 where that mean is 0.
 *   stream   cudaStream_t (NULL = legacy default stream).
 * Asynchronous on `stream`.  The first call on a device looks up that
 * device's scratch address (once, with the device current); make that first
 * call before any stream capture.  Every call on a device shares the one
 * scratch array, which keeps the previous call's contents (the call clears
 * the parts that must start at zero), so calls that overlap on the GPU --
 * two streams, or two host threads -- race and must be ordered by the caller.
 * Errors: LOPT_E_ARG / LOPT_E_ALIGN / LOPT_E_SHAPE / LOPT_E_ALIAS
 * (validation, nothing enqueued), LOPT_E_TOO_LARGE (the tensor needs more
 * than LOPT_STATIC_SCRATCH_BYTES of scratch; nothing enqueued),
 * LOPT_E_CUDA.
 */
#define LOPT_STATIC_SCRATCH_BYTES (2u << 20)
int lopt_rowcol_static(const float* grad, float* const* row, float* const* col,
                       int64_t rows, int64_t cols, float* inv_rho, void* stream);

/* Release every device allocation of the handle (waits for its work). */
/*
 * Self-test of failure detection, for the current device.  Every wait of
 * the library's kernels on an mbarrier (a pipeline stage, an MMA
 * completion) is bounded by %globaltimer: when it runs out, the kernel
 * raises a timeout flag that lopt_check() reports as LOPT_E_TIMEOUT, every
 * role stops, and the CUDA context stays usable.  This call runs that same
 * bounded wait in one block of 32 threads on a barrier that expects two
 * arrivals and gets one, so that it must run out after limit_ns
 * nanoseconds (1 .. 1e9), and synchronises with the device.
 * Returns LOPT_E_TIMEOUT when the wait gave up and raised the flag, as
 * designed; LOPT_OK would mean that the wait had returned on a phase that
 * never completed.  Errors: LOPT_E_ARG (limit out of range), LOPT_E_OOM,
 * LOPT_E_CUDA.
 */
int lopt_selftest_wait(int64_t limit_ns);

int lopt_destroy(lopt_handle h);

/* Static string naming an error code. */
const char* lopt_strerror(int code);

/*
 * Name and description of the last CUDA error on which a call made by this
 * host thread returned LOPT_E_CUDA or LOPT_E_OOM ("" if none yet).  The
 * string belongs to the library and stays valid until the thread's next
 * failing call.
 */
const char* lopt_last_cuda_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int lopt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LOPT_H */
