/*
 * snack.h -- C ABI of the GB300 truly sparse linear layer.
 *
 * Source: "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks
 * on GPU" (abstract).  The abstract describes a GPU layer that keeps and
 * multiplies only the weights that exist (a COO SpMM kernel), computes its
 * gradients without ever forming a dense weight, and lets the user rewire
 * its connections during Dynamic Sparse Training.  This header makes those
 * four operations concrete:
 *
 *   forward        Y[b,r]  = bias[r] + sum_{k: row[k]=r} val[k] * X[b,col[k]]
 *   input grad     dX[b,c] = sum_{k: col[k]=c} val[k] * dY[b,row[k]]
 *   weight grad    dW[k]   = sum_b dY[b,row[k]] * X[b,col[k]]  (stored positions only)
 *                  db[r]   = sum_b dY[b,r]
 *   restructure    prune the n_prune smallest |val|, regrow as many at uniformly
 *                  random positions that were empty, value +0, re-sort the COO.
 *
 * Layout.  W is out_f x in_f, stored as row-sorted COO: int32 row[nnz] and
 * col[nnz], strictly increasing in (row, col) (no duplicates), plus val[nnz]
 * in fp32 or bf16.  X is [batch, in_f] and Y is [batch, out_f], row-major
 * (torch Linear convention, Y = X W^T + b); dY and dX likewise.  bias, dW and
 * db are fp32.  Accumulation is fp32 in every kernel.
 *
 * Memory ownership.  Every device buffer -- indices, values, activations,
 * outputs, the plan and the workspaces -- is allocated and freed by the
 * caller.  The library never allocates device memory.  A handle owns host
 * metadata, and after its first restructure also two CUDA streams, five
 * events and 32 bytes of mapped pinned host memory; snack_destroy frees them.
 *
 * Streams.  Every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream), except snack_create with validate != 0, which
 * synchronises `stream`, and snack_restructure, which waits on the host for
 * its draw count (see there).  A plan and a workspace may be used by one call
 * in flight at a time.  After either restructure the update of the plan's
 * column view may still be running on a stream of the handle; every call
 * that reads the column view (snack_spmm_dx, snack_spmm_dx_gelu,
 * snack_sddmm_dw, snack_backward and both restructures) first makes its
 * stream wait for it, so results never depend on the timing.  The forward
 * reads only the row half of the plan and does not wait.  snack_wait_plan
 * orders any stream after that update.  The update's stream has the lowest
 * stream priority: calls queued next on a stream of higher priority (see
 * cudaStreamCreateWithPriority) run ahead of it, and it fills the gaps they
 * leave.
 *
 * Host threads.  Calls may come from several host threads.  The launchers
 * raise a kernel's dynamic shared-memory limit (a per-process, per-device
 * setting) through one table kept under a lock, and never lower it, so
 * threads launching one kernel for layers of different sizes do not disturb
 * each other.  Calls on one handle, plan or workspace must still be ordered
 * (one call in flight at a time, see Streams).
 *
 * Errors.  Every entry point returns a snack_status.  Arguments are checked
 * on the host before any launch; a failed launch or CUDA call returns
 * SNACK_ERR_CUDA.  The library never aborts, exits or traps on the device.
 *
 * Tensor-core path.  A bf16 layer with at least 8 % of W stored, out_f and
 * in_f multiples of 8 and at most 65536, created with max_batch >= 16, runs
 * calls with batch >= 16 (activations 16-byte aligned) as dense contractions
 * on the tensor cores (tcgen05), never densifying W in memory: each CTA
 * builds W tiles in shared memory from a per-(64-column block, row) mask and
 * value-offset table that the plan keeps, and multiplies them with activation
 * tiles brought in by TMA; the weight gradient is read back from the
 * accumulators at the stored positions only.  snack_query_sizes reserves the
 * tables in the plan and the path's scratch (split-K partial sums and
 * transposed activations) in the workspace; a call given a smaller workspace
 * takes the gather kernels instead.  Results follow the same tolerance
 * contract.
 *
 * Plan contract.  snack_create derives a plan (row offsets, load-balanced
 * tiles, a column-ordered view) from row/col.  row/col may change only through
 * snack_restructure, which rebuilds the plan for the new pattern; the values
 * may change freely between calls.  Passing a different pattern than the one
 * the plan was built from gives undefined results (no fault: every index the
 * kernels use is read from the plan, whose entries are in range).
 */
#ifndef SNACK_H
#define SNACK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SNACK_VERSION 1

/* Opaque layer handle (host memory only). */
typedef struct snack_layer *snack_handle;

/* A cudaStream_t. */
typedef struct CUstream_st *snack_stream_t;

typedef enum snack_status {
  SNACK_OK = 0,
  SNACK_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad size, aliasing, batch > max_batch */
  SNACK_ERR_UNSORTED = 2,     /* validation: (row, col) not strictly increasing */
  SNACK_ERR_OUT_OF_RANGE = 3, /* validation: an index outside [0,out_f) x [0,in_f) */
  SNACK_ERR_WORKSPACE = 4,    /* plan or workspace smaller than the call needs (the queried sizes always do) */
  SNACK_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
  SNACK_ERR_TIMEOUT = 6,      /* restructure: a bounded device-side wait gave up (not expected); nothing was changed */
  SNACK_ERR_UNSUPPORTED = 7,  /* val and act dtypes differ, or max(out_f, in_f) x padded batch >= 2^32 */
  SNACK_ERR_NO_SPACE = 8      /* restructure: too few empty positions, or draw budget spent */
} snack_status;

typedef enum snack_dtype { SNACK_F32 = 0, SNACK_BF16 = 1 } snack_dtype;

/*
 * Sizes of the caller-allocated buffers for a layer.
 *   plan_bytes       persistent plan, alive as long as the handle;
 *   workspace_bytes  scratch for snack_create and for fwd / dx / dw with
 *                    batch <= max_batch (contents need not survive calls).
 *                    Calls with batch <= 8 whose gathered operand (x for the
 *                    forward, dy for the gradients) fits 96 KB at the batch
 *                    rounded up to 1, 2, 4 or 8 run one small-batch kernel
 *                    that uses none of it; other calls check ws_bytes against
 *                    what they use and return SNACK_ERR_WORKSPACE before any
 *                    launch when it is short.
 * For layers whose column view is rebuilt after the call returns (256 <
 * in_f <= 131072 and row plus column index bits <= 32), plan_bytes also holds
 * that rebuild's scratch (8 bytes per stored weight and two small tables), so
 * it never uses the caller's workspace.
 * Limits: 1 <= out_f, in_f < 2^31; 0 <= nnz <= out_f*in_f and nnz < 2^31 - 1;
 * 1 <= max_batch <= 65535.  val_t must equal act_t (fp32/fp32 or bf16/bf16).
 * Either output pointer may be NULL.
 */
snack_status snack_query_sizes(int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch,
                               snack_dtype val_t, snack_dtype act_t, size_t *plan_bytes,
                               size_t *workspace_bytes);

/*
 * Build a layer handle and its plan from the pattern row/col (device, nnz
 * entries each, caller-owned; only read during the call).  `plan` (device,
 * 256-byte aligned, plan_bytes >= the queried size) receives the plan;
 * `ws` (device, 256-byte aligned) is scratch.  With validate != 0 the pattern
 * is checked on the device (ranges, strict order) and the call synchronises
 * `stream` to return SNACK_ERR_OUT_OF_RANGE or SNACK_ERR_UNSORTED; with
 * validate == 0 an invalid pattern gives undefined results.  When nnz is a
 * multiple of out_f the call also checks on the device whether every row
 * holds nnz / out_f stored weights (a constant fan-in, as Structured RigL
 * keeps and snack_restructure_rows preserves) and synchronises `stream` once
 * to read the answer; such layers run their forward with whole rows per warp.
 * The handle is bound to the CUDA device current at this call.
 */
snack_status snack_create(snack_handle *out_handle, int32_t out_f, int32_t in_f, int64_t nnz,
                          int32_t max_batch, snack_dtype val_t, snack_dtype act_t,
                          const int32_t *row, const int32_t *col, void *plan, size_t plan_bytes,
                          void *ws, size_t ws_bytes, int validate, snack_stream_t stream);

/*
 * Forward (the SNACK-COO SpMM of the abstract, over stored weights only):
 *   y[b, r] = bias[r] + sum_{k : row[k] = r} val[k] * x[b, col[k]]
 * x [batch, in_f] and y [batch, out_f] in act dtype; bias fp32 [out_f] or
 * NULL (zero).  0 <= batch <= max_batch.  y must not overlap x.  Rows without
 * stored weights get bias[r].  Deterministic (no atomics on outputs).
 */
snack_status snack_spmm_fwd(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                            const void *x, int32_t batch, const float *bias, void *y, void *ws,
                            size_t ws_bytes, snack_stream_t stream);

/*
 * Forward without a workspace argument (the paper has no counterpart; this is
 * a convenience of this library).  For callers that may not allocate device
 * memory on their call path -- e.g. a plugin run from an inference engine's
 * enqueue step, or a real-time loop whose memory is fixed at start-up -- and
 * so cannot pass the scratch buffer snack_spmm_fwd takes.  Same arguments and
 * result as snack_spmm_fwd; its scratch is a 32 MiB array inside the
 * library's device image, held by every GPU that loads the library until the
 * process exits.  A call needing more scratch than that (large in_f * batch)
 * returns SNACK_ERR_WORKSPACE before any launch.  The call takes the path
 * snack_spmm_fwd would take with a 32 MiB workspace: a layer on the
 * tensor-core path whose scratch for this batch exceeds it runs on the gather
 * kernels instead (same results within the tolerance contract, not bit for
 * bit).  The first call on a device
 * looks up the array's device address (with that device current), so make it
 * before any stream capture.  All calls share the array: calls that overlap on
 * the GPU race, so order them (one stream, or events).  Allocates nothing.
 */
snack_status snack_spmm_fwd_noalloc(snack_handle h, const int32_t *row, const int32_t *col,
                                    const void *val, const void *x, int32_t batch, const float *bias,
                                    void *y, snack_stream_t stream);

/*
 * Input gradient (transposed SpMM; the sparse backward pass of the abstract):
 *   dx[b, c] = sum_{k : col[k] = c} val[k] * dy[b, row[k]]
 * dy [batch, out_f], dx [batch, in_f] in act dtype; dx must not overlap dy.
 * Deterministic.
 */
snack_status snack_spmm_dx(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                           const void *dy, int32_t batch, void *dx, void *ws, size_t ws_bytes,
                           snack_stream_t stream);

/*
 * Forward with a GELU epilogue, for the sparse MLP block of the abstract's
 * GPT-2 experiment (two sparse layers with GELU between them):
 *   y_pre[b, r] = bias[r] + sum_{k : row[k] = r} val[k] * x[b, col[k]]
 *   y[b, r]     = GELU(y_pre[b, r]) = y_pre * Phi(y_pre)   (exact erf form, fp32)
 * y_pre (same shape and dtype as y) may be NULL; keep it when the backward
 * pass needs GELU'.  y_pre and y must not overlap x or each other.
 */
snack_status snack_spmm_fwd_gelu(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                                 const void *x, int32_t batch, const float *bias, void *y_pre, void *y, void *ws,
                                 size_t ws_bytes, snack_stream_t stream);

/*
 * Input gradient through a GELU that preceded this layer:
 *   dx[b, c] = GELU'(x_pre[b, c]) * sum_{k : col[k] = c} val[k] * dy[b, row[k]]
 * x_pre [batch, in_f] is the pre-activation this layer's input came from (the
 * y_pre of the previous layer's snack_spmm_fwd_gelu); GELU'(t) = Phi(t) +
 * t phi(t).  dx must not overlap dy or x_pre.
 */
snack_status snack_spmm_dx_gelu(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                                const void *dy, int32_t batch, const void *x_pre, void *dx, void *ws,
                                size_t ws_bytes, snack_stream_t stream);

/*
 * Weight gradient at the stored positions only (sampled dense-dense product):
 *   dw[k] = sum_b dy[b, row[k]] * x[b, col[k]]     fp32 [nnz]
 *   db[r] = sum_b dy[b, r]                         fp32 [out_f], or NULL to skip
 * x [batch, in_f], dy [batch, out_f] in act dtype.  Deterministic.
 */
snack_status snack_sddmm_dw(snack_handle h, const int32_t *row, const int32_t *col, const void *x,
                            const void *dy, int32_t batch, float *dw, float *db, void *ws,
                            size_t ws_bytes, snack_stream_t stream);

/*
 * The whole sparse backward pass in one call: the input gradient of
 * snack_spmm_dx, the weight gradient of snack_sddmm_dw, and db (NULL to
 * skip).  When one batch tile covers the batch (batch <= 128 for fp32, 256
 * for bf16) the two gradients come from one pass over the column view: each
 * gathered dY row slice is also dotted with the current column of X, so the
 * index and value streams are read once.  Wider batches run the two kernels
 * one after the other.  Outputs as in snack_spmm_dx / snack_sddmm_dw; dx must
 * not overlap x or dy.  Deterministic.
 */
snack_status snack_backward(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                            const void *x, const void *dy, int32_t batch, void *dx, float *dw, float *db,
                            void *ws, size_t ws_bytes, snack_stream_t stream);

/*
 * Workspace needed by snack_restructure for a given n_prune.
 */
snack_status snack_restructure_workspace_size(snack_handle h, int64_t n_prune, size_t *bytes);

/*
 * Dynamic Sparse Training restructure (the abstract's connection rewiring):
 *  1. rank stored weights by (|val|, k) ascending, NaN above every number;
 *     the first n_prune are pruned;
 *  2. survivors keep order and value bits;
 *  3. draws i = 0, 1, ... of SplitMix64 (state mix(seed ^ mix(step)),
 *     advanced by 0x9E3779B97F4A7C15 before each draw) are mapped to
 *     positions p_i = floor(u_i * out_f*in_f / 2^64); p_i is accepted when it
 *     was empty before this call and is not already accepted; stop at n_prune;
 *  4. regrown entries (p / in_f, p mod in_f) get value +0;
 *  5. the output is survivors and regrown merged in (row, col) order.
 * Outputs (device, nnz entries, must not overlap the inputs): row_out, col_out,
 * val_out (val dtype), src_out (optional, NULL to skip): old index k of each
 * survivor, -1 for a regrown entry.  The handle's plan is rebuilt for the new
 * pattern; later calls must pass row_out/col_out.  Needs ws_bytes >=
 * snack_restructure_workspace_size(h, n_prune).  The regrow (draws,
 * acceptance, sort of the new positions) runs on `stream`; the prune select
 * runs concurrently on the handle's second stream (lowest priority), forked
 * from and joined back into `stream`; the host waits once per batch of
 * draws (normally once) for that batch's accepted count, while the device
 * keeps working.  When the call
 * returns, the new COO, the source map and the row half of the plan are
 * ordered on `stream`; the workspace is free for the next call at once.  For
 * layers with the deferred scratch in their plan (see snack_query_sizes) the
 * column view is updated from the plan alone (the old view, each weight's new
 * index, the regrown positions in column order) on a third stream of the
 * handle, of the lowest priority, after `stream`'s work, overlapping whatever
 * the caller queues next; the calls that read it wait for it (see Streams),
 * snack_wait_plan orders a stream after it, and snack_destroy waits for it.
 * It reads neither the workspace nor row_out/col_out; row_out and col_out
 * are the layer's pattern from now on.
 * Returns SNACK_ERR_NO_SPACE when fewer than
 * n_prune positions are empty or the draw budget (sized in the workspace
 * query: twice the expected number of draws plus 4096) runs out; the handle's
 * plan is then unchanged.
 */
snack_status snack_restructure(snack_handle h, const int32_t *row, const int32_t *col,
                               const void *val, int64_t n_prune, uint64_t seed, uint64_t step,
                               int32_t *row_out, int32_t *col_out, void *val_out, int32_t *src_out,
                               void *ws, size_t ws_bytes, snack_stream_t stream);

/*
 * Workspace needed by snack_restructure_rows.
 */
snack_status snack_restructure_rows_workspace_size(snack_handle h, int64_t n_per_row, size_t *bytes);

/*
 * Per-row (constant fan-in) restructure, the structured DST variant: Structured
 * RigL (in the pages' list of N:M sparsification work) keeps a constant fan-in;
 * restructuring row by row with equal counts preserves it.  Row r prunes its
 * p_r = min(n_per_row, length of row r) smallest (|val|, k), ranked as in
 * snack_restructure, and regrows p_r columns of row r that were empty before
 * the call, with value +0, from the row's own stream:
 *   base_r = mix(seed ^ mix(step ^ (r * 0xD1B54A32D192ED03))),
 *   draw i: u = mix(base_r + (i + 1) * 0x9E3779B97F4A7C15),
 *   column  = floor(u * in_f / 2^64),
 * accepting a draw whose column was empty in the row and is not yet accepted,
 * until p_r are accepted (64 * n_per_row + 2^20 draws at most per row).  Row
 * 0's stream is snack_restructure's stream.  Every row keeps its count and its
 * offsets, so the outputs (same meaning and rules as snack_restructure) hold
 * row r at the same index range as the input, and only the column view of the
 * plan changes.  Needs ws_bytes >= snack_restructure_rows_workspace_size(h,
 * n_per_row).  With the deferred scratch in the plan (see snack_query_sizes)
 * and out_f * n_per_row within it (one quarter of nnz) and at most 2^20, the
 * kernel also files the regrown positions into column-order buckets in the
 * workspace; the call ranks them on `stream` and then updates the column
 * view from the plan alone on the handle's lowest-priority stream, as
 * snack_restructure does (it reads neither the workspace nor the outputs
 * there).  Otherwise, or when a bucket ran out of slots (not expected), the
 * column view is rebuilt on `stream` before the call returns.
 * Returns SNACK_ERR_UNSUPPORTED when n_per_row > 256 or in_f > 65536, and
 * SNACK_ERR_NO_SPACE when a row has fewer empty columns than it prunes or runs
 * out of draws (the outputs are then undefined and the plan is unchanged).
 * The host waits once for the device's error words.
 */
snack_status snack_restructure_rows(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                                    int64_t n_per_row, uint64_t seed, uint64_t step, int32_t *row_out,
                                    int32_t *col_out, void *val_out, int32_t *src_out, void *ws, size_t ws_bytes,
                                    snack_stream_t stream);

/*
 * Order `stream` after everything the last snack_restructure left running on
 * the handle's own streams (the column-view update of the plan); returns at
 * once, asynchronous like every call.  Use it before timing, freeing or
 * reading anything that the update touches (the plan).  A handle that has
 * not restructured has nothing pending.
 */
snack_status snack_wait_plan(snack_handle h, snack_stream_t stream);

/* Free the handle: its host memory, and the stream, events and pinned word of
 * a handle that has restructured (waits for that stream, so for any pending
 * plan rebuild).  No device memory of the caller is touched.  NULL is allowed. */
void snack_destroy(snack_handle h);

/* Static description of a status code. */
const char *snack_status_string(snack_status st);

/* SNACK_VERSION of the built library. */
int snack_version(void);

/*
 * Kernel trace of the calling host thread (a profiling aid).  While a trace
 * is open, every kernel the library launches from this thread is bracketed by
 * two CUDA events recorded on its stream, in a ring of `capacity` records:
 * the event between two launches keeps the second from starting before the
 * first ends, so a traced kernel's time includes its launch.  Events belong
 * to the device current at snack_trace_start; trace launches on that device
 * only.
 *   snack_trace_start: open a ring of `capacity` >= 1 records (an open trace
 *     is closed first).  SNACK_ERR_INVALID_ARG for capacity < 1,
 *     SNACK_ERR_CUDA when an event cannot be created.
 *   snack_trace_read: wait for the recorded launches to finish and return the
 *     last min(recorded, capacity, max) of them, oldest first: names[i] the
 *     kernel's name as the CUDA runtime gives it (mangled; owned by the
 *     runtime), us[i] the time between its two events in microseconds; *n
 *     the count.  The trace stays open.  SNACK_ERR_INVALID_ARG without an
 *     open trace or for bad pointers.
 *   snack_trace_stop: close the trace and free its events (no-op if none).
 */
snack_status snack_trace_start(int32_t capacity);
snack_status snack_trace_read(const char **names, float *us, int32_t max, int32_t *n);
snack_status snack_trace_stop(void);

#ifdef __cplusplus
}
#endif

#endif /* SNACK_H */
