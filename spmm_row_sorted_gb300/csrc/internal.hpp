// Host-side internals shared by the translation units of libsnack.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"
#include "spmm.cuh"

namespace snack {

// Device pointers into the caller's plan buffer.
struct PlanPtrs {
  int32_t *rp;       // [out_f + 1]   row offsets of the row-sorted COO
  int32_t *tiles_f;  // [(nt_f + 1) * 2] forward merge-path split points
  int32_t *cp;       // [in_f + 1]    column offsets of the column view
  int32_t *tiles_t;  // [(nt_t + 1) * 2] input-gradient split points
  int32_t *row_t;    // [nnz]         row of each column-view entry (not kept up to date when rowt16 exists:
                     //               every reader takes the 16-bit copy then)
  int32_t *src_t;    // [nnz]         storage index of each column-view entry
  uint32_t *flags;   // [64]          validation flags and small device scalars
  uint16_t *col16;   // [nnz]         16-bit copy of col (in_f <= 65536), else null
  uint16_t *rowt16;  // [nnz]         16-bit copy of row_t (out_f <= 65536), else null
  // Incremental update of the column view after a restructure (present when
  // the row and column bits fit 31 together): a second column view, written
  // by the update while the current one is read (the handle swaps the two
  // when the update is queued), and the update's scratch, which must outlive
  // the call because the update runs on a stream of the handle after it returns.
  int32_t *cp_alt, *tiles_t_alt, *row_t_alt, *src_t_alt;
  uint16_t *rowt16_alt;
  uint32_t *newidx;   // [nnz] output index of each stored weight (~0u: pruned)
  uint32_t *gq;       // [cv_pmax] output index of each regrown weight, by acceptance rank
  uint32_t *gc_key;   // [cv_pmax] regrown positions in column order, col << rbits | row
  uint32_t *gc_q;     // [cv_pmax] and their acceptance ranks
  uint32_t *cv_pcnt;  // [in_f] pruned weights per column (written by the restructure's merge)
  uint32_t *cv_ppre;  // [in_f] their exclusive prefix (16-byte aligned)
  void *cv_bnd;       // bounds of the update's tiles of kScanTile entries (32 bytes per tile, and one more)
  int64_t cv_pmax;    // most weights a restructure may prune and still update (else rebuild)
  // Moderately sparse bf16 layers (dense_layer): per 64-column block and row,
  // the stored-position mask (u64) and the storage index of the block's
  // first stored weight (dense.cu, build_tables); else null.
  void *tables;
};

// Words of PlanPtrs::flags: [0] pattern validation, [1] constant fan-in check,
// [kPlanFlagColOk] set when the last restructure's column-order list of the
// regrown positions is complete (its column-view update, which runs after
// the call returns, may write; the word lives in the plan because the caller
// may reuse the workspace by then).
constexpr int kPlanFlagColOk = 2;

struct PlanLayout {
  size_t off_rp, off_tf, off_cp, off_tt, off_rowt, off_srct, off_flags, off_col16, off_rowt16, off_cpa, off_tta,
      off_rowta, off_srcta, off_rowt16a, off_newidx, off_gq, off_gck, off_gcq, off_cvs, off_cvq, off_cvb, off_tab, total;
  bool c16, r16;  // the 16-bit index copies exist
  bool cv;        // the second column view and the incremental update's scratch exist
  int64_t cv_pmax;
  bool dense;     // the tensor-core path's mask and offset tables exist
  TileGeom gf, gt;
};

PlanLayout plan_layout(int32_t out_f, int32_t in_f, int64_t nnz, int bt_max, int n_btiles, bool dense);
PlanPtrs plan_ptrs(const PlanLayout &lay, void *base);
size_t plan_build_ws_bytes(int32_t out_f, int32_t in_f, int64_t nnz);

// Fill the plan for the pattern (row, col).  Asynchronous on s.  `ready`
// names what is already in place: kPlanNothingReady (create),
// kPlanRowsReady (the row offsets and the 16-bit column copy, written by a
// restructure's merge), kPlanRowTilesReady (also the forward tiles: a
// per-row restructure keeps every row's offsets).  With colview = false the
// column view is left alone (a restructure updates it itself).
constexpr int kPlanNothingReady = 0, kPlanRowsReady = 1, kPlanRowTilesReady = 2;
cudaError_t build_plan(int32_t out_f, int32_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
                       const PlanPtrs &p, const TileGeom &gf, const TileGeom &gt, void *ws, cudaStream_t s,
                       int ready, bool colview = true);

// Merge-path split points of a row- or column-offset array (k_tiles).
cudaError_t cut_tiles(const int32_t *ptr, int32_t n_rows, int64_t nnz, const TileGeom &g, int32_t *tiles,
                      cudaStream_t s);

// The second column view and the update's scratch exist when both index
// widths fit 31 bits together; the update takes up to a quarter of nnz.
bool colview_update_ok(int32_t out_f, int32_t in_f, int64_t nnz);

// The column view's first level scatters (row, col) by the column's high 8
// bits when 9..17-bit columns and row + column bits fit 32: then *shift =
// column bits - 8 and the digit of an entry is (col >> shift) & 0xFF, per
// tile of 2048 entries (the histogram is digit-major: [256][tiles]).
bool colview_digits(int32_t out_f, int32_t in_f, int64_t nnz, int *shift);

// *flag = 1 unless rp[r] == r * K for every r <= out_f (a constant fan-in of K).
cudaError_t check_fan_in(const int32_t *rp, int32_t out_f, int32_t K, uint32_t *flag, cudaStream_t s);

// dst[i] = (uint16_t)src[i] for i < n (the plan's 16-bit index copies); nothing when dst is null.
cudaError_t pack16(const int32_t *src, int64_t n, uint16_t *dst, cudaStream_t s);

// flags[0] |= 1 (index out of range), |= 2 (not strictly increasing).
cudaError_t validate_pattern(int32_t out_f, int32_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
                             uint32_t *flag, cudaStream_t s);

// Restructure driver (restructure.cu).
struct RestructureArgs {
  int32_t out_f, in_f;
  int64_t nnz, n_prune;
  snack_dtype val_t;
  uint64_t seed, step;
  const int32_t *row, *col;
  const void *val;
  int32_t *row_out, *col_out;
  void *val_out;
  int32_t *src_out;  // may be null
  // The plan of the input pattern: the draws read its row offsets and 16-bit
  // columns, the merge rewrites them (and the forward tiles) for the output;
  // when `update` is set the column view is updated into the plan's second
  // view on `aux_lo` after the call returns (the caller then swaps the
  // views), else it is rebuilt on s.
  const PlanPtrs *plan;
  TileGeom gf, gt;
  bool update;
  uint32_t *host_counts;  // pinned, mapped host memory, 8 words: a draw chunk's accepted count, table and bucket
                          // overflows, and the acceptance scan's look-back error
  uint32_t *counts_dev;   // the same words' device address (written by a kernel, no copy)
  cudaEvent_t counts_ready;  // recorded after the kernel that writes host_counts
  cudaStream_t aux;          // second stream of the handle (the prune select), lowest priority
  cudaStream_t aux_lo;       // third stream (the deferred column-view update), lowest priority
  cudaEvent_t ev_fork, ev_join, ev_aux;
};
size_t restructure_ws_bytes(int32_t out_f, int32_t in_f, int64_t nnz, int64_t n_prune);
// Returns SNACK_OK, SNACK_ERR_NO_SPACE, SNACK_ERR_WORKSPACE or SNACK_ERR_CUDA;
// *updated is set when the column view was queued into the plan's second
// view (the caller swaps the views).
snack_status run_restructure(const RestructureArgs &a, void *ws, size_t ws_bytes, cudaStream_t s, bool *updated);

// Tensor-core path for moderately sparse bf16 layers (dense.cu): layers with
// >= 8 % of W stored, feature counts multiples of 8 and <= 65536, created
// with max_batch >= kDenseMinBatch; used for calls with batch >=
// kDenseMinBatch whose activations are 16-byte aligned and whose workspace
// holds the path's scratch (snack_query_sizes reserves it).
// Measured on GB300: the 4096^2 bf16 layer at 10 % stored runs its forward
// faster on the tensor cores from batch 16 (25.6 / 27.0 us at batch 16 / 64
// against 29.7 / 38.9 us on the gather kernels).
#ifndef SNACK_DENSE_MIN_BATCH
#define SNACK_DENSE_MIN_BATCH 16
#endif
#ifndef SNACK_DENSE_MIN_DENSITY
#define SNACK_DENSE_MIN_DENSITY 0.08
#endif
constexpr int kDenseMinBatch = SNACK_DENSE_MIN_BATCH;
constexpr double kDenseMinDensity = SNACK_DENSE_MIN_DENSITY;
bool dense_layer(int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch, snack_dtype val_t);
size_t dense_table_bytes(int32_t out_f, int32_t in_f);
cudaError_t build_tables(const int32_t *rp, const uint16_t *col16, int32_t out_f, int32_t in_f, void *tables,
                         cudaStream_t s);
// scratch of one call at `batch` on a device with num_sms SMs (a larger
// num_sms never needs less)
size_t dense_ws_bytes(int32_t out_f, int32_t in_f, int32_t batch, int num_sms);

// Per-row (constant fan-in) restructure (restructure.cu): rows keep their
// counts and offsets; the plan's row offsets and forward tiles stay valid.
struct RowsRestructureArgs {
  int32_t out_f, in_f;
  int64_t nnz, n_per_row;
  snack_dtype val_t;
  uint64_t seed, step;
  const int32_t *rp, *col;
  const void *val;
  int32_t *row_out, *col_out;
  void *val_out;
  int32_t *src_out;   // may be null
  uint16_t *col16;    // plan's 16-bit column copy, or null
  // device words: err[0] nonzero after the kernel when a row cannot be
  // restructured; with plan set also err[1] (a column-order bucket of the
  // regrown positions ran out of slots) and err[2] (the regrown count)
  uint32_t *err;
  // With plan set, the kernel also writes the inputs of the incremental
  // column-view update: each old weight's new index and the pruned weights
  // per column into the plan, the regrown positions into column-order
  // buckets in bws (rows_update_ws_bytes bytes, kAlign-aligned).
  const PlanPtrs *plan = nullptr;
  void *bws = nullptr;
};
// SNACK_OK, SNACK_ERR_UNSUPPORTED (n_per_row > 256 or in_f > 65536) or SNACK_ERR_CUDA; row
// failures are reported through *err.
snack_status run_restructure_rows(const RowsRestructureArgs &a, cudaStream_t s);
// Bytes of the bucket region of a per-row restructure's column-view update;
// 0 when the update does not apply (more regrown weights than the buckets
// take).
size_t rows_update_ws_bytes(int32_t out_f, int64_t n_per_row);
// After run_restructure_rows with plan set: the regrown positions'
// column-order list into the plan, on s (it reads bws; it writes nothing
// when err[0] or err[1] is set).
cudaError_t queue_rows_rank(const RowsRestructureArgs &a, cudaStream_t s);
// After queue_rows_rank, with no row error and no bucket overflow: on s_lo,
// once s reaches ev, the merge of the old column view with the n_grown
// regrown positions into the plan's second view, and that view's tiles.
cudaError_t queue_rows_colview(const RowsRestructureArgs &a, int64_t n_grown, const TileGeom &gt, cudaStream_t s,
                               cudaStream_t s_lo, cudaEvent_t ev);

// Host SplitMix64 (state increment and finaliser of Steele, Lea and Flood 2014).
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ULL;
__host__ __device__ inline uint64_t sm64_finalise(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

}  // namespace snack

struct snack_layer {
  int device;
  int32_t out_f, in_f;
  int64_t nnz;
  int32_t max_batch;
  snack_dtype val_t, act_t;
  snack::PlanLayout lay;
  snack::PlanPtrs p;
  size_t plan_bytes;
  int num_sms;
  uint32_t *host_counts = nullptr;  // restructure read-back (pinned, mapped), made on first use
  uint32_t *host_counts_dev = nullptr;  // its device address
  cudaEvent_t counts_ready = nullptr;
  cudaStream_t aux = nullptr;     // restructure's second stream (its select) and fork/join events, made on first use
  cudaStream_t aux_lo = nullptr;  // and its third stream (lowest priority)
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_aux = nullptr;
  // The column view of the last restructure is updated on `aux_lo` after the
  // call returns; ev_colview marks the end of everything the call left on
  // `aux` and `aux_lo`, and the calls that read the column view make their
  // stream wait for it.
  cudaEvent_t ev_colview = nullptr;
  bool colview_pending = false;
  bool dense = false;   // the layer takes the tensor-core path for wide batches
  int32_t fan_in = 0;   // K when every row holds K stored weights (rows at r * K), else 0
};

namespace snack {
bool dense_call_ok(const snack_layer *h, int32_t batch, const void *act, size_t ws_bytes);
snack_status dense_fwd(snack_layer *h, const void *val, const void *x, int32_t batch, const float *bias, void *y,
                       void *ws, size_t ws_bytes, cudaStream_t s);
snack_status dense_dx(snack_layer *h, const void *val, const void *dy, int32_t batch, void *dx, void *ws,
                      size_t ws_bytes, cudaStream_t s);
snack_status dense_dw(snack_layer *h, const void *x, const void *dy, int32_t batch, float *dw, float *db, void *ws,
                      size_t ws_bytes, cudaStream_t s);
}  // namespace snack
