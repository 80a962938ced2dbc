// The C ABI of libsnack (declared in include/snack.h): argument checks on the
// host, workspace carving, and dispatch to the kernels.  No device memory is
// allocated here; every buffer comes from the caller.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <new>
#include <utility>

#include "internal.hpp"

using namespace snack;

namespace snack {

cudaError_t raise_smem_limit(const void *kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;  // within the default limit of every kernel
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, size_t> granted;
  std::lock_guard<std::mutex> lock(mu);
  size_t &g = granted[std::make_pair(dev, kernel)];
  if (g >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) g = bytes;
  return e;
}

thread_local KernelTrace *g_kernel_trace = nullptr;

}  // namespace snack

namespace {

// The calling thread's trace: the ring's storage and events (created on the
// device current at snack_trace_start).
struct TraceOwner {
  KernelTrace t{};
  ~TraceOwner() { release(); }
  void release() {
    if (t.ev)
      for (int i = 0; i < 2 * t.cap; ++i)
        if (t.ev[i]) cudaEventDestroy(t.ev[i]);
    delete[] t.ev;
    delete[] t.fn;
    t = KernelTrace{};
  }
};
thread_local TraceOwner g_trace_owner;

}  // namespace

namespace {

struct DevGuard {
  int prev = -1;
  bool ok = true;
  explicit DevGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      prev = -1;
      ok = false;
      return;
    }
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DevGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return na && nb && x < y + nb && y < x + na;
}

inline bool dtype_ok(snack_dtype t) { return t == SNACK_F32 || t == SNACK_BF16; }

struct SpmmWs {
  size_t xt, carry, head, total;
};

SpmmWs spmm_ws(int32_t n_src, const TileGeom &tg, const BatchGeom &bg, size_t s_act, int batch) {
  SpmmWs w;
  size_t o = 0;
  w.xt = o;
  if (batch > 1) o += align_up((size_t)n_src * bg.ldx * s_act, kAlign);
  w.carry = o;
  o += align_up((size_t)bg.n_btiles * tg.n_tiles * bg.bt * 4, kAlign);
  w.head = o;
  o += align_up((size_t)bg.n_btiles * tg.n_tiles * bg.bt * 4, kAlign);
  w.total = o;
  return w;
}

struct DwWs {
  size_t xt, dyt, total;
};

DwWs dw_ws(int32_t out_f, int32_t in_f, const BatchGeom &bg, size_t s_act, int batch) {
  DwWs w;
  size_t o = 0;
  w.xt = o;
  if (batch > 1) o += align_up((size_t)in_f * bg.ldx * s_act, kAlign);
  w.dyt = o;
  if (batch > 1) o += align_up((size_t)out_f * bg.ldx * s_act, kAlign);
  w.total = o;
  return w;
}

// fused backward: dY transposed + X transposed + the input-gradient tile partials
struct BwdWs {
  size_t dyt, xt, carry, head, total;
};

BwdWs bwd_ws(int32_t out_f, int32_t in_f, const TileGeom &gt, const BatchGeom &bg, size_t s_act, int batch) {
  BwdWs w;
  size_t o = 0;
  w.dyt = o;
  if (batch > 1) o += align_up((size_t)out_f * bg.ldx * s_act, kAlign);
  w.xt = o;
  if (batch > 1) o += align_up((size_t)in_f * bg.ldx * s_act, kAlign);
  w.carry = o;
  o += align_up((size_t)bg.n_btiles * gt.n_tiles * bg.bt * 4, kAlign);
  w.head = o;
  o += align_up((size_t)bg.n_btiles * gt.n_tiles * bg.bt * 4, kAlign);
  w.total = o;
  return w;
}

size_t ops_ws_bytes(int32_t out_f, int32_t in_f, int batch, snack_dtype act, const PlanLayout &lay) {
  BatchGeom bg = batch_geom(batch, act);
  size_t s = dtype_size(act);
  size_t a = spmm_ws(in_f, lay.gf, bg, s, batch).total;
  size_t b = spmm_ws(out_f, lay.gt, bg, s, batch).total;
  size_t c = dw_ws(out_f, in_f, bg, s, batch).total;
  size_t d = bwd_ws(out_f, in_f, lay.gt, bg, s, batch).total;
  size_t m = a > b ? a : b;
  m = m > c ? m : c;
  return m > d ? m : d;
}

snack_status check_shape(int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch, snack_dtype val_t,
                         snack_dtype act_t) {
  if (out_f < 1 || in_f < 1 || nnz < 0 || nnz >= INT32_MAX) return SNACK_ERR_INVALID_ARG;
  if ((uint64_t)nnz > (uint64_t)out_f * (uint64_t)in_f) return SNACK_ERR_INVALID_ARG;
  if (max_batch < 1 || max_batch > 65535) return SNACK_ERR_INVALID_ARG;
  if (!dtype_ok(val_t) || !dtype_ok(act_t)) return SNACK_ERR_INVALID_ARG;
  if (val_t != act_t) return SNACK_ERR_UNSUPPORTED;
  // the kernels address a feature's batch vector by a 32-bit element offset
  const BatchGeom bg = batch_geom(max_batch, act_t);
  if ((uint64_t)(out_f > in_f ? out_f : in_f) * (uint64_t)bg.ldx > 0xFFFFFFFFull) return SNACK_ERR_UNSUPPORTED;
  return SNACK_OK;
}

#define SNACK_CUDA(x)                              \
  do {                                             \
    if ((x) != cudaSuccess) return SNACK_ERR_CUDA; \
  } while (0)

// Column-view parameters of the small-batch path: rows are the input
// features, the gathered operand is dY [batch][out_f].
SpmmParams small_colview_params(snack_handle h, const void *val, const void *dy, int32_t batch, void *dx) {
  SpmmParams p = {};
  p.n_rows = h->in_f;
  p.n_src = h->out_f;
  p.ptr = h->p.cp;
  p.nnz = h->nnz;
  p.idx = h->p.row_t;
  p.idx16 = h->p.rowt16;
  p.val = val;
  p.val_src = h->p.src_t;
  p.xt = dy;
  p.y = dx;
  p.batch = batch;
  p.act = kActNone;
  return p;
}

template <typename T>
snack_status run_fwd(snack_handle h, const int32_t *col, const void *val, const void *x, int32_t batch,
                     const float *bias, void *y, void *ws, size_t ws_bytes, cudaStream_t s, int act = kActNone,
                     void *pre_out = nullptr) {
  if (small_path_ok(batch, h->in_f, sizeof(T))) {  // one launch, X read batch-major
    SpmmParams p = {};
    p.n_rows = h->out_f;
    p.n_src = h->in_f;
    p.ptr = h->p.rp;
    p.nnz = h->nnz;
    p.idx = col;
    p.idx16 = h->p.col16;
    p.val = val;
    p.xt = x;
    p.bias = bias;
    p.y = y;
    p.batch = batch;
    p.act = act;
    p.pre_out = pre_out;
    SNACK_CUDA(run_spmm_small<T>(p, false, false, h->num_sms, s));
    return SNACK_OK;
  }
  BatchGeom bg = batch_geom(batch, h->act_t);
  SpmmWs W = spmm_ws(h->in_f, h->lay.gf, bg, sizeof(T), batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const T *xt = reinterpret_cast<const T *>(x);
  if (batch > 1) {
    T *xt_w = reinterpret_cast<T *>(b + W.xt);
    SNACK_CUDA(run_transpose<T>(reinterpret_cast<const T *>(x), batch, h->in_f, xt_w, bg.ldx, s));
    xt = xt_w;
  }
  SpmmParams p = {};
  p.n_rows = h->out_f;
  p.n_src = h->in_f;
  p.ptr = h->p.rp;
  p.tiles = h->p.tiles_f;
  p.tg = h->lay.gf;
  p.nnz = h->nnz;
  p.idx = col;
  p.idx16 = h->p.col16;
  p.val = val;
  p.val_src = nullptr;
  p.xt = xt;
  p.bias = bias;
  p.y = y;
  p.batch = batch;
  p.carry = reinterpret_cast<float *>(b + W.carry);
  p.head = reinterpret_cast<float *>(b + W.head);
  p.xt_dw = nullptr;
  p.dw = nullptr;
  p.act = act;
  p.pre_in = nullptr;
  p.pre_out = pre_out;
  if (h->fan_in > 0) {  // constant fan-in: whole rows per warp, no split rows
    SNACK_CUDA(run_ell<T>(p, bg, h->fan_in, s));
    return SNACK_OK;
  }
  SNACK_CUDA(run_spmm<T>(p, bg, false, false, s));
  return SNACK_OK;
}

template <typename T>
snack_status run_dx(snack_handle h, const void *val, const void *dy, int32_t batch, void *dx, void *ws,
                    size_t ws_bytes, cudaStream_t s, int act = kActNone, const void *pre_in = nullptr) {
  if (small_path_ok(batch, h->out_f, sizeof(T))) {  // one launch over the column view, dY read batch-major
    SpmmParams p = small_colview_params(h, val, dy, batch, dx);
    p.act = act;
    p.pre_in = pre_in;
    SNACK_CUDA(run_spmm_small<T>(p, true, false, h->num_sms, s));
    return SNACK_OK;
  }
  BatchGeom bg = batch_geom(batch, h->act_t);
  SpmmWs W = spmm_ws(h->out_f, h->lay.gt, bg, sizeof(T), batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const T *dyt = reinterpret_cast<const T *>(dy);
  if (batch > 1) {
    T *w = reinterpret_cast<T *>(b + W.xt);
    SNACK_CUDA(run_transpose<T>(reinterpret_cast<const T *>(dy), batch, h->out_f, w, bg.ldx, s));
    dyt = w;
  }
  SpmmParams p = {};
  p.n_rows = h->in_f;
  p.n_src = h->out_f;
  p.ptr = h->p.cp;
  p.tiles = h->p.tiles_t;
  p.tg = h->lay.gt;
  p.nnz = h->nnz;
  p.idx = h->p.row_t;
  p.idx16 = h->p.rowt16;
  p.val = val;
  p.val_src = h->p.src_t;
  p.xt = dyt;
  p.bias = nullptr;
  p.y = dx;
  p.batch = batch;
  p.carry = reinterpret_cast<float *>(b + W.carry);
  p.head = reinterpret_cast<float *>(b + W.head);
  p.xt_dw = nullptr;
  p.dw = nullptr;
  p.act = act;
  p.pre_in = pre_in;
  p.pre_out = nullptr;
  SNACK_CUDA(run_spmm<T>(p, bg, true, false, s));
  return SNACK_OK;
}

template <typename T>
snack_status run_dw(snack_handle h, const int32_t *row, const int32_t *col, const void *x, const void *dy,
                    int32_t batch, float *dw, float *db, void *ws, size_t ws_bytes, cudaStream_t s) {
  if (small_dw_flat_ok(batch, h->nnz)) {  // one flat pass over the stored weights
    SNACK_CUDA(run_sddmm_small<T>(h->nnz, row, col, h->out_f, h->in_f, reinterpret_cast<const T *>(x),
                                  reinterpret_cast<const T *>(dy), batch, dw, db, h->num_sms, s));
    return SNACK_OK;
  }
  if (small_path_ok(batch, h->out_f, sizeof(T))) {  // the column-view pass with dW and db only
    SpmmParams p = small_colview_params(h, nullptr, dy, batch, nullptr);
    p.xt_dw = x;
    p.dw = dw;
    p.db = db;
    SNACK_CUDA(run_spmm_small<T>(p, true, true, h->num_sms, s));
    return SNACK_OK;
  }
  BatchGeom bg = batch_geom(batch, h->act_t);
  DwWs W = dw_ws(h->out_f, h->in_f, bg, sizeof(T), batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const T *xt = reinterpret_cast<const T *>(x);
  const T *dyt = reinterpret_cast<const T *>(dy);
  if (h->nnz == 0) {
    if (db) SNACK_CUDA(run_colsum<T>(reinterpret_cast<const T *>(dy), batch, h->out_f, db, s));
    return SNACK_OK;
  }
  bool db_done = false;
  if (batch > 1) {
    T *a = reinterpret_cast<T *>(b + W.xt);
    T *c = reinterpret_cast<T *>(b + W.dyt);
    TransposePair<T> tp{reinterpret_cast<const T *>(dy), reinterpret_cast<const T *>(x), c, a, h->out_f, h->in_f,
                        bg.ldx <= 32 ? db : nullptr};
    SNACK_CUDA(run_transpose2<T>(tp, batch, bg.ldx, s));
    db_done = tp.db0 != nullptr;
    xt = a;
    dyt = c;
  }
  // db from the feature-major dY (contiguous per output feature), unless the
  // transpose already summed a single batch tile
  if (db && !db_done) SNACK_CUDA(run_rowsum_t<T>(dyt, batch > 1 ? bg.ldx : 1, batch, h->out_f, db, s));
  SNACK_CUDA(run_sddmm<T>(h->nnz, row, col, h->out_f, h->in_f, xt, dyt, bg, dw, h->num_sms, s));
  return SNACK_OK;
}

// Fused backward: one pass over the column view gives dX and dW (one batch
// tile); wider batches run the input gradient and the SDDMM separately, over
// one transpose of dY and X.
template <typename T>
snack_status run_bwd(snack_handle h, const int32_t *row, const int32_t *col, const void *val, const void *x,
                     const void *dy, int32_t batch, void *dx, float *dw, float *db, void *ws, size_t ws_bytes,
                     cudaStream_t s) {
  if (small_path_ok(batch, h->out_f, sizeof(T))) {  // dX, dW and db in one launch
    SpmmParams p = small_colview_params(h, val, dy, batch, dx);
    p.xt_dw = x;
    p.dw = dw;
    p.db = db;
    SNACK_CUDA(run_spmm_small<T>(p, true, true, h->num_sms, s));
    return SNACK_OK;
  }
  BatchGeom bg = batch_geom(batch, h->act_t);
  if (h->nnz == 0) {
    snack_status st = run_dx<T>(h, val, dy, batch, dx, ws, ws_bytes, s);
    if (st != SNACK_OK) return st;
    return run_dw<T>(h, row, col, x, dy, batch, dw, db, ws, ws_bytes, s);
  }
  // one batch tile: dX and dW in one pass over the column view; wider
  // batches: the input gradient's tiles, then the SDDMM, both reading the
  // same transposed dY (and the SDDMM the transposed X)
  const bool fused = bg.n_btiles == 1;
  BwdWs W = bwd_ws(h->out_f, h->in_f, h->lay.gt, bg, sizeof(T), batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const T *dyt = reinterpret_cast<const T *>(dy);
  const T *xt = reinterpret_cast<const T *>(x);
  bool db_done = false;
  if (batch > 1) {
    T *a = reinterpret_cast<T *>(b + W.dyt);
    T *c = reinterpret_cast<T *>(b + W.xt);
    TransposePair<T> tp{reinterpret_cast<const T *>(dy), reinterpret_cast<const T *>(x), a, c, h->out_f, h->in_f,
                        bg.ldx <= 32 ? db : nullptr};
    SNACK_CUDA(run_transpose2<T>(tp, batch, bg.ldx, s));
    db_done = tp.db0 != nullptr;
    dyt = a;
    xt = c;
  }
  if (db && !db_done) SNACK_CUDA(run_rowsum_t<T>(dyt, batch > 1 ? bg.ldx : 1, batch, h->out_f, db, s));
  SpmmParams p = {};
  p.n_rows = h->in_f;
  p.n_src = h->out_f;
  p.ptr = h->p.cp;
  p.tiles = h->p.tiles_t;
  p.tg = h->lay.gt;
  p.nnz = h->nnz;
  p.idx = h->p.row_t;
  p.idx16 = h->p.rowt16;
  p.val = val;
  p.val_src = h->p.src_t;
  p.xt = dyt;
  p.bias = nullptr;
  p.y = dx;
  p.batch = batch;
  p.carry = reinterpret_cast<float *>(b + W.carry);
  p.head = reinterpret_cast<float *>(b + W.head);
  p.xt_dw = fused ? xt : nullptr;
  p.dw = fused ? dw : nullptr;
  p.act = kActNone;
  p.pre_in = nullptr;
  p.pre_out = nullptr;
  SNACK_CUDA(run_spmm<T>(p, bg, true, fused, s));
  if (!fused) SNACK_CUDA(run_sddmm<T>(h->nnz, row, col, h->out_f, h->in_f, xt, dyt, bg, dw, h->num_sms, s));
  return SNACK_OK;
}

// Pinned host words and an event for reading small device results back
// (made on a handle's first restructure).
bool readback_ready(snack_handle h) {
  if (!h->host_counts) {  // mapped, so a kernel writes the words and the host reads them with no copy
    void *hp = nullptr, *dp = nullptr;
    if (cudaHostAlloc(&hp, 8 * sizeof(uint32_t), cudaHostAllocMapped) != cudaSuccess) return false;
    if (cudaHostGetDevicePointer(&dp, hp, 0) != cudaSuccess || !dp) {
      cudaFreeHost(hp);
      return false;
    }
    h->host_counts = reinterpret_cast<uint32_t *>(hp);
    h->host_counts_dev = reinterpret_cast<uint32_t *>(dp);
  }
  if (!h->counts_ready && cudaEventCreateWithFlags(&h->counts_ready, cudaEventDisableTiming) != cudaSuccess)
    return false;
  return true;
}

// The restructures' streams and events, made on first use.
bool restructure_streams(snack_handle h) {
  if (!h->ev_fork && cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess) return false;
  if (!h->ev_join && cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) return false;
  if (!h->ev_colview && cudaEventCreateWithFlags(&h->ev_colview, cudaEventDisableTiming) != cudaSuccess) return false;
  if (!h->ev_aux && cudaEventCreateWithFlags(&h->ev_aux, cudaEventDisableTiming) != cudaSuccess) return false;
  if (!h->aux || !h->aux_lo) {
    // The regrow branch (draws, acceptance, sort) is the longer of the two
    // that meet at the merge and runs on the caller's stream; the select
    // beside it gets the second stream at the lowest priority, so the
    // regrow's blocks are scheduled ahead of the select's when both wait for
    // SMs.  The column-view update that runs on after the call returns gets
    // the third, also of the lowest priority, so the caller's next calls go
    // ahead of it where their streams have a higher priority.
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
    (void)greatest;
    if (!h->aux && cudaStreamCreateWithPriority(&h->aux, cudaStreamNonBlocking, least) != cudaSuccess) return false;
    if (!h->aux_lo && cudaStreamCreateWithPriority(&h->aux_lo, cudaStreamNonBlocking, least) != cudaSuccess)
      return false;
  }
  return true;
}

// The column view of a restructured handle may still be updating on a
// stream of the handle: order `s` after it.  The forward reads only the
// row half of the plan and does not wait.
bool wait_colview(snack_handle h, cudaStream_t s) {
  return !h->colview_pending || cudaStreamWaitEvent(s, h->ev_colview, 0) == cudaSuccess;
}

snack_status common_call_checks(snack_handle h, int32_t batch, void *ws) {
  if (!h) return SNACK_ERR_INVALID_ARG;
  if (batch < 0 || batch > h->max_batch) return SNACK_ERR_INVALID_ARG;
  if (batch > 0 && (!ws || !aligned(ws, kAlign))) return SNACK_ERR_INVALID_ARG;
  return SNACK_OK;
}

}  // namespace

extern "C" {

snack_status snack_query_sizes(int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch, snack_dtype val_t,
                               snack_dtype act_t, size_t *plan_bytes, size_t *workspace_bytes) {
  snack_status st = check_shape(out_f, in_f, nnz, max_batch, val_t, act_t);
  if (st != SNACK_OK) return st;
  const BatchGeom mbg = batch_geom(max_batch, act_t);
  PlanLayout lay = plan_layout(out_f, in_f, nnz, mbg.bt, mbg.n_btiles, dense_layer(out_f, in_f, nnz, max_batch, val_t));
  if (plan_bytes) *plan_bytes = lay.total;
  if (workspace_bytes) {
    size_t a = ops_ws_bytes(out_f, in_f, max_batch, act_t, lay);
    size_t b = plan_build_ws_bytes(out_f, in_f, nnz);
    // the tensor-core path's scratch at max_batch on any GPU (more SMs never need less)
    size_t c = dense_layer(out_f, in_f, nnz, max_batch, val_t) ? dense_ws_bytes(out_f, in_f, max_batch, 1 << 20) : 0;
    a = a > b ? a : b;
    *workspace_bytes = a > c ? a : c;
  }
  return SNACK_OK;
}

snack_status snack_create(snack_handle *out_handle, int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch,
                          snack_dtype val_t, snack_dtype act_t, const int32_t *row, const int32_t *col, void *plan,
                          size_t plan_bytes, void *ws, size_t ws_bytes, int validate, snack_stream_t stream) {
  if (!out_handle) return SNACK_ERR_INVALID_ARG;
  *out_handle = nullptr;
  snack_status st = check_shape(out_f, in_f, nnz, max_batch, val_t, act_t);
  if (st != SNACK_OK) return st;
  if (nnz > 0 && (!row || !col)) return SNACK_ERR_INVALID_ARG;
  if (!plan || !aligned(plan, kAlign) || !ws || !aligned(ws, kAlign)) return SNACK_ERR_INVALID_ARG;
  const BatchGeom mbg = batch_geom(max_batch, act_t);
  PlanLayout lay = plan_layout(out_f, in_f, nnz, mbg.bt, mbg.n_btiles, dense_layer(out_f, in_f, nnz, max_batch, val_t));
  if (plan_bytes < lay.total) return SNACK_ERR_WORKSPACE;
  if (ws_bytes < plan_build_ws_bytes(out_f, in_f, nnz)) return SNACK_ERR_WORKSPACE;
  int dev = 0;
  SNACK_CUDA(cudaGetDevice(&dev));
  int sms = 0;
  SNACK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  PlanPtrs p = plan_ptrs(lay, plan);
  SNACK_CUDA(cudaMemsetAsync(p.flags, 0, sizeof(uint32_t) * 64, s));  // every flag word starts clear
  if (validate) {
    SNACK_CUDA(validate_pattern(out_f, in_f, nnz, row, col, p.flags, s));
    uint32_t flag = 0;
    SNACK_CUDA(cudaMemcpyAsync(&flag, p.flags, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    SNACK_CUDA(cudaStreamSynchronize(s));
    if (flag & 1u) return SNACK_ERR_OUT_OF_RANGE;
    if (flag & 2u) return SNACK_ERR_UNSORTED;
  }
  SNACK_CUDA(build_plan(out_f, in_f, nnz, row, col, p, lay.gf, lay.gt, ws, s, kPlanNothingReady));
  // a constant fan-in (every row K stored weights) lets the forward take whole
  // rows per warp: checked on the device and read back once
  int32_t fan_in = 0;
#ifndef SNACK_NO_FAN_IN_PATH  // a comparison build: every layer takes the general kernels
  if (nnz > 0 && nnz % out_f == 0) {
    const int32_t K = (int32_t)(nnz / out_f);
    SNACK_CUDA(check_fan_in(p.rp, out_f, K, p.flags + 1, s));
    uint32_t bad = 1;
    SNACK_CUDA(cudaMemcpyAsync(&bad, p.flags + 1, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    SNACK_CUDA(cudaStreamSynchronize(s));
    fan_in = bad ? 0 : K;
  }
#endif
  snack_layer *h = new (std::nothrow) snack_layer;
  if (!h) return SNACK_ERR_INVALID_ARG;
  h->device = dev;
  h->out_f = out_f;
  h->in_f = in_f;
  h->nnz = nnz;
  h->max_batch = max_batch;
  h->val_t = val_t;
  h->act_t = act_t;
  h->lay = lay;
  h->p = p;
  h->plan_bytes = plan_bytes;
  h->num_sms = sms > 0 ? sms : 1;
  h->dense = lay.dense;
  h->fan_in = fan_in;
  *out_handle = h;
  return SNACK_OK;
}

snack_status snack_spmm_fwd(snack_handle h, const int32_t *row, const int32_t *col, const void *val, const void *x,
                            int32_t batch, const float *bias, void *y, void *ws, size_t ws_bytes,
                            snack_stream_t stream) {
  snack_status st = common_call_checks(h, batch, ws);
  if (st != SNACK_OK) return st;
  (void)row;
  if (batch == 0) return SNACK_OK;
  if (!x || !y || (h->nnz > 0 && (!col || !val))) return SNACK_ERR_INVALID_ARG;
  const size_t s_act = dtype_size(h->act_t);
  if (overlap(y, (size_t)batch * h->out_f * s_act, x, (size_t)batch * h->in_f * s_act)) return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dense_call_ok(h, batch, x, ws_bytes)) return dense_fwd(h, val, x, batch, bias, y, ws, ws_bytes, s);
  if (h->act_t == SNACK_BF16) return run_fwd<bf16>(h, col, val, x, batch, bias, y, ws, ws_bytes, s);
  return run_fwd<float>(h, col, val, x, batch, bias, y, ws, ws_bytes, s);
}

snack_status snack_spmm_dx(snack_handle h, const int32_t *row, const int32_t *col, const void *val, const void *dy,
                           int32_t batch, void *dx, void *ws, size_t ws_bytes, snack_stream_t stream) {
  snack_status st = common_call_checks(h, batch, ws);
  if (st != SNACK_OK) return st;
  (void)row;
  (void)col;
  if (batch == 0) return SNACK_OK;
  if (!dy || !dx || (h->nnz > 0 && !val)) return SNACK_ERR_INVALID_ARG;
  const size_t s_act = dtype_size(h->act_t);
  if (overlap(dx, (size_t)batch * h->in_f * s_act, dy, (size_t)batch * h->out_f * s_act)) return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wait_colview(h, s)) return SNACK_ERR_CUDA;
  if (dense_call_ok(h, batch, dy, ws_bytes)) return dense_dx(h, val, dy, batch, dx, ws, ws_bytes, s);
  if (h->act_t == SNACK_BF16) return run_dx<bf16>(h, val, dy, batch, dx, ws, ws_bytes, s);
  return run_dx<float>(h, val, dy, batch, dx, ws, ws_bytes, s);
}

snack_status snack_sddmm_dw(snack_handle h, const int32_t *row, const int32_t *col, const void *x, const void *dy,
                            int32_t batch, float *dw, float *db, void *ws, size_t ws_bytes, snack_stream_t stream) {
  snack_status st = common_call_checks(h, batch, ws);
  if (st != SNACK_OK) return st;
  if (h->nnz > 0 && (!row || !col || !dw)) return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wait_colview(h, s)) return SNACK_ERR_CUDA;
  if (batch == 0) {  // empty sums
    if (h->nnz > 0) SNACK_CUDA(cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)h->nnz, s));
    if (db) SNACK_CUDA(cudaMemsetAsync(db, 0, sizeof(float) * (size_t)h->out_f, s));
    return SNACK_OK;
  }
  if (!x || !dy) return SNACK_ERR_INVALID_ARG;
  if (dense_call_ok(h, batch, dy, ws_bytes)) return dense_dw(h, x, dy, batch, dw, db, ws, ws_bytes, s);
  if (h->act_t == SNACK_BF16) return run_dw<bf16>(h, row, col, x, dy, batch, dw, db, ws, ws_bytes, s);
  return run_dw<float>(h, row, col, x, dy, batch, dw, db, ws, ws_bytes, s);
}

snack_status snack_spmm_fwd_gelu(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                                 const void *x, int32_t batch, const float *bias, void *y_pre, void *y, void *ws,
                                 size_t ws_bytes, snack_stream_t stream) {
  snack_status st = common_call_checks(h, batch, ws);
  if (st != SNACK_OK) return st;
  (void)row;
  if (batch == 0) return SNACK_OK;
  if (!x || !y || (h->nnz > 0 && (!col || !val))) return SNACK_ERR_INVALID_ARG;
  const size_t s_act = dtype_size(h->act_t);
  const size_t ny = (size_t)batch * h->out_f * s_act, nx = (size_t)batch * h->in_f * s_act;
  if (overlap(y, ny, x, nx) || (y_pre && (overlap(y_pre, ny, x, nx) || overlap(y_pre, ny, y, ny))))
    return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (h->act_t == SNACK_BF16) return run_fwd<bf16>(h, col, val, x, batch, bias, y, ws, ws_bytes, s, kActGelu, y_pre);
  return run_fwd<float>(h, col, val, x, batch, bias, y, ws, ws_bytes, s, kActGelu, y_pre);
}

snack_status snack_spmm_dx_gelu(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                                const void *dy, int32_t batch, const void *x_pre, void *dx, void *ws, size_t ws_bytes,
                                snack_stream_t stream) {
  snack_status st = common_call_checks(h, batch, ws);
  if (st != SNACK_OK) return st;
  (void)row;
  (void)col;
  if (batch == 0) return SNACK_OK;
  if (!dy || !dx || !x_pre || (h->nnz > 0 && !val)) return SNACK_ERR_INVALID_ARG;
  const size_t s_act = dtype_size(h->act_t);
  const size_t nd = (size_t)batch * h->in_f * s_act, ny = (size_t)batch * h->out_f * s_act;
  if (overlap(dx, nd, dy, ny) || overlap(dx, nd, x_pre, nd)) return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wait_colview(h, s)) return SNACK_ERR_CUDA;
  if (h->act_t == SNACK_BF16) return run_dx<bf16>(h, val, dy, batch, dx, ws, ws_bytes, s, kActGeluGrad, x_pre);
  return run_dx<float>(h, val, dy, batch, dx, ws, ws_bytes, s, kActGeluGrad, x_pre);
}

snack_status snack_backward(snack_handle h, const int32_t *row, const int32_t *col, const void *val, const void *x,
                            const void *dy, int32_t batch, void *dx, float *dw, float *db, void *ws, size_t ws_bytes,
                            snack_stream_t stream) {
  snack_status st = common_call_checks(h, batch, ws);
  if (st != SNACK_OK) return st;
  if (h->nnz > 0 && (!row || !col || !val || !dw)) return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wait_colview(h, s)) return SNACK_ERR_CUDA;
  if (batch == 0) {  // empty sums
    if (h->nnz > 0) SNACK_CUDA(cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)h->nnz, s));
    if (db) SNACK_CUDA(cudaMemsetAsync(db, 0, sizeof(float) * (size_t)h->out_f, s));
    return SNACK_OK;
  }
  if (!x || !dy || !dx) return SNACK_ERR_INVALID_ARG;
  const size_t s_act = dtype_size(h->act_t);
  if (overlap(dx, (size_t)batch * h->in_f * s_act, dy, (size_t)batch * h->out_f * s_act) ||
      overlap(dx, (size_t)batch * h->in_f * s_act, x, (size_t)batch * h->in_f * s_act))
    return SNACK_ERR_INVALID_ARG;
  if (dense_call_ok(h, batch, dy, ws_bytes)) {
    snack_status r = dense_dx(h, val, dy, batch, dx, ws, ws_bytes, s);
    return r != SNACK_OK ? r : dense_dw(h, x, dy, batch, dw, db, ws, ws_bytes, s);
  }
  if (h->act_t == SNACK_BF16) return run_bwd<bf16>(h, row, col, val, x, dy, batch, dx, dw, db, ws, ws_bytes, s);
  return run_bwd<float>(h, row, col, val, x, dy, batch, dx, dw, db, ws, ws_bytes, s);
}

snack_status snack_restructure_workspace_size(snack_handle h, int64_t n_prune, size_t *bytes) {
  if (!h || !bytes || n_prune < 0 || n_prune > h->nnz) return SNACK_ERR_INVALID_ARG;
  *bytes = restructure_ws_bytes(h->out_f, h->in_f, h->nnz, n_prune);
  return SNACK_OK;
}

snack_status snack_restructure(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                               int64_t n_prune, uint64_t seed, uint64_t step, int32_t *row_out, int32_t *col_out,
                               void *val_out, int32_t *src_out, void *ws, size_t ws_bytes, snack_stream_t stream) {
  if (!h || n_prune < 0 || n_prune > h->nnz) return SNACK_ERR_INVALID_ARG;
  const int64_t nnz = h->nnz;
  if (!ws || !aligned(ws, kAlign)) return SNACK_ERR_INVALID_ARG;
  if (nnz > 0 && (!row || !col || !val || !row_out || !col_out || !val_out)) return SNACK_ERR_INVALID_ARG;
  const uint64_t n_pos = (uint64_t)h->out_f * (uint64_t)h->in_f;
  if ((uint64_t)n_prune > n_pos - (uint64_t)nnz) return SNACK_ERR_NO_SPACE;
  const size_t n4 = 4 * (size_t)nnz, nv = dtype_size(h->val_t) * (size_t)nnz;
  const void *ins[3] = {row, col, val};
  const size_t in_sz[3] = {n4, n4, nv};
  const void *outs[4] = {row_out, col_out, val_out, src_out};
  const size_t out_sz[4] = {n4, n4, nv, src_out ? n4 : 0};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], out_sz[i], ins[j], in_sz[j])) return SNACK_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], out_sz[i], outs[j], out_sz[j])) return SNACK_ERR_INVALID_ARG;
  }
  if (ws_bytes < restructure_ws_bytes(h->out_f, h->in_f, nnz, n_prune)) return SNACK_ERR_WORKSPACE;
  if (nnz == 0) return SNACK_OK;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wait_colview(h, s)) return SNACK_ERR_CUDA;
  RestructureArgs a;
  a.out_f = h->out_f;
  a.in_f = h->in_f;
  a.nnz = nnz;
  a.n_prune = n_prune;
  a.val_t = h->val_t;
  a.seed = seed;
  a.step = step;
  a.row = row;
  a.col = col;
  a.val = val;
  a.row_out = row_out;
  a.col_out = col_out;
  a.val_out = val_out;
  a.src_out = src_out;
  a.plan = &h->p;
  a.gf = h->lay.gf;
  a.gt = h->lay.gt;
  a.update = h->lay.cv && n_prune <= h->lay.cv_pmax;
  if (!readback_ready(h) || !restructure_streams(h)) return SNACK_ERR_CUDA;
  a.host_counts = h->host_counts;
  a.counts_dev = h->host_counts_dev;
  a.counts_ready = h->counts_ready;
  a.aux = h->aux;
  a.aux_lo = h->aux_lo;
  a.ev_fork = h->ev_fork;
  a.ev_join = h->ev_join;
  a.ev_aux = h->ev_aux;
  bool updated = false;
  snack_status st = run_restructure(a, ws, ws_bytes, s, &updated);
  if (st == SNACK_OK) h->fan_in = 0;  // regrowth lands in any row: row counts change
  if (updated) {  // the new column view is being written into the second view: it becomes the current one
    std::swap(h->p.cp, h->p.cp_alt);
    std::swap(h->p.tiles_t, h->p.tiles_t_alt);
    std::swap(h->p.row_t, h->p.row_t_alt);
    std::swap(h->p.src_t, h->p.src_t_alt);
    std::swap(h->p.rowt16, h->p.rowt16_alt);
  }
  // Whatever is still queued on the second and third streams (the
  // column-view update, or work an error left behind) is what the
  // column-view readers wait for.
  if (cudaEventRecord(h->ev_aux, h->aux) != cudaSuccess || cudaStreamWaitEvent(h->aux_lo, h->ev_aux, 0) != cudaSuccess ||
      cudaEventRecord(h->ev_colview, h->aux_lo) != cudaSuccess) {
    cudaStreamSynchronize(h->aux);
    cudaStreamSynchronize(h->aux_lo);
    h->colview_pending = false;
    return SNACK_ERR_CUDA;
  }
  h->colview_pending = true;
  return st;
}

snack_status snack_restructure_rows_workspace_size(snack_handle h, int64_t n_per_row, size_t *bytes) {
  if (!h || !bytes || n_per_row < 0) return SNACK_ERR_INVALID_ARG;
  *bytes = kAlign + std::max(plan_build_ws_bytes(h->out_f, h->in_f, h->nnz), rows_update_ws_bytes(h->out_f, n_per_row));
  return SNACK_OK;
}

snack_status snack_restructure_rows(snack_handle h, const int32_t *row, const int32_t *col, const void *val,
                                    int64_t n_per_row, uint64_t seed, uint64_t step, int32_t *row_out,
                                    int32_t *col_out, void *val_out, int32_t *src_out, void *ws, size_t ws_bytes,
                                    snack_stream_t stream) {
  if (!h || n_per_row < 0) return SNACK_ERR_INVALID_ARG;
  if (n_per_row > 256 || h->in_f > 65536) return SNACK_ERR_UNSUPPORTED;
  const int64_t nnz = h->nnz;
  if (!ws || !aligned(ws, kAlign)) return SNACK_ERR_INVALID_ARG;
  if (nnz > 0 && (!row || !col || !val || !row_out || !col_out || !val_out)) return SNACK_ERR_INVALID_ARG;
  const size_t n4 = 4 * (size_t)nnz, nv = dtype_size(h->val_t) * (size_t)nnz;
  const void *ins[3] = {row, col, val};
  const size_t in_sz[3] = {n4, n4, nv};
  const void *outs[4] = {row_out, col_out, val_out, src_out};
  const size_t out_sz[4] = {n4, n4, nv, src_out ? n4 : 0};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], out_sz[i], ins[j], in_sz[j])) return SNACK_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], out_sz[i], outs[j], out_sz[j])) return SNACK_ERR_INVALID_ARG;
  }
  if (ws_bytes < kAlign + plan_build_ws_bytes(h->out_f, h->in_f, nnz)) return SNACK_ERR_WORKSPACE;
  if (nnz == 0) return SNACK_OK;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  // Every row keeps its length, so the row view stays; the column view is
  // updated from the old one (after the call returns, on the lowest-priority
  // stream) where the plan keeps a second view and the workspace holds the
  // buckets of the regrown positions, else rebuilt before the call returns.
  const size_t upd_bytes = rows_update_ws_bytes(h->out_f, n_per_row);
  const bool update = h->lay.cv && (int64_t)h->out_f * n_per_row <= h->lay.cv_pmax && upd_bytes > 0 &&
                      ws_bytes >= kAlign + upd_bytes;
  if (!readback_ready(h) || (update && !restructure_streams(h))) return SNACK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wait_colview(h, s)) return SNACK_ERR_CUDA;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  RowsRestructureArgs a;
  a.out_f = h->out_f;
  a.in_f = h->in_f;
  a.nnz = nnz;
  a.n_per_row = n_per_row;
  a.val_t = h->val_t;
  a.seed = seed;
  a.step = step;
  a.rp = h->p.rp;
  a.col = col;
  a.val = val;
  a.row_out = row_out;
  a.col_out = col_out;
  a.val_out = val_out;
  a.src_out = src_out;
  a.col16 = h->p.col16;
  a.err = reinterpret_cast<uint32_t *>(b);
  if (update) {
    a.plan = &h->p;
    a.bws = b + kAlign;
  }
  snack_status st = run_restructure_rows(a, s);
  if (st != SNACK_OK) return st;
  const int n_words = update ? 3 : 1;
  SNACK_CUDA(cudaMemcpyAsync(h->host_counts, a.err, sizeof(uint32_t) * n_words, cudaMemcpyDeviceToHost, s));
  SNACK_CUDA(cudaEventRecord(h->counts_ready, s));
  // the column-order list runs while the host waits for the words (it
  // writes nothing if they say the update will not be taken)
  if (update) SNACK_CUDA(queue_rows_rank(a, s));
  SNACK_CUDA(cudaEventSynchronize(h->counts_ready));
  if (h->host_counts[0]) {
    // the rows that finished wrote their new columns into the plan's 16-bit
    // copy: put back the input's, so the plan still serves (row, col)
    SNACK_CUDA(pack16(col, nnz, h->p.col16, s));
    return SNACK_ERR_NO_SPACE;
  }
  if (update && !h->host_counts[1]) {
    if (h->p.tables && h->p.col16) SNACK_CUDA(build_tables(h->p.rp, h->p.col16, h->out_f, h->in_f, h->p.tables, s));
    const cudaError_t e = queue_rows_colview(a, (int64_t)h->host_counts[2], h->lay.gt, s, h->aux_lo, h->ev_fork);
    if (e == cudaSuccess) {  // the second view becomes the current one
      std::swap(h->p.cp, h->p.cp_alt);
      std::swap(h->p.tiles_t, h->p.tiles_t_alt);
      std::swap(h->p.row_t, h->p.row_t_alt);
      std::swap(h->p.src_t, h->p.src_t_alt);
      std::swap(h->p.rowt16, h->p.rowt16_alt);
    }
    if (e != cudaSuccess || cudaEventRecord(h->ev_colview, h->aux_lo) != cudaSuccess) {
      cudaStreamSynchronize(h->aux_lo);
      h->colview_pending = false;
      return SNACK_ERR_CUDA;
    }
    h->colview_pending = true;
    return SNACK_OK;
  }
  SNACK_CUDA(build_plan(h->out_f, h->in_f, nnz, row_out, col_out, h->p, h->lay.gf, h->lay.gt, b + kAlign, s,
                        kPlanRowTilesReady));
  return SNACK_OK;
}

snack_status snack_wait_plan(snack_handle h, snack_stream_t stream) {
  if (!h) return SNACK_ERR_INVALID_ARG;
  DevGuard g(h->device);
  if (!g.ok) return SNACK_ERR_CUDA;
  return wait_colview(h, reinterpret_cast<cudaStream_t>(stream)) ? SNACK_OK : SNACK_ERR_CUDA;
}

void snack_destroy(snack_handle h) {
  if (!h) return;
  if (h->counts_ready || h->aux || h->aux_lo || h->ev_fork || h->ev_join || h->ev_aux || h->ev_colview) {
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(h->device);
    if (h->aux) {
      cudaStreamSynchronize(h->aux);
      cudaStreamDestroy(h->aux);
    }
    if (h->aux_lo) {
      cudaStreamSynchronize(h->aux_lo);
      cudaStreamDestroy(h->aux_lo);
    }
    if (h->ev_aux) cudaEventDestroy(h->ev_aux);
    if (h->counts_ready) cudaEventDestroy(h->counts_ready);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->ev_colview) cudaEventDestroy(h->ev_colview);
    if (prev >= 0) cudaSetDevice(prev);
  }
  if (h->host_counts) cudaFreeHost(h->host_counts);
  delete h;
}

const char *snack_status_string(snack_status st) {
  switch (st) {
    case SNACK_OK: return "ok";
    case SNACK_ERR_INVALID_ARG: return "invalid argument";
    case SNACK_ERR_UNSORTED: return "pattern not strictly increasing in (row, col)";
    case SNACK_ERR_OUT_OF_RANGE: return "index out of range";
    case SNACK_ERR_WORKSPACE: return "plan or workspace too small";
    case SNACK_ERR_CUDA: return "CUDA error";
    case SNACK_ERR_TIMEOUT: return "device wait timed out";
    case SNACK_ERR_UNSUPPORTED: return "unsupported combination";
    case SNACK_ERR_NO_SPACE: return "not enough empty positions or draw budget exhausted";
  }
  return "unknown status";
}

int snack_version(void) { return SNACK_VERSION; }

snack_status snack_trace_start(int32_t capacity) {
  if (capacity < 1) return SNACK_ERR_INVALID_ARG;
  g_kernel_trace = nullptr;
  g_trace_owner.release();
  KernelTrace &t = g_trace_owner.t;
  t.fn = new (std::nothrow) const void *[capacity]();
  t.ev = new (std::nothrow) cudaEvent_t[2 * (size_t)capacity]();
  t.cap = capacity;
  t.n = 0;
  if (!t.fn || !t.ev) {
    g_trace_owner.release();
    return SNACK_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 2 * capacity; ++i)
    if (cudaEventCreate(&t.ev[i]) != cudaSuccess) {
      g_trace_owner.release();
      return SNACK_ERR_CUDA;
    }
  g_kernel_trace = &t;
  return SNACK_OK;
}

snack_status snack_trace_read(const char **names, float *us, int32_t max, int32_t *n) {
  if (!n || max < 0 || (max > 0 && (!names || !us))) return SNACK_ERR_INVALID_ARG;
  *n = 0;
  const KernelTrace &t = g_trace_owner.t;
  if (!t.fn) return SNACK_ERR_INVALID_ARG;
  const long long have = t.n < t.cap ? t.n : t.cap;
  const long long k = have < max ? have : max;
  for (long long j = 0; j < k; ++j) {  // the last k records, oldest first
    const int slot = (int)((t.n - k + j) % t.cap);
    float ms = 0.f;
    if (cudaEventSynchronize(t.ev[2 * slot + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, t.ev[2 * slot], t.ev[2 * slot + 1]) != cudaSuccess)
      return SNACK_ERR_CUDA;
    const char *name = nullptr;
    if (cudaFuncGetName(&name, t.fn[slot]) != cudaSuccess || !name) name = "?";
    names[j] = name;
    us[j] = 1000.f * ms;
  }
  *n = (int32_t)k;
  return SNACK_OK;
}

snack_status snack_trace_stop(void) {
  g_kernel_trace = nullptr;
  g_trace_owner.release();
  return SNACK_OK;
}

}  // extern "C"
