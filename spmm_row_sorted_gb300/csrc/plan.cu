// Plan of a sparse layer: row offsets, load-balanced merge-path tiles for the
// forward pass, and a column-ordered view (column offsets, row and storage
// index per entry) with its own tiles for the input gradient.
//
// Offsets are counts (histogram + exclusive scan of clamped indices), so they
// are monotone and in [0, nnz] even for an invalid pattern; every index a
// kernel later derives from the plan is therefore in range.
#include "internal.hpp"
#include "prims.cuh"

namespace snack {

namespace {

__device__ __forceinline__ uint32_t clamp_idx(int32_t v, int32_t n) {
  uint32_t u = (uint32_t)v, m = (uint32_t)(n - 1);
  return u < m ? u : m;
}

// First pass of the column sort reads the pattern directly: key = clamped
// column, value = storage index.
struct ColSrc {
  const int32_t *col;
  int32_t in_f;
  __device__ uint32_t key(int64_t i) const { return clamp_idx(col[i], in_f); }
  __device__ uint32_t val(int64_t i) const { return (uint32_t)i; }
};

// Last pass of the column sort writes the column view itself: the sorted
// column (for the offsets), the storage index, and that entry's row.
struct ColviewDst {
  uint32_t *keys;
  int32_t *row_t, *src_t;
  const int32_t *row;
  int32_t out_f;
  __device__ int load(uint32_t k) const { return row[k]; }
  __device__ void put(uint32_t pos, uint32_t key, uint32_t k, int r) const {
    keys[pos] = key;
    src_t[pos] = (int32_t)k;
    row_t[pos] = (int32_t)clamp_idx(r, out_f);
  }
};

// counts[clamp(idx[k])] += 1, aggregated over equal indices within a warp
__global__ void k_count(const int32_t *__restrict__ idx, int64_t nnz, int32_t n, uint32_t *__restrict__ counts) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < nnz; base += stride) {
    int64_t k = base + threadIdx.x;
    bool ok = k < nnz;
    int key = ok ? (int)clamp_idx(idx[k], n) : -1;
    unsigned peers = __match_any_sync(0xffffffffu, key);
    int lane = threadIdx.x & 31;
    if (ok && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(&counts[key], (uint32_t)__popc(peers));
  }
}

struct CountRead {
  const uint32_t *c;
  int64_t n;
  __device__ uint32_t operator()(int64_t i) const { return i < n ? c[i] : 0u; }
};
struct WriteOffsets {
  int32_t *o;
  __device__ void operator()(int64_t i, uint32_t ex, uint32_t, int) const { o[i] = (int32_t)ex; }
};

// Split point of the merge path (row ends cost w, stored weights cost 1) at
// cost D: i = max{i : w*i + ptr[i] <= D}, j = min(ptr[i+1], D - w*i).
// One warp per split point; each round probes 32 evenly spaced rows at once,
// so a 16K-row search takes three dependent rounds instead of fourteen.
__global__ void k_tiles(const int32_t *__restrict__ ptr, int32_t n_rows, int64_t nnz, int32_t C, int32_t w,
                        int32_t n_tiles, int32_t *__restrict__ tiles) {
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t > n_tiles) return;
  const int64_t total = (int64_t)w * n_rows + nnz;
  int64_t D = t * (int64_t)C;
  if (D > total || t == n_tiles) D = total;
  int lo = 0, hi = n_rows;  // f(lo) <= D always (f(0) = 0); answer in [lo, hi]
  while (hi - lo > 31) {  // leaves at most 32 candidates for the final probe
    const int64_t span = hi - lo;
    const int p = lo + (int)(span * (lane + 1) / 33);
    const bool ok = (int64_t)w * p + ptr[p] <= D;
    const unsigned ball = __ballot_sync(0xffffffffu, ok);
    const int cnt = __popc(ball);  // f is increasing: the true lanes are a prefix
    const int new_lo = cnt > 0 ? lo + (int)(span * cnt / 33) : lo;
    const int new_hi = cnt < 32 ? lo + (int)(span * (cnt + 1) / 33) - 1 : hi;
    lo = new_lo;
    hi = new_hi;
  }
  {
    const int p = lo + lane;
    const bool ok = p <= hi && (int64_t)w * p + ptr[p] <= D;
    const int cnt = __popc(__ballot_sync(0xffffffffu, ok));
    lo = lo + cnt - 1;
  }
  if (lane == 0) {
    int64_t j = lo < n_rows ? D - (int64_t)w * lo : nnz;
    if (lo < n_rows && j > ptr[lo + 1]) j = ptr[lo + 1];
    tiles[2 * t] = lo;
    tiles[2 * t + 1] = (int32_t)j;
  }
}

// Offsets of sorted indices (a restructure's rows, or the column keys after
// the column sort): ptr[r] for r in (idx[k-1], idx[k]] is k.  One pass, no
// atomics; indices are clamped, so writes stay in [0, n].
template <typename I>
__global__ void k_offsets_sorted(const I *__restrict__ idx, int64_t nnz, int32_t n, int32_t *__restrict__ ptr) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k <= nnz; k += stride) {
    const int r_prev = k > 0 ? (int)clamp_idx((int32_t)idx[k - 1], n) : -1;
    const int r_cur = k < nnz ? (int)clamp_idx((int32_t)idx[k], n) : n;
    for (int r = r_prev + 1; r <= r_cur; ++r) ptr[r] = (int32_t)k;
  }
}

__global__ void k_validate(const int32_t *__restrict__ row, const int32_t *__restrict__ col, int64_t nnz, int32_t out_f,
                           int32_t in_f, uint32_t *__restrict__ flag) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t bad = 0;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += stride) {
    int32_t r = row[k], c = col[k];
    if (r < 0 || r >= out_f || c < 0 || c >= in_f) bad |= 1u;
    if (k > 0) {
      int32_t rq = row[k - 1], cq = col[k - 1];
      if (!(rq < r || (rq == r && cq < c))) bad |= 2u;
    }
  }
  if (bad) atomicOr(flag, bad);
}

int bits_for(uint64_t max_value) {
  int b = 0;
  while (b < 64 && (max_value >> b) != 0) ++b;
  return b;
}

unsigned grid_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > 65535 * 8) b = 65535 * 8;
  return (unsigned)b;
}

cudaError_t build_offsets(const int32_t *idx, int64_t nnz, int32_t n, int32_t *ptr, uint32_t *counts, void *stemp,
                          cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(uint32_t) * ((size_t)n + 1), s);
  if (e != cudaSuccess) return e;
  if (nnz > 0) k_count<<<grid_for(nnz, 256), 256, 0, s>>>(idx, nnz, n, counts);
  return scan_apply<uint32_t>(CountRead{counts, (int64_t)n}, (int64_t)n + 1, WriteOffsets{ptr}, (uint32_t *)nullptr,
                              stemp, s);
}

}  // namespace

PlanLayout plan_layout(int32_t out_f, int32_t in_f, int64_t nnz, int bt_max, int n_btiles) {
  PlanLayout L;
  L.gf = tile_geom(out_f, nnz, bt_max, n_btiles);
  L.gt = tile_geom(in_f, nnz, bt_max, n_btiles);
  size_t o = 0;
  L.off_rp = o;
  o += align_up(sizeof(int32_t) * ((size_t)out_f + 1), kAlign);
  L.off_tf = o;
  o += align_up(sizeof(int32_t) * 2 * ((size_t)L.gf.n_tiles + 1), kAlign);
  L.off_cp = o;
  o += align_up(sizeof(int32_t) * ((size_t)in_f + 1), kAlign);
  L.off_tt = o;
  o += align_up(sizeof(int32_t) * 2 * ((size_t)L.gt.n_tiles + 1), kAlign);
  L.off_rowt = o;
  o += align_up(sizeof(int32_t) * (size_t)(nnz > 0 ? nnz : 1), kAlign);
  L.off_srct = o;
  o += align_up(sizeof(int32_t) * (size_t)(nnz > 0 ? nnz : 1), kAlign);
  L.off_flags = o;
  o += align_up(sizeof(uint32_t) * 64, kAlign);
  L.total = o;
  return L;
}

PlanPtrs plan_ptrs(const PlanLayout &L, void *base) {
  uint8_t *b = reinterpret_cast<uint8_t *>(base);
  PlanPtrs p;
  p.rp = reinterpret_cast<int32_t *>(b + L.off_rp);
  p.tiles_f = reinterpret_cast<int32_t *>(b + L.off_tf);
  p.cp = reinterpret_cast<int32_t *>(b + L.off_cp);
  p.tiles_t = reinterpret_cast<int32_t *>(b + L.off_tt);
  p.row_t = reinterpret_cast<int32_t *>(b + L.off_rowt);
  p.src_t = reinterpret_cast<int32_t *>(b + L.off_srct);
  p.flags = reinterpret_cast<uint32_t *>(b + L.off_flags);
  return p;
}

namespace {
struct BuildWs {
  size_t counts, keys_a, vals_a, keys_b, vals_b, keys_out, radix, scan, total;
};

BuildWs build_ws_layout(int32_t out_f, int32_t in_f, int64_t nnz) {
  BuildWs w;
  const size_t n = (size_t)(nnz > 0 ? nnz : 1);
  const size_t nmax = (size_t)(out_f > in_f ? out_f : in_f) + 1;
  size_t o = 0;
  w.counts = o;
  o += align_up(sizeof(uint32_t) * nmax, kAlign);
  w.keys_a = o;
  o += align_up(sizeof(uint32_t) * n, kAlign);
  w.vals_a = o;
  o += align_up(sizeof(uint32_t) * n, kAlign);
  w.keys_b = o;
  o += align_up(sizeof(uint32_t) * n, kAlign);
  w.vals_b = o;
  o += align_up(sizeof(uint32_t) * n, kAlign);
  w.keys_out = o;
  o += align_up(sizeof(uint32_t) * n, kAlign);
  w.radix = o;
  o += radix_temp_bytes((int64_t)n);
  w.scan = o;
  o += scan_temp_bytes<uint32_t>((int64_t)nmax);
  w.total = o;
  return w;
}
}  // namespace

size_t plan_build_ws_bytes(int32_t out_f, int32_t in_f, int64_t nnz) { return build_ws_layout(out_f, in_f, nnz).total; }

cudaError_t build_plan(int32_t out_f, int32_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
                       const PlanPtrs &p, const TileGeom &gf, const TileGeom &gt, void *ws, cudaStream_t s,
                       bool rp_ready) {
  BuildWs W = build_ws_layout(out_f, in_f, nnz);
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  uint32_t *counts = reinterpret_cast<uint32_t *>(b + W.counts);
  void *stemp = b + W.scan;
  cudaError_t e;

  // row offsets: already written by a restructure's merge, counts otherwise
  if (!rp_ready) {
    e = build_offsets(row, nnz, out_f, p.rp, counts, stemp, s);
    if (e != cudaSuccess) return e;
  }
  k_tiles<<<grid_for(32 * ((int64_t)gf.n_tiles + 1), 256), 256, 0, s>>>(p.rp, out_f, nnz, gf.cost_per_tile,
                                                                         gf.row_weight, gf.n_tiles, p.tiles_f);
  // column view: stable sort by column (rows stay in order within a column);
  // column offsets from the sorted keys
  if (nnz > 0) {
    uint32_t *ka = reinterpret_cast<uint32_t *>(b + W.keys_a);
    uint32_t *va = reinterpret_cast<uint32_t *>(b + W.vals_a);
    uint32_t *kb = reinterpret_cast<uint32_t *>(b + W.keys_b);
    uint32_t *vb = reinterpret_cast<uint32_t *>(b + W.vals_b);
    uint32_t *keys_out = reinterpret_cast<uint32_t *>(b + W.keys_out);
    e = radix_sort_custom<uint32_t>(ColSrc{col, in_f}, ColviewDst{keys_out, p.row_t, p.src_t, row, out_f}, nnz,
                                    bits_for((uint64_t)(in_f - 1)), ka, va, kb, vb, b + W.radix, s);
    if (e != cudaSuccess) return e;
    k_offsets_sorted<uint32_t><<<grid_for(nnz + 1, 256), 256, 0, s>>>(keys_out, nnz, in_f, p.cp);
  } else {
    k_offsets_sorted<int32_t><<<1, 256, 0, s>>>(col, 0, in_f, p.cp);
  }
  k_tiles<<<grid_for(32 * ((int64_t)gt.n_tiles + 1), 256), 256, 0, s>>>(p.cp, in_f, nnz, gt.cost_per_tile,
                                                                         gt.row_weight, gt.n_tiles, p.tiles_t);
  return cudaGetLastError();
}

cudaError_t validate_pattern(int32_t out_f, int32_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
                             uint32_t *flag, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (nnz > 0) k_validate<<<grid_for(nnz, 256), 256, 0, s>>>(row, col, nnz, out_f, in_f, flag);
  return cudaGetLastError();
}

}  // namespace snack
