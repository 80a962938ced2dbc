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

// Column sort source with the row packed above the column (when both fit
// in 32 bits): key = row << cbits | col, value = storage index.  Digits of
// the column bits never see the row bits.
struct ColRowSrc {
  const int32_t *row, *col;
  int32_t out_f, in_f;
  int cbits;
  __device__ uint32_t key(int64_t i) const { return (clamp_idx(row[i], out_f) << cbits) | clamp_idx(col[i], in_f); }
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
  pdl_wait();
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

// Second half of the column view for columns of 9..17 bits (and rows that
// fit beside them in 32 bits).  The entries arrive as row << cbits | col,
// grouped by the column's high 8 bits (a stable scatter, so storage order
// within each group); block b sorts group b by the low `shift` bits,
// stably, and writes the column view (row, storage index) and the column
// offsets of its 2^shift columns.  The group is taken in chunks of
// kRadixTile entries in storage order; warp w holds entries w*256.. of a
// chunk, item i of lane l being entry i*32 + l of that range, so ranks from
// ballots plus per-warp counts keep storage order within every column.
constexpr int kColLowMax = 512;  // 2^shift bins at most

template <int kShift>
__global__ void __launch_bounds__(kRadixThreads) k_colview_bucket(const uint32_t *__restrict__ keys,
                                                                  const uint32_t *__restrict__ vals, int64_t n,
                                                                  int cbits,
                                                                  const uint32_t *__restrict__ offs, int64_t nb,
                                                                  int32_t in_f, int32_t *__restrict__ row_t,
                                                                  int32_t *__restrict__ src_t, int32_t *__restrict__ cp,
                                                                  uint16_t *__restrict__ rowt16) {
  pdl_wait();
  __shared__ uint32_t wc[kRadixWarps][kColLowMax];  // per-warp counts of a chunk, then local offsets
  __shared__ uint32_t run[kColLowMax];              // next free global slot of each column
  __shared__ uint32_t lstart[kColLowMax];           // start of each column's run inside the staged chunk
  __shared__ uint32_t s_src[kRadixTile], s_row[kRadixTile];
  __shared__ uint16_t s_col[kRadixTile];
  const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int shift = kShift;  // low column bits sorted here (the group holds 2^shift columns)
  constexpr int L = 1 << shift;
  constexpr uint32_t lmask = (uint32_t)(L - 1);
  const int64_t start = offs[(int64_t)b * nb];
  const int64_t end = b + 1 < kRadixBins ? (int64_t)offs[(int64_t)(b + 1) * nb] : n;
  // column counts of the group, then exclusive offsets = column starts
  for (int i = threadIdx.x; i < L; i += kRadixThreads) run[i] = 0;
  __syncthreads();
  for (int64_t k0 = start; k0 < end; k0 += (int64_t)kRadixThreads * kRadixItems) {
    uint32_t kk[kRadixItems];  // all loads in flight before the atomics
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i) {
      const int64_t k = k0 + i * kRadixThreads + threadIdx.x;
      kk[i] = k < end ? keys[k] : 0u;
    }
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i)
      if (k0 + i * kRadixThreads + threadIdx.x < end) atomicAdd(&run[kk[i] & lmask], 1u);
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // one warp scans the L counts in order
    uint32_t carry = (uint32_t)start;
    for (int c0 = 0; c0 < L; c0 += 32) {
      const int c = c0 + lane;
      const uint32_t v = c < L ? run[c] : 0u;
      const uint32_t inc = warp_inclusive_scan(v);
      if (c < L) {
        run[c] = carry + inc - v;
        const int64_t col = ((int64_t)b << shift) + c;
        if (col < in_f) cp[col] = (int32_t)(carry + inc - v);
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  if (b == 0 && threadIdx.x == 0) cp[in_f] = (int32_t)n;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t nkey[kRadixItems], nsrc[kRadixItems];  // next chunk, loaded ahead
  auto load = [&](int64_t c0) {
    const int64_t wbase = c0 + (int64_t)warp * (kRadixItems * 32);
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i) {
      const int64_t k = wbase + i * 32 + lane;
      const bool ok = k < end;
      nkey[i] = ok ? keys[k] : 0u;
      nsrc[i] = ok ? vals[k] : 0u;
    }
  };
  load(start);
  for (int64_t c0 = start; c0 < end; c0 += kRadixTile) {
    const int m = (int)(end - c0 < kRadixTile ? end - c0 : kRadixTile);
    uint32_t key[kRadixItems], src[kRadixItems];
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i) {
      key[i] = nkey[i];
      src[i] = nsrc[i];
    }
    if (c0 + kRadixTile < end) load(c0 + kRadixTile);
    __syncthreads();  // the previous chunk is done with wc, lstart and the staging arrays
    for (int i = threadIdx.x; i < kRadixWarps * L; i += kRadixThreads) wc[i >> shift][i & (L - 1)] = 0;
    __syncthreads();
    int dig[kRadixItems];
    uint32_t rank[kRadixItems];
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i) {
      const int64_t k = c0 + (int64_t)warp * (kRadixItems * 32) + i * 32 + lane;
      dig[i] = k < end ? (int)(key[i] & lmask) : L;  // L: sentinel for past the group
    }
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i) {
      unsigned peers = 0xffffffffu;
#pragma unroll
      for (int bit = 0; bit <= shift; ++bit) {  // shift + 1 bits cover the sentinel
        const bool on = (dig[i] >> bit) & 1;
        const unsigned bal = __ballot_sync(0xffffffffu, on);
        peers &= on ? bal : ~bal;
      }
      const uint32_t c = dig[i] < L ? wc[warp][dig[i]] : 0u;
      rank[i] = c + (uint32_t)__popc(peers & lt_mask);
      __syncwarp();
      if ((peers >> lane) == 1u && dig[i] < L) wc[warp][dig[i]] = c + (uint32_t)__popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // per column: its count in the chunk (kept in lstart for now) and the
    // warps' exclusive offsets inside the column's run
    for (int c = threadIdx.x; c < L; c += kRadixThreads) {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < kRadixWarps; ++w) {
        const uint32_t x = wc[w][c];
        wc[w][c] = t;
        t += x;
      }
      lstart[c] = t;
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // exclusive scan of the chunk's column counts: run starts in the staging arrays
      uint32_t carry = 0;
      for (int cc = 0; cc < L; cc += 32) {
        const int c = cc + lane;
        const uint32_t v = c < L ? lstart[c] : 0u;
        const uint32_t inc = warp_inclusive_scan(v);
        if (c < L) lstart[c] = carry + inc - v;
        carry += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRadixItems; ++i) {
      if (dig[i] < L) {
        const uint32_t lp = lstart[dig[i]] + wc[warp][dig[i]] + rank[i];
        s_src[lp] = src[i];
        s_row[lp] = key[i] >> cbits;
        s_col[lp] = (uint16_t)dig[i];
      }
    }
    __syncthreads();
    // write the staged chunk in order: each column's run lands on consecutive slots
    for (int e = threadIdx.x; e < m; e += kRadixThreads) {
      const int c = s_col[e];
      const uint32_t pos = run[c] + (uint32_t)e - lstart[c];
      src_t[pos] = (int32_t)s_src[e];
      if (rowt16)
        rowt16[pos] = (uint16_t)s_row[e];
      else
        row_t[pos] = (int32_t)s_row[e];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < L; c += kRadixThreads) {  // advance each column by its count in the chunk
      const uint32_t next = c + 1 < L ? lstart[c + 1] : (uint32_t)m;
      run[c] += next - lstart[c];
    }
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
  pdl_wait();
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
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k <= nnz; k += stride) {
    const int r_prev = k > 0 ? (int)clamp_idx((int32_t)idx[k - 1], n) : -1;
    const int r_cur = k < nnz ? (int)clamp_idx((int32_t)idx[k], n) : n;
    for (int r = r_prev + 1; r <= r_cur; ++r) ptr[r] = (int32_t)k;
  }
}

// 16-bit copy of an index array whose values fit (the caller checks the
// bound on the host): dst[k] = min(src[k], 65535) as uint16, clamped so a
// bad input can never produce an index past the bound.
__global__ void k_pack16(const int32_t *__restrict__ src, int64_t n, uint16_t *__restrict__ dst) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
    const uint32_t v = (uint32_t)src[k];
    dst[k] = (uint16_t)(v < 65535u ? v : 65535u);
  }
}

__global__ void k_validate(const int32_t *__restrict__ row, const int32_t *__restrict__ col, int64_t nnz, int32_t out_f,
                           int32_t in_f, uint32_t *__restrict__ flag) {
  pdl_wait();
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
  if (nnz > 0) launch_pdl(k_count, grid_for(nnz, 256), 256, 0, s, idx, nnz, n, counts);
  return scan_apply<uint32_t>(CountRead{counts, (int64_t)n}, (int64_t)n + 1, WriteOffsets{ptr}, (uint32_t *)nullptr,
                              stemp, s);
}

}  // namespace

PlanLayout plan_layout(int32_t out_f, int32_t in_f, int64_t nnz, int bt_max, int n_btiles, bool dense) {
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
  L.c16 = in_f <= 65536;
  L.r16 = out_f <= 65536;
  L.off_col16 = o;
  if (L.c16) o += align_up(sizeof(uint16_t) * (size_t)(nnz > 0 ? nnz : 1), kAlign);
  L.off_rowt16 = o;
  if (L.r16) o += align_up(sizeof(uint16_t) * (size_t)(nnz > 0 ? nnz : 1), kAlign);
  L.cv = colview_update_ok(out_f, in_f, nnz);
  L.cv_pmax = L.cv ? (nnz + 3) / 4 : 0;
  L.off_cpa = L.off_tta = L.off_rowta = L.off_srcta = L.off_rowt16a = L.off_newidx = L.off_gq = L.off_gck =
      L.off_gcq = L.off_cvs = L.off_cvq = L.off_cvb = o;
  if (L.cv) {
    const size_t n = (size_t)nnz, pm = (size_t)L.cv_pmax;
    L.off_cpa = o;
    o += align_up(sizeof(int32_t) * ((size_t)in_f + 1), kAlign);
    L.off_tta = o;
    o += align_up(sizeof(int32_t) * 2 * ((size_t)L.gt.n_tiles + 1), kAlign);
    L.off_rowta = o;
    o += align_up(sizeof(int32_t) * n, kAlign);
    L.off_srcta = o;
    o += align_up(sizeof(int32_t) * n, kAlign);
    L.off_rowt16a = o;
    if (L.r16) o += align_up(sizeof(uint16_t) * n, kAlign);
    L.off_newidx = o;
    o += align_up(sizeof(uint32_t) * n, kAlign);
    L.off_gq = o;
    o += align_up(sizeof(uint32_t) * pm, kAlign);
    L.off_gck = o;
    o += align_up(sizeof(uint32_t) * pm, kAlign);
    L.off_gcq = o;
    o += align_up(sizeof(uint32_t) * pm, kAlign);
    L.off_cvs = o;
    o += align_up(sizeof(uint32_t) * (size_t)in_f, kAlign);
    L.off_cvq = o;
    o += align_up(sizeof(uint32_t) * (size_t)in_f, kAlign);
    L.off_cvb = o;
    o += align_up(32 * (size_t)(ceil_div(nnz, kScanTile) + 1), kAlign);
  }
  L.dense = dense;
  L.off_tab = o;
  if (dense) o += dense_table_bytes(out_f, in_f);
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
  p.col16 = L.c16 ? reinterpret_cast<uint16_t *>(b + L.off_col16) : nullptr;
  p.rowt16 = L.r16 ? reinterpret_cast<uint16_t *>(b + L.off_rowt16) : nullptr;
  p.cp_alt = L.cv ? reinterpret_cast<int32_t *>(b + L.off_cpa) : nullptr;
  p.tiles_t_alt = L.cv ? reinterpret_cast<int32_t *>(b + L.off_tta) : nullptr;
  p.row_t_alt = L.cv ? reinterpret_cast<int32_t *>(b + L.off_rowta) : nullptr;
  p.src_t_alt = L.cv ? reinterpret_cast<int32_t *>(b + L.off_srcta) : nullptr;
  p.rowt16_alt = L.cv && L.r16 ? reinterpret_cast<uint16_t *>(b + L.off_rowt16a) : nullptr;
  p.newidx = L.cv ? reinterpret_cast<uint32_t *>(b + L.off_newidx) : nullptr;
  p.gq = L.cv ? reinterpret_cast<uint32_t *>(b + L.off_gq) : nullptr;
  p.gc_key = L.cv ? reinterpret_cast<uint32_t *>(b + L.off_gck) : nullptr;
  p.gc_q = L.cv ? reinterpret_cast<uint32_t *>(b + L.off_gcq) : nullptr;
  p.cv_pcnt = L.cv ? reinterpret_cast<uint32_t *>(b + L.off_cvs) : nullptr;
  p.cv_ppre = L.cv ? reinterpret_cast<uint32_t *>(b + L.off_cvq) : nullptr;
  p.cv_bnd = L.cv ? reinterpret_cast<void *>(b + L.off_cvb) : nullptr;
  p.cv_pmax = L.cv_pmax;
  p.tables = L.dense ? reinterpret_cast<void *>(b + L.off_tab) : nullptr;
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

namespace {
template <int kShift>
cudaError_t launch_cvb(const uint32_t *ka, const uint32_t *va, int64_t nnz, int cbits, const uint32_t *offs, int64_t nb,
                       int32_t in_f, const PlanPtrs &p, cudaStream_t s) {
  launch_pdl(k_colview_bucket<kShift>, kRadixBins, kRadixThreads, 0, s, ka, va, nnz, cbits, offs, nb, in_f, p.row_t,
             p.src_t, p.cp, p.rowt16);
  return cudaGetLastError();
}
// the group kernel for 1..9 low column bits
cudaError_t launch_colview_bucket(int shift, const uint32_t *ka, const uint32_t *va, int64_t nnz, int cbits,
                                  const uint32_t *offs, int64_t nb, int32_t in_f, const PlanPtrs &p, cudaStream_t s) {
  switch (shift) {
    case 1: return launch_cvb<1>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 2: return launch_cvb<2>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 3: return launch_cvb<3>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 4: return launch_cvb<4>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 5: return launch_cvb<5>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 6: return launch_cvb<6>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 7: return launch_cvb<7>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 8: return launch_cvb<8>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
    case 9: return launch_cvb<9>(ka, va, nnz, cbits, offs, nb, in_f, p, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace

bool colview_digits(int32_t out_f, int32_t in_f, int64_t nnz, int *shift) {
  const int cbits = bits_for((uint64_t)(in_f - 1)), rbits = bits_for((uint64_t)(out_f - 1));
  const bool ok = nnz > 0 && cbits > 8 && cbits - 8 <= 9 && cbits + rbits <= 32;
  if (shift) *shift = ok ? cbits - 8 : 0;
  return ok;
}

bool colview_update_ok(int32_t out_f, int32_t in_f, int64_t nnz) {
  return nnz > 0 && bits_for((uint64_t)(in_f - 1)) + bits_for((uint64_t)(out_f - 1)) <= 31;
}

cudaError_t cut_tiles(const int32_t *ptr, int32_t n_rows, int64_t nnz, const TileGeom &g, int32_t *tiles,
                      cudaStream_t s) {
  launch_pdl(k_tiles, grid_for(32 * ((int64_t)g.n_tiles + 1), 256), 256, 0, s, ptr, n_rows, nnz, g.cost_per_tile,
             g.row_weight, g.n_tiles, tiles);
  return cudaGetLastError();
}

cudaError_t build_plan(int32_t out_f, int32_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
                       const PlanPtrs &p, const TileGeom &gf, const TileGeom &gt, void *ws, cudaStream_t s,
                       int ready, bool colview) {
  BuildWs W = build_ws_layout(out_f, in_f, nnz);
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  uint32_t *counts = reinterpret_cast<uint32_t *>(b + W.counts);
  void *stemp = b + W.scan;
  cudaError_t e;
  const int cbits = bits_for((uint64_t)(in_f - 1));

  // row offsets and the 16-bit column copy: already written by a
  // restructure's merge, made here otherwise
  if (ready < kPlanRowsReady && p.col16 && nnz > 0) launch_pdl(k_pack16, grid_for(nnz, 256), 256, 0, s, col, nnz, p.col16);
  if (ready < kPlanRowsReady) {
    e = build_offsets(row, nnz, out_f, p.rp, counts, stemp, s);
    if (e != cudaSuccess) return e;
  }
  // the tensor-core path's per-(block, row) masks and offsets, from the row half
  if (p.tables && p.col16) {
    e = build_tables(p.rp, p.col16, out_f, in_f, p.tables, s);
    if (e != cudaSuccess) return e;
  }
  if (ready < kPlanRowTilesReady) {
    e = cut_tiles(p.rp, out_f, nnz, gf, p.tiles_f, s);
    if (e != cudaSuccess) return e;
  }
  if (!colview) return cudaGetLastError();
  // column view: stable sort by column (rows stay in order within a column);
  // column offsets from the sorted keys
  if (colview_digits(out_f, in_f, nnz, nullptr)) {
    // 9..17-bit columns: stable scatter of (row, col) by the column's high 8
    // bits, then one block per group sorts by the low bits and writes the
    // column offsets
    uint32_t *ka = reinterpret_cast<uint32_t *>(b + W.keys_a);
    uint32_t *va = reinterpret_cast<uint32_t *>(b + W.vals_a);
    const int shift = cbits - 8;
    const int64_t nb = ceil_div(nnz, kRadixTile);
    uint8_t *t = b + W.radix;
    const size_t hbytes = align_up((size_t)nb * kRadixBins * sizeof(uint32_t), kAlign);
    uint32_t *hist = reinterpret_cast<uint32_t *>(t);
    const uint32_t *offs = reinterpret_cast<uint32_t *>(t + hbytes);
    e = radix_pass<uint32_t>(ColRowSrc{row, col, out_f, in_f, cbits}, ArrayDst<uint32_t>{ka, va}, nnz, shift, hist,
                             reinterpret_cast<uint32_t *>(t + hbytes), t + 2 * hbytes, s);
    if (e != cudaSuccess) return e;
    e = launch_colview_bucket(shift, ka, va, nnz, cbits, offs, nb, in_f, p, s);
    if (e != cudaSuccess) return e;
  } else if (nnz > 0) {
    uint32_t *ka = reinterpret_cast<uint32_t *>(b + W.keys_a);
    uint32_t *va = reinterpret_cast<uint32_t *>(b + W.vals_a);
    uint32_t *kb = reinterpret_cast<uint32_t *>(b + W.keys_b);
    uint32_t *vb = reinterpret_cast<uint32_t *>(b + W.vals_b);
    uint32_t *keys_out = reinterpret_cast<uint32_t *>(b + W.keys_out);
    e = radix_sort_custom<uint32_t>(ColSrc{col, in_f}, ColviewDst{keys_out, p.row_t, p.src_t, row, out_f}, nnz,
                                    cbits, ka, va, kb, vb, b + W.radix, s);
    if (e != cudaSuccess) return e;
    launch_pdl(k_offsets_sorted<uint32_t>, grid_for(nnz + 1, 256), 256, 0, s, keys_out, nnz, in_f, p.cp);
    if (p.rowt16) launch_pdl(k_pack16, grid_for(nnz, 256), 256, 0, s, p.row_t, nnz, p.rowt16);
  } else {
    launch_pdl(k_offsets_sorted<int32_t>, 1, 256, 0, s, col, 0, in_f, p.cp);
  }
  return cut_tiles(p.cp, in_f, nnz, gt, p.tiles_t, s);
}

// *flag |= 1 when some row r does not start at r * K (K stored weights per row)
__global__ void k_check_fan_in(const int32_t *__restrict__ rp, int32_t out_f, int32_t K, uint32_t *flag) {
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r <= out_f && rp[r] != (int64_t)r * K) atomicOr(flag, 1u);
}

cudaError_t check_fan_in(const int32_t *rp, int32_t out_f, int32_t K, uint32_t *flag, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  launch_pdl(k_check_fan_in, grid_for((int64_t)out_f + 1, 256), 256, 0, s, rp, out_f, K, flag);
  return cudaGetLastError();
}

cudaError_t pack16(const int32_t *src, int64_t n, uint16_t *dst, cudaStream_t s) {
  if (n > 0 && dst) launch_pdl(k_pack16, grid_for(n, 256), 256, 0, s, src, n, dst);
  return cudaGetLastError();
}

cudaError_t validate_pattern(int32_t out_f, int32_t in_f, int64_t nnz, const int32_t *row, const int32_t *col,
                             uint32_t *flag, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (nnz > 0) launch_pdl(k_validate, grid_for(nnz, 256), 256, 0, s, row, col, nnz, out_f, in_f, flag);
  return cudaGetLastError();
}

}  // namespace snack
