// SpMM over row-sorted COO (forward and input gradient), the weight-gradient
// SDDMM, and the activation transposes they gather from.
//
// Work decomposition (forward; the input gradient runs the same kernel on the
// column-ordered view of W):
//  * The merge path of (row ends, stored weights) is cut into tiles of equal
//    cost, a row end costing `row_weight` and a stored weight costing 1, so
//    every tile has at most cost_per_tile weights AND a bounded number of rows
//    whatever the row-length skew.  One CTA per (tile, batch tile).
//  * Inside a CTA the tile is cut again into 8 equal-cost warp ranges.
//  * A warp walks its rows.  Its 32 lanes form 32/G slots of G lanes; a slot
//    takes one stored weight at a time and its G lanes each gather a 16-byte
//    slice (V batch elements) of the transposed activation row Xt[col], so
//    one weight's batch vector is read as whole 32-byte sectors.
//  * Row sums reduce across slots with xor shuffles and land in shared
//    memory; rows split between warps are combined in warp order, rows split
//    between CTAs leave a partial ("carry" / "head") that a fix-up kernel adds
//    in tile order.  No atomics on outputs: results are deterministic.
//  * Outputs leave shared memory as contiguous runs of Y[b, r0:r1].
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace snack {

constexpr int kSpmmThreads = 256;
constexpr int kSpmmWarps = kSpmmThreads / 32;

// Resident CTAs per SM the tile kernel is compiled for (caps registers), and
// the largest unroll depth (stored weights per slot in flight).  Defaults are
// the fastest measured on GB300 for the 16384^2 / batch-32 layer.
#ifndef SNACK_SPMM_MIN_CTAS
#define SNACK_SPMM_MIN_CTAS 5  // resident CTAs per SM the register budget is sized for
#endif
#ifndef SNACK_SPMM_MIN_CTAS_FUSED
#define SNACK_SPMM_MIN_CTAS_FUSED 4  // the fused backward keeps more live values
#endif
#ifndef SNACK_TILE_COST
#define SNACK_TILE_COST 65536  // tile cost C = SNACK_TILE_COST / batch tile width, clamped to [1024, 8192]
#endif
#ifndef SNACK_SPMM_UNROLL
#define SNACK_SPMM_UNROLL 4
#endif

// Batch geometry of one call.
struct BatchGeom {
  int V;         // activation elements per lane slice (1, 4 or 8)
  int G;         // lanes per stored weight (power of two <= 32)
  int bt;        // batch elements per CTA = G * V
  int n_btiles;  // CTAs along the batch
  int ldx;       // row stride of the transposed activations (= n_btiles * bt; 1 when batch == 1)
};

inline BatchGeom batch_geom(int batch, snack_dtype act) {
  BatchGeom g;
  if (batch <= 1) {
    g.V = 1;
    g.G = 1;
    g.bt = 1;
    g.n_btiles = 1;
    g.ldx = 1;
    return g;
  }
  g.V = act == SNACK_BF16 ? 8 : 4;
  int bp = (batch + g.V - 1) / g.V * g.V;
  int lanes = bp / g.V;
  int G = 1;
  while (G < lanes && G < 32) G <<= 1;
  g.G = G;
  g.bt = G * g.V;
  g.n_btiles = (bp + g.bt - 1) / g.bt;
  g.ldx = g.n_btiles * g.bt;
  return g;
}

// Tile geometry of one merge path (fixed per plan).
struct TileGeom {
  int32_t cost_per_tile;  // C
  int32_t row_weight;     // w
  int32_t n_tiles;
  int32_t max_rows;       // rows a tile can touch, partial rows included
};

inline TileGeom tile_geom(int32_t n_rows, int64_t nnz, int bt_max, int n_btiles = 1) {
  TileGeom t;
  int c = SNACK_TILE_COST / (bt_max > 0 ? bt_max : 1);
  if (c < 1024) c = 1024;  // batch tiles of 128 and 256: 1024 measured faster than 512 (768x3072 and 3072x768 at B 1024)
  if (c > 8192) c = 8192;
  // keep the staged rows of a tile within ~16 KB of shared memory
  int rows_target = 16384 / ((bt_max + 1) * 4);
  if (rows_target < 16) rows_target = 16;
  auto weight = [&](int cost) {
    int w = (cost + rows_target - 1) / rows_target;
    return w < 2 ? 2 : w;
  };
  int w = weight(c);
  int64_t total = (int64_t)w * n_rows + nnz;
  // small layers: smaller tiles (down to 128 cost units) until the grid has
  // about 1024 CTAs, so the work still spreads over every SM
  const int64_t want = 1024 / (n_btiles > 0 ? n_btiles : 1) + 1;
  if ((total + c - 1) / c < want) {
    int64_t c2 = (total + want - 1) / want;
    if (c2 < 128) c2 = 128;
    if (c2 < c) {
      c = (int)c2;
      w = weight(c);
      total = (int64_t)w * n_rows + nnz;
    }
  }
  t.cost_per_tile = c;
  t.row_weight = w;
  int64_t nt = (total + c - 1) / c;
  t.n_tiles = (int32_t)(nt > 0 ? nt : 1);
  t.max_rows = (c + w - 1) / w + 2;
  return t;
}

// stored weights a tile can hold: cost C plus the part of a row end that did not fit
inline __host__ __device__ int tile_stage_cap(const TileGeom &tg) { return tg.cost_per_tile + tg.row_weight; }
// The staged arrays run kStagePad entries past the tile (zero offsets and
// weights), so the inner loop reads whole groups of slots without bounds
// tests; weights past a row's end are masked to zero.
constexpr int kStagePad = 256;  // >= slots per warp x weights per slot
inline __host__ __device__ int tile_stage_len(const TileGeom &tg) { return tile_stage_cap(tg) + kStagePad; }

inline size_t spmm_smem_bytes(const TileGeom &tg, int bt) {
  return (size_t)tg.max_rows * (bt + 1) * 4 + (size_t)kSpmmWarps * bt * 4 + (size_t)(tg.max_rows + 1) * 4 +
         (size_t)(kSpmmWarps + 1) * 2 * 4 + 8 + (size_t)tile_stage_len(tg) * 8;  // + 8: alignment of the staged pairs
}

struct SpmmParams {
  int32_t n_rows;         // outputs per batch row (fwd: out_f, dx: in_f)
  int32_t n_src;          // rows of the gathered operand (fwd: in_f, dx: out_f)
  const int32_t *ptr;     // [n_rows + 1] segment offsets
  const int32_t *tiles;   // [(n_tiles + 1) * 2] (row, nnz) split points
  TileGeom tg;
  int64_t nnz;
  const int32_t *idx;     // [nnz] gather index (fwd: col, dx: row of the column view)
  const uint16_t *idx16;  // [nnz] the same index in 16 bits (from the plan), or null
  const void *val;        // [nnz] weights, storage order
  const int32_t *val_src; // dx: storage index of each column-view entry; fwd: null
  const void *xt;         // [n_src][ldx] transposed activations
  const float *bias;      // [n_rows] or null
  void *y;                // [batch][n_rows]
  int32_t batch;
  float *carry;           // [n_btiles][n_tiles][bt]
  float *head;            // [n_btiles][n_tiles][bt]
  const void *xt_dw;      // fused backward: transposed X [n_rows][ldx] (dx mode, rows = input features)
  float *dw;              // fused backward: weight gradient [nnz], written at storage index
  int32_t act;            // output epilogue: kActNone, kActGelu, kActGeluGrad
  const void *pre_in;     // kActGeluGrad: pre-activation [batch][n_rows] (act dtype)
  void *pre_out;          // kActGelu: pre-activation written here when non-null
  float *db;              // small-batch fused backward: bias gradient [n_src], or null
};

// Output epilogues of the SpMM kernels.
constexpr int kActNone = 0;
constexpr int kActGelu = 1;      // y = GELU(s), s optionally kept in pre_out
constexpr int kActGeluGrad = 2;  // y = s * GELU'(pre_in)

// GELU in the exact (erf) form and its derivative Phi(x) + x phi(x).
__device__ __forceinline__ float gelu_f(float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad_f(float x) {
  return 0.5f * (1.f + erff(x * 0.70710678118654752f)) + x * 0.39894228040143267794f * expf(-0.5f * x * x);
}

// Final value of output (b, r) given its fp32 sum s (bias included).
template <typename TA>
__device__ __forceinline__ TA spmm_epilogue(const SpmmParams &P, float s, size_t off) {
  if (P.act == kActGelu) {
    if (P.pre_out) reinterpret_cast<TA *>(P.pre_out)[off] = from_f32<TA>(s);
    return from_f32<TA>(gelu_f(s));
  }
  if (P.act == kActGeluGrad) return from_f32<TA>(s * gelu_grad_f(to_f32(reinterpret_cast<const TA *>(P.pre_in)[off])));
  return from_f32<TA>(s);
}

// ------------------------------------------------------------------ kernels

// Unroll: stored weights per slot in flight, keeping kU * V <= 32 gathered floats.
template <int V, int G>
struct SpmmUnroll {
  static constexpr int kSlots = 32 / G;
  static constexpr int kMax = SNACK_SPMM_UNROLL;
  static constexpr int base = kSlots >= 8 ? (V >= 8 ? 2 : 4) : (V >= 8 ? 4 : 8);
  static constexpr int value = base < kMax ? base : kMax;
};

// kFuseDw (column-view mode, one batch tile): each gathered dY row slice is
// also dotted with the current column's X slice, giving dW at that entry's
// storage index in the same pass.
template <typename TA, typename TV, int V, int G, bool kGatherVal, bool kFuseDw>
__global__ void __launch_bounds__(kSpmmThreads, kFuseDw ? SNACK_SPMM_MIN_CTAS_FUSED : SNACK_SPMM_MIN_CTAS)
    k_spmm_tiles(SpmmParams P, BatchGeom bg) {
  pdl_wait();
  constexpr int kSlots = 32 / G;
  constexpr int kU = SpmmUnroll<V, G>::value;
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane / G, g = lane % G;
  const int t = blockIdx.x, bi = blockIdx.y;
  const int bt = bg.bt;
  const int b0 = bi * bt;
  const int max_rows = P.tg.max_rows;
  const int w = P.tg.row_weight;
  const int cap = tile_stage_cap(P.tg);
  const int ys_ld = bt + 1;
  float *Ys = smem;
  float *wcar = Ys + (size_t)max_rows * ys_ld;
  int *rps = reinterpret_cast<int *>(wcar + kSpmmWarps * bt);
  int *wsp = rps + max_rows + 1;
  // s_iv: each weight's gather offset in elements (index * ldx) and its value bits
  uint2 *s_iv = reinterpret_cast<uint2 *>(
      (reinterpret_cast<uintptr_t>(wsp + 2 * (kSpmmWarps + 1)) + 7) & ~(uintptr_t)7);  // 8-byte aligned
  uint32_t *s_src = reinterpret_cast<uint32_t *>(s_iv + cap + kStagePad);  // kFuseDw only

  const int i0 = P.tiles[2 * t], j0 = P.tiles[2 * t + 1];
  int i1 = P.tiles[2 * t + 2];
  int j1 = P.tiles[2 * t + 3];
  if (i1 - i0 + 1 > max_rows) i1 = i0 + max_rows - 1;  // defensive: never overrun shared memory
  if (j1 - j0 > cap) j1 = j0 + cap;
  const int nr = i1 - i0 + 1;

  for (int q = tid; q <= nr; q += kSpmmThreads) {
    int r = i0 + q;
    rps[q] = P.ptr[r < P.n_rows ? r : P.n_rows];
  }
  for (int b = tid; b < bt; b += kSpmmThreads) Ys[(size_t)(nr - 1) * ys_ld + b] = 0.f;

  // stage the tile's gather indices and weights (one memory round trip)
  {
    const TV *val = reinterpret_cast<const TV *>(P.val);
    const uint32_t src_max = (uint32_t)(P.n_src - 1);
    const uint32_t nnz_max = (uint32_t)(P.nnz > 0 ? P.nnz - 1 : 0);
    const int nn = j1 - j0;
    for (int q0 = 0; q0 < nn; q0 += 4 * kSpmmThreads) {
      uint32_t cc[4], ss[4];
      float vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * kSpmmThreads + tid;
        cc[u] = 0u;
        ss[u] = 0u;
        vv[u] = 0.f;
        if (q < nn) {
          cc[u] = P.idx16 ? (uint32_t)ld_stream(P.idx16 + j0 + q) : (uint32_t)ld_stream(P.idx + j0 + q);
          if (kGatherVal) {
            uint32_t sidx = (uint32_t)ld_stream(P.val_src + j0 + q);
            ss[u] = sidx < nnz_max ? sidx : nnz_max;
            vv[u] = to_f32(ld_keep(val + ss[u]));
          } else {
            vv[u] = to_f32(ld_stream(val + j0 + q));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * kSpmmThreads + tid;
        if (q < nn) {
          s_iv[q] = make_uint2((cc[u] < src_max ? cc[u] : src_max) * (uint32_t)bg.ldx, __float_as_uint(vv[u]));
          if (kFuseDw) s_src[q] = ss[u];
        }
      }
    }
    for (int q = nn + tid; q < nn + kStagePad; q += kSpmmThreads) {
      s_iv[q] = make_uint2(0u, 0u);
      if (kFuseDw) s_src[q] = 0u;
    }
  }
  __syncthreads();

  // warp ranges: equal cost slices of [c0, c1]
  if (tid <= kSpmmWarps) {
    const int64_t c0 = (int64_t)w * i0 + j0, c1 = (int64_t)w * i1 + j1;
    const int64_t D = c0 + (c1 - c0) * tid / kSpmmWarps;
    int lo = i0, hi = i1;
    while (lo < hi) {
      int mid = lo + (hi - lo + 1) / 2;
      if ((int64_t)w * mid + rps[mid - i0] <= D)
        lo = mid;
      else
        hi = mid - 1;
    }
    int64_t j = D - (int64_t)w * lo;
    int64_t lim = rps[lo - i0 + 1];
    if (j > lim) j = lim;
    if (j > j1) j = j1;
    if (j < j0) j = j0;
    if (tid == kSpmmWarps) j = j1;
    wsp[2 * tid] = lo;
    wsp[2 * tid + 1] = (int)j;
  }
  __syncthreads();

  const int wi0 = wsp[2 * warp], wj0 = wsp[2 * warp + 1];
  const int wi1 = wsp[2 * warp + 2], wj1 = wsp[2 * warp + 3];
  const TA *xt = reinterpret_cast<const TA *>(P.xt) + b0 + g * V;

  for (int i = wi0; i <= wi1; ++i) {
    const int ps = max(rps[i - i0], wj0) - j0;
    const int pe = min(i < wi1 ? rps[i - i0 + 1] : wj1, j1) - j0;
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    float xc[V];  // kFuseDw: this column's X slice
    if (kFuseDw) {
      const int ci = i < P.n_rows ? i : P.n_rows - 1;
      if (ps < pe)
        Slice<TA, V>::load(reinterpret_cast<const TA *>(P.xt_dw) + (size_t)ci * bg.ldx + b0 + g * V, xc);
      else
#pragma unroll
        for (int e = 0; e < V; ++e) xc[e] = 0.f;
    }
    for (int base = ps; base < pe; base += kSlots * kU) {
      uint32_t c[kU];
      float v[kU];
      const int k0 = base + slot;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint2 iv = s_iv[k0 + u * kSlots];
        c[u] = iv.x;
        v[u] = __uint_as_float(iv.y);
      }
      if (base + kSlots * kU > pe) {  // last group of the row: weights past its end count zero
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = k0 + u * kSlots < pe ? v[u] : 0.f;
      }
      float x[kU][V];
#pragma unroll
      for (int u = 0; u < kU; ++u) Slice<TA, V>::load(xt + c[u], x[u]);
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(v[u], x[u][e], acc[e]);
      if (kFuseDw) {
        float d[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          d[u] = 0.f;
#pragma unroll
          for (int e = 0; e < V; ++e) d[u] = fmaf(x[u][e], xc[e], d[u]);
        }
        if constexpr (kU == 4 && G >= 4) {
          // transposed reduction over the slot's G lanes: the first two steps
          // halve the values each lane carries (4 -> 2 -> 1), so four
          // shuffles (plus log2(G/4)) replace 4 * log2(G); lane g with
          // g % (G/4) == 0 ends with the full sum of weight u = g / (G/4)
          constexpr int h1 = G / 2, h2 = G / 4;
          const bool up1 = (g & h1) != 0, up2 = (g & h2) != 0;
          const float e0 = (up1 ? d[2] : d[0]) + __shfl_xor_sync(0xffffffffu, up1 ? d[0] : d[2], h1);
          const float e1 = (up1 ? d[3] : d[1]) + __shfl_xor_sync(0xffffffffu, up1 ? d[1] : d[3], h1);
          float f = (up2 ? e1 : e0) + __shfl_xor_sync(0xffffffffu, up2 ? e0 : e1, h2);
#pragma unroll
          for (int off = 1; off < h2; off <<= 1) f += __shfl_xor_sync(0xffffffffu, f, off);
          if ((g & (h2 - 1)) == 0) {
            const int k = base + ((up1 ? 2 : 0) + (up2 ? 1 : 0)) * kSlots + slot;
            if (k < pe) P.dw[s_src[k]] = f;
          }
        } else {
#pragma unroll
          for (int off = 1; off < G; off <<= 1)
#pragma unroll
            for (int u = 0; u < kU; ++u) d[u] += __shfl_xor_sync(0xffffffffu, d[u], off);
          if (g == 0) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const int k = base + u * kSlots + slot;
              if (k < pe) P.dw[s_src[k]] = d[u];
            }
          }
        }
      }
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    if (slot == 0) {
      float *dst = i < wi1 ? Ys + (size_t)(i - i0) * ys_ld + g * V : wcar + warp * bt + g * V;
#pragma unroll
      for (int e = 0; e < V; ++e) dst[e] = acc[e];
    }
  }
  __syncthreads();

  // rows split between warps: add the carries in warp order
  for (int b = tid; b < bt; b += kSpmmThreads) {
#pragma unroll 1
    for (int k = 0; k < kSpmmWarps; ++k) {
      int r = wsp[2 * k + 2];
      Ys[(size_t)(r - i0) * ys_ld + b] += wcar[k * bt + b];
    }
  }
  __syncthreads();

  const int nfin = nr - 1;  // rows i0 .. i1-1 end in this tile
  const bool continued = rps[0] < j0;
  const size_t slot_base = ((size_t)bi * P.tg.n_tiles + t) * bt;
  if (i1 < P.n_rows)
    for (int b = tid; b < bt; b += kSpmmThreads) P.carry[slot_base + b] = Ys[(size_t)(nr - 1) * ys_ld + b];
  if (nfin >= 1 && continued)
    for (int b = tid; b < bt; b += kSpmmThreads) P.head[slot_base + b] = Ys[b];
  const int rs = continued ? 1 : 0;
  const int nw = nfin - rs;
  if (nw > 0) {
    TA *y = reinterpret_cast<TA *>(P.y);
    const int bmax = min(bt, P.batch - b0);
    if (nw <= 32) {  // a warp covers 32 / 2^lg batch rows of up to 2^lg outputs at once
      const int lg = nw <= 1 ? 0 : 32 - __clz(nw - 1);
      const int per = 32 >> lg, sub = lane >> lg, q = lane & ((1 << lg) - 1);
      if (q < nw) {
        const float bq = P.bias ? P.bias[i0 + rs + q] : 0.f;
        for (int b = warp * per + sub; b < bmax; b += kSpmmWarps * per) {
          const size_t off = (size_t)(b0 + b) * P.n_rows + i0 + rs + q;
          float s = Ys[(size_t)(q + rs) * ys_ld + b];
          if (P.bias) s = bq + s;
          y[off] = spmm_epilogue<TA>(P, s, off);
        }
      }
    } else {
      for (int b = warp; b < bmax; b += kSpmmWarps) {
        const size_t rowoff = (size_t)(b0 + b) * P.n_rows + i0 + rs;
        for (int q = lane; q < nw; q += 32) {
          float s = Ys[(size_t)(q + rs) * ys_ld + b];
          if (P.bias) s = P.bias[i0 + rs + q] + s;
          y[rowoff + q] = spmm_epilogue<TA>(P, s, rowoff + q);
        }
      }
    }
  }
}

// Rows whose first stored weights sit in earlier tiles: bias + carries (tile
// order) + head, written once.
template <typename TA>
__global__ void k_spmm_fixup(SpmmParams P, BatchGeom bg) {
  pdl_wait();
  const int t = blockIdx.x, bi = blockIdx.y;
  const int i0 = P.tiles[2 * t], j0 = P.tiles[2 * t + 1], i1 = P.tiles[2 * t + 2];
  if (i1 <= i0 || i0 >= P.n_rows) return;
  if (P.ptr[i0] >= j0) return;
  int first = t - 1;
  while (first > 0 && P.tiles[2 * first] == i0) --first;
  const int bt = bg.bt, b0 = bi * bt;
  TA *y = reinterpret_cast<TA *>(P.y);
  for (int b = threadIdx.x; b < bt && b0 + b < P.batch; b += blockDim.x) {
    float s = 0.f;
    for (int u = first; u < t; ++u) s += P.carry[((size_t)bi * P.tg.n_tiles + u) * bt + b];
    s += P.head[((size_t)bi * P.tg.n_tiles + t) * bt + b];
    if (P.bias) s = P.bias[i0] + s;
    const size_t off = (size_t)(b0 + b) * P.n_rows + i0;
    y[off] = spmm_epilogue<TA>(P, s, off);
  }
}

// a [batch][n] -> at [n][ldx], zero-filled for b in [batch, ldx)
template <typename T>
__global__ void k_transpose(const T *__restrict__ a, int batch, int n, T *__restrict__ at, int ldx) {
  pdl_wait();
  __shared__ T tile[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int c0 = blockIdx.x * 32, b0 = blockIdx.y * 32;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int b = b0 + ty + 8 * j, c = c0 + tx;
    T v = from_f32<T>(0.f);
    if (b < batch && c < n) v = a[(size_t)b * n + c];
    tile[ty + 8 * j][tx] = v;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int c = c0 + ty + 8 * j, b = b0 + tx;
    if (c < n && b < ldx) at[(size_t)c * ldx + b] = tile[tx][ty + 8 * j];
  }
}

// Two transposes in one launch (blockIdx.z picks the matrix): a0 [batch][n0]
// -> at0 [n0][ldx] and a1 [batch][n1] -> at1 [n1][ldx].  When the whole
// batch fits one 32-row tile, the blocks of the first matrix also write its
// column sums db0[c] = sum_b a0[b][c] (b increasing) from the staged tile.
template <typename T>
struct TransposePair {
  const T *a0, *a1;
  T *at0, *at1;
  int n0, n1;
  float *db0;  // or null
};

template <typename T>
__global__ void k_transpose2(TransposePair<T> tp, int batch, int ldx) {
  pdl_wait();
  __shared__ T tile[32][33];
  const bool second = blockIdx.z == 1;
  const T *a = second ? tp.a1 : tp.a0;
  T *at = second ? tp.at1 : tp.at0;
  const int n = second ? tp.n1 : tp.n0;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int c0 = blockIdx.x * 32, b0 = blockIdx.y * 32;
  if (c0 >= n) return;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int b = b0 + ty + 8 * j, c = c0 + tx;
    T v = from_f32<T>(0.f);
    if (b < batch && c < n) v = a[(size_t)b * n + c];
    tile[ty + 8 * j][tx] = v;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int c = c0 + ty + 8 * j, b = b0 + tx;
    if (c < n && b < ldx) at[(size_t)c * ldx + b] = tile[tx][ty + 8 * j];
  }
  if (!second && tp.db0 && gridDim.y == 1 && ty == 0 && c0 + tx < n) {
    float s = 0.f;
    for (int b = 0; b < batch; ++b) s += to_f32(tile[b][tx]);
    tp.db0[c0 + tx] = s;
  }
}

// out[c] = sum_b a[b][c], b increasing
template <typename T>
__global__ void k_colsum(const T *__restrict__ a, int batch, int n, float *__restrict__ out) {
  pdl_wait();
  int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= n) return;
  float s = 0.f;
  for (int b = 0; b < batch; ++b) s += to_f32(a[(size_t)b * n + c]);
  out[c] = s;
}

// out[r] = sum_b at[r][b] over the feature-major copy (rows ldx apart): one
// warp per row, each lane adding 16-byte runs of the row (single elements,
// lane-strided, when rows are not 16-byte aligned), the lanes' sums combined
// by a fixed shuffle tree, so the result does not depend on scheduling.
template <typename T>
__global__ void __launch_bounds__(256) k_rowsum_t(const T *__restrict__ at, int ldx, int batch, int n,
                                                  float *__restrict__ out) {
  pdl_wait();
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= n) return;
  const T *p = at + (size_t)r * ldx;
  float s = 0.f;
  constexpr int kV = 16 / (int)sizeof(T);  // elements per 16-byte load
  if (ldx % kV == 0) {  // rows start on 16-byte boundaries: a lane adds kV consecutive elements per load
    const int nv = batch / kV;
#pragma unroll 2
    for (int v = lane; v < nv; v += 32) {
      const uint4 q = *reinterpret_cast<const uint4 *>(p + (size_t)v * kV);
      const T *e = reinterpret_cast<const T *>(&q);
#pragma unroll
      for (int k = 0; k < kV; ++k) s += to_f32(e[k]);
    }
    for (int b = nv * kV + lane; b < batch; b += 32) s += to_f32(p[b]);
  } else {
#pragma unroll 4
    for (int b = lane; b < batch; b += 32) s += to_f32(p[b]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) out[r] = s;
}

// dw[k] = sum_b dyt[row[k]][b] * xt[col[k]][b].  One CTA per chunk of at
// most kDwChunk stored weights (fewer for wide batches, so the grid still
// fills the GPU): indices staged in shared memory, results gathered in shared
// memory and written back contiguously.
constexpr int kDwChunk = 2048;

template <int V, int G>
struct DwUnroll {
  static constexpr int kSlots = 32 / G;
  static constexpr int value = V >= 8 ? 2 : (kSlots >= 8 && V >= 4 ? 2 : 4);
};

template <typename TA, int V, int G>
__global__ void __launch_bounds__(256) k_sddmm(int64_t nnz, const int32_t *__restrict__ row,
                                               const int32_t *__restrict__ col, int32_t out_f, int32_t in_f,
                                               const TA *__restrict__ xt, const TA *__restrict__ dyt, int ldx,
                                               int n_chunks, int chunk, float *__restrict__ dw) {
  pdl_wait();
  constexpr int kSlots = 32 / G;
  constexpr int kU = DwUnroll<V, G>::value;
  const int per_warp = (chunk + 7) / 8;
  __shared__ uint32_t s_row[kDwChunk];
  __shared__ uint32_t s_col[kDwChunk];
  __shared__ float s_out[kDwChunk];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane / G, g = lane % G;
  const int64_t k0 = (int64_t)blockIdx.x * chunk;
  const int n = (int)min((int64_t)chunk, nnz - k0);
  const uint32_t rmax = (uint32_t)(out_f - 1), cmax = (uint32_t)(in_f - 1);
  for (int q0 = 0; q0 < n; q0 += 4 * 256) {
    uint32_t rr[4], cc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      int q = q0 + u * 256 + tid;
      rr[u] = q < n ? (uint32_t)ld_stream(row + k0 + q) : 0u;
      cc[u] = q < n ? (uint32_t)ld_stream(col + k0 + q) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      int q = q0 + u * 256 + tid;
      if (q < n) {
        s_row[q] = rr[u] < rmax ? rr[u] : rmax;
        s_col[q] = cc[u] < cmax ? cc[u] : cmax;
      }
    }
  }
  __syncthreads();
  const int bt = G * V;
  const int wq0 = min(n, warp * per_warp), wq1 = min(n, wq0 + per_warp);
  for (int base = wq0; base < wq1; base += kSlots * kU) {
    uint32_t r[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      int q = base + u * kSlots + slot;
      bool ok = q < wq1;
      r[u] = ok ? s_row[q] : 0u;
      c[u] = ok ? s_col[q] : 0u;
    }
    float acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = 0.f;
    for (int ch = 0; ch < n_chunks; ++ch) {
      const int off = ch * bt + g * V;
      float dyv[kU][V], xv[kU][V];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        Slice<TA, V>::load(dyt + (size_t)r[u] * ldx + off, dyv[u]);
        Slice<TA, V>::load(xt + (size_t)c[u] * ldx + off, xv[u]);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[u] = fmaf(dyv[u][e], xv[u][e], acc[u]);
    }
#pragma unroll
    for (int off = 1; off < G; off <<= 1)
#pragma unroll
      for (int u = 0; u < kU; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
    if (g == 0) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        int q = base + u * kSlots + slot;
        if (q < wq1) s_out[q] = acc[u];
      }
    }
  }
  __syncthreads();
  for (int q = tid; q < n; q += 256) dw[k0 + q] = s_out[q];
}

// Weight gradient in storage (row) order when one batch tile covers the
// batch: a slot keeps the dY slice of its current row in registers and
// reloads it only when its next stored weight starts a new row, so each
// stored weight gathers one activation slice (X[col]) instead of two.
// Chunks, staging and output as in k_sddmm.
template <typename TA, int V, int G>
__global__ void __launch_bounds__(256) k_sddmm_rows(int64_t nnz, const int32_t *__restrict__ row,
                                                    const int32_t *__restrict__ col, int32_t out_f, int32_t in_f,
                                                    const TA *__restrict__ xt, const TA *__restrict__ dyt, int ldx,
                                                    int chunk, float *__restrict__ dw) {
  pdl_wait();
  constexpr int kSlots = 32 / G;
  constexpr int kU = DwUnroll<V, G>::value;
  const int per_warp = (chunk + 7) / 8;
  __shared__ uint32_t s_row[kDwChunk];
  __shared__ uint32_t s_col[kDwChunk];
  __shared__ float s_out[kDwChunk];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane / G, g = lane % G;
  const int64_t k0 = (int64_t)blockIdx.x * chunk;
  const int n = (int)min((int64_t)chunk, nnz - k0);
  const uint32_t rmax = (uint32_t)(out_f - 1), cmax = (uint32_t)(in_f - 1);
  for (int q0 = 0; q0 < n; q0 += 4 * 256) {
    uint32_t rr[4], cc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      int q = q0 + u * 256 + tid;
      rr[u] = q < n ? (uint32_t)ld_stream(row + k0 + q) : 0u;
      cc[u] = q < n ? (uint32_t)ld_stream(col + k0 + q) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      int q = q0 + u * 256 + tid;
      if (q < n) {
        s_row[q] = rr[u] < rmax ? rr[u] : rmax;
        s_col[q] = cc[u] < cmax ? cc[u] : cmax;
      }
    }
  }
  __syncthreads();
  const int wq0 = min(n, warp * per_warp), wq1 = min(n, wq0 + per_warp);
  uint32_t cur = 0xFFFFFFFFu;  // the row whose dY slice dyv holds
  float dyv[V];
#pragma unroll
  for (int e = 0; e < V; ++e) dyv[e] = 0.f;
  const TA *xb = xt + g * V;
  const TA *db = dyt + g * V;
  for (int base = wq0; base < wq1; base += kSlots * kU) {
    uint32_t c[kU];
    float xv[kU][V];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = base + u * kSlots + slot;
      c[u] = q < wq1 ? s_col[q] : 0u;
      Slice<TA, V>::load(xb + (size_t)c[u] * ldx, xv[u]);
    }
    float acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = base + u * kSlots + slot;
      const uint32_t r = q < wq1 ? s_row[q] : cur;
      if (r != cur) {  // the G lanes of a slot take this branch together
        Slice<TA, V>::load(db + (size_t)r * ldx, dyv);
        cur = r;
      }
      acc[u] = 0.f;
#pragma unroll
      for (int e = 0; e < V; ++e) acc[u] = fmaf(dyv[e], xv[u][e], acc[u]);
    }
#pragma unroll
    for (int off = 1; off < G; off <<= 1)
#pragma unroll
      for (int u = 0; u < kU; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
    if (g == 0) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int q = base + u * kSlots + slot;
        if (q < wq1) s_out[q] = acc[u];
      }
    }
  }
  __syncthreads();
  for (int q = tid; q < n; q += 256) dw[k0 + q] = s_out[q];
}

// Forward of a layer with a constant fan-in (every row holds K stored
// weights, rows at k = r K): kEllRows whole rows per CTA, a warp per row at a
// time, no merge-path search, no split rows, no fix-up.  The warp loads its
// row's indices and weights 32 at a time (one per lane), slots of G lanes
// take them in turn and gather their Xt slices; the row sums reduce across
// slots into shared memory, and outputs leave as contiguous runs of Y[b, r0:].
constexpr int kEllRows = 32;
constexpr int kEllThreads = 256;

template <typename TA, typename TV, int V, int G>
__global__ void __launch_bounds__(kEllThreads) k_ell_fwd(SpmmParams P, BatchGeom bg, int32_t K) {
  pdl_wait();
  constexpr int kSlots = 32 / G;
  constexpr int kSteps = 32 / kSlots;           // slot steps per group of 32 stored weights
  constexpr int kU = kSteps < 4 ? kSteps : 4;   // steps in flight
  extern __shared__ __align__(16) float ys[];  // [kEllRows][bt + 1]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = lane / G, g = lane % G;
  const int bt = bg.bt, ys_ld = bt + 1;
  const int r0 = blockIdx.x * kEllRows, b0 = blockIdx.y * bt;
  const TA *xt = reinterpret_cast<const TA *>(P.xt) + b0 + g * V;
  const TV *val = reinterpret_cast<const TV *>(P.val);
  const uint32_t src_max = (uint32_t)(P.n_src - 1);
  for (int rr = warp; rr < kEllRows; rr += kEllThreads / 32) {
    const int r = r0 + rr;
    if (r >= P.n_rows) break;
    const int64_t k0 = (int64_t)r * K, k1 = k0 + K;
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    for (int64_t kb = k0; kb < k1; kb += 32) {
      const int64_t k = kb + lane;
      uint32_t c = 0u;
      float v = 0.f;
      if (k < k1) {
        c = P.idx16 ? (uint32_t)ld_stream(P.idx16 + k) : (uint32_t)ld_stream(P.idx + k);
        c = c < src_max ? c : src_max;
        v = to_f32(ld_stream(val + k));
      }
#pragma unroll
      for (int s0 = 0; s0 < kSteps; s0 += kU) {
        float x[kU][V], vv[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int e = (s0 + u) * kSlots + slot;  // < 32
          const uint32_t cc = __shfl_sync(0xffffffffu, c, e);
          vv[u] = __shfl_sync(0xffffffffu, v, e);
          Slice<TA, V>::load(xt + (size_t)cc * bg.ldx, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = fmaf(vv[u], x[u][e], acc[e]);
      }
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    if (slot == 0)
#pragma unroll
      for (int e = 0; e < V; ++e) ys[rr * ys_ld + g * V + e] = acc[e];
  }
  __syncthreads();
  TA *y = reinterpret_cast<TA *>(P.y);
  const int nr = min(kEllRows, P.n_rows - r0);
  const int bmax = min(bt, P.batch - b0);
  for (int i = threadIdx.x; i < nr * bmax; i += kEllThreads) {
    const int b = i / nr, q = i % nr;  // consecutive threads: consecutive outputs of one batch row
    float s = ys[q * ys_ld + b];
    if (P.bias) s = P.bias[r0 + q] + s;
    const size_t off = (size_t)(b0 + b) * P.n_rows + r0 + q;
    y[off] = spmm_epilogue<TA>(P, s, off);
  }
}

// ------------------------------------------------------------------ host

template <typename TA, typename TV, int V, int G, bool kGV, bool kFuse>
cudaError_t launch_spmm_v(const SpmmParams &p, const BatchGeom &bg, cudaStream_t s) {
  size_t smem = spmm_smem_bytes(p.tg, bg.bt) + (kFuse ? (size_t)tile_stage_len(p.tg) * 4 : 0);
  auto kern = k_spmm_tiles<TA, TV, V, G, kGV, kFuse>;
  cudaError_t e = raise_smem_limit(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.tg.n_tiles, bg.n_btiles);
  launch_pdl(kern, grid, kSpmmThreads, smem, s, p, bg);
  int fx = bg.bt < 32 ? 32 : (bg.bt > 256 ? 256 : bg.bt);
  launch_pdl(k_spmm_fixup<TA>, grid, fx, 0, s, p, bg);
  return cudaGetLastError();
}

template <typename TA, typename TV, bool kGV, bool kFuse>
cudaError_t launch_spmm(const SpmmParams &p, const BatchGeom &bg, cudaStream_t s) {
  constexpr int VV = ActTraits<TA>::kVec;
  if (bg.V == 1) return launch_spmm_v<TA, TV, 1, 1, kGV, kFuse>(p, bg, s);
  switch (bg.G) {
    case 1: return launch_spmm_v<TA, TV, VV, 1, kGV, kFuse>(p, bg, s);
    case 2: return launch_spmm_v<TA, TV, VV, 2, kGV, kFuse>(p, bg, s);
    case 4: return launch_spmm_v<TA, TV, VV, 4, kGV, kFuse>(p, bg, s);
    case 8: return launch_spmm_v<TA, TV, VV, 8, kGV, kFuse>(p, bg, s);
    case 16: return launch_spmm_v<TA, TV, VV, 16, kGV, kFuse>(p, bg, s);
    case 32: return launch_spmm_v<TA, TV, VV, 32, kGV, kFuse>(p, bg, s);
  }
  return cudaErrorInvalidValue;
}

template <typename TA, typename TV, int V, int G>
cudaError_t launch_ell_v(const SpmmParams &p, const BatchGeom &bg, int32_t K, cudaStream_t s) {
  const size_t smem = (size_t)kEllRows * (bg.bt + 1) * sizeof(float);
  cudaError_t e = raise_smem_limit(k_ell_fwd<TA, TV, V, G>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.n_rows + kEllRows - 1) / kEllRows), bg.n_btiles);
  launch_pdl(k_ell_fwd<TA, TV, V, G>, grid, kEllThreads, smem, s, p, bg, K);
  return cudaGetLastError();
}

template <typename TA, typename TV>
cudaError_t launch_ell(const SpmmParams &p, const BatchGeom &bg, int32_t K, cudaStream_t s) {
  constexpr int VV = ActTraits<TA>::kVec;
  if (bg.V == 1) return launch_ell_v<TA, TV, 1, 1>(p, bg, K, s);
  switch (bg.G) {
    case 1: return launch_ell_v<TA, TV, VV, 1>(p, bg, K, s);
    case 2: return launch_ell_v<TA, TV, VV, 2>(p, bg, K, s);
    case 4: return launch_ell_v<TA, TV, VV, 4>(p, bg, K, s);
    case 8: return launch_ell_v<TA, TV, VV, 8>(p, bg, K, s);
    case 16: return launch_ell_v<TA, TV, VV, 16>(p, bg, K, s);
    case 32: return launch_ell_v<TA, TV, VV, 32>(p, bg, K, s);
  }
  return cudaErrorInvalidValue;
}

template <typename TA, int V, int G>
cudaError_t launch_sddmm_v(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                           const TA *xt, const TA *dyt, const BatchGeom &bg, float *dw, int num_sms,
                           cudaStream_t s) {
  // chunk: ~64K batch elements of work per CTA, at least two CTAs per SM
  int64_t chunk = 65536 / (bg.ldx > 0 ? bg.ldx : 1);
  int64_t fill = (nnz + 2 * (int64_t)num_sms - 1) / (2 * (int64_t)num_sms);
  if (chunk > fill) chunk = fill;
  chunk = (chunk + 63) / 64 * 64;
  if (chunk < 64) chunk = 64;
  if (chunk > kDwChunk) chunk = kDwChunk;
  int64_t blocks = (nnz + chunk - 1) / chunk;
  int n_chunks = bg.ldx / bg.bt;
  if (n_chunks == 1)  // one batch tile: each slot keeps its row's dY slice
    launch_pdl(k_sddmm_rows<TA, V, G>, (unsigned)blocks, 256, 0, s, nnz, row, col, out_f, in_f, xt, dyt, bg.ldx,
               (int)chunk, dw);
  else
    launch_pdl(k_sddmm<TA, V, G>, (unsigned)blocks, 256, 0, s, nnz, row, col, out_f, in_f, xt, dyt, bg.ldx, n_chunks,
               (int)chunk, dw);
  return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_sddmm(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                         const TA *xt, const TA *dyt, const BatchGeom &bg, float *dw, int num_sms,
                         cudaStream_t s) {
  constexpr int VV = ActTraits<TA>::kVec;
  if (nnz <= 0) return cudaSuccess;
  if (bg.V == 1) return launch_sddmm_v<TA, 1, 1>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
  switch (bg.G) {
    case 1: return launch_sddmm_v<TA, VV, 1>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
    case 2: return launch_sddmm_v<TA, VV, 2>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
    case 4: return launch_sddmm_v<TA, VV, 4>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
    case 8: return launch_sddmm_v<TA, VV, 8>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
    case 16: return launch_sddmm_v<TA, VV, 16>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
    case 32: return launch_sddmm_v<TA, VV, 32>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_transpose(const T *a, int batch, int n, T *at, int ldx, cudaStream_t s) {
  dim3 grid((n + 31) / 32, (ldx + 31) / 32);
  launch_pdl(k_transpose<T>, grid, dim3(32, 8), 0, s, a, batch, n, at, ldx);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_colsum(const T *a, int batch, int n, float *out, cudaStream_t s) {
  launch_pdl(k_colsum<T>, (n + 255) / 256, 256, 0, s, a, batch, n, out);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_transpose2(const TransposePair<T> &tp, int batch, int ldx, cudaStream_t s) {
  const int n = tp.n0 > tp.n1 ? tp.n0 : tp.n1;
  dim3 grid((n + 31) / 32, (ldx + 31) / 32, 2);
  launch_pdl(k_transpose2<T>, grid, dim3(32, 8), 0, s, tp, batch, ldx);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rowsum_t(const T *at, int ldx, int batch, int n, float *out, cudaStream_t s) {
  launch_pdl(k_rowsum_t<T>, (n + 7) / 8, 256, 0, s, at, ldx, batch, n, out);
  return cudaGetLastError();
}

// per-dtype entry points (explicitly instantiated in spmm_f32.cu / spmm_bf16.cu)
// gather_val: column-view mode (input gradient); fuse_dw: also the weight
// gradient (column-view mode with a single batch tile only)
template <typename T>
cudaError_t run_spmm(const SpmmParams &p, const BatchGeom &bg, bool gather_val, bool fuse_dw, cudaStream_t s);
template <typename T>
cudaError_t run_sddmm(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                      const T *xt, const T *dyt, const BatchGeom &bg, float *dw, int num_sms, cudaStream_t s);
template <typename T>
cudaError_t run_transpose(const T *a, int batch, int n, T *at, int ldx, cudaStream_t s);
// forward of a constant-fan-in layer (K stored weights in every row)
template <typename T>
cudaError_t run_ell(const SpmmParams &p, const BatchGeom &bg, int32_t K, cudaStream_t s);
template <typename T>
cudaError_t run_colsum(const T *a, int batch, int n, float *out, cudaStream_t s);
template <typename T>
cudaError_t run_rowsum_t(const T *at, int ldx, int batch, int n, float *out, cudaStream_t s);
template <typename T>
cudaError_t run_transpose2(const TransposePair<T> &tp, int batch, int ldx, cudaStream_t s);

// Small-batch path (spmm_small.cu): batch <= kSmallMaxBatch, the gathered
// operand read batch-major (no transposed copy), one launch per call.  In
// column-view mode with fuse_dw it also writes dw at storage index and, when
// p.db is set, the bias gradient; p.y == null skips the input gradient.
constexpr int kSmallMaxBatch = 8;
constexpr size_t kSmallMaxStage = 96 * 1024;  // bytes of the operand copy a CTA stages
int small_batch_width(int batch);
bool small_path_ok(int batch, int n_src, size_t elem);
template <typename T>
cudaError_t run_spmm_small(const SpmmParams &p, bool gather_val, bool fuse_dw, int num_sms, cudaStream_t s);
// Weight gradient alone on a small layer at small batch: a flat pass over
// the stored weights (no row structure, no transposed copies) when nnz times
// the padded batch width is at most kSmallDwFlatLoads.
constexpr int64_t kSmallDwFlatLoads = int64_t(1) << 22;
bool small_dw_flat_ok(int batch, int64_t nnz);
template <typename T>
cudaError_t run_sddmm_small(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                            const T *x, const T *dy, int batch, float *dw, float *db, int num_sms, cudaStream_t s);

}  // namespace snack
