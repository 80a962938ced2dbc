// Device-wide building blocks used by the plan builder and the restructure:
//  * scan_apply: exclusive prefix sum over a generated sequence f(i), then a
//    per-element callback out(i, exclusive, value) -- reduce-then-scan in
//    two launches (each second-pass block sums the tile totals before it),
//    no inter-block waiting;
//  * radix_sort: stable LSD radix sort of 32/64-bit keys with an optional
//    32-bit payload, 8-bit digits, per-warp stable ranking via match_any.
// All results are deterministic.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace snack {

// ------------------------------------------------------------------ scan

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T u = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

// Exclusive scan across the block (blockDim.x == kThreads, at most 1024).
// Returns the thread's exclusive prefix; *total gets the block sum.
template <typename T, int kThreads = kScanThreads>
__device__ __forceinline__ T block_exclusive_scan(T v, T *total) {
  constexpr int kNW = kThreads / 32;
  __shared__ T warp_tot[kNW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T inc = warp_inclusive_scan(v);
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = lane < kNW ? warp_tot[lane] : T(0);
    T wi = warp_inclusive_scan(w);
    if (lane < kNW) warp_tot[lane] = wi - w;  // exclusive over warps
    if (lane == kNW - 1) *total = wi;
  }
  __syncthreads();
  T excl = warp_tot[warp] + inc - v;
  __syncthreads();  // warp_tot may be reused by the next call
  return excl;
}

// One padding element per 128 bytes keeps the blocked read (thread t reads
// elements 8t..8t+7) free of bank conflicts.
template <typename T>
__device__ __forceinline__ int scan_pad(int e) {
  return e + e / (int)(128 / sizeof(T));
}

// Payload loaded with the scanned value (before the block scan), so the
// callback's operands do not cost a second memory round trip.
struct NoPayload {
  __device__ int operator()(int64_t) const { return 0; }
};

template <typename T, typename F>
__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(F f, int64_t n, T *block_sums) {
  pdl_wait();
  const int64_t base = (int64_t)blockIdx.x * kScanTile;
  T s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    int64_t idx = base + (int64_t)i * kScanThreads + threadIdx.x;
    if (idx < n) s += f(idx);
  }
  __shared__ T tot;
  T ignored = block_exclusive_scan<T>(s, &tot);
  (void)ignored;
  if (threadIdx.x == 0) block_sums[blockIdx.x] = tot;
}

// One block: exclusive scan of the block sums in place; grand total to *total.
template <typename T>
__global__ void __launch_bounds__(kScanThreads) k_scan_spine(T *sums, int64_t nb, T *total) {
  pdl_wait();
  __shared__ T chunk_tot;
  T carry = 0;
  for (int64_t c = 0; c < nb; c += kScanThreads) {
    int64_t idx = c + threadIdx.x;
    T v = idx < nb ? sums[idx] : T(0);
    T ex = block_exclusive_scan<T>(v, &chunk_tot);
    if (idx < nb) sums[idx] = carry + ex;
    carry += chunk_tot;
    __syncthreads();
  }
  if (threadIdx.x == 0 && total) *total = carry;
}

// Up to this many tiles, every block of the second pass adds up the sums of
// the tiles before it itself (no spine launch).
constexpr int64_t kScanDirectTiles = 2048;

// Second pass: block b scans its tile and runs the callbacks.  kDirect: its
// prefix is the sum of block_sums[0..b) (and the last block writes the
// total); otherwise block_sums already holds exclusive prefixes.
template <typename T, bool kDirect, typename F, typename PL, typename Out>
__global__ void __launch_bounds__(kScanThreads) k_scan_down(F f, PL pl, int64_t n, const T *block_sums, Out out,
                                                            T *d_total) {
  pdl_wait();
  constexpr int kPadded = kScanTile + kScanTile / (128 / sizeof(T));
  __shared__ T tile[kPadded];
  __shared__ T tile_ex[kPadded];
  __shared__ T tot, pre_tot;
  const int64_t base = (int64_t)blockIdx.x * kScanTile;
  T in[kScanItems];
  decltype(pl(0)) pay[kScanItems];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    int64_t idx = base + i * kScanThreads + threadIdx.x;
    in[i] = idx < n ? f(idx) : T(0);
    pay[i] = idx < n ? pl(idx) : decltype(pl(0))();
  }
  T prefix;
  if (kDirect) {
    T ps = 0;
    for (int64_t q = threadIdx.x; q < (int64_t)blockIdx.x; q += kScanThreads) ps += block_sums[q];
    T ignored = block_exclusive_scan<T>(ps, &pre_tot);
    (void)ignored;
    prefix = pre_tot;
  } else {
    prefix = block_sums[blockIdx.x];
  }
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) tile[scan_pad<T>(i * kScanThreads + threadIdx.x)] = in[i];
  __syncthreads();
  T v[kScanItems];
  T sum = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = tile[scan_pad<T>(threadIdx.x * kScanItems + i)];
    sum += v[i];
  }
  T ex = block_exclusive_scan<T>(sum, &tot) + prefix;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    tile_ex[scan_pad<T>(threadIdx.x * kScanItems + i)] = ex;
    ex += v[i];
  }
  __syncthreads();
  // callbacks in striped order: consecutive threads touch consecutive elements
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int e = i * kScanThreads + threadIdx.x;
    const int64_t idx = base + e;
    if (idx < n) out(idx, tile_ex[scan_pad<T>(e)], in[i], pay[i]);
  }
  if (kDirect && d_total && threadIdx.x == 0 && blockIdx.x == gridDim.x - 1) *d_total = prefix + tot;
}

template <typename T>
inline size_t scan_temp_bytes(int64_t n) {
  int64_t nb = ceil_div(n > 0 ? n : 1, kScanTile);
  return align_up((size_t)(nb + 2) * sizeof(T), kAlign);
}

// Exclusive scan of f(0..n-1); calls out(i, exclusive_i, f(i), pl(i)) for
// every i and writes the total to *d_total (device pointer, may be null).
// temp needs scan_temp_bytes<T>(n).  Reduce-then-scan: two launches on
// `stream` (three above kScanDirectTiles tiles); no block waits on another.
template <typename T, typename F, typename PL, typename Out>
cudaError_t scan_apply_pl(F f, PL pl, int64_t n, Out out, T *d_total, void *temp, cudaStream_t stream) {
  if (n <= 0) {
    if (d_total) return cudaMemsetAsync(d_total, 0, sizeof(T), stream);
    return cudaSuccess;
  }
  const int64_t nb = ceil_div(n, kScanTile);
  T *sums = reinterpret_cast<T *>(temp);
  launch_pdl(k_scan_reduce<T, F>, (unsigned)nb, kScanThreads, 0, stream, f, n, sums);
  if (nb <= kScanDirectTiles) {
    launch_pdl(k_scan_down<T, true, F, PL, Out>, (unsigned)nb, kScanThreads, 0, stream, f, pl, n, sums, out, d_total);
  } else {
    launch_pdl(k_scan_spine<T>, 1, kScanThreads, 0, stream, sums, nb, d_total);
    launch_pdl(k_scan_down<T, false, F, PL, Out>, (unsigned)nb, kScanThreads, 0, stream, f, pl, n, sums, out, d_total);
  }
  return cudaGetLastError();
}

// Without payload: out(i, exclusive_i, f(i), 0).
template <typename T, typename F, typename Out>
cudaError_t scan_apply(F f, int64_t n, Out out, T *d_total, void *temp, cudaStream_t stream) {
  return scan_apply_pl<T>(f, NoPayload{}, n, out, d_total, temp, stream);
}

// ------------------------------------------------------------- radix sort

constexpr int kRadixThreads = 256;
constexpr int kRadixItems = 8;  // per lane, striped within the warp
constexpr int kRadixWarps = kRadixThreads / 32;
constexpr int kRadixTile = kRadixThreads * kRadixItems;  // 2048
constexpr int kRadixBins = 256;

// Sources and sinks of a radix pass: the first pass may generate its keys
// (e.g. from a column array) and the last pass may write its own outputs.
template <typename K>
struct ArraySrc {
  const K *k;
  const uint32_t *v;
  __device__ K key(int64_t i) const { return k[i]; }
  __device__ uint32_t val(int64_t i) const { return v ? v[i] : 0u; }
};

// A sink may gather something per element first (load), all loads of a
// thread in flight together, then write (put).
template <typename K>
struct ArrayDst {
  K *k;
  uint32_t *v;
  __device__ int load(uint32_t) const { return 0; }
  __device__ void put(uint32_t pos, K key, uint32_t val, int) const {
    k[pos] = key;
    if (v) v[pos] = val;
  }
};

template <typename K, typename Src>
__global__ void __launch_bounds__(kRadixThreads) k_radix_hist(Src src, int64_t n, int shift, uint32_t *hist,
                                                              int64_t nb) {
  pdl_wait();
  __shared__ uint32_t h[kRadixWarps][kRadixBins];  // one histogram per warp: less atomic contention
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kRadixWarps * kRadixBins; i += kRadixThreads) (&h[0][0])[i] = 0;
  const int64_t base = (int64_t)blockIdx.x * kRadixTile;
  K kk[kRadixItems];
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {  // all loads in flight before any use
    int64_t idx = base + (int64_t)i * kRadixThreads + threadIdx.x;
    kk[i] = idx < n ? src.key(idx) : K(0);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    int64_t idx = base + (int64_t)i * kRadixThreads + threadIdx.x;
    if (idx < n) atomicAdd(&h[warp][(uint32_t)(kk[i] >> shift) & 0xFF], 1u);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kRadixBins; d += kRadixThreads) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kRadixWarps; ++w) c += h[w][d];
    hist[(int64_t)d * nb + blockIdx.x] = c;
  }
}

// Stable scatter of one tile.  Warp w owns kRadixItems*32 consecutive tile
// elements, striped: item i of lane l is element i*32 + l of that range, so
// visiting items in order and lanes in order visits elements in index order.
// Lanes with equal digits are found with one ballot per digit bit.  Each element gets
// its rank inside the tile's digit-grouped order, the tile is rearranged in
// shared memory, and each digit's run is written to its global slots by
// consecutive threads (coalesced).
template <typename K, typename Src, typename Dst>
__global__ void __launch_bounds__(kRadixThreads) k_radix_scatter(Src src, Dst dst, int64_t n, int shift,
                                                                 const uint32_t *offs, int64_t nb) {
  pdl_wait();
  __shared__ uint32_t cnt[kRadixWarps][kRadixBins];
  __shared__ uint32_t dig_start[kRadixBins];
  __shared__ uint32_t glob[kRadixBins];
  __shared__ uint32_t tile_total;
  extern __shared__ __align__(16) unsigned char rs_smem[];
  K *s_key = reinterpret_cast<K *>(rs_smem);
  uint32_t *s_val = reinterpret_cast<uint32_t *>(s_key + kRadixTile);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kRadixWarps * kRadixBins; i += kRadixThreads) (&cnt[0][0])[i] = 0;
  for (int d = threadIdx.x; d < kRadixBins; d += kRadixThreads)
    glob[d] = offs[(int64_t)d * nb + blockIdx.x];
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kRadixTile + (int64_t)warp * (kRadixItems * 32);
  const uint32_t lt_mask = (1u << lane) - 1u;
  K key[kRadixItems];
  uint32_t val[kRadixItems];
  uint32_t rank[kRadixItems];
  int digit[kRadixItems];
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    int64_t idx = base + i * 32 + lane;
    bool ok = idx < n;
    key[i] = ok ? src.key(idx) : K(0);
    val[i] = ok ? src.val(idx) : 0u;
  }
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    int64_t idx = base + i * 32 + lane;
    digit[i] = idx < n ? (int)((uint32_t)(key[i] >> shift) & 0xFF) : kRadixBins;  // sentinel bin
  }
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    // lanes holding the same digit (sentinel included), from nine ballots
    unsigned peers = 0xffffffffu;
#pragma unroll
    for (int bit = 0; bit < 9; ++bit) {
      const bool on = (digit[i] >> bit) & 1;
      const unsigned bal = __ballot_sync(0xffffffffu, on);
      peers &= on ? bal : ~bal;
    }
    uint32_t before = (uint32_t)__popc(peers & lt_mask);
    uint32_t c = digit[i] < kRadixBins ? cnt[warp][digit[i]] : 0u;
    rank[i] = c + before;
    __syncwarp();
    bool last = (peers >> lane) == 1u;  // highest lane of its group
    if (last && digit[i] < kRadixBins) cnt[warp][digit[i]] = c + (uint32_t)__popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per digit: exclusive offsets across warps, and the digit's total in the tile
  uint32_t tot = 0;
  {
    const int d = threadIdx.x;  // kRadixThreads == kRadixBins
#pragma unroll
    for (int w = 0; w < kRadixWarps; ++w) {
      uint32_t c = cnt[w][d];
      cnt[w][d] = tot;
      tot += c;
    }
  }
  {
    __shared__ uint32_t scan_total;
    uint32_t ex = block_exclusive_scan<uint32_t>(tot, &scan_total);
    dig_start[threadIdx.x] = ex;
    if (threadIdx.x == 0) tile_total = scan_total;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    if (digit[i] < kRadixBins) {
      const uint32_t lpos = dig_start[digit[i]] + cnt[warp][digit[i]] + rank[i];
      s_key[lpos] = key[i];
      s_val[lpos] = val[i];
    }
  }
  __syncthreads();
  const int m = (int)tile_total;
  K ok[kRadixItems];
  uint32_t ov[kRadixItems], opos[kRadixItems];
  int oaux[kRadixItems];
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    const int e = i * kRadixThreads + threadIdx.x;
    if (e < m) {
      ok[i] = s_key[e];
      ov[i] = s_val[e];
      const uint32_t d = (uint32_t)(ok[i] >> shift) & 0xFF;
      opos[i] = glob[d] + (uint32_t)e - dig_start[d];
      oaux[i] = dst.load(ov[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    const int e = i * kRadixThreads + threadIdx.x;
    if (e < m) dst.put(opos[i], ok[i], ov[i], oaux[i]);
  }
}

struct HistRead {
  const uint32_t *h;
  __device__ uint32_t operator()(int64_t i) const { return h[i]; }
};
struct WriteExcl32 {
  uint32_t *o;
  __device__ void operator()(int64_t i, uint32_t ex, uint32_t, int) const { o[i] = ex; }
};

inline size_t radix_temp_bytes(int64_t n) {
  int64_t nb = ceil_div(n > 0 ? n : 1, kRadixTile);
  size_t h = align_up((size_t)nb * kRadixBins * sizeof(uint32_t), kAlign);
  return 2 * h + scan_temp_bytes<uint32_t>(nb * kRadixBins);
}

template <typename K, typename Src, typename Dst>
cudaError_t radix_pass(Src src, Dst dst, int64_t n, int shift, uint32_t *hist, uint32_t *offs, void *stemp,
                       cudaStream_t stream) {
  const int64_t nb = ceil_div(n, kRadixTile);
  launch_pdl(k_radix_hist<K, Src>, (unsigned)nb, kRadixThreads, 0, stream, src, n, shift, hist, nb);
  cudaError_t e = scan_apply<uint32_t>(HistRead{hist}, nb * kRadixBins, WriteExcl32{offs}, (uint32_t *)nullptr,
                                       stemp, stream);
  if (e != cudaSuccess) return e;
  const size_t dyn = (size_t)kRadixTile * (sizeof(K) + sizeof(uint32_t));
  e = raise_smem_limit(k_radix_scatter<K, Src, Dst>, dyn);
  if (e != cudaSuccess) return e;
  launch_pdl(k_radix_scatter<K, Src, Dst>, (unsigned)nb, kRadixThreads, dyn, stream, src, dst, n, shift, offs, nb);
  return cudaGetLastError();
}

// The scatter half of a pass, when the digit-major offsets (exclusive scan of
// the tile histograms, tiles of kRadixTile elements) were made elsewhere.
template <typename K, typename Src, typename Dst>
cudaError_t radix_scatter_only(Src src, Dst dst, int64_t n, int shift, const uint32_t *offs, cudaStream_t stream) {
  const int64_t nb = ceil_div(n, kRadixTile);
  const size_t dyn = (size_t)kRadixTile * (sizeof(K) + sizeof(uint32_t));
  cudaError_t e = raise_smem_limit(k_radix_scatter<K, Src, Dst>, dyn);
  if (e != cudaSuccess) return e;
  launch_pdl(k_radix_scatter<K, Src, Dst>, (unsigned)nb, kRadixThreads, dyn, stream, src, dst, n, shift, offs, nb);
  return cudaGetLastError();
}

// Stable sort by the low `bits` bits of the keys, 8 bits per pass (at least
// one pass).  The first pass reads `first`, the last writes `last`; passes in
// between ping-pong between (k0, v0) and (k1, v1).
template <typename K, typename Src0, typename DstLast>
cudaError_t radix_sort_custom(Src0 first, DstLast last, int64_t n, int bits, K *k0, uint32_t *v0, K *k1,
                              uint32_t *v1, void *temp, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t nb = ceil_div(n, kRadixTile);
  uint8_t *t = reinterpret_cast<uint8_t *>(temp);
  size_t hbytes = align_up((size_t)nb * kRadixBins * sizeof(uint32_t), kAlign);
  uint32_t *hist = reinterpret_cast<uint32_t *>(t);
  uint32_t *offs = reinterpret_cast<uint32_t *>(t + hbytes);
  void *stemp = t + 2 * hbytes;
  const int passes = bits <= 8 ? 1 : (bits + 7) / 8;
  cudaError_t e = cudaSuccess;
  if (passes == 1) return radix_pass<K>(first, last, n, 0, hist, offs, stemp, stream);
  e = radix_pass<K>(first, ArrayDst<K>{k0, v0}, n, 0, hist, offs, stemp, stream);
  if (e != cudaSuccess) return e;
  K *ka = k0, *kb = k1;
  uint32_t *va = v0, *vb = v1;
  for (int p = 1; p < passes - 1; ++p) {
    e = radix_pass<K>(ArraySrc<K>{ka, va}, ArrayDst<K>{kb, vb}, n, 8 * p, hist, offs, stemp, stream);
    if (e != cudaSuccess) return e;
    K *tk = ka;
    ka = kb;
    kb = tk;
    uint32_t *tv = va;
    va = vb;
    vb = tv;
  }
  return radix_pass<K>(ArraySrc<K>{ka, va}, last, n, 8 * (passes - 1), hist, offs, stemp, stream);
}

// ------------------------------------------------------------- bucket sort
//
// Sort n distinct 64-bit keys in [0, key_range): keys are spread over
// equal-width buckets of the key range (about 16 keys per bucket for keys
// drawn uniformly), each bucket is filled in arbitrary order with atomics, and
// one warp per bucket then places every key by its rank within the bucket
// (the number of smaller keys).  Distinct keys make the result unique.

constexpr int kBucketTarget = 16;
constexpr int kBucketSmem = 256;  // keys per warp ranked from shared memory

__device__ __forceinline__ uint32_t bucket_of(uint64_t key, double scale, uint32_t nb) {
  const double b = (double)key * scale;  // monotone in key
  const uint32_t u = b < (double)nb ? (uint32_t)b : nb - 1;
  return u;
}

static __global__ void k_bucket_count(const uint64_t *__restrict__ keys, int64_t n, double scale, uint32_t nb,
                               uint32_t *__restrict__ counts) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    atomicAdd(&counts[bucket_of(keys[i], scale, nb)], 1u);
}

static __global__ void k_bucket_fill(const uint64_t *__restrict__ keys, int64_t n, double scale, uint32_t nb,
                              const uint32_t *__restrict__ offs, uint32_t *__restrict__ fill,
                              uint64_t *__restrict__ tmp) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t k = keys[i];
    const uint32_t b = bucket_of(k, scale, nb);
    tmp[offs[b] + atomicAdd(&fill[b], 1u)] = k;
  }
}

static __global__ void __launch_bounds__(256) k_bucket_rank(const uint64_t *__restrict__ tmp, const uint32_t *__restrict__ offs,
                                                     uint32_t nb, uint64_t *__restrict__ out) {
  pdl_wait();
  __shared__ uint64_t s[8][kBucketSmem];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = (int64_t)blockIdx.x * 8 + warp;
  if (b >= nb) return;
  const uint32_t o = offs[b], L = offs[b + 1] - o;
  if (L <= (uint32_t)kBucketSmem) {
    for (uint32_t i = lane; i < L; i += 32) s[warp][i] = tmp[o + i];
    __syncwarp();
    for (uint32_t i = lane; i < L; i += 32) {
      const uint64_t k = s[warp][i];
      uint32_t r = 0;
      for (uint32_t j = 0; j < L; ++j) r += s[warp][j] < k ? 1u : 0u;
      out[o + r] = k;
    }
  } else {  // rare long bucket: rank from global memory
    for (uint32_t i = lane; i < L; i += 32) {
      const uint64_t k = tmp[o + i];
      uint32_t r = 0;
      for (uint32_t j = 0; j < L; ++j) r += tmp[o + j] < k ? 1u : 0u;
      out[o + r] = k;
    }
  }
}

struct CountRead64 {
  const uint32_t *c;
  __device__ uint32_t operator()(int64_t i) const { return c[i]; }
};
struct WriteOffs {
  uint32_t *o;
  __device__ void operator()(int64_t i, uint32_t ex, uint32_t, int) const { o[i] = ex; }
};

inline uint32_t bucket_count_for(int64_t n) {
  int64_t nb = n / kBucketTarget;
  if (nb < 1) nb = 1;
  if (nb > (1 << 24)) nb = 1 << 24;
  return (uint32_t)nb;
}

inline size_t bucket_sort_temp_bytes(int64_t n) {
  const uint32_t nb = bucket_count_for(n);
  return 2 * align_up((size_t)(nb + 1) * 4, kAlign) + align_up((size_t)(n > 0 ? n : 1) * 8, kAlign) +
         scan_temp_bytes<uint32_t>((int64_t)nb + 1);
}

// keys (n distinct, < key_range) -> out, ascending.  keys and out may not alias.
inline cudaError_t bucket_sort_u64(const uint64_t *keys, int64_t n, uint64_t key_range, uint64_t *out, void *temp,
                                   cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const uint32_t nb = bucket_count_for(n);
  uint8_t *t = reinterpret_cast<uint8_t *>(temp);
  const size_t cb = align_up((size_t)(nb + 1) * 4, kAlign);
  uint32_t *offs = reinterpret_cast<uint32_t *>(t);
  uint32_t *fill = reinterpret_cast<uint32_t *>(t + cb);
  uint64_t *tmp = reinterpret_cast<uint64_t *>(t + 2 * cb);
  void *stemp = t + 2 * cb + align_up((size_t)n * 8, kAlign);
  const double scale = (double)nb / ((double)key_range + 1.0);
  cudaError_t e = cudaMemsetAsync(offs, 0, 2 * cb, stream);  // counts and fill cursors
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((n + 255) / 256 < 65535 * 8 ? (n + 255) / 256 : 65535 * 8);
  launch_pdl(k_bucket_count, grid, 256, 0, stream, keys, n, scale, nb, offs);
  e = scan_apply<uint32_t>(CountRead64{offs}, (int64_t)nb, WriteOffs{offs}, offs + nb, stemp, stream);
  if (e != cudaSuccess) return e;
  launch_pdl(k_bucket_fill, grid, 256, 0, stream, keys, n, scale, nb, offs, fill, tmp);
  launch_pdl(k_bucket_rank, (nb + 7) / 8, 256, 0, stream, tmp, offs, nb, out);
  return cudaGetLastError();
}

// Stable sort by the low `bits` bits of the keys, ping-ponging between
// (k0, v0) and (k1, v1) (v0/v1 may be null); *in_second is set when the
// result ends in (k1, v1).
template <typename K>
cudaError_t radix_sort(K *k0, uint32_t *v0, K *k1, uint32_t *v1, int64_t n, int bits, void *temp,
                       cudaStream_t stream, bool *in_second) {
  *in_second = false;
  if (n <= 1 || bits <= 0) return cudaSuccess;
  const int64_t nb = ceil_div(n, kRadixTile);
  uint8_t *t = reinterpret_cast<uint8_t *>(temp);
  size_t hbytes = align_up((size_t)nb * kRadixBins * sizeof(uint32_t), kAlign);
  uint32_t *hist = reinterpret_cast<uint32_t *>(t);
  uint32_t *offs = reinterpret_cast<uint32_t *>(t + hbytes);
  void *stemp = t + 2 * hbytes;
  K *ka = k0, *kb = k1;
  uint32_t *va = v0, *vb = v1;
  for (int shift = 0; shift < bits; shift += 8) {
    cudaError_t e = radix_pass<K>(ArraySrc<K>{ka, va}, ArrayDst<K>{kb, vb}, n, shift, hist, offs, stemp, stream);
    if (e != cudaSuccess) return e;
    K *tk = ka;
    ka = kb;
    kb = tk;
    uint32_t *tv = va;
    va = vb;
    vb = tv;
    *in_second = !*in_second;
  }
  return cudaSuccess;
}

}  // namespace snack
