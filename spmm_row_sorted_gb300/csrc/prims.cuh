// Device-wide building blocks used by the plan builder and the restructure:
//  * scan_apply: exclusive prefix sum over a generated sequence f(i), then a
//    per-element callback out(i, exclusive, value) -- reduce-then-scan in
//    three launches, no inter-block waiting;
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

// Exclusive scan across the block (blockDim.x == kScanThreads).  Returns the
// thread's exclusive prefix; *total gets the block sum.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T *total) {
  constexpr int kNW = kScanThreads / 32;
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

template <typename T, typename F>
__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(F f, int64_t n, T *block_sums) {
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

template <typename T, typename F, typename Out>
__global__ void __launch_bounds__(kScanThreads) k_scan_down(F f, int64_t n, const T *block_offs,
                                                            Out out) {
  __shared__ T tile[kScanTile];
  const int64_t base = (int64_t)blockIdx.x * kScanTile;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    int e = i * kScanThreads + threadIdx.x;
    int64_t idx = base + e;
    tile[e] = idx < n ? f(idx) : T(0);
  }
  __syncthreads();
  T v[kScanItems];
  T s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = tile[threadIdx.x * kScanItems + i];
    s += v[i];
  }
  __shared__ T tot;
  T ex = block_exclusive_scan<T>(s, &tot) + block_offs[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    int64_t idx = base + threadIdx.x * kScanItems + i;
    if (idx < n) out(idx, ex, v[i]);
    ex += v[i];
  }
}

template <typename T>
inline size_t scan_temp_bytes(int64_t n) {
  int64_t nb = ceil_div(n > 0 ? n : 1, kScanTile);
  return align_up((size_t)(nb + 2) * sizeof(T), kAlign);
}

// Exclusive scan of f(0..n-1); calls out(i, exclusive_i, f(i)) for every i and
// writes the total to *d_total (device pointer, may be null).  temp needs
// scan_temp_bytes<T>(n).  Three launches on `stream`.
template <typename T, typename F, typename Out>
cudaError_t scan_apply(F f, int64_t n, Out out, T *d_total, void *temp, cudaStream_t stream) {
  int64_t nb = ceil_div(n > 0 ? n : 1, kScanTile);
  T *sums = reinterpret_cast<T *>(temp);
  if (n <= 0) {
    if (d_total) return cudaMemsetAsync(d_total, 0, sizeof(T), stream);
    return cudaSuccess;
  }
  k_scan_reduce<T, F><<<(unsigned)nb, kScanThreads, 0, stream>>>(f, n, sums);
  k_scan_spine<T><<<1, kScanThreads, 0, stream>>>(sums, nb, d_total);
  k_scan_down<T, F, Out><<<(unsigned)nb, kScanThreads, 0, stream>>>(f, n, sums, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------- radix sort

constexpr int kRadixThreads = 256;
constexpr int kRadixItems = 16;  // per lane, striped within the warp
constexpr int kRadixWarps = kRadixThreads / 32;
constexpr int kRadixTile = kRadixThreads * kRadixItems;  // 4096
constexpr int kRadixBins = 256;

template <typename K>
__global__ void __launch_bounds__(kRadixThreads) k_radix_hist(const K *keys, int64_t n, int shift,
                                                              uint32_t *hist, int64_t nb) {
  __shared__ uint32_t h[kRadixBins];
  for (int i = threadIdx.x; i < kRadixBins; i += kRadixThreads) h[i] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kRadixTile;
#pragma unroll 4
  for (int i = 0; i < kRadixItems; ++i) {
    int64_t idx = base + (int64_t)i * kRadixThreads + threadIdx.x;
    if (idx < n) atomicAdd(&h[(uint32_t)(keys[idx] >> shift) & 0xFF], 1u);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kRadixBins; d += kRadixThreads) hist[(int64_t)d * nb + blockIdx.x] = h[d];
}

// Stable scatter of one tile.  Warp w owns tile elements [w*512, w*512+512),
// striped: item i of lane l is element w*512 + i*32 + l, so visiting items in
// order and lanes in order visits elements in index order.
template <typename K, bool kHasVal>
__global__ void __launch_bounds__(kRadixThreads) k_radix_scatter(const K *kin, const uint32_t *vin,
                                                                 K *kout, uint32_t *vout, int64_t n,
                                                                 int shift, const uint32_t *offs,
                                                                 int64_t nb) {
  __shared__ uint32_t cnt[kRadixWarps][kRadixBins];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kRadixWarps * kRadixBins; i += kRadixThreads) (&cnt[0][0])[i] = 0;
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
    key[i] = ok ? kin[idx] : K(0);
    if (kHasVal) val[i] = ok ? vin[idx] : 0u;
    digit[i] = ok ? (int)((uint32_t)(key[i] >> shift) & 0xFF) : kRadixBins;  // sentinel bin
  }
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    unsigned peers = __match_any_sync(0xffffffffu, digit[i]);
    uint32_t before = (uint32_t)__popc(peers & lt_mask);
    uint32_t c = digit[i] < kRadixBins ? cnt[warp][digit[i]] : 0u;
    rank[i] = c + before;
    __syncwarp();
    bool last = (peers >> lane) == 1u;  // highest lane of its group
    if (last && digit[i] < kRadixBins) cnt[warp][digit[i]] = c + (uint32_t)__popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // exclusive scan across warps, per digit
  for (int d = threadIdx.x; d < kRadixBins; d += kRadixThreads) {
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kRadixWarps; ++w) {
      uint32_t c = cnt[w][d];
      cnt[w][d] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kRadixItems; ++i) {
    if (digit[i] < kRadixBins) {
      uint32_t pos = offs[(int64_t)digit[i] * nb + blockIdx.x] + cnt[warp][digit[i]] + rank[i];
      kout[pos] = key[i];
      if (kHasVal) vout[pos] = val[i];
    }
  }
}

struct HistRead {
  const uint32_t *h;
  __device__ uint32_t operator()(int64_t i) const { return h[i]; }
};
struct WriteExcl32 {
  uint32_t *o;
  __device__ void operator()(int64_t i, uint32_t ex, uint32_t) const { o[i] = ex; }
};

inline size_t radix_temp_bytes(int64_t n) {
  int64_t nb = ceil_div(n > 0 ? n : 1, kRadixTile);
  size_t h = align_up((size_t)nb * kRadixBins * sizeof(uint32_t), kAlign);
  return 2 * h + scan_temp_bytes<uint32_t>(nb * kRadixBins);
}

// Stable sort by the low `bits` bits of the keys (bits <= 8*sizeof(K)).
// Ping-pongs between (k0, v0) and (k1, v1); *in_second is set when the
// result ends in (k1, v1).  v0/v1 may be null (keys only).
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
  const bool has_val = v0 != nullptr;
  for (int shift = 0; shift < bits; shift += 8) {
    k_radix_hist<K><<<(unsigned)nb, kRadixThreads, 0, stream>>>(ka, n, shift, hist, nb);
    cudaError_t e = scan_apply<uint32_t>(HistRead{hist}, nb * kRadixBins, WriteExcl32{offs},
                                         (uint32_t *)nullptr, stemp, stream);
    if (e != cudaSuccess) return e;
    if (has_val)
      k_radix_scatter<K, true><<<(unsigned)nb, kRadixThreads, 0, stream>>>(ka, va, kb, vb, n, shift,
                                                                          offs, nb);
    else
      k_radix_scatter<K, false><<<(unsigned)nb, kRadixThreads, 0, stream>>>(ka, nullptr, kb, nullptr,
                                                                           n, shift, offs, nb);
    K *tk = ka;
    ka = kb;
    kb = tk;
    uint32_t *tv = va;
    va = vb;
    vb = tv;
    *in_second = !*in_second;
  }
  return cudaGetLastError();
}

}  // namespace snack
