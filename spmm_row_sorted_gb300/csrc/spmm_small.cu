// Small-batch SpMM (batch <= 8): one launch per call, no transposed copy of
// the activations and no fix-up pass.
//
//  * Each CTA owns a run of whole rows, so no row is split between CTAs and
//    every output is written once, by one CTA, with no atomics.
//  * Inside the CTA the (row ends, stored weights) merge path is cut into 8
//    equal-cost warp ranges, as in the tile kernel; rows split between warps
//    are combined in shared memory in warp order.
//  * A lane takes one stored weight at a time and all kB batch elements of
//    it (kB = the batch rounded up to 1, 2, 4 or 8).  When a CTA's stored
//    weights reach half the gathered operand's features and the copy fits
//    96 KB, the operand (X for the forward, dY for the column view) is first
//    copied into shared memory, feature-major, so a weight's batch vector is
//    one short vector load from a bank instead of kB random lines of L1;
//    otherwise the gathers read the operand through L1.
//  * Row sums reduce across the warp with a transposed shuffle tree (each
//    step halves the values a lane carries), leaving batch element b in lanes
//    b * 32/kB .. b * 32/kB + 32/kB - 1.
//  * Column-view mode with kFuseDw also gives dW at each entry's storage
//    index (the lane holds the whole dY batch vector of its entry, so the dot
//    product with the current input feature's X vector needs no shuffles) and
//    the bias gradient db (a slice of the output features per CTA).
#include "spmm.cuh"

namespace snack {

namespace {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallRowCost = 32;  // merge-path cost of a row end, in stored weights

template <int kB>
struct SmallUnroll {  // stored weights per lane in flight
  static constexpr int value = kB >= 8 ? 4 : (kB >= 2 ? 8 : 16);
};

// kB elements of a staged feature-major row, widened to fp32
template <typename T, int kB>
__device__ __forceinline__ void load_staged(const T *p, float (&o)[kB]);

template <>
__device__ __forceinline__ void load_staged<float, 1>(const float *p, float (&o)[1]) {
  o[0] = *p;
}
template <>
__device__ __forceinline__ void load_staged<float, 2>(const float *p, float (&o)[2]) {
  const float2 v = *reinterpret_cast<const float2 *>(p);
  o[0] = v.x;
  o[1] = v.y;
}
template <>
__device__ __forceinline__ void load_staged<float, 4>(const float *p, float (&o)[4]) {
  const float4 v = *reinterpret_cast<const float4 *>(p);
  o[0] = v.x;
  o[1] = v.y;
  o[2] = v.z;
  o[3] = v.w;
}
template <>
__device__ __forceinline__ void load_staged<float, 8>(const float *p, float (&o)[8]) {
  const float4 v = reinterpret_cast<const float4 *>(p)[0], w = reinterpret_cast<const float4 *>(p)[1];
  o[0] = v.x;
  o[1] = v.y;
  o[2] = v.z;
  o[3] = v.w;
  o[4] = w.x;
  o[5] = w.y;
  o[6] = w.z;
  o[7] = w.w;
}
template <>
__device__ __forceinline__ void load_staged<bf16, 1>(const bf16 *p, float (&o)[1]) {
  o[0] = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(p) << 16);
}
template <>
__device__ __forceinline__ void load_staged<bf16, 2>(const bf16 *p, float (&o)[2]) {
  const uint32_t v = *reinterpret_cast<const uint32_t *>(p);
  o[0] = bf16_lo(v);
  o[1] = bf16_hi(v);
}
template <>
__device__ __forceinline__ void load_staged<bf16, 4>(const bf16 *p, float (&o)[4]) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  o[0] = bf16_lo(v.x);
  o[1] = bf16_hi(v.x);
  o[2] = bf16_lo(v.y);
  o[3] = bf16_hi(v.y);
}
template <>
__device__ __forceinline__ void load_staged<bf16, 8>(const bf16 *p, float (&o)[8]) {
  const uint4 v = *reinterpret_cast<const uint4 *>(p);
  o[0] = bf16_lo(v.x);
  o[1] = bf16_hi(v.x);
  o[2] = bf16_lo(v.y);
  o[3] = bf16_hi(v.y);
  o[4] = bf16_lo(v.z);
  o[5] = bf16_hi(v.z);
  o[6] = bf16_lo(v.w);
  o[7] = bf16_hi(v.w);
}

// Sum over the 32 lanes of a[0..kB), transposed: the first log2(kB) xor steps
// each hand half of the remaining values to the partner lane, the rest are
// plain.  Returns, in every lane, the total of batch element lane >> (5 - log2 kB).
template <int kB>
__device__ __forceinline__ float warp_sum_t(const float (&a)[kB], int lane) {
  float g;
  if constexpr (kB == 8) {
    const bool u4 = (lane & 16) != 0, u3 = (lane & 8) != 0, u2 = (lane & 4) != 0;
    float e[4], f[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) e[j] = (u4 ? a[4 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, u4 ? a[j] : a[4 + j], 16);
#pragma unroll
    for (int j = 0; j < 2; ++j) f[j] = (u3 ? e[2 + j] : e[j]) + __shfl_xor_sync(0xffffffffu, u3 ? e[j] : e[2 + j], 8);
    g = (u2 ? f[1] : f[0]) + __shfl_xor_sync(0xffffffffu, u2 ? f[0] : f[1], 4);
    g += __shfl_xor_sync(0xffffffffu, g, 2);
    g += __shfl_xor_sync(0xffffffffu, g, 1);
  } else if constexpr (kB == 4) {
    const bool u4 = (lane & 16) != 0, u3 = (lane & 8) != 0;
    float e[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) e[j] = (u4 ? a[2 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, u4 ? a[j] : a[2 + j], 16);
    g = (u3 ? e[1] : e[0]) + __shfl_xor_sync(0xffffffffu, u3 ? e[0] : e[1], 8);
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
  } else if constexpr (kB == 2) {
    const bool u4 = (lane & 16) != 0;
    g = (u4 ? a[1] : a[0]) + __shfl_xor_sync(0xffffffffu, u4 ? a[0] : a[1], 16);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
  } else {
    g = a[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
  }
  return g;
}

template <int kB>
struct Log2 {
  static constexpr int value = kB <= 1 ? 0 : (kB == 2 ? 1 : (kB == 4 ? 2 : 3));
};

// Shared memory of one CTA: [staged operand][ys (R+1) x kB][wcar 8 x kB][bias R][rps R+2][wsp 18]
__host__ __device__ inline size_t small_stage_bytes(int n_src, int kB, size_t elem, bool stage) {
  return stage ? align_up((size_t)n_src * kB * elem, 16) : 0;
}
inline size_t small_smem_bytes(int n_src, int kB, size_t elem, int R, bool stage) {
  return small_stage_bytes(n_src, kB, elem, stage) + (size_t)(R + 1) * kB * 4 + (size_t)kSmallWarps * kB * 4 +
         (size_t)R * 4 + (size_t)(R + 2) * 4 + (size_t)2 * (kSmallWarps + 1) * 4;
}

// kB elements into a staged feature-major row (vector stores)
__device__ __forceinline__ uint32_t pack_bf16(bf16 lo, bf16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}
template <typename T, int kB>
__device__ __forceinline__ void store_staged(T *p, const T (&t)[kB]);
template <>
__device__ __forceinline__ void store_staged<float, 1>(float *p, const float (&t)[1]) {
  *p = t[0];
}
template <>
__device__ __forceinline__ void store_staged<bf16, 1>(bf16 *p, const bf16 (&t)[1]) {
  *p = t[0];
}
template <>
__device__ __forceinline__ void store_staged<float, 2>(float *p, const float (&t)[2]) {
  *reinterpret_cast<float2 *>(p) = make_float2(t[0], t[1]);
}
template <>
__device__ __forceinline__ void store_staged<float, 4>(float *p, const float (&t)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(t[0], t[1], t[2], t[3]);
}
template <>
__device__ __forceinline__ void store_staged<float, 8>(float *p, const float (&t)[8]) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(t[0], t[1], t[2], t[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(t[4], t[5], t[6], t[7]);
}
template <>
__device__ __forceinline__ void store_staged<bf16, 2>(bf16 *p, const bf16 (&t)[2]) {
  *reinterpret_cast<uint32_t *>(p) = pack_bf16(t[0], t[1]);
}
template <>
__device__ __forceinline__ void store_staged<bf16, 4>(bf16 *p, const bf16 (&t)[4]) {
  *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16(t[0], t[1]), pack_bf16(t[2], t[3]));
}
template <>
__device__ __forceinline__ void store_staged<bf16, 8>(bf16 *p, const bf16 (&t)[8]) {
  *reinterpret_cast<uint4 *>(p) =
      make_uint4(pack_bf16(t[0], t[1]), pack_bf16(t[2], t[3]), pack_bf16(t[4], t[5]), pack_bf16(t[6], t[7]));
}

// kStage: copy the operand into shared memory first -- chosen when
// a CTA's stored weights outnumber the operand's features enough to repay the
// copy; otherwise each weight's kB values are read through L1.
template <typename TA, typename TV, int kB, bool kStage, bool kGatherVal, bool kFuseDw>
__global__ void __launch_bounds__(kSmallThreads) k_spmm_small(SpmmParams P, int R) {
  pdl_wait();
  constexpr int kU = SmallUnroll<kB>::value;
  constexpr int kLg = Log2<kB>::value;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ns = P.n_src, batch = P.batch;
  const int r0 = blockIdx.x * R;
  const int r1 = min(r0 + R, P.n_rows);
  const int nr = r1 - r0;
  const size_t stage = small_stage_bytes(ns, kB, sizeof(TA), kStage);
  TA *xs = reinterpret_cast<TA *>(smem_raw);
  float *ys = reinterpret_cast<float *>(smem_raw + stage);
  float *wcar = ys + (size_t)(R + 1) * kB;
  float *sbias = wcar + kSmallWarps * kB;
  int *rps = reinterpret_cast<int *>(sbias + R);
  int *wsp = rps + R + 2;
  const TA *xg = reinterpret_cast<const TA *>(P.xt);  // [batch][n_src]
  const bool want_out = P.y != nullptr;                // the weight-gradient-only call leaves dX alone

  for (int q = tid; q <= nr; q += kSmallThreads) rps[q] = P.ptr[r0 + q];
  if (P.bias)
    for (int q = tid; q < nr; q += kSmallThreads) sbias[q] = P.bias[r0 + q];
  for (int q = tid; q < kB; q += kSmallThreads) ys[(size_t)nr * kB + q] = 0.f;
  // bias gradient: this CTA's slice of the gathered operand's features
  if (kFuseDw && P.db) {
    const int per = (ns + gridDim.x - 1) / gridDim.x;
    const int q0 = blockIdx.x * per, q1 = min(q0 + per, ns);
    for (int q = q0 + tid; q < q1; q += kSmallThreads) {
      float t[kB], sacc = 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) t[b] = b < batch ? to_f32(ld_keep(xg + (size_t)b * ns + q)) : 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) sacc += t[b];
      P.db[q] = sacc;
    }
  }
  if constexpr (kStage) {  // the operand feature-major, zero past the batch; 16 loads in flight
    constexpr int kH = 16 / kB;
    for (int c0 = tid; c0 < ns; c0 += kH * kSmallThreads) {
      TA t[kH][kB];
#pragma unroll
      for (int h = 0; h < kH; ++h)
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const int c = c0 + h * kSmallThreads;
          t[h][b] = (b < batch && c < ns) ? ld_keep(xg + (size_t)b * ns + c) : from_f32<TA>(0.f);
        }
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        const int c = c0 + h * kSmallThreads;
        if (c < ns) store_staged<TA, kB>(xs + (size_t)c * kB, t[h]);
      }
    }
  }
  __syncthreads();

  // warp ranges: equal-cost slices of the CTA's rows [r0, r1)
  const int w = kSmallRowCost;
  const int j0 = rps[0], j1 = rps[nr];
  if (tid <= kSmallWarps) {
    const int64_t c0 = (int64_t)w * r0 + j0, c1 = (int64_t)w * r1 + j1;
    const int64_t D = c0 + (c1 - c0) * tid / kSmallWarps;
    int lo = r0, hi = r1;
    while (lo < hi) {
      const int mid = lo + (hi - lo + 1) / 2;
      if ((int64_t)w * mid + rps[mid - r0] <= D)
        lo = mid;
      else
        hi = mid - 1;
    }
    int64_t j = D - (int64_t)w * lo;
    const int64_t lim = lo < r1 ? rps[lo - r0 + 1] : j1;
    if (j > lim) j = lim;
    if (j > j1) j = j1;
    if (j < j0) j = j0;
    if (tid == kSmallWarps) j = j1;
    wsp[2 * tid] = lo;
    wsp[2 * tid + 1] = (int)j;
  }
  __syncthreads();

  const int wi0 = wsp[2 * warp], wj0 = wsp[2 * warp + 1];
  const int wi1 = wsp[2 * warp + 2], wj1 = wsp[2 * warp + 3];
  const TV *val = reinterpret_cast<const TV *>(P.val);
  const uint32_t src_max = (uint32_t)(ns - 1);
  const uint32_t nnz_max = (uint32_t)(P.nnz > 0 ? P.nnz - 1 : 0);
  for (int i = wi0; i <= wi1; ++i) {
    const int ps = max(rps[i - r0], wj0);
    const int pe = min(i < wi1 ? rps[i - r0 + 1] : wj1, j1);
    float acc[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) acc[b] = 0.f;
    float xc[kB];  // kFuseDw: this input feature's X batch vector
    if (kFuseDw) {
      const TA *xr = reinterpret_cast<const TA *>(P.xt_dw);  // [batch][n_rows]
#pragma unroll
      for (int b = 0; b < kB; ++b) xc[b] = (b < batch && ps < pe) ? to_f32(xr[(size_t)b * P.n_rows + i]) : 0.f;
    }
    for (int base = ps; base < pe; base += 32 * kU) {
      uint32_t c[kU], sidx[kU];
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int k = base + u * 32 + lane;
        const bool ok = k < pe;
        uint32_t cc = 0u;
        if (ok) cc = P.idx16 ? (uint32_t)ld_stream(P.idx16 + k) : (uint32_t)ld_stream(P.idx + k);
        c[u] = cc < src_max ? cc : src_max;
        sidx[u] = 0u;
        v[u] = 0.f;
        if (kGatherVal) {
          if (ok) {
            const uint32_t sx = (uint32_t)ld_stream(P.val_src + k);
            sidx[u] = sx < nnz_max ? sx : nnz_max;
          }
          if (ok && want_out) v[u] = to_f32(ld_keep(val + sidx[u]));
        } else if (ok) {
          v[u] = to_f32(ld_stream(val + k));
        }
      }
      float x[kU][kB];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if constexpr (kStage) {
          load_staged<TA, kB>(xs + (size_t)c[u] * kB, x[u]);
        } else {
#pragma unroll
          for (int b = 0; b < kB; ++b) x[u][b] = b < batch ? to_f32(ld_keep(xg + (size_t)b * ns + c[u])) : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int b = 0; b < kB; ++b) acc[b] = fmaf(v[u], x[u][b], acc[b]);
      if (kFuseDw) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          float d = 0.f;
#pragma unroll
          for (int b = 0; b < kB; ++b) d = fmaf(x[u][b], xc[b], d);
          if (base + u * 32 + lane < pe) P.dw[sidx[u]] = d;
        }
      }
    }
    const float tot = warp_sum_t<kB>(acc, lane);
    if ((lane & ((32 >> kLg) - 1)) == 0) {
      const int b = lane >> (5 - kLg);
      float *dst = i < wi1 ? ys + (size_t)(i - r0) * kB : wcar + warp * kB;
      dst[b] = tot;
    }
  }
  __syncthreads();
  if (!want_out) return;

  // rows split between warps: add the carries in warp order
  for (int b = tid; b < kB; b += kSmallThreads) {
#pragma unroll 1
    for (int k = 0; k < kSmallWarps; ++k) ys[(size_t)(wsp[2 * k + 2] - r0) * kB + b] += wcar[k * kB + b];
  }
  __syncthreads();

  TA *y = reinterpret_cast<TA *>(P.y);
  for (int q = tid; q < nr * batch; q += kSmallThreads) {
    const int b = q / nr, r = q - b * nr;
    const size_t off = (size_t)b * P.n_rows + r0 + r;
    float sv = ys[(size_t)r * kB + b];
    if (P.bias) sv = sbias[r] + sv;
    y[off] = spmm_epilogue<TA>(P, sv, off);
  }
}

// Rows per CTA: one wave of resident CTAs (at least one row each, at most 64).
template <typename K>
int small_rows_per_cta(K kern, size_t smem, int n_rows, int num_sms) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSmallThreads, smem) != cudaSuccess || occ < 1)
    occ = 1;
  const int64_t slots = (int64_t)occ * num_sms;
  int64_t R = (n_rows + slots - 1) / slots;
  if (R < 1) R = 1;
  if (R > 64) R = 64;
  return (int)R;
}

// Host-side state a launch would otherwise query every call: the rows per
// CTA last derived for a (device, shared memory, rows) triple.  Per host
// thread.  Shared-memory limits live in the process-wide table of
// raise_smem_limit, which only ever raises them.
struct SmallLaunchCache {
  int dev = -1, n_rows = -1, num_sms = -1, R = 0;
  size_t smem = 0;
};

template <typename TA, typename TV, int kB, bool kStage, bool kGV, bool kFuse>
cudaError_t launch_small_s(const SpmmParams &p, int num_sms, cudaStream_t s) {
  auto kern = k_spmm_small<TA, TV, kB, kStage, kGV, kFuse>;
  thread_local SmallLaunchCache cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (cache.dev != dev) {
    cache = SmallLaunchCache{};
    cache.dev = dev;
  }
  const size_t smem_max = small_smem_bytes(p.n_src, kB, sizeof(TA), 64, kStage);
  auto fused = k_spmm_small<TA, TV, kB, kStage, true, true>;  // sizes the column-view calls' CTAs
  e = raise_smem_limit(kern, smem_max);
  if (e == cudaSuccess && kGV)  // the occupancy query below must see a limit that fits smem_max
    e = raise_smem_limit(fused, smem_max);
  if (e != cudaSuccess) return e;
  // the column-view calls size their CTAs by the fused kernel, so dX comes
  // out of the same row partition (and summation order) with or without dW
  if (cache.smem != smem_max || cache.n_rows != p.n_rows || cache.num_sms != num_sms) {
    cache.R = kGV ? small_rows_per_cta(fused, smem_max, p.n_rows, num_sms)
                  : small_rows_per_cta(kern, smem_max, p.n_rows, num_sms);
    cache.smem = smem_max;
    cache.n_rows = p.n_rows;
    cache.num_sms = num_sms;
  }
  const int R = cache.R;
  const size_t smem = small_smem_bytes(p.n_src, kB, sizeof(TA), R, kStage);
  const unsigned grid = (unsigned)((p.n_rows + R - 1) / R);
  launch_pdl(kern, grid, kSmallThreads, smem, s, p, R);
  return cudaGetLastError();
}

// Stage the operand when a CTA's expected stored weights reach half its
// feature count (the copy is then cheaper than reading kB values per weight
// through L1).
template <typename TA, typename TV, int kB, bool kGV, bool kFuse>
cudaError_t launch_small_b(const SpmmParams &p, int num_sms, cudaStream_t s) {
  const int64_t ctas = p.n_rows < 4 * (int64_t)num_sms ? p.n_rows : 4 * (int64_t)num_sms;
  const double per_cta = (double)p.nnz / (double)(ctas > 0 ? ctas : 1);
  const bool fits = (size_t)p.n_src * kB * sizeof(TA) <= kSmallMaxStage;
  if (fits && per_cta * 2.0 >= (double)p.n_src) return launch_small_s<TA, TV, kB, true, kGV, kFuse>(p, num_sms, s);
  return launch_small_s<TA, TV, kB, false, kGV, kFuse>(p, num_sms, s);
}

template <typename TA, typename TV, bool kGV, bool kFuse>
cudaError_t launch_small(const SpmmParams &p, int num_sms, cudaStream_t s) {
  const int b = p.batch;
  if (b <= 1) return launch_small_b<TA, TV, 1, kGV, kFuse>(p, num_sms, s);
  if (b <= 2) return launch_small_b<TA, TV, 2, kGV, kFuse>(p, num_sms, s);
  if (b <= 4) return launch_small_b<TA, TV, 4, kGV, kFuse>(p, num_sms, s);
  if (b <= kSmallMaxBatch) return launch_small_b<TA, TV, 8, kGV, kFuse>(p, num_sms, s);
  return cudaErrorInvalidValue;
}

// Weight gradient alone at small batch: every stored weight is independent,
// so a flat pass needs no row structure -- dw[k] = sum_b dy[b, row[k]] *
// x[b, col[k]] from the batch-major operands through L1, two weights per
// thread in flight, plus db over a slice of the output features per CTA.
template <typename TA, int kB>
__global__ void __launch_bounds__(kSmallThreads) k_sddmm_small(int64_t nnz, const int32_t *__restrict__ row,
                                                               const int32_t *__restrict__ col, int32_t out_f,
                                                               int32_t in_f, const TA *__restrict__ x,
                                                               const TA *__restrict__ dy, int batch,
                                                               float *__restrict__ dw, float *__restrict__ db) {
  pdl_wait();
  constexpr int kW = 2;
  const int tid = threadIdx.x;
  if (db) {
    const int per = (out_f + gridDim.x - 1) / gridDim.x;
    const int q0 = blockIdx.x * per, q1 = min(q0 + per, out_f);
    for (int q = q0 + tid; q < q1; q += kSmallThreads) {
      float t[kB], sacc = 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) t[b] = b < batch ? to_f32(ld_keep(dy + (size_t)b * out_f + q)) : 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) sacc += t[b];
      db[q] = sacc;
    }
  }
  const uint32_t rmax = (uint32_t)(out_f - 1), cmax = (uint32_t)(in_f - 1);
  const int64_t stride = (int64_t)gridDim.x * kSmallThreads;
  for (int64_t k0 = (int64_t)blockIdx.x * kSmallThreads + tid; k0 < nnz; k0 += kW * stride) {
    uint32_t r[kW], c[kW];
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int64_t k = k0 + w * stride;
      const uint32_t rr = k < nnz ? (uint32_t)ld_stream(row + k) : 0u, cc = k < nnz ? (uint32_t)ld_stream(col + k) : 0u;
      r[w] = rr < rmax ? rr : rmax;
      c[w] = cc < cmax ? cc : cmax;
    }
    float a[kW][kB], xv[kW][kB];
#pragma unroll
    for (int w = 0; w < kW; ++w)
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        a[w][b] = b < batch ? to_f32(ld_keep(dy + (size_t)b * out_f + r[w])) : 0.f;
        xv[w][b] = b < batch ? to_f32(ld_keep(x + (size_t)b * in_f + c[w])) : 0.f;
      }
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int64_t k = k0 + w * stride;
      float d = 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) d = fmaf(a[w][b], xv[w][b], d);
      if (k < nnz) dw[k] = d;
    }
  }
}

template <typename TA, int kB>
cudaError_t launch_sddmm_small_b(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                                 const TA *x, const TA *dy, int batch, float *dw, float *db, int num_sms,
                                 cudaStream_t s) {
  int64_t blocks = (nnz + 2 * kSmallThreads - 1) / (2 * kSmallThreads);
  if (blocks > 8 * (int64_t)num_sms) blocks = 8 * (int64_t)num_sms;
  if (blocks < 1) blocks = 1;
  launch_pdl(k_sddmm_small<TA, kB>, (unsigned)blocks, kSmallThreads, 0, s, nnz, row, col, out_f, in_f, x, dy, batch,
             dw, db);
  return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_sddmm_small(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                               const TA *x, const TA *dy, int batch, float *dw, float *db, int num_sms,
                               cudaStream_t s) {
  switch (small_batch_width(batch)) {
    case 1: return launch_sddmm_small_b<TA, 1>(nnz, row, col, out_f, in_f, x, dy, batch, dw, db, num_sms, s);
    case 2: return launch_sddmm_small_b<TA, 2>(nnz, row, col, out_f, in_f, x, dy, batch, dw, db, num_sms, s);
    case 4: return launch_sddmm_small_b<TA, 4>(nnz, row, col, out_f, in_f, x, dy, batch, dw, db, num_sms, s);
    default: return launch_sddmm_small_b<TA, 8>(nnz, row, col, out_f, in_f, x, dy, batch, dw, db, num_sms, s);
  }
}

}  // namespace

int small_batch_width(int batch) { return batch <= 1 ? 1 : (batch <= 2 ? 2 : (batch <= 4 ? 4 : 8)); }

bool small_path_ok(int batch, int n_src, size_t elem) {
  if (batch < 1 || batch > kSmallMaxBatch) return false;
  const int kB = small_batch_width(batch);
  return kB == 1 || (size_t)n_src * kB * elem <= kSmallMaxStage;
}

bool small_dw_flat_ok(int batch, int64_t nnz) {
  return batch >= 1 && batch <= kSmallMaxBatch && nnz * small_batch_width(batch) <= kSmallDwFlatLoads;
}

template <>
cudaError_t run_sddmm_small<float>(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                                   const float *x, const float *dy, int batch, float *dw, float *db, int num_sms,
                                   cudaStream_t s) {
  return launch_sddmm_small<float>(nnz, row, col, out_f, in_f, x, dy, batch, dw, db, num_sms, s);
}

template <>
cudaError_t run_sddmm_small<bf16>(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                                  const bf16 *x, const bf16 *dy, int batch, float *dw, float *db, int num_sms,
                                  cudaStream_t s) {
  return launch_sddmm_small<bf16>(nnz, row, col, out_f, in_f, x, dy, batch, dw, db, num_sms, s);
}

template <>
cudaError_t run_spmm_small<float>(const SpmmParams &p, bool gather_val, bool fuse_dw, int num_sms, cudaStream_t s) {
  if (!gather_val) return launch_small<float, float, false, false>(p, num_sms, s);
  return fuse_dw ? launch_small<float, float, true, true>(p, num_sms, s)
                 : launch_small<float, float, true, false>(p, num_sms, s);
}

template <>
cudaError_t run_spmm_small<bf16>(const SpmmParams &p, bool gather_val, bool fuse_dw, int num_sms, cudaStream_t s) {
  if (!gather_val) return launch_small<bf16, bf16, false, false>(p, num_sms, s);
  return fuse_dw ? launch_small<bf16, bf16, true, true>(p, num_sms, s)
                 : launch_small<bf16, bf16, true, false>(p, num_sms, s);
}

}  // namespace snack
