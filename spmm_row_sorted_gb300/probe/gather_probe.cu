// Gather-throughput probes for the SpMM tile kernels (measurement only; not
// part of libsnack).  Each probe streams the stored weights of a layer once
// and, per weight, brings the 128-byte batch vector Xt[col] (32 fp32 batch
// elements of the feature-major activations) to the SM and multiplies it by
// the weight -- the inner loop of the forward SpMM with the row structure
// removed -- by one of three routes:
//
//   kind 0  LDG.128 gathers through L1: 8 lanes per weight, 4 weights per warp
//           instruction, 8 weights per lane in flight;
//   kind 1  TMA tile::gather4 (four 128-byte rows per instruction) into a ring
//           of shared-memory stages completed on mbarriers, read back with
//           LDS.128 by consumer warps;
//   kind 2  one 1-D bulk copy (cp.async.bulk, 128 bytes) per weight into the
//           same ring.
//
// and three reference streams for the other costs of the backward pass:
//
//   kind 3  random 4-byte loads val[perm[k]] (the column view's value gather);
//   kind 4  random 4-byte stores dst[perm[k]] (a weight gradient written at
//           storage index from column order);
//   kind 5  a sequential read of the index and value streams.
//
// Every spin on an mbarrier is bounded; when a bound runs out the probe sets
// an error word and the CTA still waits (bounded) for its own copies before
// it returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kSpinLimit = 1 << 22;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// true when the phase of the given parity has completed, false when the bound ran out
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  for (int i = 0; i < kSpinLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int x, int r0, int r1, int r2, int r3,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

constexpr int kB = 32;  // batch elements per gathered row (fp32: 128 bytes)

// kind 0
__global__ void __launch_bounds__(256) k_probe_ldg(const float *__restrict__ xt, const int32_t *__restrict__ col,
                                                   const float *__restrict__ val, int64_t nnz, int n_src,
                                                   float *__restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int slot = lane >> 3, g = lane & 7;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w * 32 < nnz; w += warps) {
    const int64_t k = w * 32 + lane;
    int c = k < nnz ? col[k] : 0;
    c = c < 0 ? 0 : (c >= n_src ? n_src - 1 : c);
    const float v = k < nnz ? val[k] : 0.f;
    float4 x[8];
    float vv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = u * 4 + slot;
      const int cc = __shfl_sync(0xffffffffu, c, e);
      vv[u] = __shfl_sync(0xffffffffu, v, e);
      x[u] = __ldg(reinterpret_cast<const float4 *>(xt + (size_t)cc * kB) + g);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc[0] = fmaf(vv[u], x[u].x, acc[0]);
      acc[1] = fmaf(vv[u], x[u].y, acc[1]);
      acc[2] = fmaf(vv[u], x[u].z, acc[2]);
      acc[3] = fmaf(vv[u], x[u].w, acc[3]);
    }
  }
  out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = acc[0] + acc[1] + acc[2] + acc[3];
}

// kinds 1 and 2: one producer warp, kCons consumer warps, kStages stages of 32 rows
constexpr int kCons = 4;
constexpr int kStages = 8;
constexpr int kStageBytes = 32 * kB * 4;
constexpr int kRingThreads = 32 * (1 + kCons);

template <bool kTensor>
__global__ void __launch_bounds__(kRingThreads) k_probe_ring(const __grid_constant__ CUtensorMap map,
                                                             const float *__restrict__ xt,
                                                             const int32_t *__restrict__ col,
                                                             const float *__restrict__ val, int64_t nnz, int n_src,
                                                             float *__restrict__ out, uint32_t *__restrict__ err) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
  uint64_t *empty = full + kStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCons);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t n_chunks = (nnz + 31) / 32;
  int64_t issued = 0;
  bool ok = true;
  if (warp == 0) {
    for (int64_t ch = blockIdx.x; ch < n_chunks && ok; ch += gridDim.x, ++issued) {
      const int s = (int)(issued % kStages);
      const uint32_t par = (uint32_t)((issued / kStages) & 1);
      if (!mbar_wait(&empty[s], par ^ 1u)) {
        ok = false;
        break;
      }
      const int64_t k = ch * 32 + lane;
      int c = k < nnz ? col[k] : 0;
      c = c < 0 ? 0 : (c >= n_src ? n_src - 1 : c);
      unsigned char *dst = smem + s * kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], kStageBytes);
      __syncwarp();
      if (kTensor) {
        const int q = (lane & 7) * 4;
        const int r0 = __shfl_sync(0xffffffffu, c, q), r1 = __shfl_sync(0xffffffffu, c, q + 1);
        const int r2 = __shfl_sync(0xffffffffu, c, q + 2), r3 = __shfl_sync(0xffffffffu, c, q + 3);
        if (lane < 8) tma_gather4(dst + lane * 4 * kB * 4, &map, 0, r0, r1, r2, r3, &full[s]);
      } else {
        bulk_copy(dst + lane * kB * 4, xt + (size_t)c * kB, kB * 4, &full[s]);
      }
    }
  } else {
    const int cw = warp - 1;
    const int slot = lane >> 3, g = lane & 7;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t ch = blockIdx.x; ch < n_chunks; ch += gridDim.x, ++issued) {
      const int s = (int)(issued % kStages);
      const uint32_t par = (uint32_t)((issued / kStages) & 1);
      if (!mbar_wait(&full[s], par)) {
        ok = false;
        break;
      }
      const unsigned char *src = smem + s * kStageBytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = cw * 8 + u * 4 + slot;
        const int64_t k = ch * 32 + e;
        const float v = k < nnz ? __ldg(val + k) : 0.f;
        const float4 x = *reinterpret_cast<const float4 *>(src + e * kB * 4 + g * 16);
        acc[0] = fmaf(v, x.x, acc[0]);
        acc[1] = fmaf(v, x.y, acc[1]);
        acc[2] = fmaf(v, x.z, acc[2]);
        acc[3] = fmaf(v, x.w, acc[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    out[(size_t)blockIdx.x * kRingThreads + threadIdx.x] = acc[0] + acc[1] + acc[2] + acc[3];
  }
  if (!ok && lane == 0) atomicOr(err, 1u);
  __syncthreads();
  // every copy this CTA issued has completed before it exits (bounded)
  if (threadIdx.x == 0) {
    const int64_t last = issued;  // the producer's count of issued chunks
    for (int64_t i = last > kStages ? last - kStages : 0; i < last; ++i)
      if (!mbar_wait(&full[i % kStages], (uint32_t)((i / kStages) & 1))) atomicOr(err, 2u);
  }
}

// kind 3: random 4-byte loads
__global__ void __launch_bounds__(256) k_probe_rand_load(const float *__restrict__ val, const int32_t *__restrict__ perm,
                                                         int64_t nnz, float *__restrict__ out) {
  float acc = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += 4 * stride) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = k + u * stride;
      int p = q < nnz ? perm[q] : 0;
      p = p < 0 ? 0 : (p >= nnz ? (int)(nnz - 1) : p);
      v[u] = q < nnz ? __ldg(val + p) : 0.f;
    }
    acc += v[0] + v[1] + v[2] + v[3];
  }
  out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// kind 4: random 4-byte stores
__global__ void __launch_bounds__(256) k_probe_rand_store(const float *__restrict__ val,
                                                          const int32_t *__restrict__ perm, int64_t nnz,
                                                          float *__restrict__ dst) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += stride) {
    int p = perm[k];
    p = p < 0 ? 0 : (p >= nnz ? (int)(nnz - 1) : p);
    dst[p] = val[k];
  }
}

// kind 5: sequential read of col and val
__global__ void __launch_bounds__(256) k_probe_stream(const int32_t *__restrict__ col, const float *__restrict__ val,
                                                      int64_t nnz, float *__restrict__ out) {
  float acc = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += stride)
    acc += (float)__ldcs(col + k) + __ldcs(val + k);
  out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

// Launch one probe.  out needs probe_out_elems(kind) floats; dst (kind 4)
// nnz floats; err one word (zeroed by the caller).  Returns 0, or a negative
// code: -1 bad arguments, -2 tensor map, -3 launch.
extern "C" int probe_gather(int kind, const float *xt, int n_src, const int32_t *col, const float *val,
                            const int32_t *perm, int64_t nnz, float *out, float *dst, uint32_t *err, int grid,
                            cudaStream_t s) {
  if (nnz <= 0 || n_src <= 0 || grid <= 0) return -1;
  switch (kind) {
    case 0:
      k_probe_ldg<<<grid, 256, 0, s>>>(xt, col, val, nnz, n_src, out);
      break;
    case 1:
    case 2: {
      CUtensorMap map = {};
      if (kind == 1) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
          return -2;
        const cuuint64_t dims[2] = {(cuuint64_t)kB, (cuuint64_t)n_src};
        const cuuint64_t strides[1] = {(cuuint64_t)kB * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kB, 1u};
        const cuuint32_t estr[2] = {1u, 1u};
        if (reinterpret_cast<EncodeTiled>(fn)(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(xt), dims,
                                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return -2;
      }
      const size_t smem = (size_t)kStages * kStageBytes + 2 * kStages * sizeof(uint64_t);
      auto kern = kind == 1 ? k_probe_ring<true> : k_probe_ring<false>;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -3;
      kern<<<grid, kRingThreads, smem, s>>>(map, xt, col, val, nnz, n_src, out, err);
      break;
    }
    case 3:
      k_probe_rand_load<<<grid, 256, 0, s>>>(val, perm, nnz, out);
      break;
    case 4:
      k_probe_rand_store<<<grid, 256, 0, s>>>(val, perm, nnz, dst);
      break;
    case 5:
      k_probe_stream<<<grid, 256, 0, s>>>(col, val, nnz, out);
      break;
    default:
      return -1;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

// floats of `out` a launch of `grid` CTAs writes
extern "C" int64_t probe_out_elems(int kind, int grid) {
  return (int64_t)grid * (kind == 1 || kind == 2 ? kRingThreads : 256);
}
