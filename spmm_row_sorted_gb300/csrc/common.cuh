// Device helpers shared by the kernels of the sparse layer (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/snack.h"

namespace snack {

constexpr int kWarp = 32;
constexpr size_t kAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

typedef __nv_bfloat16 bf16;

// ------------------------------------------------------- dependent launches
//
// Every kernel of the library is launched with programmatic stream
// serialization: its blocks may be scheduled while the kernel before it on
// the stream is still draining, and its first instruction waits until that
// kernel has completed and its writes are visible (griddepcontrol.wait).
// Nothing a kernel does comes before that wait, so the stream order of
// results is unchanged; what overlaps is the launch and block scheduling,
// about 4 us per dependent launch on GB300 otherwise.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ kernel trace
//
// While the calling host thread has a trace open (snack_trace_start), every
// launch is bracketed by two CUDA events recorded on its stream, kept with
// the kernel's entry point in the next slot of a ring of `cap` slots.  (The
// event between two launches also keeps the second from starting early, so a
// traced kernel's time includes its launch.)
struct KernelTrace {
  const void **fn;
  cudaEvent_t *ev;  // two per slot: before, after
  int cap;
  long long n;  // launches recorded; slot n % cap is next
};
extern thread_local KernelTrace *g_kernel_trace;

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KernelTrace *tr = g_kernel_trace;
  int slot = 0;
  if (tr) {
    slot = (int)(tr->n % tr->cap);
    tr->fn[slot] = reinterpret_cast<const void *>(kernel);
    cudaEventRecord(tr->ev[2 * slot], s);
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
  if (tr) {
    cudaEventRecord(tr->ev[2 * slot + 1], s);
    ++tr->n;
  }
  return e;
}

// ------------------------------------------------ shared-memory limits
//
// A kernel's dynamic shared-memory limit (cudaFuncAttributeMaxDynamicSharedMemorySize)
// is process-wide per device.  Every launcher raises it through this one
// call: a table keyed by (device, kernel), under a lock, records the largest
// limit granted so far and the attribute is only ever raised, so host threads
// launching the same kernel for layers of different sizes, or one launcher
// that also sizes another kernel, never lower a limit another launch needs.
cudaError_t raise_smem_limit(const void *kernel, size_t bytes);
template <typename... KArgs>
inline cudaError_t raise_smem_limit(void (*kernel)(KArgs...), size_t bytes) {
  return raise_smem_limit(reinterpret_cast<const void *>(kernel), bytes);
}

// ---------------------------------------------------------------- loads

// Streamed once: evict-first in L1 and L2.
template <typename T>
__device__ __forceinline__ T ld_stream(const T *p) {
  return __ldcs(p);
}

// Reused from L2 / L1 (activations gathered by column).
template <typename T>
__device__ __forceinline__ T ld_keep(const T *p) {
  return __ldg(p);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float v) {
  return __float2bfloat16_rn(v);
}

// A lane's slice of a gathered activation row: V consecutive elements,
// widened to fp32.  V = 4 (fp32, 16 B), V = 8 (bf16, 16 B) or V = 1.
template <typename T, int V>
struct Slice;

template <>
struct Slice<float, 4> {
  __device__ __forceinline__ static void load(const float *p, float (&o)[4]) {
    float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
  }
};

template <>
struct Slice<bf16, 8> {
  __device__ __forceinline__ static void load(const bf16 *p, float (&o)[8]) {
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
    o[0] = bf16_lo(v.x);
    o[1] = bf16_hi(v.x);
    o[2] = bf16_lo(v.y);
    o[3] = bf16_hi(v.y);
    o[4] = bf16_lo(v.z);
    o[5] = bf16_hi(v.z);
    o[6] = bf16_lo(v.w);
    o[7] = bf16_hi(v.w);
  }
};

template <>
struct Slice<float, 1> {
  __device__ __forceinline__ static void load(const float *p, float (&o)[1]) { o[0] = __ldg(p); }
};

template <>
struct Slice<bf16, 1> {
  __device__ __forceinline__ static void load(const bf16 *p, float (&o)[1]) {
    o[0] = __bfloat162float(__ldg(p));
  }
};

template <typename T>
struct ActTraits;
template <>
struct ActTraits<float> {
  static constexpr int kVec = 4;  // elements per 16-byte slice
};
template <>
struct ActTraits<bf16> {
  static constexpr int kVec = 8;
};

__host__ __device__ inline size_t dtype_size(snack_dtype t) { return t == SNACK_BF16 ? 2 : 4; }

}  // namespace snack
