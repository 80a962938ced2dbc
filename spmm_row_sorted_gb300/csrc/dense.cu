// Moderately sparse bf16 layers (a quarter or more of W stored, batch >= 32)
// on the tensor cores.  At that density the product is a dense contraction,
// so it runs as tcgen05 matrix multiplies with fp32 accumulators in tensor
// memory (TMEM).  W is never densified in HBM: every CTA builds its W tiles
// in shared memory straight from the row-sorted COO (16-bit columns from the
// plan, the caller's bf16 values), using the plan's per-(64-column block, row)
// offset table to find each row's entries in a block; the activation tiles
// arrive by TMA.
//
//   forward      D[r][b] = sum_c W[r][c] X[b][c]     A = W tile (rows x 64 cols, scattered)
//                                                    B = X tile (batch x 64 cols, TMA)
//                Y[b][r] = bf16(bias[r] + D[r][b])   one rounding, after the bias
//   input grad   D[c][b] = sum_r W[r][c] dY[b][r]    A = W^T tile (cols x 64 rows, scattered)
//                                                    B = dY tile (batch x 64 rows, TMA)
//   weight grad  D[r][c] = sum_b dY[b][r] X[b][c]    A = dY^T, B = X^T (feature-major copies, TMA)
//                dW[k] = D[row_k][col_k]             read back at the stored positions only
//
// Every operand tile is K-major with the 128-byte swizzle: a tile row holds
// 64 bf16 of K (128 bytes), 8 rows form a 1024-byte atom whose 16-byte chunks
// are permuted by chunk ^= row % 8.  The TMA writes that layout itself
// (CU_TENSOR_MAP_SWIZZLE_128B, box inner extent 128 bytes); the scatter
// computes it.  One CTA per output tile (persistent over tiles when there
// are more than SMs); warps 0-3 build the W tiles and run the epilogue
// (TMEM lanes 0-127), warp 4 issues the TMA loads and warp 5 the MMAs.  Wide reductions are split along K into partial sums that a
// second kernel adds in split order (deterministic).
//
// Every wait on an mbarrier is bounded: when a bound runs out the kernel
// records an error word, stops issuing work, waits (bounded) for what it has
// in flight, frees its TMEM and returns.
#include <cuda.h>

#include "internal.hpp"

namespace snack {

namespace {

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t su32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}

constexpr int kSpinLimit = 1 << 20;  // try_wait rounds before a wait is declared stuck (far above any real wait)

// true once the phase of the given parity has completed; false when the bound ran out
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = su32(bar);
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

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// one full warp; the TMEM address lands in *dst
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (TMEM) (+)= A (smem) * B (smem)^T, both K-major, fp32 accumulate
__device__ __forceinline__ void umma_bf16(uint32_t taddr, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(taddr),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on *bar once every MMA issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major tile with the 128-byte
// swizzle: start address (16-byte units), leading byte offset (unused for
// this layout, 1), stride byte offset 1024 (one 8-row atom to the next),
// descriptor version 1, layout type 2 (128-byte swizzle).  The tile base is
// 1024-byte aligned; a K step of 16 elements inside the 128-byte row moves
// the start by 32 bytes and the hardware applies the swizzle to the result.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bit 4), A and B
// bf16 (bits 7 and 10), both K-major, N / 8 at bit 17, M / 16 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// byte offset of element (row i, k j) in a K-major 128-byte-swizzled tile of 64-wide rows
__device__ __forceinline__ uint32_t sw128_off(uint32_t i, uint32_t j) {
  return i * 128u + ((((j >> 3) ^ (i & 7u))) << 4) + ((j & 7u) << 1);
}

// ------------------------------------------------------------------ kernel

constexpr int kM = 128;         // UMMA M: rows of the A tile, TMEM lanes
constexpr int kKb = 64;         // K per stage (one 128-byte swizzle row of bf16), and the plan's column block
constexpr int kStages = 3;      // A/B stages
constexpr int kIdx = 8;         // index slices in flight (mask + offsets of a stage)
constexpr int kIdxBytes = 2048; // one slice: up to 128 x (8 + 4) bytes
constexpr int kProdWarps = 16;  // W tiles and epilogue
constexpr int kProd = kProdWarps * 32;
constexpr int kThreads = kProd + 64;  // + warp 16 (TMA) + warp 17 (MMA)
constexpr int kATileBytes = kM * kKb * 2;
constexpr int kDwN = 256;       // weight-gradient tile width (columns)
constexpr int kLook = 2;        // stages of value loads a producer keeps in flight ahead of the one it writes

enum { kModeFwd = 0, kModeDx = 1, kModeDw = 2 };

// The plan's tables of a moderately sparse layer, both [block][row] with
// 64-column blocks (nkb = ceil(in_f / 64)):
//   mask[kb * out_f + r]  bit c of row r's 64 columns 64 kb .. 64 kb + 63 is set
//                         when that weight is stored;
//   koff[kb * out_f + r]  storage index of row r's first stored weight at a
//                         column >= 64 kb (kb = nkb: the row's end).
// Row r's stored values of block kb are then val[koff .. koff + popc(mask)),
// in column order.
struct TcArgs {
  int32_t out_f, in_f, batch;
  int32_t nkb;
  const uint64_t *mask;
  const int32_t *koff;
  const uint16_t *val;     // [nnz] bf16 bits
  const float *bias;       // forward, or null
  bf16 *out;               // forward Y [batch][out_f], input gradient dX [batch][in_f] (no split)
  float *part;             // split partial sums [n_split][batch][n_out]
  float *dw;               // weight gradient [nnz]
  int32_t n_out;           // forward: out_f; input gradient: in_f
  int32_t nt;              // N of a tile: the batch tile (forward, input gradient) or kDwN
  int32_t m_tiles, n_tiles, n_split;
  int32_t k_chunks;        // 64-wide K chunks in all (forward: nkb; input gradient: ceil(out_f/64); weight gradient: ldx/64)
  uint32_t *err;           // error word: bit 0 a wait ran out
};

// One producer warp's part of a stage's A tile: 8 W rows x one 64-column
// block; lane l owns the block's columns 2l and 2l + 1, so every value load of
// the warp reads within one row's contiguous run of stored values.
//   forward: A row i = W row m0 + i, i in [8w, 8w + 8), K = the block's 64 columns;
//   input gradient: W rows 64 kc + 8 (w >> 1) .. + 7 (K), block h = w & 1 of
//            the CTA's 128 columns (A rows 64 h .. 64 h + 63).
// The index slice of a stage holds mask[] then koff[] of its rows x blocks:
// forward [1 block][128 rows], input gradient [2 blocks][64 rows].
template <int kMode>
__device__ __forceinline__ int slice_row(int w, int r8) {
  return kMode == kModeFwd ? 8 * w + r8 : (w & 1) * 64 + 8 * (w >> 1) + r8;
}

// v[2 r8 + b]: the value of row r8 at column 2 lane + b, or zero
template <int kMode>
__device__ __forceinline__ void seg_load(const uint8_t *slice, int w, int lane, const uint16_t *__restrict__ val,
                                         uint16_t (&v)[16]) {
  const uint64_t *mk = reinterpret_cast<const uint64_t *>(slice);
  const int32_t *ko = reinterpret_cast<const int32_t *>(slice + 1024);
  const uint64_t below = (1ull << (2 * lane)) - 1ull;
#pragma unroll
  for (int r8 = 0; r8 < 8; ++r8) {
    const int idx = slice_row<kMode>(w, r8);
    const uint64_t m = mk[idx];
    const int p = ko[idx] + __popcll(m & below);
    const uint32_t b = (uint32_t)(m >> (2 * lane)) & 3u;
    v[2 * r8] = (b & 1u) ? val[p] : (uint16_t)0;
    v[2 * r8 + 1] = (b & 2u) ? val[p + (int)(b & 1u)] : (uint16_t)0;
  }
}

template <int kMode>
__device__ __forceinline__ void seg_store(uint8_t *a, int w, int lane, const uint16_t (&v)[16]) {
  if (kMode == kModeFwd) {
    // row i: columns 2 lane, 2 lane + 1 are one 4-byte word of chunk lane / 4
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) {
      const uint32_t i = (uint32_t)(8 * w + r8);
      *reinterpret_cast<uint32_t *>(a + i * 128 + ((((uint32_t)lane >> 2) ^ (i & 7u)) << 4) + ((lane & 3) << 2)) =
          v[2 * r8] | ((uint32_t)v[2 * r8 + 1] << 16);
    }
  } else {
    // A rows 64 h + 2 lane + b hold the column; their K chunk w >> 1 gets the 8 rows' values
    const uint32_t kch = (uint32_t)(w >> 1);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t i = (uint32_t)((w & 1) * 64 + 2 * lane + b);
      uint4 c;
      c.x = v[0 + b] | ((uint32_t)v[2 + b] << 16);
      c.y = v[4 + b] | ((uint32_t)v[6 + b] << 16);
      c.z = v[8 + b] | ((uint32_t)v[10 + b] << 16);
      c.w = v[12 + b] | ((uint32_t)v[14 + b] << 16);
      *reinterpret_cast<uint4 *>(a + i * 128 + ((kch ^ (i & 7u)) << 4)) = c;
    }
  }
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1) k_tc(const __grid_constant__ CUtensorMap map_a,
                                                    const __grid_constant__ CUtensorMap map_b,
                                                    const __grid_constant__ CUtensorMap map_mask,
                                                    const __grid_constant__ CUtensorMap map_koff, TcArgs P) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int nt = P.nt;
  const uint32_t b_bytes = (uint32_t)nt * kKb * 2;
  const uint32_t stage_bytes = kATileBytes + b_bytes;
  constexpr bool kW = kMode != kModeDw;  // the CTA builds W tiles
  uint8_t *stage0 = smem;
  uint8_t *idx0 = smem + kStages * stage_bytes;  // kIdx index slices (kW only)
  uint64_t *bars = reinterpret_cast<uint64_t *>(idx0 + (kW ? kIdx * kIdxBytes : 0));
  uint64_t *b_full = bars;                  // TMA bytes of a stage (kStages)
  uint64_t *a_full = bars + kStages;        // the producer warps have written a stage's A tile (kStages)
  uint64_t *empty = bars + 2 * kStages;     // the MMAs of a stage have completed (kStages)
  uint64_t *i_full = bars + 3 * kStages;    // an index slice has landed (kIdx)
  uint64_t *i_free = i_full + kIdx;         // the producers are done with an index slice (kIdx)
  uint64_t *done = i_free + kIdx;           // the MMAs of a tile have completed
  uint64_t *tfree = done + 1;               // the epilogue has read the tile's accumulator
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfree + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  int *mma_tiles = abort_flag + 1;          // tiles whose MMAs the issuer committed to `done`
  int *tma_issued = abort_flag + 2;         // stage loads the TMA warp issued
  int *idx_issued = abort_flag + 3;         // index slices the TMA warp issued
  float *ep = reinterpret_cast<float *>(tmem_slot + 8);  // weight gradient: [16 warps][32][33]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tcols = kMode == kModeDw ? (uint32_t)kDwN : (nt <= 32 ? 32u : nt <= 64 ? 64u : nt <= 128 ? 128u : 256u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&a_full[s], kProdWarps);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kIdx; ++s) {
      mbar_init(&i_full[s], 1);
      mbar_init(&i_free[s], kProdWarps);
    }
    mbar_init(done, 1);
    mbar_init(tfree, kProdWarps);
    *abort_flag = 0;
    *mma_tiles = 0;
    *tma_issued = 0;
    *idx_issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles = P.m_tiles * P.n_tiles * P.n_split;
  const int kpb = (P.k_chunks + P.n_split - 1) / P.n_split;  // K chunks per split
  bool ok = true;
  // stage and slice counters run on across the tiles of a CTA
  uint32_t it = 0;
  int tile_iter = 0;
  for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tile_iter) {
    const int split = tile % P.n_split;
    const int mn = tile / P.n_split;
    const int mt = mn % P.m_tiles, ntile = mn / P.m_tiles;
    const int m0 = mt * kM, n0 = ntile * nt;
    const int kc0 = split * kpb;
    const int kc1 = min(P.k_chunks, kc0 + kpb);
    const int nk = max(0, kc1 - kc0);

    if (warp == kProdWarps) {  // ------------------------------------ TMA
      if (lane == 0) {
        // index slices run up to kIdx stages ahead of the producers; the
        // activation tiles up to kStages ahead of the MMAs
        int qi = 0;
        auto issue_idx = [&](int upto) -> bool {
          for (; qi < upto && qi < nk; ++qi) {
            const uint32_t g = it + qi;
            const int s = (int)(g % kIdx);
            if (!mbar_wait(&i_free[s], ((g / kIdx) & 1) ^ 1)) return false;
            uint8_t *sl = idx0 + s * kIdxBytes;
            mbar_expect_tx(&i_full[s], kMode == kModeFwd ? 128 * 12 : 2 * 64 * 12);
            if (kMode == kModeFwd) {
              tma_load_2d(sl, &map_mask, m0, kc0 + qi, &i_full[s]);
              tma_load_2d(sl + 1024, &map_koff, m0, kc0 + qi, &i_full[s]);
            } else {
              tma_load_2d(sl, &map_mask, (kc0 + qi) * kKb, m0 / kKb, &i_full[s]);
              tma_load_2d(sl + 1024, &map_koff, (kc0 + qi) * kKb, m0 / kKb, &i_full[s]);
            }
            *idx_issued = (int)(g + 1);
          }
          return true;
        };
        if (kW && !issue_idx(kIdx)) ok = false;
        for (int q = 0; q < nk && ok; ++q) {
          const uint32_t g = it + q;
          const int s = (int)(g % kStages);
          if (!mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1)) {
            ok = false;
            break;
          }
          uint8_t *st = stage0 + s * stage_bytes;
          const int kx = (kc0 + q) * kKb;
          if (kMode == kModeDw) {
            mbar_expect_tx(&b_full[s], stage_bytes);
            tma_load_2d(st, &map_a, kx, m0, &b_full[s]);
          } else {
            mbar_expect_tx(&b_full[s], b_bytes);
          }
          tma_load_2d(st + kATileBytes, &map_b, kx, n0, &b_full[s]);
          *tma_issued = (int)(g + 1);
          if (kW && !issue_idx(q + 1 + kIdx)) {
            ok = false;
            break;
          }
        }
      }
    } else if (warp == kProdWarps + 1) {  // ------------------------------ MMA issuer
      if (lane == 0) {
        if (tile_iter > 0 && !mbar_wait(tfree, (tile_iter - 1) & 1)) ok = false;  // the last tile's accumulator was read
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(kM, kMode == kModeDw ? kDwN : nt);
        for (int q = 0; q < nk && ok; ++q) {
          const uint32_t g = it + q;
          const int s = (int)(g % kStages);
          const uint32_t ph = (g / kStages) & 1;
          if (kW && !mbar_wait(&a_full[s], ph)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&b_full[s], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = su32(stage0 + s * stage_bytes);
          const uint32_t sb = sa + kATileBytes;
#pragma unroll
          for (int k = 0; k < kKb / 16; ++k)
            umma_bf16(tmem, sw128_desc(sa + 32 * k), sw128_desc(sb + 32 * k), idesc, (q > 0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[s]);  // frees the stage once these MMAs have read it
        }
        umma_commit(done);  // the tile's accumulator is complete (also on abort)
        *mma_tiles = tile_iter + 1;
      }
    } else if (kW && nk > 0) {  // ----------------------- W tiles (warps 0-15)
      // value loads run kLook stages ahead of the stage being written: three
      // register sets, rotated by unrolling, so a load in flight is never moved
      uint16_t v0[16], v1[16], v2[16];
      auto fetch = [&](int q, uint16_t(&v)[16]) -> bool {
        if (q >= nk) return true;
        const uint32_t g = it + q;
        const int s = (int)(g % kIdx);
        if (!mbar_wait(&i_full[s], (g / kIdx) & 1)) return false;
        seg_load<kMode>(idx0 + s * kIdxBytes, warp, lane, P.val, v);
        __syncwarp();
        if (lane == 0) mbar_arrive(&i_free[s]);  // the warp has read the slice: it may be refilled
        return true;
      };
      auto write = [&](int q, const uint16_t(&v)[16]) -> bool {
        if (q >= nk) return true;
        const uint32_t g = it + q;
        const int s = (int)(g % kStages);
        if (!mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1)) return false;
        seg_store<kMode>(stage0 + s * stage_bytes, warp, lane, v);
        fence_async_shared();  // the tensor core reads the tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
        return true;
      };
      bool good = fetch(0, v0) && fetch(1, v1);
      for (int q = 0; q < nk && good; q += 3) {
        good = fetch(q + 2, v2) && write(q, v0) && fetch(q + 3, v0) && write(q + 1, v1) && fetch(q + 4, v1) &&
               write(q + 2, v2);
      }
      if (!good) ok = false;
    }
    it += nk;

    // ---------------------------------------------------------- epilogue
    if (warp < kProdWarps) {
      const int quarter = warp & 3, grp = warp >> 2;  // TMEM lanes 32 quarter .. +31; column chunks grp, grp+4, ...
      const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
      if (kMode != kModeDw) {
        if (!mbar_wait(done, tile_iter & 1)) ok = false;
        tc_fence_after();
        const int o = m0 + quarter * 32 + lane;  // output feature of this TMEM lane
        const bool o_ok = o < P.n_out;
        const float bo = (kMode == kModeFwd && P.bias && o_ok && P.n_split == 1) ? P.bias[o] : 0.f;
        for (int c0 = grp * 32; c0 < nt; c0 += 4 * 32) {
          float v[32];
          tmem_ld32(lane_base + (uint32_t)c0, v);
          if (o_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int b = n0 + c0 + j;
              if (b < P.batch) {
                if (P.n_split == 1)
                  P.out[(size_t)b * P.n_out + o] = __float2bfloat16_rn(bo + v[j]);
                else
                  P.part[((size_t)split * P.batch + b) * P.n_out + o] = v[j];
              }
            }
          }
        }
      } else {
        // weight gradient: row r's stored weights among the chunk's 32 columns
        // are the set bits of its mask, stored contiguously from dw[base]: each
        // lane compacts its row's values into shared memory, then the warp
        // writes row after row as contiguous runs
        const int r = m0 + quarter * 32 + lane;
        float *eb = ep + warp * 32 * 33;
        uint32_t bits[2];
        int base[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // this warp's chunks: grp and grp + 4 (32 columns each)
          const int c = n0 + (grp + 4 * h) * 32;
          bits[h] = 0u;
          base[h] = 0;
          if (r < P.out_f && c < P.in_f) {
            const int kb = c / kKb;
            const uint64_t m = P.mask[(size_t)kb * P.out_f + r];
            const bool hi = (c & 63) != 0;
            bits[h] = hi ? (uint32_t)(m >> 32) : (uint32_t)m;
            base[h] = P.koff[(size_t)kb * P.out_f + r] + (hi ? __popc((uint32_t)m) : 0);
          }
        }
        if (!mbar_wait(done, tile_iter & 1)) ok = false;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v[32];
          tmem_ld32(lane_base + (uint32_t)((grp + 4 * h) * 32), v);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if ((bits[h] >> j) & 1u) eb[lane * 33 + __popc(bits[h] & ((1u << j) - 1u))] = v[j];
          __syncwarp();
          for (int ii = 0; ii < 32; ++ii) {
            const int n = __popc(__shfl_sync(0xffffffffu, bits[h], ii));
            const int b0 = __shfl_sync(0xffffffffu, base[h], ii);
            if (lane < n) P.dw[b0 + lane] = eb[ii * 33 + lane];
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tfree);
    }
  }
  if (!ok) {
    atomicOr(P.err, 1u);
    *abort_flag = 1;
  }
  __syncthreads();
  // after an abort: every load and MMA issued has completed (bounded) before
  // the TMEM is given back and the CTA exits
  if (threadIdx.x == 0 && *abort_flag) {
    const int issued = *tma_issued;
    for (int g = issued - 1; g >= 0 && g >= issued - kStages; --g) mbar_wait(&b_full[g % kStages], (g / kStages) & 1);
    const int ii = *idx_issued;
    for (int g = ii - 1; g >= 0 && g >= ii - kIdx; --g) mbar_wait(&i_full[g % kIdx], (g / kIdx) & 1);
    const int mt_done = *mma_tiles;
    if (mt_done > 0) mbar_wait(done, (mt_done - 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, tcols);
}

// y[b][o] = bf16((bias[o]) + sum_s part[s][b][o]), s ascending; four outputs
// per thread (n_out is a multiple of 8, so a group never crosses a row)
__global__ void __launch_bounds__(256) k_tc_finish(const float *__restrict__ part, int n_split, int batch, int n_out,
                                                   const float *__restrict__ bias, bf16 *__restrict__ y) {
  pdl_wait();
  const int64_t total = (int64_t)batch * n_out, groups = total / 4;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += (int64_t)gridDim.x * blockDim.x) {
    float4 a = __ldcs(reinterpret_cast<const float4 *>(part) + g);
    for (int k = 1; k < n_split; ++k) {
      const float4 c = __ldcs(reinterpret_cast<const float4 *>(part + (size_t)k * total) + g);
      a.x += c.x;
      a.y += c.y;
      a.z += c.z;
      a.w += c.w;
    }
    if (bias) {  // the caller's bias and output need only their element alignment
      const float *bb = bias + (g * 4) % n_out;
      a.x = bb[0] + a.x;
      a.y = bb[1] + a.y;
      a.z = bb[2] + a.z;
      a.w = bb[3] + a.w;
    }
    bf16 *yo = y + g * 4;
    yo[0] = __float2bfloat16_rn(a.x);
    yo[1] = __float2bfloat16_rn(a.y);
    yo[2] = __float2bfloat16_rn(a.z);
    yo[3] = __float2bfloat16_rn(a.w);
  }
}

// The plan's mask and offset tables (see TcArgs): one warp per row, the
// row's bits gathered per block in shared memory (kTabWarps rows per CTA).
constexpr int kTabWarps = 4;
__global__ void __launch_bounds__(kTabWarps * 32) k_tables(const int32_t *__restrict__ rp,
                                                         const uint16_t *__restrict__ col16, int32_t out_f,
                                                         int32_t nkb, uint64_t *__restrict__ mask,
                                                         int32_t *__restrict__ koff) {
  pdl_wait();
  extern __shared__ unsigned long long tab_bits[];  // [kTabWarps][nkb]
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kTabWarps + w;
  unsigned long long *bits = tab_bits + (size_t)w * nkb;
  for (int kb = lane; kb < nkb; kb += 32) bits[kb] = 0ull;
  __syncwarp();
  if (r < out_f) {
    const int k0 = rp[r], k1 = rp[r + 1];
    for (int k = k0 + lane; k < k1; k += 32) {
      const int c = col16[k];
      atomicOr(&bits[c >> 6], 1ull << (c & 63));
      const int b = c >> 6;
      const int bp = k > k0 ? (col16[k - 1] >> 6) : -1;
      for (int q = bp + 1; q <= b; ++q) koff[(size_t)q * out_f + r] = k;  // first entry at a column >= 64 q
    }
    const int blast = k1 > k0 ? (col16[k1 - 1] >> 6) : -1;
    for (int q = blast + 1 + lane; q <= nkb; q += 32) koff[(size_t)q * out_f + r] = k1;
  }
  __syncwarp();
  if (r < out_f)
    for (int kb = lane; kb < nkb; kb += 32) mask[(size_t)kb * out_f + r] = bits[kb];
}

typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows][cols] (cols contiguous, ld elements apart), boxes of
// 64 columns x box_rows rows, 128-byte swizzle, zero fill outside
bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kKb, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// one of the plan's [block][row] tables (elements of 4 or 8 bytes) in boxes
// of box_rows rows x box_blocks blocks (no swizzle; zero fill outside, which
// reads as blocks without stored weights)
bool make_table_map(CUtensorMap *m, const void *table, int32_t out_f, int32_t blocks, bool wide, uint32_t box_rows,
                    uint32_t box_blocks) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const size_t es = wide ? 8 : 4;
  const cuuint64_t dims[2] = {(cuuint64_t)out_f, (cuuint64_t)blocks};
  const cuuint64_t strides[1] = {(cuuint64_t)out_f * es};
  const cuuint32_t box[2] = {box_rows, box_blocks};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, wide ? CU_TENSOR_MAP_DATA_TYPE_INT64 : CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void *>(table), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int batch_tile(int batch) {
  if (batch > 256) return 256;
  return (batch + 15) / 16 * 16;
}

size_t tc_smem(int mode, int nt) {
  const size_t stage = kATileBytes + (size_t)nt * kKb * 2;
  return 1024 + (size_t)kStages * stage + (mode == kModeDw ? 0 : (size_t)kIdx * kIdxBytes) + 256 +
         (mode == kModeDw ? (size_t)kProdWarps * 32 * 33 * 4 : 0);
}
static_assert(8 * (3 * kStages + 2 * kIdx + 2) + 32 <= 256, "barriers and flags fit their 256 bytes");
static_assert(kProdWarps == 16, "a stage is 16 warp parts: 128 rows / 8, or 64 rows / 8 x 2 blocks");
static_assert(128 * 8 <= 1024 && 128 * 4 <= kIdxBytes - 1024, "an index slice fits");

struct DenseWs {
  size_t part, xt, dyt, err, total;
  int split_fwd, split_dx;
};

int pick_split(int mn_tiles, int k_chunks, int num_sms) {
  int s = num_sms / (mn_tiles > 0 ? mn_tiles : 1);
  if (s < 1) s = 1;
  if (s > 8) s = 8;
  // every split keeps a few K chunks, and none is empty
  while (s > 1 && (k_chunks / s < 4 || (s - 1) * ((k_chunks + s - 1) / s) >= k_chunks)) --s;
  return s;
}

DenseWs dense_ws(int32_t out_f, int32_t in_f, int32_t batch, int num_sms) {
  DenseWs w;
  const int nt = batch_tile(batch);
  const int btiles = (batch + nt - 1) / nt;
  const int nkb = (in_f + kKb - 1) / kKb;
  w.split_fwd = pick_split(((out_f + kM - 1) / kM) * btiles, nkb, num_sms);
  w.split_dx = pick_split(((in_f + kM - 1) / kM) * btiles, (out_f + kKb - 1) / kKb, num_sms);
  const BatchGeom bg = batch_geom(batch, SNACK_BF16);
  size_t o = 0;
  w.part = o;
  const size_t pf = w.split_fwd > 1 ? (size_t)w.split_fwd * batch * out_f * 4 : 0;
  const size_t pd = w.split_dx > 1 ? (size_t)w.split_dx * batch * in_f * 4 : 0;
  o += align_up(pf > pd ? pf : pd, kAlign);
  w.xt = o;
  o += align_up((size_t)in_f * bg.ldx * 2, kAlign);
  w.dyt = o;
  o += align_up((size_t)out_f * bg.ldx * 2, kAlign);
  w.err = o;
  o += kAlign;
  w.total = o;
  return w;
}

template <int kMode>
cudaError_t launch_tc(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mm, const CUtensorMap &mk,
                      const TcArgs &a, int num_sms, cudaStream_t s) {
  const size_t smem = tc_smem(kMode, a.nt);
  cudaError_t e = raise_smem_limit(k_tc<kMode>, smem);
  if (e != cudaSuccess) return e;
  const int tiles = a.m_tiles * a.n_tiles * a.n_split;
  const int grid = tiles < num_sms ? tiles : num_sms;
  launch_pdl(k_tc<kMode>, (unsigned)grid, kThreads, smem, s, ma, mb, mm, mk, a);
  return cudaGetLastError();
}

unsigned grid_of(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > 65535 * 8) b = 65535 * 8;
  return (unsigned)b;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

bool dense_layer(int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch, snack_dtype val_t) {
  return val_t == SNACK_BF16 && max_batch >= kDenseMinBatch && (double)nnz >= kDenseMinDensity * (double)out_f * (double)in_f &&
         out_f % 8 == 0 && in_f % 8 == 0 && out_f <= 65536 && in_f <= 65536;
}

size_t dense_table_bytes(int32_t out_f, int32_t in_f) {
  const size_t nkb = (size_t)(in_f + kKb - 1) / kKb;
  return align_up(nkb * out_f * sizeof(uint64_t), kAlign) + align_up((nkb + 1) * out_f * sizeof(int32_t), kAlign);
}

cudaError_t build_tables(const int32_t *rp, const uint16_t *col16, int32_t out_f, int32_t in_f, void *tables,
                         cudaStream_t s) {
  const int nkb = (in_f + kKb - 1) / kKb;
  uint64_t *mask = reinterpret_cast<uint64_t *>(tables);
  int32_t *koff =
      reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(tables) + align_up((size_t)nkb * out_f * 8, kAlign));
  const size_t smem = (size_t)kTabWarps * nkb * sizeof(uint64_t);
  cudaError_t e = raise_smem_limit(k_tables, smem);
  if (e != cudaSuccess) return e;
  launch_pdl(k_tables, (unsigned)((out_f + kTabWarps - 1) / kTabWarps), kTabWarps * 32, smem, s, rp, col16, out_f, nkb,
             mask, koff);
  return cudaGetLastError();
}

size_t dense_ws_bytes(int32_t out_f, int32_t in_f, int32_t max_batch, int num_sms) {
  return dense_ws(out_f, in_f, max_batch, num_sms).total;
}

namespace {
// the layer's tables in the plan, and the maps of their stage slices
void set_tables(TcArgs &a, const snack_layer *h) {
  a.nkb = (h->in_f + kKb - 1) / kKb;
  a.mask = reinterpret_cast<const uint64_t *>(h->p.tables);
  a.koff = reinterpret_cast<const int32_t *>(reinterpret_cast<const uint8_t *>(h->p.tables) +
                                             align_up((size_t)a.nkb * h->out_f * 8, kAlign));
}
bool table_maps(CUtensorMap *mm, CUtensorMap *mk, const TcArgs &a, uint32_t rows, uint32_t blocks) {
  return make_table_map(mm, a.mask, a.out_f, a.nkb, true, rows, blocks) &&
         make_table_map(mk, a.koff, a.out_f, a.nkb + 1, false, rows, blocks);
}
}  // namespace

bool dense_call_ok(const snack_layer *h, int32_t batch, const void *act, size_t ws_bytes) {
  return h->dense && h->p.tables && batch >= kDenseMinBatch && aligned16(act) &&
         ws_bytes >= dense_ws(h->out_f, h->in_f, batch, h->num_sms).total;
}

snack_status dense_fwd(snack_layer *h, const void *val, const void *x, int32_t batch, const float *bias, void *y,
                       void *ws, size_t ws_bytes, cudaStream_t s) {
  const DenseWs W = dense_ws(h->out_f, h->in_f, batch, h->num_sms);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const int nt = batch_tile(batch);
  TcArgs a = {};
  a.out_f = h->out_f;
  a.in_f = h->in_f;
  a.batch = batch;
  set_tables(a, h);
  a.val = reinterpret_cast<const uint16_t *>(val);
  a.bias = bias;
  a.out = reinterpret_cast<bf16 *>(y);
  a.part = reinterpret_cast<float *>(b + W.part);
  a.n_out = h->out_f;
  a.nt = nt;
  a.m_tiles = (h->out_f + kM - 1) / kM;
  a.n_tiles = (batch + nt - 1) / nt;
  a.n_split = W.split_fwd;
  a.k_chunks = (h->in_f + kKb - 1) / kKb;
  a.err = reinterpret_cast<uint32_t *>(b + W.err);
  CUtensorMap mx, mm, mk;
  if (!make_map(&mx, x, (uint64_t)h->in_f, (uint64_t)batch, (uint64_t)h->in_f, (uint32_t)nt) ||
      !table_maps(&mm, &mk, a, kM, 1))
    return SNACK_ERR_CUDA;
  if (launch_tc<kModeFwd>(mx, mx, mm, mk, a, h->num_sms, s) != cudaSuccess) return SNACK_ERR_CUDA;
  if (a.n_split > 1) {
    launch_pdl(k_tc_finish, grid_of((int64_t)batch * h->out_f / 4, 256), 256, 0, s, (const float *)a.part, a.n_split, batch,
               h->out_f, bias, a.out);
    if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  }
  return SNACK_OK;
}

snack_status dense_dx(snack_layer *h, const void *val, const void *dy, int32_t batch, void *dx, void *ws,
                      size_t ws_bytes, cudaStream_t s) {
  const DenseWs W = dense_ws(h->out_f, h->in_f, batch, h->num_sms);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const int nt = batch_tile(batch);
  TcArgs a = {};
  a.out_f = h->out_f;
  a.in_f = h->in_f;
  a.batch = batch;
  set_tables(a, h);
  a.val = reinterpret_cast<const uint16_t *>(val);
  a.out = reinterpret_cast<bf16 *>(dx);
  a.part = reinterpret_cast<float *>(b + W.part);
  a.n_out = h->in_f;
  a.nt = nt;
  a.m_tiles = (h->in_f + kM - 1) / kM;
  a.n_tiles = (batch + nt - 1) / nt;
  a.n_split = W.split_dx;
  a.k_chunks = (h->out_f + kKb - 1) / kKb;
  a.err = reinterpret_cast<uint32_t *>(b + W.err);
  CUtensorMap md, mm, mk;
  if (!make_map(&md, dy, (uint64_t)h->out_f, (uint64_t)batch, (uint64_t)h->out_f, (uint32_t)nt) ||
      !table_maps(&mm, &mk, a, 64, 2))
    return SNACK_ERR_CUDA;
  if (launch_tc<kModeDx>(md, md, mm, mk, a, h->num_sms, s) != cudaSuccess) return SNACK_ERR_CUDA;
  if (a.n_split > 1) {
    launch_pdl(k_tc_finish, grid_of((int64_t)batch * h->in_f / 4, 256), 256, 0, s, (const float *)a.part, a.n_split, batch,
               h->in_f, (const float *)nullptr, a.out);
    if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  }
  return SNACK_OK;
}

snack_status dense_dw(snack_layer *h, const void *x, const void *dy, int32_t batch, float *dw, float *db, void *ws,
                      size_t ws_bytes, cudaStream_t s) {
  const DenseWs W = dense_ws(h->out_f, h->in_f, batch, h->num_sms);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  const BatchGeom bg = batch_geom(batch, SNACK_BF16);
  bf16 *xt = reinterpret_cast<bf16 *>(b + W.xt);
  bf16 *dyt = reinterpret_cast<bf16 *>(b + W.dyt);
  // feature-major copies (batch contiguous, zero-padded to ldx): the K-major operands of dY^T X
  TransposePair<bf16> tp{reinterpret_cast<const bf16 *>(dy), reinterpret_cast<const bf16 *>(x), dyt, xt, h->out_f,
                         h->in_f, bg.ldx <= 32 ? db : nullptr};
  if (run_transpose2<bf16>(tp, batch, bg.ldx, s) != cudaSuccess) return SNACK_ERR_CUDA;
  if (db && !tp.db0 && run_rowsum_t<bf16>(dyt, bg.ldx, batch, h->out_f, db, s) != cudaSuccess) return SNACK_ERR_CUDA;
  if (h->nnz == 0) return SNACK_OK;
  TcArgs a = {};
  a.out_f = h->out_f;
  a.in_f = h->in_f;
  a.batch = batch;
  set_tables(a, h);
  a.dw = dw;
  a.nt = kDwN;
  a.m_tiles = (h->out_f + kM - 1) / kM;
  a.n_tiles = (h->in_f + kDwN - 1) / kDwN;
  a.n_split = 1;
  a.k_chunks = (bg.ldx + kKb - 1) / kKb;
  a.err = reinterpret_cast<uint32_t *>(b + W.err);
  CUtensorMap ma, mb;
  if (!make_map(&ma, dyt, (uint64_t)bg.ldx, (uint64_t)h->out_f, (uint64_t)bg.ldx, (uint32_t)kM) ||
      !make_map(&mb, xt, (uint64_t)bg.ldx, (uint64_t)h->in_f, (uint64_t)bg.ldx, (uint32_t)kDwN))
    return SNACK_ERR_CUDA;
  if (launch_tc<kModeDw>(ma, mb, mb, mb, a, h->num_sms, s) != cudaSuccess) return SNACK_ERR_CUDA;
  return SNACK_OK;
}

}  // namespace snack
