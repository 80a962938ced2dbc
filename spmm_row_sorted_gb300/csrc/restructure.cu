// Dynamic Sparse Training restructure on the GPU (prune smallest |w|, regrow
// at random empty positions with value +0, re-sort the COO).
//
//  1. prune set: radix select (digits of 11, 10 and 10 bits, high to low) of
//     the n_prune-th smallest magnitude key t; ties at t are pruned in
//     storage order, so the pruned set is exactly the n_prune smallest (|w|, k);
//  2. survivors: one scan of the packed pair (key > t, key == t) gives every
//     survivor its output slot (stable compaction);
//  3. regrow: draws i of SplitMix64 map to positions by multiply-high; a draw
//     is a candidate when the position was empty (binary search in its old
//     row), and is accepted when it is the first draw of its position -- a
//     hash table keeps the minimum draw index per position (atomicMin, so the
//     outcome does not depend on thread order); a scan over draw order keeps
//     the first n_prune accepted.  Draws run in chunks until enough are
//     accepted; the first chunk is queued before steps 1 and 2 and the host
//     reads its count back while the device runs them;
//  4. regrown positions are sorted: the accept scan drops each accepted
//     position into an equal-width bucket of the position range, one block
//     turns the bucket counts into offsets and one warp per bucket places its
//     positions by rank (a general sort takes over after extra draw chunks or
//     a full bucket); then they are merged with the survivors by position
//     (merge path), writing row/col/val/src.
// Every step is integer work, so the output is bit-exact with the sequential
// definition.
#include <math.h>

#include "internal.hpp"
#include "prims.cuh"

namespace snack {

namespace {

constexpr uint64_t kEmpty = ~0ull;
constexpr int kMergeThreads = 256;
constexpr int kMergeItems = 4;
constexpr int kMergeTile = kMergeThreads * kMergeItems;
static_assert(2 * kMergeTile == kRadixTile, "two merge tiles make one tile of the column view's first radix pass");

// The column view's first-level tile histogram of the merged pattern, from
// the merge's split points alone (beside the merge, on the other stream):
// radix tile t holds the outputs of merge tiles 2t and 2t+1, i.e. survivor
// keys A[a0, a1) and regrown keys B[d0 - a0, d1 - a1); each output's digit is
// its column's high 8 bits.  Every bin is written (digit-major [256][tiles]).
__global__ void __launch_bounds__(256) k_col_hist(const uint64_t *__restrict__ A, const uint64_t *__restrict__ B,
                                                  const int64_t *__restrict__ part, int64_t n_merge_tiles, int64_t n,
                                                  int cbits, int cshift, uint32_t *__restrict__ chist, int64_t cnb) {
  pdl_wait();
  __shared__ uint32_t h[8][kRadixBins];  // one histogram per warp: less atomic contention
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 8 * kRadixBins; i += 256) (&h[0][0])[i] = 0u;
  __syncthreads();
  const int64_t t = blockIdx.x;
  const int64_t d0 = t * kRadixTile, d1 = d0 + kRadixTile < n ? d0 + kRadixTile : n;
  const int64_t m1 = 2 * t + 2 < n_merge_tiles ? 2 * t + 2 : n_merge_tiles;
  const int64_t a0 = part[2 * t], a1 = part[m1];
  const int64_t b0 = d0 - a0, b1 = d1 - a1;
  const uint64_t cmask = (1ull << cbits) - 1ull;
  for (int64_t q = a0 + threadIdx.x; q < a1; q += 256)
    atomicAdd(&h[warp][(uint32_t)((A[q] & cmask) >> cshift) & 0xFFu], 1u);
  for (int64_t q = b0 + threadIdx.x; q < b1; q += 256)
    atomicAdd(&h[warp][(uint32_t)((B[q] & cmask) >> cshift) & 0xFFu], 1u);
  __syncthreads();
  for (int d = threadIdx.x; d < kRadixBins; d += 256) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += h[w][d];
    chist[(int64_t)d * cnb + t] = c;
  }
}

struct SelState {
  uint32_t prefix, remaining, n_prune, total;  // prefix = threshold key t, remaining = ties to prune
  uint32_t overflow;                           // a draw found the position table full
  uint32_t pfx, mask, rem;                     // select progress: digits fixed so far, ranks left within them
  uint32_t arrive[4];                          // blocks finished per pass
  uint32_t hist0[2048], hist1[1024], hist2[1024];  // digit histograms: key bits 30..20, 19..10, 9..0
};

__device__ __forceinline__ uint32_t canon_mag(uint32_t m) { return m > 0x7F800000u ? 0x7F800001u : m; }

template <typename TV>
__device__ __forceinline__ uint32_t mag_key(const TV *val, int64_t k);
template <>
__device__ __forceinline__ uint32_t mag_key<float>(const float *val, int64_t k) {
  return canon_mag(__float_as_uint(val[k]) & 0x7FFFFFFFu);
}
template <>
__device__ __forceinline__ uint32_t mag_key<bf16>(const bf16 *val, int64_t k) {
  uint32_t b = reinterpret_cast<const uint16_t *>(val)[k];
  return canon_mag((b & 0x7FFFu) << 16);
}

template <int kPass>
struct SelDigit {
  static constexpr int kShift = kPass == 0 ? 20 : (kPass == 1 ? 10 : 0);
  static constexpr int kBins = kPass == 0 ? 2048 : 1024;
};

// One pass of the radix select over the 31-bit magnitude keys (digits of 11,
// 10 and 10 bits, high first).  Every block histograms the digit of the keys
// that match the digits fixed so far, adds its counts to the global
// histogram, and the last block to finish picks the digit holding rank
// `rem` (no extra launch, no waiting: the last arrival does the pick).
template <typename TV, int kPass>
__global__ void __launch_bounds__(256) k_sel_pass(const TV *__restrict__ val, int64_t nnz, SelState *st) {
  pdl_wait();
  constexpr int kItems = 16;
  constexpr int kShift = SelDigit<kPass>::kShift, kBins = SelDigit<kPass>::kBins, kPer = kBins / 256;
  __shared__ uint32_t h[kBins];
  __shared__ uint32_t s_scan[256];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + tid;
  uint32_t key[kItems];
#pragma unroll
  for (int u = 0; u < kItems; ++u) key[u] = first + u * stride < nnz ? mag_key<TV>(val, first + u * stride) : 0u;
  __shared__ uint32_t s_pm[2];
  for (int i = tid; i < kBins; i += 256) h[i] = 0;
  if (tid == 0) {  // one load per block: the digits fixed by the previous pass
    s_pm[0] = kPass ? st->pfx : 0u;
    s_pm[1] = kPass ? st->mask : 0u;
  }
  __syncthreads();
  const uint32_t pfx = s_pm[0], mask = s_pm[1];
#pragma unroll
  for (int u = 0; u < kItems; ++u)
    if (first + u * stride < nnz && (key[u] & mask) == pfx) atomicAdd(&h[(key[u] >> kShift) & (kBins - 1)], 1u);
  for (int64_t k0 = first + kItems * stride; k0 < nnz; k0 += kItems * stride) {
#pragma unroll
    for (int u = 0; u < kItems; ++u) key[u] = k0 + u * stride < nnz ? mag_key<TV>(val, k0 + u * stride) : 0u;
#pragma unroll
    for (int u = 0; u < kItems; ++u)
      if (k0 + u * stride < nnz && (key[u] & mask) == pfx) atomicAdd(&h[(key[u] >> kShift) & (kBins - 1)], 1u);
  }
  __syncthreads();
  uint32_t *gh = kPass == 0 ? st->hist0 : (kPass == 1 ? st->hist1 : st->hist2);
  for (int i = tid; i < kBins; i += 256)
    if (h[i]) atomicAdd(&gh[i], h[i]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&st->arrive[kPass], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last block: exclusive scan of the global histogram, then the digit d at
  // which the running count first reaches rem
  const uint32_t rem = kPass ? st->rem : st->n_prune;
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    c[j] = __ldcg(&gh[tid * kPer + j]);
    sum += c[j];
  }
  s_scan[tid] = sum;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    uint32_t v = tid >= off ? s_scan[tid - off] : 0u;
    __syncthreads();
    s_scan[tid] += v;
    __syncthreads();
  }
  uint32_t ex = s_scan[tid] - sum;
  if (ex < rem && ex + sum >= rem) {
#pragma unroll 1
    for (int j = 0; j < kPer; ++j) {
      if (ex + c[j] >= rem) {
        const uint32_t d = (uint32_t)(tid * kPer + j);
        const uint32_t np = pfx | (d << kShift), nm = mask | ((uint32_t)(kBins - 1) << kShift);
        st->pfx = np;
        st->mask = nm;
        st->rem = rem - ex;
        if (kPass == 2) {
          st->prefix = np;
          st->remaining = rem - ex;
        }
        break;
      }
      ex += c[j];
    }
  }
}

__global__ void k_sel_init(SelState *st, uint32_t n_prune) {
  pdl_wait();
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) st->hist0[i] = 0;
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) {
    st->hist1[i] = 0;
    st->hist2[i] = 0;
  }
  if (threadIdx.x < 4) st->arrive[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    st->prefix = 0;
    st->remaining = 0;
    st->n_prune = n_prune;
    st->total = 0;
    st->overflow = 0;
    st->pfx = 0;
    st->mask = 0;
    st->rem = n_prune;
  }
}

template <typename TV>
struct KeepVal {
  const TV *val;
  const SelState *st;
  __device__ uint64_t operator()(int64_t k) const {
    // every element reads the threshold: through the read-only cache, so the
    // SMs do not all queue on one L2 line
    uint32_t key = mag_key<TV>(val, k), t = __ldg(&st->prefix);
    return (uint64_t)(key > t) | ((uint64_t)(key == t) << 32);
  }
};

// position key (row << cbits) | col of stored weight k, loaded with the scan
// value; keys order positions as row * in_f + col does, and split with a
// shift and a mask
struct PosPayload {
  const int32_t *row, *col;
  int cbits;
  __device__ uint64_t operator()(int64_t k) const {
    return ((uint64_t)(uint32_t)row[k] << cbits) | (uint32_t)col[k];
  }
};

struct KeepOut {
  const SelState *st;
  uint64_t *surv_pos;
  uint32_t *surv_src;
  __device__ void operator()(int64_t k, uint64_t ex, uint64_t v, uint64_t pos) const {
    const uint32_t m = __ldg(&st->remaining);
    const uint32_t gt = (uint32_t)ex, eq = (uint32_t)(ex >> 32);
    const bool keep = (v & 1ull) || ((v >> 32) && eq >= m);
    if (keep) {
      uint32_t s = gt + (eq > m ? eq - m : 0u);
      surv_pos[s] = pos;
      surv_src[s] = (uint32_t)k;
    }
  }
};

__device__ __forceinline__ uint32_t hash_min(const uint64_t *keys, const uint32_t *mins, uint64_t mask, uint64_t p) {
  uint64_t h = sm64_finalise(p) & mask;
  for (uint64_t probe = 0; probe <= mask; ++probe) {
    uint64_t k = keys[h];
    if (k == p) return mins[h];
    if (k == kEmpty) return 0xFFFFFFFFu;
    h = (h + 1) & mask;
  }
  return 0xFFFFFFFFu;
}

__global__ void k_draw(uint64_t base, uint64_t i0, int64_t m, uint64_t n_pos, int32_t in_f, int cbits,
                       const int32_t *__restrict__ rp, const int32_t *__restrict__ col, uint64_t *__restrict__ cand,
                       uint64_t *hkeys, uint32_t *hmin, uint64_t hmask, uint32_t *overflow) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < m; idx += stride) {
    const uint64_t i = i0 + (uint64_t)idx;
    const uint64_t u = sm64_finalise(base + (i + 1) * kGolden);
    const uint64_t p = __umul64hi(u, n_pos);
    const uint64_t r = p / (uint64_t)in_f;
    const int32_t c = (int32_t)(p - r * (uint64_t)in_f);
    int32_t lo = rp[r], hi = rp[r + 1];
    while (lo < hi) {
      int32_t mid = lo + (hi - lo) / 2;
      if (col[mid] < c)
        lo = mid + 1;
      else
        hi = mid;
    }
    const bool member = lo < rp[r + 1] && col[lo] == c;
    if (member) {
      cand[idx] = kEmpty;
      continue;
    }
    const uint64_t key = (r << cbits) | (uint32_t)c;  // position key of the draw
    cand[idx] = key;
    uint64_t h = sm64_finalise(key) & hmask;
    bool done = false;
    for (uint64_t probe = 0; probe <= hmask; ++probe) {
      unsigned long long prev =
          atomicCAS(reinterpret_cast<unsigned long long *>(hkeys + h), (unsigned long long)kEmpty,
                    (unsigned long long)key);
      if (prev == kEmpty || prev == key) {
        atomicMin(hmin + h, (uint32_t)i);
        done = true;
        break;
      }
      h = (h + 1) & hmask;
    }
    if (!done) atomicOr(overflow, 1u);
  }
}

// flag[idx] = 1 when draw i0+idx found an empty position and is the first
// draw of that position (its index is the minimum recorded for it)
__global__ void k_accept_flags(const uint64_t *__restrict__ cand, int64_t m, uint64_t i0,
                               const uint64_t *__restrict__ hkeys, const uint32_t *__restrict__ hmin, uint64_t hmask,
                               uint32_t *__restrict__ flags) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < m; idx += stride) {
    const uint64_t p = cand[idx];
    flags[idx] = (p != kEmpty && hash_min(hkeys, hmin, hmask, p) == (uint32_t)(i0 + (uint64_t)idx)) ? 1u : 0u;
  }
}

struct FlagRead {
  const uint32_t *f;
  __device__ uint32_t operator()(int64_t i) const { return f[i]; }
};

struct CandPayload {
  const uint64_t *cand;
  __device__ uint64_t operator()(int64_t idx) const { return cand[idx]; }
};

// Accepted draws in draw order: slot q of the regrown list, and -- for the
// sort -- a slot in the position's bucket (equal-width buckets of the
// position range, kBktCap slots each, filled in any order; a full bucket
// raises `bovf` and the caller sorts the list the general way instead).
constexpr int kBktTarget = 32;  // positions expected per bucket
constexpr int kBktCap = 128;    // slots per bucket

struct AcceptOut {
  uint64_t *grown;
  int64_t before, n_prune;
  uint32_t *bcnt;     // [nb] positions placed per bucket
  uint64_t *bslots;   // [nb][kBktCap]
  double scale;       // bucket = floor(p * scale)
  uint32_t nb;
  uint32_t *bovf;
  __device__ void operator()(int64_t idx, uint32_t ex, uint32_t v, uint64_t p) const {
    if (v) {
      int64_t q = before + (int64_t)ex;
      if (q < n_prune) {
        grown[q] = p;
        const uint32_t bk = bucket_of(p, scale, nb);
        const uint32_t slot = atomicAdd(&bcnt[bk], 1u);
        if (slot < (uint32_t)kBktCap)
          bslots[(size_t)bk * kBktCap + slot] = p;
        else
          atomicOr(bovf, 1u);
      }
    }
  }
};

// Counters of the regrow branch (it runs beside the select on a second stream).
struct DrawState {
  uint32_t total, overflow;  // accepted draws of the last chunk; a draw found the position table full
  uint32_t bucket_overflow;  // a sort bucket of the regrown positions ran out of slots
};

// Bucket offsets: exclusive prefix of min(count, kBktCap) over the nb
// buckets, one block of light threads (it runs beside the other stream's
// kernels): each thread sums a contiguous run of counts, 16 loads in flight
// per round, the block scans the sums, and the thread writes its run's
// offsets; offs[nb] = the number of positions placed.  Thread 0 first copies
// the draw chunk's counters to the host's mapped words (the accept scan that
// wrote them precedes this kernel), so the host reads them with no copy on
// the stream.
constexpr int kBktScanThreads = 1024;
__global__ void __launch_bounds__(kBktScanThreads) k_bkt_scan(const uint32_t *__restrict__ bcnt, uint32_t nb,
                                                              uint32_t *__restrict__ offs, const DrawState *ds,
                                                              volatile uint32_t *host_words) {
  pdl_wait();
  __shared__ uint32_t s_warp[kBktScanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    host_words[0] = ds->total;
    host_words[1] = ds->overflow;
    host_words[2] = ds->bucket_overflow;
  }
  const uint32_t per = (nb + kBktScanThreads - 1) / kBktScanThreads;
  const uint32_t b0 = min((uint32_t)tid * per, nb), b1 = min(b0 + per, nb);
  uint32_t sum = 0;
  for (uint32_t i0 = b0; i0 < b1; i0 += 16) {
    uint32_t c[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) c[i] = i0 + i < b1 ? min(__ldg(&bcnt[i0 + i]), (uint32_t)kBktCap) : 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) sum += c[i];
  }
  const uint32_t inc = warp_inclusive_scan(sum);
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) s_warp[lane] = warp_inclusive_scan(s_warp[lane]);
  __syncthreads();
  uint32_t run = inc - sum + (warp > 0 ? s_warp[warp - 1] : 0u);
  for (uint32_t i0 = b0; i0 < b1; i0 += 16) {
    uint32_t c[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) c[i] = i0 + i < b1 ? min(__ldg(&bcnt[i0 + i]), (uint32_t)kBktCap) : 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i0 + i < b1) offs[i0 + i] = run;
      run += c[i];
    }
  }
  if (tid == kBktScanThreads - 1) offs[nb] = run;
}

// Start of a restructure's regrow branch: counters and bucket counts to zero,
// the position table to empty (one launch instead of four fills).
__global__ void k_rs_init(DrawState *ds, uint64_t *__restrict__ hkeys, uint32_t *__restrict__ hmin, int64_t cap,
                          uint32_t *__restrict__ bcnt, int64_t nb) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 == 0) {
    ds->total = 0u;
    ds->overflow = 0u;
    ds->bucket_overflow = 0u;
  }
  for (int64_t i = i0; i < cap; i += stride) {
    hkeys[i] = kEmpty;
    hmin[i] = 0xFFFFFFFFu;
  }
  for (int64_t i = i0; i < nb; i += stride) bcnt[i] = 0u;
}

// One warp per bucket: each position's rank among its bucket's (distinct)
// positions gives its place in the sorted list.  Slots past the placed
// positions get key_space + q, larger than every position key, in order.
__global__ void __launch_bounds__(256) k_bkt_rank(const uint64_t *__restrict__ bslots, const uint32_t *__restrict__ bcnt,
                                                  const uint32_t *__restrict__ offs, uint32_t nb, int64_t n,
                                                  uint64_t key_space, uint64_t *__restrict__ out) {
  pdl_wait();
  __shared__ uint64_t sk[8][kBktCap];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tot = offs[nb];
  for (int64_t q = tot + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += (int64_t)gridDim.x * blockDim.x)
    out[q] = key_space + (uint64_t)q;
  const int64_t b = (int64_t)blockIdx.x * 8 + warp;
  if (b >= nb) return;
  const uint32_t L = min(bcnt[b], (uint32_t)kBktCap), o = offs[b];
  for (uint32_t i = lane; i < L; i += 32) sk[warp][i] = bslots[(size_t)b * kBktCap + i];
  __syncwarp();
  for (uint32_t i = lane; i < L; i += 32) {
    const uint64_t k = sk[warp][i];
    uint32_t r = 0;
    for (uint32_t j = 0; j < L; ++j) r += sk[warp][j] < k ? 1u : 0u;
    out[o + r] = k;
  }
}

// Number of A elements among the first d outputs of the merge (A first on
// ties), by one warp: the predicate A[a] <= B[d-1-a] holds on a prefix of
// candidate a, so each round probes 32 points and keeps the crossing.
__device__ int64_t merge_split_warp(const uint64_t *A, int64_t na, const uint64_t *B, int64_t nb, int64_t d) {
  const int lane = threadIdx.x & 31;
  int64_t lo = d > nb ? d - nb : 0, hi = d < na ? d : na;  // answer in [lo, hi]
  while (hi - lo > 32) {
    const int64_t span = hi - lo;
    const int64_t p = lo + span * (lane + 1) / 33;  // lo < p < hi
    const bool ok = A[p] <= B[d - 1 - p];
    const int cnt = __popc(__ballot_sync(0xffffffffu, ok));
    const int64_t new_lo = cnt > 0 ? lo + span * cnt / 33 + 1 : lo;
    const int64_t new_hi = cnt < 32 ? lo + span * (cnt + 1) / 33 : hi;
    lo = new_lo;
    hi = new_hi;
  }
  const int64_t a = lo + lane;
  const bool ok = a < hi && A[a] <= B[d - 1 - a];
  return lo + __popc(__ballot_sync(0xffffffffu, ok));
}

// part[t] = A elements among the first t*kMergeTile outputs, one warp per split
__global__ void k_merge_splits(const uint64_t *__restrict__ A, int64_t na, const uint64_t *__restrict__ B, int64_t nb,
                               int64_t n_tiles, int64_t *__restrict__ part) {
  pdl_wait();
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t > n_tiles) return;
  int64_t d = t * kMergeTile;
  if (d > na + nb) d = na + nb;
  const int64_t sp = merge_split_warp(A, na, B, nb, d);
  if ((threadIdx.x & 31) == 0) part[t] = sp;
}

template <typename TV>
__global__ void __launch_bounds__(kMergeThreads)
    k_merge(const uint64_t *__restrict__ A, const uint32_t *__restrict__ As, int64_t na, const uint64_t *__restrict__ B,
            int64_t nb, const int64_t *__restrict__ part, int cbits, int32_t out_f, const TV *__restrict__ val,
            int32_t *__restrict__ row_out, int32_t *__restrict__ col_out, TV *__restrict__ val_out,
            int32_t *__restrict__ src_out, int32_t *__restrict__ rp, uint16_t *__restrict__ col16) {
  pdl_wait();
  __shared__ uint64_t sA[kMergeTile];
  __shared__ uint64_t sB[kMergeTile];
  __shared__ uint32_t sS[kMergeTile];  // survivor sources; then the output sources (oS)
  int32_t *oS = reinterpret_cast<int32_t *>(sS);
  // after the merge, the two key arrays hold the outputs' rows and columns as 32-bit words
  uint32_t *oR = reinterpret_cast<uint32_t *>(sA), *oC = reinterpret_cast<uint32_t *>(sB);
  const int64_t t = blockIdx.x;
  const int64_t n = na + nb;
  const uint64_t cmask = (1ull << cbits) - 1ull;
  const int64_t d0 = t * kMergeTile;
  const int64_t d1 = d0 + kMergeTile < n ? d0 + kMergeTile : n;
  const int64_t a0 = part[t], a1 = part[t + 1];
  const int64_t b0 = d0 - a0, b1 = d1 - a1;
  const int la = (int)(a1 - a0), lb = (int)(b1 - b0);
  for (int q = threadIdx.x; q < la; q += kMergeThreads) {
    sA[q] = A[a0 + q];
    sS[q] = As[a0 + q];
  }
  for (int q = threadIdx.x; q < lb; q += kMergeThreads) sB[q] = B[b0 + q];
  __syncthreads();
  int ld = threadIdx.x * kMergeItems;
  if (ld > la + lb) ld = la + lb;
  int lo = ld > lb ? ld - lb : 0, hi = ld < la ? ld : la;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (sA[mid] <= sB[ld - 1 - mid])
      lo = mid + 1;
    else
      hi = mid;
  }
  int ai = lo, bi = ld - lo;
  uint64_t pos[kMergeItems];
  int32_t src[kMergeItems];
#pragma unroll
  for (int it = 0; it < kMergeItems; ++it) {
    src[it] = -2;
    if (ld + it >= la + lb) continue;
    bool take_a = bi >= lb || (ai < la && sA[ai] <= sB[bi]);
    if (take_a) {
      pos[it] = sA[ai];
      src[it] = (int32_t)sS[ai];
      ++ai;
    } else {
      pos[it] = sB[bi];
      src[it] = -1;
      ++bi;
    }
  }
  __syncthreads();
  // stage rows / cols / sources in shared memory, then write coalesced
#pragma unroll
  for (int it = 0; it < kMergeItems; ++it)
    if (src[it] != -2) {
      const uint32_t c = (uint32_t)(pos[it] & cmask);
      oR[ld + it] = (uint32_t)(pos[it] >> cbits);
      oC[ld + it] = c;
      oS[ld + it] = src[it];
    }
  __syncthreads();
  // row offsets of the output: rp[r] = o for the rows r in (row[o-1], row[o]];
  // the row before the tile is that of the larger of the two inputs' last
  // elements consumed by earlier tiles
  int r_before = -1;
  if (d0 > 0) {
    uint64_t last = 0;
    if (a0 > 0) last = A[a0 - 1];
    if (b0 > 0 && B[b0 - 1] > last) last = B[b0 - 1];
    r_before = (int)(last >> cbits);
  }
  for (int q = threadIdx.x; q < la + lb; q += kMergeThreads) {
    const int64_t o = d0 + q;
    const int32_t s = oS[q];
    const uint32_t rr = oR[q], cc = oC[q];
    row_out[o] = (int32_t)rr;
    col_out[o] = (int32_t)cc;
    if (col16) col16[o] = (uint16_t)cc;
    val_out[o] = s >= 0 ? val[s] : from_f32<TV>(0.f);
    if (src_out) src_out[o] = s;
    const int r_cur = (int)rr;
    const int r_prev = q > 0 ? (int)oR[q - 1] : r_before;
    for (int r = r_prev + 1; r <= r_cur && r <= out_f; ++r) rp[r] = (int32_t)o;
  }
  if (d1 == n && threadIdx.x == 0) {  // rows after the last stored weight
    const int64_t r_last = la + lb > 0 ? (int64_t)oR[la + lb - 1] : r_before;
    for (int64_t r = r_last + 1; r <= out_f; ++r) rp[r] = (int32_t)n;  // 64-bit: out_f may be 2^31 - 1
  }
}

unsigned grid_for(int64_t n, int threads, int64_t cap = 65535 * 8) {
  int64_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return (unsigned)b;
}

int bits_for(uint64_t v) {
  int b = 0;
  while (b < 64 && (v >> b) != 0) ++b;
  return b;
}

// Expected number of draws to accept `need` distinct positions out of `empty`
// empty ones, among n_pos equally likely positions: n_pos * (H(empty) -
// H(empty - need)), using ln((e + 1/2) / (e - need + 1/2)) for the difference.
double expected_draws(double n_pos, double empty, double need) {
  if (need <= 0) return 0.0;
  return n_pos * log((empty + 0.5) / (empty - need + 0.5));
}

struct RWs {
  size_t state, dstate, scan, scan2, surv_pos, surv_src, grown_a, grown_b, cand, flags, hkeys, hmin, radix, part, bcnt,
      boffs, bslots, total;
  int64_t d_max, cap, n_merge_tiles;
  uint32_t n_bkt;  // sort buckets of the regrown positions
};

RWs rws_layout(int32_t out_f, int32_t in_f, int64_t nnz, int64_t n_prune) {
  RWs w;
  const double n_pos = (double)out_f * (double)in_f;
  double e = expected_draws(n_pos, n_pos - (double)nnz, (double)n_prune);
  double dm = n_prune > 0 ? ceil(2.0 * e) + 4096.0 : 0.0;
  if (dm > 2147483647.0) dm = 2147483647.0;
  w.d_max = (int64_t)dm;
  int64_t cap = 16;
  while (cap < w.d_max + w.d_max / 4 + 16) cap <<= 1;  // load factor below 0.8 even if every draw is made
  w.cap = cap;
  w.n_merge_tiles = (nnz + kMergeTile - 1) / kMergeTile;
  const size_t n = (size_t)(nnz > 0 ? nnz : 1), np = (size_t)(n_prune > 0 ? n_prune : 1);
  size_t o = 0;
  w.state = o;
  o += align_up(sizeof(SelState), kAlign);
  w.dstate = o;
  o += align_up(sizeof(DrawState), kAlign);
  w.scan = o;
  o += scan_temp_bytes<uint64_t>(nnz > 0 ? nnz : 1);
  w.scan2 = o;  // the accept scan, then the column histogram's scan
  const int64_t col_scan = ceil_div(nnz > 0 ? nnz : 1, kRadixTile) * kRadixBins;
  o += scan_temp_bytes<uint32_t>(w.d_max > col_scan ? w.d_max : col_scan);
  w.surv_pos = o;
  o += align_up(8 * n, kAlign);
  w.surv_src = o;
  o += align_up(4 * n, kAlign);
  w.grown_a = o;
  o += align_up(8 * np, kAlign);
  w.grown_b = o;
  o += align_up(8 * np, kAlign);
  w.cand = o;
  o += align_up(8 * (size_t)(w.d_max > 0 ? w.d_max : 1), kAlign);
  w.flags = o;
  o += align_up(4 * (size_t)(w.d_max > 0 ? w.d_max : 1), kAlign);
  w.hkeys = o;
  o += align_up(8 * (size_t)cap, kAlign);
  w.hmin = o;
  o += align_up(4 * (size_t)cap, kAlign);
  w.radix = o;
  o += bucket_sort_temp_bytes((int64_t)np);
  w.part = o;
  o += align_up(8 * (size_t)(w.n_merge_tiles + 2), kAlign);
  w.n_bkt = (uint32_t)((int64_t)np / kBktTarget > 0 ? (int64_t)np / kBktTarget : 1);
  w.bcnt = o;
  o += align_up(4 * ((size_t)w.n_bkt + 1), kAlign);
  w.boffs = o;
  o += align_up(4 * ((size_t)w.n_bkt + 1), kAlign);
  w.bslots = o;
  o += align_up(8 * (size_t)w.n_bkt * kBktCap, kAlign);
  w.total = o;
  return w;
}

template <typename TV>
snack_status restructure_impl(const RestructureArgs &a, void *ws, size_t ws_bytes, cudaStream_t s) {
  const RWs W = rws_layout(a.out_f, a.in_f, a.nnz, a.n_prune);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  SelState *st = reinterpret_cast<SelState *>(b + W.state);
  void *stemp = b + W.scan;
  uint64_t *surv_pos = reinterpret_cast<uint64_t *>(b + W.surv_pos);
  uint32_t *surv_src = reinterpret_cast<uint32_t *>(b + W.surv_src);
  uint64_t *grown_a = reinterpret_cast<uint64_t *>(b + W.grown_a);
  uint64_t *grown_b = reinterpret_cast<uint64_t *>(b + W.grown_b);
  uint64_t *cand = reinterpret_cast<uint64_t *>(b + W.cand);
  uint64_t *hkeys = reinterpret_cast<uint64_t *>(b + W.hkeys);
  uint32_t *hmin = reinterpret_cast<uint32_t *>(b + W.hmin);
  uint32_t *flags = reinterpret_cast<uint32_t *>(b + W.flags);
  int64_t *part = reinterpret_cast<int64_t *>(b + W.part);
  uint32_t *bcnt = reinterpret_cast<uint32_t *>(b + W.bcnt);
  uint32_t *boffs = reinterpret_cast<uint32_t *>(b + W.boffs);
  uint64_t *bslots = reinterpret_cast<uint64_t *>(b + W.bslots);
  const TV *val = reinterpret_cast<const TV *>(a.val);
  const int64_t nnz = a.nnz, n_prune = a.n_prune, n_surv = nnz - n_prune;
  const uint64_t n_pos = (uint64_t)a.out_f * (uint64_t)a.in_f;
  // positions travel as keys (row << cbits) | col: same order as row * in_f + col
  const int cbits = bits_for((uint64_t)(a.in_f - 1));
  const uint64_t key_space = (uint64_t)a.out_f << cbits;
  // the column view's first-level histogram and offsets are made from the
  // merge's split points on the second stream, beside the merge
  int cshift = 0;
  const bool col_offs = a.cv_offs && a.cv_hist && colview_digits(a.out_f, a.in_f, nnz, &cshift);
  const int64_t cnb = ceil_div(nnz, kRadixTile);
  uint32_t *coffs = a.cv_offs;
  uint32_t *chist = a.cv_hist;
  cudaError_t e;
#define SNACK_TRY(x)                       \
  do {                                     \
    e = (x);                               \
    if (e != cudaSuccess) return SNACK_ERR_CUDA; \
  } while (0)

  // Two branches meet at the merge: the regrow (draws, acceptance, sort of
  // the grown positions) depends only on the old pattern and runs on the
  // handle's second stream, beside the prune select and the survivor scan on
  // the caller's stream.  The host reads each draw chunk's accepted count
  // from mapped pinned words that a kernel writes (an event on the second
  // stream marks them ready) while the device goes on.  Every return after the fork joins the branches first, so no
  // work on the second stream outlives the call's work on s.
  cudaStream_t s2 = a.aux;
  DrawState *ds = reinterpret_cast<DrawState *>(b + W.dstate);
  void *stemp2 = b + W.scan2;
  SNACK_TRY(cudaEventRecord(a.ev_fork, s));
  SNACK_TRY(cudaStreamWaitEvent(s2, a.ev_fork, 0));
  auto join = [&]() -> cudaError_t {
    cudaError_t err = cudaEventRecord(a.ev_join, s2);
    if (err != cudaSuccess) return err;
    return cudaStreamWaitEvent(s, a.ev_join, 0);
  };
  const uint64_t base = sm64_finalise(a.seed ^ sm64_finalise(a.step));
  const double bscale = (double)W.n_bkt / (double)key_space;  // position keys are < key_space
  const double empty = (double)n_pos - (double)nnz;
  int64_t done = 0, acc = 0;
  auto draw_chunk = [&](int64_t m) -> cudaError_t {
    launch_pdl(k_draw, grid_for(m, 256), 256, 0, s2, base, (uint64_t)done, m, n_pos, a.in_f, cbits, a.rp_old, a.col, cand,
                                             hkeys, hmin, (uint64_t)(W.cap - 1), &ds->overflow);
    launch_pdl(k_accept_flags, grid_for(m, 256), 256, 0, s2, cand, m, (uint64_t)done, hkeys, hmin, (uint64_t)(W.cap - 1),
                                                     flags);
    const AcceptOut out{grown_a, acc, n_prune, bcnt, bslots, bscale, W.n_bkt, &ds->bucket_overflow};
    cudaError_t err = scan_apply_pl<uint32_t>(FlagRead{flags}, CandPayload{cand}, m, out, &ds->total, stemp2, s2);
    if (err != cudaSuccess) return err;
    launch_pdl(k_bkt_scan, 1, kBktScanThreads, 0, s2, bcnt, W.n_bkt, boffs, (const DrawState *)ds, a.counts_dev);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return cudaEventRecord(a.counts_ready, s2);
  };
  auto chunk_size = [&]() -> int64_t {
    double want = 1.1 * expected_draws((double)n_pos, empty - (double)acc, (double)(n_prune - acc)) + 1024.0;
    int64_t m = (int64_t)ceil(want);
    return m > W.d_max - done ? W.d_max - done : m;
  };
  int64_t m = 0;
  cudaError_t e2 = cudaSuccess;
  // When at least twice n_prune positions are empty the first chunk is all but
  // certain to accept enough, so the sort of the regrown positions is queued
  // right behind it, before the host has read the count (and redone if more
  // chunks turn out to be needed).
  const bool speculative = n_prune > 1 && (double)n_pos - (double)nnz >= 2.0 * (double)n_prune;
  // The first chunk's accepted positions already sit in their buckets
  // (AcceptOut): bucket offsets, then a rank inside each bucket, with slots
  // the chunk left empty filled past key_space.  After more chunks, or when a
  // bucket overflowed, the whole list is sorted the general way.
  auto sort_grown = [&](bool first_chunk_only) -> cudaError_t {
    if (!first_chunk_only)  // every slot filled by accepted draws
      return bucket_sort_u64(grown_a, n_prune, key_space - 1, grown_b, b + W.radix, s2);
    launch_pdl(k_bkt_rank, (W.n_bkt + 7) / 8, 256, 0, s2, bslots, bcnt, boffs, W.n_bkt, n_prune, key_space, grown_b);
    return cudaGetLastError();
  };
  if (n_prune > 0) {
    launch_pdl(k_rs_init, grid_for(W.cap, 256, 1184), 256, 0, s2, ds, hkeys, hmin, (int64_t)W.cap, bcnt,
               (int64_t)W.n_bkt);
    e2 = cudaGetLastError();
    if (e2 == cudaSuccess) {
      m = chunk_size();
      e2 = draw_chunk(m);
    }
    if (e2 == cudaSuccess && speculative) e2 = sort_grown(true);
  }
  // 1. prune threshold: three digit passes (11, 10, 10 bits), high to low
  launch_pdl(k_sel_init, 1, 256, 0, s, st, (uint32_t)n_prune);
  if (n_prune > 0) {
    const unsigned g = grid_for((nnz + 15) / 16, 256, 1184);
    launch_pdl(k_sel_pass<TV, 0>, g, 256, 0, s, val, nnz, st);
    launch_pdl(k_sel_pass<TV, 1>, g, 256, 0, s, val, nnz, st);
    launch_pdl(k_sel_pass<TV, 2>, g, 256, 0, s, val, nnz, st);
  }
  // 2. survivors
  e = cudaGetLastError();
  if (e == cudaSuccess)
    e = scan_apply_pl<uint64_t>(KeepVal<TV>{val, st}, PosPayload{a.row, a.col, cbits}, nnz,
                                KeepOut{st, surv_pos, surv_src}, (uint64_t *)nullptr, stemp, s);
  if (e != cudaSuccess || e2 != cudaSuccess) {
    join();
    return SNACK_ERR_CUDA;
  }
  // 3. regrow: further chunks only when the first fell short (rare)
  snack_status verdict = SNACK_OK;
  bool resort = !speculative;
  while (n_prune > 0) {
    if (cudaEventSynchronize(a.counts_ready) != cudaSuccess) {
      verdict = SNACK_ERR_CUDA;
      break;
    }
    if (a.host_counts[1]) {
      verdict = SNACK_ERR_WORKSPACE;
      break;
    }
    acc += a.host_counts[0];
    done += m;
    if (a.host_counts[2]) resort = true;  // a bucket overflowed: sort the list the general way
    if (acc >= n_prune) break;
    if (done >= W.d_max) {
      verdict = SNACK_ERR_NO_SPACE;
      break;
    }
    m = chunk_size();
    resort = true;
    if (draw_chunk(m) != cudaSuccess) {
      verdict = SNACK_ERR_CUDA;
      break;
    }
  }
  // 4. sort regrown positions (bucket sort: they are uniform over the empty
  //    positions), then join and merge with the survivors
  const uint64_t *grown = n_prune > 1 ? grown_b : grown_a;
  if (verdict == SNACK_OK && n_prune > 1 && resort && sort_grown(false) != cudaSuccess) verdict = SNACK_ERR_CUDA;
  if (join() != cudaSuccess && verdict == SNACK_OK) verdict = SNACK_ERR_CUDA;
  if (verdict != SNACK_OK) return verdict;
  if (nnz > 0) {
    launch_pdl(k_merge_splits, grid_for(32 * (W.n_merge_tiles + 1), 256), 256, 0, s, surv_pos, n_surv, grown, n_prune,
                                                                              W.n_merge_tiles, part);
    if (col_offs) {  // fork: the column histogram and its scan beside the merge, into the plan, for the
                     // column-view rebuild that follows on the second stream
      SNACK_TRY(cudaEventRecord(a.ev_fork, s));
      SNACK_TRY(cudaStreamWaitEvent(s2, a.ev_fork, 0));
      launch_pdl(k_col_hist, (unsigned)cnb, 256, 0, s2, (const uint64_t *)surv_pos, grown, (const int64_t *)part,
                 W.n_merge_tiles, nnz, cbits, cshift, chist, cnb);
      e = scan_apply<uint32_t>(HistRead{chist}, cnb * kRadixBins, WriteExcl32{coffs}, (uint32_t *)nullptr, stemp2, s2);
      if (e != cudaSuccess) {
        join();
        return SNACK_ERR_CUDA;
      }
    }
    launch_pdl(k_merge<TV>, (unsigned)W.n_merge_tiles, kMergeThreads, 0, s, surv_pos, surv_src, n_surv, grown, n_prune,
               part, cbits, a.out_f, val, a.row_out, a.col_out, reinterpret_cast<TV *>(a.val_out), a.src_out, a.rp_new,
               a.col16_new);
    // the column histogram read the merge's inputs and scanned in the
    // workspace: it is ordered on s before the call returns
    if (col_offs) SNACK_TRY(join());
  }
  SNACK_TRY(cudaGetLastError());
#undef SNACK_TRY
  return SNACK_OK;
}

// ------------------------------------------------------------------------
// Per-row (constant fan-in) restructure: every row prunes its
// p = min(n_per_row, length) smallest (|w|, k) and regrows p columns of the
// same row that were empty, from the row's own draw stream
// (base_r = mix(seed ^ mix(step ^ r*K))), so row counts and offsets do not
// change.  One warp per row:
//  1. radix select of the row's p-th smallest magnitude key (four 8-bit
//     digits, a 256-bin histogram per warp) and the number of ties to prune;
//  2. draws in groups of 32: a draw is a candidate when its column was empty
//     in the row (binary search) and is not yet accepted; the first
//     occurrence in the group (match_any) in draw order is accepted until p;
//  3. the accepted columns are sorted (bitonic, shared memory), each with
//     the number of old entries left of it;
//  4. one pass over the row: survivor s lands at s + (grown columns left of
//     it), the pruned columns are listed; regrown g lands at
//     g + (old entries left of it) - (pruned entries left of it).

constexpr int kRowsWarps = 8;
constexpr int kRowsMaxPrune = 256;  // per row
constexpr uint64_t kRowStreamK = 0xD1B54A32D192ED03ull;

struct RowsArgs {
  const int32_t *rp, *col;
  const void *val;
  int32_t out_f, in_f, n_per_row;
  uint64_t seed, step;
  int64_t max_draws;
  int32_t *row_out, *col_out;
  void *val_out;
  int32_t *src_out;
  uint16_t *col16;
  uint32_t *err;  // bit 0: a row has fewer empty columns than it prunes; bit 1: a row ran out of draws
};

// one warp: the digit d of hist (256 bins) where the running count reaches
// rank rem (1-based), and the count below d
__device__ void warp_pick256(const uint32_t *hist, uint32_t rem, uint32_t *digit, uint32_t *before) {
  const int lane = threadIdx.x & 31;
  uint32_t h[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = hist[lane * 8 + i];
    sum += h[i];
  }
  uint32_t inc = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += u;
  }
  const uint32_t ex = inc - sum;
  const unsigned hit = __ballot_sync(0xffffffffu, inc >= rem && ex < rem);
  const int src = hit ? __ffs(hit) - 1 : 31;
  uint32_t dg = 255, bf = 0;
  if (lane == src) {
    uint32_t c = ex;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      if (c + h[i] >= rem) {
        dg = lane * 8 + i;
        bf = c;
        break;
      }
      c += h[i];
    }
  }
  *digit = __shfl_sync(0xffffffffu, dg, src);
  *before = __shfl_sync(0xffffffffu, bf, src);
}

// first index in a[0..n) with a[i] >= v (a ascending)
template <typename P>
__device__ __forceinline__ int lower_bound_by(P at, int n, uint32_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (at(mid) < v)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

template <typename TV>
__global__ void __launch_bounds__(kRowsWarps * 32) k_restructure_rows(RowsArgs A) {
  pdl_wait();
  __shared__ uint32_t s_hist[kRowsWarps][256];
  __shared__ uint32_t s_gcol[kRowsWarps][kRowsMaxPrune];
  __shared__ uint32_t s_glb[kRowsWarps][kRowsMaxPrune];
  __shared__ uint32_t s_pcol[kRowsWarps][kRowsMaxPrune];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r = blockIdx.x * kRowsWarps + w;
  if (r >= A.out_f) return;
  const unsigned full = 0xffffffffu, lt = (1u << lane) - 1u;
  const TV *val = reinterpret_cast<const TV *>(A.val);
  TV *val_out = reinterpret_cast<TV *>(A.val_out);
  const int64_t k0 = A.rp[r];
  const int L = (int)(A.rp[r + 1] - k0);
  const int p = A.n_per_row < L ? A.n_per_row : L;
  if (p > A.in_f - L) {
    if (lane == 0) atomicOr(A.err, 1u);
    return;
  }
  const int32_t *crow = A.col + k0;
  uint32_t *hist = s_hist[w], *gcol = s_gcol[w], *glb = s_glb[w], *pcol = s_pcol[w];

  // 1. threshold key t of rank p and the ties to prune
  uint32_t t = 0, remaining = 0;
  if (p > 0) {
    uint32_t pfx = 0, mask = 0, rem = (uint32_t)p;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
#pragma unroll
      for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0;
      __syncwarp();
      for (int j = lane; j < L; j += 32) {
        const uint32_t key = mag_key<TV>(val, k0 + j);
        if ((key & mask) == pfx) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
      }
      __syncwarp();
      uint32_t d, before;
      warp_pick256(hist, rem, &d, &before);
      pfx |= d << shift;
      mask |= 0xFFu << shift;
      rem -= before;
      __syncwarp();
    }
    t = pfx;
    remaining = rem;
  }

  // 2. regrow draws, groups of 32 in draw order
  int n_acc = 0;
  if (p > 0) {
    const uint64_t base = sm64_finalise(A.seed ^ sm64_finalise(A.step ^ ((uint64_t)r * kRowStreamK)));
    for (int64_t i0 = 0; n_acc < p; i0 += 32) {
      if (i0 >= A.max_draws) {
        if (lane == 0) atomicOr(A.err, 2u);
        return;
      }
      const int64_t i = i0 + lane;
      const uint64_t u = sm64_finalise(base + ((uint64_t)i + 1) * kGolden);
      const uint32_t c = (uint32_t)__umul64hi(u, (uint64_t)A.in_f);
      const int lb = lower_bound_by([&](int m) { return (uint32_t)crow[m]; }, L, c);
      bool cand = i < A.max_draws && !(lb < L && (uint32_t)crow[lb] == c);
      for (int a = 0; cand && a < n_acc; ++a) cand = gcol[a] != c;
      const unsigned peers = __match_any_sync(full, cand ? c : (0x80000000u | (uint32_t)lane));
      const bool first = cand && (__ffs(peers) - 1) == lane;
      const unsigned bal = __ballot_sync(full, first);
      const int rank = __popc(bal & lt);
      if (first && n_acc + rank < p) {
        gcol[n_acc + rank] = c;
        glb[n_acc + rank] = (uint32_t)lb;
      }
      n_acc = min(p, n_acc + __popc(bal));
      __syncwarp();
    }
    // 3. sort the accepted columns (and their left counts) ascending
    int n2 = 1;
    while (n2 < p) n2 <<= 1;
    for (int q = p + lane; q < n2; q += 32) {
      gcol[q] = 0xFFFFFFFFu;
      glb[q] = 0;
    }
    __syncwarp();
    for (int size = 2; size <= n2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int q = lane; q < n2; q += 32) {
          const int o = q ^ stride;
          if (o > q) {
            const bool up = (q & size) == 0;
            const uint32_t a = gcol[q], b = gcol[o];
            if ((a > b) == up) {
              gcol[q] = b;
              gcol[o] = a;
              const uint32_t x = glb[q];
              glb[q] = glb[o];
              glb[o] = x;
            }
          }
        }
        __syncwarp();
      }
    }
  }

  // 4. survivors in storage order; the pruned columns are listed in order
  uint32_t carry_eq = 0, carry_keep = 0, n_pr = 0;
  for (int j0 = 0; j0 < L; j0 += 32) {
    const int j = j0 + lane;
    const bool in = j < L;
    const uint32_t key = in ? mag_key<TV>(val, k0 + j) : 0u;
    const uint32_t c = in ? (uint32_t)crow[j] : 0u;
    const bool eq = in && p > 0 && key == t;
    const unsigned eqb = __ballot_sync(full, eq);
    const uint32_t eq_rank = carry_eq + __popc(eqb & lt);
    const bool keep = in && (p == 0 || key > t || (eq && eq_rank >= remaining));
    const unsigned kb = __ballot_sync(full, keep), pb = __ballot_sync(full, in && !keep);
    const uint32_t pos =
        keep ? carry_keep + __popc(kb & lt) + (uint32_t)lower_bound_by([&](int m) { return gcol[m]; }, p, c) : 0u;
    if (keep && pos < (uint32_t)L) {  // always true; the test keeps every store inside the row
      const int64_t o = k0 + pos;
      A.row_out[o] = r;
      A.col_out[o] = (int32_t)c;
      val_out[o] = val[k0 + j];
      if (A.src_out) A.src_out[o] = (int32_t)(k0 + j);
      if (A.col16) A.col16[o] = (uint16_t)c;
    } else if (in && !keep && n_pr + __popc(pb & lt) < (uint32_t)kRowsMaxPrune) {
      pcol[n_pr + __popc(pb & lt)] = c;
    }
    carry_eq += __popc(eqb);
    carry_keep += __popc(kb);
    n_pr += __popc(pb);
  }
  __syncwarp();
  // 5. regrown entries
  for (int g = lane; g < p; g += 32) {
    const uint32_t c = gcol[g];
    const int pl = lower_bound_by([&](int m) { return pcol[m]; }, (int)min(n_pr, (uint32_t)kRowsMaxPrune), c);
    const int64_t off = g + (int64_t)glb[g] - pl;
    if (off < 0 || off >= L) continue;  // never; keeps every store inside the row
    const int64_t o = k0 + off;
    A.row_out[o] = r;
    A.col_out[o] = (int32_t)c;
    val_out[o] = from_f32<TV>(0.f);
    if (A.src_out) A.src_out[o] = -1;
    if (A.col16) A.col16[o] = (uint16_t)c;
  }
}

}  // namespace

// The restructure's own scratch, or the plan rebuild's when that is larger
// (the rebuild runs on the caller's stream for layers whose column view is
// not rebuilt on the second stream).
size_t restructure_ws_bytes(int32_t out_f, int32_t in_f, int64_t nnz, int64_t n_prune) {
  size_t r = rws_layout(out_f, in_f, nnz, n_prune).total;
  size_t p = plan_build_ws_bytes(out_f, in_f, nnz);
  return align_up(r > p ? r : p, kAlign);
}

snack_status run_restructure_rows(const RowsRestructureArgs &a, cudaStream_t s) {
  if (a.n_per_row > kRowsMaxPrune || a.in_f > 65536) return SNACK_ERR_UNSUPPORTED;
  RowsArgs A;
  A.rp = a.rp;
  A.col = a.col;
  A.val = a.val;
  A.out_f = a.out_f;
  A.in_f = a.in_f;
  A.n_per_row = (int32_t)a.n_per_row;
  A.seed = a.seed;
  A.step = a.step;
  A.max_draws = 64 * (int64_t)a.n_per_row + (1 << 20);
  A.row_out = a.row_out;
  A.col_out = a.col_out;
  A.val_out = a.val_out;
  A.src_out = a.src_out;
  A.col16 = a.col16;
  A.err = a.err;
  if (cudaMemsetAsync(a.err, 0, sizeof(uint32_t), s) != cudaSuccess) return SNACK_ERR_CUDA;
  const unsigned grid = (unsigned)((a.out_f + kRowsWarps - 1) / kRowsWarps);
  if (a.val_t == SNACK_BF16)
    launch_pdl(k_restructure_rows<bf16>, grid, kRowsWarps * 32, 0, s, A);
  else
    launch_pdl(k_restructure_rows<float>, grid, kRowsWarps * 32, 0, s, A);
  if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  return SNACK_OK;
}

snack_status run_restructure(const RestructureArgs &a, void *ws, size_t ws_bytes, cudaStream_t s) {
  if (a.val_t == SNACK_BF16) return restructure_impl<bf16>(a, ws, ws_bytes, s);
  return restructure_impl<float>(a, ws, ws_bytes, s);
}

}  // namespace snack
