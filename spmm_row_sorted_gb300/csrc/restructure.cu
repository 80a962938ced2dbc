// Dynamic Sparse Training restructure on the GPU (prune smallest |w|, regrow
// at random empty positions with value +0, re-sort the COO).
//
//  1. prune set (on the handle's second stream, of the lowest priority,
//     beside step 2): radix select (digits of 11, 10 and 10 bits, high to low) of
//     the n_prune-th smallest magnitude key t; ties at t are pruned in
//     storage order, so the pruned set is exactly the n_prune smallest
//     (|w|, k); one more pass counts, per tile of stored weights, those above
//     t and those equal to it;
//  2. regrow, on the caller's stream beside step 1: draws i of
//     SplitMix64 map to positions by multiply-high; a draw is a candidate when
//     the position was empty (binary search in its old row), and is accepted
//     when it is the first draw of its position -- a hash table keeps the
//     minimum draw index per position (atomicMin, so the outcome does not
//     depend on thread order); a scan over draw order keeps the first n_prune
//     accepted and drops each into an equal-width bucket of the position range
//     (and, when the column view is updated, of the column-major range); one
//     warp per bucket ranks its positions, giving the regrown positions sorted
//     in row order (and in column order);
//  3. one pass merges the survivors with the regrown positions: tile t of the
//     stored weights owns the regrown positions from its first key up to the
//     next tile's, so a survivor lands at (survivors before it) + (regrown
//     below it) and a regrown position at (its rank) + (survivors below it);
//     the same pass writes the row offsets and the 16-bit columns;
//  4. the column view is updated the same way on the handle's lowest-priority
//     stream after the call returns: the current view's kept entries (column order) merged with
//     the regrown positions in column order, into the plan's second view.
// Steps 3 and 4 are queued before the host has read how many draws the first
// chunk accepted, behind a device flag that step 2 sets only when the chunk
// sufficed; when it did not (rare: more draws are needed, or a bucket ran
// over) the flagged passes write nothing, and the host queues the remaining
// draws, a general sort and the passes again.
// Every step is integer work, so the output is bit-exact with the sequential
// definition.
#include <math.h>

#include "internal.hpp"
#include "prims.cuh"

namespace snack {

namespace {

constexpr uint64_t kEmpty = ~0ull;

// Decoupled look-back, by one full warp, for tile b of a pass whose tiles are
// taken in ticket order (every earlier tile has a block running): publish the
// tile's total `agg` (a 62-bit value whose fields add without carries), add up
// the predecessors' published values going back from the nearest, 32 at a
// time, until one that includes everything before it, publish b's inclusive
// total and return the exclusive one (in every lane).  Words: flag in bits
// 62..63 (1: the tile's own total, 2: everything up to it), value below.
// Every wait is bounded: after kLbMaxSpins polls *err is set and the sum so
// far is returned.
constexpr uint64_t kLbAggregate = 1ull << 62, kLbInclusive = 2ull << 62, kLbValue = (1ull << 62) - 1;
constexpr uint32_t kLbMaxSpins = 1u << 20;  // about 0.1 s of polling

__device__ uint64_t look_back(uint64_t *status, int64_t b, uint64_t agg, uint32_t *err) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) *reinterpret_cast<volatile uint64_t *>(&status[b]) = (b == 0 ? kLbInclusive : kLbAggregate) | agg;
  uint64_t excl = 0;
  int64_t i = b - 1;
  uint32_t spins = 0;
  while (i >= 0) {
    const int64_t idx = i - lane;
    const uint64_t v = idx >= 0 ? *reinterpret_cast<const volatile uint64_t *>(&status[idx]) : kLbInclusive;
    const unsigned incl = __ballot_sync(0xffffffffu, (v >> 62) == 2u);
    const int first = incl ? __ffs(incl) - 1 : 31;
    const unsigned upto = first == 31 ? 0xffffffffu : ((2u << first) - 1u);  // lanes 0 .. first
    const unsigned missing = __ballot_sync(0xffffffffu, (v >> 62) == 0u) & upto;
    if (missing) {
      if (++spins > kLbMaxSpins) {
        if (lane == 0) atomicOr(err, 1u);
        break;
      }
      __nanosleep(64);
      continue;
    }
    uint64_t val = (unsigned)lane <= (unsigned)first ? (v & kLbValue) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) val += __shfl_down_sync(0xffffffffu, val, o);
    excl += __shfl_sync(0xffffffffu, val, 0);
    if (incl) break;
    i -= 32;
  }
  if (lane == 0 && b > 0) *reinterpret_cast<volatile uint64_t *>(&status[b]) = kLbInclusive | ((excl + agg) & kLbValue);
  return excl;
}

struct SelState {
  uint32_t prefix, remaining, n_prune, total;  // prefix = threshold key t, remaining = ties to prune
  uint32_t overflow;                           // a draw found the position table full
  uint32_t pfx, mask, rem;                     // select progress: digits fixed so far, ranks left within them
  uint32_t arrive[4];                          // blocks finished per pass
  uint32_t n_cand;                             // keys in the first digit's bucket (the candidates)
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
    st->n_cand = 0;
  }
}

// Second pass of the two-pass select, one block per scan tile (2048 stored
// weights): the tile's keys above the first digit's bucket are counted (its
// keep count so far, sums[t]), and the keys in the bucket are listed as
// candidates, key << 32 | storage index (one list append per block).
template <typename TV>
__global__ void __launch_bounds__(kScanThreads) k_sel_bucket(const TV *__restrict__ val, int64_t nnz, SelState *st,
                                                             uint64_t *__restrict__ sums, uint64_t *__restrict__ cand) {
  pdl_wait();
  __shared__ uint32_t s_above[kScanThreads / 32], s_cnt[kScanThreads / 32];
  __shared__ uint32_t s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = (int64_t)blockIdx.x * kScanTile;
  const uint32_t d0 = st->pfx >> 20;
  uint32_t key[kScanItems];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t k = base + i * kScanThreads + tid;
    key[i] = k < nnz ? mag_key<TV>(val, k) : 0u;
  }
  uint32_t n_above = 0, n_mine = 0;
  unsigned bal[kScanItems];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t k = base + i * kScanThreads + tid;
    const bool in = k < nnz;
    n_above += in && (key[i] >> 20) > d0 ? 1u : 0u;
    bal[i] = __ballot_sync(0xffffffffu, in && (key[i] >> 20) == d0);
    n_mine += (uint32_t)__popc(bal[i]);  // the warp's candidates (same in every lane)
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n_above += __shfl_down_sync(0xffffffffu, n_above, o);
  if (lane == 0) {
    s_above[warp] = n_above;
    s_cnt[warp] = n_mine;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t ta = 0, tc = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) {
      ta += s_above[w];
      const uint32_t c = s_cnt[w];
      s_cnt[w] = tc;  // the warp's first slot within the block's run
      tc += c;
    }
    sums[blockIdx.x] = ta;
    s_base = tc ? atomicAdd(&st->n_cand, tc) : 0u;
  }
  __syncthreads();
  uint32_t at = s_base + s_cnt[warp];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if ((bal[i] >> lane) & 1u)
      cand[at + __popc(bal[i] & ((1u << lane) - 1u))] = ((uint64_t)key[i] << 32) | (uint32_t)(base + i * kScanThreads + tid);
    at += (uint32_t)__popc(bal[i]);
  }
}

// A digit pass of the select over the candidate list (bits 19..10, then
// 9..0, of the keys matching the digits fixed so far): per-block histograms
// (equal bins of a warp added once), added to the global one; the last block
// to finish picks the digit that holds rank rem (as the first pass does).
constexpr int kSelCandBlocks = 304;
template <int kPass>
__global__ void __launch_bounds__(256) k_sel_cand(const uint64_t *__restrict__ cand, SelState *st) {
  pdl_wait();
  constexpr int kShift = kPass == 1 ? 10 : 0, kBins = 1024, kPer = kBins / 256;
  __shared__ uint32_t h[kBins];
  __shared__ uint32_t s_scan[256];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t nc = st->n_cand, pfx = st->pfx, mask = st->mask;
  for (int i = tid; i < kBins; i += 256) h[i] = 0u;
  __syncthreads();
  const uint32_t stride = gridDim.x * 256u;
  for (uint32_t i0 = blockIdx.x * 256u; i0 < nc; i0 += stride) {  // whole warps per round (ballots below)
    const uint32_t i = i0 + tid;
    const uint32_t key = i < nc ? (uint32_t)(cand[i] >> 32) : 0u;
    const bool on = i < nc && (key & mask) == pfx;
    const uint32_t bin = on ? (key >> kShift) & (kBins - 1) : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (on && (peers & ((1u << lane) - 1u)) == 0u) atomicAdd(&h[bin], (uint32_t)__popc(peers));
  }
  __syncthreads();
  uint32_t *gh = kPass == 1 ? st->hist1 : st->hist2;
  for (int i = tid; i < kBins; i += 256)
    if (h[i]) atomicAdd(&gh[i], h[i]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&st->arrive[kPass], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const uint32_t rem = st->rem;
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    c[j] = __ldcg(&gh[tid * kPer + j]);
    sum += c[j];
  }
  s_scan[tid] = sum;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    const uint32_t v = tid >= off ? s_scan[tid - off] : 0u;
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
        st->pfx = pfx | (d << kShift);
        st->mask = mask | ((uint32_t)(kBins - 1) << kShift);
        st->rem = rem - ex;
        if (kPass == 2) {
          st->prefix = pfx | (d << kShift);
          st->remaining = rem - ex;
        }
        break;
      }
      ex += c[j];
    }
  }
}

// The tiles' keep counts: each candidate above the threshold t adds one kept
// weight to its tile, each equal to t one tie.  Candidates were listed a
// tile at a time, so a warp's lanes of one tile add their counts at once.
__global__ void __launch_bounds__(256) k_sel_tiles(const uint64_t *__restrict__ cand, const SelState *st,
                                                   uint64_t *__restrict__ sums) {
  pdl_wait();
  const uint32_t nc = st->n_cand, t = st->prefix;
  const int lane = threadIdx.x & 31;
  const uint32_t stride = gridDim.x * 256u;
  for (uint32_t i0 = blockIdx.x * 256u; i0 < nc; i0 += stride) {  // whole warps per round (ballots below)
    const uint32_t i = i0 + threadIdx.x;
    uint32_t key = 0, tile = 0xFFFFFFFFu;
    if (i < nc) {
      const uint64_t cw = cand[i];
      key = (uint32_t)(cw >> 32);
      tile = (uint32_t)cw / kScanTile;
    }
    const bool gt = i < nc && key > t, eq = i < nc && key == t;
    const unsigned gtm = __ballot_sync(0xffffffffu, gt), eqm = __ballot_sync(0xffffffffu, eq);
    const unsigned peers = __match_any_sync(0xffffffffu, (gt || eq) ? tile : 0xFFFFFFFFu);
    if ((gt || eq) && (peers & ((1u << lane) - 1u)) == 0u) {
      const uint64_t add = (uint64_t)__popc(peers & gtm) | ((uint64_t)__popc(peers & eqm) << 32);
      atomicAdd(reinterpret_cast<unsigned long long *>(&sums[tile]), add);
    }
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


// Position table: the first (smallest) draw index of every drawn empty
// position, open addressing with linear probing.  Packed (positions below
// 2^32): one 64-bit word per slot, position << 32 | draw index, so a first
// insertion is one compare-and-swap and a repeat one atomicMin on the same
// word; otherwise 64-bit positions and 32-bit minima in two arrays.
struct PosTable {
  uint64_t *keys;
  uint32_t *mins;  // unused when packed
  uint64_t mask;
  bool packed;
  __device__ bool insert(uint64_t key, uint32_t i) const {
    uint64_t h = sm64_finalise(key) & mask;
    if (packed) {
      const unsigned long long w = (key << 32) | i;  // never kEmpty: i < 2^32 - 1
      for (uint64_t probe = 0; probe <= mask; ++probe) {
        const unsigned long long prev =
            atomicCAS(reinterpret_cast<unsigned long long *>(keys + h), (unsigned long long)kEmpty, w);
        if (prev == kEmpty) return true;
        if ((prev >> 32) == key) {
          atomicMin(reinterpret_cast<unsigned long long *>(keys + h), w);
          return true;
        }
        h = (h + 1) & mask;
      }
      return false;
    }
    for (uint64_t probe = 0; probe <= mask; ++probe) {
      const unsigned long long prev = atomicCAS(reinterpret_cast<unsigned long long *>(keys + h),
                                                (unsigned long long)kEmpty, (unsigned long long)key);
      if (prev == kEmpty || prev == key) {
        atomicMin(mins + h, i);
        return true;
      }
      h = (h + 1) & mask;
    }
    return false;
  }
  __device__ uint64_t home(uint64_t key) const { return sm64_finalise(key) & mask; }
  // the smallest draw index recorded for key, probing from slot h whose word is k
  __device__ uint32_t min_from(uint64_t key, uint64_t h, uint64_t k) const {
    for (uint64_t probe = 0; probe <= mask; ++probe) {
      if (k == kEmpty) return 0xFFFFFFFFu;
      if (packed) {
        if ((k >> 32) == key) return (uint32_t)k;
      } else if (k == key) {
        return mins[h];
      }
      h = (h + 1) & mask;
      k = keys[h];
    }
    return 0xFFFFFFFFu;
  }
};

__device__ __forceinline__ uint32_t mag_of(float v) { return canon_mag(__float_as_uint(v) & 0x7FFFFFFFu); }
__device__ __forceinline__ uint32_t mag_of(bf16 v) {
  return canon_mag(((uint32_t)__bfloat16_as_ushort(v) & 0x7FFFu) << 16);
}

// A draw: position by multiply-high of SplitMix64 output i; empty test by a
// binary search of its column in the old row, over the plan's 16-bit column
// copy or the 32-bit columns (CI); insertion into the position table.
template <typename CI>
__global__ void k_draw(uint64_t base, uint64_t i0, int64_t m, uint64_t n_pos, int32_t in_f, int cbits,
                       const int32_t *__restrict__ rp, const CI *__restrict__ col, uint64_t *__restrict__ cand,
                       PosTable tab, uint32_t *overflow) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < m; idx += stride) {
    const uint64_t i = i0 + (uint64_t)idx;
    const uint64_t u = sm64_finalise(base + (i + 1) * kGolden);
    const uint64_t p = __umul64hi(u, n_pos);
    const uint64_t r = p / (uint64_t)in_f;
    const int32_t c = (int32_t)(p - r * (uint64_t)in_f);
    int32_t lo = rp[r], hi = rp[r + 1];
    const int32_t end = hi;
    while (lo < hi) {
      const int32_t mid = lo + (hi - lo) / 2;
      if ((int32_t)col[mid] < c)
        lo = mid + 1;
      else
        hi = mid;
    }
    const bool member = lo < end && (int32_t)col[lo] == c;
    if (member) {
      cand[idx] = kEmpty;
      continue;
    }
    const uint64_t key = (r << cbits) | (uint32_t)c;  // position key of the draw
    cand[idx] = key;
    if (!tab.insert(key, (uint32_t)i)) atomicOr(overflow, 1u);
  }
}

constexpr int kBktTarget = 64;               // positions expected per bucket
constexpr int kBktCap = 256;                 // slots per bucket
constexpr uint32_t kBktMaxBuckets = 16384;   // more buckets: the regrown positions take the general sort

// Equal-width buckets of a key range, filled in any order (atomic slots);
// each key keeps its acceptance rank.  The bucket of a key is the high word
// of key * mult, mult = floor(2^64 * nb / range): monotone in the key and
// below nb.  Counters sit one per 32-byte sector (kCntStride words apart), so
// the atomics on neighbouring buckets do not queue on one sector.
constexpr int kCntStride = 8;
struct BucketSet {
  uint32_t *cnt;  // [nb * kCntStride] keys dropped per bucket
  uint64_t *key;  // [nb][kBktCap]
  uint32_t *q;    // [nb][kBktCap]
  uint64_t mult;
  uint32_t nb;    // 0: not used
  __device__ uint32_t count(uint32_t b) const { return min(__ldg(&cnt[(size_t)b * kCntStride]), (uint32_t)kBktCap); }
  __device__ void place(uint64_t k, uint32_t qq, uint32_t *ovf) const {
    const uint32_t b = (uint32_t)__umul64hi(k, mult);
    const uint32_t slot = atomicAdd(&cnt[(size_t)b * kCntStride], 1u);
    if (slot < (uint32_t)kBktCap) {
      key[(size_t)b * kBktCap + slot] = k;
      q[(size_t)b * kBktCap + slot] = qq;
    } else {
      atomicOr(ovf, 1u);
    }
  }
};

uint64_t bucket_mult(uint32_t nb, uint64_t range) {
  const unsigned __int128 m = ((unsigned __int128)nb << 64) / (unsigned __int128)range;
  return m >> 64 ? ~0ull : (uint64_t)m;
}

// column-major key col << rbits | row of a row-major key row << cbits | col
__device__ __forceinline__ uint64_t col_major(uint64_t p, int cbits, int rbits) {
  return ((p & ((1ull << cbits) - 1ull)) << rbits) | (p >> cbits);
}

// Counters of the regrow branch (it runs beside the select, which has a stream of its own).
struct DrawState {
  uint32_t total, overflow;  // accepted draws of the last chunk; a draw found the position table full
  uint32_t bucket_overflow;  // a row-order bucket of the regrown positions ran out of slots
  uint32_t col_overflow;     // a column-order bucket did
  uint32_t lb_fail;          // the acceptance scan gave up waiting for a predecessor tile (never expected)
  uint32_t lists_ok;         // the row-order list is complete: the merge may write
};

// The lists' verdict (the column-order one into the plan word col_ok) and,
// with host_words, the chunk's counters to the host's mapped words.
__device__ __forceinline__ void publish(DrawState *ds, int64_t n_prune, uint32_t *host_words, bool made,
                                        uint32_t *col_ok) {
  const uint32_t tot = ds->total, ovf = ds->overflow, bovf = ds->bucket_overflow, covf = ds->col_overflow;
  const uint32_t lbf = ds->lb_fail;
  if (host_words) {
    volatile uint32_t *hw = host_words;
    hw[0] = tot;
    hw[1] = ovf;
    hw[2] = bovf;
    hw[3] = covf;
    hw[4] = lbf;
  }
  const bool ok = made && (int64_t)tot >= n_prune && !ovf && !bovf && !lbf;
  ds->lists_ok = ok ? 1u : 0u;
  *col_ok = ok && !covf ? 1u : 0u;
}

__global__ void k_publish(DrawState *ds, int64_t n_prune, uint32_t *host_words, int made, uint32_t *col_ok) {
  pdl_wait();
  publish(ds, n_prune, host_words, made != 0, col_ok);
}

__global__ void k_set_word(uint32_t *w, uint32_t v) {
  pdl_wait();
  *w = v;
}

// Start of a restructure's regrow branch: counters, bucket counts and the
// column-view update's pruned counts per column to zero, the position table
// to empty (one launch instead of several fills).
__global__ void k_rs_init(DrawState *ds, PosTable tab, uint32_t *__restrict__ bcnt, int64_t nb,
                          uint64_t *__restrict__ lb_status, int64_t n_lb, uint32_t *lb_ticket,
                          uint32_t *__restrict__ pcnt, int64_t n_pc, uint32_t *col_ok) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 == 0) {
    ds->total = 0u;
    ds->overflow = 0u;
    ds->bucket_overflow = 0u;
    ds->col_overflow = 0u;
    ds->lb_fail = 0u;
    ds->lists_ok = 0u;
    *col_ok = 0u;
    *lb_ticket = 0u;
  }
  // 16-byte stores: the table (a power of two of at least 16 slots) and the
  // bucket counts (a multiple of 16 words) start on 16-byte boundaries
  const int64_t cap = (int64_t)tab.mask + 1;
  const uint4 ones = make_uint4(~0u, ~0u, ~0u, ~0u), zeros = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = i0; i < cap / 2; i += stride) reinterpret_cast<uint4 *>(tab.keys)[i] = ones;
  if (!tab.packed)
    for (int64_t i = i0; i < cap / 4; i += stride) reinterpret_cast<uint4 *>(tab.mins)[i] = ones;
  for (int64_t i = i0; i < nb / 4; i += stride) reinterpret_cast<uint4 *>(bcnt)[i] = zeros;
  for (int64_t i = (nb / 4) * 4 + i0; i < nb; i += stride) bcnt[i] = 0u;
  for (int64_t i = i0; i < n_lb; i += stride) lb_status[i] = 0ull;
  for (int64_t i = i0; i < n_pc; i += stride) pcnt[i] = 0u;
}

// The acceptance scan's block: a scan tile of draws over 1024 threads, two
// per thread (its phases are dependent round trips; more warps per tile keep
// more of them in flight).
constexpr int kAccThreads = 1024, kAccItems = kScanTile / kAccThreads;
static_assert(kAccItems * kAccThreads == kScanTile, "one acceptance block per scan tile");

// Acceptance of a draw chunk, its scan over draw order and (first chunk) the
// bucket placement of the regrown positions, in one pass: tiles of kScanTile
// draws taken in ticket order.  A block flags its tile's draws (an empty
// position, and that position's first draw), scans the flags, learns the
// accepted draws before its tile by look-back, and writes the first n_prune
// accepted positions in draw order: grown[q] for acceptance rank q, and
// (key, q) into the position's row-order bucket and, for the column-view
// update, (col << rbits | row, q) into its column-order bucket.  The last
// tile's block writes the chunk's accepted count.
struct AcceptArgs {
  const uint64_t *cand;
  int64_t m;
  uint64_t i0;
  PosTable tab;
  uint64_t *grown;
  int64_t before, n_prune;
  BucketSet br;  // br.nb == 0: no placement (chunks after the first)
  uint32_t *bovf;
  BucketSet bc;  // bc.nb == 0: no column-order placement
  uint32_t *covf;
  int cbits, rbits;
  uint64_t *status;  // [tiles], zero before the launch
  uint32_t *ticket;  // zero before the launch
  uint32_t *err;
  uint32_t *total;
};

__global__ void __launch_bounds__(kAccThreads) k_accept_scan(AcceptArgs a) {
  constexpr int kPadded = kScanTile + kScanTile / 32 + 1;
  __shared__ uint32_t sF[kPadded];  // flags, then exclusive counts (one pad word per 32)
  __shared__ int64_t s_tile;
  __shared__ uint32_t s_tot;
  __shared__ uint64_t s_pre;
  auto pad = [](int e) { return e + (e >> 5); };
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_tile = atomicAdd(a.ticket, 1u);
  __syncthreads();
  const int64_t t = s_tile, base = t * kScanTile;
  uint64_t p[kAccItems], h[kAccItems], w[kAccItems];
#pragma unroll
  for (int i = 0; i < kAccItems; ++i) {
    const int64_t idx = base + i * kAccThreads + tid;
    p[i] = idx < a.m ? a.cand[idx] : kEmpty;
  }
#pragma unroll
  for (int i = 0; i < kAccItems; ++i) {  // every item's first probe in flight at once
    h[i] = a.tab.home(p[i]);
    w[i] = p[i] != kEmpty ? a.tab.keys[h[i]] : kEmpty;
  }
  uint32_t f[kAccItems];
#pragma unroll
  for (int i = 0; i < kAccItems; ++i) {
    const int64_t idx = base + i * kAccThreads + tid;
    f[i] = p[i] != kEmpty && a.tab.min_from(p[i], h[i], w[i]) == (uint32_t)(a.i0 + (uint64_t)idx) ? 1u : 0u;
    sF[pad(i * kAccThreads + tid)] = f[i];
  }
  __syncthreads();
  {
    uint32_t v[kAccItems], tsum = 0;
#pragma unroll
    for (int i = 0; i < kAccItems; ++i) {
      v[i] = sF[pad(tid * kAccItems + i)];
      tsum += v[i];
    }
    uint32_t ex = block_exclusive_scan<uint32_t, kAccThreads>(tsum, &s_tot);
#pragma unroll
    for (int i = 0; i < kAccItems; ++i) {
      sF[pad(tid * kAccItems + i)] = ex;
      ex += v[i];
    }
  }
  if (warp == 0) {  // accepted draws of the tiles before this one
    const uint64_t excl = look_back(a.status, t, s_tot, a.err);
    if (lane == 0) {
      s_pre = excl;
      if (t == ceil_div(a.m, kScanTile) - 1) *a.total = (uint32_t)(excl + s_tot);
    }
  }
  __syncthreads();
  int64_t q[kAccItems];
  bool put[kAccItems];
#pragma unroll
  for (int i = 0; i < kAccItems; ++i) {
    q[i] = a.before + (int64_t)s_pre + sF[pad(i * kAccThreads + tid)];
    put[i] = f[i] && q[i] < a.n_prune;
    if (put[i]) a.grown[q[i]] = p[i];
  }
  if (a.br.nb) {  // bucket slots: every atomic in flight before the stores that use them
    const bool col = a.bc.nb != 0;
    uint32_t bk[kAccItems], slot[kAccItems], ck[kAccItems], bkc[kAccItems], slotc[kAccItems];
#pragma unroll
    for (int i = 0; i < kAccItems; ++i) {
      bk[i] = put[i] ? (uint32_t)__umul64hi(p[i], a.br.mult) : 0u;
      slot[i] = put[i] ? atomicAdd(&a.br.cnt[(size_t)bk[i] * kCntStride], 1u) : 0u;
      ck[i] = put[i] && col ? (uint32_t)col_major(p[i], a.cbits, a.rbits) : 0u;
      bkc[i] = put[i] && col ? (uint32_t)__umul64hi((uint64_t)ck[i], a.bc.mult) : 0u;
      slotc[i] = put[i] && col ? atomicAdd(&a.bc.cnt[(size_t)bkc[i] * kCntStride], 1u) : 0u;
    }
#pragma unroll
    for (int i = 0; i < kAccItems; ++i) {
      if (!put[i]) continue;
      if (slot[i] < (uint32_t)kBktCap) {
        a.br.key[(size_t)bk[i] * kBktCap + slot[i]] = p[i];
        a.br.q[(size_t)bk[i] * kBktCap + slot[i]] = (uint32_t)q[i];
      } else {
        atomicOr(a.bovf, 1u);
      }
      if (!col) continue;
      if (slotc[i] < (uint32_t)kBktCap) {
        a.bc.key[(size_t)bkc[i] * kBktCap + slotc[i]] = ck[i];
        a.bc.q[(size_t)bkc[i] * kBktCap + slotc[i]] = (uint32_t)q[i];
      } else {
        atomicOr(a.covf, 1u);
      }
    }
  }
}

struct RankDst {
  uint64_t *key64;  // row order: 64-bit keys, or
  uint32_t *key32;  // column order: 32-bit keys
  uint32_t *q;      // acceptance ranks
};

// The sorted lists from the first chunk's buckets, one warp per bucket: the
// bucket's first slot is the number of keys in the buckets before it (its
// block adds up those counts), and each key lands at its rank among the
// bucket's keys (all distinct).  Blocks [0, nr) rank the row-order buckets
// R, the others the column-order buckets C.  Block 0 first sets the lists'
// verdict (and, with host_words, publishes the chunk's counters); without ds
// there is no verdict to set.  With stop set, the launch writes nothing when
// stop[0] or stop[1] is nonzero.
__global__ void __launch_bounds__(256) k_bkt_rank(BucketSet R, RankDst DR, bool k32r, uint32_t nr, BucketSet C,
                                                  RankDst DC, int64_t n_prune, DrawState *ds, uint32_t *host_words,
                                                  uint32_t *col_ok, const uint32_t *stop) {
  pdl_wait();
  if (stop && (stop[0] | stop[1])) return;
  __shared__ __align__(16) uint64_t sk[8][kBktCap];
  __shared__ uint32_t s_red[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0 && ds) publish(ds, n_prune, host_words, true, col_ok);
  const bool rows = blockIdx.x < nr;
  const BucketSet S = rows ? R : C;
  const RankDst D = rows ? DR : DC;
  const bool k32 = rows ? k32r : true;
  const uint32_t b0 = (rows ? blockIdx.x : blockIdx.x - nr) * 8;
  uint32_t part = 0;
  for (uint32_t i0 = threadIdx.x; i0 < b0; i0 += 256 * 8) {  // eight loads in flight per round
    uint32_t c[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) c[u] = i0 + u * 256 < b0 ? S.count(i0 + u * 256) : 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) part += c[u];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(0xffffffffu, part, o);
  if (lane == 0) s_red[warp] = part;
  __syncthreads();
  uint32_t before = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) before += s_red[w];
  const uint32_t b = b0 + warp;
  if (b >= S.nb) return;
  for (uint32_t w = 0; w < (uint32_t)warp; ++w) before += S.count(b0 + w);
  const uint32_t L = S.count(b);
  const size_t sb = (size_t)b * kBktCap;
  auto put = [&](uint32_t i, uint64_t k, uint32_t r) {
    const int64_t dst = (int64_t)before + r;
    if (dst < n_prune) {  // always, unless a bucket ran over (then the lists are discarded)
      if (D.key64)
        D.key64[dst] = k;
      else
        D.key32[dst] = (uint32_t)k;
      D.q[dst] = S.q[sb + i];
    }
  };
  if (k32) {
    // keys below 2^32: staged as 32-bit words padded with ~0u (never below a
    // key) to a multiple of four; a lane ranks two keys per sweep, reading
    // four staged keys per 16-byte load
    uint32_t *s32 = reinterpret_cast<uint32_t *>(sk[warp]);
    const uint32_t L4 = (L + 3u) & ~3u;
    for (uint32_t i = lane; i < L4; i += 32) s32[i] = i < L ? (uint32_t)S.key[sb + i] : ~0u;
    __syncwarp();
    for (uint32_t i = lane; i < L; i += 64) {
      const bool two = i + 32 < L;
      const uint32_t ka = s32[i], kb = two ? s32[i + 32] : 0u;
      uint32_t ra = 0, rb = 0;
      for (uint32_t j = 0; j < L4; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(s32 + j);
        ra += (v.x < ka ? 1u : 0u) + (v.y < ka ? 1u : 0u) + (v.z < ka ? 1u : 0u) + (v.w < ka ? 1u : 0u);
        rb += (v.x < kb ? 1u : 0u) + (v.y < kb ? 1u : 0u) + (v.z < kb ? 1u : 0u) + (v.w < kb ? 1u : 0u);
      }
      put(i, ka, ra);
      if (two) put(i + 32, kb, rb);
    }
  } else {
    for (uint32_t i = lane; i < L; i += 32) sk[warp][i] = S.key[sb + i];
    __syncwarp();
    for (uint32_t i = lane; i < L; i += 32) {
      const uint64_t k = sk[warp][i];
      uint32_t r = 0;
      for (uint32_t j = 0; j < L; ++j) r += sk[warp][j] < k ? 1u : 0u;
      put(i, k, r);
    }
  }
}

// Sources of the general sort of the regrown positions (acceptance rank as
// the payload): row order, and column order.
struct GrownRowSrc {
  const uint64_t *grown;
  __device__ uint64_t key(int64_t q) const { return grown[q]; }
  __device__ uint32_t val(int64_t q) const { return (uint32_t)q; }
};
struct GrownColSrc {
  const uint64_t *grown;
  int cbits, rbits;
  __device__ uint32_t key(int64_t q) const { return (uint32_t)col_major(grown[q], cbits, rbits); }
  __device__ uint32_t val(int64_t q) const { return (uint32_t)q; }
};

// ---------------------------------------------------------------------------
// Merge of the kept elements of a sorted stream with a sorted list.
//
// The stream holds n elements with strictly increasing keys; each has a
// packed count g | e << 16 (the scan tile sums pack g | e << 32): kept
// (g = 1), or a tie (e = 1) -- the first m ties in stream order are dropped,
// the rest kept.  The list's keys increase strictly and none equals a stream
// key.  Output index of a kept element: (kept elements before it) + (list
// keys below its key); of list entry j: j + (kept elements below it).  Tile
// t of the stream (kMkTile elements) owns the list keys from its first key up
// to the next tile's first key (tile 0 from the start, the last tile to the
// end): every list entry is written by one tile, and a tile's outputs are one
// contiguous range.  Major offsets (rows, or columns): off[M] = outputs whose
// major index (key >> minor_bits) is below M, written by the tile after
// whose element major M starts.
//
// A block loads its tile striped (coalesced), counts each of its list keys
// on the last element below it (a binary search over the tile's keys in
// shared memory), scans the counts blocked (thread t: elements 8t .. 8t+7)
// and writes striped again.

constexpr int kMkThreads = 256, kMkItems = 8, kMkTile = kMkThreads * kMkItems;
static_assert(kMkTile == kScanTile, "a tile's keep counts are one scan tile's sum");
constexpr int kMkListCap = 2048;  // list keys of a tile staged in shared memory
// Tile arrays are read both striped (thread t: t, t + 256, ...) and blocked
// (thread t: 8t .. 8t+7); one pad word per 32 words keeps both free of bank
// conflicts (one 8-byte pad per 16 keys for 64-bit keys).
template <typename K>
__device__ __forceinline__ int kpad(int e) {
  return sizeof(K) == 4 ? e + (e >> 5) : e + (e >> 4);
}
template <typename K>
__host__ __device__ constexpr int kpad_words(int n) {
  return sizeof(K) == 4 ? n + n / 32 + 1 : n + n / 16 + 1;
}
template <typename K>
struct PadKeys {  // sK[e] through the padded index
  K *p;
  __device__ K &operator[](int e) const { return p[kpad<K>(e)]; }
};

// Bounds of tile t: its first key and the list keys below it (tile n_tiles:
// key ~0, every list key), and the policy's notes on the first element (the
// column view: its column, and that column's first entry).
struct MkBound {
  uint64_t key;
  int64_t lo;
  uint32_t aux, aux2;
};
static_assert(sizeof(MkBound) <= 32, "the plan reserves 32 bytes per tile bound");

struct MkArgs {
  int64_t n, n_list;
  int64_t n_out;          // output slots (every index written is checked against it)
  const MkBound *bnd;     // [n_tiles + 1]
  const uint64_t *sums;   // per-tile packed keep counts (kMkDirect), or their exclusive prefixes (kMkGiven)
  const uint32_t *guard;  // when set and zero, every block returns at once
  int minor_bits;
  int64_t n_major;
  int32_t *off;  // [n_major + 1]
  // kMkByColumn: pruned entries in the columns before each column, exclusive
  // prefix (null when nothing is pruned)
  const uint32_t *col_pre;
};

// How a merge block learns the keep counts before its tile: given as
// exclusive prefixes, added up from the per-tile counts, or (the column
// view) its first entry's index less the pruned entries before it, which
// are those of the columns before the tile's first column plus those of
// that column ahead of the tile.
constexpr int kMkGiven = 0, kMkDirect = 1, kMkByColumn = 2;

// number of entries of an ascending sequence at(0..n) below v, by one warp:
// each round probes 32 evenly spaced entries and keeps the bracket of the
// crossing (the probes below v are a prefix)
template <typename F>
__device__ int64_t lb_warp(F at, int64_t n, uint64_t v) {
  const int lane = threadIdx.x & 31;
  int64_t lo = 0, hi = n;  // answer in [lo, hi]
  while (hi - lo > 32) {
    const int64_t span = hi - lo;
    const bool below = at(lo + span * (lane + 1) / 33) < v;  // probes strictly inside [lo, hi)
    const int cnt = __popc(__ballot_sync(0xffffffffu, below));
    const int64_t new_lo = cnt > 0 ? lo + span * cnt / 33 + 1 : lo;
    const int64_t new_hi = cnt < 32 ? lo + span * (cnt + 1) / 33 : hi;
    lo = new_lo;
    hi = new_hi;
  }
  const bool below = lo + lane < hi && at(lo + lane) < v;
  return lo + __popc(__ballot_sync(0xffffffffu, below));
}

// number of entries of an ascending sequence at(0..n) below v
template <typename F, typename V>
__device__ __forceinline__ int lb_seq(F at, int n, V v) {
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

template <class Pol>
constexpr size_t mk_smem_bytes() {
  using K = typename Pol::Key;
  return sizeof(K) * (kpad_words<K>(kMkTile + 1) + kMkListCap) + sizeof(uint64_t) * kpad_words<uint64_t>(kMkTile + 1) +
         sizeof(uint16_t) * kMkListCap + sizeof(typename Pol::Shared);
}

// Exclusive prefix sums pre[c] = cnt[0] + .. + cnt[c - 1], c < n, by one
// block of kScanThreads, kPfxItems consecutive counts per thread a round:
// added up, block-scanned, then read again (from L1) to write the prefixes,
// so no thread holds its counts across the scan.
constexpr int kPfxItems = 64;
__device__ void block_prefix_u32(const uint32_t *cnt, uint32_t *pre, int64_t n) {
  __shared__ uint32_t s_tot;
  uint32_t carry = 0;
  for (int64_t r0 = 0; r0 < n; r0 += (int64_t)kScanThreads * kPfxItems) {
    const int64_t b = r0 + (int64_t)threadIdx.x * kPfxItems;
    const bool whole = b + kPfxItems <= n;  // 16-byte aligned: b is a multiple of kPfxItems
    uint32_t sum = 0;
    if (whole) {
      const uint4 *p = reinterpret_cast<const uint4 *>(cnt + b);
#pragma unroll
      for (int i = 0; i < kPfxItems / 4; ++i) {
        const uint4 q = p[i];
        sum += q.x + q.y + q.z + q.w;
      }
    } else {
      for (int i = 0; i < kPfxItems; ++i) sum += b + i < n ? cnt[b + i] : 0u;
    }
    uint32_t ex = carry + block_exclusive_scan<uint32_t>(sum, &s_tot);
    if (whole) {
      const uint4 *p = reinterpret_cast<const uint4 *>(cnt + b);
      uint4 *o = reinterpret_cast<uint4 *>(pre + b);
#pragma unroll 4
      for (int i = 0; i < kPfxItems / 4; ++i) {
        const uint4 q = p[i];
        uint4 w;
        w.x = ex;
        w.y = w.x + q.x;
        w.z = w.y + q.y;
        w.w = w.z + q.z;
        ex = w.w + q.w;
        o[i] = w;
      }
    } else {
      for (int i = 0; i < kPfxItems && b + i < n; ++i) {
        const uint32_t x = cnt[b + i];
        pre[b + i] = ex;
        ex += x;
      }
    }
    carry += s_tot;
  }
}

// Tile bounds, one warp per tile t in [0, n_tiles], all at once (so the merge
// blocks start with their bounds instead of searching the list themselves);
// with pcnt, one more block (the last) writes the exclusive prefix of the
// n_cols counts pcnt into ppre.
template <class Pol>
__global__ void k_bounds(Pol pol, int64_t n_list, int64_t n_tiles, MkBound *bnd, const uint32_t *pcnt,
                         uint32_t *ppre, int64_t n_cols) {
  pdl_wait();
  if constexpr (Pol::kByColumn) {
    if (pcnt && blockIdx.x == gridDim.x - 1) {
      block_prefix_u32(pcnt, ppre, n_cols);
      return;
    }
  }
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t > n_tiles) return;
  MkBound r{~0ull, n_list, 0u, 0u};
  if (t < n_tiles) {
    r.key = pol.key_at_warp(t * (int64_t)kMkTile, &r.aux);
    r.lo = t == 0 ? 0 : lb_warp([&](int64_t j) { return pol.list_key(j); }, n_list, r.key);
    if constexpr (Pol::kByColumn) r.aux2 = (uint32_t)pol.cp[r.aux];
  }
  if ((threadIdx.x & 31) == 0) bnd[t] = r;
}

// Each element's 64-bit count: bits 0..15 kept (unless a tie), 16..31 tie,
// 32..47 list keys placed right after it.  After the exclusive scan, the
// fields at element e count the kept elements, ties and list keys of the tile
// below e's key (list keys below the tile's first element are counted apart).
template <class Pol, int kMode>
__global__ void __launch_bounds__(kMkThreads, 4) k_merge_kept(Pol pol, MkArgs a) {
  constexpr bool kDirect = kMode == kMkDirect;
  using K = typename Pol::Key;
  extern __shared__ __align__(16) uint8_t mk_smem[];
  uint64_t *sX = reinterpret_cast<uint64_t *>(mk_smem);                    // counts (padded), then exclusive sums
  K *sKp = reinterpret_cast<K *>(sX + kpad_words<uint64_t>(kMkTile + 1));  // tile keys (padded)
  K *sL = sKp + kpad_words<K>(kMkTile + 1);                                // the tile's list keys
  uint16_t *sPj = reinterpret_cast<uint16_t *>(sL + kMkListCap);          // elements below each list key
  typename Pol::Shared &ps = *reinterpret_cast<typename Pol::Shared *>(sPj + kMkListCap);
  const PadKeys<K> sK{sKp};
  __shared__ uint64_t s_pre;
  __shared__ uint64_t s_red[kMkThreads / 32];
  __shared__ uint64_t s_tot;
  __shared__ uint32_t s_c00;
  pdl_wait();
  // every load of the tile's inputs is issued before the first wait on one
  const uint32_t go = a.guard ? *reinterpret_cast<const volatile uint32_t *>(a.guard) : 1u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t b = blockIdx.x;
  const int64_t base = b * (int64_t)kMkTile;
  const int len = (int)(a.n - base < kMkTile ? a.n - base : kMkTile);
  const bool last = b == (int64_t)gridDim.x - 1;
  const MkBound bd0 = a.bnd[b], bd1 = a.bnd[b + 1];
  const uint32_t m = pol.ties_dropped();
  typename Pol::Item it[kMkItems];
  uint32_t fl[kMkItems];
  // (the column view: this thread's share of the pruned entries of the
  // tile's first column ahead of the tile, and those of the columns before)
  uint32_t ahead = pol.load(base, len, last, bd0, bd1.aux, it, fl, sK, ps);
  const uint32_t col_pre = kMode == kMkByColumn && a.col_pre && tid == 0 ? a.col_pre[bd0.aux] : 0u;
  if constexpr (kMode == kMkByColumn) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ahead += __shfl_down_sync(0xffffffffu, ahead, o);
    if (lane == 0) s_red[warp] = ahead;
  }
  const int64_t lo = bd0.lo, cnt = bd1.lo - bd0.lo;
  const bool lsm = cnt <= kMkListCap;
  if (lsm)
    for (int j = tid; j < (int)cnt; j += kMkThreads) sL[j] = (K)pol.list_key(lo + j);
  uint64_t part = 0;
  if (kDirect) {
    for (int64_t q0 = tid; q0 < b; q0 += kMkThreads * 8) {  // eight loads in flight per round
      uint64_t c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = q0 + u * kMkThreads < b ? a.sums[q0 + u * kMkThreads] : 0ull;
#pragma unroll
      for (int u = 0; u < 8; ++u) part += c[u];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(0xffffffffu, part, o);
    if (lane == 0) s_red[warp] = part;
  }
#pragma unroll
  for (int i = 0; i < kMkItems; ++i) {
    const int e = i * kMkThreads + tid;
    sX[kpad<uint64_t>(e)] = fl[i];
  }
  if (go == 0u) return;  // a speculative launch whose lists were not made: write nothing
  if (tid == 0) {
    sK[len] = (K)bd1.key;
    sX[kpad<uint64_t>(kMkTile)] = 0ull;
    s_c00 = 0u;
  }
  __syncthreads();
  if (tid == 0) {
    uint64_t p = 0;
    if (kDirect) {
#pragma unroll
      for (int w = 0; w < kMkThreads / 32; ++w) p += s_red[w];
    } else if (kMode == kMkByColumn) {  // kept entries before the tile (no ties in this order)
      uint32_t np = col_pre;
#pragma unroll
      for (int w = 0; w < kMkThreads / 32; ++w) np += s_red[w];
      p = (uint64_t)((uint32_t)base - np);
    } else {
      p = a.sums[b];
    }
    s_pre = p;
  }
  if (pol.keys_blocked(base, len, last, bd0.aux, bd1.aux, sK, ps)) __syncthreads();
  auto lkey = [&](int j) -> K { return lsm ? sL[j] : (K)pol.list_key(lo + j); };
  auto lb_keys = [&](K v) -> int { return lb_seq([&](int i) { return sK[i]; }, len, v); };
  // each list key after the last element below it
  for (int j = tid; j < (int)cnt; j += kMkThreads) {
    const int p = lb_keys(lkey(j));
    if (lsm) sPj[j] = (uint16_t)p;
    if (p > 0)
      atomicAdd(reinterpret_cast<unsigned long long *>(&sX[kpad<uint64_t>(p - 1)]), 1ull << 32);
    else
      atomicAdd(&s_c00, 1u);
  }
  __syncthreads();
  {  // exclusive scan of the counts in element order (thread t: elements 8t .. 8t+7)
    uint64_t v[kMkItems], tsum = 0;
#pragma unroll
    for (int i = 0; i < kMkItems; ++i) {
      v[i] = sX[kpad<uint64_t>(tid * kMkItems + i)];
      tsum += v[i];
    }
    uint64_t ex = block_exclusive_scan<uint64_t>(tsum, &s_tot);
#pragma unroll
    for (int i = 0; i < kMkItems; ++i) {
      sX[kpad<uint64_t>(tid * kMkItems + i)] = ex;
      ex += v[i];
    }
    if (tid == 0) sX[kpad<uint64_t>(kMkTile)] = s_tot;
  }
  __syncthreads();
  const uint32_t preG = (uint32_t)s_pre, preE = (uint32_t)(s_pre >> 32), lo32 = (uint32_t)lo, c00 = s_c00;
  auto surv = [&](uint64_t x) -> uint32_t {  // kept elements below, from an exclusive count
    const uint32_t g = preG + (uint32_t)(x & 0xFFFFu), e = preE + (uint32_t)((x >> 16) & 0xFFFFu);
    return g + (e > m ? e - m : 0u);
  };
  auto below = [&](uint64_t x) -> uint32_t { return c00 + (uint32_t)((x >> 32) & 0xFFFFu); };  // list keys below
  const int mb = a.minor_bits;
  const uint32_t nmaj = (uint32_t)a.n_major;
  // kept and dropped elements, striped (coalesced writes), and the offsets of
  // the majors that start after each element
#pragma unroll
  for (int i = 0; i < kMkItems; ++i) {
    const int e = i * kMkThreads + tid;
    if (e < len) {
      const uint64_t x = sX[kpad<uint64_t>(e)];
      const uint32_t keep = (fl[i] & 0xFFFFu) | ((fl[i] >> 16) & (preE + (uint32_t)((x >> 16) & 0xFFFFu) >= m ? 1u : 0u));
      const K key = sK[e];
      if (keep) {
        const uint32_t pos = surv(x) + lo32 + below(x);
        if ((int64_t)pos < a.n_out) pol.write_kept(it[i], base + e, pos, key);
      } else {
        pol.write_dropped(it[i], base + e, key);
      }
      const uint32_t maj = (uint32_t)(key >> mb);
      const uint32_t nxt = e + 1 == len && last ? nmaj : min((uint32_t)(sK[e + 1] >> mb), nmaj);
      if (nxt > maj) {
        const uint32_t sv = surv(sX[kpad<uint64_t>(e + 1)]) + lo32;
        for (uint32_t M = maj + 1; M <= nxt; ++M)
          a.off[M] = (int32_t)(sv + (uint32_t)lb_seq(lkey, (int)cnt, (K)M << mb));
      }
    }
  }
  if (b == 0) {  // majors up to the first element's: no kept element before them
    const uint32_t maj0 = min((uint32_t)(sK[0] >> mb), nmaj);
    for (uint32_t M = tid; M <= maj0; M += kMkThreads) a.off[M] = (int32_t)lb_seq(lkey, (int)cnt, (K)M << mb);
  }
  // the tile's list entries
  for (int j = tid; j < (int)cnt; j += kMkThreads) {
    const K key = lkey(j);
    const int p = lsm ? (int)sPj[j] : lb_keys(key);
    const uint32_t pos = lo32 + (uint32_t)j + surv(sX[kpad<uint64_t>(p)]);
    if ((int64_t)pos < a.n_out) pol.write_list(lo + j, key, pos);
  }
}

// The stored weights (row order) merged with the regrown positions: writes
// the output pattern, values (+0 for the regrown), sources (-1 for the
// regrown), 16-bit columns, and -- for the column-view update -- the output
// index of every old weight (~0u when pruned), of every regrown position (by
// acceptance rank), and the pruned weights per column.  K: 32-bit keys when
// row and column bits fit 31.
template <typename TV, typename K>
struct RowPol {
  using Key = K;
  static constexpr bool kByColumn = false;
  const int32_t *row, *col;
  const TV *val;
  const SelState *st;
  int cbits;
  const uint64_t *B;   // regrown positions, row order
  const uint32_t *Bq;  // their acceptance ranks
  int32_t *row_out, *col_out;
  TV *val_out;
  int32_t *src_out;  // or null
  uint16_t *col16;   // or null
  uint32_t *newidx;  // or null
  uint32_t *gq;      // or null
  uint32_t *pcnt;    // or null: pruned weights per column, added to
  struct Shared {
    uint32_t unused;
  };
  struct Item {
    TV v;
  };
  __device__ uint32_t ties_dropped() const { return st->remaining; }
  __device__ uint32_t load(int64_t base, int len, bool, const MkBound &, uint32_t, Item (&it)[kMkItems],
                           uint32_t (&fl)[kMkItems], const PadKeys<K> &sK, Shared &) const {
    const uint32_t t = st->prefix;
    uint32_t r[kMkItems], c[kMkItems];
#pragma unroll
    for (int i = 0; i < kMkItems; ++i) {
      const int e = i * kMkThreads + threadIdx.x;
      if (e < len) {
        r[i] = (uint32_t)ld_stream(row + base + e);
        c[i] = (uint32_t)ld_stream(col + base + e);
        it[i].v = ld_stream(val + base + e);
      }
    }
#pragma unroll
    for (int i = 0; i < kMkItems; ++i) {
      const int e = i * kMkThreads + threadIdx.x;
      fl[i] = 0u;
      if (e < len) {
        sK[e] = ((K)r[i] << cbits) | (K)c[i];
        const uint32_t mk = mag_of(it[i].v);
        fl[i] = (mk > t ? 1u : 0u) | (mk == t ? 0x10000u : 0u);
      }
    }
    return 0u;
  }
  __device__ bool keys_blocked(int64_t, int, bool, uint32_t, uint32_t, const PadKeys<K> &, Shared &) const {
    return false;
  }
  __device__ uint64_t key_at_warp(int64_t k, uint32_t *) const {
    return ((uint64_t)(uint32_t)row[k] << cbits) | (uint32_t)col[k];
  }
  __device__ uint64_t list_key(int64_t j) const { return B[j]; }
  __device__ void write_kept(const Item &x, int64_t k, uint32_t pos, K key) const {
    const uint32_t c = (uint32_t)(key & (((K)1 << cbits) - 1));
    row_out[pos] = (int32_t)(key >> cbits);
    col_out[pos] = (int32_t)c;
    val_out[pos] = x.v;
    if (src_out) src_out[pos] = (int32_t)k;
    if (col16) col16[pos] = (uint16_t)c;
    if (newidx) newidx[k] = pos;
  }
  __device__ void write_dropped(const Item &, int64_t k, K key) const {
    if (newidx) newidx[k] = ~0u;
    if (pcnt) atomicAdd(&pcnt[(uint32_t)(key & (((K)1 << cbits) - 1))], 1u);
  }
  __device__ void write_list(int64_t j, K key, uint32_t pos) const {
    const uint32_t c = (uint32_t)(key & (((K)1 << cbits) - 1));
    row_out[pos] = (int32_t)(key >> cbits);
    col_out[pos] = (int32_t)c;
    val_out[pos] = from_f32<TV>(0.f);
    if (src_out) src_out[pos] = -1;
    if (col16) col16[pos] = (uint16_t)c;
    if (gq) gq[Bq[j]] = pos;
  }
};

// The current column view (column order: rows, storage indices, column
// offsets) merged with the regrown positions in column order (col << rbits |
// row, 32-bit), into the second view: kept entries take their weight's new
// storage index, regrown ones theirs.
struct ColPol {
  using Key = uint32_t;
  static constexpr bool kByColumn = true;
  const int32_t *cp;       // [in_f + 1] current column offsets
  const int32_t *row_t;    // current rows in column order
  const uint16_t *rowt16;  // or null
  const int32_t *src_t;    // current storage indices in column order
  const uint32_t *newidx;
  int rbits;
  int32_t in_f;
  const uint32_t *gc_key, *gc_q, *gq;
  int32_t *row_t_new, *src_t_new;  // (the 32-bit rows only without the 16-bit copy)
  uint16_t *rowt16_new;             // or null
  static constexpr int kCpCap = 1024;  // column offsets of a tile staged in shared memory
  struct Shared {
    int32_t cp[kCpCap];
  };
  struct Item {
    uint32_t nk;
  };
  __device__ uint32_t ties_dropped() const { return 0u; }
  // rows into sK (the columns follow, blocked), the tile's column offsets
  // cp[c0 .. c1 + 1] into shared memory, each entry's weight's new index;
  // returns this thread's count of the pruned entries of column c0 ahead of
  // the tile (from the column's first entry up to base), whose loads travel
  // with the tile's
  __device__ uint32_t load(int64_t base, int len, bool last, const MkBound &bd, uint32_t c_next,
                           Item (&it)[kMkItems], uint32_t (&fl)[kMkItems], const PadKeys<uint32_t> &sK,
                           Shared &ps) const {
    const uint32_t c0 = bd.aux;
    const int64_t ncp = (int64_t)(last ? (uint32_t)in_f - 1 : c_next) - c0 + 2;
    if (ncp <= kCpCap)
      for (int i = threadIdx.x; i < ncp; i += kMkThreads) ps.cp[i] = cp[c0 + i];
    uint32_t src[kMkItems];
#pragma unroll
    for (int i = 0; i < kMkItems; ++i) {
      const int e = i * kMkThreads + threadIdx.x;
      if (e < len) {
        src[i] = (uint32_t)ld_stream(src_t + base + e);
        sK[e] = rowt16 ? (uint32_t)ld_stream(rowt16 + base + e) : (uint32_t)ld_stream(row_t + base + e);
      }
    }
    const int64_t ja = (int64_t)bd.aux2 + threadIdx.x;
    const uint32_t qa = ja < base ? (uint32_t)src_t[ja] : ~0u;
#pragma unroll
    for (int i = 0; i < kMkItems; ++i) {
      const int e = i * kMkThreads + threadIdx.x;
      fl[i] = 0u;
      if (e < len) {
        it[i].nk = newidx[src[i]];
        fl[i] = it[i].nk != ~0u ? 1u : 0u;
      }
    }
    uint32_t ahead = qa != ~0u && newidx[qa] == ~0u ? 1u : 0u;
    for (int64_t j = ja + kMkThreads; j < base; j += kMkThreads)  // columns longer than a block
      ahead += newidx[src_t[j]] == ~0u ? 1u : 0u;
    return ahead;
  }
  // columns, blocked (thread t: entries 8t .. 8t+7): one search, then forward
  // steps; the block synchronises after it
  __device__ bool keys_blocked(int64_t base, int len, bool last, uint32_t c0, uint32_t c_next,
                               const PadKeys<uint32_t> &sK, Shared &ps) const {
    const int64_t ncp = (int64_t)(last ? (uint32_t)in_f - 1 : c_next) - c0 + 2;
    const int e0 = threadIdx.x * kMkItems;
    if (e0 >= len) return true;
    const int e1 = min(e0 + kMkItems, len);
    // the last x in [0, ncp - 2] with off[x] <= base + e0, then forward steps
    // (32-bit: positions are below 2^31)
    auto walk = [&](const int32_t *off) {
      const int32_t t0 = (int32_t)base + e0;
      int lo = 0, hi = (int)ncp - 1;
      while (hi - lo > 1) {
        const int md = (lo + hi) >> 1;
        if (off[md] <= t0)
          lo = md;
        else
          hi = md;
      }
      int32_t nxt = off[lo + 1];
      for (int e = e0; e < e1; ++e) {
        const int32_t pos = (int32_t)base + e;
        while (nxt <= pos) nxt = off[++lo + 1];
        sK[e] |= (c0 + (uint32_t)lo) << rbits;
      }
    };
    if (ncp <= kCpCap)
      walk(ps.cp);
    else
      walk(cp + c0);
    return true;
  }
  // column of entry e: the number of columns c >= 1 whose offset cp[c] is at most e
  __device__ uint64_t key_at_warp(int64_t e, uint32_t *aux) const {
    const uint32_t c =
        (uint32_t)lb_warp([&](int64_t j) { return (uint64_t)(uint32_t)cp[j + 1]; }, in_f, (uint64_t)e + 1);
    *aux = c;
    const uint32_t r = rowt16 ? (uint32_t)rowt16[e] : (uint32_t)row_t[e];
    return ((uint64_t)c << rbits) | r;
  }
  __device__ uint64_t list_key(int64_t j) const { return gc_key[j]; }
  __device__ void write_kept(const Item &x, int64_t, uint32_t pos, uint32_t key) const {
    const uint32_t r = key & ((1u << rbits) - 1u);
    src_t_new[pos] = (int32_t)x.nk;
    if (rowt16_new)
      rowt16_new[pos] = (uint16_t)r;
    else
      row_t_new[pos] = (int32_t)r;
  }
  __device__ void write_dropped(const Item &, int64_t, uint32_t) const {}
  __device__ void write_list(int64_t j, uint32_t key, uint32_t pos) const {
    const uint32_t r = key & ((1u << rbits) - 1u);
    src_t_new[pos] = (int32_t)gq[gc_q[j]];
    if (rowt16_new)
      rowt16_new[pos] = (uint16_t)r;
    else
      row_t_new[pos] = (int32_t)r;
  }
};

// per-tile packed keep counts of f; exclusive prefixes in place when there are
// more tiles than each merge block adds up itself
template <typename F>
cudaError_t keep_sums(F f, int64_t n, uint64_t *sums, cudaStream_t s, bool *direct) {
  const int64_t nb = ceil_div(n, kScanTile);
  launch_pdl(k_scan_reduce<uint64_t, F>, (unsigned)nb, kScanThreads, 0, s, f, n, sums);
  *direct = nb <= kScanDirectTiles;
  if (!*direct) launch_pdl(k_scan_spine<uint64_t>, 1, kScanThreads, 0, s, sums, nb, (uint64_t *)nullptr);
  return cudaGetLastError();
}

template <class Pol, int kMode>
cudaError_t launch_merge_mode(const Pol &pol, const MkArgs &a, cudaStream_t s) {
  constexpr size_t dyn = mk_smem_bytes<Pol>();
  cudaError_t e = raise_smem_limit(k_merge_kept<Pol, kMode>, dyn);
  if (e == cudaSuccess)
    e = launch_pdl(k_merge_kept<Pol, kMode>, (unsigned)ceil_div(a.n, kMkTile), kMkThreads, dyn, s, pol, a);
  return e;
}

// The column view is merged by column counts; the row order by tile counts.
template <class Pol>
cudaError_t launch_merge(const Pol &pol, const MkArgs &a, int mode, cudaStream_t s) {
  if constexpr (Pol::kByColumn) {
    return launch_merge_mode<Pol, kMkByColumn>(pol, a, s);
  } else {
    if (mode == kMkDirect) return launch_merge_mode<Pol, kMkDirect>(pol, a, s);
    return launch_merge_mode<Pol, kMkGiven>(pol, a, s);
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

// The column-view update on stream s3: the old view merged with the n_list
// regrown positions in column order (pl.gc_key, pl.gc_q, pl.gq), kept
// entries taking pl.newidx, tile prefixes from the pruned counts per column
// (pl.cv_pcnt, n_list > 0), into the plan's second view, then its column
// tiles.  `guard`: when set and zero, the merge writes nothing.
cudaError_t queue_colview_merge(const PlanPtrs &pl, int32_t in_f, int64_t nnz, int64_t n_list, int rbits,
                                const uint32_t *guard, const TileGeom &gt, cudaStream_t s3) {
  const int64_t n_tiles = ceil_div(nnz, kMkTile);
  const ColPol cpol{pl.cp,     pl.row_t, pl.rowt16, pl.src_t,     pl.newidx,    rbits,
                    in_f,      pl.gc_key, pl.gc_q,  pl.gq,        pl.row_t_alt, pl.src_t_alt,
                    pl.rowt16_alt};
  MkBound *cbnd = reinterpret_cast<MkBound *>(pl.cv_bnd);
  // with pruned weights, one more block of the bounds launch turns their
  // counts per column into exclusive prefixes
  const bool pruned = n_list > 0;
  launch_pdl(k_bounds<ColPol>, grid_for(32 * (n_tiles + 1), 256) + (pruned ? 1u : 0u), 256, 0, s3, cpol, n_list,
             n_tiles, cbnd, pruned ? (const uint32_t *)pl.cv_pcnt : nullptr, pl.cv_ppre, (int64_t)in_f);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = launch_merge(cpol,
                     MkArgs{nnz, n_list, nnz, cbnd, nullptr, guard, rbits, in_f, pl.cp_alt,
                            pruned ? (const uint32_t *)pl.cv_ppre : nullptr},
                     kMkByColumn, s3);
  if (err != cudaSuccess) return err;
  return cut_tiles(pl.cp_alt, in_f, nnz, gt, pl.tiles_t_alt, s3);
}

// Expected number of draws to accept `need` distinct positions out of `empty`
// empty ones, among n_pos equally likely positions: n_pos * (H(empty) -
// H(empty - need)), using ln((e + 1/2) / (e - need + 1/2)) for the difference.
double expected_draws(double n_pos, double empty, double need) {
  if (need <= 0) return 0.0;
  return n_pos * log((empty + 0.5) / (empty - need + 0.5));
}

// Standard deviation of that number: the draws for the k-th new position are
// geometric with success probability q = u / n_pos (u = empty - k positions
// left), variance (1 - q) / q^2 = n_pos (n_pos - u) / u^2; summed over u from
// empty - need + 1 to empty with the same half-step sums as above.
double draws_sd(double n_pos, double empty, double need) {
  if (need <= 0) return 0.0;
  const double lo = empty - need + 0.5, hi = empty + 0.5;
  const double var = n_pos * n_pos * (1.0 / lo - 1.0 / hi) - n_pos * log(hi / lo);
  return var > 0.0 ? sqrt(var) : 0.0;
}

struct RWs {
  size_t state, dstate, sums, above, scand, scan2, grown_a, B, Bq, cand, alb, hkeys, hmin, bcnt, bnd, bkey, bq,
      rk0, rv0, rk1, rv1, rtemp, plan, total;
  int64_t d_max, cap;
  bool packed;     // positions below 2^32: one 64-bit word per table slot
  uint32_t n_bkt;  // buckets per order (row, column)
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
  const size_t np = (size_t)(n_prune > 0 ? n_prune : 1), dmx = (size_t)(w.d_max > 0 ? w.d_max : 1);
  w.n_bkt = (uint32_t)((int64_t)np / kBktTarget > 0 ? (int64_t)np / kBktTarget : 1);
  if (w.n_bkt > (1u << 30)) w.n_bkt = 1u << 30;
  size_t o = 0;
  w.state = o;
  o += align_up(sizeof(SelState), kAlign);
  w.dstate = o;
  o += align_up(sizeof(DrawState), kAlign);
  w.sums = o;
  o += scan_temp_bytes<uint64_t>(nnz > 0 ? nnz : 1);
  w.above = o;
  w.scand = o;  // the keys in the select's first-digit bucket
  if (n_prune > 0) o += align_up(8 * (size_t)(nnz > 0 ? nnz : 1), kAlign);
  w.scan2 = o;
  o += scan_temp_bytes<uint32_t>((int64_t)dmx);
  w.grown_a = o;
  o += align_up(8 * np, kAlign);
  w.B = o;
  o += align_up(8 * np, kAlign);
  w.Bq = o;
  o += align_up(4 * np, kAlign);
  w.cand = o;
  o += align_up(8 * dmx, kAlign);
  w.alb = o;  // the acceptance scan's look-back words (one per tile of draws) and its ticket
  o += align_up(8 * ((size_t)ceil_div((int64_t)dmx, kScanTile) + 1), kAlign);
  w.packed = ((uint64_t)out_f << bits_for((uint64_t)(in_f - 1))) <= (1ull << 32);
  w.hkeys = o;
  o += align_up(8 * (size_t)cap, kAlign);
  w.hmin = o;
  if (!w.packed) o += align_up(4 * (size_t)cap, kAlign);
  const bool bk = w.n_bkt <= kBktMaxBuckets;
  w.bcnt = o;  // both orders' bucket counts, one launch clears them
  if (bk) o += align_up(4 * 2 * (size_t)w.n_bkt * kCntStride, kAlign);
  w.bnd = o;  // tile bounds of the merge
  o += align_up(sizeof(MkBound) * (size_t)(ceil_div(nnz > 0 ? nnz : 1, kMkTile) + 1), kAlign);
  // the buckets' slots, or (the general sort) its key / rank buffers
  const size_t region = o;
  w.bkey = o;
  if (bk) o += align_up(8 * 2 * (size_t)w.n_bkt * kBktCap, kAlign);
  w.bq = o;
  if (bk) o += align_up(4 * 2 * (size_t)w.n_bkt * kBktCap, kAlign);
  const size_t bucket_end = o;
  o = region;
  w.rk0 = o;
  o += align_up(8 * np, kAlign);
  w.rv0 = o;
  o += align_up(4 * np, kAlign);
  w.rk1 = o;
  o += align_up(8 * np, kAlign);
  w.rv1 = o;
  o += align_up(4 * np, kAlign);
  w.rtemp = o;
  o += radix_temp_bytes((int64_t)np);
  if (o < bucket_end) o = bucket_end;
  w.plan = o;  // a plan rebuild's scratch (layers without the column-view update)
  o += plan_build_ws_bytes(out_f, in_f, nnz);
  w.total = o;
  return w;
}

template <typename TV>
snack_status restructure_impl(const RestructureArgs &a, void *ws, size_t ws_bytes, cudaStream_t s, bool *updated) {
  *updated = false;
  const RWs W = rws_layout(a.out_f, a.in_f, a.nnz, a.n_prune);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  SelState *st = reinterpret_cast<SelState *>(b + W.state);
  DrawState *ds = reinterpret_cast<DrawState *>(b + W.dstate);
  uint64_t *sums = reinterpret_cast<uint64_t *>(b + W.sums);
  void *stemp2 = b + W.scan2;
  uint64_t *grown_a = reinterpret_cast<uint64_t *>(b + W.grown_a);
  uint64_t *B = reinterpret_cast<uint64_t *>(b + W.B);
  uint32_t *Bq = reinterpret_cast<uint32_t *>(b + W.Bq);
  uint64_t *cand = reinterpret_cast<uint64_t *>(b + W.cand);
  const PosTable tab{reinterpret_cast<uint64_t *>(b + W.hkeys), reinterpret_cast<uint32_t *>(b + W.hmin),
                     (uint64_t)(W.cap - 1), W.packed};
  uint32_t *bcnt = reinterpret_cast<uint32_t *>(b + W.bcnt);
  const PlanPtrs &pl = *a.plan;
  const TV *val = reinterpret_cast<const TV *>(a.val);
  const int64_t nnz = a.nnz, n_prune = a.n_prune;
  const uint64_t n_pos = (uint64_t)a.out_f * (uint64_t)a.in_f;
  // positions travel as keys (row << cbits) | col: same order as row * in_f + col
  const int cbits = bits_for((uint64_t)(a.in_f - 1)), rbits = bits_for((uint64_t)(a.out_f - 1));
  const uint64_t key_space = (uint64_t)a.out_f << cbits;
  const int kbits = cbits + rbits;
  const bool update = a.update && pl.newidx && kbits <= 32 && n_prune <= pl.cv_pmax;
  const bool buckets = n_prune > 0 && W.n_bkt <= kBktMaxBuckets;
  BucketSet br{}, bc{};
  if (buckets) {
    uint64_t *bkey = reinterpret_cast<uint64_t *>(b + W.bkey);
    uint32_t *bq = reinterpret_cast<uint32_t *>(b + W.bq);
    const size_t per = (size_t)W.n_bkt * kBktCap;
    br = BucketSet{bcnt, bkey, bq, bucket_mult(W.n_bkt, key_space), W.n_bkt};
    if (update)
      bc = BucketSet{bcnt + (size_t)W.n_bkt * kCntStride, bkey + per, bq + per,
                     bucket_mult(W.n_bkt, (uint64_t)a.in_f << rbits), W.n_bkt};
  }
  cudaError_t e;
#define SNACK_TRY(x)                             \
  do {                                           \
    e = (x);                                     \
    if (e != cudaSuccess) return SNACK_ERR_CUDA; \
  } while (0)

  // Two branches meet at the merge: the regrow (draws, acceptance, sort of
  // the regrown positions) depends only on the old pattern; it is the longer
  // of the two and runs on the caller's stream (s2 = s), while the prune
  // select runs beside it on the handle's second stream ss, of the lowest
  // priority (so the regrow's blocks go first), forked from s at the start
  // and joined back before the merge.  The host reads each draw chunk's
  // accepted count from mapped pinned words that a kernel writes (an event
  // marks them ready).
  cudaStream_t s2 = s, ss = a.aux;
  auto fork = [&]() -> cudaError_t {
    cudaError_t err = cudaEventRecord(a.ev_fork, s);
    return err != cudaSuccess ? err : cudaStreamWaitEvent(ss, a.ev_fork, 0);
  };
  auto join = [&]() -> cudaError_t {
    cudaError_t err = cudaEventRecord(a.ev_join, ss);
    return err != cudaSuccess ? err : cudaStreamWaitEvent(s, a.ev_join, 0);
  };
  SNACK_TRY(fork());
  const uint64_t base = sm64_finalise(a.seed ^ sm64_finalise(a.step));
  const double empty = (double)n_pos - (double)nnz;
  int64_t done = 0, acc = 0;
  auto draw_chunk = [&](int64_t m, bool first) -> cudaError_t {
    if (pl.col16)
      launch_pdl(k_draw<uint16_t>, grid_for(m, 256), 256, 0, s2, base, (uint64_t)done, m, n_pos, a.in_f, cbits, pl.rp,
                 (const uint16_t *)pl.col16, cand, tab, &ds->overflow);
    else
      launch_pdl(k_draw<int32_t>, grid_for(m, 256), 256, 0, s2, base, (uint64_t)done, m, n_pos, a.in_f, cbits, pl.rp,
                 a.col, cand, tab, &ds->overflow);
    const int64_t n_at = ceil_div(m, kScanTile);
    uint64_t *alb = reinterpret_cast<uint64_t *>(b + W.alb);
    uint32_t *aticket = reinterpret_cast<uint32_t *>(alb + n_at);
    if (!first) {  // the first chunk's words were cleared with the table
      cudaError_t err = cudaMemsetAsync(alb, 0, sizeof(uint64_t) * (size_t)n_at + sizeof(uint32_t), s2);
      if (err != cudaSuccess) return err;
    }
    const AcceptArgs aa{cand,
                        m,
                        (uint64_t)done,
                        tab,
                        grown_a,
                        acc,
                        n_prune,
                        first && buckets ? br : BucketSet{},
                        &ds->bucket_overflow,
                        first && buckets && update ? bc : BucketSet{},
                        &ds->col_overflow,
                        cbits,
                        rbits,
                        alb,
                        aticket,
                        &ds->lb_fail,
                        &ds->total};
    launch_pdl(k_accept_scan, (unsigned)n_at, kAccThreads, 0, s2, aa);
    return cudaGetLastError();
  };
  auto chunk_size = [&]() -> int64_t {
    // the expected draws and eight standard deviations (then the chunk falls
    // short with a probability far below 1e-9), or 1.1 x the expected draws
    // where that is less (crowded layers: more chunks are cheaper than many
    // wasted draws)
    const double e_left = empty - (double)acc, need = (double)(n_prune - acc);
    const double ex = expected_draws((double)n_pos, e_left, need);
    const double want = fmin(ex + 8.0 * draws_sd((double)n_pos, e_left, need), 1.1 * ex) + 1024.0;
    int64_t m = (int64_t)ceil(want);
    return m > W.d_max - done ? W.d_max - done : m;
  };
  // general sorts of the n_prune regrown positions: row order, column order
  uint64_t *rk0 = reinterpret_cast<uint64_t *>(b + W.rk0), *rk1 = reinterpret_cast<uint64_t *>(b + W.rk1);
  uint32_t *rv0 = reinterpret_cast<uint32_t *>(b + W.rv0), *rv1 = reinterpret_cast<uint32_t *>(b + W.rv1);
  auto sort_rows_general = [&]() -> cudaError_t {
    return radix_sort_custom<uint64_t>(GrownRowSrc{grown_a}, ArrayDst<uint64_t>{B, Bq}, n_prune, kbits, rk0, rv0, rk1,
                                       rv1, b + W.rtemp, s2);
  };
  auto sort_cols_general = [&]() -> cudaError_t {
    if (!update) return cudaSuccess;
    return radix_sort_custom<uint32_t>(GrownColSrc{grown_a, cbits, rbits}, ArrayDst<uint32_t>{pl.gc_key, pl.gc_q},
                                       n_prune, kbits, reinterpret_cast<uint32_t *>(rk0), rv0,
                                       reinterpret_cast<uint32_t *>(rk1), rv1, b + W.rtemp, s2);
  };
  const int64_t n_tiles = ceil_div(nnz, kMkTile);
  const uint32_t *row_guard = n_prune > 0 ? &ds->lists_ok : nullptr;
  uint32_t *col_ok = pl.flags + kPlanFlagColOk;
  const uint32_t *col_guard = n_prune > 0 ? col_ok : nullptr;
  // 3: the merge (after s waits for the row-order list) and the plan's row half
  bool row_direct = true;  // set with the keep counts below, before the first call
  auto queue_rows = [&]() -> cudaError_t {
    const MkBound *rbnd = reinterpret_cast<MkBound *>(b + W.bnd);
    const uint32_t *nix = nullptr;
    cudaError_t err;
    auto run = [&](auto rpol) -> cudaError_t {
      using P = decltype(rpol);
      launch_pdl(k_bounds<P>, grid_for(32 * (n_tiles + 1), 256), 256, 0, s, rpol, n_prune, n_tiles,
                 const_cast<MkBound *>(rbnd), (const uint32_t *)nullptr, (uint32_t *)nullptr, (int64_t)0);
      cudaError_t r = cudaGetLastError();
      return r != cudaSuccess ? r
                              : launch_merge(rpol,
                                             MkArgs{nnz, n_prune, nnz, rbnd, sums, row_guard, cbits, a.out_f, pl.rp,
                                                    nullptr},
                                             row_direct ? kMkDirect : kMkGiven, s);
    };
    (void)nix;
    TV *vo = reinterpret_cast<TV *>(a.val_out);
    uint32_t *ni = update ? pl.newidx : nullptr, *gq = update ? pl.gq : nullptr;
    uint32_t *pc = update && n_prune > 0 ? pl.cv_pcnt : nullptr;
    if (kbits <= 31)
      err = run(RowPol<TV, uint32_t>{a.row, a.col, val, st, cbits, B, Bq, a.row_out, a.col_out, vo, a.src_out,
                                     pl.col16, ni, gq, pc});
    else
      err = run(RowPol<TV, uint64_t>{a.row, a.col, val, st, cbits, B, Bq, a.row_out, a.col_out, vo, a.src_out,
                                     pl.col16, ni, gq, pc});
    if (err != cudaSuccess) return err;
    return build_plan(a.out_f, a.in_f, nnz, a.row_out, a.col_out, pl, a.gf, a.gt, b + W.plan, s, kPlanRowsReady,
                      !update);
  };
  // 4: the column-view update, on the third stream (lowest priority), after
  // s's work so far (which waits for the select)
  cudaStream_t s3 = a.aux_lo;
  auto queue_cols = [&]() -> cudaError_t {
    cudaError_t err = cudaEventRecord(a.ev_fork, s);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(s3, a.ev_fork, 0);
    if (err != cudaSuccess) return err;
    return queue_colview_merge(pl, a.in_f, nnz, n_prune, rbits, col_guard, a.gt, s3);
  };
  auto mark = [&]() -> cudaError_t { return cudaEventRecord(a.ev_join, ss); };
  auto wait_mark = [&]() -> cudaError_t { return cudaStreamWaitEvent(s, a.ev_join, 0); };

  // 2. regrow, first chunk, and its sorted lists (on s2 = s): the merge
  //    follows them in stream order
  int64_t m = 0;
  e = cudaSuccess;
  if (n_prune > 0) {
    const int64_t n_at1 = ceil_div(chunk_size(), kScanTile);
    uint64_t *alb = reinterpret_cast<uint64_t *>(b + W.alb);
    launch_pdl(k_rs_init, grid_for(W.cap, 256, 1184), 256, 0, s2, ds, tab, bcnt,
               (int64_t)(buckets ? 2 * (int64_t)W.n_bkt * kCntStride : 0), alb, n_at1,
               reinterpret_cast<uint32_t *>(alb + n_at1), update ? pl.cv_pcnt : (uint32_t *)nullptr,
               (int64_t)(update ? a.in_f : 0), col_ok);
    m = chunk_size();
    e = draw_chunk(m, true);
    if (e == cudaSuccess) {
      const bool k32 = kbits <= 32;
      if (buckets) {  // both orders' lists in one launch
        const uint32_t nr = (br.nb + 7) / 8, nc = update ? (bc.nb + 7) / 8 : 0u;
        launch_pdl(k_bkt_rank, nr + nc, 256, 0, s2, br, RankDst{B, nullptr, Bq}, k32, nr, bc,
                   RankDst{nullptr, pl.gc_key, pl.gc_q}, n_prune, ds, a.counts_dev, col_ok, (const uint32_t *)nullptr);
        e = cudaGetLastError();
      } else {
        e = sort_rows_general();
        if (e == cudaSuccess) e = sort_cols_general();
        if (e == cudaSuccess) {
          launch_pdl(k_publish, 1, 1, 0, s2, ds, n_prune, a.counts_dev, 1, col_ok);
          e = cudaGetLastError();
        }
      }
    }
    if (e == cudaSuccess) e = cudaEventRecord(a.counts_ready, s2);
  }
  if (e != cudaSuccess) {
    join();
    return SNACK_ERR_CUDA;
  }
  // 1. prune threshold (on ss): three digit passes (11, 10, 10 bits), high to
  //    low; keep counts per tile
  launch_pdl(k_sel_init, 1, 256, 0, ss, st, (uint32_t)n_prune);
  if (n_prune > 0) {
    // first digit over every key; the keys in its bucket listed while each
    // tile counts those above it; the rest of the select and the tiles' keep
    // counts from the list
    launch_pdl(k_sel_pass<TV, 0>, grid_for((nnz + 15) / 16, 256, 1184), 256, 0, ss, val, nnz, st);
    uint64_t *scand = reinterpret_cast<uint64_t *>(b + W.scand);
    launch_pdl(k_sel_bucket<TV>, (unsigned)n_tiles, kScanThreads, 0, ss, val, nnz, st, sums, scand);
    launch_pdl(k_sel_cand<1>, kSelCandBlocks, 256, 0, ss, (const uint64_t *)scand, st);
    launch_pdl(k_sel_cand<2>, kSelCandBlocks, 256, 0, ss, (const uint64_t *)scand, st);
    launch_pdl(k_sel_tiles, kSelCandBlocks, 256, 0, ss, (const uint64_t *)scand, (const SelState *)st, sums);
    row_direct = n_tiles <= kScanDirectTiles;
    if (!row_direct) launch_pdl(k_scan_spine<uint64_t>, 1, kScanThreads, 0, ss, sums, n_tiles, (uint64_t *)nullptr);
    e = cudaGetLastError();
  } else {
    e = keep_sums(KeepVal<TV>{val, st}, nnz, sums, ss, &row_direct);
  }
  if (e == cudaSuccess) e = mark();
  // With the update, 3 and 4 are queued at once behind the lists' flags (they
  // write nothing unless the first chunk's lists came out whole); a plan
  // rebuild on s cannot be undone, so without the update they wait for the
  // host's verdict.
  if (e == cudaSuccess && update) e = wait_mark();
  if (e == cudaSuccess && update) e = queue_rows();
  if (e == cudaSuccess && update) e = queue_cols();
  if (e != cudaSuccess) {
    join();
    return SNACK_ERR_CUDA;
  }
  snack_status verdict = SNACK_OK;
  bool rows_queued = update, cols_queued = update;
  if (n_prune > 0) {
    if (cudaEventSynchronize(a.counts_ready) != cudaSuccess) {
      join();
      return SNACK_ERR_CUDA;
    }
    if (a.host_counts[1]) {  // the position table ran full (nothing of the output was written)
      join();
      return SNACK_ERR_WORKSPACE;
    }
    if (a.host_counts[4]) {  // the acceptance scan gave up waiting for a predecessor tile: the
      join();                 // lists were not made, so the queued passes wrote nothing
      return SNACK_ERR_TIMEOUT;
    }
    acc = a.host_counts[0] < (uint32_t)n_prune ? (int64_t)a.host_counts[0] : n_prune;
    done = m;
    if (acc < n_prune || a.host_counts[2]) {
      // the first chunk fell short or a row-order bucket ran over: more draws
      // (after everything queued so far), the general sorts, and 3 and 4 again
      rows_queued = cols_queued = false;
      while (acc < n_prune) {
        if (done >= W.d_max) {
          verdict = SNACK_ERR_NO_SPACE;
          break;
        }
        m = chunk_size();
        if (draw_chunk(m, false) != cudaSuccess) {
          verdict = SNACK_ERR_CUDA;
          break;
        }
        launch_pdl(k_publish, 1, 1, 0, s2, ds, n_prune, a.counts_dev, 0, col_ok);
        if (cudaGetLastError() != cudaSuccess || cudaEventRecord(a.counts_ready, s2) != cudaSuccess ||
            cudaEventSynchronize(a.counts_ready) != cudaSuccess) {
          verdict = SNACK_ERR_CUDA;
          break;
        }
        if (a.host_counts[1]) {
          verdict = SNACK_ERR_WORKSPACE;
          break;
        }
        if (a.host_counts[4]) {
          verdict = SNACK_ERR_TIMEOUT;
          break;
        }
        acc += a.host_counts[0];
        done += m;
      }
      if (verdict == SNACK_OK && (sort_rows_general() != cudaSuccess || sort_cols_general() != cudaSuccess))
        verdict = SNACK_ERR_CUDA;
      if (verdict == SNACK_OK) {
        launch_pdl(k_set_word, 1, 1, 0, s2, &ds->lists_ok, 1u);
        launch_pdl(k_set_word, 1, 1, 0, s2, col_ok, 1u);
        if (cudaGetLastError() != cudaSuccess) verdict = SNACK_ERR_CUDA;
      }
      if (join() != cudaSuccess && verdict == SNACK_OK) verdict = SNACK_ERR_CUDA;
      if (verdict != SNACK_OK) return verdict;
    } else if (update && a.host_counts[3]) {
      // only a column-order bucket ran over: the merge has written the
      // output; the column-order list the general way and 4 again
      cols_queued = false;
      SNACK_TRY(sort_cols_general());
      launch_pdl(k_set_word, 1, 1, 0, s2, col_ok, 1u);
      SNACK_TRY(cudaGetLastError());
      SNACK_TRY(join());  // the sort's scratch is in the workspace: done before the call returns
    }
  }
  if (!rows_queued) {
    SNACK_TRY(wait_mark());
    SNACK_TRY(queue_rows());
  }
  if (update && !cols_queued) SNACK_TRY(queue_cols());
  *updated = update;
#undef SNACK_TRY
  return SNACK_OK;
}

// ------------------------------------------------------------------------
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
  // With newidx set, the inputs of the incremental column-view update: each
  // old weight's new index (~0u: pruned), the pruned weights per column, the
  // new index of regrown weight q = row * n_per_row + g in gq, and (col <<
  // rbits | row, q) of every regrown weight in its column-order bucket;
  // *bovf set when a bucket ran out of slots; *n_grown the regrown count.
  uint32_t *newidx, *pcnt, *gq;
  BucketSet bc;
  uint32_t *bovf, *n_grown;
  int rbits;
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
      if (A.newidx) A.newidx[k0 + j] = (uint32_t)o;
    } else if (in && !keep) {
      if (n_pr + __popc(pb & lt) < (uint32_t)kRowsMaxPrune) pcol[n_pr + __popc(pb & lt)] = c;
      if (A.newidx) {
        A.newidx[k0 + j] = ~0u;
        atomicAdd(&A.pcnt[c], 1u);
      }
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
    if (A.gq) {
      const uint32_t q = (uint32_t)r * (uint32_t)A.n_per_row + (uint32_t)g;
      A.gq[q] = (uint32_t)o;
      A.bc.place((uint64_t)((c << A.rbits) | (uint32_t)r), q, A.bovf);
    }
  }
  if (A.n_grown && lane == 0 && p > 0) atomicAdd(A.n_grown, (uint32_t)p);
}

// The column-order buckets of a per-row restructure's regrown positions
// (out_f * n_per_row at most) in its workspace.
struct RowsBkt {
  uint32_t nb;
  size_t cnt, key, q, total;
};
RowsBkt rows_bkt_layout(int32_t out_f, int64_t n_per_row) {
  RowsBkt L{};
  const int64_t np = (int64_t)out_f * n_per_row, nb = np / kBktTarget;
  L.nb = (uint32_t)(nb < 1 ? 1 : nb > (int64_t)kBktMaxBuckets ? (int64_t)kBktMaxBuckets + 1 : nb);
  size_t o = 0;
  L.cnt = o;
  o += align_up(4 * (size_t)L.nb * kCntStride, kAlign);
  L.key = o;
  o += align_up(8 * (size_t)L.nb * kBktCap, kAlign);
  L.q = o;
  o += align_up(4 * (size_t)L.nb * kBktCap, kAlign);
  L.total = o;
  return L;
}

BucketSet rows_buckets(const RowsBkt &L, void *bws, int32_t in_f, int rbits) {
  uint8_t *b = reinterpret_cast<uint8_t *>(bws);
  return BucketSet{reinterpret_cast<uint32_t *>(b + L.cnt), reinterpret_cast<uint64_t *>(b + L.key),
                   reinterpret_cast<uint32_t *>(b + L.q), bucket_mult(L.nb, (uint64_t)in_f << rbits), L.nb};
}

}  // namespace

size_t rows_update_ws_bytes(int32_t out_f, int64_t n_per_row) {
  const RowsBkt L = rows_bkt_layout(out_f, n_per_row);
  return L.nb > kBktMaxBuckets ? 0 : L.total;
}

cudaError_t queue_rows_rank(const RowsRestructureArgs &a, cudaStream_t s) {
  const PlanPtrs &pl = *a.plan;
  const int rbits = bits_for((uint64_t)(a.out_f - 1));
  const BucketSet C = rows_buckets(rows_bkt_layout(a.out_f, a.n_per_row), a.bws, a.in_f, rbits);
  launch_pdl(k_bkt_rank, (C.nb + 7) / 8, 256, 0, s, BucketSet{}, RankDst{nullptr, nullptr, nullptr}, true, 0u, C,
             RankDst{nullptr, pl.gc_key, pl.gc_q}, (int64_t)a.out_f * a.n_per_row, (DrawState *)nullptr,
             (uint32_t *)nullptr, (uint32_t *)nullptr, (const uint32_t *)a.err);
  return cudaGetLastError();
}

cudaError_t queue_rows_colview(const RowsRestructureArgs &a, int64_t n_grown, const TileGeom &gt, cudaStream_t s,
                               cudaStream_t s_lo, cudaEvent_t ev) {
  const PlanPtrs &pl = *a.plan;
  const int rbits = bits_for((uint64_t)(a.out_f - 1));
  cudaError_t e = cudaEventRecord(ev, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_lo, ev, 0);
  if (e != cudaSuccess) return e;
  return queue_colview_merge(pl, a.in_f, a.nnz, n_grown, rbits, nullptr, gt, s_lo);
}

size_t restructure_ws_bytes(int32_t out_f, int32_t in_f, int64_t nnz, int64_t n_prune) {
  return align_up(rws_layout(out_f, in_f, nnz, n_prune).total, kAlign);
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
  A.newidx = A.pcnt = A.gq = A.bovf = A.n_grown = nullptr;
  A.bc = BucketSet{};
  A.rbits = 0;
  if (cudaMemsetAsync(a.err, 0, sizeof(uint32_t) * (a.plan ? 3 : 1), s) != cudaSuccess) return SNACK_ERR_CUDA;
  if (a.plan) {
    const RowsBkt L = rows_bkt_layout(a.out_f, a.n_per_row);
    if (L.nb > kBktMaxBuckets || !a.bws || !a.plan->newidx) return SNACK_ERR_INVALID_ARG;
    A.rbits = bits_for((uint64_t)(a.out_f - 1));
    A.bc = rows_buckets(L, a.bws, a.in_f, A.rbits);
    A.newidx = a.plan->newidx;
    A.pcnt = a.plan->cv_pcnt;
    A.gq = a.plan->gq;
    A.bovf = a.err + 1;
    A.n_grown = a.err + 2;
    if (cudaMemsetAsync(A.bc.cnt, 0, sizeof(uint32_t) * (size_t)L.nb * kCntStride, s) != cudaSuccess ||
        cudaMemsetAsync(A.pcnt, 0, sizeof(uint32_t) * (size_t)a.in_f, s) != cudaSuccess)
      return SNACK_ERR_CUDA;
  }
  const unsigned grid = (unsigned)((a.out_f + kRowsWarps - 1) / kRowsWarps);
  if (a.val_t == SNACK_BF16)
    launch_pdl(k_restructure_rows<bf16>, grid, kRowsWarps * 32, 0, s, A);
  else
    launch_pdl(k_restructure_rows<float>, grid, kRowsWarps * 32, 0, s, A);
  if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  return SNACK_OK;
}

snack_status run_restructure(const RestructureArgs &a, void *ws, size_t ws_bytes, cudaStream_t s, bool *updated) {
  if (a.val_t == SNACK_BF16) return restructure_impl<bf16>(a, ws, ws_bytes, s, updated);
  return restructure_impl<float>(a, ws, ws_bytes, s, updated);
}

}  // namespace snack
