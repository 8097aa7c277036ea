// Backward preprocessing: expand, radix sort, run-length encode, classify.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Backward:
// invert 'which rows did this sample use?'": transposition, sorting and
// run-length encoding turn the bags' lookups into runs, one per unique
// (table,row), listing the samples that touched it; section "Fewer reads and
// synchronizations can beat more parallel work": the number of long runs is
// known only on the device, so task lists are compacted on the GPU and later
// kernels read the counts from device memory (never copied to the host).
// "HugeCTR DistributedSlotSparseEmbeddingHash backward" (eqicode.com),
// steps 1-4: expand each lookup's sample id, radix-sort (row, sample) pairs
// over only the bits the row range needs (end_bit), flag run starts, prefix-
// sum the flags and scatter run starts with a sentinel entry.
//
// GB300 design:
//  * keys are 32-bit linear keys hash_base[t] + row (the index range of every
//    supported problem is below 2^32); values are the bag b within its table;
//    per-sample weights ride along as a second value.
//  * LSD radix sort over ceil(log2(total_E+1)) bits in passes of at most 9
//    bits.  Each pass is reduce-then-scan over persistent CTAs that own
//    contiguous tile ranges: a digit histogram per CTA, one scan, then a
//    downsweep that ranks every 4096-key tile stably in shared memory
//    (warp match + per-warp digit counters) and writes each digit's keys as
//    one contiguous segment, so global stores stay coalesced.
//  * invalid lookups get the key total_E and sort after every valid key.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace tbe {
namespace {

constexpr int kRleThreads = 256;
constexpr int kRleItems = 8;
constexpr int kRleTile = kRleThreads * kRleItems;

// ------------------------------------------------------------------ expand
// One CTA per tile of kHotTileBags consecutive bags of one table.  A lookup
// whose row is in the table's hot set adds its weight (1 without per-sample
// weights) to the bag's histogram row; every other valid lookup is cold and
// goes to the sort.  Out-of-range lookups go nowhere.  Without per-sample
// weights a bag's row is stored as bytes (hot_hist8) while no count exceeds
// 255; a tile with any larger count, and every tile with per-sample weights,
// is wide: all its bags get fp32 rows (hot_hist) with per-bag scales.  The
// tile's kind (bytes, wide, or no hot rows) goes to tile_kind.
// Pass 1 (count) fills the histogram and counts cold lookups per bag and per
// tile; a scan of the tile counts gives each tile's first sort position;
// pass 2 (write) writes the cold lookups in position order, so the sort's
// input order, and hence its stability, is the lookup order.

// Hot-set membership: the two-choice hash of the table's hot keys (see
// kCuckooHalf); entry = key | slot << 32, empty = kEmptyKey.
constexpr uint64_t kEmptyEntry = kEmptyKey;

struct HotHash {
  uint64_t e[kCuckooSize];
};

// The table's hot set as the kernels read it.
struct HotSet {
  const uint32_t* keys;   // [T][kHot]
  const uint32_t* place;  // [T][kHot]
  const uint32_t* n;      // [T]
  const uint32_t* m1;     // [T]
  const uint32_t* m2;     // [T]
};

// Slot of `key` in the hot set, or -1.
__device__ __forceinline__ int hot_lookup(const HotHash& h, uint32_t m1, uint32_t m2,
                                          uint32_t key) {
  const uint64_t e1 = h.e[cuckoo_h1(key, m1)];
  const uint64_t e2 = h.e[cuckoo_h2(key, m2)];
  return static_cast<uint32_t>(e1) == key   ? static_cast<int>(e1 >> 32)
         : static_cast<uint32_t>(e2) == key ? static_cast<int>(e2 >> 32)
                                            : -1;
}

struct TileInfo {
  int t;
  int64_t b0;
  int nbags;
};

__device__ __forceinline__ TileInfo tile_info(int B) {
  const int64_t per_table = (B + kHotTileBags - 1) / kHotTileBags;
  TileInfo ti;
  ti.t = static_cast<int>(blockIdx.x / per_table);
  ti.b0 = (blockIdx.x % per_table) * kHotTileBags;
  ti.nbags = static_cast<int>(B - ti.b0 < kHotTileBags ? B - ti.b0 : kHotTileBags);
  return ti;
}

// The tile's nbags + 1 offsets, clamped to [0, n], into shared memory (one
// coalesced load per CTA instead of a dependent load at every bag); bag lb
// of the tile then spans [off[lb], max(off[lb + 1], off[lb])), as bag_range
// gives.  The caller synchronises before reading them.
template <typename IndexT>
__device__ __forceinline__ void load_tile_offsets(const IndexT* offsets, const TileInfo& ti, int B,
                                                  int64_t n, int64_t* off) {
  for (int i = threadIdx.x; i <= ti.nbags; i += blockDim.x) {
    const int64_t v = load_index(offsets, static_cast<int64_t>(ti.t) * B + ti.b0 + i);
    off[i] = v < 0 ? 0 : (v > n ? n : v);
  }
}

// Builds the hash of table t's hot set (empty when the histogram is disabled
// or the table is too wide for the hot path); returns the number of hot
// slots.  Contains __syncthreads.
__device__ int build_hot_hash(HotHash& h, uint32_t* m1, uint32_t* m2, const HotSet& hs,
                              const int64_t* D_offsets, int64_t h0, int64_t E, int t,
                              bool enabled) {
  int nh = 0;
  if (enabled) {
    const int D = static_cast<int>(__ldg(D_offsets + t + 1) - __ldg(D_offsets + t));
    nh = D <= kHotMaxD ? static_cast<int>(min(hs.n[t], static_cast<uint32_t>(kHot))) : 0;
  }
  for (int i = threadIdx.x; i < kCuckooSize; i += blockDim.x) h.e[i] = kEmptyEntry;
  __syncthreads();
  for (int slot = threadIdx.x; slot < nh; slot += blockDim.x) {
    // a key outside the table (a workspace last used for other tables) or a
    // place outside the hash is left out: its slot stays empty
    const uint32_t key = hs.keys[t * kHot + slot];
    const uint32_t at = hs.place[t * kHot + slot];
    if (key >= h0 && key < h0 + E && at < static_cast<uint32_t>(kCuckooSize))
      h.e[at] = key | (static_cast<uint64_t>(slot) << 32);
  }
  *m1 = hs.m1[t];
  *m2 = hs.m2[t];
  __syncthreads();
  return nh;
}

// Per-bag exponent of an fp32 histogram row: the row's largest magnitude
// times 2^scale lands in [2^14, 2^15).
__device__ __forceinline__ int8_t bag_scale(float peak) {
  int sc = 0;
  if (peak > 0.f) sc = 14 - ilogbf(peak);
  return static_cast<int8_t>(sc < -126 ? -126 : (sc > 126 ? 126 : sc));
}

// Histogram slots written per bag: nh rounded up to the 64-slot MMA chunk.
__device__ __forceinline__ int hot_slots_padded(int nh) { return (nh + 63) & ~63; }

template <typename IndexT, bool kWeighted>
struct ExpandSmem {
  HotHash hash;
  int64_t bag_off[kHotTileBags + 1];  // the tile's offsets, clamped to [0, n]
  unsigned long long warp_cold[8];
  uint32_t wide_bags[kHotTileBags / 32];  // bit lb: bag lb has an fp32 row
  uint32_t slot_cnt[kHot];
  // the bag each warp is on: per-slot weight (exact sums: integer counts, or
  // fp32 weights summed in double, so the result does not depend on atomic
  // order) and, weighted, per-slot lookups
  alignas(16) typename std::conditional<kWeighted, double, uint32_t>::type row[8][kHot];
  uint32_t cnt_row[kWeighted ? 8 : 1][kWeighted ? kHot : 1];
};

#ifndef TBE_EXPAND_LOADS
#define TBE_EXPAND_LOADS 8
#endif
constexpr int kExpandLoads = TBE_EXPAND_LOADS;  // index loads in flight per lane
// Unweighted lookups of a table's first kTopVoteSlots hot slots (the set is
// ordered by lookups, so these are its most looked-up rows: about 60 % of
// the hot lookups under Zipf(1.4) for four slots) can be counted by one warp
// vote per slot instead of shared atomics that many lanes of a warp aim at
// the same counter.  Off: on GB300 the votes cost more than the contention
// they remove (hot-row preprocess 0.83 ms without, 0.95 ms with four slots,
// 1.05 ms with eight).
#ifndef TBE_TOP_VOTE_SLOTS
#define TBE_TOP_VOTE_SLOTS 0
#endif
constexpr int kTopVoteSlots = TBE_TOP_VOTE_SLOTS;

template <typename IndexT, bool kWeighted>
__global__ void __launch_bounds__(256)
    expand_count_kernel(const IndexT* __restrict__ indices, const IndexT* __restrict__ offsets,
                        const float* __restrict__ psw, const int64_t* __restrict__ hash_base,
                        const int64_t* __restrict__ D_offsets, int64_t n, int B, HotSet hs,
                        uint8_t* __restrict__ hot_hist8, float* __restrict__ hot_hist,
                        int8_t* __restrict__ hot_scale, uint8_t* __restrict__ tile_kind,
                        uint32_t* __restrict__ hot_cnt, uint32_t* __restrict__ bag_cold,
                        uint32_t* __restrict__ tile_cold, uint32_t* __restrict__ sp_keys,
                        float* __restrict__ sp_psw, int* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ExpandSmem<IndexT, kWeighted>& sm = *reinterpret_cast<ExpandSmem<IndexT, kWeighted>*>(smem_raw);
  const TileInfo ti = tile_info(B);
  const int warp = threadIdx.x >> 5;
  const unsigned lane = lane_id();
  for (int i = threadIdx.x; i < 8 * kHot; i += blockDim.x) {
    sm.row[i / kHot][i % kHot] = 0;
    if constexpr (kWeighted) sm.cnt_row[i / kHot][i % kHot] = 0;
  }
  for (int i = threadIdx.x; i < kHot; i += blockDim.x) sm.slot_cnt[i] = 0;
  if (threadIdx.x < kHotTileBags / 32) sm.wide_bags[threadIdx.x] = 0;
  load_tile_offsets(offsets, ti, B, n, sm.bag_off);  // read after build_hot_hash's barriers
  const int64_t h0 = __ldg(hash_base + ti.t);
  const int64_t E = __ldg(hash_base + ti.t + 1) - h0;
  uint32_t m1, m2;
  const int nh = build_hot_hash(sm.hash, &m1, &m2, hs, D_offsets, h0, E, ti.t,
                                hot_hist != nullptr);
  const int nh_pad = hot_slots_padded(nh);
  constexpr int kPerLane = kHot / 32;
  static_assert(kPerLane == 8, "byte rows: eight slots per lane");
  // lookups of this lane's slots over the tile: slots l, l + 32, ... with
  // per-sample weights, slots 8 l .. 8 l + 7 without
  uint32_t cnt[kPerLane];
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) cnt[j] = 0;
  bool bad = false;
  // this warp's cold lookups over its bags: 64-bit, because bags of malformed
  // (overlapping) offsets can together hold more than n lookups
  unsigned long long cold_w = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int lb = warp; lb < ti.nbags; lb += 8) {
    const int64_t bag = static_cast<int64_t>(ti.t) * B + ti.b0 + lb;
    const int64_t s = sm.bag_off[lb];
    const int64_t e = sm.bag_off[lb + 1] > s ? sm.bag_off[lb + 1] : s;
    uint32_t cold = 0;  // this bag's cold lookups so far (the same in every lane)
    uint32_t top[kTopVoteSlots > 0 ? kTopVoteSlots : 1];  // votes of the first slots (uniform)
#pragma unroll
    for (int j = 0; j < kTopVoteSlots; ++j) top[j] = 0;
    // 32-bit arithmetic relative to the bag's start (a bag holds fewer than
    // 2^32 lookups, and keys are below 2^32): the lane's position o, the
    // sparse-list position `cold + ...`, the key h0 + row
    const uint32_t len = static_cast<uint32_t>(e - s);
    const IndexT* __restrict__ ib = indices + s;
    const float* __restrict__ pb = kWeighted ? psw + s : nullptr;
    uint32_t* __restrict__ kb = sp_keys + s;
    float* __restrict__ wb = kWeighted ? sp_psw + s : nullptr;
    const uint32_t h0_32 = static_cast<uint32_t>(h0);
    for (uint32_t base = 0; base < len; base += 32 * kExpandLoads) {
      IndexT r[kExpandLoads];
#pragma unroll
      for (int u = 0; u < kExpandLoads; ++u) {
        const uint32_t o = base + u * 32 + lane;
        r[u] = o < len ? __ldg(ib + o) : IndexT(0);
      }
#pragma unroll
      for (int u = 0; u < kExpandLoads; ++u) {
        if (base + u * 32 >= len) break;  // warp-uniform
        const uint32_t o = base + u * 32 + lane;
        const bool inside = o < len;
        // a row outside [0, E) (negative ones too, as unsigned) is skipped
        const bool ok = inside && static_cast<uint64_t>(static_cast<int64_t>(r[u])) <
                                      static_cast<uint64_t>(E);
        bad |= inside && !ok;
        const uint32_t key = h0_32 + static_cast<uint32_t>(r[u]);
        // the probe is always in bounds and finds nothing in an empty set
        // (every entry then holds kEmptyKey, never a key): no branch
        const int hit = hot_lookup(sm.hash, m1, m2, key);
        const int slot = ok ? hit : -1;
        // cold lookups go, in lookup order, to the front of the bag's own
        // range [s, e) of the sparse list
        const bool is_cold = ok && slot < 0;
        const unsigned cm = __ballot_sync(kFull, is_cold);
        if (is_cold) {  // the bag of each entry is its range's: expand_write adds it
          const uint32_t at = cold + __popc(cm & lt);
          kb[at] = key;
          if (kWeighted) wb[at] = __ldg(pb + o);
        }
        cold += __popc(cm);
        if constexpr (kWeighted) {
          // double sums of fp32 weights are exact: atomic order does not matter
          if (slot >= 0) {
            atomicAdd(&sm.row[warp][slot], static_cast<double>(__ldg(pb + o)));
            atomicAdd(&sm.cnt_row[warp][slot], 1u);
          }
        } else {
          // the first slots by votes; the rest one shared atomic per hot
          // lookup (lanes on the same row are merged by the shared-memory
          // unit, which measured faster than combining them first with a
          // warp match)
#pragma unroll
          for (int j = 0; j < kTopVoteSlots; ++j) top[j] += __popc(__ballot_sync(kFull, slot == j));
          if (slot >= kTopVoteSlots) atomicAdd(&sm.row[warp][slot], 1u);
        }
      }
    }
    if (lane == 0) bag_cold[bag] = cold;
    cold_w += cold;
    if (nh_pad) {
      // flush the bag's row: histogram entries, per-bag scale, slot counts
      __syncwarp();
      float* dst = hot_hist + bag * kHot;
      if constexpr (kWeighted) {
        float peak = 0.f;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
          const int slot = lane + 32 * j;
          if (slot < nh_pad) {
            const float f = static_cast<float>(sm.row[warp][slot]);
            dst[slot] = f;
            peak = fmaxf(peak, fabsf(f));
            cnt[j] += sm.cnt_row[warp][slot];
            sm.cnt_row[warp][slot] = 0;
            sm.row[warp][slot] = 0;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) peak = fmaxf(peak, __shfl_xor_sync(kFull, peak, o));
        if (lane == 0) hot_scale[bag] = bag_scale(peak);
      } else {
        // the voted slots join the row (only this warp writes it)
        if (lane == 0)
#pragma unroll
          for (int j = 0; j < kTopVoteSlots; ++j) sm.row[warp][j] = top[j];
        __syncwarp();
        // lane l: slots 8 l .. 8 l + 7 (two 16-byte shared loads)
        uint4* rw = reinterpret_cast<uint4*>(&sm.row[warp][8 * lane]);
        const uint4 q0 = rw[0], q1 = rw[1];
        rw[0] = make_uint4(0u, 0u, 0u, 0u);
        rw[1] = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t v[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint32_t peak = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          cnt[k] += v[k];
          peak = max(peak, v[k]);
        }
        peak = __reduce_max_sync(kFull, peak);
        if (peak <= 255u) {
          // slots past nh hold zeros: the whole 256-byte row is written
          uint2 packed;
          packed.x = v[0] | (v[1] << 8) | (v[2] << 16) | (v[3] << 24);
          packed.y = v[4] | (v[5] << 8) | (v[6] << 16) | (v[7] << 24);
          *reinterpret_cast<uint2*>(hot_hist8 + bag * kHot + 8 * lane) = packed;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (8 * lane + k < nh_pad) dst[8 * lane + k] = static_cast<float>(v[k]);
          if (lane == 0) {
            hot_scale[bag] = bag_scale(static_cast<float>(peak));
            atomicOr(&sm.wide_bags[lb >> 5], 1u << (lb & 31));
          }
        }
      }
      __syncwarp();
    }
  }
  if (lane == 0) sm.warp_cold[warp] = cold_w;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j)
    if (cnt[j]) atomicAdd(&sm.slot_cnt[kWeighted ? lane + 32 * j : 8 * lane + j], cnt[j]);
  __syncthreads();
  if (threadIdx.x == 0) {
    // saturated at n: with well-formed offsets the tile holds at most n cold
    // lookups; overlapping bags may count more, and only the first n of all
    // cold lookups are kept (see capped_scan_kernel)
    unsigned long long c = 0;
    for (int w = 0; w < 8; ++w) c += sm.warp_cold[w];
    tile_cold[blockIdx.x] = static_cast<uint32_t>(c < static_cast<unsigned long long>(n) ? c : n);
  }
  if (nh_pad) {
    bool wide = kWeighted;
#pragma unroll
    for (int i = 0; i < kHotTileBags / 32; ++i) wide |= sm.wide_bags[i] != 0;
    if (!kWeighted && wide) {
      // a wide tile is read as fp32 rows only: the byte rows written above
      // (this CTA's own global writes, visible after the barrier) become
      // fp32 rows with scale 0 (counts of at most 255 are exact as they are)
      for (int lb = warp; lb < ti.nbags; lb += 8) {
        if ((sm.wide_bags[lb >> 5] >> (lb & 31)) & 1u) continue;
        const int64_t bag = static_cast<int64_t>(ti.t) * B + ti.b0 + lb;
        for (int slot = lane; slot < nh_pad; slot += 32)
          hot_hist[bag * kHot + slot] = static_cast<float>(hot_hist8[bag * kHot + slot]);
        if (lane == 0) hot_scale[bag] = 0;
      }
    }
    if (threadIdx.x == 0) tile_kind[blockIdx.x] = wide ? kTileWide : kTileBytes;
  } else if (hot_hist != nullptr && threadIdx.x == 0) {
    tile_kind[blockIdx.x] = kTileNoHot;
  }
  for (int i = threadIdx.x; i < nh; i += blockDim.x)
    if (sm.slot_cnt[i]) atomicAdd(&hot_cnt[ti.t * kHot + i], sm.slot_cnt[i]);
  if (status && __any_sync(kFull, bad) && lane == 0) set_status(status, TBE_ERR_INDEX_RANGE);
}

// Compaction of the cold lookups: each bag's cold keys, which the count
// kernel left at the front of the bag's own range of the sparse list, move to
// the dense list at the bag's first cold entry (tile base + in-tile prefix of
// the per-bag counts), keeping lookup order, each with its bag (the range's
// own, so the sparse list holds no bags); cold_off gets each bag's first
// entry.  Only the cold entries are read, not the indices.
template <typename IndexT, bool kWeighted>
__global__ void __launch_bounds__(256)
    expand_write_kernel(const IndexT* __restrict__ offsets, int64_t n, int B,
                        const uint32_t* __restrict__ bag_cold,
                        const uint32_t* __restrict__ tile_base, uint32_t* __restrict__ cold_off,
                        const uint32_t* __restrict__ sp_keys,
                        const float* __restrict__ sp_psw, uint32_t* __restrict__ keys,
                        uint32_t* __restrict__ vals, float* __restrict__ psw_out) {
  __shared__ uint32_t rel[kHotTileBags + 1];  // each bag's first entry relative to the tile's
  __shared__ unsigned long long scan[33];
  __shared__ int64_t bag_off[kHotTileBags + 1];
  const TileInfo ti = tile_info(B);
  load_tile_offsets(offsets, ti, B, n, bag_off);  // read after the scan's barriers
  unsigned long long tile_total = 0;
  {
    // exclusive prefix of the tile's per-bag cold counts = the bags' first
    // entries in the dense list.  In 64 bits and capped at n: with
    // well-formed offsets no cap applies; bags of malformed (overlapping)
    // offsets can hold more than n cold lookups in all, and then only
    // positions below n are written (every one of them, since positions are
    // a dense prefix), so the dense list never leaves its n entries.
    const int lb = threadIdx.x;
    const unsigned long long c =
        lb < ti.nbags ? bag_cold[static_cast<int64_t>(ti.t) * B + ti.b0 + lb] : 0ull;
    unsigned long long total;
    const unsigned long long inc = block_inclusive_scan(c, OpSum(), 0ull, scan, &total);
    const unsigned long long cap = static_cast<unsigned long long>(n);
    const unsigned long long first = tile_base[blockIdx.x] + inc - c;
    const uint32_t first_c = static_cast<uint32_t>(first < cap ? first : cap);
    // relative starts saturate at 2^32 - 1: the entries copied below lie
    // below n - tile base < 2^32, where the saturated values still order them
    const unsigned long long r = inc - c;
    if (lb < kHotTileBags) rel[lb] = static_cast<uint32_t>(r < 0xffffffffull ? r : 0xffffffffull);
    if (lb < ti.nbags) cold_off[static_cast<int64_t>(ti.t) * B + ti.b0 + lb] = first_c;
    tile_total = total;
    if (lb == 0 && blockIdx.x == gridDim.x - 1) {
      const unsigned long long last = tile_base[blockIdx.x] + total;
      cold_off[static_cast<int64_t>(ti.t) * B + ti.b0 + ti.nbags] =
          static_cast<uint32_t>(last < cap ? last : cap);
    }
  }
  __syncthreads();
  // The tile's entries as one dense range, the threads striding over it
  // (a bag holds about as many cold entries as a warp has lanes, so a
  // warp per bag left lanes idle and waited on each bag's loads in turn).
  // Entry i belongs to the last bag whose relative start is at most i;
  // entries at or past n are dropped (malformed offsets only; see above).
  const unsigned long long tb = tile_base[blockIdx.x];
  const unsigned long long un = static_cast<unsigned long long>(n);
  const unsigned long long room = tb < un ? un - tb : 0ull;
  const uint32_t lim = static_cast<uint32_t>(tile_total < room ? tile_total : room);
  const uint64_t pos0 = tb;
#pragma unroll 4
  for (uint32_t i = threadIdx.x; i < lim; i += blockDim.x) {
    int lo = 0, hi = ti.nbags - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rel[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int64_t src = bag_off[lo] + static_cast<int64_t>(i - rel[lo]);
    keys[pos0 + i] = __ldg(sp_keys + src);
    vals[pos0 + i] = static_cast<uint32_t>(ti.b0 + lo);
    if (kWeighted) psw_out[pos0 + i] = __ldg(sp_psw + src);
  }
}

// One CTA per array (blockIdx.x = k): exclusive scan in place of the
// classify blocks' totals blk[k][0 .. nblk) and the array's total into
// counters[dest[k]] (medium runs, long runs, chunks, tree nodes).
struct ScanDests {
  int d[4];
};
__global__ void __launch_bounds__(1024)
    block_totals_scan_kernel(uint32_t* __restrict__ blk, int nblk, uint32_t* counters,
                             ScanDests dest) {
  __shared__ uint32_t sm[33];
  uint32_t* data = blk + static_cast<int64_t>(blockIdx.x) * nblk;
  const int per = (nblk + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
  const int b = static_cast<int>(threadIdx.x) * per;
  const int e = b + per < nblk ? b + per : nblk;
  uint32_t s = 0;
  for (int i = b; i < e; ++i) s += data[i];
  uint32_t agg;
  const uint32_t inc = block_inclusive_scan(s, OpSum(), 0u, sm, &agg);
  uint32_t run = inc - s;
  for (int i = b; i < e; ++i) {
    const uint32_t v = data[i];
    data[i] = run;
    run += v;
  }
  if (threadIdx.x == 0) counters[dest.d[blockIdx.x]] = agg;
}

// Single CTA: exclusive scan of the expand tiles' cold counts in place,
// capped at `cap` (= n): entry i becomes min(sum of the counts before i, cap)
// and *sum_out min(sum of all, cap), the number of entries the sort takes.
// Sums are formed in 64 bits, so counts of malformed offsets cannot wrap.
__global__ void __launch_bounds__(1024)
    capped_scan_kernel(uint32_t* __restrict__ data, int64_t total, uint32_t cap,
                       uint32_t* sum_out) {
  __shared__ unsigned long long sm[33];
  const int64_t per = (total + blockDim.x - 1) / blockDim.x;
  const int64_t b = threadIdx.x * per;
  const int64_t e = b + per < total ? b + per : total;
  unsigned long long s = 0;
  for (int64_t i = b; i < e; ++i) s += data[i];
  unsigned long long agg;
  const unsigned long long inc = block_inclusive_scan(s, OpSum(), 0ull, sm, &agg);
  unsigned long long run = inc - s;
  for (int64_t i = b; i < e; ++i) {
    const uint32_t v = data[i];
    data[i] = static_cast<uint32_t>(run < cap ? run : cap);
    run += v;
  }
  if (threadIdx.x == 0) *sum_out = static_cast<uint32_t>(agg < cap ? agg : cap);
}

// -------------------------------------------------------------- radix sort
// Persistent CTAs over the sorted range.  The number of entries is read from
// device memory (counters[kCntSortN]), so it can be decided on the device;
// the grid is sized on the host from an upper bound.
struct SortGeom {
  int ctas;              // persistent CTAs
  const uint32_t* n_dev; // entries to process
};

__device__ __forceinline__ int64_t geom_n(const SortGeom& g) { return static_cast<int64_t>(*g.n_dev); }

// Tile range of this CTA: contiguous kSortTile-key tiles, split evenly.
__device__ __forceinline__ void cta_range(const SortGeom& g, int64_t n, int64_t* b, int64_t* e) {
  const int64_t tiles = (n + kSortTile - 1) / kSortTile;
  const int64_t per_cta = (tiles + g.ctas - 1) / g.ctas;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * per_cta;
  const int64_t t1 = t0 + per_cta < tiles ? t0 + per_cta : tiles;
  *b = t0 * kSortTile;
  *e = t1 * kSortTile < n ? t1 * kSortTile : n;
  if (*b > n) *b = n;
}

// Per-CTA digit histogram; counts stored CTA-major: counts[cta * 2^width + d].
__global__ void __launch_bounds__(kSortThreads)
    radix_upsweep_kernel(const uint32_t* __restrict__ keys, SortGeom g, int shift,
                         int width, uint32_t* __restrict__ counts) {
  const int64_t n = geom_n(g);
  __shared__ uint32_t hist[kSortThreads / 32][1 << kMaxRadixBits];
  const int nd = 1 << width;
  const uint32_t mask = static_cast<uint32_t>(nd - 1);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kSortThreads / 32) * nd; i += kSortThreads)
    hist[i / nd][i % nd] = 0;
  __syncthreads();
  int64_t b, e;
  cta_range(g, n, &b, &e);
  // b is a multiple of the tile size, hence 16-byte aligned.
  int64_t i = b + static_cast<int64_t>(threadIdx.x) * 4;
  for (; i + 3 < e; i += kSortThreads * 4) {
    const uint4 k = __ldg(reinterpret_cast<const uint4*>(keys + i));
    atomicAdd(&hist[warp][(k.x >> shift) & mask], 1u);
    atomicAdd(&hist[warp][(k.y >> shift) & mask], 1u);
    atomicAdd(&hist[warp][(k.z >> shift) & mask], 1u);
    atomicAdd(&hist[warp][(k.w >> shift) & mask], 1u);
  }
  for (; i < e; ++i) atomicAdd(&hist[warp][(__ldg(keys + i) >> shift) & mask], 1u);
  __syncthreads();
  for (int d = threadIdx.x; d < nd; d += kSortThreads) {
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < kSortThreads / 32; ++w) s += hist[w][d];
    counts[static_cast<int64_t>(blockIdx.x) * nd + d] = s;
  }
}

// Output position of every (digit, CTA) in digit-major order: for digit d and
// CTA c, the keys of smaller digits plus the keys of digit d in CTAs before c.
// One CTA, one thread per digit walking the CTAs (loads are coalesced across
// threads), then a scan of the digit totals.  In place on counts[c][d].
// Digit-parallel scan of the upsweep's counts: one warp per digit d turns
// counts[c][d] into the exclusive prefix over CTAs c of digit d and writes the
// digit's total to totals[d]; the downsweep adds the exclusive prefix of the
// totals over digits (its digit base).  Lane l owns CTAs [l k, (l + 1) k).
constexpr int kScanPerLane = kMaxSortCtas / 32;

__global__ void __launch_bounds__(256)
    radix_scan_kernel(uint32_t* __restrict__ counts, int ctas, int nd,
                      uint32_t* __restrict__ totals) {
  const int d = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (d >= nd) return;  // warp-uniform
  const int lane = static_cast<int>(lane_id());
  const int k = (ctas + 31) / 32;
  uint32_t v[kScanPerLane];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < kScanPerLane; ++j) {
    const int c = lane * k + j;
    v[j] = (j < k && c < ctas) ? counts[static_cast<int64_t>(c) * nd + d] : 0u;
    sum += v[j];
  }
  const uint32_t inc = warp_inclusive_scan(sum, OpSum());
  uint32_t run = inc - sum;
#pragma unroll
  for (int j = 0; j < kScanPerLane; ++j) {
    const int c = lane * k + j;
    if (j < k && c < ctas) counts[static_cast<int64_t>(c) * nd + d] = run;
    run += v[j];
  }
  if (lane == 31) totals[d] = inc;
}

// Single CTA: exclusive scan over `total` counts in place (digit-major order
// yields, for each (digit, cta), the first output position of that CTA's keys
// of that digit).  Optionally writes the grand total to *sum_out.
__global__ void __launch_bounds__(1024)
    exclusive_scan_kernel(uint32_t* __restrict__ data, int64_t total, uint32_t* sum_out) {
  __shared__ uint32_t sm[33];
  const int64_t per = (total + blockDim.x - 1) / blockDim.x;
  const int64_t b = threadIdx.x * per;
  const int64_t e = b + per < total ? b + per : total;
  uint32_t s = 0;
  for (int64_t i = b; i < e; ++i) s += data[i];
  uint32_t agg;
  const uint32_t inc = block_inclusive_scan(s, OpSum(), 0u, sm, &agg);
  uint32_t run = inc - s;
  for (int64_t i = b; i < e; ++i) {
    const uint32_t v = data[i];
    data[i] = run;
    run += v;
  }
  if (sum_out && threadIdx.x == 0) *sum_out = agg;
}

template <bool kWeighted>
struct DownSmem {
  // Two tile buffers: one being loaded while the other is ranked, permuted
  // in place into digit order and written out.
  uint32_t keys[2][kSortTile];
  uint32_t vals[2][kSortTile];
  float psw[2][kWeighted ? kSortTile : 4];
  uint32_t run_off[1 << kMaxRadixBits];  // next output position per digit
  uint32_t tile_cnt[1 << kMaxRadixBits];
  uint32_t tile_start[1 << kMaxRadixBits];
  uint32_t wcnt[kSortThreads / 32][1 << kMaxRadixBits];
  uint32_t scan[33];
};

// Queue the copies of tile [tb, tb + valid) into buffer `buf`.
template <bool kWeighted>
__device__ __forceinline__ void load_tile_async(DownSmem<kWeighted>& sm, int buf,
                                                const uint32_t* keys_in, const uint32_t* vals_in,
                                                const float* psw_in, int64_t tb, int valid) {
  for (int c = threadIdx.x; c < kSortTile / 4; c += kSortThreads) {
    const int rem = valid - 4 * c;
    const int bytes = rem >= 4 ? 16 : (rem > 0 ? rem * 4 : 0);
    const int64_t src = rem > 0 ? tb + 4 * c : 0;  // no global read when bytes == 0
    cp_async16(&sm.keys[buf][4 * c], keys_in + src, bytes);
    cp_async16(&sm.vals[buf][4 * c], vals_in + src, bytes);
    if (kWeighted) cp_async16(&sm.psw[buf][4 * c], psw_in + src, bytes);
  }
}

template <bool kWeighted>
__global__ void __launch_bounds__(kSortThreads, 2)
    radix_downsweep_kernel(const uint32_t* __restrict__ keys_in,
                           const uint32_t* __restrict__ vals_in,
                           const float* __restrict__ psw_in, uint32_t* __restrict__ keys_out,
                           uint32_t* __restrict__ vals_out, float* __restrict__ psw_out,
                           SortGeom g, int shift, int width,
                           const uint32_t* __restrict__ counts,
                           const uint32_t* __restrict__ totals) {
  const int64_t n = geom_n(g);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  DownSmem<kWeighted>& sm = *reinterpret_cast<DownSmem<kWeighted>*>(smem_raw);
  const int nd = 1 << width;
  const uint32_t mask = static_cast<uint32_t>(nd - 1);
  const int warp = threadIdx.x >> 5;
  const unsigned lane = lane_id();
  const unsigned lt_mask = (1u << lane) - 1u;
  {
    // output start of each digit: the digit's base (exclusive prefix of the
    // digit totals) plus this CTA's prefix within the digit
    const int d0 = threadIdx.x * 2;
    const uint32_t t0 = d0 < nd ? totals[d0] : 0u;
    const uint32_t t1 = d0 + 1 < nd ? totals[d0 + 1] : 0u;
    const uint32_t inc = block_inclusive_scan(t0 + t1, OpSum(), 0u, sm.scan);
    if (d0 < nd) sm.run_off[d0] = inc - t0 - t1 + counts[static_cast<int64_t>(blockIdx.x) * nd + d0];
    if (d0 + 1 < nd)
      sm.run_off[d0 + 1] = inc - t1 + counts[static_cast<int64_t>(blockIdx.x) * nd + d0 + 1];
  }
  int64_t b, e;
  cta_range(g, n, &b, &e);
  if (b < e) {
    load_tile_async(sm, 0, keys_in, vals_in, psw_in, b,
                    static_cast<int>(e - b < kSortTile ? e - b : kSortTile));
  }
  cp_async_commit();

  int cur = 0;
  for (int64_t tb = b; tb < e; tb += kSortTile, cur ^= 1) {
    const int valid = static_cast<int>(e - tb < kSortTile ? e - tb : kSortTile);
    const int64_t nb = tb + kSortTile;
    if (nb < e)
      load_tile_async(sm, cur ^ 1, keys_in, vals_in, psw_in, nb,
                      static_cast<int>(e - nb < kSortTile ? e - nb : kSortTile));
    cp_async_commit();
    cp_async_wait<1>();  // this tile's copies are done (the next tile's may still run)
    for (int d = lane; d < nd; d += 32) sm.wcnt[warp][d] = 0;
    __syncthreads();
    // Rank this warp's 512 keys (16 rounds of 32 consecutive keys) stably
    // among keys of the same digit within the warp.
    uint32_t key[kSortItems];
    uint32_t rank[kSortItems / 2];  // two 16-bit ranks per word (a rank is below 512)
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
      const int p = warp * (kSortItems * 32) + r * 32 + static_cast<int>(lane);
      // Keys past the end take the largest digit: they rank after every
      // valid key of the tile and are never written out.
      key[r] = p < valid ? sm.keys[cur][p] : 0xffffffffu;
      const uint32_t d = (key[r] >> shift) & mask;
      const unsigned peers = __match_any_sync(kFull, d);
      // the digit's leader adds the round's count; atomics on one address
      // return in issue order, so the rounds need no barrier between them
      const int leader = 31 - __clz(peers);
      uint32_t old = 0;
      if (static_cast<int>(lane) == leader) old = atomicAdd(&sm.wcnt[warp][d], __popc(peers));
      const uint32_t before = __shfl_sync(kFull, old, leader);
      const uint32_t rk = before + __popc(peers & lt_mask);
      if (r & 1) rank[r >> 1] |= rk << 16; else rank[r >> 1] = rk;
    }
    __syncthreads();
    // Exclusive prefix over warps per digit, and the tile's digit counts.
    for (int d = threadIdx.x; d < nd; d += kSortThreads) {
      uint32_t s = 0;
#pragma unroll
      for (int w = 0; w < kSortThreads / 32; ++w) {
        const uint32_t c = sm.wcnt[w][d];
        sm.wcnt[w][d] = s;
        s += c;
      }
      sm.tile_cnt[d] = s;
    }
    __syncthreads();
    {
      // Exclusive scan of the tile counts over digits (two digits per thread).
      const int d0 = threadIdx.x * 2;
      const uint32_t c0 = d0 < nd ? sm.tile_cnt[d0] : 0u;
      const uint32_t c1 = d0 + 1 < nd ? sm.tile_cnt[d0 + 1] : 0u;
      const uint32_t inc = block_inclusive_scan(c0 + c1, OpSum(), 0u, sm.scan);
      if (d0 < nd) sm.tile_start[d0] = inc - c0 - c1;
      if (d0 + 1 < nd) sm.tile_start[d0 + 1] = inc - c1;
    }
    // Take this thread's values out of the buffer, then write keys and
    // values back in digit order (the block scan above ended on a barrier,
    // and the reads below finish before the barrier that precedes the writes).
    uint32_t val[kSortItems];
    float pw[kWeighted ? kSortItems : 1];
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
      const int p = warp * (kSortItems * 32) + r * 32 + static_cast<int>(lane);
      val[r] = sm.vals[cur][p];
      if (kWeighted) pw[r] = sm.psw[cur][p];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
      const uint32_t d = (key[r] >> shift) & mask;
      const uint32_t pos = sm.tile_start[d] + sm.wcnt[warp][d] +
                           ((rank[r >> 1] >> (16 * (r & 1))) & 0xffffu);
      sm.keys[cur][pos] = key[r];
      sm.vals[cur][pos] = val[r];
      if (kWeighted) sm.psw[cur][pos] = pw[r];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < valid; i += kSortThreads) {
      const uint32_t k = sm.keys[cur][i];
      const uint32_t d = (k >> shift) & mask;
      const uint32_t dst = sm.run_off[d] + (static_cast<uint32_t>(i) - sm.tile_start[d]);
      keys_out[dst] = k;
      vals_out[dst] = sm.vals[cur][i];
      if (kWeighted) psw_out[dst] = sm.psw[cur][i];
    }
    __syncthreads();
    for (int d = threadIdx.x; d < nd; d += kSortThreads) sm.run_off[d] += sm.tile_cnt[d];
    // The next iteration's barrier orders these updates before their use.
  }
  cp_async_wait<0>();
}

// --------------------------------------------------------------------- RLE
// Two levels over the sorted lookups: runs (one per table row) and pairs (the
// lookups of a run from one bag).  Each thread owns kRleItems consecutive
// lookups; the loads of the next tile are issued before the current tile is
// processed.
struct RleItems {
  uint32_t k[kRleItems];
  uint32_t b[kRleItems];
  uint32_t pk, pb;  // the lookup before the first one (lane 0: from memory)
  bool first;       // no lookup before the first one
  bool run_head[kRleItems];
  bool pair_head[kRleItems];
};

// Issue the loads of a thread's kRleItems lookups starting at i0 (and, on
// lane 0, of the lookup before them); rle_heads consumes them later.
__device__ __forceinline__ void rle_load(const uint32_t* __restrict__ keys,
                                         const uint32_t* __restrict__ bags, int64_t i0, int64_t e,
                                         uint32_t sentinel, RleItems& it) {
  if (i0 + kRleItems <= e) {
#pragma unroll
    for (int j = 0; j < kRleItems; j += 4) {
      const uint4 kk = __ldg(reinterpret_cast<const uint4*>(keys + i0 + j));
      const uint4 bb = __ldg(reinterpret_cast<const uint4*>(bags + i0 + j));
      it.k[j] = kk.x; it.k[j + 1] = kk.y; it.k[j + 2] = kk.z; it.k[j + 3] = kk.w;
      it.b[j] = bb.x; it.b[j + 1] = bb.y; it.b[j + 2] = bb.z; it.b[j + 3] = bb.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kRleItems; ++j) {
      const bool in = i0 + j < e;
      it.k[j] = in ? __ldg(keys + i0 + j) : sentinel;
      it.b[j] = in ? __ldg(bags + i0 + j) : 0u;
    }
  }
  it.first = false;
  it.pk = sentinel;
  it.pb = 0;
  if (lane_id() == 0) {
    if (i0 > 0 && i0 - 1 < e) {
      it.pk = __ldg(keys + i0 - 1);
      it.pb = __ldg(bags + i0 - 1);
    } else if (i0 == 0) {
      it.first = true;
    }
  }
}

// A run starts where the key changes (a new table row), a pair where the key
// or the bag changes; lookups with the invalid key start nothing.  The
// lookup before a thread's first one is its neighbour lane's last one.
__device__ __forceinline__ void rle_heads(RleItems& it, uint32_t sentinel) {
  uint32_t pk = __shfl_up_sync(kFull, it.k[kRleItems - 1], 1);
  uint32_t pb = __shfl_up_sync(kFull, it.b[kRleItems - 1], 1);
  bool first = false;
  if (lane_id() == 0) {
    pk = it.pk;
    pb = it.pb;
    first = it.first;
  }
#pragma unroll
  for (int j = 0; j < kRleItems; ++j) {
    const bool valid = it.k[j] < sentinel;
    const bool newkey = first || it.k[j] != pk;
    it.run_head[j] = valid && newkey;
    it.pair_head[j] = valid && (newkey || it.b[j] != pb);
    first = false;
    pk = it.k[j];
    pb = it.b[j];
  }
}

__global__ void __launch_bounds__(kRleThreads)
    rle_count_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ bags,
                     SortGeom g, uint32_t sentinel, uint32_t* __restrict__ cta_runs,
                     uint32_t* __restrict__ cta_pairs) {
  const int64_t n = geom_n(g);
  __shared__ unsigned long long sm[33];
  int64_t b, e;
  cta_range(g, n, &b, &e);
  unsigned long long c = 0;  // runs in the high word, pairs in the low word
  RleItems it, nx;
  if (b < e) rle_load(keys, bags, b + static_cast<int64_t>(threadIdx.x) * kRleItems, e, sentinel, nx);
  for (int64_t tb = b; tb < e; tb += kRleTile) {
    it = nx;
    if (tb + kRleTile < e)  // next tile's loads in flight while this one is counted
      rle_load(keys, bags, tb + kRleTile + static_cast<int64_t>(threadIdx.x) * kRleItems, e,
               sentinel, nx);
    rle_heads(it, sentinel);
#pragma unroll
    for (int j = 0; j < kRleItems; ++j)
      c += (static_cast<unsigned long long>(it.run_head[j]) << 32) | it.pair_head[j];
  }
  unsigned long long total;
  block_inclusive_scan(c, OpSum(), 0ull, sm, &total);
  if (threadIdx.x == 0) {
    cta_runs[blockIdx.x] = static_cast<uint32_t>(total >> 32);
    cta_pairs[blockIdx.x] = static_cast<uint32_t>(total);
  }
}

__global__ void __launch_bounds__(kRleThreads)
    rle_write_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ bags,
                     SortGeom g, uint32_t sentinel,
                     const uint32_t* __restrict__ run_base, const uint32_t* __restrict__ pair_base,
                     uint32_t* __restrict__ unique_keys, uint32_t* __restrict__ run_starts,
                     uint32_t* __restrict__ run_pairs, uint32_t* __restrict__ pair_starts,
                     uint32_t* __restrict__ pair_bags, uint32_t* __restrict__ counters) {
  __shared__ uint32_t sm[33];
  // the tile's pairs and runs, in order, before their coalesced write-out
  __shared__ uint32_t s_pstart[kRleTile], s_pbag[kRleTile];
  __shared__ uint32_t s_ukey[kRleTile], s_rstart[kRleTile], s_rpair[kRleTile];
  const int64_t n = geom_n(g);
  int64_t b, e;
  cta_range(g, n, &b, &e);
  uint32_t r = run_base[blockIdx.x];
  uint32_t p = pair_base[blockIdx.x];
  const uint32_t R = run_base[g.ctas];
  const uint32_t P = pair_base[g.ctas];
  RleItems it, nx;
  if (b < e) rle_load(keys, bags, b + static_cast<int64_t>(threadIdx.x) * kRleItems, e, sentinel, nx);
  for (int64_t tb = b; tb < e; tb += kRleTile) {
    const int64_t i0 = tb + static_cast<int64_t>(threadIdx.x) * kRleItems;
    it = nx;
    if (tb + kRleTile < e)  // next tile's loads in flight while this one is written
      rle_load(keys, bags, i0 + kRleTile, e, sentinel, nx);
    const bool first_here = it.first;
    const uint32_t up_key = __shfl_up_sync(kFull, it.k[kRleItems - 1], 1);  // all lanes
    const uint32_t before_key = lane_id() == 0 ? it.pk : up_key;
    rle_heads(it, sentinel);
    uint32_t c = 0;  // runs << 16 | pairs: at most kRleTile each per tile
#pragma unroll
    for (int j = 0; j < kRleItems; ++j) c += (static_cast<uint32_t>(it.run_head[j]) << 16) | it.pair_head[j];
    uint32_t total;
    const uint32_t inc = block_inclusive_scan(c, OpSum(), 0u, sm, &total);
    const uint32_t exc = inc - c;
    uint32_t rr = exc >> 16;      // within the tile
    uint32_t pp = exc & 0xffffu;
#pragma unroll
    for (int j = 0; j < kRleItems; ++j) {
      const int64_t i = i0 + j;
      if (it.pair_head[j]) {
        s_pstart[pp] = static_cast<uint32_t>(i);
        s_pbag[pp] = it.b[j];
        if (it.run_head[j]) {
          s_ukey[rr] = it.k[j];
          s_rstart[rr] = static_cast<uint32_t>(i);
          s_rpair[rr] = p + pp;
          ++rr;
        }
        ++pp;
      }
      // End of the valid keys: the first invalid key, or the end of the array.
      if (i < e) {
        const bool invalid = it.k[j] >= sentinel;
        const uint32_t prev = j > 0 ? it.k[j - 1] : before_key;
        const bool first_invalid = invalid && ((j == 0 && first_here) || prev < sentinel);
        const bool last_valid = !invalid && i == n - 1;
        if (first_invalid || last_valid) {
          const uint32_t nv = first_invalid ? static_cast<uint32_t>(i) : static_cast<uint32_t>(n);
          run_starts[R] = nv;
          pair_starts[P] = nv;
          run_pairs[R] = P;
          counters[kCntValid] = nv;
        }
      }
    }
    __syncthreads();
    const uint32_t nr = total >> 16, np = total & 0xffffu;
    for (uint32_t k = threadIdx.x; k < np; k += kRleThreads) {
      pair_starts[p + k] = s_pstart[k];
      pair_bags[p + k] = s_pbag[k];
    }
    for (uint32_t k = threadIdx.x; k < nr; k += kRleThreads) {
      unique_keys[r + k] = s_ukey[k];
      run_starts[r + k] = s_rstart[k];
      run_pairs[r + k] = s_rpair[k];
    }
    __syncthreads();  // the staging arrays are rewritten by the next tile
    r += nr;
    p += np;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    counters[kCntRuns] = R;
    counters[kCntPairs] = P;
  }
}

// ---------------------------------------------------------------- classify
// One CTA: first run of every table (binary search of its first key among
// the unique keys) and the prefix of short-run warp tasks per table.
__global__ void __launch_bounds__(1024)
    table_runs_kernel(const uint32_t* __restrict__ unique_keys, const uint32_t* counters,
                      const int64_t* __restrict__ hash_base, const int64_t* __restrict__ D_offsets,
                      int T, uint32_t* __restrict__ table_runs, uint32_t* __restrict__ table_tasks,
                      uint32_t* counters_out) {  // counters and counters_out: the same array
  __shared__ uint32_t sm[33];
  const uint32_t R = counters[kCntRuns];
  for (int t = threadIdx.x; t <= T; t += blockDim.x) {
    const uint32_t target = static_cast<uint32_t>(__ldg(hash_base + t));
    uint32_t lo = 0, hi = R;
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      if (unique_keys[mid] < target) lo = mid + 1; else hi = mid;
    }
    table_runs[t] = t == T ? R : lo;
  }
  __syncthreads();
  uint32_t carry = 0;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    uint32_t c = 0;
    if (t < T) {
      const int D = static_cast<int>(__ldg(D_offsets + t + 1) - __ldg(D_offsets + t));
      const int G = 32 / update_lanes(D >> 2);
      c = (table_runs[t + 1] - table_runs[t] + G - 1) / G;
    }
    uint32_t total;
    const uint32_t inc = block_inclusive_scan(c, OpSum(), 0u, sm, &total);
    if (t < T) table_tasks[t] = carry + inc - c;
    carry += total;
  }
  if (threadIdx.x == 0) {
    table_tasks[T] = carry;
    counters_out[kCntTasks] = carry;
  }
}

// Medium runs (kMediumRun <= pairs < kLongThreshold) and long runs (at least
// kLongThreshold pairs) compacted into lists on the device, each long run
// with a contiguous range of chunk slots and of tree nodes.  Each block takes
// a contiguous range of runs in passes of 256; a pass places its runs by
// block scans.  kMode 0: each pass takes its list ranges with one atomic per
// counter (the lists' order across blocks is arbitrary).  With
// TBE_ORDERED_CLASSIFY the lists follow the run order (table-major, so the
// medium-run kernel works through one table's gradient rows at a time):
// kMode 1 only counts each block's medium runs, long runs, chunks and tree
// nodes into blk[4][grid], an exclusive scan of each turns them into the
// blocks' list bases, and kMode 2 writes the lists from those bases.
#ifndef TBE_ORDERED_CLASSIFY
#define TBE_ORDERED_CLASSIFY 1
#endif
template <int kMode>
__global__ void __launch_bounds__(256)
    classify_kernel(const uint32_t* __restrict__ run_pairs, uint32_t* __restrict__ counters,
                    uint32_t* __restrict__ long_run, uint32_t* __restrict__ long_chunk0,
                    uint32_t* __restrict__ long_tree0, uint32_t* __restrict__ medium_run,
                    uint32_t* __restrict__ blk) {
  __shared__ uint32_t sm32[33];
  __shared__ unsigned long long sm64[33];
  __shared__ uint32_t base[4];
  __shared__ uint32_t run_base[4];  // kMode 1: the block's totals; 2: its next list slots
  if (threadIdx.x < 4)
    run_base[threadIdx.x] = kMode == 2 ? blk[threadIdx.x * gridDim.x + blockIdx.x] : 0u;
  __syncthreads();
  const uint32_t R = counters[kCntRuns];
  const uint32_t per_block = ((R + gridDim.x - 1) / gridDim.x + 255u) & ~255u;
  const uint32_t j0 = blockIdx.x * per_block;
  const uint32_t j1 = j0 + per_block < R ? j0 + per_block : R;
  for (uint32_t jb = j0; jb < j1; jb += 256) {  // uniform over the block
    const uint32_t j = jb + threadIdx.x;
    const uint32_t SL = j < j1 ? run_pairs[j + 1] - run_pairs[j] : 0u;
    const bool medium = SL >= static_cast<uint32_t>(kMediumRun) &&
                        SL < static_cast<uint32_t>(kLongThreshold);
    const bool lng = SL >= static_cast<uint32_t>(kLongThreshold);
    const uint32_t nch = lng ? (SL + kChunk - 1) / kChunk : 0u;
    const uint32_t nodes = lng ? static_cast<uint32_t>(tree_nodes(nch)) : 0u;
    // medium count in the low half, long count in the high half (<= 256 each)
    const uint32_t f = (medium ? 1u : 0u) | (lng ? 1u << 16 : 0u);
    uint32_t ftot;
    const uint32_t fex = block_inclusive_scan(f, OpSum(), 0u, sm32, &ftot) - f;
    const unsigned long long c = nch | (static_cast<unsigned long long>(nodes) << 32);
    unsigned long long ctot;
    const unsigned long long cex = block_inclusive_scan(c, OpSum(), 0ull, sm64, &ctot) - c;
    if (threadIdx.x == 0) {
      const uint32_t tot[4] = {ftot & 0xffffu, ftot >> 16, static_cast<uint32_t>(ctot),
                               static_cast<uint32_t>(ctot >> 32)};
      if (kMode == 0) {
        base[0] = tot[0] ? atomicAdd(&counters[kCntMedium], tot[0]) : 0u;
        base[1] = tot[1] ? atomicAdd(&counters[kCntLong], tot[1]) : 0u;
        base[2] = tot[2] ? atomicAdd(&counters[kCntChunks], tot[2]) : 0u;
        base[3] = tot[3] ? atomicAdd(&counters[kCntTree], tot[3]) : 0u;
      } else {
        for (int k = 0; k < 4; ++k) {
          base[k] = run_base[k];
          run_base[k] += tot[k];
        }
      }
    }
    __syncthreads();
    if (kMode == 1) continue;  // uniform; the next pass's barriers follow
    if (medium) medium_run[base[0] + (fex & 0xffffu)] = j;
    if (lng) {
      const uint32_t slot = base[1] + (fex >> 16);
      long_run[slot] = j;
      long_chunk0[slot] = base[2] + static_cast<uint32_t>(cex);
      long_tree0[slot] = base[3] + static_cast<uint32_t>(cex >> 32);
    }
    __syncthreads();  // base is rewritten by the next pass
  }
  if (kMode == 1 && threadIdx.x < 4) blk[threadIdx.x * gridDim.x + blockIdx.x] = run_base[threadIdx.x];
}

// One warp per long run: its info record, the descriptors of its chunks, and
// the arrival counters of its reduction tree (children per node).
__global__ void __launch_bounds__(256)
    chunk_fill_kernel(const uint32_t* __restrict__ run_pairs, const uint32_t* __restrict__ counters,
                      const uint32_t* __restrict__ unique_keys,
                      const int64_t* __restrict__ hash_base, int T,
                      const uint32_t* __restrict__ long_run, const uint32_t* __restrict__ long_chunk0,
                      const uint32_t* __restrict__ long_tree0, LongRunInfo* __restrict__ info,
                      ChunkDesc* __restrict__ chunk_desc, uint32_t* __restrict__ tree_cnt) {
  const uint32_t nlong = counters[kCntLong];
  const unsigned lane = lane_id();
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t k = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; k < nlong; k += warps) {
    const uint32_t j = long_run[k];
    const uint32_t p0 = run_pairs[j];
    const uint32_t np = run_pairs[j + 1] - p0;
    const uint32_t nch = (np + kChunk - 1) / kChunk;
    const uint32_t c0 = long_chunk0[k];
    const uint32_t key = unique_keys[j];
    if (lane == 0) {
      int lo = 0, hi = T - 1;  // table of the key
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(hash_base + mid) <= static_cast<int64_t>(key)) lo = mid; else hi = mid - 1;
      }
      LongRunInfo r;
      r.key = key;
      r.table = static_cast<uint32_t>(lo);
      r.nch = nch;
      r.chunk0 = c0;
      r.tree0 = long_tree0[k];
      r.pad0 = j;
      r.pad1 = r.pad2 = 0;
      info[k] = r;
    }
    for (uint32_t c = lane; c < nch; c += 32) {
      ChunkDesc cd;
      cd.first = p0 + c * kChunk;
      cd.end = cd.first + kChunk < p0 + np ? cd.first + kChunk : p0 + np;
      cd.run = k;
      cd.c = c;
      chunk_desc[c0 + c] = cd;
    }
    uint32_t node = long_tree0[k];
    uint32_t below = nch;
    while (below > 1) {
      const uint32_t here = (below + kFanIn - 1) / kFanIn;
      for (uint32_t i = lane; i < here; i += 32) {
        const uint32_t kids = below - i * kFanIn;
        tree_cnt[node + i] = kids < static_cast<uint32_t>(kFanIn) ? kids : kFanIn;
      }
      node += here;
      below = here;
    }
  }
}

// Processing order of the long-run chunks: binned by the first bag each
// chunk gathers (counting sort over bag bands; order within a band is free).
// With TBE_TABLE_BANDS the bins are (table, band) in table-major order,
// bands_per_table bins per table: the chunks in flight then gather from one
// table's gradient rows at a time instead of every table's.
#ifndef TBE_TABLE_BANDS
#define TBE_TABLE_BANDS 1
#endif
__global__ void __launch_bounds__(256)
    chunk_band_count_kernel(const uint32_t* __restrict__ counters,
                            const ChunkDesc* __restrict__ chunk_desc,
                            const LongRunInfo* __restrict__ info,
                            const uint32_t* __restrict__ pair_bags, int band_shift,
                            int bands_per_table,
                            uint32_t* __restrict__ chunk_band, uint32_t* __restrict__ band_count) {
  const uint32_t nchunks = counters[kCntChunks];
  for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < nchunks; q += gridDim.x * blockDim.x) {
    const ChunkDesc cd = chunk_desc[q];
    uint32_t band = pair_bags[cd.first] >> band_shift;
    if (TBE_TABLE_BANDS) {
      const uint32_t bpt = static_cast<uint32_t>(bands_per_table);
      band = info[cd.run].table * bpt + (band < bpt ? band : bpt - 1);
    }
    band = band < kBagBands ? band : kBagBands - 1;
    chunk_band[q] = band;
    atomicAdd(&band_count[band], 1u);
  }
}

__global__ void __launch_bounds__(256)
    chunk_band_scatter_kernel(const uint32_t* __restrict__ counters,
                              const ChunkDesc* __restrict__ chunk_desc,
                              const uint32_t* __restrict__ chunk_band,
                              uint32_t* __restrict__ band_cursor, ChunkDesc* __restrict__ chunk_order) {
  const uint32_t nchunks = counters[kCntChunks];
  for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < nchunks; q += gridDim.x * blockDim.x)
    chunk_order[atomicAdd(&band_cursor[chunk_band[q]], 1u)] = chunk_desc[q];
}

int key_bits(const tbe_desc* d) {
  // keys range over [0, total_E], total_E being the invalid-lookup key
  const uint64_t maxkey = static_cast<uint64_t>(d->total_E);
  int bits = 0;
  while (bits < 32 && (maxkey >> bits) != 0) ++bits;
  return bits < 1 ? 1 : bits;
}

// Grid of the sort / RLE kernels for at most n entries.
SortGeom sort_geom(int64_t n, int num_sms, int per_sm, const uint32_t* n_dev) {
  SortGeom g;
  const int64_t tiles = (n + kSortTile - 1) / kSortTile;
  int64_t ctas = static_cast<int64_t>(per_sm) * num_sms;
  if (ctas > kMaxSortCtas) ctas = kMaxSortCtas;
  if (ctas > tiles) ctas = tiles;
  if (ctas < 1) ctas = 1;
  g.ctas = static_cast<int>(ctas);
  g.n_dev = n_dev;
  return g;
}

template <typename IndexT>
cudaError_t preprocess_t(const Launch& L, const WsLayout& W, char* ws, const IndexT* indices,
                         const IndexT* offsets, const float* psw, bool check) {
  const tbe_desc* d = L.d;
  const int64_t n = L.n;
  cudaStream_t s = L.s;  // the side stream after the expand
  int* status = check ? reinterpret_cast<int*>(ws + W.status) : nullptr;
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + W.counts);
  const uint32_t sentinel = static_cast<uint32_t>(d->total_E);
  const bool weighted = psw != nullptr;
  uint32_t* keys[3];
  uint32_t* vals[3];
  float* pw[3];
  for (int i = 0; i < 3; ++i) {
    keys[i] = reinterpret_cast<uint32_t*>(ws + W.keys[i]);
    vals[i] = reinterpret_cast<uint32_t*>(ws + W.vals[i]);
    pw[i] = weighted ? reinterpret_cast<float*>(ws + W.psw[i]) : nullptr;
  }
  uint32_t* uk = reinterpret_cast<uint32_t*>(ws + W.unique_keys);
  uint32_t* rs = reinterpret_cast<uint32_t*>(ws + W.run_starts);

  SideFlow* sf = side_flow(ws);
  if (!sf) return cudaErrorNotReady;
  // the previous call's side work (sort chain, hot-set refresh) still reads
  // the buffers this one rewrites (a record on the other side of a graph
  // capture is not waited for: every backward joins its side work into the
  // caller's stream before it returns)
  cudaError_t err = flow_wait(s, sf->done);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(counters, 0, kNumCounters * sizeof(uint32_t), s);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(rs, 0, sizeof(uint32_t), s);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(ws + W.run_pairs, 0, sizeof(uint32_t), s);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(ws + W.pair_starts, 0, sizeof(uint32_t), s);
  if (err != cudaSuccess) return err;

  // Expand: hot lookups into the histogram, cold ones (in lookup order) to the sort.
  uint32_t* tile_cold = reinterpret_cast<uint32_t*>(ws + W.tile_cold);
  {
    err = cudaMemsetAsync(ws + W.hot_cnt, 0, static_cast<size_t>(d->T) * kHot * 4, s);
    if (err != cudaSuccess) return err;
    // this batch's hot set: the one the last backward chose
    err = cudaMemcpyAsync(ws + W.hot_cur, ws + W.hot_next, W.hot_set_bytes,
                          cudaMemcpyDeviceToDevice, s);
    if (err != cudaSuccess) return err;
    HotSet hs;
    hs.keys = reinterpret_cast<const uint32_t*>(ws + W.hot_keys(W.hot_cur));
    hs.place = reinterpret_cast<const uint32_t*>(ws + W.hot_place(W.hot_cur));
    hs.n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
    hs.m1 = reinterpret_cast<const uint32_t*>(ws + W.hot_m1(W.hot_cur));
    hs.m2 = reinterpret_cast<const uint32_t*>(ws + W.hot_m2(W.hot_cur));
    float* hh = W.hot_enabled ? reinterpret_cast<float*>(ws + W.hot_hist) : nullptr;
    uint8_t* hh8 = W.hot_enabled ? reinterpret_cast<uint8_t*>(ws + W.hot_hist8) : nullptr;
    int8_t* hsc = reinterpret_cast<int8_t*>(ws + W.hot_scale);
    uint8_t* tk = reinterpret_cast<uint8_t*>(ws + W.tile_kind);
    uint32_t* hc = reinterpret_cast<uint32_t*>(ws + W.hot_cnt);
    uint32_t* bc = reinterpret_cast<uint32_t*>(ws + W.bag_cold);
    uint32_t* co = reinterpret_cast<uint32_t*>(ws + W.cold_off);
    const unsigned tiles = static_cast<unsigned>(W.hot_tiles);
    // the cold lookups go first to buffer 0 at their bags' own positions,
    // then, compacted, to buffer 2 (the sort reads buffer 2 before it
    // writes buffer 0)
    if (weighted)
      { probe_begin(TBE_PROBE_EXPAND_COUNT, s); expand_count_kernel<IndexT, true><<<tiles, 256, sizeof(ExpandSmem<IndexT, true>), s>>>(
          indices, offsets, psw, d->hash_base, d->D_offsets, n, d->B, hs, hh8, hh, hsc, tk, hc, bc,
          tile_cold, keys[0], pw[0], status); note_launch(); probe_end(TBE_PROBE_EXPAND_COUNT, s); }
    else
      { probe_begin(TBE_PROBE_EXPAND_COUNT, s); expand_count_kernel<IndexT, false><<<tiles, 256, sizeof(ExpandSmem<IndexT, false>), s>>>(
          indices, offsets, psw, d->hash_base, d->D_offsets, n, d->B, hs, hh8, hh, hsc, tk, hc, bc,
          tile_cold, keys[0], pw[0], status); note_launch(); probe_end(TBE_PROBE_EXPAND_COUNT, s); }
    { capped_scan_kernel<<<1, 1024, 0, s>>>(tile_cold, W.hot_tiles, static_cast<uint32_t>(n),
                                            counters + kCntSortN); note_launch(); }
    if (weighted)
      { expand_write_kernel<IndexT, true><<<tiles, 256, 0, s>>>(
          offsets, n, d->B, bc, tile_cold, co, keys[0], pw[0], keys[2], vals[2],
          pw[2]); note_launch(); }
    else
      { expand_write_kernel<IndexT, false><<<tiles, 256, 0, s>>>(
          offsets, n, d->B, bc, tile_cold, co, keys[0], pw[0], keys[2], vals[2],
          pw[2]); note_launch(); }
  }
  // The sort chain (sort, run-length encoding, classification) goes to the
  // side stream: the forward needs only the expand's outputs and runs
  // concurrently on the caller's stream; the backward waits for `sorted`.
  err = fork_to(sf, s);
  if (err != cudaSuccess) return err;
  s = sf->side;
  if (n > 0) {
    const SortGeom g = sort_geom(n, L.num_sms, 2, counters + kCntSortN);
    const int bits = key_bits(d);
    const int passes = (bits + kMaxRadixBits - 1) / kMaxRadixBits;
    const int rb = (bits + passes - 1) / passes;
    uint32_t* counts = reinterpret_cast<uint32_t*>(ws + W.radix_counts);
    uint32_t* totals = counts + static_cast<size_t>(kMaxSortCtas) * (1 << kMaxRadixBits);
    const size_t smem = weighted ? sizeof(DownSmem<true>) : sizeof(DownSmem<false>);
    for (int p = 0; p < passes; ++p) {
      const int shift = p * rb;
      const int width = rb < bits - shift ? rb : bits - shift;
      // pass 0 reads the expand output (buffer 2), later passes ping-pong
      // between 1 and 0, so the sorted result is in buffer passes & 1
      const int src = p == 0 ? 2 : (p & 1), dst = (p & 1) ^ 1;
      { radix_upsweep_kernel<<<g.ctas, kSortThreads, 0, s>>>(keys[src], g, shift, width, counts); note_launch(); }
      { radix_scan_kernel<<<((1 << width) + 7) / 8, 256, 0, s>>>(counts, g.ctas, 1 << width, totals); note_launch(); }
      if (weighted)
        { probe_begin(TBE_PROBE_RADIX_DOWNSWEEP, s); radix_downsweep_kernel<true><<<g.ctas, kSortThreads, smem, s>>>(
            keys[src], vals[src], pw[src], keys[dst], vals[dst], pw[dst], g, shift, width,
            counts, totals); note_launch(); probe_end(TBE_PROBE_RADIX_DOWNSWEEP, s); }
      else
        { probe_begin(TBE_PROBE_RADIX_DOWNSWEEP, s); radix_downsweep_kernel<false><<<g.ctas, kSortThreads, smem, s>>>(
            keys[src], vals[src], pw[src], keys[dst], vals[dst], pw[dst], g, shift, width,
            counts, totals); note_launch(); probe_end(TBE_PROBE_RADIX_DOWNSWEEP, s); }
    }
    const int fin = passes & 1;
    const SortGeom gr = sort_geom(n, L.num_sms, 6, counters + kCntSortN);
    uint32_t* cta_runs = reinterpret_cast<uint32_t*>(ws + W.cta_counts);
    uint32_t* cta_pairs = cta_runs + (kMaxSortCtas + 1);
    { rle_count_kernel<<<gr.ctas, kRleThreads, 0, s>>>(keys[fin], vals[fin], gr, sentinel,
                                                     cta_runs, cta_pairs); note_launch(); }
    { exclusive_scan_kernel<<<1, 1024, 0, s>>>(cta_runs, gr.ctas, cta_runs + gr.ctas); note_launch(); }
    { exclusive_scan_kernel<<<1, 1024, 0, s>>>(cta_pairs, gr.ctas, cta_pairs + gr.ctas); note_launch(); }
    { rle_write_kernel<<<gr.ctas, kRleThreads, 0, s>>>(
        keys[fin], vals[fin], gr, sentinel, cta_runs, cta_pairs, uk, rs,
        reinterpret_cast<uint32_t*>(ws + W.run_pairs),
        reinterpret_cast<uint32_t*>(ws + W.pair_starts),
        reinterpret_cast<uint32_t*>(ws + W.pair_bags), counters); note_launch(); }
  }
  { table_runs_kernel<<<1, 1024, 0, s>>>(uk, counters, d->hash_base, d->D_offsets, d->T,
                                       reinterpret_cast<uint32_t*>(ws + W.table_runs),
                                       reinterpret_cast<uint32_t*>(ws + W.table_tasks), counters); note_launch(); }
  if (n > 0) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 8LL * L.num_sms) blocks = 8LL * L.num_sms;
    uint32_t* cl_args[5] = {reinterpret_cast<uint32_t*>(ws + W.long_run),
                            reinterpret_cast<uint32_t*>(ws + W.long_chunk0),
                            reinterpret_cast<uint32_t*>(ws + W.long_tree0),
                            reinterpret_cast<uint32_t*>(ws + W.medium_run),
                            reinterpret_cast<uint32_t*>(ws + W.radix_counts)};  // sort done: free
    const uint32_t* rp = reinterpret_cast<uint32_t*>(ws + W.run_pairs);
    const unsigned cb0 = static_cast<unsigned>(blocks);
    if (TBE_ORDERED_CLASSIFY) {
      classify_kernel<1><<<cb0, 256, 0, s>>>(rp, counters, cl_args[0], cl_args[1], cl_args[2],
                                              cl_args[3], cl_args[4]);
      note_launch();
      const ScanDests dest{{kCntMedium, kCntLong, kCntChunks, kCntTree}};
      block_totals_scan_kernel<<<4, 1024, 0, s>>>(cl_args[4], static_cast<int>(cb0), counters,
                                                 dest);
      note_launch();
      classify_kernel<2><<<cb0, 256, 0, s>>>(rp, counters, cl_args[0], cl_args[1], cl_args[2],
                                              cl_args[3], cl_args[4]);
      note_launch();
    } else {
      classify_kernel<0><<<cb0, 256, 0, s>>>(rp, counters, cl_args[0], cl_args[1], cl_args[2],
                                              cl_args[3], cl_args[4]);
      note_launch();
    }
    int64_t fb = (W.max_long * 32 + 255) / 256;
    if (fb > 8LL * L.num_sms) fb = 8LL * L.num_sms;
    if (fb < 1) fb = 1;
    { chunk_fill_kernel<<<static_cast<unsigned>(fb), 256, 0, s>>>(
        reinterpret_cast<uint32_t*>(ws + W.run_pairs), counters, uk, d->hash_base, d->T,
        reinterpret_cast<uint32_t*>(ws + W.long_run),
        reinterpret_cast<uint32_t*>(ws + W.long_chunk0),
        reinterpret_cast<uint32_t*>(ws + W.long_tree0),
        reinterpret_cast<LongRunInfo*>(ws + W.long_info),
        reinterpret_cast<ChunkDesc*>(ws + W.chunk_desc),
        reinterpret_cast<uint32_t*>(ws + W.tree_cnt)); note_launch(); }
    const int bands_per_table =
        TBE_TABLE_BANDS ? (d->T < kBagBands ? kBagBands / d->T : 1) : kBagBands;
    int band_shift = 0;
    while ((static_cast<int64_t>(d->B - 1) >> band_shift) >= bands_per_table) ++band_shift;
    uint32_t* band_count = reinterpret_cast<uint32_t*>(ws + W.band_count);
    err = cudaMemsetAsync(band_count, 0, kBagBands * sizeof(uint32_t), s);
    if (err != cudaSuccess) return err;
    int64_t cb = (W.max_chunks + 255) / 256;
    if (cb > 8LL * L.num_sms) cb = 8LL * L.num_sms;
    if (cb < 1) cb = 1;
    { chunk_band_count_kernel<<<static_cast<unsigned>(cb), 256, 0, s>>>(
        counters, reinterpret_cast<ChunkDesc*>(ws + W.chunk_desc),
        reinterpret_cast<const LongRunInfo*>(ws + W.long_info),
        reinterpret_cast<uint32_t*>(ws + W.pair_bags), band_shift, bands_per_table,
        reinterpret_cast<uint32_t*>(ws + W.chunk_band), band_count); note_launch(); }
    { exclusive_scan_kernel<<<1, 1024, 0, s>>>(band_count, kBagBands, nullptr); note_launch(); }
    { chunk_band_scatter_kernel<<<static_cast<unsigned>(cb), 256, 0, s>>>(
        counters, reinterpret_cast<ChunkDesc*>(ws + W.chunk_desc),
        reinterpret_cast<uint32_t*>(ws + W.chunk_band), band_count,
        reinterpret_cast<ChunkDesc*>(ws + W.chunk_order)); note_launch(); }
  }
  err = flow_record(sf->sorted, s);
  if (err != cudaSuccess) return err;
  if (TBE_REFRESH_IN_PREPROCESS) {
    // the next hot set needs only this batch's runs and hot-row counts;
    // the backward does not wait for it (only the next preprocess does)
    Launch Ls = L;
    Ls.s = s;
    err = launch_hot_refresh(Ls, W, ws);
    if (err != cudaSuccess) return err;
  }
  err = flow_record(sf->done, s);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

int radix_passes(const tbe_desc* d) {
  const int bits = key_bits(d);
  return (bits + kMaxRadixBits - 1) / kMaxRadixBits;
}

cudaError_t prepare_preprocess_kernels() {
  cudaError_t e = cudaFuncSetAttribute(expand_count_kernel<int32_t, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(ExpandSmem<int32_t, true>)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(expand_count_kernel<int64_t, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(ExpandSmem<int64_t, true>)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(radix_downsweep_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(DownSmem<true>)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(radix_downsweep_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(DownSmem<false>)));
}

cudaError_t launch_preprocess(const Launch& L, const WsLayout& W, char* ws, const void* indices,
                              const void* offsets, const float* psw, bool check) {
  if (L.d->index_dtype == TBE_DT_I32)
    return preprocess_t<int32_t>(L, W, ws, static_cast<const int32_t*>(indices),
                                 static_cast<const int32_t*>(offsets), psw, check);
  return preprocess_t<int64_t>(L, W, ws, static_cast<const int64_t*>(indices),
                               static_cast<const int64_t*>(offsets), psw, check);
}

}  // namespace tbe
