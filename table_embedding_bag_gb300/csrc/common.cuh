// Internal helpers shared by the CUDA translation units of the TBE library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "tbe.h"

// Build-time tuning knobs (defaults are the measured choices on GB300):
//   TBE_CHUNK_PAIRS   pairs per long-run chunk and the long-run threshold
//   TBE_LONG_VECS     row vectors in flight per lane on long-run chunks
//   TBE_LONG_MINB     resident CTAs per SM the long-run kernel is built for
//   TBE_SHORT_VECS    row vectors in flight per lane on short runs
//   TBE_FWD_UNROLL    row vectors in flight per lane in the forward
//   TBE_SHORT_MINB, TBE_FWD_MINB  resident CTAs per SM for those kernels
#ifndef TBE_SHORT_MINB
#define TBE_SHORT_MINB 3
#endif
#ifndef TBE_FWD_MINB
#define TBE_FWD_MINB 4
#endif
#ifndef TBE_LONG_VECS
#define TBE_LONG_VECS 8
#endif
#ifndef TBE_LONG_MINB
#define TBE_LONG_MINB 3
#endif
#ifndef TBE_SHORT_VECS
#define TBE_SHORT_VECS 4
#endif
#ifndef TBE_FWD_UNROLL
#define TBE_FWD_UNROLL 4
#endif
// TBE_DYNAMIC_RUNS: the short-, medium- and long-run update kernels take
// their next task from a counter (in task order) instead of a fixed stride,
// so that the warps in flight stay on a narrow window of runs.
#ifndef TBE_DYNAMIC_RUNS
#define TBE_DYNAMIC_RUNS 1
#endif

namespace tbe {

constexpr unsigned kFull = 0xffffffffu;

// Work threshold from which a run takes the chunked (cooperative) path and
// the work per chunk.  Work is counted in distinct (row, bag) pairs: every
// lookup of a bag into the same row shares one gradient-row gather.  The
// FBTriton backward uses 256 lookups for both; here both are 128 pairs (the
// fastest on GB300 in a sweep of 128/256/512), and they stay equal, so a long
// run always has at least one full chunk.
#ifndef TBE_CHUNK_PAIRS
#define TBE_CHUNK_PAIRS 128
#endif
constexpr int kLongThreshold = TBE_CHUNK_PAIRS;
// Runs of at least kMediumRun pairs (and fewer than kLongThreshold) are
// updated by a whole warp each instead of sharing a warp with other runs.
#ifndef TBE_MEDIUM_RUN
#define TBE_MEDIUM_RUN 16
#endif
constexpr int kMediumRun = TBE_MEDIUM_RUN;
static_assert(kMediumRun <= TBE_CHUNK_PAIRS, "medium runs lie below the long threshold");
constexpr int kChunk = TBE_CHUNK_PAIRS;
// Fan-in of the last-arriver reduction tree over a long run's chunk partials.
constexpr int kFanIn = 32;
// Widest supported table row (elements); rows are moved in 16-byte vectors.
constexpr int kMaxD = 1024;

// Hot rows: per table, up to kHot rows (the most looked-up ones of the
// previous backward) bypass the sort; their gradients are histogram(bag x hot
// row)^T x grad_out.  The histogram (a byte per entry, plus fp32 rows for
// the tiles whose entries a byte cannot hold) is kept only if it fits
// kHotBudgetBytes,
// and tables wider than kHotMaxD take no hot rows.
#ifndef TBE_HOT_ROWS
#define TBE_HOT_ROWS 256
#endif
constexpr int kHot = TBE_HOT_ROWS;
constexpr int kHotTileBags = 128;  // bags per expand CTA (one table)
// Histogram storage of a tile of kHotTileBags bags: every count of the tile
// fits a byte (unweighted lookups, at most 255 of one row in a bag), or the
// tile's rows are fp32 with per-bag scales, or its table has no hot rows.
constexpr uint8_t kTileBytes = 0;
constexpr uint8_t kTileWide = 1;
constexpr uint8_t kTileNoHot = 2;
constexpr int kHotMaxD = 256;
constexpr size_t kHotBudgetBytes = size_t(2) << 30;
// CTAs of the hot-gradient kernels (bag partitions over all tables): one
// wave at 2 per SM on 152 SMs
#ifndef TBE_HOT_CTA_TARGET
#define TBE_HOT_CTA_TARGET 304
#endif
constexpr int kHotCtaTarget = TBE_HOT_CTA_TARGET;
constexpr int kHotMinPartBags = 256;  // fewest bags per hot-gradient CTA
constexpr int kHotFwdMinBagLen = 64;  // preprocessed forward: mean lookups per bag to use it
constexpr int kHotBuckets = 256;    // log-scale buckets of lookup counts (8 per octave)
// A row becomes hot with at least max(B / kHotMinCountDiv, 32) lookups in a
// batch: its histogram column costs about 12 bytes per bag (written once,
// read by the forward and the gradient), a cold lookup costs several hundred
// (row gather, gradient-row gather, sort traffic).
constexpr int kHotMinCountDiv = 64;
static_assert(kHot % 64 == 0 && kHot <= 256, "hot slots: multiples of the 64-slot MMA chunk");

// Hot-set membership: a two-choice (cuckoo) hash of the table's hot keys in
// shared memory, two halves of kCuckooHalf entries.  When the set is chosen,
// multipliers m1, m2 are found under which every key has a place at
// h1 = (key * m1) >> s or kCuckooHalf + ((key * m2) >> s), and each key's place
// is stored with the set, so a lookup is two independent 64-bit shared loads.
constexpr int kCuckooHalfBits = 9;
constexpr int kCuckooHalf = 1 << kCuckooHalfBits;
constexpr int kCuckooSize = 2 * kCuckooHalf;
constexpr uint32_t kEmptyKey = 0xffffffffu;  // never a key: total_E < 2^32 - 1

__host__ __device__ __forceinline__ uint32_t cuckoo_h1(uint32_t key, uint32_t m1) {
  return (key * m1) >> (32 - kCuckooHalfBits);
}
__host__ __device__ __forceinline__ uint32_t cuckoo_h2(uint32_t key, uint32_t m2) {
  return kCuckooHalf + ((key * m2) >> (32 - kCuckooHalfBits));
}

// Long-run chunks are processed in order of the first bag they touch, binned
// into at most this many bag bands, so that the warps in flight gather
// gradient rows from a narrow band of bags and the band stays in L2.
constexpr int kBagBands = 2048;

// Radix sort: threads per CTA, keys per thread, digit width bound.
constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kMaxRadixBits = 9;
constexpr int kMaxSortCtas = 1024;

// Workspace header: status word and device-resident counters.
enum Counter : int {
  kCntRuns = 0,      // R: runs with a valid key
  kCntValid = 1,     // n_valid: sorted lookups with a valid key
  kCntLong = 2,      // long runs
  kCntChunks = 3,    // chunks of long runs
  kCntTree = 4,      // internal reduction-tree nodes
  kCntTasks = 5,     // short-run warp tasks
  kCntPairs = 6,     // P: distinct (key, bag) pairs among the valid sorted lookups
  kCntSortN = 7,     // entries in the sort (written on the device before the sort)
  kCntMedium = 8,    // medium runs (kMediumRun <= pairs < kLongThreshold)
  kCntNextShort = 9,   // work cursors of the update kernels (TBE_DYNAMIC_RUNS):
  kCntNextMedium = 10, // the next short-run task, medium run and long-run chunk
  kCntNextLong = 11,   // to hand out
  kNumCounters = 12,
};

struct WsLayout {
  size_t status;       // int32 status word
  size_t counts;       // uint32 [kNumCounters]
  size_t table_runs;   // uint32 [T+1] first run of each table
  size_t table_tasks;  // uint32 [T+1] prefix of short-run warp tasks per table
  // sort buffers: [2] is the expand output, the cold lookups in lookup order
  // (kept intact for the forward), [0] / [1] the radix passes' ping-pong
  size_t keys[3];      // uint32 [n] linear keys
  size_t vals[3];      // uint32 [n] bags
  size_t psw[3];       // float [n] (weighted only)
  size_t radix_counts; // uint32 [2^kMaxRadixBits * kMaxSortCtas]
  size_t cta_counts;   // uint32 [kMaxSortCtas + 1]
  size_t unique_keys;  // uint32 [n + 1]
  size_t run_starts;   // uint32 [n + 2] first sorted position of each run
  size_t run_pairs;    // uint32 [n + 2] first pair of each run
  size_t pair_starts;  // uint32 [n + 2] first sorted position of each (key, bag) pair
  size_t pair_bags;    // uint32 [n + 1] bag of each pair
  size_t medium_run;   // uint32 [max_medium] medium runs (any order)
  size_t long_run;     // uint32 [max_long]
  size_t long_chunk0;  // uint32 [max_long] first chunk of each long run
  size_t long_tree0;   // uint32 [max_long] first tree node of each long run
  size_t long_info;    // LongRunInfo [max_long]
  size_t chunk_desc;   // ChunkDesc [max_chunks], chunk-id order
  size_t chunk_band;   // uint32 [max_chunks] bag band of each chunk
  size_t chunk_order;  // ChunkDesc [max_chunks], sorted by bag band
  size_t band_count;   // uint32 [kBagBands] chunks per band, then band cursors
  size_t tree_cnt;     // uint32 [max_tree] arrivals still expected at each tree node
  size_t partials;     // float [max_chunks * max_D]
  size_t tree_part;    // float [max_tree * max_D]
  // Two hot sets, each uint32 keys [T][kHot] (linear keys, the most looked-up
  // first, ties by key), place
  // [T][kHot] (each key's cuckoo entry), n [T], m1 [T], m2 [T], kept across
  // calls: `hot_next` is written by the backward's refresh and copied to
  // `hot_cur` at the start of every preprocess; the preprocess, the forward
  // and the backward of one batch all read `hot_cur`.
  size_t hot_cur;
  size_t hot_next;
  size_t hot_set_bytes;
  size_t hot_keys(size_t set) const { return set; }
  size_t hot_place(size_t set) const { return set + static_cast<size_t>(T) * kHot * 4; }
  size_t hot_n(size_t set) const { return set + static_cast<size_t>(T) * kHot * 8; }
  size_t hot_m1(size_t set) const { return hot_n(set) + static_cast<size_t>(T) * 4; }
  size_t hot_m2(size_t set) const { return hot_n(set) + static_cast<size_t>(T) * 8; }
  int64_t T;
  size_t hot_cnt;      // uint32 [T][kHot] lookups of each hot row in this call
  size_t hot_hist8;    // uint8 [T][B][kHot] per-bag lookups of each hot row, byte tiles (if enabled)
  size_t hot_hist;     // float [T][B][kHot] per-bag weight of each hot row, wide tiles (if enabled)
  size_t hot_scale;    // int8 [T*B] wide tiles: histogram row x 2^scale peaks below 2^15
  size_t tile_kind;    // uint8 [hot_tiles] kTileBytes / kTileWide / kTileNoHot
  size_t cold_off;     // uint32 [T*B + 1] first cold-list entry of each bag
  size_t inv_len;      // float [T*B] mean pooling's factor per bag: 1/L for L > 1 lookups, else 1
                       // (written by mean-mode calls before their use)
  size_t hot_part;     // float [T][hot_parts][kHot][kHotMaxD] partial hot gradients
  size_t bag_cold;     // uint32 [T*B] cold lookups per bag
  size_t tile_cold;    // uint32 [hot_tiles + 1] cold lookups per expand tile, then prefix
  size_t sel_hist;     // uint32 [T][kHotBuckets] refresh: count buckets per table
  size_t sel_thresh;   // uint32 [T] refresh: lowest bucket kept
  size_t sel_keys;     // uint32 [T][kHot] refresh: the next hot set
  size_t sel_cnt;      // uint32 [T][kHot] refresh: each selected key's lookups
  size_t sel_n;        // uint32 [T]
  size_t offsets_fix;  // index type [T*B+1] repaired offsets
  size_t fix_scratch;  // int64 [blocks] block maxima for the repair scan
  size_t grad_mean;    // float [B][total_D] mean-scaled gradient (TBE_WS_MEAN only; last)
  size_t total;
  int64_t max_long, max_chunks, max_tree, max_medium;
  int64_t hot_tiles;   // expand CTAs: T * ceil(B / kHotTileBags)
  int hot_parts;       // bag partitions per table in the hot-gradient kernel
  bool hot_enabled;    // histogram fits the budget
  bool weighted;
};

// One chunk of a long run: pairs [first, end) of long run `run`, chunk index c.
struct __align__(16) ChunkDesc {
  uint32_t first, end, run, c;
};

// One long run: its key and table, chunk count, first chunk slot and first
// reduction-tree node.
struct __align__(16) LongRunInfo {
  uint32_t key, table, nch, chunk0, tree0, pad0, pad1, pad2;
};

// Lanes per gradient row for the update kernels (fp32 rows moved as float4,
// nv = D/4 vectors): small rows take next_pow2(nv) lanes; wider rows give each
// lane up to four vectors so that a warp serves several runs at once.
__host__ __device__ inline int update_lanes(int nv) {
  int p = 1;
  while (p < nv) p <<= 1;
  if (p <= 8) return p;
  int S = p / 4;
  if (S < 8) S = 8;
  return S > 32 ? 32 : S;
}

// Number of reduction-tree nodes above nch leaves (the root included when
// nch > 1): levels ceil(nch/F), ceil(ceil(nch/F)/F), ... down to 1.
__host__ __device__ inline int64_t tree_nodes(int64_t nch) {
  int64_t total = 0;
  while (nch > 1) {
    nch = (nch + kFanIn - 1) / kFanIn;
    total += nch;
  }
  return total;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// allow_hot = false lays out no hot-row histograms or partials and turns the
// hot-row path off (the no-allocation entry point's fixed scratch).
WsLayout make_layout(const tbe_desc* d, int64_t n, uint32_t ws_flags, bool allow_hot = true);

inline int index_bytes(const tbe_desc* d) { return d->index_dtype == TBE_DT_I32 ? 4 : 8; }

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

template <typename IndexT>
__device__ __forceinline__ int64_t load_index(const IndexT* p, int64_t i) {
  return static_cast<int64_t>(__ldg(p + i));
}

// Offsets of bag `bag` clamped into [0, n] with end >= start, so that no
// lookup outside indices[0, n) is ever touched whatever the offsets hold.
template <typename IndexT>
__device__ __forceinline__ void bag_range(const IndexT* offsets, int64_t bag, int64_t n,
                                          int64_t* start, int64_t* end) {
  int64_t s = load_index(offsets, bag);
  int64_t e = load_index(offsets, bag + 1);
  s = s < 0 ? 0 : (s > n ? n : s);
  e = e < s ? s : (e > n ? n : e);
  *start = s;
  *end = e;
}

// Eight fp16 values packed in a uint4 -> fp32, scaled and accumulated.
__device__ __forceinline__ void acc_half8(float* acc, uint4 v, float w) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(h[i]);
    acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
  }
}

// Eight fp16 values accumulated into fp32 without a weight: f32(h) + acc,
// rounded once, the same result as converting and then adding.
__device__ __forceinline__ void add_half8(float* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
        : "r"(w[i]));
}

// Eight bf16 values packed in a uint4 -> fp32 (a bf16 is the upper half of
// an fp32), accumulated, optionally scaled.
__device__ __forceinline__ void add_bf16x8(float* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(w[i] << 16);
    acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void acc_bf16x8(float* acc, uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(s, __uint_as_float(w[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = fmaf(s, __uint_as_float(w[i] & 0xffff0000u), acc[2 * i + 1]);
  }
}
// The forward's accumulation of eight 16-bit weights of either type.
template <bool kBf16, bool kWeighted>
__device__ __forceinline__ void acc_row8(float* acc, uint4 v, float s) {
  if constexpr (kBf16) {
    if constexpr (kWeighted) acc_bf16x8(acc, v, s);
    else add_bf16x8(acc, v);
  } else {
    if constexpr (kWeighted) acc_half8(acc, v, s);
    else add_half8(acc, v);
  }
}

__device__ __forceinline__ uint4 ldg_u4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte asynchronous global -> shared copy; bytes beyond src_bytes are
// zero-filled and not read from global memory.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}
// 4-byte asynchronous global -> shared copy through L1; when !valid nothing
// is read and the four bytes are zero-filled.
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ float4 ldg_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

}  // namespace tbe

namespace tbe {

// ------------------------------------------------------------------- scans
struct OpSum {
  template <typename T>
  __device__ __forceinline__ T operator()(T a, T b) const { return a + b; }
};
struct OpMax {
  template <typename T>
  __device__ __forceinline__ T operator()(T a, T b) const { return a > b ? a : b; }
};

template <typename T, typename Op>
__device__ __forceinline__ T warp_inclusive_scan(T v, Op op) {
  const unsigned lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(kFull, v, o);
    if (lane >= static_cast<unsigned>(o)) v = op(v, y);
  }
  return v;
}

// Inclusive scan over the CTA (blockDim.x a multiple of 32, at most 1024).
// smem must hold 33 elements.  *total receives the CTA aggregate.  Contains
// __syncthreads; every thread of the CTA must call it.
template <typename T, typename Op>
__device__ T block_inclusive_scan(T v, Op op, T identity, T* smem, T* total = nullptr) {
  const unsigned lane = lane_id();
  const unsigned warp = threadIdx.x >> 5;
  const unsigned nwarps = blockDim.x >> 5;
  v = warp_inclusive_scan(v, op);
  if (lane == 31) smem[warp] = v;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nwarps ? smem[lane] : identity;
    w = warp_inclusive_scan(w, op);
    smem[lane] = w;  // inclusive per-warp prefix
  }
  __syncthreads();
  if (warp > 0) v = op(smem[warp - 1], v);
  if (total) *total = smem[nwarps - 1];
  __syncthreads();
  return v;
}

}  // namespace tbe
