// Gather-and-sum of one bag's rows by one warp (the pooled forward's inner
// loop), shared by the generic forward and the hot-row forward.
#pragma once

#include "common.cuh"

namespace tbe {
namespace {

// How pool_bag leaves its sum: stored, or added to what out_row holds.
constexpr int kPoolStore = 0;
constexpr int kPoolAdd = 1;

// A row of zeros (kMaxD fp16 values): the gather target of lookups that are
// out of range or past a bag's end.  Static device memory is zero at module
// load and nothing writes it.
__device__ __align__(16) uint4 g_zero_row[kMaxD / 8];

// Pool one bag over the row columns [vec0*8, (vec0 + min(S, nvec - vec0))*8):
// lane sl of each group owns the 16-byte vector vec0 + sl.  Rows wider than
// 32 vectors (256 fp16) are pooled in several such column passes, so no lane
// ever holds more than eight accumulators.  The lane that loads a lookup's
// index resolves it to a row address once; a lookup that is out of range or
// past the bag's end resolves to a row of zeros, so the gather loop has no
// per-lookup branch (a skipped lookup also gets weight 0).  Row r of the
// table is the lookup value minus `rbase` (0 for raw indices, the table's
// first linear key for lists of linear keys).
template <int S, typename IndexT, bool kWeighted, int kUnroll = TBE_FWD_UNROLL, bool kBf16 = false>
__device__ __forceinline__ void pool_bag(const __half* __restrict__ Wt, int64_t E, int64_t rbase,
                                         int D, int vec0, const IndexT* __restrict__ indices,
                                         const float* __restrict__ psw, int64_t start,
                                         int64_t end, float* __restrict__ out_row, int mode,
                                         int* status, float scale = 1.f) {
  constexpr int G = 32 / S;
  constexpr int U = S < kUnroll ? S : kUnroll;  // row vectors in flight per lane
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
  const int vec = vec0 + sl;
  const bool col_ok = vec < (D >> 3);
  // lanes past the row's last vector read the row's first one and drop it
  const int col = col_ok ? vec * 8 : 0;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  bool bad = false;

  // The next batch's index (and weight) is loaded while this batch's rows are
  // gathered, so a batch waits on one memory round trip instead of two.
  int64_t nx_r = start + lane < end ? load_index(indices, start + lane) : 0;
  float nx_w = (kWeighted && start + lane < end) ? __ldg(psw + start + lane) : 0.f;
  for (int64_t base = start; base < end; base += 32) {
    const int cnt = static_cast<int>(end - base < 32 ? end - base : 32);
    const int64_t r = nx_r - rbase;
    const float w_in = nx_w;
    if (base + 32 + lane < end) {
      nx_r = load_index(indices, base + 32 + lane);
      if (kWeighted) nx_w = __ldg(psw + base + 32 + lane);
    }
    const __half* my_row = reinterpret_cast<const __half*>(g_zero_row);
    float my_w = 0.f;
    if (lane < cnt) {
      const bool ok = r >= 0 && r < E;
      bad |= !ok;
      if (ok) {
        my_row = Wt + r * D;
        if (kWeighted) my_w = w_in;
      }
    }
    const uint64_t my_addr = reinterpret_cast<uint64_t>(my_row);
    const uint32_t my_lo = static_cast<uint32_t>(my_addr);
    const uint32_t my_hi = static_cast<uint32_t>(my_addr >> 32);
#pragma unroll
    for (int u0 = 0; u0 < S; u0 += U) {
      if (G * u0 >= cnt) break;  // warp-uniform
      uint4 v[U];
      float wv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int k = g + G * (u0 + uu);  // < 32 because u0 + uu < S
        const uint64_t a = static_cast<uint64_t>(__shfl_sync(kFull, my_lo, k)) |
                           (static_cast<uint64_t>(__shfl_sync(kFull, my_hi, k)) << 32);
        if (kWeighted) wv[uu] = __shfl_sync(kFull, my_w, k);
        v[uu] = ldg_u4(reinterpret_cast<const __half*>(a) + col);
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) acc_row8<kBf16, kWeighted>(acc, v[uu], kWeighted ? wv[uu] : 1.f);
    }
  }

  // Combine the G groups (lanes sl, sl+S, sl+2S, ... hold the same columns).
#pragma unroll
  for (int off = S; off < 32; off <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += __shfl_xor_sync(kFull, acc[i], off);

  if (g == 0 && col_ok) {
    float4* o = reinterpret_cast<float4*>(out_row + vec * 8);
    if (mode == kPoolAdd) {  // out already holds a partial sum of the bag
      const float4 a = o[0], b = o[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    if (scale != 1.f)  // mean pooling
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= scale;
    // written once, not read back: evict first
    __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
    __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
  }
  if (status && __any_sync(kFull, bad) && lane == 0) set_status(status, TBE_ERR_INDEX_RANGE);
}

}  // namespace
}  // namespace tbe
