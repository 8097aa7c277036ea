// Gather-and-sum of one bag's rows by one warp (the pooled forward's inner
// loop), shared by the generic forward and the hot-row forward.
#pragma once

#include "common.cuh"

namespace tbe {
namespace {

// How pool_bag leaves its sum: stored, or added to what out_row holds.
constexpr int kPoolStore = 0;
constexpr int kPoolAdd = 1;

// A row of zeros (kMaxD fp32 values, so also kMaxD 16-bit ones): the gather
// target of lookups that are out of range or past a bag's end.  Static device
// memory is zero at module load and nothing writes it.
__device__ __align__(16) uint4 g_zero_row[kMaxD / 4];

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

// ------------------------------------------------------------ fp32 weights
// fp32 rows are pooled as an unevaluated sum hi + lo of two fp32 values per
// column: every term is added to hi by Knuth's two-sum, whose exact rounding
// error goes to lo; a weighted term's product is split exactly by a fused
// multiply-add first (Ogita, Rump and Oishi's "Sum2" and "Dot2").  The sum
// hi + lo rounded once is within the final rounding plus about
// (n 2^-24)^2 of the sum of |terms| of the exact sum, which at these bag
// lengths is what an fp64 accumulation rounded to fp32 gives.  The _rn
// intrinsics are never contracted into fused operations.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// hi + lo += x (unweighted) or w * x.
template <bool kWeighted>
__device__ __forceinline__ void comp_add(float& hi, float& lo, float x, float w) {
  float e;
  if constexpr (kWeighted) {
    const float p = __fmul_rn(w, x);
    const float pe = fmaf(w, x, -p);  // w x - p, exact
    two_sum(hi, p, hi, e);
    lo = __fadd_rn(lo, __fadd_rn(e, pe));
  } else {
    two_sum(hi, x, hi, e);
    lo = __fadd_rn(lo, e);
  }
}

// The same bag pooling as pool_bag (one warp, G groups of S lanes, lane sl
// owning columns 8 (vec0 + sl) .. + 7, passes of 256 columns) for fp32 rows:
// each column vector is two 16-byte loads, accumulated compensated.  The
// groups meet in a butterfly of two-sums (the same result in every lane of a
// column); the sum is stored, times the mean factor `scale`.
template <int S, typename IndexT, bool kWeighted, int kUnroll = TBE_FWD_UNROLL>
__device__ __forceinline__ void pool_bag_f32(const float* __restrict__ Wt, int64_t E, int D,
                                             int vec0, const IndexT* __restrict__ indices,
                                             const float* __restrict__ psw, int64_t start,
                                             int64_t end, float* __restrict__ out_row,
                                             int* status, float scale = 1.f) {
  constexpr int G = 32 / S;
  constexpr int U = S < kUnroll ? S : kUnroll;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
  const int vec = vec0 + sl;
  const bool col_ok = vec < (D >> 3);
  const int col = col_ok ? vec * 8 : 0;
  float hi[8], lo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) hi[i] = lo[i] = 0.f;
  bool bad = false;
  int64_t nx_r = start + lane < end ? load_index(indices, start + lane) : 0;
  float nx_w = (kWeighted && start + lane < end) ? __ldg(psw + start + lane) : 0.f;
  for (int64_t base = start; base < end; base += 32) {
    const int cnt = static_cast<int>(end - base < 32 ? end - base : 32);
    const int64_t r = nx_r;
    const float w_in = nx_w;
    if (base + 32 + lane < end) {
      nx_r = load_index(indices, base + 32 + lane);
      if (kWeighted) nx_w = __ldg(psw + base + 32 + lane);
    }
    const float* my_row = reinterpret_cast<const float*>(g_zero_row);
    float my_w = 0.f;
    if (lane < cnt) {
      const bool ok = r >= 0 && r < E;
      bad |= !ok;
      if (ok) {
        my_row = Wt + r * D;
        my_w = kWeighted ? w_in : 1.f;
      }
    }
    const uint64_t my_addr = reinterpret_cast<uint64_t>(my_row);
    const uint32_t my_lo = static_cast<uint32_t>(my_addr);
    const uint32_t my_hi = static_cast<uint32_t>(my_addr >> 32);
#pragma unroll
    for (int u0 = 0; u0 < S; u0 += U) {
      if (G * u0 >= cnt) break;  // warp-uniform
      float4 v[U][2];
      float wv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int k = g + G * (u0 + uu);
        const uint64_t a = static_cast<uint64_t>(__shfl_sync(kFull, my_lo, k)) |
                           (static_cast<uint64_t>(__shfl_sync(kFull, my_hi, k)) << 32);
        wv[uu] = __shfl_sync(kFull, my_w, k);
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a) + col);
        v[uu][0] = __ldg(p);
        v[uu][1] = __ldg(p + 1);
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const float x[8] = {v[uu][0].x, v[uu][0].y, v[uu][0].z, v[uu][0].w,
                            v[uu][1].x, v[uu][1].y, v[uu][1].z, v[uu][1].w};
        // a zero row (skipped or padding lookup) adds exact zeros
#pragma unroll
        for (int i = 0; i < 8; ++i) comp_add<kWeighted>(hi[i], lo[i], x[i], wv[uu]);
      }
    }
  }
#pragma unroll
  for (int off = S; off < 32; off <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float ho = __shfl_xor_sync(kFull, hi[i], off);
      const float lw = __shfl_xor_sync(kFull, lo[i], off);
      float e;
      two_sum(hi[i], ho, hi[i], e);
      lo[i] = __fadd_rn(__fadd_rn(lo[i], lw), e);
    }
  if (g == 0 && col_ok) {
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r[i] = __fadd_rn(hi[i], lo[i]);
      if (scale != 1.f) r[i] = __fmul_rn(r[i], scale);  // mean pooling
    }
    float4* o = reinterpret_cast<float4*>(out_row + vec * 8);
    __stcs(o, make_float4(r[0], r[1], r[2], r[3]));
    __stcs(o + 1, make_float4(r[4], r[5], r[6], r[7]));
  }
  if (status && __any_sync(kFull, bad) && lane == 0) set_status(status, TBE_ERR_INDEX_RANGE);
}

}  // namespace
}  // namespace tbe
