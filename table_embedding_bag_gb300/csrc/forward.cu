// Pooled forward (generic gather-and-sum path) and the offsets checker.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Forward:
// keep a narrowly specialized path beside the general one": one launch covers
// every table; each bag gathers the rows its lookups index and sums them,
// fp16 (or bf16) weights accumulating in fp32; the bounds / offset check is a
// separate small kernel and is off by default.
//
// GB300 mapping: one warp per bag.  A row of D_t 16-bit values is D_t/8 16-byte
// vectors; S = next_pow2(D_t/8) lanes (at most 32) cover one row, so a warp
// holds G = 32/S lookups of the bag at once and every lane keeps U row
// vectors in flight.  The G partial sums meet through a shuffle butterfly.
// Narrow tables therefore do not leave lanes sized for the widest table idle;
// rows wider than 256 values take several 256-column passes.  Unweighted
// bags accumulate with the mixed-precision add (f16 operand, f32 sum).
#include "common.cuh"
#include "internal.h"
#include "pool.cuh"

namespace tbe {
namespace {

// Weight types of the generic forward: fp16, bf16 (fp32 accumulation) and
// fp32 (compensated accumulation, pool_bag_f32).
constexpr int kWF16 = 0, kWBF16 = 1, kWF32 = 2;

template <typename IndexT, bool kWeighted, int kWT>
__global__ void __launch_bounds__(256, TBE_FWD_MINB)
    forward_generic_kernel(const void* __restrict__ Wv, const int64_t* __restrict__ D_offsets,
                           const int64_t* __restrict__ hash_base,
                           const int64_t* __restrict__ w_offsets,
                           const IndexT* __restrict__ indices, const IndexT* __restrict__ offsets,
                           const float* __restrict__ psw, int64_t n, int T, int B,
                           int64_t total_D, float* __restrict__ out, int* status, bool mean) {
  const int warps = blockDim.x >> 5;
  const int64_t nbags = static_cast<int64_t>(T) * B;
  for (int64_t bag = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); bag < nbags;
       bag += static_cast<int64_t>(gridDim.x) * warps) {
    const int t = static_cast<int>(bag / B);
    const int64_t b = bag - static_cast<int64_t>(t) * B;
    const int64_t d0 = __ldg(D_offsets + t);
    const int D = static_cast<int>(__ldg(D_offsets + t + 1) - d0);
    if (D < 8 || D > kMaxD || (D & 7)) continue;  // widths the vector path cannot move
    const int64_t h0 = __ldg(hash_base + t);
    const int64_t E = __ldg(hash_base + t + 1) - h0;
    const int64_t rbase = 0;
    const int mode = kPoolStore;
    int64_t s, e;
    bag_range(offsets, bag, n, &s, &e);
    // mean pooling: the sum times 1/L for L > 1 lookups
    const float scale = mean && e - s > 1 ? 1.f / static_cast<float>(e - s) : 1.f;
    float* orow = out + b * total_D + d0;
    const int nvec = D >> 3;
    if constexpr (kWT == kWF32) {
      const float* Wt = static_cast<const float*>(Wv) + __ldg(w_offsets + t);
      if (nvec <= 1)
        pool_bag_f32<1, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status, scale);
      else if (nvec <= 2)
        pool_bag_f32<2, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status, scale);
      else if (nvec <= 4)
        pool_bag_f32<4, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status, scale);
      else if (nvec <= 8)
        pool_bag_f32<8, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status, scale);
      else if (nvec <= 16)
        pool_bag_f32<16, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status, scale);
      else
        for (int vec0 = 0; vec0 < nvec; vec0 += 32)
          pool_bag_f32<32, IndexT, kWeighted>(Wt, E, D, vec0, indices, psw, s, e, orow, status,
                                              scale);
      continue;
    }
    constexpr bool kBf16 = kWT == kWBF16;
    const __half* Wt = static_cast<const __half*>(Wv) + __ldg(w_offsets + t);
    if (nvec <= 1)
      pool_bag<1, IndexT, kWeighted, TBE_FWD_UNROLL, kBf16>(Wt, E, rbase, D, 0, indices, psw, s, e, orow, mode, status, scale);
    else if (nvec <= 2)
      pool_bag<2, IndexT, kWeighted, TBE_FWD_UNROLL, kBf16>(Wt, E, rbase, D, 0, indices, psw, s, e, orow, mode, status, scale);
    else if (nvec <= 4)
      pool_bag<4, IndexT, kWeighted, TBE_FWD_UNROLL, kBf16>(Wt, E, rbase, D, 0, indices, psw, s, e, orow, mode, status, scale);
    else if (nvec <= 8)
      pool_bag<8, IndexT, kWeighted, TBE_FWD_UNROLL, kBf16>(Wt, E, rbase, D, 0, indices, psw, s, e, orow, mode, status, scale);
    else if (nvec <= 16)
      pool_bag<16, IndexT, kWeighted, TBE_FWD_UNROLL, kBf16>(Wt, E, rbase, D, 0, indices, psw, s, e, orow, mode, status, scale);
    else
      for (int vec0 = 0; vec0 < nvec; vec0 += 32)
        pool_bag<32, IndexT, kWeighted, TBE_FWD_UNROLL, kBf16>(Wt, E, rbase, D, vec0, indices, psw, s, e, orow, mode,
                                          status, scale);
  }
}

// Cold lists after tbe_preprocess: short bags, so a warp pools G = 32 / S
// consecutive bags at once, one per group of S lanes (S = next_pow2(D / 8)
// for the widest table, at most 32), which multiplies the loads in flight per
// warp by G.  Lookups are linear keys (row = key - hash_base[t]); each
// group's next index batch is loaded while the current one is gathered, and
// when the bag's hot rows were already pooled into out (hot_n given, the
// table has hot rows, D_t <= kHotMaxD) the out row is read at the start and
// added to.  Rows wider than 8 S values take several column passes.
template <int S, bool kWeighted, bool kBf16>
__global__ void __launch_bounds__(256, TBE_FWD_MINB)
    forward_cold_kernel(const __half* __restrict__ W, const int64_t* __restrict__ D_offsets,
                        const int64_t* __restrict__ hash_base, const int64_t* __restrict__ w_offsets,
                        const uint32_t* __restrict__ keys, const uint32_t* __restrict__ cold_off,
                        const float* __restrict__ psw, int T, int B, int64_t total_D,
                        float* __restrict__ out, const uint32_t* __restrict__ hot_n,
                        const float* __restrict__ inv_len) {
  constexpr int G = 32 / S;
  constexpr int U = S < TBE_FWD_UNROLL ? S : TBE_FWD_UNROLL;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
  const int warps = blockDim.x >> 5;
  const int64_t nbags = static_cast<int64_t>(T) * B;
  for (int64_t bag0 = (static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5)) * G;
       bag0 < nbags; bag0 += static_cast<int64_t>(gridDim.x) * warps * G) {
    const int64_t bag = bag0 + g;  // this group's bag
    const bool live = bag < nbags;
    const int t = live ? static_cast<int>(bag / B) : 0;
    const int64_t b = bag - static_cast<int64_t>(t) * B;
    const int64_t d0 = __ldg(D_offsets + t);
    const int D = static_cast<int>(__ldg(D_offsets + t + 1) - d0);
    const int64_t h0 = __ldg(hash_base + t);
    const int64_t E = __ldg(hash_base + t + 1) - h0;
    const __half* Wt = W + __ldg(w_offsets + t);
    const bool add = live && hot_n && D <= kHotMaxD && hot_n[t] != 0;
    const int64_t s = live ? static_cast<int64_t>(__ldg(cold_off + bag)) : 0;
    const int64_t e = live ? static_cast<int64_t>(__ldg(cold_off + bag + 1)) : 0;
    float* orow = out + b * total_D + d0;
    const int nvec = D >> 3;
    // groups may hold tables of different widths: passes run to the widest
    int nvec_max = nvec;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) nvec_max = max(nvec_max, __shfl_xor_sync(kFull, nvec_max, o));
    for (int vec0 = 0; vec0 < nvec_max; vec0 += S) {  // warp-uniform
      const int vec = vec0 + sl;
      const bool col_ok = live && vec < nvec;
      const int col = col_ok ? vec * 8 : 0;
      float acc[8];
      if (add && col_ok) {
        const float4 o0 = reinterpret_cast<const float4*>(orow + col)[0];
        const float4 o1 = reinterpret_cast<const float4*>(orow + col)[1];
        acc[0] = o0.x; acc[1] = o0.y; acc[2] = o0.z; acc[3] = o0.w;
        acc[4] = o1.x; acc[5] = o1.y; acc[6] = o1.z; acc[7] = o1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      }
      int64_t p = s;
      uint32_t nx_key = p + sl < e ? __ldg(keys + p + sl) : 0u;
      float nx_w = (kWeighted && p + sl < e) ? __ldg(psw + p + sl) : 0.f;
      for (;;) {
        const int cnt = static_cast<int>(e - p < S ? (e - p > 0 ? e - p : 0) : S);
        int cmax = cnt;
#pragma unroll
        for (int o = S; o < 32; o <<= 1) cmax = max(cmax, __shfl_xor_sync(kFull, cmax, o));
        if (cmax == 0) break;  // warp-uniform
        const uint32_t key = nx_key;
        const float w_in = nx_w;
        if (p + S + sl < e) {
          nx_key = __ldg(keys + p + S + sl);
          if (kWeighted) nx_w = __ldg(psw + p + S + sl);
        }
        const __half* my_row = reinterpret_cast<const __half*>(g_zero_row);
        float my_w = 0.f;
        if (sl < cnt) {
          const int64_t r = static_cast<int64_t>(key) - h0;
          if (r >= 0 && r < E) {
            my_row = Wt + r * D;
            if (kWeighted) my_w = w_in;
          }
        }
        const uint64_t my_addr = reinterpret_cast<uint64_t>(my_row);
        const uint32_t my_lo = static_cast<uint32_t>(my_addr);
        const uint32_t my_hi = static_cast<uint32_t>(my_addr >> 32);
#pragma unroll
        for (int u0 = 0; u0 < S; u0 += U) {
          if (u0 >= cmax) break;  // warp-uniform
          uint4 v[U];
          float wv[U];
#pragma unroll
          for (int uu = 0; uu < U; ++uu) {
            const int src = g * S + u0 + uu;  // lane of this group holding lookup u0 + uu
            const uint64_t ad = static_cast<uint64_t>(__shfl_sync(kFull, my_lo, src)) |
                                (static_cast<uint64_t>(__shfl_sync(kFull, my_hi, src)) << 32);
            if (kWeighted) wv[uu] = __shfl_sync(kFull, my_w, src);
            v[uu] = ldg_u4(reinterpret_cast<const __half*>(ad) + col);
          }
#pragma unroll
          for (int uu = 0; uu < U; ++uu) acc_row8<kBf16, kWeighted>(acc, v[uu], kWeighted ? wv[uu] : 1.f);
        }
        p += S;
      }
      if (col_ok) {
        if (inv_len) {  // mean pooling: this kernel writes every bag last
          const float sc = __ldg(inv_len + bag);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] *= sc;
        }
        float4* o = reinterpret_cast<float4*>(orow + vec * 8);
        __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
        __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
      }
    }
  }
}

// The same pooling with persistent warps that loop over their bag groups
// through a software pipeline whose intermediate data lives in shared
// memory: while bag group i is pooled, the first S cold keys (and weights)
// of each bag of group i + 1 and the list offsets of group i + 2 are copied
// there by cp.async.  A group then waits for its rows only, not for its
// offsets and keys.
#ifndef TBE_COLD_PIPE
#define TBE_COLD_PIPE 1
#endif

template <int S>
struct ColdPipe {  // one per warp
  uint32_t off[3][32 / S + 1];  // slot: cold_off of the group's bags and the end
  uint32_t key[2][32];          // slot: the first S keys of bag g at [g S + sl]
  float w[2][32];               // and their per-sample weights
};

template <int S, bool kWeighted, bool kBf16>
__global__ void __launch_bounds__(256, TBE_FWD_MINB)
    forward_cold_piped_kernel(const __half* __restrict__ W, const int64_t* __restrict__ D_offsets,
                              const int64_t* __restrict__ hash_base,
                              const int64_t* __restrict__ w_offsets,
                              const uint32_t* __restrict__ keys, const uint32_t* __restrict__ cold_off,
                              const float* __restrict__ psw, int T, int B, int64_t total_D,
                              float* __restrict__ out, const uint32_t* __restrict__ hot_n,
                              const float* __restrict__ inv_len) {
  constexpr int G = 32 / S;
  constexpr int U = S < TBE_FWD_UNROLL ? S : TBE_FWD_UNROLL;
  __shared__ ColdPipe<S> pipes[8];
  ColdPipe<S>& cp = pipes[threadIdx.x >> 5];
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
  const int64_t nbags = static_cast<int64_t>(T) * B;
  const int64_t ngroups = (nbags + G - 1) / G;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  // list offsets of group q into slot os: lanes 0 .. G copy cold_off[q G + l]
  auto stage_off = [&](int64_t q, int os) {
    if (q >= ngroups) return;  // warp-uniform
    if (lane <= G) {
      const int64_t bb = q * G + lane;
      const bool v = bb <= nbags;
      cp_async4(&cp.off[os][lane], cold_off + (v ? bb : 0), v);
    }
  };
  // the first S keys of each bag of group q (offsets in slot os) into slot ks
  auto stage_keys = [&](int64_t q, int os, int ks) {
    if (q >= ngroups) return;
    const bool live = q * G + g < nbags;
    const uint32_t s = cp.off[os][g];
    const uint32_t e = cp.off[os][g + 1];
    const bool v = live && s + static_cast<uint32_t>(sl) < e;
    const uint32_t at = v ? s + static_cast<uint32_t>(sl) : 0u;
    cp_async4(&cp.key[ks][lane], keys + at, v);
    if (kWeighted) cp_async4(&cp.w[ks][lane], psw + at, v);
  };
  const int64_t q0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  stage_off(q0, 0);
  cp_async_commit();
  stage_off(q0 + stride, 1);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  stage_keys(q0, 0, 0);
  cp_async_commit();
  for (uint32_t it = 0;; ++it) {
    const int64_t q = q0 + static_cast<int64_t>(it) * stride;
    if (q >= ngroups) break;
    const int os0 = static_cast<int>(it % 3u), ks0 = static_cast<int>(it & 1u);
    const int os1 = os0 == 2 ? 0 : os0 + 1, os2 = os1 == 2 ? 0 : os1 + 1;
    __syncwarp();  // every lane is done reading the slots refilled below
    stage_off(q + 2 * stride, os2);
    cp_async_commit();
    cp_async_wait<1>();  // group q + 1's offsets and group q's keys are in
    __syncwarp();
    stage_keys(q + stride, os1, ks0 ^ 1);
    cp_async_commit();

    const int64_t bag = q * G + g;  // this group's bag
    const bool live = bag < nbags;
    const int t = live ? static_cast<int>(bag / B) : 0;
    const int64_t b = bag - static_cast<int64_t>(t) * B;
    const int64_t d0 = __ldg(D_offsets + t);
    const int D = static_cast<int>(__ldg(D_offsets + t + 1) - d0);
    const int64_t h0 = __ldg(hash_base + t);
    const int64_t E = __ldg(hash_base + t + 1) - h0;
    const __half* Wt = W + __ldg(w_offsets + t);
    const bool add = live && hot_n && D <= kHotMaxD && hot_n[t] != 0;
    const int64_t s = live ? static_cast<int64_t>(cp.off[os0][g]) : 0;
    const int64_t e = live ? static_cast<int64_t>(cp.off[os0][g + 1]) : 0;
    float* orow = out + b * total_D + d0;
    const int nvec = D >> 3;
    int nvec_max = nvec;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) nvec_max = max(nvec_max, __shfl_xor_sync(kFull, nvec_max, o));
    for (int vec0 = 0; vec0 < nvec_max; vec0 += S) {  // warp-uniform
      const int vec = vec0 + sl;
      const bool col_ok = live && vec < nvec;
      const int col = col_ok ? vec * 8 : 0;
      float acc[8];
      if (add && col_ok) {
        const float4 o0 = reinterpret_cast<const float4*>(orow + col)[0];
        const float4 o1 = reinterpret_cast<const float4*>(orow + col)[1];
        acc[0] = o0.x; acc[1] = o0.y; acc[2] = o0.z; acc[3] = o0.w;
        acc[4] = o1.x; acc[5] = o1.y; acc[6] = o1.z; acc[7] = o1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      }
      int64_t p = s;
      // the first batch of keys is in shared memory (zero past the bag)
      uint32_t nx_key = cp.key[ks0][lane];
      float nx_w = kWeighted ? cp.w[ks0][lane] : 0.f;
      for (;;) {
        const int cnt = static_cast<int>(e - p < S ? (e - p > 0 ? e - p : 0) : S);
        int cmax = cnt;
#pragma unroll
        for (int o = S; o < 32; o <<= 1) cmax = max(cmax, __shfl_xor_sync(kFull, cmax, o));
        if (cmax == 0) break;  // warp-uniform
        const uint32_t key = nx_key;
        const float w_in = nx_w;
        if (p + S + sl < e) {
          nx_key = __ldg(keys + p + S + sl);
          if (kWeighted) nx_w = __ldg(psw + p + S + sl);
        }
        const __half* my_row = reinterpret_cast<const __half*>(g_zero_row);
        float my_w = 0.f;
        if (sl < cnt) {
          const int64_t r = static_cast<int64_t>(key) - h0;
          if (r >= 0 && r < E) {
            my_row = Wt + r * D;
            if (kWeighted) my_w = w_in;
          }
        }
        const uint64_t my_addr = reinterpret_cast<uint64_t>(my_row);
        const uint32_t my_lo = static_cast<uint32_t>(my_addr);
        const uint32_t my_hi = static_cast<uint32_t>(my_addr >> 32);
#pragma unroll
        for (int u0 = 0; u0 < S; u0 += U) {
          if (u0 >= cmax) break;  // warp-uniform
          uint4 v[U];
          float wv[U];
#pragma unroll
          for (int uu = 0; uu < U; ++uu) {
            const int src = g * S + u0 + uu;  // lane of this group holding lookup u0 + uu
            const uint64_t ad = static_cast<uint64_t>(__shfl_sync(kFull, my_lo, src)) |
                                (static_cast<uint64_t>(__shfl_sync(kFull, my_hi, src)) << 32);
            if (kWeighted) wv[uu] = __shfl_sync(kFull, my_w, src);
            v[uu] = ldg_u4(reinterpret_cast<const __half*>(ad) + col);
          }
#pragma unroll
          for (int uu = 0; uu < U; ++uu) acc_row8<kBf16, kWeighted>(acc, v[uu], kWeighted ? wv[uu] : 1.f);
        }
        p += S;
      }
      if (col_ok) {
        if (inv_len) {  // mean pooling: this kernel writes every bag last
          const float sc = __ldg(inv_len + bag);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] *= sc;
        }
        float4* o = reinterpret_cast<float4*>(orow + vec * 8);
        __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
        __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
      }
    }
  }
  cp_async_wait<0>();  // no copy outlives the block's shared memory
}

// Mean pooling's factor of every bag, from its offsets clamped as every
// kernel reads them: 1/L for L > 1 lookups (rows out of range included), else 1.
template <typename IndexT>
__global__ void __launch_bounds__(256)
    mean_factor_kernel(const IndexT* __restrict__ offsets, int64_t nbags, int64_t n,
                       float* __restrict__ inv_len) {
  for (int64_t bag = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; bag < nbags;
       bag += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t s, e;
    bag_range(offsets, bag, n, &s, &e);
    inv_len[bag] = e - s > 1 ? 1.f / static_cast<float>(e - s) : 1.f;
  }
}

// ----------------------------------------------------------- offsets check
// Valid offsets: o[0] = 0, 0 <= o[i] <= o[i+1], o[T*B] <= n.
template <typename IndexT>
__global__ void check_offsets_kernel(const IndexT* __restrict__ offsets, int64_t nb, int64_t n,
                                     int* status) {
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i <= nb;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t o = load_index(offsets, i);
    bad |= o < 0 || o > n || (i == 0 && o != 0);
    if (i < nb) bad |= o > load_index(offsets, i + 1);
  }
  if (__any_sync(kFull, bad) && lane_id() == 0) set_status(status, TBE_ERR_OFFSETS);
}

// Repair o'[0] = 0, o'[i] = max over j <= i of clamp(o[j], 0, n): a prefix
// maximum, done as per-block maxima, a scan of those, and a local scan.
constexpr int kFixThreads = 256;
constexpr int kFixItems = 4;
constexpr int kFixTile = kFixThreads * kFixItems;

template <typename IndexT>
__device__ __forceinline__ int64_t clamped(const IndexT* offsets, int64_t i, int64_t n) {
  if (i == 0) return 0;
  int64_t o = load_index(offsets, i);
  return o < 0 ? 0 : (o > n ? n : o);
}

template <typename IndexT>
__global__ void __launch_bounds__(kFixThreads)
    repair_block_max_kernel(const IndexT* __restrict__ offsets, int64_t nb1, int64_t n,
                            int64_t* __restrict__ block_max) {
  __shared__ int64_t sm[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kFixTile + threadIdx.x * kFixItems;
  int64_t m = 0;
#pragma unroll
  for (int k = 0; k < kFixItems; ++k)
    if (base + k < nb1) m = max(m, clamped(offsets, base + k, n));
  int64_t total;
  block_inclusive_scan(m, OpMax(), int64_t(0), sm, &total);
  if (threadIdx.x == 0) block_max[blockIdx.x] = total;
}

// Single CTA: exclusive prefix maximum of the block maxima, in place.
__global__ void __launch_bounds__(1024) repair_scan_kernel(int64_t* block_max, int64_t nblocks) {
  __shared__ int64_t sm[33];
  __shared__ int64_t inc_of[1024];
  int64_t carry = 0;
  for (int64_t base = 0; base < nblocks; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    const int64_t v = i < nblocks ? block_max[i] : 0;
    int64_t total;
    inc_of[threadIdx.x] = block_inclusive_scan(v, OpMax(), int64_t(0), sm, &total);
    __syncthreads();
    const int64_t exc = threadIdx.x == 0 ? 0 : inc_of[threadIdx.x - 1];
    if (i < nblocks) block_max[i] = max(carry, exc);
    carry = max(carry, total);
    __syncthreads();
  }
}

template <typename IndexT>
__global__ void __launch_bounds__(kFixThreads)
    repair_apply_kernel(const IndexT* __restrict__ offsets, int64_t nb1, int64_t n,
                        const int64_t* __restrict__ carry_in, IndexT* __restrict__ fixed) {
  __shared__ int64_t sm[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kFixTile + threadIdx.x * kFixItems;
  int64_t v[kFixItems];
  int64_t m = 0;
#pragma unroll
  for (int k = 0; k < kFixItems; ++k) {
    v[k] = base + k < nb1 ? clamped(offsets, base + k, n) : 0;
    m = max(m, v[k]);
  }
  __shared__ int64_t inc_of[kFixThreads];
  inc_of[threadIdx.x] = block_inclusive_scan(m, OpMax(), int64_t(0), sm);
  __syncthreads();
  const int64_t exc = threadIdx.x == 0 ? 0 : inc_of[threadIdx.x - 1];
  int64_t run = max(carry_in[blockIdx.x], exc);
#pragma unroll
  for (int k = 0; k < kFixItems; ++k) {
    run = max(run, v[k]);
    if (base + k < nb1) fixed[base + k] = static_cast<IndexT>(run);
  }
}

template <typename IndexT>
cudaError_t launch_forward_t(const Launch& L, const void* W, const IndexT* indices,
                             const IndexT* offsets, const float* psw, float* out, int* status,
                             bool mean) {
  const tbe_desc* d = L.d;
  const int64_t nbags = static_cast<int64_t>(d->T) * d->B;
  const int warps = 8;
  int64_t blocks = (nbags + warps - 1) / warps;
  if (blocks > (1 << 22)) blocks = 1 << 22;
  if (blocks < 1) blocks = 1;
  auto go = [&](auto kernel) {
    kernel<<<static_cast<unsigned>(blocks), warps * 32, 0, L.s>>>(
        W, d->D_offsets, d->hash_base, d->weights_offsets, indices, offsets, psw, L.n, d->T,
        d->B, d->total_D, out, status, mean);
    note_launch();
  };
  const int wt = d->weights_dtype;
  if (psw) {
    if (wt == TBE_DT_F32) go(forward_generic_kernel<IndexT, true, kWF32>);
    else if (wt == TBE_DT_BF16) go(forward_generic_kernel<IndexT, true, kWBF16>);
    else go(forward_generic_kernel<IndexT, true, kWF16>);
  } else {
    if (wt == TBE_DT_F32) go(forward_generic_kernel<IndexT, false, kWF32>);
    else if (wt == TBE_DT_BF16) go(forward_generic_kernel<IndexT, false, kWBF16>);
    else go(forward_generic_kernel<IndexT, false, kWF16>);
  }
  return cudaGetLastError();
}

template <typename IndexT>
cudaError_t launch_offsets_t(const Launch& L, const IndexT* offsets, bool repair, IndexT* fixed,
                             int64_t* scratch, int* status) {
  const int64_t nb = static_cast<int64_t>(L.d->T) * L.d->B;
  int64_t blocks = (nb + 1 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  { check_offsets_kernel<IndexT><<<static_cast<unsigned>(blocks), 256, 0, L.s>>>(offsets, nb, L.n,
                                                                               status); note_launch(); }
  if (!repair) return cudaGetLastError();
  const int64_t nfix = (nb + 1 + kFixTile - 1) / kFixTile;
  { repair_block_max_kernel<IndexT><<<static_cast<unsigned>(nfix), kFixThreads, 0, L.s>>>(
      offsets, nb + 1, L.n, scratch); note_launch(); }
  { repair_scan_kernel<<<1, 1024, 0, L.s>>>(scratch, nfix); note_launch(); }
  { repair_apply_kernel<IndexT><<<static_cast<unsigned>(nfix), kFixThreads, 0, L.s>>>(
      offsets, nb + 1, L.n, scratch, fixed); note_launch(); }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_generic(const Launch& L, const void* weights, const void* indices,
                                   const void* offsets, const float* psw, float* out,
                                   int* status, bool mean) {
  const void* W = weights;
  if (L.d->index_dtype == TBE_DT_I32)
    return launch_forward_t<int32_t>(L, W, static_cast<const int32_t*>(indices),
                                     static_cast<const int32_t*>(offsets), psw, out, status, mean);
  return launch_forward_t<int64_t>(L, W, static_cast<const int64_t*>(indices),
                                   static_cast<const int64_t*>(offsets), psw, out, status, mean);
}

template <int S>
cudaError_t launch_cold_s(const Launch& L, const __half* W, const uint32_t* keys,
                          const uint32_t* cold_off, const float* psw, float* out,
                          const uint32_t* hot_n, const float* inv_len) {
  const tbe_desc* d = L.d;
  const int64_t tasks = (static_cast<int64_t>(d->T) * d->B + (32 / S) - 1) / (32 / S);
  const int warps = 8;
  int64_t blocks = (tasks + warps - 1) / warps;
  if (blocks > (1 << 22)) blocks = 1 << 22;
  // persistent warps for the pipelined kernel: the CTAs the SMs hold at once
  if (TBE_COLD_PIPE && blocks > static_cast<int64_t>(L.num_sms) * TBE_FWD_MINB)
    blocks = static_cast<int64_t>(L.num_sms) * TBE_FWD_MINB;
  if (blocks < 1) blocks = 1;
  auto go = [&](auto kernel) {
    probe_begin(TBE_PROBE_FORWARD_COLD, L.s);
    kernel<<<static_cast<unsigned>(blocks), warps * 32, 0, L.s>>>(
        W, d->D_offsets, d->hash_base, d->weights_offsets, keys, cold_off, psw, d->T, d->B,
        d->total_D, out, hot_n, inv_len);
    note_launch();
    probe_end(TBE_PROBE_FORWARD_COLD, L.s);
  };
  const bool bf16 = d->weights_dtype == TBE_DT_BF16;
#if TBE_COLD_PIPE
  if (psw) {
    if (bf16) go(forward_cold_piped_kernel<S, true, true>);
    else go(forward_cold_piped_kernel<S, true, false>);
  } else {
    if (bf16) go(forward_cold_piped_kernel<S, false, true>);
    else go(forward_cold_piped_kernel<S, false, false>);
  }
#else
  if (psw) {
    if (bf16) go(forward_cold_kernel<S, true, true>);
    else go(forward_cold_kernel<S, true, false>);
  } else {
    if (bf16) go(forward_cold_kernel<S, false, true>);
    else go(forward_cold_kernel<S, false, false>);
  }
#endif
  return cudaGetLastError();
}

cudaError_t launch_forward_cold(const Launch& L, const void* weights, const uint32_t* cold_keys,
                                const uint32_t* cold_off, const float* cold_psw, float* out,
                                const uint32_t* hot_n, const float* inv_len) {
  const __half* W = static_cast<const __half*>(weights);
  const int64_t nvec = L.d->max_D / 8;  // lanes per row for the widest table
  if (nvec <= 1) return launch_cold_s<1>(L, W, cold_keys, cold_off, cold_psw, out, hot_n, inv_len);
  if (nvec <= 2) return launch_cold_s<2>(L, W, cold_keys, cold_off, cold_psw, out, hot_n, inv_len);
  if (nvec <= 4) return launch_cold_s<4>(L, W, cold_keys, cold_off, cold_psw, out, hot_n, inv_len);
  if (nvec <= 8) return launch_cold_s<8>(L, W, cold_keys, cold_off, cold_psw, out, hot_n, inv_len);
  if (nvec <= 16) return launch_cold_s<16>(L, W, cold_keys, cold_off, cold_psw, out, hot_n, inv_len);
  return launch_cold_s<32>(L, W, cold_keys, cold_off, cold_psw, out, hot_n, inv_len);
}

cudaError_t launch_mean_factors(const Launch& L, const void* offsets, float* inv_len) {
  const int64_t nbags = static_cast<int64_t>(L.d->T) * L.d->B;
  int64_t blocks = (nbags + 255) / 256;
  if (blocks > 8LL * L.num_sms) blocks = 8LL * L.num_sms;
  if (blocks < 1) blocks = 1;
  if (L.d->index_dtype == TBE_DT_I32)
    mean_factor_kernel<int32_t><<<static_cast<unsigned>(blocks), 256, 0, L.s>>>(
        static_cast<const int32_t*>(offsets), nbags, L.n, inv_len);
  else
    mean_factor_kernel<int64_t><<<static_cast<unsigned>(blocks), 256, 0, L.s>>>(
        static_cast<const int64_t*>(offsets), nbags, L.n, inv_len);
  note_launch();
  return cudaGetLastError();
}

int64_t repair_scratch_blocks(int64_t nb1) { return (nb1 + kFixTile - 1) / kFixTile; }

cudaError_t launch_check_offsets(const Launch& L, const void* offsets, bool repair, void* fixed,
                                 int64_t* scratch, int* status) {
  if (L.d->index_dtype == TBE_DT_I32)
    return launch_offsets_t<int32_t>(L, static_cast<const int32_t*>(offsets), repair,
                                     static_cast<int32_t*>(fixed), scratch, status);
  return launch_offsets_t<int64_t>(L, static_cast<const int64_t*>(offsets), repair,
                                   static_cast<int64_t*>(fixed), scratch, status);
}

}  // namespace tbe
