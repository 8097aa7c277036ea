// Pooled forward after tbe_preprocess: hot rows on the tensor cores, cold
// lookups gathered.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Forward:
// keep a narrowly specialized path beside the general one", counts how often
// each row occurs in each bag and multiplies the counts by the table for one
// small table.  Here the same product serves the few rows of every table
// that take most of the lookups: tbe_preprocess has already built, per table
// t and tile of 128 bags, the histogram H[slot][bag] of the table's hot rows
// (at most 64, chosen by the previous backward) and the list of the other,
// cold, lookups of each bag in lookup order.  For bag b of table t
//
//   out[b, D_off[t] : D_off[t] + D_t] = sum_slot H[slot][b] * W_t[hot(slot)]
//                                      + sum over b's cold lookups of W_t[row]
//
// which is the plain pooled sum with the hot lookups grouped by row.
//
// GB300 design (persistent CTAs of 16 warps, one tile of 128 bags of one
// table at a time):
//  * the hot rows of the tile's table are staged in shared memory as the B
//    operand (N = D_t rounded up to 16, K = 64 slots, tf32 = the fp16 values
//    widened, exactly), rebuilt only when the table changes;
//  * the histogram tile becomes the A operand (M = 128 bags x K = 64), split
//    exactly into a tf32 high part and a remainder (zero for integer counts
//    below 2^11, which then costs nothing);
//  * one thread issues tcgen05.mma kind::tf32 into a 128 x N fp32
//    accumulator in tensor memory while all warps gather the tile's cold
//    lookups (warp per bag, the generic forward's gather loop) and store the
//    cold sums;
//  * after a bounded wait on the MMA's mbarrier the warps add the
//    accumulator (tcgen05.ld) to the stored cold sums.
// Tables without hot rows (no histogram, D_t > 256, or an empty set) take
// only the gather.  On an mbarrier time-out the CTA records TBE_ERR_TIMEOUT,
// drains its MMAs (bounded), frees its tensor memory and stops.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "pool.cuh"
#include "tcgen05.cuh"

namespace tbe {
namespace {

#ifndef TBE_FWDHOT_UNROLL
#define TBE_FWDHOT_UNROLL 4  // cold-gather row vectors in flight per lane
#endif

constexpr int kFM = kHotTileBags;          // bags per tile = MMA M (128)
constexpr int kFK = kHot;                  // hot slots = MMA K (64)
constexpr int kFThreads = 512;             // 16 warps
constexpr int kFWarps = kFThreads / 32;
constexpr uint32_t kFLBO = 128;            // K-adjacent core matrices
constexpr uint32_t kFSBO = (kFK / 4) * 128;  // 8-row groups: 16 cores of 4 tf32 (2048 bytes)
constexpr int kAOperandBytes = kFM * kFK * 4;

static_assert(kFM == 128, "tile = MMA M = 128");
static_assert(kFK % 8 == 0, "tf32 MMA K step is 8");
static_assert((kFM * kFK) % kFThreads == 0, "A tile splits evenly over the threads");

// Byte offset of element (row, k) of a K-major tf32 operand.
__device__ __forceinline__ uint32_t canon_tf32(int row, int k) {
  return static_cast<uint32_t>((row >> 3) * kFSBO + (k >> 2) * kFLBO + (row & 7) * 16 + (k & 3) * 4);
}

struct FwdHotArgs {
  const __half* W;
  const int64_t* D_offsets;
  const int64_t* hash_base;
  const int64_t* w_offsets;
  const uint32_t* cold_keys;   // linear keys of the cold lookups, per bag in lookup order
  const float* cold_psw;       // their per-sample weights (weighted only)
  const uint32_t* bag_cold;    // [T*B] cold lookups per bag
  const uint32_t* tile_base;   // [tiles] first cold entry of each tile
  const uint32_t* hot_keys;    // [T][kHot] this batch's hot rows
  const uint32_t* hot_n;       // [T]
  const float* hot_hist;       // [T][kHot][B], or null: no hot rows
  float* out;
  int* error_word;
  int64_t total_D;
  int T;
  int B;
  int n_max;                   // B operand rows allotted in shared memory
};

// Shared memory: A high part, A remainder, B (n_max rows), then the small
// fields.  The MMA operands sit at 1024-byte multiples from the aligned base.
struct FwdHotTail {
  uint32_t cold_off[kFM + 1];
  uint32_t scan[33];
  alignas(8) unsigned long long mbar;
  uint32_t tmem_base;
  int need_lo;
  int timed_out;
  int b_table;
};

__host__ __device__ constexpr size_t fwd_hot_smem_bytes(int n_max) {
  return 1024 + 2 * static_cast<size_t>(kAOperandBytes) + static_cast<size_t>(n_max) * kFK * 4 +
         sizeof(FwdHotTail);
}

template <typename F>
__device__ __forceinline__ void pool_cold(int D, F&& pool) {
  const int nvec = D >> 3;
  if (nvec <= 1) pool(std::integral_constant<int, 1>(), 0);
  else if (nvec <= 2) pool(std::integral_constant<int, 2>(), 0);
  else if (nvec <= 4) pool(std::integral_constant<int, 4>(), 0);
  else if (nvec <= 8) pool(std::integral_constant<int, 8>(), 0);
  else if (nvec <= 16) pool(std::integral_constant<int, 16>(), 0);
  else
    for (int vec0 = 0; vec0 < nvec; vec0 += 32) pool(std::integral_constant<int, 32>(), vec0);
}

template <bool kWeighted>
__global__ void __launch_bounds__(kFThreads, 2) forward_hot_kernel(FwdHotArgs a, uint32_t tmem_cols) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* a_hi = base;
  unsigned char* a_lo = base + kAOperandBytes;
  unsigned char* b_op = base + 2 * kAOperandBytes;
  FwdHotTail& tl = *reinterpret_cast<FwdHotTail*>(b_op + static_cast<size_t>(a.n_max) * kFK * 4);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();

  if (warp == 0) tmem_alloc(&tl.tmem_base, tmem_cols);
  if (tid == 0) {
    mbar_init(&tl.mbar, 1);
    tl.timed_out = 0;
    tl.b_table = -1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tl.tmem_base;
  uint32_t phase = 0, drain_phase = 0;
  bool pending = false;  // an MMA commit whose phase the drain must wait for

  // each CTA takes a contiguous range of tiles: consecutive tiles share a
  // table, so its hot rows stay staged
  const int64_t per_table = (a.B + kFM - 1) / kFM;
  const int64_t tiles = per_table * a.T;
  const int64_t tile_begin = tiles * blockIdx.x / gridDim.x;
  const int64_t tile_end = tiles * (blockIdx.x + 1) / gridDim.x;
  for (int64_t tile = tile_begin; tile < tile_end; ++tile) {
    const int t = static_cast<int>(tile / per_table);
    const int64_t b0 = (tile % per_table) * kFM;
    const int nbags = static_cast<int>(a.B - b0 < kFM ? a.B - b0 : kFM);
    const int64_t d0 = __ldg(a.D_offsets + t);
    const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - d0);
    const int64_t h0 = __ldg(a.hash_base + t);
    const int64_t E = __ldg(a.hash_base + t + 1) - h0;
    const __half* Wt = a.W + __ldg(a.w_offsets + t);
    const int n_pad = (D + 15) & ~15;
    const int nh = (a.hot_hist != nullptr && D <= kHotMaxD && n_pad <= a.n_max)
                       ? static_cast<int>(min(a.hot_n[t], static_cast<uint32_t>(kHot)))
                       : 0;

    // cold list offsets of the tile's bags
    {
      const uint32_t c = tid < nbags ? a.bag_cold[static_cast<int64_t>(t) * a.B + b0 + tid] : 0u;
      uint32_t total;
      const uint32_t inc = block_inclusive_scan(c, OpSum(), 0u, tl.scan, &total);
      const uint32_t tb = a.tile_base[tile];
      if (tid < kFM) tl.cold_off[tid] = tb + inc - c;
      if (tid == 0) tl.cold_off[kFM] = tb + total;
    }

    if (nh > 0) {
      // B operand: element (n, k) = W_t[hot row k][n], zero past D or nh
      if (tl.b_table != t) {
        // 8 columns (one 16-byte load) per item
        const int ng = n_pad >> 3;
        for (int i = tid; i < ng * kFK; i += kFThreads) {
          const int k = i / ng, n0 = (i % ng) * 8;
          uint4 raw = make_uint4(0u, 0u, 0u, 0u);
          if (k < nh && n0 < D) {
            // a key outside the table never had lookups counted: zero row
            const int64_t row = static_cast<int64_t>(a.hot_keys[t * kHot + k]) - h0;
            if (row >= 0 && row < E) raw = ldg_u4(Wt + row * D + n0);
          }
          const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(h2[j]);
            *reinterpret_cast<float*>(b_op + canon_tf32(n0 + 2 * j, k)) = f.x;
            *reinterpret_cast<float*>(b_op + canon_tf32(n0 + 2 * j + 1, k)) = f.y;
          }
        }
      }
      // A operand: histogram tile, high part and remainder (all of a
      // thread's loads are issued before the first store)
      int lo_here = 0;
      constexpr int kPer = kFM * kFK / kFThreads;
      float hv[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = tid + j * kFThreads;
        const int k = i / kFM, m = i % kFM;
        hv[j] = (k < nh && m < nbags)
                    ? __ldg(a.hot_hist + (static_cast<int64_t>(t) * kHot + k) * a.B + b0 + m)
                    : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = tid + j * kFThreads;
        const int k = i / kFM, m = i % kFM;
        const float hi = __uint_as_float(__float_as_uint(hv[j]) & 0xffffe000u);
        const float lo = hv[j] - hi;
        *reinterpret_cast<float*>(a_hi + canon_tf32(m, k)) = hi;
        *reinterpret_cast<float*>(a_lo + canon_tf32(m, k)) = lo;
        lo_here |= lo != 0.f;
      }
      const int need_lo = __syncthreads_or(lo_here);
      if (tid == 0) tl.b_table = t;
      fence_proxy_async();
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
      if (tid == 0) {
        const uint32_t idesc = make_idesc(kFmtTF32, kFM, n_pad);
        uint32_t acc = 0;
        for (int part = 0; part < (need_lo ? 2 : 1); ++part) {
          const unsigned char* aop = part == 0 ? a_hi : a_lo;
#pragma unroll
          for (int ks = 0; ks < kFK / 8; ++ks) {
            mma_tf32(tmem, make_smem_desc(aop + ks * 2 * kFLBO, kFLBO, kFSBO),
                     make_smem_desc(b_op + ks * 2 * kFLBO, kFLBO, kFSBO), idesc, acc);
            acc = 1;
          }
        }
        mma_commit(&tl.mbar);
      }
      pending = true;
      __syncwarp();
    } else {
      __syncthreads();  // cold offsets visible
    }

    // cold lookups: one warp per bag
    for (int lb = warp; lb < nbags; lb += kFWarps) {
      const int64_t s = tl.cold_off[lb], e = tl.cold_off[lb + 1];
      float* orow = a.out + (b0 + lb) * a.total_D + d0;
      pool_cold(D, [&](auto S_, int vec0) {
        constexpr int S = decltype(S_)::value;
        pool_bag<S, uint32_t, kWeighted, TBE_FWDHOT_UNROLL>(Wt, E, h0, D, vec0, a.cold_keys,
                                                            a.cold_psw, s, e, orow, nh == 0,
                                                            nullptr);
      });
    }

    if (nh > 0) {
      const bool done = mbar_wait(&tl.mbar, phase);
      drain_phase = phase;
      phase ^= 1u;
      if (!done) atomicOr(&tl.timed_out, 1);
      else pending = false;
      fence_after_sync();
      __syncthreads();  // also makes the cold sums visible to every warp
      if (tl.timed_out) break;
      // out += accumulator: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its
      // bags) and every fourth 32-column block starting at block w / 4
      const int q = warp & 3;
      const int m = q * 32 + static_cast<int>(lane);
      for (int c0 = (warp >> 2) * 32; c0 < n_pad; c0 += 128) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
        if (m < nbags) {
          float* o = a.out + (b0 + m) * a.total_D + d0 + c0;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            if (c0 + j < D) {
              float4 x = *reinterpret_cast<float4*>(o + j);
              x.x += v[j]; x.y += v[j + 1]; x.z += v[j + 2]; x.w += v[j + 3];
              __stcs(reinterpret_cast<float4*>(o + j), x);
            }
        }
      }
    }
    fence_before_sync();
    __syncthreads();  // operands, accumulator and cold offsets free for the next tile
    fence_after_sync();
  }

  if (tl.timed_out) {
    if (tid == 0) {
      atomicOr(a.error_word, TBE_ERR_TIMEOUT);
      if (pending) mbar_wait(&tl.mbar, drain_phase);
    }
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

template <bool kWeighted>
cudaError_t launch_hot_t(const Launch& L, const FwdHotArgs& a, size_t smem, uint32_t tmem_cols) {
  static size_t attr_bytes[64][2] = {};
  static int ctas_per_sm[64][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int wi = kWeighted ? 1 : 0;
  if (attr_bytes[dev][wi] != smem) {
    e = cudaFuncSetAttribute(forward_hot_kernel<kWeighted>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // all of the unified L1 / shared storage as shared memory, so that the
    // two CTAs the registers allow also fit
    e = cudaFuncSetAttribute(forward_hot_kernel<kWeighted>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int smem_per_sm = 0;
    e = cudaDeviceGetAttribute(&smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    // 1 KB of each CTA's shared memory is reserved by the driver; the
    // launch bounds (512 threads, 2 CTAs) fix the register share
    int per_sm = static_cast<int>(static_cast<size_t>(smem_per_sm) / (smem + 1024));
    if (per_sm > 2) per_sm = 2;
    ctas_per_sm[dev][wi] = per_sm < 1 ? 1 : per_sm;
    attr_bytes[dev][wi] = smem;
  }
  const int64_t tiles = static_cast<int64_t>(a.T) * ((a.B + kFM - 1) / kFM);
  // at most 512 TMEM columns per SM: resident CTAs x tmem_cols must fit
  int per_sm = ctas_per_sm[dev][wi];
  if (per_sm * static_cast<int>(tmem_cols) > 512) per_sm = static_cast<int>(512 / tmem_cols);
  int64_t grid = static_cast<int64_t>(per_sm) * L.num_sms;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  { forward_hot_kernel<kWeighted><<<static_cast<unsigned>(grid), kFThreads, smem, L.s>>>(a, tmem_cols); note_launch(); }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_hot(const Launch& L, const WsLayout& W, char* ws, const void* weights,
                               const float* psw, float* out) {
  const tbe_desc* d = L.d;
  FwdHotArgs a;
  a.W = static_cast<const __half*>(weights);
  a.D_offsets = d->D_offsets;
  a.hash_base = d->hash_base;
  a.w_offsets = d->weights_offsets;
  a.cold_keys = reinterpret_cast<const uint32_t*>(ws + W.keys[2]);
  a.cold_psw = psw ? reinterpret_cast<const float*>(ws + W.psw[2]) : nullptr;
  a.bag_cold = reinterpret_cast<const uint32_t*>(ws + W.bag_cold);
  a.tile_base = reinterpret_cast<const uint32_t*>(ws + W.tile_cold);
  a.hot_keys = reinterpret_cast<const uint32_t*>(ws + W.hot_keys(W.hot_cur));
  a.hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
  a.hot_hist = W.hot_enabled ? reinterpret_cast<const float*>(ws + W.hot_hist) : nullptr;
  a.out = out;
  a.error_word = reinterpret_cast<int*>(ws + W.status);
  a.total_D = d->total_D;
  a.T = d->T;
  a.B = d->B;
  // B operand rows: the widest table that can hold hot rows, rounded to 16
  const int64_t widest = d->max_D < kHotMaxD ? d->max_D : kHotMaxD;
  a.n_max = static_cast<int>((widest + 15) & ~15);
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(a.n_max)) tmem_cols <<= 1;
  const size_t smem = fwd_hot_smem_bytes(a.n_max);
  return psw ? launch_hot_t<true>(L, a, smem, tmem_cols) : launch_hot_t<false>(L, a, smem, tmem_cols);
}

}  // namespace tbe
