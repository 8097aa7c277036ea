// Pooled forward (generic gather-and-sum path) and the offsets checker.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Forward:
// keep a narrowly specialized path beside the general one": one launch covers
// every table; each bag gathers the rows its lookups index and sums them,
// fp16 weights accumulating in fp32; the bounds / offset check is a separate
// small kernel and is off by default.
//
// GB300 mapping: one warp per bag.  A row of D_t fp16 values is D_t/8 16-byte
// vectors; S = next_pow2(D_t/8) lanes (at most 32) cover one row, so a warp
// holds G = 32/S lookups of the bag at once and every lane keeps U row
// vectors in flight.  The G partial sums meet through a shuffle butterfly.
// Narrow tables therefore do not leave lanes sized for the widest table idle;
// rows wider than 256 values take several 256-column passes.  Unweighted
// bags accumulate with the mixed-precision add (f16 operand, f32 sum).
#include "common.cuh"
#include "internal.h"

namespace tbe {
namespace {

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
// per-lookup branch (a skipped lookup also gets weight 0).
template <int S, typename IndexT, bool kWeighted>
__device__ __forceinline__ void pool_bag(const __half* __restrict__ Wt, int64_t E, int D, int vec0,
                                         const IndexT* __restrict__ indices,
                                         const float* __restrict__ psw, int64_t start,
                                         int64_t end, float* __restrict__ out_row, int* status) {
  constexpr int G = 32 / S;
  constexpr int U = S < TBE_FWD_UNROLL ? S : TBE_FWD_UNROLL;  // row vectors in flight per lane
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
    const int64_t r = nx_r;
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
      for (int uu = 0; uu < U; ++uu) {
        if (kWeighted) acc_half8(acc, v[uu], wv[uu]);
        else add_half8(acc, v[uu]);
      }
    }
  }

  // Combine the G groups (lanes sl, sl+S, sl+2S, ... hold the same columns).
#pragma unroll
  for (int off = S; off < 32; off <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += __shfl_xor_sync(kFull, acc[i], off);

  if (g == 0 && col_ok) {
    float4* o = reinterpret_cast<float4*>(out_row + vec * 8);
    __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
    __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
  }
  if (status && __any_sync(kFull, bad) && lane == 0) set_status(status, TBE_ERR_INDEX_RANGE);
}

template <typename IndexT, bool kWeighted>
__global__ void __launch_bounds__(256, TBE_FWD_MINB)
    forward_generic_kernel(const __half* __restrict__ W, const int64_t* __restrict__ D_offsets,
                           const int64_t* __restrict__ hash_base,
                           const int64_t* __restrict__ w_offsets,
                           const IndexT* __restrict__ indices, const IndexT* __restrict__ offsets,
                           const float* __restrict__ psw, int64_t n, int T, int B,
                           int64_t total_D, float* __restrict__ out, int* status) {
  const int warps = blockDim.x >> 5;
  const int64_t nbags = static_cast<int64_t>(T) * B;
  for (int64_t bag = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); bag < nbags;
       bag += static_cast<int64_t>(gridDim.x) * warps) {
    const int t = static_cast<int>(bag / B);
    const int64_t b = bag - static_cast<int64_t>(t) * B;
    const int64_t d0 = __ldg(D_offsets + t);
    const int D = static_cast<int>(__ldg(D_offsets + t + 1) - d0);
    if (D < 8 || D > kMaxD || (D & 7)) continue;  // widths the vector path cannot move
    const int64_t E = __ldg(hash_base + t + 1) - __ldg(hash_base + t);
    const __half* Wt = W + __ldg(w_offsets + t);
    int64_t s, e;
    bag_range(offsets, bag, n, &s, &e);
    float* orow = out + b * total_D + d0;
    const int nvec = D >> 3;
    if (nvec <= 1)
      pool_bag<1, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status);
    else if (nvec <= 2)
      pool_bag<2, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status);
    else if (nvec <= 4)
      pool_bag<4, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status);
    else if (nvec <= 8)
      pool_bag<8, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status);
    else if (nvec <= 16)
      pool_bag<16, IndexT, kWeighted>(Wt, E, D, 0, indices, psw, s, e, orow, status);
    else
      for (int vec0 = 0; vec0 < nvec; vec0 += 32)
        pool_bag<32, IndexT, kWeighted>(Wt, E, D, vec0, indices, psw, s, e, orow, status);
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
cudaError_t launch_forward_t(const Launch& L, const __half* W, const IndexT* indices,
                             const IndexT* offsets, const float* psw, float* out, int* status) {
  const tbe_desc* d = L.d;
  const int64_t nbags = static_cast<int64_t>(d->T) * d->B;
  const int warps = 8;
  int64_t blocks = (nbags + warps - 1) / warps;
  if (blocks > (1 << 22)) blocks = 1 << 22;
  if (blocks < 1) blocks = 1;
  if (psw)
    { forward_generic_kernel<IndexT, true><<<static_cast<unsigned>(blocks), warps * 32, 0, L.s>>>(
        W, d->D_offsets, d->hash_base, d->weights_offsets, indices, offsets, psw, L.n, d->T,
        d->B, d->total_D, out, status); note_launch(); }
  else
    { forward_generic_kernel<IndexT, false><<<static_cast<unsigned>(blocks), warps * 32, 0, L.s>>>(
        W, d->D_offsets, d->hash_base, d->weights_offsets, indices, offsets, psw, L.n, d->T,
        d->B, d->total_D, out, status); note_launch(); }
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
                                   int* status) {
  const __half* W = static_cast<const __half*>(weights);
  if (L.d->index_dtype == TBE_DT_I32)
    return launch_forward_t<int32_t>(L, W, static_cast<const int32_t*>(indices),
                                     static_cast<const int32_t*>(offsets), psw, out, status);
  return launch_forward_t<int64_t>(L, W, static_cast<const int64_t*>(indices),
                                   static_cast<const int64_t*>(offsets), psw, out, status);
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
