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
#include "pool.cuh"

namespace tbe {
namespace {

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
      pool_bag<1, IndexT, kWeighted>(Wt, E, 0, D, 0, indices, psw, s, e, orow, true, status);
    else if (nvec <= 2)
      pool_bag<2, IndexT, kWeighted>(Wt, E, 0, D, 0, indices, psw, s, e, orow, true, status);
    else if (nvec <= 4)
      pool_bag<4, IndexT, kWeighted>(Wt, E, 0, D, 0, indices, psw, s, e, orow, true, status);
    else if (nvec <= 8)
      pool_bag<8, IndexT, kWeighted>(Wt, E, 0, D, 0, indices, psw, s, e, orow, true, status);
    else if (nvec <= 16)
      pool_bag<16, IndexT, kWeighted>(Wt, E, 0, D, 0, indices, psw, s, e, orow, true, status);
    else
      for (int vec0 = 0; vec0 < nvec; vec0 += 32)
        pool_bag<32, IndexT, kWeighted>(Wt, E, 0, D, vec0, indices, psw, s, e, orow, true,
                                          status);
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
