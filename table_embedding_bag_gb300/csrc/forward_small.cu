// Small-table forward on the 5th-generation tensor cores.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Forward:
// keep a narrowly specialized path beside the general one": for one small
// table, count how often each row occurs in each bag, then multiply the
// counts by the table, turning irregular reads into tensor-core work;
// eligibility is one table with E <= 64, 64 <= D <= 128, bags of at least 64
// lookups, fp16 weights, fp32 output and no per-sample weights.
//
// GB300 design (one CTA per tile of 128 bags, persistent over tiles):
//  * the table is staged once per CTA in shared memory as the B operand
//    (N = D rows of K = 64 fp16, K-major, no swizzle; rows E..63 are zero);
//  * the CTA streams the tile's index range (contiguous: 128 consecutive
//    bags) with 8 loads in flight per thread and builds the histogram
//    H[bag][row] with shared-memory atomics, then converts it to fp16 into
//    the A operand (M = 128 bags x K = 64);
//    A count c is split into c_hi = c & ~2047 and c_lo = c & 2047, both exact
//    in fp16; the c_hi operand is multiplied only when some count reaches
//    2048, so the result is exact in the counts whatever the bag length;
//  * one thread issues tcgen05.mma (kind::f16, fp32 accumulate) into a
//    128 x D fp32 accumulator in tensor memory and commits to an mbarrier;
//    the warps then move the accumulator out with tcgen05.ld and store the
//    pooled rows.  Every wait on the mbarrier is bounded: on time-out the CTA
//    records an error in the status word, drains its MMAs (also bounded),
//    frees its tensor memory and stops.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace tbe {
namespace {

constexpr int kM = 128;              // bags per tile (MMA M)
constexpr int kK = 64;               // table rows (MMA K, zero-padded)
constexpr int kThreads = 256;        // 8 warps
constexpr int kCoreBytes = 128;      // 8 rows x 16 bytes
constexpr int kLBO = kCoreBytes;     // next 8 K-elements of the same 8 rows
constexpr int kSBO = (kK / 8) * kCoreBytes;  // next 8 rows (1024 bytes)
constexpr int kTmemCols = 128;       // fp32 accumulator columns (>= D, power of two)

struct SmallSmem {
  alignas(1024) __half a_lo[kM * kK];  // H & 2047, canonical K-major layout
  alignas(1024) __half a_hi[kM * kK];  // H & ~2047
  alignas(1024) __half b[128 * kK];    // W^T rows (N = D <= 128), canonical K-major
  uint32_t counts[kM * kK];            // integer histogram of the tile
  int64_t bag_off[kM + 1];             // the tile's bag offsets, clamped to [0, n]
  alignas(8) unsigned long long mbar;
  uint32_t tmem_base;
  int need_hi;
  int timed_out;
};

// Byte offset of element (row, k) of a K-major operand in the canonical
// no-swizzle layout: 8x8 core matrices of 128 contiguous bytes, K-adjacent
// cores kLBO apart, 8-row groups kSBO apart.
__device__ __forceinline__ int canon_offset(int row, int k) {
  return (row >> 3) * kSBO + (k >> 3) * kLBO + (row & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ uint64_t make_desc(const void* smem_ptr) {
  return make_smem_desc(smem_ptr, kLBO, kSBO);
}

template <typename IndexT>
__global__ void __launch_bounds__(kThreads, 2)
    forward_small_kernel(const __half* __restrict__ W, const IndexT* __restrict__ indices,
                         const IndexT* __restrict__ offsets, int64_t n, int B, int E, int D,
                         float* __restrict__ out, int64_t ld_out, int* status, int* error_word) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  SmallSmem& sm = *reinterpret_cast<SmallSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();

  // Table -> B operand: element (n, k) = W[k][n] for k < E, zero otherwise.
  for (int i = tid; i < 128 * kK; i += kThreads) {
    const int nn = i / kK, k = i % kK;
    const __half v = (nn < D && k < E) ? W[static_cast<int64_t>(k) * D + nn] : __float2half(0.f);
    *reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(sm.b) + canon_offset(nn, k)) = v;
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
  if (tid == 0) {
    mbar_init(&sm.mbar, 1);
    sm.timed_out = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t idesc = make_idesc(kFmtF16, kM, D <= 64 ? 64 : 128);
  const int n_mma = D <= 64 ? 64 : 128;
  uint32_t phase = 0;
  uint32_t drain_phase = 0;
  bool bad = false;
  const int64_t tiles = (static_cast<int64_t>(B) + kM - 1) / kM;

  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t bag0 = tile * kM;
    // 1. histogram of the tile's bags.  The tile's lookups are one contiguous
    //    range of indices; every thread keeps kLoads index loads in flight
    //    and finds each lookup's bag by binary search in the tile offsets.
    for (int i = tid; i < kM * kK; i += kThreads) sm.counts[i] = 0;
    for (int j = tid; j <= kM; j += kThreads) {
      const int64_t bag = bag0 + j < B ? bag0 + j : B;
      int64_t o = load_index(offsets, bag);
      o = o < 0 ? 0 : (o > n ? n : o);
      sm.bag_off[j] = o;
    }
    if (tid == 0) sm.need_hi = 0;
    __syncthreads();
    {
      const int64_t p0 = sm.bag_off[0];
      const int64_t p1 = sm.bag_off[kM];
      constexpr int kLoads = 8;
      for (int64_t base = p0; base < p1; base += static_cast<int64_t>(kThreads) * kLoads) {
        int64_t r[kLoads];
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
          const int64_t p = base + u * kThreads + tid;
          r[u] = p < p1 ? load_index(indices, p) : -1;
        }
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
          const int64_t p = base + u * kThreads + tid;
          if (p >= p1) continue;
          int lo = 0, hi = kM - 1;  // largest bag j with bag_off[j] <= p
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm.bag_off[mid] <= p) lo = mid; else hi = mid - 1;
          }
          if (p >= sm.bag_off[lo + 1]) continue;  // in no bag of the tile
          if (r[u] >= 0 && r[u] < E) atomicAdd(&sm.counts[lo * kK + static_cast<int>(r[u])], 1u);
          else bad = true;
        }
      }
    }
    __syncthreads();
    // 2. counts -> fp16 A operands (exact split at 2048)
    int hi_here = 0;
    for (int i = tid; i < kM * kK; i += kThreads) {
      const int m = i / kK, k = i % kK;
      const uint32_t c = sm.counts[i];
      const int off = canon_offset(m, k);
      *reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(sm.a_lo) + off) =
          __uint2half_rn(c & 2047u);
      *reinterpret_cast<__half*>(reinterpret_cast<unsigned char*>(sm.a_hi) + off) =
          __uint2half_rn(c & ~2047u);
      hi_here |= c > 2047u;
    }
    if (__syncthreads_or(hi_here) && tid == 0) sm.need_hi = 1;
    fence_proxy_async();  // make the generic-proxy smem writes visible to the tensor core
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // 3. one thread issues the MMAs (K = 64 in four steps of 16)
    if (tid == 0) {
      const int parts = sm.need_hi ? 2 : 1;
      uint32_t acc = 0;
      for (int part = 0; part < parts; ++part) {
        const __half* a = part == 0 ? sm.a_lo : sm.a_hi;
#pragma unroll
        for (int ks = 0; ks < kK / 16; ++ks) {
          const uint64_t ad = make_desc(reinterpret_cast<const unsigned char*>(a) + ks * 2 * kLBO);
          const uint64_t bd =
              make_desc(reinterpret_cast<const unsigned char*>(sm.b) + ks * 2 * kLBO);
          mma_f16(tmem, ad, bd, idesc, acc);
          acc = 1;
        }
      }
      mma_commit(&sm.mbar);
    }
    __syncwarp();
    // 4. wait for the accumulator, then store the pooled rows
    const bool done = mbar_wait(&sm.mbar, phase);
    drain_phase = phase;
    phase ^= 1u;
    if (!done) atomicOr(&sm.timed_out, 1);
    fence_after_sync();
    __syncthreads();
    if (sm.timed_out) break;
    {
      const int lane_grp = warp & 3;               // TMEM lanes 32*lane_grp ..
      const int col_half = warp >> 2;              // warps 4..7 take the upper columns
      const int m = lane_grp * 32 + static_cast<int>(lane);
      const int64_t bag = bag0 + m;
      for (int c0 = col_half * 32; c0 < n_mma; c0 += 64) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(lane_grp * 32) << 16) + static_cast<uint32_t>(c0), v);
        if (bag < B) {
          float* o = out + bag * ld_out;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            if (c0 + j < D) __stcs(reinterpret_cast<float4*>(o + c0 + j), make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]));
        }
      }
    }
    fence_before_sync();
    __syncthreads();  // accumulator and A buffers free for the next tile
    fence_after_sync();
  }

  if (sm.timed_out) {
    // Drain: give outstanding MMAs a bounded time to finish before the
    // tensor memory is released.
    if (tid == 0) {
      atomicOr(error_word, TBE_ERR_TIMEOUT);
      mbar_wait(&sm.mbar, drain_phase);
    }
    __syncthreads();
  }
  if (status && __any_sync(kFull, bad) && lane == 0) set_status(status, TBE_ERR_INDEX_RANGE);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

constexpr size_t kSmallSmemBytes = sizeof(SmallSmem) + 1024;

template <typename IndexT>
cudaError_t launch_small_t(const Launch& L, const __half* W, const IndexT* indices,
                           const IndexT* offsets, float* out, int* status, int* error_word) {
  const tbe_desc* d = L.d;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(forward_small_kernel<IndexT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmallSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t tiles = (static_cast<int64_t>(d->B) + kM - 1) / kM;
  int64_t grid = 2LL * L.num_sms;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  { forward_small_kernel<IndexT><<<static_cast<unsigned>(grid), kThreads, kSmallSmemBytes, L.s>>>(
      W, indices, offsets, L.n, d->B, static_cast<int>(d->total_E), static_cast<int>(d->total_D),
      out, d->total_D, status, error_word); note_launch(); }
  return cudaGetLastError();
}

}  // namespace

bool small_table_eligible(const tbe_desc* d, int64_t n, bool weighted) {
  if (weighted || d->T != 1 || d->weights_dtype != TBE_DT_F16) return false;
  if (d->total_E < 1 || d->total_E > kK) return false;
  if (d->total_D < 64 || d->total_D > 128 || (d->total_D & 15)) return false;
  return n >= 64LL * d->B;  // bags of at least 64 lookups on average
}

cudaError_t launch_forward_small(const Launch& L, const void* weights, const void* indices,
                                 const void* offsets, float* out, int* status, int* error_word) {
  const __half* W = static_cast<const __half*>(weights);
  if (L.d->index_dtype == TBE_DT_I32)
    return launch_small_t<int32_t>(L, W, static_cast<const int32_t*>(indices),
                                   static_cast<const int32_t*>(offsets), out, status, error_word);
  return launch_small_t<int64_t>(L, W, static_cast<const int64_t*>(indices),
                                 static_cast<const int64_t*>(offsets), out, status, error_word);
}

}  // namespace tbe
