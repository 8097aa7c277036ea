// Gradient of each table's hot rows on the tensor cores.
//
// The backward's row gradient ("Backward: invert ...": g_r = sum over the
// lookups i of row r of psw_i * grad_out[b_i]) grouped by bag is
//   g[slot][c] = sum_b H[slot][b] * grad_out[b, D_off[t] + c]
// with H the per-bag histogram of the table's hot rows that the preprocess
// built.  For all hot rows of a table at once that is a dense product
// G^T (D_t x B) times H^T (B x 64), computed here per partition of the bags.
//
// GB300 design: CTA (t, p) owns bags [B p / P, B (p+1) / P) of table t and
// accumulates D^T[c][slot] (M = 128 columns per tile, up to two tiles for
// D_t <= 256; N = 64 slots) in tensor memory over stages of 32 bags.  Per
// stage the threads stage the gradient rows transposed (A, K-major) and the
// histogram columns (B, K-major: the histogram is already slot-major), each
// split into a tf32 high part and an exact fp32 remainder, and one thread
// issues kind::tf32 MMAs for hi*hi + lo*hi + hi*lo (the last only when the
// histogram has a remainder: per-sample weights, or counts of 2^11 and up).
// The dropped lo*lo term and the MMA's truncation of the remainders leave a
// relative error of about 2^-21 per product, below fp32 accumulation error
// over a bag partition.  The accumulator goes to hot_part[t][p][slot][c];
// the finishing kernel sums partitions in order.  Every mbarrier wait is
// bounded (time-out: TBE_ERR_TIMEOUT in the status word, drain, free).
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace tbe {
namespace {

constexpr int kGThreads = 256;
constexpr int kGStage = 32;                   // bags per stage (MMA K: 4 steps of 8)
constexpr int kGM = 128;                      // gradient columns per M tile
constexpr int kGN = kHot;                     // hot slots (MMA N)
constexpr uint32_t kGLBO = 128;               // K-adjacent core matrices
constexpr uint32_t kGSBO = (kGStage / 4) * 128;  // 8-row groups: 8 cores of 4 tf32 (1024 bytes)
constexpr int kGATileBytes = kGM * kGStage * 4;  // 16 KB
constexpr int kGBBytes = kGN * kGStage * 4;      // 8 KB

static_assert(kGN % 16 == 0 && kGN <= 256, "MMA N");

__device__ __forceinline__ void split_tf32(float v, float* hi, float* lo) {
  *hi = __uint_as_float(__float_as_uint(v) & 0xffffe000u);
  *lo = v - *hi;
}

struct HotGradArgs {
  const float* grad_out;
  const int64_t* D_offsets;
  const float* hot_hist;  // [T][kHot][B]
  const uint32_t* hot_n;  // [T]
  float* hot_part;        // [T][parts][kHot][kHotMaxD]
  int* error_word;
  int64_t total_D;
  int B;
  int parts;
};

struct HotGradTail {
  alignas(8) unsigned long long mbar;
  uint32_t tmem_base;
  int timed_out;
};

// operands: A hi / lo for two M tiles, B hi / lo
constexpr size_t kGSmemBytes = 1024 + 4 * static_cast<size_t>(kGATileBytes) + 2 * kGBBytes +
                               sizeof(HotGradTail);
constexpr uint32_t kGTmemCols = 2 * kGN;  // one 64-column accumulator per M tile

__global__ void __launch_bounds__(kGThreads, 2) hot_grad_tc_kernel(HotGradArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* a_hi[2] = {base, base + 2 * kGATileBytes};
  unsigned char* a_lo[2] = {base + kGATileBytes, base + 3 * kGATileBytes};
  unsigned char* b_hi = base + 4 * kGATileBytes;
  unsigned char* b_lo = b_hi + kGBBytes;
  HotGradTail& tl = *reinterpret_cast<HotGradTail*>(b_lo + kGBBytes);

  const int t = blockIdx.x / a.parts;
  const int p = blockIdx.x % a.parts;
  const int nh = static_cast<int>(min(a.hot_n[t], static_cast<uint32_t>(kHot)));
  const int64_t d0 = a.D_offsets[t];
  const int D = static_cast<int>(a.D_offsets[t + 1] - d0);
  if (nh == 0 || D > kHotMaxD || (D & 7)) return;  // uniform over the CTA
  const int mtiles = (D + kGM - 1) / kGM;
  const int64_t b_begin = static_cast<int64_t>(a.B) * p / a.parts;
  const int64_t b_end = static_cast<int64_t>(a.B) * (p + 1) / a.parts;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();

  if (warp == 0) tmem_alloc(&tl.tmem_base, kGTmemCols);
  if (tid == 0) {
    mbar_init(&tl.mbar, 1);
    tl.timed_out = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tl.tmem_base;
  const uint32_t idesc = make_idesc(kFmtTF32, kGM, kGN);
  uint32_t phase = 0;
  bool pending = false;
  bool first = true;

  for (int64_t c0 = b_begin; c0 < b_end; c0 += kGStage) {
    const int cnt = static_cast<int>(b_end - c0 < kGStage ? b_end - c0 : kGStage);
    // Staging maps the 32 lanes of a warp onto one 128-byte core matrix
    // (lane = 4 * (row % 8) + k % 4), so the shared-memory stores are free of
    // bank conflicts; the loads then read 32-byte pieces of 4 gradient rows
    // (A) or 8 histogram rows (B).
    // A: element (c, kb) = grad_out[c0 + kb][d0 + mt * 128 + c]
    const int lr = static_cast<int>(lane) >> 2, lk = static_cast<int>(lane) & 3;
    for (int mt = 0; mt < mtiles; ++mt) {
      constexpr int kAItems = kGM * kGStage / kGThreads;  // 16
      float g[kAItems];
#pragma unroll
      for (int j = 0; j < kAItems; ++j) {
        const int cm = (tid + j * kGThreads) >> 5;           // core matrix 0..127
        const int c = mt * kGM + (cm % (kGM / 8)) * 8 + lr;  // gradient column
        const int kb = (cm / (kGM / 8)) * 4 + lk;            // bag within the stage
        g[j] = (kb < cnt && c < D) ? __ldg(a.grad_out + (c0 + kb) * a.total_D + d0 + c) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kAItems; ++j) {
        // core matrix cm sits at (cm % 16) * SBO + (cm / 16) * LBO; inside it
        // element (row % 8, k % 4) is at 16 (row % 8) + 4 (k % 4) = 4 lane
        const int cm = (tid + j * kGThreads) >> 5;
        const uint32_t at = static_cast<uint32_t>((cm % (kGM / 8)) * kGSBO + (cm / (kGM / 8)) * kGLBO) +
                            lane * 4;
        float hi, lo;
        split_tf32(g[j], &hi, &lo);
        *reinterpret_cast<float*>(a_hi[mt] + at) = hi;
        *reinterpret_cast<float*>(a_lo[mt] + at) = lo;
      }
    }
    // B: element (slot, kb) = H[t][slot][c0 + kb]
    int lo_here = 0;
    {
      constexpr int kBItems = kGN * kGStage / kGThreads;  // 8
      float h[kBItems];
#pragma unroll
      for (int j = 0; j < kBItems; ++j) {
        const int cm = (tid + j * kGThreads) >> 5;        // core matrix 0..63
        const int slot = (cm % (kGN / 8)) * 8 + lr;
        const int kb = (cm / (kGN / 8)) * 4 + lk;
        h[j] = (slot < nh && kb < cnt)
                   ? __ldg(a.hot_hist + (static_cast<int64_t>(t) * kHot + slot) * a.B + c0 + kb)
                   : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kBItems; ++j) {
        const int cm = (tid + j * kGThreads) >> 5;
        const uint32_t at = static_cast<uint32_t>((cm % (kGN / 8)) * kGSBO + (cm / (kGN / 8)) * kGLBO) +
                            lane * 4;
        float hi, lo;
        split_tf32(h[j], &hi, &lo);
        *reinterpret_cast<float*>(b_hi + at) = hi;
        *reinterpret_cast<float*>(b_lo + at) = lo;
        lo_here |= lo != 0.f;
      }
    }
    const int need_lo = __syncthreads_or(lo_here);
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      for (int mt = 0; mt < mtiles; ++mt) {
        const uint32_t acc_tmem = tmem + static_cast<uint32_t>(mt * kGN);
        uint32_t acc = first ? 0u : 1u;
#pragma unroll
        for (int ks = 0; ks < kGStage / 8; ++ks) {
          const uint32_t off = ks * 2 * kGLBO;
          mma_tf32(acc_tmem, make_smem_desc(a_hi[mt] + off, kGLBO, kGSBO),
                   make_smem_desc(b_hi + off, kGLBO, kGSBO), idesc, acc);
          acc = 1;
          mma_tf32(acc_tmem, make_smem_desc(a_lo[mt] + off, kGLBO, kGSBO),
                   make_smem_desc(b_hi + off, kGLBO, kGSBO), idesc, 1u);
          if (need_lo)
            mma_tf32(acc_tmem, make_smem_desc(a_hi[mt] + off, kGLBO, kGSBO),
                     make_smem_desc(b_lo + off, kGLBO, kGSBO), idesc, 1u);
        }
      }
      mma_commit(&tl.mbar);
    }
    first = false;
    pending = true;
    __syncwarp();
    // the operands are rewritten next stage: wait for the MMAs to read them
    const bool done = mbar_wait(&tl.mbar, phase);
    phase ^= 1u;
    if (!done) atomicOr(&tl.timed_out, 1);
    else pending = false;
    fence_after_sync();
    __syncthreads();
    if (tl.timed_out) break;
  }

  if (!tl.timed_out && first) {
    // no bags in this partition: its partial sums are zero
    float* dst = a.hot_part + (static_cast<int64_t>(t) * a.parts + p) * kHot * kHotMaxD;
    for (int i = tid; i < kHot * kHotMaxD; i += kGThreads) dst[i] = 0.f;
  }
  if (!tl.timed_out && !first) {
    // D^T[c][slot] -> hot_part[t][p][slot][c]: warp w reads TMEM lanes
    // 32 (w % 4) .. + 31 (columns) of M tile w / 4, all 64 slots
    const int q = warp & 3;
    const int mt = warp >> 2;
    if (mt < mtiles) {
      const int c = mt * kGM + q * 32 + static_cast<int>(lane);
      float* dst = a.hot_part + (static_cast<int64_t>(t) * a.parts + p) * kHot * kHotMaxD;
      for (int s0 = 0; s0 < kGN; s0 += 32) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                      static_cast<uint32_t>(mt * kGN + s0),
                  v);
        if (c < D)
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[(s0 + j) * kHotMaxD + c] = v[j];
      }
    }
  }
  if (tl.timed_out) {
    if (tid == 0) {
      atomicOr(a.error_word, TBE_ERR_TIMEOUT);
      if (pending) mbar_wait(&tl.mbar, phase ^ 1u);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, kGTmemCols);
}

}  // namespace

cudaError_t launch_hot_grad(const Launch& L, const WsLayout& W, char* ws, const float* grad_out) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(hot_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(hot_grad_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  HotGradArgs a;
  a.grad_out = grad_out;
  a.D_offsets = L.d->D_offsets;
  a.hot_hist = reinterpret_cast<const float*>(ws + W.hot_hist);
  a.hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
  a.hot_part = reinterpret_cast<float*>(ws + W.hot_part);
  a.error_word = reinterpret_cast<int*>(ws + W.status);
  a.total_D = L.d->total_D;
  a.B = L.d->B;
  a.parts = W.hot_parts;
  const unsigned grid = static_cast<unsigned>(L.d->T) * static_cast<unsigned>(W.hot_parts);
  { hot_grad_tc_kernel<<<grid, kGThreads, kGSmemBytes, L.s>>>(a); note_launch(); }
  return cudaGetLastError();
}

}  // namespace tbe
