// Gradient of each table's hot rows on the tensor cores.
//
// The backward's row gradient ("Backward: invert ...": g_r = sum over the
// lookups i of row r of psw_i * grad_out[b_i]) grouped by bag is
//   g[slot][c] = sum_b H[b][slot] * grad_out[b, D_off[t] + c]
// with H the per-bag histogram of the table's hot rows that the preprocess
// built.  For all hot rows of a table at once that is a dense product
// G^T (D_t x B) times H (B x slots), computed here per partition of the bags.
//
// GB300 design: CTA (t, p) owns bags [B p / P, B (p+1) / P) of table t and
// accumulates D^T[c][slot] (M = 128 columns per tile, up to two tiles for
// D_t <= 256; N = the table's hot slots rounded up to 16, at most 256) in
// tensor memory over stages of 32 bags.  Per stage the threads stage the
// gradient rows transposed (A, K-major) and the histogram rows transposed
// (B, K-major), each split into a tf32 high part and an exact fp32
// remainder, and one thread issues kind::tf32 MMAs for hi*hi + lo*hi + hi*lo
// (the last only when the histogram has a remainder: per-sample weights, or
// counts of 2^11 and up).  The next stage's loads are issued before waiting
// for the current stage's MMAs.  The dropped lo*lo term and the MMA's
// truncation of the remainders leave a relative error of about 2^-21 per
// product, below fp32 accumulation error over a bag partition.  The
// accumulator goes to hot_part[t][p][slot][c]; the finishing kernel sums the
// partitions in order.  Every mbarrier wait is bounded (time-out:
// TBE_ERR_TIMEOUT in the status word, drain, free).
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace tbe {
namespace {

constexpr int kGThreads = 256;
constexpr int kGWarps = kGThreads / 32;
constexpr int kGStage = 32;                      // bags per stage (MMA K: 4 steps of 8)
constexpr int kGM = 128;                         // gradient columns per M tile
constexpr uint32_t kGLBO = 128;                  // K-adjacent core matrices
constexpr uint32_t kGSBO = (kGStage / 4) * 128;  // 8-row groups: 8 cores of 4 tf32 (1024 bytes)
constexpr int kGATileBytes = kGM * kGStage * 4;  // 16 KB
constexpr int kGBBytes = kHot * kGStage * 4;     // 32 KB for 256 slots
constexpr int kGAItems = kGM * kGStage / kGThreads;    // 16 per M tile
constexpr int kGBItems = kHot * kGStage / kGThreads;   // up to 32

static_assert(kHot % 16 == 0 && kHot <= 256, "MMA N");
static_assert(kGStage / 4 == kGWarps, "B items: the k group of core matrix warp + 8 j is the warp");

__device__ __forceinline__ void split_tf32(float v, float* hi, float* lo) {
  *hi = __uint_as_float(__float_as_uint(v) & 0xffffe000u);
  *lo = v - *hi;
}

struct HotGradArgs {
  const float* grad_out;
  const int64_t* D_offsets;
  const float* hot_hist;  // [T][B][kHot]
  const uint32_t* hot_n;  // [T]
  float* hot_part;        // [T][parts][kHot][kHotMaxD]
  int* error_word;
  int64_t total_D;
  int B;
  int parts;
  int max_mtiles;         // M tiles the shared memory was sized for
};

struct HotGradTail {
  alignas(8) unsigned long long mbar;
  uint32_t tmem_base;
  int timed_out;
};

// operands: A hi / lo per M tile, then B hi / lo; 16-byte alignment suffices
// (no swizzle), the base is rounded to 128
__host__ __device__ constexpr size_t hot_grad_smem_bytes(int mtiles) {
  return 128 + 2 * static_cast<size_t>(mtiles) * kGATileBytes + 2 * kGBBytes +
         sizeof(HotGradTail);
}

// One stage's loads.  Each warp item covers one 128-byte core matrix,
// lane = 4 (row % 8) + k % 4: A rows are gradient columns, B rows hot slots,
// k the bag within the stage.
struct StageRegs {
  float g[2][kGAItems];
  float h[kGBItems];
};

__device__ __forceinline__ void load_stage(const HotGradArgs& a, int t, int64_t d0, int D,
                                           int mtiles, int nh, int n_slots, int64_t c0, int cnt,
                                           int warp, int lr, int lk, StageRegs& r) {
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int j = 0; j < kGAItems; ++j) {
      const int cm = warp + j * kGWarps;                   // core matrix 0..127
      const int c = mt * kGM + (cm % (kGM / 8)) * 8 + lr;  // gradient column
      const int kb = (cm / (kGM / 8)) * 4 + lk;            // bag within the stage
      r.g[mt][j] = (mt < mtiles && kb < cnt && c < D)
                       ? __ldg(a.grad_out + (c0 + kb) * a.total_D + d0 + c)
                       : 0.f;
    }
  // B items: core matrix cm = 8 sg + kg (k group fastest, a power of two),
  // rows = hot slots 8 sg .. 8 sg + 7
  const int ngroups = n_slots / 8;
  const float* hrow = a.hot_hist + (static_cast<int64_t>(t) * a.B + c0 + lk) * kHot + lr;
#pragma unroll
  for (int j = 0; j < kGBItems; ++j) {
    const int cm = warp + j * kGWarps;
    const int kg = cm & (kGStage / 4 - 1), sg = cm >> 3;
    const int slot = sg * 8 + lr;
    const int kb = kg * 4 + lk;
    r.h[j] = (sg < ngroups && slot < nh && kb < cnt) ? __ldg(hrow + kg * 4 * kHot + sg * 8) : 0.f;
  }
}

__global__ void __launch_bounds__(kGThreads, 2) hot_grad_tc_kernel(HotGradArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  unsigned char* a_hi[2] = {base, base + 2 * kGATileBytes};
  unsigned char* a_lo[2] = {base + kGATileBytes, base + 3 * kGATileBytes};
  unsigned char* b_hi = base + 2 * a.max_mtiles * kGATileBytes;
  unsigned char* b_lo = b_hi + kGBBytes;
  HotGradTail& tl = *reinterpret_cast<HotGradTail*>(b_lo + kGBBytes);

  const int t = blockIdx.x / a.parts;
  const int p = blockIdx.x % a.parts;
  const int64_t d0 = a.D_offsets[t];
  const int D = static_cast<int>(a.D_offsets[t + 1] - d0);
  const int nh = D <= kHotMaxD ? static_cast<int>(min(a.hot_n[t], static_cast<uint32_t>(kHot))) : 0;
  const int mtiles = (D + kGM - 1) / kGM;
  if (nh == 0 || (D & 7) || mtiles > a.max_mtiles) return;  // uniform over the CTA
  const int n_slots = (nh + 15) & ~15;                      // MMA N
  const uint32_t tmem_cols = mtiles == 1 ? 256u : 512u;     // 256 columns per M tile
  const int64_t b_begin = static_cast<int64_t>(a.B) * p / a.parts;
  const int64_t b_end = static_cast<int64_t>(a.B) * (p + 1) / a.parts;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();
  const int lr = static_cast<int>(lane) >> 2, lk = static_cast<int>(lane) & 3;

  if (warp == 0) tmem_alloc(&tl.tmem_base, tmem_cols);
  if (tid == 0) {
    mbar_init(&tl.mbar, 1);
    tl.timed_out = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tl.tmem_base;
  const uint32_t idesc = make_idesc(kFmtTF32, kGM, n_slots);
  uint32_t phase = 0;
  bool pending = false;
  bool first = true;

  StageRegs r;
  if (b_begin < b_end)
    load_stage(a, t, d0, D, mtiles, nh, n_slots, b_begin,
               static_cast<int>(b_end - b_begin < kGStage ? b_end - b_begin : kGStage), warp, lr,
               lk, r);
  for (int64_t c0 = b_begin; c0 < b_end; c0 += kGStage) {
    // stage the loaded values: core matrix cm sits at (cm % groups) * SBO +
    // (cm / groups) * LBO; inside it element (row % 8, k % 4) is at 4 lane
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      if (mt >= mtiles) break;
#pragma unroll
      for (int j = 0; j < kGAItems; ++j) {
        const int cm = warp + j * kGWarps;
        const uint32_t at =
            static_cast<uint32_t>((cm % (kGM / 8)) * kGSBO + (cm / (kGM / 8)) * kGLBO) + lane * 4;
        float hi, lo;
        split_tf32(r.g[mt][j], &hi, &lo);
        *reinterpret_cast<float*>(a_hi[mt] + at) = hi;
        *reinterpret_cast<float*>(a_lo[mt] + at) = lo;
      }
    }
    int lo_here = 0;
    {
      const int ngroups = n_slots / 8;
#pragma unroll
      for (int j = 0; j < kGBItems; ++j) {
        const int cm = warp + j * kGWarps;
        const int kg = cm & (kGStage / 4 - 1), sg = cm >> 3;
        if (sg < ngroups) {
          const uint32_t at = static_cast<uint32_t>(sg * kGSBO + kg * kGLBO) + lane * 4;
          float hi, lo;
          split_tf32(r.h[j], &hi, &lo);
          *reinterpret_cast<float*>(b_hi + at) = hi;
          *reinterpret_cast<float*>(b_lo + at) = lo;
          lo_here |= lo != 0.f;
        }
      }
    }
    // the next stage's loads overlap this stage's MMAs
    const int64_t c1 = c0 + kGStage;
    if (c1 < b_end)
      load_stage(a, t, d0, D, mtiles, nh, n_slots, c1,
                 static_cast<int>(b_end - c1 < kGStage ? b_end - c1 : kGStage), warp, lr, lk, r);
    const int need_lo = __syncthreads_or(lo_here);
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      for (int mt = 0; mt < mtiles; ++mt) {
        const uint32_t acc_tmem = tmem + static_cast<uint32_t>(mt * 256);
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

  float* dst = a.hot_part + (static_cast<int64_t>(t) * a.parts + p) * kHot * kHotMaxD;
  if (!tl.timed_out && first) {
    // no bags in this partition: its partial sums are zero
    for (int i = tid; i < nh * kHotMaxD; i += kGThreads) dst[i] = 0.f;
  }
  if (!tl.timed_out && !first) {
    // D^T[c][slot] -> hot_part[t][p][slot][c]: warp w reads TMEM lanes
    // 32 (w % 4) .. + 31 (columns) of M tile w / 4, the slots in blocks of 32
    const int q = warp & 3;
    const int mt = warp >> 2;
    if (mt < mtiles) {
      const int c = mt * kGM + q * 32 + static_cast<int>(lane);
      for (int s0 = 0; s0 < n_slots; s0 += 32) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                      static_cast<uint32_t>(mt * 256 + s0),
                  v);
        if (c < D)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (s0 + j < nh) dst[(s0 + j) * kHotMaxD + c] = v[j];
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
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

}  // namespace

cudaError_t launch_hot_grad(const Launch& L, const WsLayout& W, char* ws, const float* grad_out) {
  const int max_mtiles = L.d->max_D > kGM ? 2 : 1;
  const size_t smem = hot_grad_smem_bytes(max_mtiles);
  static size_t attr_bytes[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_bytes[dev] != smem) {
    e = cudaFuncSetAttribute(hot_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(hot_grad_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_bytes[dev] = smem;
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
  a.max_mtiles = max_mtiles;
  const unsigned grid = static_cast<unsigned>(L.d->T) * static_cast<unsigned>(W.hot_parts);
  { probe_begin(TBE_PROBE_HOT_GRAD, L.s); hot_grad_tc_kernel<<<grid, kGThreads, smem, L.s>>>(a); note_launch(); probe_end(TBE_PROBE_HOT_GRAD, L.s); }
  return cudaGetLastError();
}

}  // namespace tbe
