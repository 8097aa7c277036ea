// Gradient of each table's hot rows on the tensor cores.
//
// The backward's row gradient ("Backward: invert ...": g_r = sum over the
// lookups i of row r of psw_i * grad_out[b_i]) grouped by bag is
//   g[slot][c] = sum_b H[b][slot] * grad_out[b, D_off[t] + c]
// with H the per-bag histogram of the table's hot rows that the preprocess
// built.  For all hot rows of a table at once that is a dense product
// G^T (D_t x B) times H (B x slots), computed here per partition of the bags.
//
// GB300 design: CTA (t, p) owns the p-th of P runs of whole 32-bag stages of
// table t (so that a stage never straddles two 128-bag histogram tiles) and
// accumulates D^T[c][slot] (M = 128 columns per tile, up to two tiles for
// D_t <= 256; N = the table's hot slots rounded up to 16, at most 256) in
// tensor memory over stages of 32 bags.  Per stage the threads stage the
// gradient rows transposed (A, K-major) and the histogram rows transposed
// (B, K-major; from the byte histogram for byte tiles, the fp32 one for wide
// tiles), each split into a tf32 high part and an exact fp32
// remainder, and one thread issues kind::tf32 MMAs for hi*hi + lo*hi + hi*lo
// (the last only when the histogram has a remainder: per-sample weights, or
// counts of 2^11 and up).  The next stage's loads are issued before waiting
// for the current stage's MMAs.  The dropped lo*lo term and the MMA's
// truncation of the remainders leave a relative error of about 2^-21 per
// product, below fp32 accumulation error over a bag partition.  The tensor
// core's accumulation into tensor memory does not round to nearest, and its
// error grows with the number of MMAs summed into one accumulator (hundreds
// over a long partition); so every few stages (kHotFlushStages,
// kHotFlushStagesWide) the accumulator is added (fp32, round to nearest,
// reductions at L2) into the partition's partial sums in
// hot_part[t][p][slot][c] and restarted.  The finishing kernel sums the
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
// Stages summed into the tensor-memory accumulator between two flushes into
// the partials: byte tiles (hot_grad_bytes_kernel, 2 MMAs per K step of 8
// bags) every 8 stages, wide tiles (hot_grad_tc_kernel, up to 3 MMAs per K
// step, fp32 histogram values with remainders) every 2 stages.  Measured on
// GB300: at 8 stages the wide tiles of the weighted recipe left 0.4 % of the
// element-wise accumulators beyond 1e-5 of the oracle, at 2 stages none
// beyond the 0.1 % the cold rows' fp32 sums allow; the hot-row recipe's byte
// tiles meet 1e-5 (row-wise) at 8.
#ifndef TBE_HOT_FLUSH_STAGES
#define TBE_HOT_FLUSH_STAGES 8
#endif
#ifndef TBE_HOT_FLUSH_STAGES_WIDE
#define TBE_HOT_FLUSH_STAGES_WIDE 2
#endif
constexpr int kHotFlushStages = TBE_HOT_FLUSH_STAGES;
constexpr int kHotFlushStagesWide = TBE_HOT_FLUSH_STAGES_WIDE;

// The accumulator D^T[c][slot] of this CTA stored (add: added) into
// hot_part[t][p][slot][c].  Warps w and w + 4 read TMEM lanes 32 (w % 4) ..
// + 31 (columns): with two M tiles warp w takes tile w / 4, with one the two
// warps share the slot blocks of 32.  Additions are reductions at L2
// (red.global.add.f32: fire and forget, rounded to nearest); each element is
// written by one thread, so a CTA's flushes reach it in program order and
// the result does not depend on timing.  The caller orders the MMAs before
// and after it.
__device__ __forceinline__ void flush_partials(uint32_t tmem, float* dst, int mtiles, int D,
                                               int nh, int n_slots, bool add) {
  const int warp = threadIdx.x >> 5;
  const int q = warp & 3;
  const int half = warp >> 2;
  const int mt = mtiles == 2 ? half : 0;
  const int s_first = mtiles == 2 ? 0 : 32 * half;
  const int s_step = mtiles == 2 ? 32 : 64;
  const int c = mt * 128 + q * 32 + static_cast<int>(lane_id());
  for (int s0 = s_first; s0 < n_slots; s0 += s_step) {
    float v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(mt * 256 + s0), v);
    if (c < D)
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (s0 + j < nh) {
          float* o = dst + (s0 + j) * kHotMaxD + c;
          if (add) atomicAdd(o, v[j]);
          else *o = v[j];
        }
  }
}

__device__ __forceinline__ void split_tf32(float v, float* hi, float* lo) {
  *hi = __uint_as_float(__float_as_uint(v) & 0xffffe000u);
  *lo = v - *hi;
}

struct HotGradArgs {
  const float* grad_out;
  const int64_t* D_offsets;
  const uint8_t* hot_hist8;  // [T][B][kHot] byte tiles
  const float* hot_hist;     // [T][B][kHot] wide tiles
  const uint8_t* tile_kind;  // [T * ceil(B / kHotTileBags)]
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

template <bool kMixed>
__device__ __forceinline__ void load_stage(const HotGradArgs& a, int t, int64_t d0, int D,
                                           int mtiles, int nh, int n_slots, int64_t c0, int cnt,
                                           bool bytes, int warp, int lr, int lk, StageRegs& r) {
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
  const int64_t hoff = (static_cast<int64_t>(t) * a.B + c0 + lk) * kHot + lr;
  if (kMixed && bytes) {
    const uint8_t* hrow = a.hot_hist8 + hoff;
#pragma unroll
    for (int j = 0; j < kGBItems; ++j) {
      const int cm = warp + j * kGWarps;
      const int kg = cm & (kGStage / 4 - 1), sg = cm >> 3;
      const int slot = sg * 8 + lr;
      const int kb = kg * 4 + lk;
      r.h[j] = (sg < ngroups && slot < nh && kb < cnt)
                   ? static_cast<float>(__ldg(hrow + kg * 4 * kHot + sg * 8))
                   : 0.f;
    }
  } else {
    const float* hrow = a.hot_hist + hoff;
#pragma unroll
    for (int j = 0; j < kGBItems; ++j) {
      const int cm = warp + j * kGWarps;
      const int kg = cm & (kGStage / 4 - 1), sg = cm >> 3;
      const int slot = sg * 8 + lr;
      const int kb = kg * 4 + lk;
      r.h[j] = (sg < ngroups && slot < nh && kb < cnt) ? __ldg(hrow + kg * 4 * kHot + sg * 8) : 0.f;
    }
  }
}

// Bags [*b_begin, *b_end) of partition p: whole 32-bag stages, so that a
// stage lies inside one 128-bag histogram tile.
__device__ __forceinline__ void partition_bags(const HotGradArgs& a, int p, int64_t* b_begin,
                                               int64_t* b_end) {
  static_assert(kHotTileBags % kGStage == 0, "stages inside histogram tiles");
  const int64_t nstages = (a.B + kGStage - 1) / kGStage;
  *b_begin = nstages * p / a.parts * kGStage;
  const int64_t e = nstages * (p + 1) / a.parts * kGStage;
  *b_end = e < a.B ? e : a.B;
}

// Which kernel takes a partition: its histogram tiles all bytes, all wide (or
// none), or both.  Contains __syncthreads_or.
enum PartClass { kPartWide = 0, kPartBytes = 1, kPartMixed = 2 };
__device__ __forceinline__ int partition_class(const HotGradArgs& a, int t, int64_t b_begin,
                                               int64_t b_end) {
  const int64_t per_table = (a.B + kHotTileBags - 1) / kHotTileBags;
  int any_bytes = 0, any_wide = 0;
  if (b_begin < b_end)
    for (int64_t i = b_begin / kHotTileBags + threadIdx.x; i <= (b_end - 1) / kHotTileBags;
         i += blockDim.x) {
      const uint8_t k = a.tile_kind[t * per_table + i];
      any_bytes |= k == kTileBytes;
      any_wide |= k != kTileBytes;
    }
  any_bytes = __syncthreads_or(any_bytes);
  any_wide = __syncthreads_or(any_wide);
  return any_bytes ? (any_wide ? kPartMixed : kPartBytes) : kPartWide;
}

// Partitions with wide tiles (kMixed: with byte tiles too; otherwise every
// tile wide, or no bags): register-staged, one stage of loads in flight.
template <bool kMixed>
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
  int64_t b_begin, b_end;
  partition_bags(a, p, &b_begin, &b_end);
  if (partition_class(a, t, b_begin, b_end) != (kMixed ? kPartMixed : kPartWide)) return;
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

  // histogram kind of the stage at bag c (byte or wide tile); read one stage
  // ahead of its loads, so that it adds no latency in front of them
  const uint8_t* kinds = a.tile_kind + static_cast<int64_t>(t) * ((a.B + kHotTileBags - 1) / kHotTileBags);
  auto kind_at = [&](int64_t c) { return c < b_end ? kinds[c / kHotTileBags] : kTileWide; };
  StageRegs r;
  uint8_t kind_next = kind_at(b_begin + kGStage);
  if (b_begin < b_end)
    load_stage<kMixed>(a, t, d0, D, mtiles, nh, n_slots, b_begin,
               static_cast<int>(b_end - b_begin < kGStage ? b_end - b_begin : kGStage),
               kind_at(b_begin) == kTileBytes, warp, lr, lk, r);
  float* dst = a.hot_part + (static_cast<int64_t>(t) * a.parts + p) * kHot * kHotMaxD;
  int flushed = 0;  // flushes of the accumulator into dst so far
  int in_acc = 0;   // stages summed in the accumulator since the last flush
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
    if (c1 < b_end) {
      const bool bytes = kind_next == kTileBytes;
      kind_next = kind_at(c1 + kGStage);
      load_stage<kMixed>(a, t, d0, D, mtiles, nh, n_slots, c1,
                 static_cast<int>(b_end - c1 < kGStage ? b_end - c1 : kGStage), bytes, warp, lr,
                 lk, r);
    }
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
    if (++in_acc == kHotFlushStagesWide && c0 + kGStage < b_end) {
      // into the partials; the next stage restarts the accumulator
      flush_partials(tmem, dst, mtiles, D, nh, n_slots, flushed > 0);
      ++flushed;
      in_acc = 0;
      first = true;
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
    }
  }

  if (!tl.timed_out && first && flushed == 0) {
    // no bags in this partition: its partial sums are zero
    for (int i = tid; i < nh * kHotMaxD; i += kGThreads) dst[i] = 0.f;
  }
  if (!tl.timed_out && !first) flush_partials(tmem, dst, mtiles, D, nh, n_slots, flushed > 0);
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

// ------------------------------------------------------ byte partitions
// Partitions whose tiles all hold byte counts.  Each 32-bag stage is one
// bulk copy of the 8 KB byte histogram plus one bulk copy per gradient row
// (D_t floats) into a ring of kGRing shared buffers, kGRing stages ahead.
// The threads build the operands from shared memory: the gradient split
// into tf32 high part and exact remainder (A, K-major; M = columns), the
// counts as tf32 (B; exact, so no remainder term); one thread issues the
// MMAs (hi x B + lo x B) into the accumulator in tensor memory.  Operands
// are single-buffered: the next stage's conversion waits for this stage's
// MMAs, two CTAs per SM interleave.  Bags past the end of the partition are
// zero in both operands (their ring rows are not copied).
constexpr int kGRing = 2;
constexpr int kGHistBytes = kGStage * kHot;  // 8 KB

struct HotGradBytesTail {
  alignas(8) unsigned long long full[kGRing];
  alignas(8) unsigned long long mma_done;
  uint32_t tmem_base;
  int timed_out;
};

// ring stage: byte histogram, then kGStage gradient rows of up to mtiles x 128 floats
__host__ __device__ constexpr size_t grad_ring_stage_bytes(int mtiles) {
  return kGHistBytes + static_cast<size_t>(kGStage) * mtiles * kGM * 4;
}
__host__ __device__ constexpr size_t hot_grad_bytes_smem_bytes(int mtiles) {
  return 128 + 2 * static_cast<size_t>(mtiles) * kGATileBytes + kGBBytes +
         kGRing * grad_ring_stage_bytes(mtiles) + sizeof(HotGradBytesTail);
}

__global__ void __launch_bounds__(kGThreads, 2) hot_grad_bytes_kernel(HotGradArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  unsigned char* a_hi[2] = {base, base + 2 * kGATileBytes};
  unsigned char* a_lo[2] = {base + kGATileBytes, base + 3 * kGATileBytes};
  unsigned char* b_op = base + 2 * a.max_mtiles * kGATileBytes;
  unsigned char* ring = b_op + kGBBytes;
  const size_t stage_bytes = grad_ring_stage_bytes(a.max_mtiles);
  HotGradBytesTail& tl = *reinterpret_cast<HotGradBytesTail*>(ring + kGRing * stage_bytes);

  const int t = blockIdx.x / a.parts;
  const int p = blockIdx.x % a.parts;
  const int64_t d0 = a.D_offsets[t];
  const int D = static_cast<int>(a.D_offsets[t + 1] - d0);
  const int nh = D <= kHotMaxD ? static_cast<int>(min(a.hot_n[t], static_cast<uint32_t>(kHot))) : 0;
  const int mtiles = (D + kGM - 1) / kGM;
  if (nh == 0 || (D & 7) || mtiles > a.max_mtiles) return;  // uniform over the CTA
  int64_t b_begin, b_end;
  partition_bags(a, p, &b_begin, &b_end);
  if (partition_class(a, t, b_begin, b_end) != kPartBytes) return;
  const int n_slots = (nh + 15) & ~15;
  const uint32_t tmem_cols = mtiles == 1 ? 256u : 512u;
  const int nstages = static_cast<int>((b_end - b_begin + kGStage - 1) / kGStage);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();

  if (warp == 0) tmem_alloc(&tl.tmem_base, tmem_cols);
  if (tid == 0) {
    for (int i = 0; i < kGRing; ++i) mbar_init(&tl.full[i], 1);
    mbar_init(&tl.mma_done, 1);
    tl.timed_out = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tl.tmem_base;
  const uint32_t idesc = make_idesc(kFmtTF32, kGM, n_slots);

  // warp 0 issues stage i into ring slot i % kGRing
  auto issue = [&](int i) {
    const int slot = i % kGRing;
    const int64_t c0 = b_begin + static_cast<int64_t>(i) * kGStage;
    const int cnt = static_cast<int>(b_end - c0 < kGStage ? b_end - c0 : kGStage);
    unsigned char* st = ring + slot * stage_bytes;
    if (lane == 0)
      mbar_expect_tx(&tl.full[slot], static_cast<uint32_t>(cnt) * (kHot + D * 4));
    __syncwarp();
    if (lane == 0)
      bulk_copy_g2s(st, a.hot_hist8 + (static_cast<int64_t>(t) * a.B + c0) * kHot,
                    static_cast<uint32_t>(cnt) * kHot, &tl.full[slot]);
    if (static_cast<int>(lane) < cnt)
      bulk_copy_g2s(st + kGHistBytes + lane * D * 4, a.grad_out + (c0 + lane) * a.total_D + d0,
                    static_cast<uint32_t>(D) * 4, &tl.full[slot]);
  };
  if (warp == 0)
    for (int i = 0; i < kGRing && i < nstages; ++i) issue(i);

  float* dst = a.hot_part + (static_cast<int64_t>(t) * a.parts + p) * kHot * kHotMaxD;
  int consumed = 0, committed = 0, done = 0;
  for (int i = 0; i < nstages; ++i) {
    const int slot = i % kGRing;
    bool ok = mbar_wait(&tl.full[slot], static_cast<uint32_t>(i / kGRing) & 1u);
    ++consumed;
    if (committed > done) {
      const bool mma_ok = mbar_wait(&tl.mma_done, static_cast<uint32_t>(done) & 1u);
      if (mma_ok) ++done;
      ok = ok && mma_ok;
    }
    fence_after_sync();
    if (!ok) atomicOr(&tl.timed_out, 1);
    __syncthreads();
    if (tl.timed_out) break;
    const int64_t c0 = b_begin + static_cast<int64_t>(i) * kGStage;
    const int cnt = static_cast<int>(b_end - c0 < kGStage ? b_end - c0 : kGStage);
    const unsigned char* st = ring + slot * stage_bytes;
    const float* g = reinterpret_cast<const float*>(st + kGHistBytes);
    // A: thread (column cl of each M tile, bag groups kgb + 2 j) reads rows
    // 4 kg .. 4 kg + 3 of its column (consecutive columns across the warp)
    // and writes one 16-byte row of a core matrix (eight consecutive columns
    // hit eight bank groups)
    static_assert(kGThreads == 2 * kGM, "A: two bag groups per pass");
    {
      const int cl = tid & (kGM - 1), kgb = tid >> 7;
      for (int mt = 0; mt < mtiles; ++mt) {
        const int c = mt * kGM + cl;
        const bool col_ok = c < D;
#pragma unroll
        for (int j = 0; j < kGStage / 8; ++j) {
          const int kg = kgb + 2 * j;
          float hi[4], lo[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kb = kg * 4 + q;
            const float v = (kb < cnt && col_ok) ? g[kb * D + c] : 0.f;
            split_tf32(v, &hi[q], &lo[q]);
          }
          const uint32_t at = static_cast<uint32_t>((cl >> 3) * kGSBO + kg * kGLBO + (cl & 7) * 16);
          *reinterpret_cast<float4*>(a_hi[mt] + at) = make_float4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<float4*>(a_lo[mt] + at) = make_float4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
    // B: thread n (one hot slot, n_slots <= 256 threads): the four counts of
    // each bag group as tf32, exact (2^23 + b is a float, minus 2^23)
    static_assert(kGThreads >= kHot, "B: one slot per thread");
    if (tid < n_slots) {
      const int n = tid;
#pragma unroll
      for (int kg = 0; kg < kGStage / 4; ++kg) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int kb = kg * 4 + q;
          const uint32_t b = (kb < cnt && n < nh) ? st[kb * kHot + n] : 0u;
          v[q] = __uint_as_float(0x4b000000u | b) - 8388608.f;
        }
        const uint32_t at = static_cast<uint32_t>((n >> 3) * kGSBO + kg * kGLBO + (n & 7) * 16);
        *reinterpret_cast<float4*>(b_op + at) = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      for (int mt = 0; mt < mtiles; ++mt) {
        const uint32_t acc_tmem = tmem + static_cast<uint32_t>(mt * 256);
#pragma unroll
        for (int ks = 0; ks < kGStage / 8; ++ks) {
          const uint32_t off = ks * 2 * kGLBO;
          mma_tf32(acc_tmem, make_smem_desc(a_hi[mt] + off, kGLBO, kGSBO),
                   make_smem_desc(b_op + off, kGLBO, kGSBO), idesc,
                   ((i % kHotFlushStages) | ks) != 0 ? 1u : 0u);
          mma_tf32(acc_tmem, make_smem_desc(a_lo[mt] + off, kGLBO, kGSBO),
                   make_smem_desc(b_op + off, kGLBO, kGSBO), idesc, 1u);
        }
      }
      mma_commit(&tl.mma_done);
    }
    ++committed;
    // the ring slot just read is free: warp 0 refills it kGRing stages ahead
    if (warp == 0 && i + kGRing < nstages) {
      fence_proxy_async();
      issue(i + kGRing);
    }
    if ((i + 1) % kHotFlushStages == 0 && i + 1 < nstages) {
      // into the partials; stage i + 1 restarts the accumulator
      const bool ok = mbar_wait(&tl.mma_done, static_cast<uint32_t>(done) & 1u);
      if (ok) ++done;
      fence_after_sync();
      if (!ok) atomicOr(&tl.timed_out, 1);
      __syncthreads();
      if (tl.timed_out) break;
      flush_partials(tmem, dst, mtiles, D, nh, n_slots, (i + 1) > kHotFlushStages);
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
    }
  }
  if (!tl.timed_out && committed > done) {
    const bool ok = mbar_wait(&tl.mma_done, static_cast<uint32_t>(done) & 1u);
    if (ok) ++done;
    fence_after_sync();
    if (!ok) atomicOr(&tl.timed_out, 1);
  }
  __syncthreads();
  if (!tl.timed_out) {
    flush_partials(tmem, dst, mtiles, D, nh, n_slots, nstages > kHotFlushStages);
  } else if (tid == 0) {
    atomicOr(a.error_word, TBE_ERR_TIMEOUT);
    // drain (bounded): committed MMAs, issued copies (the stage that timed
    // out included; a completed phase passes)
    if (committed > done) mbar_wait(&tl.mma_done, static_cast<uint32_t>(done) & 1u);
    const int issued = nstages < consumed - 1 + kGRing ? nstages : consumed - 1 + kGRing;
    for (int f = consumed > 0 ? consumed - 1 : 0; f < issued; ++f)
      mbar_wait(&tl.full[f % kGRing], static_cast<uint32_t>(f / kGRing) & 1u);
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
  const size_t bsmem = hot_grad_bytes_smem_bytes(max_mtiles);
  static size_t attr_bytes[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_bytes[dev] != smem) {
    for (const void* k : {reinterpret_cast<const void*>(hot_grad_tc_kernel<false>),
                          reinterpret_cast<const void*>(hot_grad_tc_kernel<true>)}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(hot_grad_bytes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bsmem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(hot_grad_bytes_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_bytes[dev] = smem;
  }
  HotGradArgs a;
  a.grad_out = grad_out;
  a.D_offsets = L.d->D_offsets;
  a.hot_hist8 = reinterpret_cast<const uint8_t*>(ws + W.hot_hist8);
  a.hot_hist = reinterpret_cast<const float*>(ws + W.hot_hist);
  a.tile_kind = reinterpret_cast<const uint8_t*>(ws + W.tile_kind);
  a.hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
  a.hot_part = reinterpret_cast<float*>(ws + W.hot_part);
  a.error_word = reinterpret_cast<int*>(ws + W.status);
  a.total_D = L.d->total_D;
  a.B = L.d->B;
  a.parts = W.hot_parts;
  a.max_mtiles = max_mtiles;
  // every partition is taken by exactly one of the three kernels (byte
  // tiles only, wide tiles only or no bags, both kinds); the others leave
  const unsigned grid = static_cast<unsigned>(L.d->T) * static_cast<unsigned>(W.hot_parts);
  probe_begin(TBE_PROBE_HOT_GRAD, L.s);
  hot_grad_bytes_kernel<<<grid, kGThreads, bsmem, L.s>>>(a);
  note_launch();
  hot_grad_tc_kernel<false><<<grid, kGThreads, smem, L.s>>>(a);
  note_launch();
  hot_grad_tc_kernel<true><<<grid, kGThreads, smem, L.s>>>(a);
  note_launch();
  probe_end(TBE_PROBE_HOT_GRAD, L.s);
  return cudaGetLastError();
}

}  // namespace tbe
