// Pooled forward after tbe_preprocess: hot rows on the tensor cores, then
// the cold lookups gathered on top.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Forward:
// keep a narrowly specialized path beside the general one", counts how often
// each row occurs in each bag and multiplies the counts by the table for one
// small table.  Here the same product serves the rows of every table that
// take most of the lookups: tbe_preprocess has already built, per table t,
// the histogram H[b][slot] of the table's hot rows (up to kHot, chosen by the
// previous backward) and the per-bag lists of the other, cold, lookups.  For
// bag b of table t
//
//   out[b, D_off[t] : D_off[t] + D_t] = sum_slot H[b][slot] * W_t[hot(slot)]
//                                      + sum over b's cold lookups of W_t[row]
//
// which is the plain pooled sum with the hot lookups grouped by row.  This
// kernel writes the first term for the tables that have hot rows; the
// generic kernel over the cold lists then adds the second (forward.cu).
//
// GB300 design (persistent CTAs over contiguous ranges of 128-bag tiles, two
// per SM for D_t <= 128):
//  * the table's hot rows are staged once per table as the B operand, fp16
//    as stored (N = D_t rounded up to 16, K = the hot slots, K-major, no
//    swizzle);
//  * per 64-slot chunk, the tile's histogram rows become the A operand
//    (M = 128 bags).  Each bag's row is scaled by 2^s_b (s_b from the
//    preprocess: the row's largest entry lands in [2^14, 2^15)) and split
//    exactly into up to three fp16 parts (high, middle, low); integer counts
//    need only the high part, and the other parts' MMAs are issued only when
//    some entry needs them.  The next chunk's histogram is loaded while the
//    current chunk's MMAs run;
//  * one thread issues tcgen05.mma kind::f16 (fp32 accumulate; products of
//    fp16 values are exact) into a 128 x N accumulator in tensor memory;
//    after a bounded wait the warps store the accumulator times 2^-s_b
//    (exact) as the bags' partial sums.
// On an mbarrier time-out the CTA records TBE_ERR_TIMEOUT, drains its MMAs
// (bounded), frees its tensor memory and stops.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace tbe {
namespace {

constexpr int kFM = kHotTileBags;                 // bags per tile = MMA M (128)
constexpr int kFChunk = 64;                       // hot slots per A chunk
constexpr int kFThreads = 512;                    // 16 warps
constexpr uint32_t kFLBO = 128;                   // K-adjacent core matrices
constexpr uint32_t kFSBOA = (kFChunk / 8) * 128;  // A: 8 cores of 8 fp16 per 8-row group
constexpr uint32_t kFSBOB = (kHot / 8) * 128;     // B: all hot slots along K
constexpr int kAPartBytes = kFM * kFChunk * 2;    // 16 KB
constexpr int kFItems = kFM * kFChunk / 2 / kFThreads;  // slot pairs per thread per chunk

static_assert(kFM == 128, "tile = MMA M = 128");
static_assert(kHot % kFChunk == 0, "hot slots in whole chunks");

struct FwdHotArgs {
  const __half* W;
  const int64_t* D_offsets;
  const int64_t* hash_base;
  const int64_t* w_offsets;
  const uint32_t* hot_keys;  // [T][kHot] this batch's hot rows
  const uint32_t* hot_n;     // [T]
  const uint8_t* hot_hist8;  // [T][B][kHot] byte tiles
  const float* hot_hist;     // [T][B][kHot] wide tiles
  const int8_t* hot_scale;   // [T*B] wide tiles
  const uint8_t* tile_kind;  // [T * ceil(B / kFM)]
  float* out;
  int* error_word;
  int64_t total_D;
  int T;
  int B;
  int n_max;                 // B operand rows allotted in shared memory
};

struct FwdHotTail {
  alignas(8) unsigned long long mbar;
  uint32_t tmem_base;
  int timed_out;
  int b_table;
  int64_t row_off[kHot];  // element offset of each hot row in its table, -1: none
  int8_t scale[kFM];
};

// Operands need 16-byte alignment (no swizzle); the base is rounded to 128.
__host__ __device__ constexpr size_t fwd_hot_smem_bytes(int n_max) {
  return 128 + 3 * static_cast<size_t>(kAPartBytes) + static_cast<size_t>(n_max) * kHot * 2 +
         sizeof(FwdHotTail);
}

// 2^e as a float, for |e| <= 126 (exact scaling).
__device__ __forceinline__ float pow2(int e) { return __int_as_float((127 + e) << 23); }

// Histogram pairs (slots k, k + 1) of chunk c for this thread's items; a warp
// covers one core matrix (8 bags x 8 slots) per item, lane = 4 (m % 8) + (k % 8) / 2.
__device__ __forceinline__ void load_chunk(const FwdHotArgs& a, int t, int64_t b0, int nbags,
                                           int nh, int c, int warp, int lr, int lk,
                                           float2 (&x)[kFItems]) {
#pragma unroll
  for (int j = 0; j < kFItems; ++j) {
    const int cm = warp + j * (kFThreads / 32);  // core matrix 0..127
    const int m = (cm % (kFM / 8)) * 8 + lr;
    const int k = c * kFChunk + (cm / (kFM / 8)) * 8 + lk * 2;
    // entries of slots in [nh, nh rounded to 64) are zeros written by the preprocess
    x[j] = (m < nbags && k < nh)
               ? __ldg(reinterpret_cast<const float2*>(
                     a.hot_hist + (static_cast<int64_t>(t) * a.B + b0 + m) * kHot + k))
               : make_float2(0.f, 0.f);
  }
}

// B operand of table t (once per table and CTA): element (n, k) =
// W_t[hot row k][n], zero past D or nh.  A warp fills one 128-byte core
// matrix (8 n x 8 k) per step, lane = 4 (n % 8) + (k % 8) / 2, two k per
// lane.  row_off (kHot entries of shared memory) takes the hot rows' offsets
// first, so that the row loads are independent.  Contains __syncthreads; the
// caller makes sure no MMA still reads b_op.
__device__ __forceinline__ void stage_hot_rows(const FwdHotArgs& a, int t, int D, int nh,
                                               int nchunks, int n_pad, unsigned char* b_op,
                                               int64_t* row_off) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();
  const int lr = static_cast<int>(lane) >> 2, lk = static_cast<int>(lane) & 3;
  const int64_t h0 = __ldg(a.hash_base + t);
  const int64_t E = __ldg(a.hash_base + t + 1) - h0;
  const __half* Wt = a.W + __ldg(a.w_offsets + t);
  for (int k = tid; k < nchunks * kFChunk; k += blockDim.x) {
    int64_t off = -1;
    if (k < nh) {
      // a key outside the table never had lookups counted: zero row
      const int64_t row = static_cast<int64_t>(a.hot_keys[t * kHot + k]) - h0;
      if (row >= 0 && row < E) off = row * D;
    }
    row_off[k] = off;
  }
  __syncthreads();
  const int ngroups = n_pad / 8;
  const int ncores = ngroups * nchunks * (kFChunk / 8);
  const int nwarps = static_cast<int>(blockDim.x >> 5);
#pragma unroll 4
  for (int cm = warp; cm < ncores; cm += nwarps) {
    const int ng = cm % ngroups, kg = cm / ngroups;
    const int nn = ng * 8 + lr;
    __half v[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int64_t off = row_off[kg * 8 + lk * 2 + q];
      v[q] = (off >= 0 && nn < D) ? Wt[off + nn] : __float2half(0.f);
    }
    *reinterpret_cast<__half2*>(b_op + ng * kFSBOB + kg * kFLBO + lane * 4) =
        __halves2half2(v[0], v[1]);
  }
}

// 16-bit operand values of either weight type (kBf16: bf16, else fp16): the
// round-to-nearest conversion from fp32 and back.
template <bool kBf16>
__device__ __forceinline__ uint16_t to16(float v) {
  if constexpr (kBf16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  else return __half_as_ushort(__float2half_rn(v));
}
template <bool kBf16>
__device__ __forceinline__ float from16(uint16_t h) {
  if constexpr (kBf16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  else return __half2float(__ushort_as_half(h));
}

// Wide tiles only (per-sample weights, or counts above 255 in some bag).
// kBf16: bf16 weights, and the histogram split into bf16 parts (three 8-bit
// significands hold any fp32 value exactly, as three fp16 parts do).
template <bool kBf16>
__global__ void __launch_bounds__(kFThreads, 2) forward_hot_kernel(FwdHotArgs a, uint32_t tmem_cols) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  unsigned char* a_part[3] = {base, base + kAPartBytes, base + 2 * kAPartBytes};
  unsigned char* b_op = base + 3 * kAPartBytes;
  FwdHotTail& tl = *reinterpret_cast<FwdHotTail*>(b_op + static_cast<size_t>(a.n_max) * kHot * 2);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();
  const int lr = static_cast<int>(lane) >> 2, lk = static_cast<int>(lane) & 3;

  const int64_t per_table = (a.B + kFM - 1) / kFM;
  const int64_t tiles = per_table * a.T;
  const int64_t tile_begin = tiles * blockIdx.x / gridDim.x;
  const int64_t tile_end = tiles * (blockIdx.x + 1) / gridDim.x;
  {
    // nothing to do (the usual case without per-sample weights): leave
    // before allocating tensor memory
    int mine = 0;
    for (int64_t i = tile_begin + tid; i < tile_end; i += kFThreads)
      mine |= a.tile_kind[i] == kTileWide;
    if (!__syncthreads_or(mine)) return;
  }

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
  uint32_t phase = 0;
  bool pending = false;

  for (int64_t tile = tile_begin; tile < tile_end; ++tile) {
    if (a.tile_kind[tile] != kTileWide) continue;  // uniform
    const int t = static_cast<int>(tile / per_table);
    const int64_t d0 = __ldg(a.D_offsets + t);
    const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - d0);
    const int nh =
        D <= kHotMaxD ? static_cast<int>(min(a.hot_n[t], static_cast<uint32_t>(kHot))) : 0;
    const int n_pad = (D + 15) & ~15;
    if (nh == 0 || n_pad > a.n_max) continue;  // uniform: the cold kernel stores these bags
    const int64_t b0 = (tile % per_table) * kFM;
    const int nbags = static_cast<int>(a.B - b0 < kFM ? a.B - b0 : kFM);
    const int nchunks = (nh + kFChunk - 1) / kFChunk;
    float2 x[kFItems];
    load_chunk(a, t, b0, nbags, nh, 0, warp, lr, lk, x);

    if (tl.b_table != t) {
      stage_hot_rows(a, t, D, nh, nchunks, n_pad, b_op, tl.row_off);
      if (tid == 0) tl.b_table = t;
    }
    if (tid < kFM) tl.scale[tid] = tid < nbags ? a.hot_scale[static_cast<int64_t>(t) * a.B + b0 + tid] : 0;
    __syncthreads();

    for (int c = 0; c < nchunks; ++c) {
      // A parts of chunk c: H[b0 + m][64 c + k] * 2^s_m split exactly in
      // three fp16 parts
      int need = 0;  // bit 0: middle parts, bit 1: low parts
#pragma unroll
      for (int j = 0; j < kFItems; ++j) {
        const int cm = warp + j * (kFThreads / 32);
        const int mg = cm % (kFM / 8), kg = cm / (kFM / 8);
        const float mul = pow2(tl.scale[mg * 8 + lr]);
        const float v[2] = {x[j].x * mul, x[j].y * mul};
        uint16_t p[3][2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          p[0][q] = to16<kBf16>(v[q]);
          const float r1 = v[q] - from16<kBf16>(p[0][q]);
          p[1][q] = to16<kBf16>(r1);
          const float r2 = r1 - from16<kBf16>(p[1][q]);
          p[2][q] = to16<kBf16>(r2);
          need |= (r1 != 0.f ? 1 : 0) | (r2 != 0.f ? 2 : 0);
        }
        const uint32_t off = static_cast<uint32_t>(mg * kFSBOA + kg * kFLBO) + lane * 4;
#pragma unroll
        for (int part = 0; part < 3; ++part)
          *reinterpret_cast<uint32_t*>(a_part[part] + off) =
              static_cast<uint32_t>(p[part][0]) | (static_cast<uint32_t>(p[part][1]) << 16);
      }
      // the next chunk's histogram loads overlap this chunk's MMAs
      if (c + 1 < nchunks) load_chunk(a, t, b0, nbags, nh, c + 1, warp, lr, lk, x);
      const int need_mid = __syncthreads_or(need & 1) ? 1 : 0;
      const int need_lo = __syncthreads_or(need & 2) ? 1 : 0;
      fence_proxy_async();
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
      if (tid == 0) {
        const uint32_t idesc = make_idesc(kBf16 ? kFmtBF16 : kFmtF16, kFM, n_pad);
        const int parts = need_lo ? 3 : (need_mid ? 2 : 1);
        for (int part = 0; part < parts; ++part) {
#pragma unroll
          for (int ks = 0; ks < kFChunk / 16; ++ks) {
            const uint32_t acc = (c == 0 && part == 0 && ks == 0) ? 0u : 1u;
            mma_f16(tmem, make_smem_desc(a_part[part] + ks * 2 * kFLBO, kFLBO, kFSBOA),
                    make_smem_desc(b_op + (c * (kFChunk / 8) + ks * 2) * kFLBO, kFLBO, kFSBOB),
                    idesc, acc);
          }
        }
        mma_commit(&tl.mbar);
      }
      pending = true;
      __syncwarp();
      // the A parts are rewritten by the next chunk: wait for the MMAs
      const bool done = mbar_wait(&tl.mbar, phase);
      phase ^= 1u;
      if (!done) atomicOr(&tl.timed_out, 1);
      else pending = false;
      fence_after_sync();
      __syncthreads();
      if (tl.timed_out) break;
    }
    if (tl.timed_out) break;

    // out[b0 + m, d0 + n] = acc[m][n] * 2^-s_m: warp w reads TMEM lanes
    // 32 (w % 4) .. + 31 (its bags) and every fourth 32-column block from w / 4
    {
      const int q = warp & 3;
      const int m = q * 32 + static_cast<int>(lane);
      const float unscale = pow2(-tl.scale[m]);
      for (int c0 = (warp >> 2) * 32; c0 < n_pad; c0 += (kFThreads / 128) * 32) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
        if (m < nbags) {
          float* o = a.out + (b0 + m) * a.total_D + d0 + c0;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            if (c0 + j < D)
              *reinterpret_cast<float4*>(o + j) =
                  make_float4(v[j] * unscale, v[j + 1] * unscale, v[j + 2] * unscale,
                              v[j + 3] * unscale);
        }
      }
    }
    fence_before_sync();
    __syncthreads();  // accumulator and per-bag scales free for the next tile
    fence_after_sync();
  }

  if (tl.timed_out) {
    if (tid == 0) {
      atomicOr(a.error_word, TBE_ERR_TIMEOUT);
      if (pending) mbar_wait(&tl.mbar, phase ^ 1u);
    }
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// ------------------------------------------------------------- byte tiles
// Tiles whose counts are bytes (no per-sample weights, at most 255 lookups of
// one hot row in a bag): the tile's 128 x 256 histogram is one contiguous
// 32 KB block, fetched by one bulk copy into a ring of `stages` buffers,
// `stages` tiles ahead.  Per tile every thread converts four 16-byte pieces
// (16 slots of one bag) to fp16, exact, into the A operand (four 64-slot
// chunks, the layout of the wide kernel); one thread issues the 16 MMAs
// (K = 256) into one of two accumulators and refills the ring buffer just
// read; then the warps store the previous tile's accumulator, so that its
// epilogue overlaps this tile's MMAs.  No scaling: counts and fp16 weights
// multiply exactly, and the sums are fp32 accumulations.
constexpr int kBThreads = 512;
constexpr int kBRawBytes = kFM * kHot;             // 32 KB
constexpr int kBAOpBytes = kFM * kHot * 2;         // 64 KB: four chunks of kAPartBytes
constexpr int kBMaxStages = 4;
static_assert(kHot == 256 && kBAOpBytes == 4 * kAPartBytes, "byte tiles: 256 slots, 4 chunks");

struct FwdBytesTail {
  alignas(8) unsigned long long full[kBMaxStages];
  alignas(8) unsigned long long mma_done;
  alignas(8) unsigned long long never;  // test-only builds: nothing arrives on it
  uint32_t tmem_base;
  int timed_out;
  int b_table;
  int64_t row_off[kHot];
};

// Epilogue transpose buffer: per warp 32 rows x 16 columns of fp32.
constexpr int kBXposeBytes = (kBThreads / 32) * 32 * 16 * 4;  // 32 KB

__host__ __device__ constexpr size_t fwd_bytes_smem_bytes(int n_max, int stages, bool xpose) {
  return 128 + static_cast<size_t>(n_max) * kHot * 2 + kBAOpBytes +
         static_cast<size_t>(stages) * kBRawBytes + (xpose ? kBXposeBytes : 0) +
         sizeof(FwdBytesTail);
}

// Bytes 2 i and 2 i + 1 of w as two fp16 values: 1024 + b is exact in fp16
// (exponent 10, b in the mantissa), minus 1024 exactly.
__device__ __forceinline__ uint32_t bytes_to_half2(uint32_t w, uint32_t sel) {
  const uint32_t x = __byte_perm(w, 0x64646464u, sel);
  __half2 h = *reinterpret_cast<const __half2*>(&x);
  h = __hsub2(h, __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6400))));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The same for bf16: 2^23 + b is exact in fp32, minus 2^23 exactly gives b,
// whose upper 16 bits are its bf16 value (b has at most 8 significant bits).
__device__ __forceinline__ uint32_t bytes_to_bf162(uint32_t w, uint32_t sel) {
  const uint32_t x = __byte_perm(w, 0u, sel);  // the two bytes in bits 0-7 and 16-23
  const float f0 = __uint_as_float(0x4b000000u | (x & 0xffu)) - 8388608.f;
  const float f1 = __uint_as_float(0x4b000000u | (x >> 16)) - 8388608.f;
  return __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);
}

template <bool kBf16>
__device__ __forceinline__ uint32_t bytes_to_16x2(uint32_t w, uint32_t sel) {
  if constexpr (kBf16) return bytes_to_bf162(w, sel);
  else return bytes_to_half2(w, sel);
}

// kXpose: the epilogue goes through a per-warp shared buffer so that every
// global store instruction writes 8 rows x 64 contiguous bytes (full
// sectors); without it (no room for the buffer: D_t > 128) a lane stores its
// own row.
// kBf16: bf16 weights and counts (counts up to 255 are exact bf16 values).
template <bool kXpose, bool kBf16>
__global__ void __launch_bounds__(kBThreads, 1)
    forward_bytes_kernel(FwdHotArgs a, uint32_t tmem_cols, int stages) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  unsigned char* b_op = base;
  unsigned char* a_op = b_op + static_cast<size_t>(a.n_max) * kHot * 2;
  unsigned char* raw = a_op + kBAOpBytes;
  unsigned char* xpose = raw + static_cast<size_t>(stages) * kBRawBytes;
  FwdBytesTail& tl = *reinterpret_cast<FwdBytesTail*>(xpose + (kXpose ? kBXposeBytes : 0));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const unsigned lane = lane_id();

  const int64_t per_table = (a.B + kFM - 1) / kFM;
  const int64_t tiles = per_table * a.T;
  const int64_t tile_begin = tiles * blockIdx.x / gridDim.x;
  const int64_t tile_end = tiles * (blockIdx.x + 1) / gridDim.x;
  {
    int mine = 0;
    for (int64_t i = tile_begin + tid; i < tile_end; i += kBThreads)
      mine |= a.tile_kind[i] == kTileBytes;
    if (!__syncthreads_or(mine)) return;
  }
  // the next byte tile at or after `from` (all threads walk the same list)
  auto next_tile = [&](int64_t from) {
    while (from < tile_end && a.tile_kind[from] != kTileBytes) ++from;
    return from;
  };
  auto tile_bags = [&](int64_t tile) {
    const int64_t b0 = (tile % per_table) * kFM;
    return static_cast<int>(a.B - b0 < kFM ? a.B - b0 : kFM);
  };

  if (warp == 0) tmem_alloc(&tl.tmem_base, 2 * tmem_cols);
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) mbar_init(&tl.full[i], 1);
    mbar_init(&tl.mma_done, 1);
    mbar_init(&tl.never, 1);
    tl.timed_out = 0;
    tl.b_table = -1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tl.tmem_base;

  // producer (thread 0): tiles fetched so far and the next one to fetch
  int64_t fetch_at = tile_begin;
  uint32_t fetched = 0;
  auto fetch = [&](int slot) {
    fetch_at = next_tile(fetch_at);
    if (fetch_at >= tile_end) return;
    const int t = static_cast<int>(fetch_at / per_table);
    const int64_t b0 = (fetch_at % per_table) * kFM;
    const uint32_t bytes = static_cast<uint32_t>(tile_bags(fetch_at)) * kHot;
    mbar_expect_tx(&tl.full[slot], bytes);
    bulk_copy_g2s(raw + static_cast<size_t>(slot) * kBRawBytes,
                  a.hot_hist8 + (static_cast<int64_t>(t) * a.B + b0) * kHot, bytes, &tl.full[slot]);
    ++fetch_at;
    ++fetched;
  };
  if (tid == 0)
    for (int i = 0; i < stages; ++i) fetch(i);

  uint32_t consumed = 0;   // tiles taken from the ring
  uint32_t committed = 0;  // tiles whose MMAs were committed
  uint32_t done = 0;       // tiles whose MMAs are known complete
  int64_t prev_tile = -1;
  int prev_t = 0, prev_D = 0, prev_npad = 0;

  // out rows of a finished tile: acc[m][n] for bags m < nbags, columns < D
  auto epilogue = [&](int64_t tile, int t, int D, int n_pad, uint32_t acc_col) {
    const int64_t b0 = (tile % per_table) * kFM;
    const int nbags = tile_bags(tile);
    const int64_t d0 = __ldg(a.D_offsets + t);
    const int q = warp & 3;
    const int m = q * 32 + static_cast<int>(lane);
    for (int c0 = (warp >> 2) * 32; c0 < n_pad; c0 += (kBThreads / 128) * 32) {
      float v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc_col + static_cast<uint32_t>(c0), v);
      if constexpr (kXpose) {
        // 16 columns at a time: lane = row writes four 16-byte chunks, chunk
        // c of row r at r * 64 + (c ^ ((r >> 1) & 3)) * 16, so eight
        // consecutive rows fill eight bank groups; then four lanes per row
        // read a row's 64 bytes back (eight rows per instruction)
        unsigned char* xb = xpose + warp * (32 * 16 * 4);
        const int lr4 = static_cast<int>(lane) >> 2, lc = static_cast<int>(lane) & 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<float4*>(xb + lane * 64 + ((c ^ ((lane >> 1) & 3)) * 16)) =
                make_float4(v[16 * h + 4 * c], v[16 * h + 4 * c + 1], v[16 * h + 4 * c + 2],
                            v[16 * h + 4 * c + 3]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int r = 8 * k + lr4;
            const float4 x = *reinterpret_cast<const float4*>(xb + r * 64 + ((lc ^ ((r >> 1) & 3)) * 16));
            const int mm = q * 32 + r;
            const int col = c0 + 16 * h + 4 * lc;
            if (mm < nbags && col < D)
              *reinterpret_cast<float4*>(a.out + (b0 + mm) * a.total_D + d0 + col) = x;
          }
          __syncwarp();
        }
      } else if (m < nbags) {
        float* o = a.out + (b0 + m) * a.total_D + d0 + c0;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (c0 + j < D) *reinterpret_cast<float4*>(o + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
  };

  int t = -1, D = 0, nh = 0, n_pad = 0, nchunks = 0;  // the current tile's table
  for (int64_t tile = next_tile(tile_begin); tile < tile_end; tile = next_tile(tile + 1)) {
    if (tile / per_table != t) {
      t = static_cast<int>(tile / per_table);
      D = static_cast<int>(__ldg(a.D_offsets + t + 1) - __ldg(a.D_offsets + t));
      nh = static_cast<int>(min(a.hot_n[t], static_cast<uint32_t>(kHot)));
      n_pad = (D + 15) & ~15;
      nchunks = (nh + kFChunk - 1) / kFChunk;
    }
    const int slot = static_cast<int>(consumed % static_cast<uint32_t>(stages));
    // this tile's bytes, and the previous tile's MMAs (A and B are rewritten)
    bool ok = (TBE_TEST_STUCK_WAIT > 0 && consumed == 0)
                  ? mbar_wait(&tl.never, 0u, TBE_TEST_STUCK_WAIT)
                  : mbar_wait(&tl.full[slot], (consumed / static_cast<uint32_t>(stages)) & 1u);
    ++consumed;
    if (committed > done) {
      const bool mma_ok = mbar_wait(&tl.mma_done, done & 1u);
      if (mma_ok) ++done;
      ok = ok && mma_ok;
    }
    fence_after_sync();
    if (!ok) atomicOr(&tl.timed_out, 1);
    __syncthreads();
    if (tl.timed_out) break;
    if (tl.b_table != t) {
      // tables with hot rows are at most kHotMaxD wide, so n_pad <= n_max
      stage_hot_rows(a, t, D, nh, nchunks, n_pad, b_op, tl.row_off);
      if (tid == 0) tl.b_table = t;
    }
    // bytes -> fp16 A operand.  Item (bag m, 16 slots from k0): the eight
    // lanes of a quarter warp take bags 8 mg .. 8 mg + 7 at rotated slot
    // groups, so that both the 16-byte reads (row stride 256 bytes) and the
    // core-matrix writes fall in eight distinct bank groups.
    const unsigned char* rt = raw + static_cast<size_t>(slot) * kBRawBytes;
#pragma unroll
    for (int j = 0; j < (kFM * kHot / 16) / kBThreads; ++j) {
      const int item = tid + j * kBThreads;
      const int p = item & 7, r = item >> 3;
      const int mg = r & 15, kq = r >> 4;
      const int m = mg * 8 + p;
      const int k0 = ((kq + p) & 15) * 16;
      const uint4 w = *reinterpret_cast<const uint4*>(rt + m * kHot + k0);
      uint4 h0, h1;
      h0.x = bytes_to_16x2<kBf16>(w.x, 0x4140u);
      h0.y = bytes_to_16x2<kBf16>(w.x, 0x4342u);
      h0.z = bytes_to_16x2<kBf16>(w.y, 0x4140u);
      h0.w = bytes_to_16x2<kBf16>(w.y, 0x4342u);
      h1.x = bytes_to_16x2<kBf16>(w.z, 0x4140u);
      h1.y = bytes_to_16x2<kBf16>(w.z, 0x4342u);
      h1.z = bytes_to_16x2<kBf16>(w.w, 0x4140u);
      h1.w = bytes_to_16x2<kBf16>(w.w, 0x4342u);
      unsigned char* dst = a_op + (k0 >> 6) * kAPartBytes + mg * kFSBOA + ((k0 & 63) >> 3) * kFLBO + p * 16;
      *reinterpret_cast<uint4*>(dst) = h0;
      *reinterpret_cast<uint4*>(dst + kFLBO) = h1;
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t acc_col = (committed & 1u) * tmem_cols;
    if (tid == 0) {
      const uint32_t idesc = make_idesc(kBf16 ? kFmtBF16 : kFmtF16, kFM, n_pad);
      for (int c = 0; c < nchunks; ++c)
#pragma unroll
        for (int ks = 0; ks < kFChunk / 16; ++ks)
          mma_f16(tmem + acc_col,
                  make_smem_desc(a_op + c * kAPartBytes + ks * 2 * kFLBO, kFLBO, kFSBOA),
                  make_smem_desc(b_op + (c * (kFChunk / 8) + ks * 2) * kFLBO, kFLBO, kFSBOB), idesc,
                  (c | ks) != 0 ? 1u : 0u);
      mma_commit(&tl.mma_done);
      // the ring buffer just converted is free: fetch `stages` tiles ahead
      fence_proxy_async();
      fetch(slot);
    }
    ++committed;
    if (prev_tile >= 0) epilogue(prev_tile, prev_t, prev_D, prev_npad, ((committed - 2) & 1u) * tmem_cols);
    prev_tile = tile;
    prev_t = t;
    prev_D = D;
    prev_npad = n_pad;
    fence_before_sync();
  }
  if (!tl.timed_out && committed > done) {
    const bool ok = mbar_wait(&tl.mma_done, done & 1u);
    if (ok) ++done;
    fence_after_sync();
    if (!ok) atomicOr(&tl.timed_out, 1);
    __syncthreads();
    if (!tl.timed_out) epilogue(prev_tile, prev_t, prev_D, prev_npad, ((committed - 1) & 1u) * tmem_cols);
  }
  __syncthreads();
  if (tl.timed_out && tid == 0) {
    atomicOr(a.error_word, TBE_ERR_TIMEOUT);
    // drain (bounded): the MMAs committed and the copies issued (the last
    // tile taken may have timed out on its copy; a completed phase passes)
    if (committed > done) mbar_wait(&tl.mma_done, done & 1u);
    for (uint32_t f = consumed > 0 ? consumed - 1 : 0; f < fetched; ++f)
      mbar_wait(&tl.full[f % static_cast<uint32_t>(stages)], (f / static_cast<uint32_t>(stages)) & 1u);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 2 * tmem_cols);
}

}  // namespace

cudaError_t launch_forward_hot(const Launch& L, const WsLayout& W, char* ws, const void* weights,
                               const float* psw, float* out, bool mean) {
  const tbe_desc* d = L.d;
  const uint32_t* hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
  if (W.hot_enabled) {
    FwdHotArgs a;
    a.W = static_cast<const __half*>(weights);
    a.D_offsets = d->D_offsets;
    a.hash_base = d->hash_base;
    a.w_offsets = d->weights_offsets;
    a.hot_keys = reinterpret_cast<const uint32_t*>(ws + W.hot_keys(W.hot_cur));
    a.hot_n = hot_n;
    a.hot_hist8 = reinterpret_cast<const uint8_t*>(ws + W.hot_hist8);
    a.hot_hist = reinterpret_cast<const float*>(ws + W.hot_hist);
    a.hot_scale = reinterpret_cast<const int8_t*>(ws + W.hot_scale);
    a.tile_kind = reinterpret_cast<const uint8_t*>(ws + W.tile_kind);
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

    const bool bf16 = d->weights_dtype == TBE_DT_BF16;
    const int ti = bf16 ? 1 : 0;  // weight type: index of the per-type attribute caches
    const void* hot_k = bf16 ? reinterpret_cast<const void*>(forward_hot_kernel<true>)
                             : reinterpret_cast<const void*>(forward_hot_kernel<false>);
    static size_t attr_bytes[64][2] = {};
    static int ctas_per_sm[64][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_bytes[dev][ti] != smem) {
      e = cudaFuncSetAttribute(hot_k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      // all of the unified L1 / shared storage as shared memory, so that two
      // CTAs fit when the operands allow
      e = cudaFuncSetAttribute(hot_k, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      int smem_per_sm = 0;
      e = cudaDeviceGetAttribute(&smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
      if (e != cudaSuccess) return e;
      // 1 KB of each CTA's shared memory is reserved by the driver
      int per_sm = static_cast<int>(static_cast<size_t>(smem_per_sm) / (smem + 1024));
      if (per_sm > 2) per_sm = 2;
      ctas_per_sm[dev][ti] = per_sm < 1 ? 1 : per_sm;
      attr_bytes[dev][ti] = smem;
    }
    // resident CTAs x tensor-memory columns must fit the SM's 512
    int per_sm = ctas_per_sm[dev][ti];
    if (per_sm * static_cast<int>(tmem_cols) > 512) per_sm = static_cast<int>(512 / tmem_cols);
    const int64_t tiles = static_cast<int64_t>(d->T) * ((d->B + kFM - 1) / kFM);
    int64_t grid = static_cast<int64_t>(per_sm) * L.num_sms;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;

    // byte tiles: one CTA per SM, as many ring stages as shared memory holds
    // (the transpose buffer when at least two stages fit beside it)
    static size_t bytes_attr[64][2] = {};
    static int bytes_stages[64][2] = {};
    static int bytes_nmax[64][2] = {};
    static bool bytes_xpose[64][2] = {};
    if (bytes_nmax[dev][ti] != a.n_max) {
      int optin = 0;
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (e != cudaSuccess) return e;
      const bool xpose = fwd_bytes_smem_bytes(a.n_max, 2, true) <= static_cast<size_t>(optin);
      int stages = kBMaxStages;
      while (stages > 1 && fwd_bytes_smem_bytes(a.n_max, stages, xpose) > static_cast<size_t>(optin))
        --stages;
      const size_t bsmem = fwd_bytes_smem_bytes(a.n_max, stages, xpose);
      const void* k = xpose ? (bf16 ? reinterpret_cast<const void*>(forward_bytes_kernel<true, true>)
                                    : reinterpret_cast<const void*>(forward_bytes_kernel<true, false>))
                            : (bf16 ? reinterpret_cast<const void*>(forward_bytes_kernel<false, true>)
                                    : reinterpret_cast<const void*>(forward_bytes_kernel<false, false>));
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bsmem));
      if (e != cudaSuccess) return e;
      bytes_attr[dev][ti] = bsmem;
      bytes_stages[dev][ti] = stages;
      bytes_xpose[dev][ti] = xpose;
      bytes_nmax[dev][ti] = a.n_max;
    }
    int64_t bgrid = L.num_sms < tiles ? L.num_sms : tiles;
    if (bgrid < 1) bgrid = 1;
    // both kernels together are the hot part of the forward
    probe_begin(TBE_PROBE_FORWARD_HOT, L.s);
    const unsigned bg = static_cast<unsigned>(bgrid);
    const size_t bs = bytes_attr[dev][ti];
    const int st = bytes_stages[dev][ti];
    if (bytes_xpose[dev][ti]) {
      if (bf16) forward_bytes_kernel<true, true><<<bg, kBThreads, bs, L.s>>>(a, tmem_cols, st);
      else forward_bytes_kernel<true, false><<<bg, kBThreads, bs, L.s>>>(a, tmem_cols, st);
    } else {
      if (bf16) forward_bytes_kernel<false, true><<<bg, kBThreads, bs, L.s>>>(a, tmem_cols, st);
      else forward_bytes_kernel<false, false><<<bg, kBThreads, bs, L.s>>>(a, tmem_cols, st);
    }
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (bf16) forward_hot_kernel<true><<<static_cast<unsigned>(grid), kFThreads, smem, L.s>>>(a, tmem_cols);
    else forward_hot_kernel<false><<<static_cast<unsigned>(grid), kFThreads, smem, L.s>>>(a, tmem_cols);
    note_launch();
    probe_end(TBE_PROBE_FORWARD_HOT, L.s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_forward_cold(L, weights, reinterpret_cast<const uint32_t*>(ws + W.keys[2]),
                             reinterpret_cast<const uint32_t*>(ws + W.cold_off),
                             psw ? reinterpret_cast<const float*>(ws + W.psw[2]) : nullptr, out,
                             W.hot_enabled ? hot_n : nullptr,
                             mean ? reinterpret_cast<const float*>(ws + W.inv_len) : nullptr);
}

}  // namespace tbe
