// Backward update: sum each run's gradients, then one exact row-wise Adagrad
// step per touched row.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Backward:
// invert 'which rows did this sample use?'": short runs are handled by one
// program that gathers, accumulates in registers, updates and plain-stores
// the row (it owns the row exclusively); long runs are split into chunks
// that write partial sums; in the fused variant
// each chunk writes its partial, executes a device-scope fence and decrements
// the run's remaining count, and only the last chunk to finish updates the
// row, while the default variant finishes in a second kernel.  Section
// "Fusion boundaries are also engineering interfaces": per-sample weights
// scale each contribution before grouping, and the optimizer is the
// epilogue of the backward.  "HugeCTR DistributedSlotSparseEmbeddingHash
// backward" (eqicode.com), the Adagrad kernel: the accumulator is updated
// first and the weight step divides by sqrt(new accumulator) + eps.
//
// GB300 design:
//  * work is counted in pairs: the lookups of one run that come from the
//    same bag read the same gradient row, so each pair gathers that row once
//    and scales it by the pair's multiplicity (or the sum of its per-sample
//    weights).  On skewed inputs a hot row is hit many times per bag, and
//    this removes most of its gathers;
//  * the gradient rows are fp32; a row of D floats is D/4 float4 vectors on
//    S = next_pow2(D/4) lanes (at most 32), so one warp serves G = 32/S short
//    runs of the same table at once (tasks never straddle tables);
//  * a long run's chunk partials meet in a tree of fan-in 32: the last of a
//    node's children to arrive (fence, then atomic decrement) sums them in
//    child order and climbs; the root's last arriver applies the update.  A
//    run of millions of lookups thus has no serial tail over all its
//    partials, and the result does not depend on arrival order;
//  * partial sums are written and read at L2 (st.cg / ld.cg), never through
//    the non-coherent L1.
#include "common.cuh"
#include "internal.h"

namespace tbe {
namespace {

struct UpdArgs {
  const float* grad_out;
  __half* W;
  float* momentum;
  const int64_t* D_offsets;
  const int64_t* hash_base;
  const int64_t* w_offsets;
  const float* sorted_psw;
  const uint32_t* unique_keys;
  const uint32_t* run_pairs;
  const uint32_t* pair_starts;
  const uint32_t* pair_bags;
  const uint32_t* counters;
  const uint32_t* table_runs;
  const uint32_t* table_tasks;
  const uint32_t* long_run;
  const uint32_t* long_chunk0;
  const uint32_t* long_tree0;
  const uint32_t* chunk_task;
  const uint32_t* chunk_order;
  uint32_t* tree_cnt;
  float* partials;
  float* tree_part;
  int64_t total_D;
  int T;
  int B;
  int max_D;
  float lr;
  float eps;
};

// Largest t with table_first[t] <= x (table_first has T+1 ascending entries).
template <typename V>
__device__ __forceinline__ int find_table(const V* first, int T, V x) {
  int lo = 0, hi = T - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(first + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bag and coefficient of pair k: every lookup of the pair reads the same
// gradient row, so the row is gathered once and scaled by the number of
// lookups or, with per-sample weights, by their sum (in lookup order).
template <bool kWeighted>
__device__ __forceinline__ void load_pair(const UpdArgs& a, uint32_t k, uint32_t* bag, float* coef) {
  const uint32_t s = a.pair_starts[k];
  const uint32_t e = a.pair_starts[k + 1];
  *bag = a.pair_bags[k];
  if (kWeighted) {
    float c = 0.f;
    for (uint32_t i = s; i < e; ++i) c += a.sorted_psw[i];
    *coef = c;
  } else {
    *coef = static_cast<float>(e - s);
  }
}

// Row-wise Adagrad on one row (key, row r of table t) with the summed
// gradient held by the S lanes of a group: lane sl owns columns
// (sl + c*S)*4 .. +3 for c < NC.
template <int S, int NC>
__device__ __forceinline__ void adagrad_row(const UpdArgs& a, float (&g)[NC][4], int D,
                                            uint32_t key, int t, bool active) {
  const int sl = static_cast<int>(lane_id()) % S;
  const int nv = D >> 2;
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c)
    if (sl + c * S < nv)
#pragma unroll
      for (int i = 0; i < 4; ++i) ss = fmaf(g[c][i], g[c][i], ss);
#pragma unroll
  for (int off = 1; off < S; off <<= 1) ss += __shfl_xor_sync(kFull, ss, off);
  if (!active) return;
  const float m_new = a.momentum[key] + ss / static_cast<float>(D);
  const float denom = sqrtf(m_new) + a.eps;
  const int64_t r = static_cast<int64_t>(key) - __ldg(a.hash_base + t);
  __half* row = a.W + __ldg(a.w_offsets + t) + r * D;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int vec = sl + c * S;
    if (vec < nv) {
      uint2* p = reinterpret_cast<uint2*>(row + vec * 4);
      uint2 raw = *p;
      __half2* h = reinterpret_cast<__half2*>(&raw);
      const float2 w01 = __half22float2(h[0]);
      const float2 w23 = __half22float2(h[1]);
      h[0] = __floats2half2_rn(w01.x - a.lr * g[c][0] / denom, w01.y - a.lr * g[c][1] / denom);
      h[1] = __floats2half2_rn(w23.x - a.lr * g[c][2] / denom, w23.y - a.lr * g[c][3] / denom);
      *p = raw;
    }
  }
  if (sl == 0) a.momentum[key] = m_new;
}

// ------------------------------------------------------------- short runs
template <int S, int NC, bool kWeighted>
__device__ __forceinline__ void short_task(const UpdArgs& a, int t, uint32_t j0, uint32_t j_end) {
  constexpr int U = 4 / NC > 0 ? (4 / NC < S ? 4 / NC : S) : 1;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
  const int64_t d0 = __ldg(a.D_offsets + t);
  const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - d0);
  const int nv = D >> 2;
  const uint32_t j = j0 + g;
  uint32_t s = 0, SL = 0;  // first pair and pair count of this group's run
  if (j < j_end) {
    s = a.run_pairs[j];
    SL = a.run_pairs[j + 1] - s;
    if (SL >= static_cast<uint32_t>(kLongThreshold)) SL = 0;  // chunked path owns it
  }
  const uint32_t max_len = __reduce_max_sync(kFull, SL);
  float acc[NC][4];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  for (uint32_t base = 0; base < max_len; base += S) {
    uint32_t my_b = 0xffffffffu;
    float my_w = 0.f;
    if (base + sl < SL) load_pair<kWeighted>(a, s + base + sl, &my_b, &my_w);
#pragma unroll
    for (int u0 = 0; u0 < S; u0 += U) {
      if (base + u0 >= max_len) break;  // warp-uniform
      float4 v[U][NC];
      float wv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const uint32_t b = __shfl_sync(kFull, my_b, u0 + uu, S);
        wv[uu] = __shfl_sync(kFull, my_w, u0 + uu, S);
        const bool ok = b < static_cast<uint32_t>(a.B);  // also false past the run's end
        const float* grow = a.grad_out + static_cast<int64_t>(b) * a.total_D + d0;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int vec = sl + c * S;
          v[uu][c] = (ok && vec < nv) ? ldg_f4(grow + vec * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu)
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          acc[c][0] = fmaf(wv[uu], v[uu][c].x, acc[c][0]);
          acc[c][1] = fmaf(wv[uu], v[uu][c].y, acc[c][1]);
          acc[c][2] = fmaf(wv[uu], v[uu][c].z, acc[c][2]);
          acc[c][3] = fmaf(wv[uu], v[uu][c].w, acc[c][3]);
        }
    }
  }
  const uint32_t key = SL > 0 ? a.unique_keys[j] : 0u;
  adagrad_row<S, NC>(a, acc, D, key, t, SL > 0);
}

template <bool kWeighted>
__global__ void __launch_bounds__(256) short_runs_kernel(UpdArgs a) {
  const uint32_t ntasks = a.counters[kCntTasks];
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntasks;
       task += warps) {
    const int t = find_table(a.table_tasks, a.T, task);
    const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - __ldg(a.D_offsets + t));
    if (D < 8 || D > kMaxD || (D & 7)) continue;  // widths the vector path cannot move
    const int nv = D >> 2;
    int S = 1;
    while (S < nv && S < 32) S <<= 1;
    const uint32_t G = 32 / S;
    const uint32_t j0 = a.table_runs[t] + (task - a.table_tasks[t]) * G;
    const uint32_t j_end = a.table_runs[t + 1];
    if (nv <= 2) short_task<2, 1, kWeighted>(a, t, j0, j_end);
    else if (nv <= 4) short_task<4, 1, kWeighted>(a, t, j0, j_end);
    else if (nv <= 8) short_task<8, 1, kWeighted>(a, t, j0, j_end);
    else if (nv <= 16) short_task<16, 1, kWeighted>(a, t, j0, j_end);
    else if (nv <= 32) short_task<32, 1, kWeighted>(a, t, j0, j_end);
    else if (nv <= 64) short_task<32, 2, kWeighted>(a, t, j0, j_end);
    else if (nv <= 128) short_task<32, 4, kWeighted>(a, t, j0, j_end);
    else short_task<32, 8, kWeighted>(a, t, j0, j_end);
  }
}

// -------------------------------------------------------------- long runs
// Sum pairs [s, e) of one run over the whole warp: group g takes every G-th
// pair; the groups meet in a butterfly so every lane ends with its columns.
template <int S, int NC, bool kWeighted>
__device__ __forceinline__ void sum_lookups(const UpdArgs& a, int64_t d0, int nv, uint32_t s,
                                            uint32_t e, float (&acc)[NC][4]) {
  constexpr int G = 32 / S;
  constexpr int U = 4 / NC > 0 ? (4 / NC < S ? 4 / NC : S) : 1;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  for (uint32_t base = s; base < e; base += 32) {
    const int cnt = static_cast<int>(e - base < 32u ? e - base : 32u);
    uint32_t my_b = 0xffffffffu;
    float my_w = 0.f;
    if (lane < cnt) load_pair<kWeighted>(a, base + lane, &my_b, &my_w);
#pragma unroll
    for (int u0 = 0; u0 < S; u0 += U) {
      if (G * u0 >= cnt) break;  // warp-uniform
      float4 v[U][NC];
      float wv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int k = g + G * (u0 + uu);
        const uint32_t b = __shfl_sync(kFull, my_b, k);
        wv[uu] = __shfl_sync(kFull, my_w, k);
        const bool ok = b < static_cast<uint32_t>(a.B);
        const float* grow = a.grad_out + static_cast<int64_t>(b) * a.total_D + d0;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int vec = sl + c * S;
          v[uu][c] = (ok && vec < nv) ? ldg_f4(grow + vec * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu)
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          acc[c][0] = fmaf(wv[uu], v[uu][c].x, acc[c][0]);
          acc[c][1] = fmaf(wv[uu], v[uu][c].y, acc[c][1]);
          acc[c][2] = fmaf(wv[uu], v[uu][c].z, acc[c][2]);
          acc[c][3] = fmaf(wv[uu], v[uu][c].w, acc[c][3]);
        }
    }
  }
#pragma unroll
  for (int off = S; off < 32; off <<= 1)
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][i] += __shfl_xor_sync(kFull, acc[c][i], off);
}

// Sum `count` partial rows (stride max_D floats) starting at `base`, in
// order within each group, then across groups in a fixed butterfly.
template <int S, int NC>
__device__ __forceinline__ void sum_partials(const float* base, int max_D, uint32_t count, int nv,
                                             float (&acc)[NC][4]) {
  constexpr int G = 32 / S;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
  const int sl = lane % S;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  for (uint32_t ch = g; ch < count; ch += G) {
    const float* p = base + static_cast<int64_t>(ch) * max_D;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int vec = sl + c * S;
      if (vec < nv) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p + vec * 4));
        acc[c][0] += v.x;
        acc[c][1] += v.y;
        acc[c][2] += v.z;
        acc[c][3] += v.w;
      }
    }
  }
#pragma unroll
  for (int off = S; off < 32; off <<= 1)
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][i] += __shfl_xor_sync(kFull, acc[c][i], off);
}

template <int S, int NC>
__device__ __forceinline__ void store_partial(float* dst, int nv, const float (&acc)[NC][4]) {
  const int lane = static_cast<int>(lane_id());
  if (lane < S) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int vec = lane + c * S;
      if (vec < nv)
        __stcg(reinterpret_cast<float4*>(dst + vec * 4),
               make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]));
    }
  }
}

// Publish this warp's stores, then take one arrival off `counter`.  Returns
// true for the last arriver, which may then read every other arriver's data.
__device__ __forceinline__ bool arrive_last(uint32_t* counter) {
  __threadfence();
  __syncwarp();
  uint32_t prev = 0;
  if (lane_id() == 0) {
    prev = atomicSub(counter, 1u);
    __threadfence();
  }
  prev = __shfl_sync(kFull, prev, 0);
  __syncwarp();
  __threadfence();
  return prev == 1u;
}

template <int S, int NC, bool kWeighted>
__device__ __forceinline__ void long_chunk(const UpdArgs& a, uint32_t q, bool two_launch) {
  const uint32_t k = a.chunk_task[q];
  const uint32_t j = a.long_run[k];
  const uint32_t c = q - a.long_chunk0[k];
  const uint32_t rs0 = a.run_pairs[j];
  const uint32_t SL = a.run_pairs[j + 1] - rs0;
  const uint32_t nch = (SL + kChunk - 1) / kChunk;
  const uint32_t s = rs0 + c * kChunk;
  const uint32_t e = s + kChunk < rs0 + SL ? s + kChunk : rs0 + SL;
  const uint32_t key = a.unique_keys[j];
  const int t = find_table(a.hash_base, a.T, static_cast<int64_t>(key));
  const int64_t d0 = __ldg(a.D_offsets + t);
  const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - d0);
  const int nv = D >> 2;
  float acc[NC][4];
  sum_lookups<S, NC, kWeighted>(a, d0, nv, s, e, acc);
  if (nch == 1 && !two_launch) {
    adagrad_row<S, NC>(a, acc, D, key, t, true);
    return;
  }
  const uint32_t c0 = a.long_chunk0[k];
  store_partial<S, NC>(a.partials + static_cast<int64_t>(c0 + c) * a.max_D, nv, acc);
  if (two_launch) return;
  // Climb the run's reduction tree while this warp is the last arriver.
  const uint32_t tree0 = a.long_tree0[k];
  uint32_t level_off = 0;   // first node of the current level within the run's tree
  uint32_t below = nch;     // nodes on the level below
  uint32_t i = c / kFanIn;  // node index on the current level
  for (;;) {
    const uint32_t here = (below + kFanIn - 1) / kFanIn;
    if (!arrive_last(a.tree_cnt + tree0 + level_off + i)) return;
    const uint32_t first = i * kFanIn;
    const uint32_t kids = below - first < static_cast<uint32_t>(kFanIn) ? below - first : kFanIn;
    const float* src = level_off == 0 && below == nch
                           ? a.partials + static_cast<int64_t>(c0 + first) * a.max_D
                           : a.tree_part + static_cast<int64_t>(tree0 + level_off - below + first) *
                                               a.max_D;
    sum_partials<S, NC>(src, a.max_D, kids, nv, acc);
    if (here == 1) {
      adagrad_row<S, NC>(a, acc, D, key, t, true);
      return;
    }
    store_partial<S, NC>(a.tree_part + static_cast<int64_t>(tree0 + level_off + i) * a.max_D, nv,
                         acc);
    level_off += here;
    below = here;
    i /= kFanIn;
  }
}

template <bool kWeighted>
__global__ void __launch_bounds__(256) long_chunks_kernel(UpdArgs a, bool two_launch) {
  const uint32_t nchunks = a.counters[kCntChunks];
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t qi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; qi < nchunks; qi += warps) {
    const uint32_t q = a.chunk_order[qi];
    const uint32_t k = a.chunk_task[q];
    const uint32_t key = a.unique_keys[a.long_run[k]];
    const int t = find_table(a.hash_base, a.T, static_cast<int64_t>(key));
    const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - __ldg(a.D_offsets + t));
    if (D < 8 || D > kMaxD || (D & 7)) continue;
    const int nv = D >> 2;
    if (nv <= 2) long_chunk<2, 1, kWeighted>(a, q, two_launch);
    else if (nv <= 4) long_chunk<4, 1, kWeighted>(a, q, two_launch);
    else if (nv <= 8) long_chunk<8, 1, kWeighted>(a, q, two_launch);
    else if (nv <= 16) long_chunk<16, 1, kWeighted>(a, q, two_launch);
    else if (nv <= 32) long_chunk<32, 1, kWeighted>(a, q, two_launch);
    else if (nv <= 64) long_chunk<32, 2, kWeighted>(a, q, two_launch);
    else if (nv <= 128) long_chunk<32, 4, kWeighted>(a, q, two_launch);
    else long_chunk<32, 8, kWeighted>(a, q, two_launch);
  }
}

// Two-launch variant, second kernel: one warp per long run sums the run's
// chunk partials in chunk order and applies the update.
template <int S, int NC>
__device__ __forceinline__ void finish_run(const UpdArgs& a, uint32_t k) {
  const uint32_t j = a.long_run[k];
  const uint32_t SL = a.run_pairs[j + 1] - a.run_pairs[j];
  const uint32_t nch = (SL + kChunk - 1) / kChunk;
  const uint32_t key = a.unique_keys[j];
  const int t = find_table(a.hash_base, a.T, static_cast<int64_t>(key));
  const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - __ldg(a.D_offsets + t));
  float acc[NC][4];
  sum_partials<S, NC>(a.partials + static_cast<int64_t>(a.long_chunk0[k]) * a.max_D, a.max_D, nch,
                      D >> 2, acc);
  adagrad_row<S, NC>(a, acc, D, key, t, true);
}

__global__ void __launch_bounds__(256) long_finish_kernel(UpdArgs a) {
  const uint32_t nlong = a.counters[kCntLong];
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t k = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; k < nlong; k += warps) {
    const uint32_t key = a.unique_keys[a.long_run[k]];
    const int t = find_table(a.hash_base, a.T, static_cast<int64_t>(key));
    const int D = static_cast<int>(__ldg(a.D_offsets + t + 1) - __ldg(a.D_offsets + t));
    if (D < 8 || D > kMaxD || (D & 7)) continue;
    const int nv = D >> 2;
    if (nv <= 2) finish_run<2, 1>(a, k);
    else if (nv <= 4) finish_run<4, 1>(a, k);
    else if (nv <= 8) finish_run<8, 1>(a, k);
    else if (nv <= 16) finish_run<16, 1>(a, k);
    else if (nv <= 32) finish_run<32, 1>(a, k);
    else if (nv <= 64) finish_run<32, 2>(a, k);
    else if (nv <= 128) finish_run<32, 4>(a, k);
    else finish_run<32, 8>(a, k);
  }
}

}  // namespace

cudaError_t launch_update(const Launch& L, const WsLayout& W, char* ws, const float* grad_out,
                          void* weights, float* momentum, float lr, float eps, bool two_launch) {
  const tbe_desc* d = L.d;
  const int fin = radix_passes(d) & 1;
  UpdArgs a;
  a.grad_out = grad_out;
  a.W = static_cast<__half*>(weights);
  a.momentum = momentum;
  a.D_offsets = d->D_offsets;
  a.hash_base = d->hash_base;
  a.w_offsets = d->weights_offsets;
  a.sorted_psw = W.weighted ? reinterpret_cast<const float*>(ws + W.psw[fin]) : nullptr;
  a.unique_keys = reinterpret_cast<const uint32_t*>(ws + W.unique_keys);
  a.run_pairs = reinterpret_cast<const uint32_t*>(ws + W.run_pairs);
  a.pair_starts = reinterpret_cast<const uint32_t*>(ws + W.pair_starts);
  a.pair_bags = reinterpret_cast<const uint32_t*>(ws + W.pair_bags);
  a.counters = reinterpret_cast<const uint32_t*>(ws + W.counts);
  a.table_runs = reinterpret_cast<const uint32_t*>(ws + W.table_runs);
  a.table_tasks = reinterpret_cast<const uint32_t*>(ws + W.table_tasks);
  a.long_run = reinterpret_cast<const uint32_t*>(ws + W.long_run);
  a.long_chunk0 = reinterpret_cast<const uint32_t*>(ws + W.long_chunk0);
  a.long_tree0 = reinterpret_cast<const uint32_t*>(ws + W.long_tree0);
  a.chunk_task = reinterpret_cast<const uint32_t*>(ws + W.chunk_task);
  a.chunk_order = reinterpret_cast<const uint32_t*>(ws + W.chunk_order);
  a.tree_cnt = reinterpret_cast<uint32_t*>(ws + W.tree_cnt);
  a.partials = reinterpret_cast<float*>(ws + W.partials);
  a.tree_part = reinterpret_cast<float*>(ws + W.tree_part);
  a.total_D = d->total_D;
  a.T = d->T;
  a.B = d->B;
  a.max_D = d->max_D;
  a.lr = lr;
  a.eps = eps;
  if (L.n == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>(L.num_sms) * 8u;
  const bool weighted = a.sorted_psw != nullptr;
  if (weighted) short_runs_kernel<true><<<blocks, 256, 0, L.s>>>(a);
  else short_runs_kernel<false><<<blocks, 256, 0, L.s>>>(a);
  if (weighted) long_chunks_kernel<true><<<blocks, 256, 0, L.s>>>(a, two_launch);
  else long_chunks_kernel<false><<<blocks, 256, 0, L.s>>>(a, two_launch);
  if (two_launch) long_finish_kernel<<<blocks, 256, 0, L.s>>>(a);
  return cudaGetLastError();
}

}  // namespace tbe
