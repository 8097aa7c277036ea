// Backward update: sum each run's gradients, then one exact row-wise Adagrad
// step per touched row.
//
// "Modernizing Table Batched Embeddings with FBTriton", section "Backward:
// invert 'which rows did this sample use?'": short runs are handled by one
// program that gathers, accumulates in registers, updates and plain-stores
// the row (it owns the row exclusively); long runs are split into chunks
// that write partial sums; in the fused variant each chunk writes its
// partial, executes a device-scope fence and decrements the run's remaining
// count, and only the last chunk to finish updates the row, while the
// default variant finishes in a second kernel.  Section "Fusion boundaries
// are also engineering interfaces": per-sample weights scale each
// contribution before grouping, and the optimizer is the epilogue of the
// backward.  "HugeCTR DistributedSlotSparseEmbeddingHash backward"
// (eqicode.com), the Adagrad kernel: the accumulator is updated first and the
// weight step divides by sqrt(new accumulator) + eps.
//
// GB300 design:
//  * work is counted in pairs: the lookups of one run that come from the
//    same bag read the same gradient row, so each pair gathers that row once
//    and scales it by the pair's multiplicity (or the sum of its per-sample
//    weights).  On skewed inputs a hot row is hit many times per bag, and
//    this removes most of its gathers;
//  * the gradient rows are fp32, moved as float4: a row of D floats is
//    nv = D/4 vectors on S lanes with NC = nv/S vectors each (update_lanes),
//    so one warp serves G = 32/S runs of a table at once; a lane keeps up to
//    8 row vectors in flight on long-run chunks and 4 on short runs, whose
//    memory latency is hidden by running several of them per warp;
//  * table metadata sits in shared memory; a short run's weights row and
//    momentum are fetched at the start, in the shadow of its gradient
//    gathers; a long-run chunk is one 16-byte descriptor;
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

constexpr int kSmemTables = 256;  // tables whose metadata is cached in shared memory

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
  const LongRunInfo* long_info;
  const ChunkDesc* chunk_order;
  uint32_t* tree_cnt;
  uint32_t* cursors;  // counters + kCntNextShort: the update kernels' work cursors
  float* partials;
  float* tree_part;
  int64_t total_D;
  int T;
  int B;
  int max_D;
  float lr;
  float eps;
  bool bf16;  // weights are bf16 rather than fp16
  bool f32;   // weights are fp32 (W then points at floats)
};

// Table metadata, in shared memory when the problem has few enough tables.
struct Meta {
  const int64_t* d_off;
  const int64_t* hb;
  const int64_t* w_off;
  const uint32_t* tasks;
  const uint32_t* runs;
};

struct MetaSmem {
  int64_t d_off[kSmemTables + 1];
  int64_t hb[kSmemTables + 1];
  int64_t w_off[kSmemTables + 1];
  uint32_t tasks[kSmemTables + 1];
  uint32_t runs[kSmemTables + 1];
};

__device__ __forceinline__ Meta load_meta(const UpdArgs& a, MetaSmem& sm, bool with_tasks) {
  if (a.T > kSmemTables)
    return Meta{a.D_offsets, a.hash_base, a.w_offsets, a.table_tasks, a.table_runs};
  for (int t = threadIdx.x; t <= a.T; t += blockDim.x) {
    sm.d_off[t] = a.D_offsets[t];
    sm.hb[t] = a.hash_base[t];
    sm.w_off[t] = a.w_offsets[t];
    if (with_tasks) {
      sm.tasks[t] = a.table_tasks[t];
      sm.runs[t] = a.table_runs[t];
    }
  }
  __syncthreads();
  return Meta{sm.d_off, sm.hb, sm.w_off, sm.tasks, sm.runs};
}

// The next work item of a warp from cursor `c` (TBE_DYNAMIC_RUNS): one
// atomic by lane 0, broadcast.
__device__ __forceinline__ uint32_t grab(uint32_t* c) {
  uint32_t v = 0;
  if (lane_id() == 0) v = atomicAdd(c, 1u);
  return __shfl_sync(kFull, v, 0);
}

// grab() in two halves, for loops that take their next work item one
// iteration ahead: lane 0's atomic (grab_raw), whose result the warp reads
// (ticket) in the next iteration, so that the atomic's round trip does not
// stall the warp (it issues in order and would wait at the broadcast).
__device__ __forceinline__ uint32_t grab_raw(uint32_t* c) {
  uint32_t v = 0;
  if (lane_id() == 0) v = atomicAdd(c, 1u);
  return v;
}
__device__ __forceinline__ uint32_t ticket(uint32_t raw) { return __shfl_sync(kFull, raw, 0); }

// Largest t with first[t] <= x (first has T+1 ascending entries).
__device__ __forceinline__ int find_table(const uint32_t* first, int T, uint32_t x) {
  int lo = 0, hi = T - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (first[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bag and coefficient of pair k: every lookup of the pair reads the same
// gradient row, so the row is gathered once and scaled by the number of
// lookups or, with per-sample weights, by their sum (in lookup order).
template <bool kWeighted>
__device__ __forceinline__ void load_pair(const UpdArgs& a, uint32_t k, uint32_t* bag, float* coef) {
  const uint32_t s = __ldg(a.pair_starts + k);
  const uint32_t e = __ldg(a.pair_starts + k + 1);
  *bag = __ldg(a.pair_bags + k);
  if (kWeighted) {
    float c = 0.f;
    for (uint32_t i = s; i < e; ++i) c += __ldg(a.sorted_psw + i);
    *coef = c;
  } else {
    *coef = static_cast<float>(e - s);
  }
}

// This lane's vectors of gradient row b (columns d0 + (sl + c*S)*4 ..).
template <int S, int NC>
__device__ __forceinline__ void gather_row(const UpdArgs& a, int64_t d0, int nv, uint32_t b,
                                           float4 (&v)[NC], bool ok) {
  const int sl = static_cast<int>(lane_id()) % S;
  const float* grow = a.grad_out + static_cast<int64_t>(b) * a.total_D + d0;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int vec = sl + c * S;
    v[c] = (ok && vec < nv) ? ldg_f4(grow + vec * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int NC>
__device__ __forceinline__ void fma_rows(float (&acc)[NC][4], const float4 (&v)[NC], float w) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    acc[c][0] = fmaf(w, v[c].x, acc[c][0]);
    acc[c][1] = fmaf(w, v[c].y, acc[c][1]);
    acc[c][2] = fmaf(w, v[c].z, acc[c][2]);
    acc[c][3] = fmaf(w, v[c].w, acc[c][3]);
  }
}

// This lane's 16-bit weights of the row at element offset woff, fetched
// ahead of the gradient gathers (fp32 rows are read by the update itself).
template <int S, int NC>
__device__ __forceinline__ void load_row(const UpdArgs& a, int64_t woff, int nv,
                                         uint2 (&w_raw)[NC], bool active) {
  const int sl = static_cast<int>(lane_id()) % S;
  const __half* row = a.W + woff;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int vec = sl + c * S;
    w_raw[c] = (active && !a.f32 && vec < nv) ? *reinterpret_cast<const uint2*>(row + vec * 4)
                                              : make_uint2(0u, 0u);
  }
}

// Four weights of a row after their Adagrad step w - lr * g / den, formed as
// fma(-g, q, w) with q = lr / den (one rounding of the quotient, then one of
// the fused product and difference), each rounded to nearest even in the
// weights' own 16-bit type (bf16 when a.bf16).  The row-wise step shares q
// over the row, so a row costs one division instead of one per element.
__device__ __forceinline__ uint2 adagrad_step4(const UpdArgs& a, uint2 raw, const float (&g)[4],
                                               const float (&q)[4]) {
  if (a.bf16) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
    const float2 w01 = __bfloat1622float2(h[0]);
    const float2 w23 = __bfloat1622float2(h[1]);
    h[0] = __floats2bfloat162_rn(fmaf(-g[0], q[0], w01.x), fmaf(-g[1], q[1], w01.y));
    h[1] = __floats2bfloat162_rn(fmaf(-g[2], q[2], w23.x), fmaf(-g[3], q[3], w23.y));
  } else {
    __half2* h = reinterpret_cast<__half2*>(&raw);
    const float2 w01 = __half22float2(h[0]);
    const float2 w23 = __half22float2(h[1]);
    h[0] = __floats2half2_rn(fmaf(-g[0], q[0], w01.x), fmaf(-g[1], q[1], w01.y));
    h[1] = __floats2half2_rn(fmaf(-g[2], q[2], w23.x), fmaf(-g[3], q[3], w23.y));
  }
  return raw;
}

// Stores the four weights at element offset off after their step: 16-bit
// weights from raw (see adagrad_step4); fp32 weights are read here and
// fma(-g, q, w) is stored in fp32.
__device__ __forceinline__ void store_step4(const UpdArgs& a, int64_t off, uint2 raw,
                                            const float (&g)[4], const float (&q)[4]) {
  if (a.f32) {
    float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.W) + off);
    float4 w = *p;
    w.x = fmaf(-g[0], q[0], w.x);
    w.y = fmaf(-g[1], q[1], w.y);
    w.z = fmaf(-g[2], q[2], w.z);
    w.w = fmaf(-g[3], q[3], w.w);
    *p = w;
  } else {
    *reinterpret_cast<uint2*>(a.W + off) = adagrad_step4(a, raw, g, q);
  }
}

// Adagrad on one row with the summed gradient held by the S lanes of a group
// (lane sl owns vectors sl + c*S).  w_raw / m_old are the row's 16-bit
// weights (4 per vector; fp16, or bf16 when a.bf16) and row momentum, already
// loaded; the new weight is rounded to nearest even in its own type.
// Row-wise (default): m += mean_d g_d^2, one denominator for the row; every
// lane of the warp must call it (the sum of squares is a group shuffle).
// Element-wise (kEw): momentum holds
// one accumulator per weight element at the weight's own flat position, each
// element takes m_d += g_d^2 and its own denominator; m_old is unused.
template <int S, int NC, bool kEw>
__device__ __forceinline__ void adagrad_apply(const UpdArgs& a, float (&g)[NC][4], int D,
                                              uint32_t key, int64_t woff,
                                              const uint2 (&w_raw)[NC], float m_old, bool active) {
  const int sl = static_cast<int>(lane_id()) % S;
  const int nv = D >> 2;
  if constexpr (kEw) {
    if (!active) return;
    float* mrow = a.momentum + woff;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int vec = sl + c * S;
      if (vec < nv) {
        float4 m = *reinterpret_cast<const float4*>(mrow + vec * 4);
        m.x = fmaf(g[c][0], g[c][0], m.x);
        m.y = fmaf(g[c][1], g[c][1], m.y);
        m.z = fmaf(g[c][2], g[c][2], m.z);
        m.w = fmaf(g[c][3], g[c][3], m.w);
        const float q[4] = {a.lr / (sqrtf(m.x) + a.eps), a.lr / (sqrtf(m.y) + a.eps),
                            a.lr / (sqrtf(m.z) + a.eps), a.lr / (sqrtf(m.w) + a.eps)};
        store_step4(a, woff + vec * 4, w_raw[c], g[c], q);
        *reinterpret_cast<float4*>(mrow + vec * 4) = m;
      }
    }
    return;
  }
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c)
    if (sl + c * S < nv)
#pragma unroll
      for (int i = 0; i < 4; ++i) ss = fmaf(g[c][i], g[c][i], ss);
#pragma unroll
  for (int off = 1; off < S; off <<= 1) ss += __shfl_xor_sync(kFull, ss, off);
  if (!active) return;
  const float m_new = m_old + ss / static_cast<float>(D);
  const float qr = a.lr / (sqrtf(m_new) + a.eps);
  const float q[4] = {qr, qr, qr, qr};
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int vec = sl + c * S;
    if (vec < nv) store_step4(a, woff + vec * 4, w_raw[c], g[c], q);
  }
  if (sl == 0) a.momentum[key] = m_new;
}

// ------------------------------------------------------------- short runs
// A warp task: G consecutive runs of table t, run j0 + g for lane group g.
// Its run data is fetched one task ahead (see short_runs_kernel).
struct ShortTask {
  int t;       // table, -1 when there is no task
  int nv;      // float4 vectors per gradient row
  uint32_t p0; // this lane group's pairs [p0, p1) (none: no run)
  uint32_t p1;
  uint32_t key;
  // The pair count.  Read where it is used: the loads of p0 and p1 then
  // need not have arrived when the task is fetched.
  __device__ __forceinline__ uint32_t np() const { return p1 - p0; }
};

__device__ __forceinline__ ShortTask fetch_task(const UpdArgs& a, const Meta& m, uint32_t task,
                                                uint32_t ntasks) {
  ShortTask st{-1, 0, 0, 0, 0};
  if (task >= ntasks) return st;
  const int t = find_table(m.tasks, a.T, task);
  const int D = static_cast<int>(m.d_off[t + 1] - m.d_off[t]);
  // widths the vector path cannot move, or columns off the 32-byte grid
  if (D < 8 || D > kMaxD || (D & 7) || (m.d_off[t] & 7)) return st;
  st.t = t;
  st.nv = D >> 2;
  const int S = update_lanes(st.nv);
  const uint32_t G = 32 / S;
  const uint32_t j = m.runs[t] + (task - m.tasks[t]) * G + lane_id() / S;
  if (j < m.runs[t + 1]) {
    st.p0 = __ldg(a.run_pairs + j);
    st.p1 = __ldg(a.run_pairs + j + 1);
    st.key = __ldg(a.unique_keys + j);
  }
  return st;
}

// Group g of the warp owns one run: its pairs are loaded S at a time, one
// per lane of the group, and gathered U at a time.
template <int S, int NC, bool kWeighted, bool kEw>
__device__ __forceinline__ void short_task(const UpdArgs& a, const Meta& m, const ShortTask& st) {
  // Row vectors in flight per lane: short runs hold few pairs, so the warp's
  // G concurrent runs, not a deep unroll, hide the latency.
  constexpr int U = TBE_SHORT_VECS / NC > 0 ? (TBE_SHORT_VECS / NC < S ? TBE_SHORT_VECS / NC : S) : 1;
  const int lane = static_cast<int>(lane_id());
  const int sl = lane % S;
  const int t = st.t;
  const int64_t d0 = m.d_off[t];
  const int D = static_cast<int>(m.d_off[t + 1] - d0);
  const int nv = D >> 2;
  const uint32_t p0 = st.p0;
  const uint32_t key = st.key;
  // runs of kMediumRun pairs or more belong to medium_runs_kernel and the
  // chunked path
  const uint32_t np = st.np() >= static_cast<uint32_t>(kMediumRun) ? 0u : st.np();
  const bool active = np > 0;
  const int64_t woff = m.w_off[t] + (active ? (static_cast<int64_t>(key) - m.hb[t]) * D : 0);
  uint2 w_raw[NC];
  load_row<S, NC>(a, woff, nv, w_raw, active);
  const float m_old = active ? a.momentum[key] : 0.f;
  const uint32_t max_np = __reduce_max_sync(kFull, np);
  float acc[NC][4];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  for (uint32_t base = 0; base < max_np; base += S) {
    uint32_t my_b = 0xffffffffu;
    float my_w = 0.f;
    if (base + sl < np) load_pair<kWeighted>(a, p0 + base + sl, &my_b, &my_w);
#pragma unroll
    for (int u0 = 0; u0 < S; u0 += U) {
      if (base + u0 >= max_np) break;  // warp-uniform
      float4 v[U][NC];
      float wv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const uint32_t b = __shfl_sync(kFull, my_b, u0 + uu, S);
        wv[uu] = __shfl_sync(kFull, my_w, u0 + uu, S);
        gather_row<S, NC>(a, d0, nv, b, v[uu], b < static_cast<uint32_t>(a.B));
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) fma_rows<NC>(acc, v[uu], wv[uu]);
    }
  }
  adagrad_apply<S, NC, kEw>(a, acc, D, key, woff, w_raw, m_old, active);
}

// ------------------------------------------------------ short runs, piped
// The short-run kernel's tasks (without per-sample weights) through a
// software pipeline per warp whose intermediate data lives in shared
// memory, not registers: while task i is updated, the run data of task i + 2
// and the pair data of task i + 1 are copied there by cp.async (4-byte
// copies, no registers held while they are in flight), and the index of task
// i + 3 is taken.  A task of the tables whose rows take lane groups of S = 8
// (5 to 32 float4 vectors) then waits for its gradient rows only; other
// widths run short_task as it is.  Measured on GB300 (hot-row recipe, short
// runs): 0.618 ms with the register path, 0.567 ms piped.  Per-sample
// weights would add a dependent load of the weights to each pair; those
// launches keep the register path (0.48 ms against 0.57 ms piped, weighted
// recipe), as does a variant that gathered the four runs' rows as one stream
// with a lane per vector (0.81 ms: the per-row accumulator choice and the
// per-run reductions cost more instructions than the latency it saved).
#ifndef TBE_SHORT_PIPE
#define TBE_SHORT_PIPE 1
#endif
static_assert(kMediumRun <= 16, "a short run has at most 15 pairs");

struct ShortPipe {             // one per warp
  uint32_t run[3][16][4];      // slot, run of the task (G = 32 / S <= 16): p0, p1, key
  uint32_t bag[2][4][16];      // slot, run (four for S = 8), pair: its bag
  uint32_t start[2][4][16];    // and its first lookup; start[np] is the run's end
};

// Table of a task, and whether the vector path can move its rows.
__device__ __forceinline__ bool task_table(const UpdArgs& a, const Meta& m, uint32_t task, int* t,
                                           int* D) {
  *t = find_table(m.tasks, a.T, task);
  *D = static_cast<int>(m.d_off[*t + 1] - m.d_off[*t]);
  return *D >= 8 && *D <= kMaxD && !(*D & 7) && !(m.d_off[*t] & 7);
}

// Run data of task `task` into run slot rs: lane l < G copies run j0 + l.
__device__ __forceinline__ void pipe_runs(const UpdArgs& a, const Meta& m, uint32_t task,
                                          uint32_t ntasks, uint32_t (*rs)[4]) {
  if (task >= ntasks) return;  // warp-uniform
  int t, D;
  const bool ok = task_table(a, m, task, &t, &D);
  const uint32_t G = 32u / static_cast<uint32_t>(update_lanes(D >> 2));
  const uint32_t l = lane_id();
  if (l < G) {
    const uint32_t j = m.runs[t] + (task - m.tasks[t]) * G + l;
    const bool v = ok && j < m.runs[t + 1];
    const uint32_t jj = v ? j : 0u;
    cp_async4(&rs[l][0], a.run_pairs + jj, v);
    cp_async4(&rs[l][1], a.run_pairs + jj + 1, v);
    cp_async4(&rs[l][2], a.unique_keys + jj, v);
  }
}

// Pair data of an S = 8 task (run slot rs, complete) into pair slot
// (bag, start): lane (g, sl) copies pairs sl and sl + 8 of run g.
__device__ __forceinline__ void pipe_pairs(const UpdArgs& a, const Meta& m, uint32_t task,
                                           uint32_t ntasks, const uint32_t (*rs)[4],
                                           uint32_t (*bag)[16], uint32_t (*start)[16]) {
  if (task >= ntasks) return;
  int t, D;
  if (!task_table(a, m, task, &t, &D)) return;
  const int nv = D >> 2;
  if (nv <= 4 || nv > 32) return;  // not an S = 8 task (warp-uniform)
  const uint32_t g = lane_id() >> 3, sl = lane_id() & 7u;
  const uint32_t p0 = rs[g][0];
  uint32_t np = rs[g][1] - p0;
  if (np >= static_cast<uint32_t>(kMediumRun)) np = 0u;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t k = sl + 8u * h;
    const bool vb = k < np, vs = np > 0 && k <= np;
    cp_async4(&bag[g][k], a.pair_bags + (vb ? p0 + k : 0u), vb);
    cp_async4(&start[g][k], a.pair_starts + (vs ? p0 + k : 0u), vs);
  }
}

// Coefficient of pair k of a run: its lookup count (as load_pair forms it).
__device__ __forceinline__ float pipe_coef(const uint32_t* start, uint32_t k) {
  return static_cast<float>(start[k + 1] - start[k]);
}

// S = 8 lane groups (rows of 5 to 32 vectors), pair data from the pipe.
template <int NC, bool kEw>
__device__ __forceinline__ void short_task_piped(const UpdArgs& a, const Meta& m, int t,
                                                 const uint32_t (*rs)[4], const uint32_t (*bag)[16],
                                                 const uint32_t (*start)[16]) {
  constexpr int S = 8;
  constexpr int U = TBE_SHORT_VECS / NC > 0 ? TBE_SHORT_VECS / NC : 1;
  const int g = static_cast<int>(lane_id()) >> 3;
  const int64_t d0 = m.d_off[t];
  const int D = static_cast<int>(m.d_off[t + 1] - d0);
  const int nv = D >> 2;
  const uint32_t p0 = rs[g][0];
  const uint32_t key = rs[g][2];
  uint32_t np = rs[g][1] - p0;
  if (np >= static_cast<uint32_t>(kMediumRun)) np = 0u;
  const bool active = np > 0;
  const int64_t woff = m.w_off[t] + (active ? (static_cast<int64_t>(key) - m.hb[t]) * D : 0);
  uint2 w_raw[NC];
  load_row<S, NC>(a, woff, nv, w_raw, active);
  const float m_old = (active && !kEw) ? a.momentum[key] : 0.f;
  const uint32_t max_np = __reduce_max_sync(kFull, np);
  float acc[NC][4];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  for (uint32_t k0 = 0; k0 < max_np; k0 += U) {
    float4 v[U][NC];
    float w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool has = k0 + u < np;
      const uint32_t k = has ? k0 + u : 0u;  // in-bounds index either way
      const uint32_t b = has ? bag[g][k] : 0xffffffffu;
      w[u] = has ? pipe_coef(start[g], k) : 0.f;
      gather_row<S, NC>(a, d0, nv, b, v[u], b < static_cast<uint32_t>(a.B));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) fma_rows<NC>(acc, v[u], w[u]);
  }
  adagrad_apply<S, NC, kEw>(a, acc, D, key, woff, w_raw, m_old, active);
}

// kWide: the instantiation for rows wider than 512 values (eight vectors per
// lane); the other one skips them, so that its register budget stays small.
// kWide: the instantiation for rows wider than 512 values (eight vectors per
// lane); the other one skips them, so that its register budget stays small.
// One medium run with the whole warp.  The row's nv float4 vectors take R
// lanes (lane l holds vectors l % R + c R, c < NC), the warp's G = 32 / R lane
// groups take the run's pairs in turn (group g: pairs g, g + G, ...) with
// U = 8 / NC rows in flight per lane, and a butterfly adds the groups' sums
// (each group sums its pairs in order; the groups are combined in a fixed
// pattern).  A run of many pairs costs one round trip per G U pairs.
template <int R, int NC, bool kWeighted, bool kEw>
__device__ __forceinline__ void warp_run(const UpdArgs& a, const Meta& m, int t, uint32_t p0,
                                         uint32_t np, uint32_t key) {
  constexpr int G = 32 / R;
  constexpr int U = NC < 8 ? 8 / NC : 1;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / R;
  const int64_t d0 = m.d_off[t];
  const int D = static_cast<int>(m.d_off[t + 1] - d0);
  const int nv = D >> 2;
  const int64_t woff = m.w_off[t] + (static_cast<int64_t>(key) - m.hb[t]) * D;
  uint2 w_raw[NC];
  load_row<R, NC>(a, woff, nv, w_raw, true);
  const float m_old = a.momentum[key];
  float acc[NC][4];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  for (uint32_t base = 0; base < np; base += 32) {
    uint32_t my_b = 0xffffffffu;
    float my_w = 0.f;
    if (base + lane < np) load_pair<kWeighted>(a, p0 + base + lane, &my_b, &my_w);
    const uint32_t cnt = np - base < 32u ? np - base : 32u;
#pragma unroll
    for (int u0 = 0; u0 < R; u0 += U) {
      if (static_cast<uint32_t>(u0 * G) >= cnt) break;  // warp-uniform
      float4 v[U][NC];
      float wv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int k = (u0 + uu) * G + g;  // this group's pair within the batch
        const uint32_t b = __shfl_sync(kFull, my_b, k & 31);
        const float w = __shfl_sync(kFull, my_w, k & 31);
        const bool ok = k < 32 && b < static_cast<uint32_t>(a.B);
        wv[uu] = ok ? w : 0.f;
        gather_row<R, NC>(a, d0, nv, b, v[uu], ok);
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) fma_rows<NC>(acc, v[uu], wv[uu]);
    }
  }
#pragma unroll
  for (int off = R; off < 32; off <<= 1)
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][i] += __shfl_xor_sync(kFull, acc[c][i], off);
  adagrad_apply<R, NC, kEw>(a, acc, D, key, woff, w_raw, m_old, g == 0);
}

// Medium runs (kMediumRun <= pairs < kLongThreshold, listed by the
// preprocess): one warp per run.
// kNarrow: every table of the launch is at most 128 wide (one vector per
// lane), so the wider paths, which set the register budget, are left out.
template <bool kWeighted, bool kNarrow, bool kEw>
__global__ void __launch_bounds__(256, kNarrow ? 3 : 2)
    medium_runs_kernel(UpdArgs a, const uint32_t* __restrict__ medium_run) {
  __shared__ MetaSmem msm;
  const Meta m = load_meta(a, msm, true);
  const uint32_t nmed = a.counters[kCntMedium];
#if TBE_DYNAMIC_RUNS
  uint32_t* cur = a.cursors + (kCntNextMedium - kCntNextShort);
  for (uint32_t i = grab(cur); i < nmed; i = grab(cur)) {
#else
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < nmed; i += warps) {
#endif
    const uint32_t j = __ldg(medium_run + i);
    const uint32_t key = __ldg(a.unique_keys + j);
    const uint32_t p0 = __ldg(a.run_pairs + j);
    const uint32_t np = __ldg(a.run_pairs + j + 1) - p0;
    int lo = 0, hi = a.T - 1;  // table of the key
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (m.hb[mid] <= static_cast<int64_t>(key)) lo = mid; else hi = mid - 1;
    }
    const int t = lo;
    const int D = static_cast<int>(m.d_off[t + 1] - m.d_off[t]);
    // widths the vector path cannot move, or columns off the 32-byte grid
    if (D < 8 || D > kMaxD || (D & 7) || (m.d_off[t] & 7)) continue;
    const int nv = D >> 2;
    if (nv <= 4) warp_run<4, 1, kWeighted, kEw>(a, m, t, p0, np, key);
    else if (nv <= 8) warp_run<8, 1, kWeighted, kEw>(a, m, t, p0, np, key);
    else if (nv <= 16) warp_run<16, 1, kWeighted, kEw>(a, m, t, p0, np, key);
    else if (kNarrow || nv <= 32) warp_run<32, 1, kWeighted, kEw>(a, m, t, p0, np, key);
    else if (nv <= 64) warp_run<32, 2, kWeighted, kEw>(a, m, t, p0, np, key);
    else if (nv <= 128) warp_run<32, 4, kWeighted, kEw>(a, m, t, p0, np, key);
    else warp_run<32, 8, kWeighted, kEw>(a, m, t, p0, np, key);
  }
}

template <bool kWeighted, bool kWide, bool kEw>
__global__ void __launch_bounds__(256, TBE_SHORT_MINB) short_runs_kernel(UpdArgs a) {
  __shared__ MetaSmem msm;
  const Meta m = load_meta(a, msm, true);
  const uint32_t ntasks = a.counters[kCntTasks];
  if constexpr (!kWide && !kWeighted && TBE_SHORT_PIPE) {
    __shared__ ShortPipe pipes[8];
    ShortPipe& sp = pipes[threadIdx.x >> 5];
#if TBE_DYNAMIC_RUNS
    auto take = [&]() { return grab_raw(a.cursors); };
    auto index = [&](uint32_t raw) { return ticket(raw); };
#else
    const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
    uint32_t stride_task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    auto take = [&]() {
      const uint32_t v = stride_task;
      stride_task += warps;
      return v;
    };
    auto index = [&](uint32_t raw) { return raw; };
#endif
    // prologue: run data of tasks 0 and 1, pair data of task 0
    uint32_t task0 = index(take());
    pipe_runs(a, m, task0, ntasks, sp.run[0]);
    cp_async_commit();
    uint32_t task1 = index(take());
    pipe_runs(a, m, task1, ntasks, sp.run[1]);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    pipe_pairs(a, m, task0, ntasks, sp.run[0], sp.bag[0], sp.start[0]);
    cp_async_commit();
    uint32_t raw = take();
    int rs0 = 0, ps0 = 0;  // slots of task 0
    while (task0 < ntasks) {
      __syncwarp();  // every lane is done reading the slots refilled below
      const uint32_t task2 = index(raw);
      raw = take();
      const int rs1 = rs0 == 2 ? 0 : rs0 + 1, rs2 = rs1 == 2 ? 0 : rs1 + 1;
      pipe_runs(a, m, task2, ntasks, sp.run[rs2]);
      cp_async_commit();
      cp_async_wait<1>();  // task 1's run data and task 0's pair data are in
      __syncwarp();
      pipe_pairs(a, m, task1, ntasks, sp.run[rs1], sp.bag[ps0 ^ 1], sp.start[ps0 ^ 1]);
      cp_async_commit();
      int t, D;
      if (task_table(a, m, task0, &t, &D)) {
        const int nv = D >> 2;
        const uint32_t (*rs)[4] = sp.run[rs0];
        if (nv > 4 && nv <= 32) {
          if (nv <= 8) short_task_piped<1, kEw>(a, m, t, rs, sp.bag[ps0], sp.start[ps0]);
          else if (nv <= 16) short_task_piped<2, kEw>(a, m, t, rs, sp.bag[ps0], sp.start[ps0]);
          else short_task_piped<4, kEw>(a, m, t, rs, sp.bag[ps0], sp.start[ps0]);
        } else if (nv <= 128) {
          ShortTask st;
          st.t = t;
          st.nv = nv;
          const int grp = static_cast<int>(lane_id()) / update_lanes(nv);
          st.p0 = rs[grp][0];
          st.p1 = rs[grp][1];
          st.key = rs[grp][2];
          if (nv <= 2) short_task<2, 1, false, kEw>(a, m, st);
          else if (nv <= 4) short_task<4, 1, false, kEw>(a, m, st);
          else if (nv <= 64) short_task<16, 4, false, kEw>(a, m, st);
          else short_task<32, 4, false, kEw>(a, m, st);
        }
      }
      task0 = task1;
      task1 = task2;
      rs0 = rs1;
      ps0 ^= 1;
    }
    cp_async_wait<0>();  // no copy outlives the block's shared memory
    return;
  }
#if TBE_DYNAMIC_RUNS
  uint32_t task = grab(a.cursors);
  ShortTask cur = fetch_task(a, m, task, ntasks);
  uint32_t raw = grab_raw(a.cursors);  // the next task's index, read next iteration
  while (task < ntasks) {
    const uint32_t task_next = ticket(raw);
    raw = grab_raw(a.cursors);
    const ShortTask next = fetch_task(a, m, task_next, ntasks);  // one task ahead
    task = task_next;
#else
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  uint32_t task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  ShortTask cur = fetch_task(a, m, task, ntasks);
  for (; task < ntasks; task += warps) {
    const ShortTask next = fetch_task(a, m, task + warps, ntasks);  // one task ahead
#endif
    const int nv = cur.nv;
    if (cur.t >= 0 && (nv > 128) == kWide) {
      if (kWide) short_task<32, 8, kWeighted, kEw>(a, m, cur);
      else if (nv <= 2) short_task<2, 1, kWeighted, kEw>(a, m, cur);
      else if (nv <= 4) short_task<4, 1, kWeighted, kEw>(a, m, cur);
      else if (nv <= 8) short_task<8, 1, kWeighted, kEw>(a, m, cur);
      else if (nv <= 16) short_task<8, 2, kWeighted, kEw>(a, m, cur);
      else if (nv <= 32) short_task<8, 4, kWeighted, kEw>(a, m, cur);
      else if (nv <= 64) short_task<16, 4, kWeighted, kEw>(a, m, cur);
      else short_task<32, 4, kWeighted, kEw>(a, m, cur);
    }
    cur = next;
  }
}

// -------------------------------------------------------------- long runs
// Sum pairs [s, e) over the whole warp: group g takes every G-th pair of each
// batch of 32; the next batch's pair data is fetched while this batch's rows
// are gathered.  The groups meet in a butterfly so every lane ends with its
// columns of the sum.
template <int S, int NC, bool kWeighted>
__device__ __forceinline__ void sum_pairs(const UpdArgs& a, int64_t d0, int nv, uint32_t s,
                                          uint32_t e, float (&acc)[NC][4]) {
  constexpr int G = 32 / S;
  constexpr int U = TBE_LONG_VECS / NC > 0 ? (TBE_LONG_VECS / NC < S ? TBE_LONG_VECS / NC : S) : 1;
  const int lane = static_cast<int>(lane_id());
  const int g = lane / S;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
  uint32_t my_b = 0xffffffffu;
  float my_w = 0.f;
  if (s + lane < e) load_pair<kWeighted>(a, s + lane, &my_b, &my_w);
  for (uint32_t base = s; base < e; base += 32) {
    const int cnt = static_cast<int>(e - base < 32u ? e - base : 32u);
    uint32_t nx_b = 0xffffffffu;
    float nx_w = 0.f;
    if (base + 32 + lane < e) load_pair<kWeighted>(a, base + 32 + lane, &nx_b, &nx_w);
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
        gather_row<S, NC>(a, d0, nv, b, v[uu], b < static_cast<uint32_t>(a.B));
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) fma_rows<NC>(acc, v[uu], wv[uu]);
    }
    my_b = nx_b;
    my_w = nx_w;
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
// Release: every lane fences its own stores before lane 0's decrement.
// Acquire: only the last arriver fences again before reading.
__device__ __forceinline__ bool arrive_last(uint32_t* counter) {
  __threadfence();
  __syncwarp();
  uint32_t prev = 0;
  if (lane_id() == 0) prev = atomicSub(counter, 1u);
  prev = __shfl_sync(kFull, prev, 0);
  if (prev == 1u) __threadfence();
  __syncwarp();
  return prev == 1u;
}

// The whole warp applies the update of one long run's row (every lane holds
// the summed gradient; group 0's lanes write).
template <int S, int NC, bool kEw>
__device__ __forceinline__ void finish_long_row(const UpdArgs& a, const Meta& m,
                                                const LongRunInfo& ri, float (&acc)[NC][4]) {
  const int t = static_cast<int>(ri.table);
  const int D = static_cast<int>(m.d_off[t + 1] - m.d_off[t]);
  const int64_t woff = m.w_off[t] + (static_cast<int64_t>(ri.key) - m.hb[t]) * D;
  const bool writer = static_cast<int>(lane_id()) < S;
  uint2 w_raw[NC];
  load_row<S, NC>(a, woff, D >> 2, w_raw, writer);
  const float m_old = a.momentum[ri.key];
  adagrad_apply<S, NC, kEw>(a, acc, D, ri.key, woff, w_raw, m_old, writer);
}

template <int S, int NC, bool kWeighted, bool kEw>
__device__ __forceinline__ void long_chunk(const UpdArgs& a, const Meta& m, const ChunkDesc& cd,
                                           const LongRunInfo& ri, bool two_launch) {
  const int t = static_cast<int>(ri.table);
  const int64_t d0 = m.d_off[t];
  const int D = static_cast<int>(m.d_off[t + 1] - d0);
  const int nv = D >> 2;
  float acc[NC][4];
  sum_pairs<S, NC, kWeighted>(a, d0, nv, cd.first, cd.end, acc);
  if (ri.nch == 1 && !two_launch) {
    finish_long_row<S, NC, kEw>(a, m, ri, acc);
    return;
  }
  store_partial<S, NC>(a.partials + static_cast<int64_t>(ri.chunk0 + cd.c) * a.max_D, nv, acc);
  if (two_launch) return;
  // Climb the run's reduction tree while this warp is the last arriver.
  uint32_t level_off = 0;   // first node of the current level within the run's tree
  uint32_t below = ri.nch;  // nodes on the level below
  uint32_t i = cd.c / kFanIn;
  for (;;) {
    const uint32_t here = (below + kFanIn - 1) / kFanIn;
    if (!arrive_last(a.tree_cnt + ri.tree0 + level_off + i)) return;
    const uint32_t first = i * kFanIn;
    const uint32_t kids = below - first < static_cast<uint32_t>(kFanIn) ? below - first : kFanIn;
    const float* src = level_off == 0 && below == ri.nch
                           ? a.partials + static_cast<int64_t>(ri.chunk0 + first) * a.max_D
                           : a.tree_part + static_cast<int64_t>(ri.tree0 + level_off - below + first) *
                                               a.max_D;
    sum_partials<S, NC>(src, a.max_D, kids, nv, acc);
    if (here == 1) {
      finish_long_row<S, NC, kEw>(a, m, ri, acc);
      return;
    }
    store_partial<S, NC>(a.tree_part + static_cast<int64_t>(ri.tree0 + level_off + i) * a.max_D, nv,
                         acc);
    level_off += here;
    below = here;
    i /= kFanIn;
  }
}

template <bool kWeighted, bool kWide, bool kEw>
__global__ void __launch_bounds__(256, TBE_LONG_MINB) long_chunks_kernel(UpdArgs a, bool two_launch) {
  __shared__ MetaSmem msm;
  const Meta m = load_meta(a, msm, false);
  const uint32_t nchunks = a.counters[kCntChunks];
#if TBE_DYNAMIC_RUNS
  uint32_t* cur = a.cursors + (kCntNextLong - kCntNextShort);
  for (uint32_t qi = grab(cur); qi < nchunks; qi = grab(cur)) {
#else
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t qi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; qi < nchunks; qi += warps) {
#endif
    const ChunkDesc cd = a.chunk_order[qi];
    const LongRunInfo ri = a.long_info[cd.run];
    const int t = static_cast<int>(ri.table);
    const int D = static_cast<int>(m.d_off[t + 1] - m.d_off[t]);
    if (D < 8 || D > kMaxD || (D & 7) || (m.d_off[t] & 7)) continue;
    const int nv = D >> 2;
    if ((nv > 128) != kWide) continue;
    if (kWide) long_chunk<32, 8, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else if (nv <= 2) long_chunk<2, 1, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else if (nv <= 4) long_chunk<4, 1, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else if (nv <= 8) long_chunk<8, 1, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else if (nv <= 16) long_chunk<8, 2, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else if (nv <= 32) long_chunk<8, 4, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else if (nv <= 64) long_chunk<16, 4, kWeighted, kEw>(a, m, cd, ri, two_launch);
    else long_chunk<32, 4, kWeighted, kEw>(a, m, cd, ri, two_launch);
  }
}

// Two-launch variant, second kernel: one warp per long run sums the run's
// chunk partials in chunk order and applies the update.
template <int S, int NC, bool kEw>
__device__ __forceinline__ void finish_run(const UpdArgs& a, const Meta& m, const LongRunInfo& ri) {
  const int t = static_cast<int>(ri.table);
  const int D = static_cast<int>(m.d_off[t + 1] - m.d_off[t]);
  float acc[NC][4];
  sum_partials<S, NC>(a.partials + static_cast<int64_t>(ri.chunk0) * a.max_D, a.max_D, ri.nch,
                      D >> 2, acc);
  finish_long_row<S, NC, kEw>(a, m, ri, acc);
}

template <bool kWide, bool kEw>
__global__ void __launch_bounds__(256, 3) long_finish_kernel(UpdArgs a) {
  __shared__ MetaSmem msm;
  const Meta m = load_meta(a, msm, false);
  const uint32_t nlong = a.counters[kCntLong];
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t k = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; k < nlong; k += warps) {
    const LongRunInfo ri = a.long_info[k];
    const int t = static_cast<int>(ri.table);
    const int D = static_cast<int>(m.d_off[t + 1] - m.d_off[t]);
    if (D < 8 || D > kMaxD || (D & 7) || (m.d_off[t] & 7)) continue;
    const int nv = D >> 2;
    if ((nv > 128) != kWide) continue;
    if (kWide) finish_run<32, 8, kEw>(a, m, ri);
    else if (nv <= 2) finish_run<2, 1, kEw>(a, m, ri);
    else if (nv <= 4) finish_run<4, 1, kEw>(a, m, ri);
    else if (nv <= 8) finish_run<8, 1, kEw>(a, m, ri);
    else if (nv <= 16) finish_run<8, 2, kEw>(a, m, ri);
    else if (nv <= 32) finish_run<8, 4, kEw>(a, m, ri);
    else if (nv <= 64) finish_run<16, 4, kEw>(a, m, ri);
    else finish_run<32, 4, kEw>(a, m, ri);
  }
}

// --------------------------------------------------------------- hot rows
// The hot rows' partial gradients come from the tensor-core kernel in
// hot_grad.cu (hot_part[t][p][slot][c]).
// One CTA per hot row that was looked up in this call: warp w adds the
// partitions w, w + 8, ... in order, warp 0 adds the eight warp sums in order
// (a fixed order, so the result is reproducible), then applies the row-wise
// Adagrad step.
template <bool kEw>
__global__ void __launch_bounds__(256)
    hot_finish_kernel(UpdArgs a, const uint32_t* __restrict__ hot_keys,
                      const uint32_t* __restrict__ hot_n, const uint32_t* __restrict__ hot_cnt,
                      int parts, const float* __restrict__ hot_part) {
  __shared__ __align__(16) float wsum[8][kHotMaxD];
  const int t = static_cast<int>(blockIdx.x / kHot), slot = static_cast<int>(blockIdx.x % kHot);
  if (slot >= static_cast<int>(min(hot_n[t], static_cast<uint32_t>(kHot))) ||
      hot_cnt[blockIdx.x] == 0)
    return;  // uniform over the CTA
  const int D = static_cast<int>(a.D_offsets[t + 1] - a.D_offsets[t]);
  if (D > kHotMaxD || (D & 7) || (a.D_offsets[t] & 7)) return;
  const int warp = threadIdx.x >> 5;
  const int lane = static_cast<int>(lane_id());
  const int nv = D >> 2;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int vec = lane + c * 32;
    if (vec < nv) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      const float* src = hot_part + (static_cast<int64_t>(t) * parts * kHot + slot) * kHotMaxD + vec * 4;
#pragma unroll 4
      for (int p = warp; p < parts; p += 8) {
        const float4 v = *reinterpret_cast<const float4*>(src + static_cast<int64_t>(p) * kHot * kHotMaxD);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      *reinterpret_cast<float4*>(&wsum[warp][vec * 4]) = acc;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  float acc[2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int vec = lane + c * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
    if (vec < nv)
      for (int w = 0; w < 8; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(&wsum[w][vec * 4]);
        acc[c][0] += v.x; acc[c][1] += v.y; acc[c][2] += v.z; acc[c][3] += v.w;
      }
  }
  const uint32_t key = hot_keys[blockIdx.x];
  if (key < a.hash_base[t] || key >= a.hash_base[t + 1]) return;  // not this table's row
  const int64_t woff = a.w_offsets[t] + (static_cast<int64_t>(key) - a.hash_base[t]) * D;
  uint2 w_raw[2];
  load_row<32, 2>(a, woff, nv, w_raw, true);
  const float m_old = a.momentum[key];
  adagrad_apply<32, 2, kEw>(a, acc, D, key, woff, w_raw, m_old, true);
}

// ------------------------------------------------------ hot set refresh
// The next call's hot rows: per table, the rows with the most lookups in
// this call (cold runs and current hot rows alike), at most kHot of them and
// only rows looked up at least min_count times.  Counts go to log-scale
// buckets (8 per octave); the cut is the lowest bucket whose suffix fits.
__device__ __forceinline__ int count_bucket(uint32_t c) {
  const int e = 31 - __clz(c);
  const uint32_t frac = e >= 3 ? (c >> (e - 3)) & 7u : (c << (3 - e)) & 7u;
  return e * 8 + static_cast<int>(frac);
}

// Candidate i: cold runs first, then the current hot slots.
__device__ __forceinline__ bool hot_candidate(const UpdArgs& a, const Meta& m, uint32_t i,
                                              uint32_t R, const uint32_t* run_starts,
                                              const uint32_t* hot_keys, const uint32_t* hot_n,
                                              const uint32_t* hot_cnt, uint32_t min_count,
                                              int* t_out, uint32_t* key_out, uint32_t* cnt_out) {
  int t;
  uint32_t key, cnt;
  if (i < R) {
    key = a.unique_keys[i];
    cnt = run_starts[i + 1] - run_starts[i];
    int lo = 0, hi = a.T - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (m.hb[mid] <= static_cast<int64_t>(key)) lo = mid; else hi = mid - 1;
    }
    t = lo;
  } else {
    const uint32_t w = i - R;
    t = static_cast<int>(w / kHot);
    if (w % kHot >= min(hot_n[t], static_cast<uint32_t>(kHot))) return false;
    key = hot_keys[w];
    cnt = hot_cnt[w];
  }
  if (cnt < min_count || m.d_off[t + 1] - m.d_off[t] > kHotMaxD) return false;
  *t_out = t;
  *key_out = key;
  *cnt_out = cnt;
  return true;
}

__global__ void __launch_bounds__(256)
    hot_hist_kernel(UpdArgs a, const uint32_t* __restrict__ run_starts,
                    const uint32_t* __restrict__ hot_keys, const uint32_t* __restrict__ hot_n,
                    const uint32_t* __restrict__ hot_cnt, uint32_t min_count,
                    uint32_t* __restrict__ sel_hist) {
  __shared__ MetaSmem msm;
  const Meta m = load_meta(a, msm, false);
  const uint32_t R = a.counters[kCntRuns];
  const uint32_t total = R + static_cast<uint32_t>(a.T) * kHot;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    int t;
    uint32_t key, cnt;
    if (hot_candidate(a, m, i, R, run_starts, hot_keys, hot_n, hot_cnt, min_count, &t, &key, &cnt))
      atomicAdd(&sel_hist[t * kHotBuckets + count_bucket(cnt)], 1u);
  }
}

__global__ void hot_thresh_kernel(int T, const uint32_t* __restrict__ sel_hist,
                                  uint32_t* __restrict__ sel_thresh) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    uint32_t acc = 0, cut = 0;
    for (int b = kHotBuckets - 1; b >= 0; --b) {
      acc += sel_hist[t * kHotBuckets + b];
      if (acc > static_cast<uint32_t>(kHot)) {
        cut = static_cast<uint32_t>(b + 1);
        break;
      }
    }
    sel_thresh[t] = cut;
  }
}

__global__ void __launch_bounds__(256)
    hot_select_kernel(UpdArgs a, const uint32_t* __restrict__ run_starts,
                      const uint32_t* __restrict__ hot_keys, const uint32_t* __restrict__ hot_n,
                      const uint32_t* __restrict__ hot_cnt, uint32_t min_count,
                      const uint32_t* __restrict__ sel_thresh, uint32_t* __restrict__ sel_keys,
                      uint32_t* __restrict__ sel_cnt, uint32_t* __restrict__ sel_n) {
  __shared__ MetaSmem msm;
  const Meta m = load_meta(a, msm, false);
  const uint32_t R = a.counters[kCntRuns];
  const uint32_t total = R + static_cast<uint32_t>(a.T) * kHot;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    int t;
    uint32_t key, cnt;
    if (hot_candidate(a, m, i, R, run_starts, hot_keys, hot_n, hot_cnt, min_count, &t, &key, &cnt) &&
        static_cast<uint32_t>(count_bucket(cnt)) >= sel_thresh[t]) {
      const uint32_t slot = atomicAdd(&sel_n[t], 1u);
      if (slot < static_cast<uint32_t>(kHot)) {
        sel_keys[t * kHot + slot] = key;
        sel_cnt[t * kHot + slot] = cnt;
      }
    }
  }
}

// The selected keys, ordered per table by lookups (most first, ties by key:
// the expand counts the first slots by warp votes), become the hot set,
// together with a place for each key in the two-choice hash (see
// kCuckooHalf): one CTA per table sorts them (bitonic), then one thread
// inserts them with
// displacement under the first multiplier pair of a fixed sequence for which
// every insertion succeeds within kCuckooKicks moves.  At a load of 1/4 the
// first pair almost always succeeds; if kCuckooTries pairs fail, keys that
// find no free place without displacement under the first pair are dropped
// from the set (a smaller set stays correct, only less effective).
constexpr int kCuckooTries = 64;
constexpr int kCuckooKicks = 128;

__device__ __forceinline__ uint32_t odd_mult(int i) {
  return (0x9E3779B1u + 2u * static_cast<uint32_t>(i) * 0x3C6EF372u) | 1u;
}

// Inserts key into tab (kEmptyKey = free); false if kicks run out (the table
// then holds some other key displaced out, so the caller starts over).
__device__ bool cuckoo_insert(uint32_t* tab, uint32_t key, uint32_t m1, uint32_t m2,
                              bool displace) {
  uint32_t cur = key;
  uint32_t pos = cuckoo_h1(cur, m1);
  if (tab[pos] == kEmptyKey) { tab[pos] = cur; return true; }
  pos = cuckoo_h2(cur, m2);
  if (tab[pos] == kEmptyKey) { tab[pos] = cur; return true; }
  if (!displace) return false;
  for (int kick = 0; kick < kCuckooKicks; ++kick) {
    const uint32_t out = tab[pos];
    tab[pos] = cur;
    cur = out;
    // the displaced key moves to its other place
    pos = pos == cuckoo_h1(cur, m1) ? cuckoo_h2(cur, m2) : cuckoo_h1(cur, m1);
    if (tab[pos] == kEmptyKey) { tab[pos] = cur; return true; }
  }
  return false;
}

__global__ void __launch_bounds__(kHot)
    hot_commit_kernel(const uint32_t* __restrict__ sel_keys, const uint32_t* __restrict__ sel_cnt,
                      const uint32_t* __restrict__ sel_n,
                      uint32_t* __restrict__ hot_keys, uint32_t* __restrict__ hot_place,
                      uint32_t* __restrict__ hot_n, uint32_t* __restrict__ hot_m1,
                      uint32_t* __restrict__ hot_m2) {
  __shared__ uint32_t k[kHot];
  __shared__ unsigned long long order[kHot];  // (~count) << 32 | key: ascending = most first
  __shared__ uint32_t tab[kCuckooSize];
  __shared__ uint32_t scan[33];
  __shared__ uint32_t mults[2];
  const int t = blockIdx.x;
  const int i = threadIdx.x;
  const uint32_t nsel = min(sel_n[t], static_cast<uint32_t>(kHot));
  order[i] = i < static_cast<int>(nsel)
                 ? (static_cast<unsigned long long>(~sel_cnt[t * kHot + i]) << 32) |
                       sel_keys[t * kHot + i]
                 : ~0ull;  // padding sorts last
  // bitonic sort of kHot entries, ascending
  for (int size = 2; size <= kHot; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      const int j = i ^ stride;
      if (j > i) {
        const bool up = (i & size) == 0;
        const unsigned long long a = order[i], b = order[j];
        if ((a > b) == up) { order[i] = b; order[j] = a; }
      }
    }
  __syncthreads();
  k[i] = i < static_cast<int>(nsel) ? static_cast<uint32_t>(order[i]) : kEmptyKey;
  __syncthreads();
  if (i == 0) {
    bool ok = false;
    uint32_t m1 = odd_mult(0), m2 = odd_mult(1);
    for (int tr = 0; tr < kCuckooTries && !ok; ++tr) {
      m1 = odd_mult(2 * tr);
      m2 = odd_mult(2 * tr + 1);
      for (int e = 0; e < kCuckooSize; ++e) tab[e] = kEmptyKey;
      ok = true;
      for (uint32_t s = 0; s < nsel && ok; ++s) ok = cuckoo_insert(tab, k[s], m1, m2, true);
    }
    if (!ok) {
      m1 = odd_mult(0);
      m2 = odd_mult(1);
      for (int e = 0; e < kCuckooSize; ++e) tab[e] = kEmptyKey;
      for (uint32_t s = 0; s < nsel; ++s) cuckoo_insert(tab, k[s], m1, m2, false);
    }
    mults[0] = m1;
    mults[1] = m2;
  }
  __syncthreads();
  const uint32_t m1 = mults[0], m2 = mults[1];
  // keep the placed keys in sorted order with their places
  uint32_t place = kCuckooSize;
  if (i < static_cast<int>(nsel)) {
    const uint32_t key = k[i];
    if (tab[cuckoo_h1(key, m1)] == key) place = cuckoo_h1(key, m1);
    else if (tab[cuckoo_h2(key, m2)] == key) place = cuckoo_h2(key, m2);
  }
  const uint32_t kept = place < static_cast<uint32_t>(kCuckooSize) ? 1u : 0u;
  uint32_t total;
  const uint32_t inc = block_inclusive_scan(kept, OpSum(), 0u, scan, &total);
  if (kept) {
    hot_keys[t * kHot + inc - 1] = k[i];
    hot_place[t * kHot + inc - 1] = place;
  }
  if (i == 0) {
    hot_n[t] = total;
    hot_m1[t] = m1;
    hot_m2[t] = m2;
  }
}

// Mean pooling's backward input (the HugeCTR page's mean backward step): the
// gradient row of bag (t, b) times the bag's factor, 1/L for L > 1 lookups,
// before the regrouping.  Grid: x over the table's B x D_t/4 vectors, y = t.
__global__ void __launch_bounds__(256)
    scale_grad_kernel(const float* __restrict__ grad, const float* __restrict__ inv_len,
                      const int64_t* __restrict__ D_offsets, int B, int64_t total_D,
                      float* __restrict__ out) {
  const int t = blockIdx.y;
  const int64_t d0 = D_offsets[t];
  const int nv = static_cast<int>((D_offsets[t + 1] - d0) >> 2);
  const int64_t nvec = static_cast<int64_t>(B) * nv;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / nv;
    const int v = static_cast<int>(i - b * nv);
    const float sc = __ldg(inv_len + static_cast<int64_t>(t) * B + b);
    const int64_t at = b * total_D + d0 + v * 4;
    float4 g = ldg_f4(grad + at);
    g.x *= sc; g.y *= sc; g.z *= sc; g.w *= sc;
    *reinterpret_cast<float4*>(out + at) = g;
  }
}

#ifndef TBE_HOT_GRAD_SIDE
#define TBE_HOT_GRAD_SIDE 0
#endif

// The cold runs' update kernels (short, medium, long chunks, and the second
// long-run kernel in the two-launch variant) on L's stream, in that order.
template <bool kEw>
void launch_runs(const Launch& L, const UpdArgs& a, const uint32_t* medium, unsigned blocks,
                 bool weighted, bool wide, bool two_launch) {
  // with work cursors, the CTAs the SMs hold at once take every task: a
  // larger grid only adds CTAs that start late and find the cursor spent
  const unsigned sms = static_cast<unsigned>(L.num_sms);
  const unsigned short_blocks = TBE_DYNAMIC_RUNS ? sms * TBE_SHORT_MINB : blocks;
  const unsigned medium_blocks = TBE_DYNAMIC_RUNS ? sms * (a.max_D <= 128 ? 3u : 2u) : blocks;
  const unsigned long_blocks = TBE_DYNAMIC_RUNS ? sms * TBE_LONG_MINB : blocks;
  if (weighted) { probe_begin(TBE_PROBE_SHORT_RUNS, L.s); short_runs_kernel<true, false, kEw><<<short_blocks, 256, 0, L.s>>>(a); note_launch(); probe_end(TBE_PROBE_SHORT_RUNS, L.s); }
  else { probe_begin(TBE_PROBE_SHORT_RUNS, L.s); short_runs_kernel<false, false, kEw><<<short_blocks, 256, 0, L.s>>>(a); note_launch(); probe_end(TBE_PROBE_SHORT_RUNS, L.s); }
  {
    const bool narrow = a.max_D <= 128;
    probe_begin(TBE_PROBE_MEDIUM_RUNS, L.s);
    if (weighted && narrow) medium_runs_kernel<true, true, kEw><<<medium_blocks, 256, 0, L.s>>>(a, medium);
    else if (weighted) medium_runs_kernel<true, false, kEw><<<medium_blocks, 256, 0, L.s>>>(a, medium);
    else if (narrow) medium_runs_kernel<false, true, kEw><<<medium_blocks, 256, 0, L.s>>>(a, medium);
    else medium_runs_kernel<false, false, kEw><<<medium_blocks, 256, 0, L.s>>>(a, medium);
    note_launch();
    probe_end(TBE_PROBE_MEDIUM_RUNS, L.s);
  }
  // a second launch of a kernel with a work cursor (rows wider than 512
  // values) starts its cursor afresh
  auto reset = [&](int c) {
    if (TBE_DYNAMIC_RUNS && wide) cudaMemsetAsync(a.cursors + (c - kCntNextShort), 0, 4, L.s);
  };
  reset(kCntNextShort);
  if (wide && weighted) { probe_begin(TBE_PROBE_SHORT_RUNS, L.s); short_runs_kernel<true, true, kEw><<<short_blocks, 256, 0, L.s>>>(a); note_launch(); probe_end(TBE_PROBE_SHORT_RUNS, L.s); }
  if (wide && !weighted) { probe_begin(TBE_PROBE_SHORT_RUNS, L.s); short_runs_kernel<false, true, kEw><<<short_blocks, 256, 0, L.s>>>(a); note_launch(); probe_end(TBE_PROBE_SHORT_RUNS, L.s); }
  if (weighted) { probe_begin(TBE_PROBE_LONG_CHUNKS, L.s); long_chunks_kernel<true, false, kEw><<<long_blocks, 256, 0, L.s>>>(a, two_launch); note_launch(); probe_end(TBE_PROBE_LONG_CHUNKS, L.s); }
  else { probe_begin(TBE_PROBE_LONG_CHUNKS, L.s); long_chunks_kernel<false, false, kEw><<<long_blocks, 256, 0, L.s>>>(a, two_launch); note_launch(); probe_end(TBE_PROBE_LONG_CHUNKS, L.s); }
  reset(kCntNextLong);
  if (wide && weighted) { probe_begin(TBE_PROBE_LONG_CHUNKS, L.s); long_chunks_kernel<true, true, kEw><<<long_blocks, 256, 0, L.s>>>(a, two_launch); note_launch(); probe_end(TBE_PROBE_LONG_CHUNKS, L.s); }
  if (wide && !weighted) { probe_begin(TBE_PROBE_LONG_CHUNKS, L.s); long_chunks_kernel<false, true, kEw><<<long_blocks, 256, 0, L.s>>>(a, two_launch); note_launch(); probe_end(TBE_PROBE_LONG_CHUNKS, L.s); }
  if (two_launch) {
    { long_finish_kernel<false, kEw><<<blocks, 256, 0, L.s>>>(a); note_launch(); }
    if (wide) { long_finish_kernel<true, kEw><<<blocks, 256, 0, L.s>>>(a); note_launch(); }
  }
}

}  // namespace

cudaError_t launch_update(const Launch& L, const WsLayout& W, char* ws, const float* grad_out,
                          void* weights, float* momentum, float lr, float eps, bool two_launch,
                          bool elementwise) {
  const tbe_desc* d = L.d;
  const int fin = radix_passes(d) & 1;
  UpdArgs a;
  a.grad_out = grad_out;
  a.W = static_cast<__half*>(weights);  // 16-bit rows; a.bf16 picks the codec
  a.bf16 = d->weights_dtype == TBE_DT_BF16;
  a.f32 = d->weights_dtype == TBE_DT_F32;
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
  a.long_info = reinterpret_cast<const LongRunInfo*>(ws + W.long_info);
  a.chunk_order = reinterpret_cast<const ChunkDesc*>(ws + W.chunk_order);
  a.tree_cnt = reinterpret_cast<uint32_t*>(ws + W.tree_cnt);
  a.cursors = reinterpret_cast<uint32_t*>(ws + W.counts) + kCntNextShort;
  a.partials = reinterpret_cast<float*>(ws + W.partials);
  a.tree_part = reinterpret_cast<float*>(ws + W.tree_part);
  a.total_D = d->total_D;
  a.T = d->T;
  a.B = d->B;
  a.max_D = d->max_D;
  a.lr = lr;
  a.eps = eps;
  if (L.n == 0) return cudaSuccess;
  SideFlow* sf = side_flow(ws);
  if (!sf) return cudaErrorNotReady;
  const unsigned blocks = static_cast<unsigned>(L.num_sms) * 8u;
  const bool weighted = a.sorted_psw != nullptr;
  const bool wide = d->max_D > 512;  // rows of more than 128 float4 vectors
  // Hot rows on the side stream, concurrently with the cold rows below
  // (disjoint rows): their gradient needs grad_out (ready on the caller's
  // stream) and the histogram; the side stream has finished the sort chain
  // before it starts.
  const uint32_t* hot_keys = reinterpret_cast<const uint32_t*>(ws + W.hot_keys(W.hot_cur));
  const uint32_t* hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
  const uint32_t* hot_cnt = reinterpret_cast<const uint32_t*>(ws + W.hot_cnt);
  if (W.hot_enabled) {
    // TBE_HOT_GRAD_SIDE 0: on the caller's stream, before the cold rows
    cudaError_t e = TBE_HOT_GRAD_SIDE ? fork_to(sf, L.s) : cudaSuccess;
    if (e != cudaSuccess) return e;
    Launch Ls = L;
    if (TBE_HOT_GRAD_SIDE) Ls.s = sf->side;
    const float* part = reinterpret_cast<const float*>(ws + W.hot_part);
    e = launch_hot_grad(Ls, W, ws, grad_out);
    if (e != cudaSuccess) return e;
    if (elementwise)
      hot_finish_kernel<true><<<static_cast<unsigned>(d->T) * kHot, 256, 0, Ls.s>>>(
          a, hot_keys, hot_n, hot_cnt, W.hot_parts, part);
    else
      hot_finish_kernel<false><<<static_cast<unsigned>(d->T) * kHot, 256, 0, Ls.s>>>(
          a, hot_keys, hot_n, hot_cnt, W.hot_parts, part);
    note_launch();
    e = flow_record(sf->hot, Ls.s);
    if (e != cudaSuccess) return e;
    if (TBE_HOT_GRAD_SIDE) {  // the side stream's latest work (after the refresh)
      e = flow_record(sf->done, Ls.s);
      if (e != cudaSuccess) return e;
    }
  }
  // the cold rows need the sort chain; their work cursors start at zero
  {
    cudaError_t e = flow_wait(L.s, sf->sorted);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.cursors, 0, 3 * sizeof(uint32_t), L.s);
    if (e != cudaSuccess) return e;
  }
  const uint32_t* medium = reinterpret_cast<const uint32_t*>(ws + W.medium_run);
  if (elementwise) launch_runs<true>(L, a, medium, blocks, weighted, wide, two_launch);
  else launch_runs<false>(L, a, medium, blocks, weighted, wide, two_launch);
  cudaError_t e = cudaSuccess;
  if (W.hot_enabled) {  // without a histogram the hot set stays empty
    // the caller's stream joins the hot rows' update
    e = flow_wait(L.s, sf->hot);
    if (e != cudaSuccess) return e;
    if (!TBE_REFRESH_IN_PREPROCESS) {  // else the preprocess chose the next set
      e = launch_hot_refresh(L, W, ws);
      if (e != cudaSuccess) return e;
    }
  }
  // and every side-stream segment of this call and of its preprocess (the
  // sort chain, the hot-set refresh): once the call's work on the caller's
  // stream is done, all of it is, and a CUDA graph that captures whole steps
  // has no unjoined work
  e = flow_wait(L.s, sf->done);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The next call's hot set, chosen from this call's lookups: the cold runs'
// lengths and the hot rows' counts (none of the gradients), written to the
// workspace's second hot set on L's stream.
cudaError_t launch_hot_refresh(const Launch& L, const WsLayout& W, char* ws) {
  const tbe_desc* d = L.d;
  if (L.n == 0 || !W.hot_enabled) return cudaSuccess;
  UpdArgs a{};
  a.D_offsets = d->D_offsets;
  a.hash_base = d->hash_base;
  a.w_offsets = d->weights_offsets;
  a.unique_keys = reinterpret_cast<const uint32_t*>(ws + W.unique_keys);
  a.counters = reinterpret_cast<const uint32_t*>(ws + W.counts);
  a.T = d->T;
  a.B = d->B;
  a.max_D = d->max_D;
  const unsigned blocks = static_cast<unsigned>(L.num_sms) * 8u;
  const uint32_t* hot_keys = reinterpret_cast<const uint32_t*>(ws + W.hot_keys(W.hot_cur));
  const uint32_t* hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_cur));
  const uint32_t* hot_cnt = reinterpret_cast<const uint32_t*>(ws + W.hot_cnt);
  cudaError_t e = cudaMemsetAsync(ws + W.sel_hist, 0, static_cast<size_t>(d->T) * kHotBuckets * 4, L.s);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ws + W.sel_n, 0, static_cast<size_t>(d->T) * 4, L.s);
  if (e != cudaSuccess) return e;
  const uint32_t min_count =
      d->B / kHotMinCountDiv > 32 ? static_cast<uint32_t>(d->B / kHotMinCountDiv) : 32u;
  const uint32_t* rs = reinterpret_cast<const uint32_t*>(ws + W.run_starts);
  uint32_t* sel_hist = reinterpret_cast<uint32_t*>(ws + W.sel_hist);
  uint32_t* sel_thresh = reinterpret_cast<uint32_t*>(ws + W.sel_thresh);
  uint32_t* sel_keys = reinterpret_cast<uint32_t*>(ws + W.sel_keys);
  uint32_t* sel_cnt = reinterpret_cast<uint32_t*>(ws + W.sel_cnt);
  uint32_t* sel_n = reinterpret_cast<uint32_t*>(ws + W.sel_n);
  { hot_hist_kernel<<<blocks, 256, 0, L.s>>>(a, rs, hot_keys, hot_n, hot_cnt, min_count, sel_hist); note_launch(); }
  { hot_thresh_kernel<<<(d->T + 127) / 128, 128, 0, L.s>>>(d->T, sel_hist, sel_thresh); note_launch(); }
  { hot_select_kernel<<<blocks, 256, 0, L.s>>>(a, rs, hot_keys, hot_n, hot_cnt, min_count,
                                             sel_thresh, sel_keys, sel_cnt, sel_n); note_launch(); }
  { hot_commit_kernel<<<static_cast<unsigned>(d->T), kHot, 0, L.s>>>(
      sel_keys, sel_cnt, sel_n, reinterpret_cast<uint32_t*>(ws + W.hot_keys(W.hot_next)),
      reinterpret_cast<uint32_t*>(ws + W.hot_place(W.hot_next)),
      reinterpret_cast<uint32_t*>(ws + W.hot_n(W.hot_next)),
      reinterpret_cast<uint32_t*>(ws + W.hot_m1(W.hot_next)),
      reinterpret_cast<uint32_t*>(ws + W.hot_m2(W.hot_next))); note_launch(); }
  return cudaGetLastError();
}

cudaError_t launch_scale_grad(const Launch& L, const float* grad_out, const float* inv_len,
                              float* out) {
  const tbe_desc* d = L.d;
  const int64_t vecs = static_cast<int64_t>(d->B) * (d->max_D / 4);
  int64_t bx = (vecs + 255) / 256;
  const int64_t cap = 8LL * L.num_sms;
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  if (d->T > 65535) return cudaErrorInvalidConfiguration;
  scale_grad_kernel<<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(d->T)), 256, 0, L.s>>>(
      grad_out, inv_len, d->D_offsets, d->B, d->total_D, out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tbe
