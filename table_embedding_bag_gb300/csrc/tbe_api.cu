// C ABI entry points: argument validation, workspace layout and launch order.
// The operations themselves are specified in include/tbe.h.
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace tbe {

std::atomic<uint64_t> g_kernel_launches{0};

void note_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

#ifndef TBE_SIDE_PRIORITY
#define TBE_SIDE_PRIORITY 1
#endif

namespace {
// Side flows by (device, workspace address).  Entries live until the process
// exits (a stream and four events each); a workspace freed and another
// allocated at the same address shares the entry, which only orders the new
// workspace's calls after the old one's.
std::mutex g_flow_mu;
std::map<std::pair<int, const void*>, SideFlow*> g_flows;

SideFlow* lookup_flow(const void* ws, bool create) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_flow_mu);
  const auto key = std::make_pair(dev, ws);
  auto it = g_flows.find(key);
  if (it != g_flows.end()) return it->second;
  if (!create) return nullptr;
  SideFlow f;
  const unsigned ef = cudaEventDisableTiming;
  // TBE_SIDE_PRIORITY: the side stream at the device's greatest priority
  // (its blocks are scheduled ahead of the caller's default-priority ones)
  int prio_least = 0, prio_greatest = 0;
  if (TBE_SIDE_PRIORITY && cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest) != cudaSuccess)
    prio_greatest = 0;
  const int prio = TBE_SIDE_PRIORITY ? prio_greatest : 0;
  const bool ok = cudaStreamCreateWithPriority(&f.side, cudaStreamNonBlocking, prio) == cudaSuccess &&
                  cudaEventCreateWithFlags(&f.fork, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&f.sorted.ev, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&f.hot.ev, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&f.done.ev, ef) == cudaSuccess;
  if (!ok) {
    // give back what was created; the next call tries again
    for (cudaEvent_t e : {f.fork, f.sorted.ev, f.hot.ev, f.done.ev})
      if (e) cudaEventDestroy(e);
    if (f.side) cudaStreamDestroy(f.side);
    return nullptr;
  }
  SideFlow* p = new SideFlow(f);
  g_flows.emplace(key, p);
  return p;
}
}  // namespace

SideFlow* side_flow(const void* ws) { return lookup_flow(ws, true); }
SideFlow* find_side_flow(const void* ws) { return lookup_flow(ws, false); }

cudaError_t fork_to(SideFlow* f, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(f->fork, s);
  if (e != cudaSuccess) return e;
  return cudaStreamWaitEvent(f->side, f->fork, 0);
}

namespace {
// The id of the capture s is in, 0 when it is not being captured.
cudaError_t capture_id(cudaStream_t s, unsigned long long* id) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  unsigned long long v = 0;
  const cudaError_t e = cudaStreamGetCaptureInfo(s, &cs, &v);
  *id = cs == cudaStreamCaptureStatusActive ? v : 0ull;
  return e;
}
}  // namespace

cudaError_t flow_record(FlowEvent& e, cudaStream_t s) {
  unsigned long long id = 0;
  const cudaError_t err = capture_id(s, &id);
  if (err != cudaSuccess) return err;
  e.capture = id;
  return cudaEventRecord(e.ev, s);
}

cudaError_t flow_wait(cudaStream_t s, const FlowEvent& e) {
  unsigned long long id = 0;
  const cudaError_t err = capture_id(s, &id);
  if (err != cudaSuccess) return err;
  if (id != e.capture) return cudaSuccess;
  return cudaStreamWaitEvent(s, e.ev, 0);
}


namespace {
constexpr int kProbeMax = 256;
std::mutex g_probe_mu;
std::atomic<uint32_t> g_probe_kernel{0};
cudaEvent_t g_probe_ev[kProbeMax][2] = {};
int g_probe_used = 0;   // launches recorded
bool g_probe_open = false;
}  // namespace

void probe_begin(uint32_t kernel, cudaStream_t s) {
  if (g_probe_kernel.load(std::memory_order_relaxed) != kernel || kernel == 0) return;
  std::lock_guard<std::mutex> lk(g_probe_mu);
  if (g_probe_used >= kProbeMax || g_probe_open) return;
  cudaEvent_t* ev = g_probe_ev[g_probe_used];
  if (!ev[0] && cudaEventCreate(&ev[0]) != cudaSuccess) return;
  if (!ev[1] && cudaEventCreate(&ev[1]) != cudaSuccess) return;
  if (cudaEventRecord(ev[0], s) == cudaSuccess) g_probe_open = true;
}

void probe_end(uint32_t kernel, cudaStream_t s) {
  if (g_probe_kernel.load(std::memory_order_relaxed) != kernel || kernel == 0) return;
  std::lock_guard<std::mutex> lk(g_probe_mu);
  if (!g_probe_open) return;
  g_probe_open = false;
  if (cudaEventRecord(g_probe_ev[g_probe_used][1], s) == cudaSuccess) ++g_probe_used;
}

cudaError_t prepare_preprocess_kernels();

WsLayout make_layout(const tbe_desc* d, int64_t n, uint32_t ws_flags, bool allow_hot) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.weighted = (ws_flags & TBE_WS_WEIGHTED) != 0;
  const size_t un = static_cast<size_t>(n);
  // State kept across calls comes first, at offsets that depend only on T,
  // so calls with different n (or weightedness) on one workspace agree.
  L.status = take(64);
  L.T = d->T;
  L.hot_set_bytes = static_cast<size_t>(d->T) * (2 * kHot + 3) * 4;
  L.hot_cur = take(L.hot_set_bytes);
  L.hot_next = take(L.hot_set_bytes);
  L.counts = take(kNumCounters * sizeof(uint32_t));
  L.table_runs = take((d->T + 1) * sizeof(uint32_t));
  L.table_tasks = take((d->T + 1) * sizeof(uint32_t));
  // sort buffers keep 64 spare bytes: whole 16-byte tile copies stay inside
  for (int i = 0; i < 3; ++i) L.keys[i] = take(un * 4 + 64);
  for (int i = 0; i < 3; ++i) L.vals[i] = take(un * 4 + 64);
  for (int i = 0; i < 3; ++i) L.psw[i] = L.weighted ? take(un * 4 + 64) : 0;
  L.radix_counts = take(sizeof(uint32_t) * (1u << kMaxRadixBits) * (kMaxSortCtas + 1));
  L.cta_counts = take(sizeof(uint32_t) * 2 * (kMaxSortCtas + 1));
  L.unique_keys = take((un + 1) * 4);
  L.run_starts = take((un + 2) * 4);
  L.run_pairs = take((un + 2) * 4);
  L.pair_starts = take((un + 2) * 4);
  L.pair_bags = take((un + 1) * 4);
  L.max_long = n / kLongThreshold + 1;
  L.max_chunks = n / kChunk + L.max_long + 1;
  L.max_tree = L.max_chunks / (kFanIn - 1) + 8 * L.max_long + 1;
  L.max_medium = n / kMediumRun + 1;
  L.medium_run = take(L.max_medium * 4);
  L.long_run = take(L.max_long * 4);
  L.long_chunk0 = take(L.max_long * 4);
  L.long_tree0 = take(L.max_long * 4);
  L.long_info = take(L.max_long * sizeof(LongRunInfo));
  L.chunk_desc = take(L.max_chunks * sizeof(ChunkDesc));
  L.chunk_band = take(L.max_chunks * 4);
  L.chunk_order = take(L.max_chunks * sizeof(ChunkDesc));
  L.band_count = take(kBagBands * 4);
  L.tree_cnt = take(L.max_tree * 4);
  L.partials = take(static_cast<size_t>(L.max_chunks) * d->max_D * 4);
  L.tree_part = take(static_cast<size_t>(L.max_tree) * d->max_D * 4);
  const int64_t T = d->T, B = d->B;
  L.hot_tiles = T * ((B + kHotTileBags - 1) / kHotTileBags);
  // hot-gradient partitions: about kHotCtaTarget CTAs in all, at least
  // kHotMinPartBags bags each
  L.hot_parts = static_cast<int>(kHotCtaTarget / T > 0 ? kHotCtaTarget / T : 1);
  const int64_t max_parts = (B + kHotMinPartBags - 1) / kHotMinPartBags;
  if (L.hot_parts > max_parts) L.hot_parts = static_cast<int>(max_parts);
  // the hot rows' tensor-core kernels take 16-bit weights (fp16 or bf16)
  L.hot_enabled = allow_hot &&
                  (d->weights_dtype == TBE_DT_F16 || d->weights_dtype == TBE_DT_BF16) &&
                  static_cast<size_t>(T) * kHot * B * (sizeof(float) + 1) <= kHotBudgetBytes;
  L.hot_cnt = take(T * kHot * 4);
  L.hot_hist8 = L.hot_enabled ? take(static_cast<size_t>(T) * kHot * B) : 0;
  L.hot_hist = L.hot_enabled ? take(static_cast<size_t>(T) * kHot * B * sizeof(float)) : 0;
  L.tile_kind = take(L.hot_tiles);
  L.hot_part = L.hot_enabled ? take(static_cast<size_t>(T) * L.hot_parts * kHot * kHotMaxD * 4) : 0;
  L.hot_scale = take(static_cast<size_t>(T) * B);
  L.bag_cold = take(static_cast<size_t>(T) * B * 4);
  L.cold_off = take((static_cast<size_t>(T) * B + 1) * 4);
  L.inv_len = take(static_cast<size_t>(T) * B * 4);
  L.tile_cold = take((L.hot_tiles + 1) * 4);
  L.sel_hist = take(T * kHotBuckets * 4);
  L.sel_thresh = take(T * 4);
  L.sel_keys = take(T * kHot * 4);
  L.sel_cnt = take(T * kHot * 4);
  L.sel_n = take(T * 4);
  const int64_t nb1 = T * B + 1;
  L.offsets_fix = take(nb1 * index_bytes(d));
  L.fix_scratch = take(repair_scratch_blocks(nb1) * sizeof(int64_t));
  // last, so layouts with and without it agree on every other offset
  L.grad_mean = (ws_flags & TBE_WS_MEAN) ? take(static_cast<size_t>(B) * d->total_D * 4) : 0;
  L.total = off;
  return L;
}

namespace {

tbe_status check_desc(const tbe_desc* d) {
  if (!d) return TBE_EINVAL;
  if (d->T < 1 || d->B < 1 || !d->D_offsets || !d->hash_base || !d->weights_offsets)
    return TBE_EINVAL;
  if (d->weights_dtype != TBE_DT_F16 && d->weights_dtype != TBE_DT_BF16 &&
      d->weights_dtype != TBE_DT_F32)
    return TBE_EUNSUPPORTED;
  if (d->index_dtype != TBE_DT_I32 && d->index_dtype != TBE_DT_I64) return TBE_EUNSUPPORTED;
  if (d->min_D < 8 || d->max_D > kMaxD || d->min_D > d->max_D || (d->min_D & 7) ||
      (d->max_D & 7) || d->total_D < d->max_D || (d->total_D & 7))
    return TBE_EUNSUPPORTED;
  if (d->total_E < 1 || d->total_E >= 0xffffffffLL) return TBE_EUNSUPPORTED;
  if (static_cast<int64_t>(d->B) * d->T >= 0x7fffffffLL) return TBE_EUNSUPPORTED;
  return TBE_OK;
}

tbe_status check_n(int64_t n) {
  if (n < 0) return TBE_EINVAL;
  if (n >= 0xfffffff0LL) return TBE_EUNSUPPORTED;
  return TBE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device, and the device's kernel set-up (shared
// memory attributes), done once per device; a set-up that fails is tried
// again by the next call.
int device_sms() {
  static int sms[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
      return 148;
    if (prepare_preprocess_kernels() != cudaSuccess) return v;
    sms[dev] = v;
  }
  return sms[dev];
}

tbe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TBE_OK : TBE_ECUDA; }

// Offsets check / repair shared by every entry point.  Returns the offsets
// pointer the kernels should read.
tbe_status run_checks(const Launch& L, const WsLayout& W, char* ws, const void* offsets,
                      uint32_t flags, const void** offsets_eff, int** status) {
  *offsets_eff = offsets;
  *status = nullptr;
  if (!(flags & (TBE_F_CHECK_BOUNDS | TBE_F_REPAIR_OFFSETS))) return TBE_OK;
  *status = reinterpret_cast<int*>(ws + W.status);
  const bool repair = (flags & TBE_F_REPAIR_OFFSETS) != 0;
  cudaError_t e = launch_check_offsets(L, offsets, repair, ws + W.offsets_fix,
                                       reinterpret_cast<int64_t*>(ws + W.fix_scratch), *status);
  if (e != cudaSuccess) return TBE_ECUDA;
  if (repair) *offsets_eff = ws + W.offsets_fix;
  return TBE_OK;
}

tbe_status common_args(const tbe_desc* d, const void* indices, const void* offsets, int64_t n,
                       void* workspace, size_t ws_bytes, bool weighted, WsLayout* W,
                       bool mean = false) {
  tbe_status st = check_desc(d);
  if (st != TBE_OK) return st;
  st = check_n(n);
  if (st != TBE_OK) return st;
  if (!offsets || (n > 0 && !indices)) return TBE_EINVAL;
  if (!workspace || !aligned16(workspace)) return TBE_EWORKSPACE;
  *W = make_layout(d, n, (weighted ? TBE_WS_WEIGHTED : 0u) | (mean ? TBE_WS_MEAN : 0u));
  if (ws_bytes < W->total) return TBE_EWORKSPACE;
  return TBE_OK;
}

}  // namespace
}  // namespace tbe

using namespace tbe;

extern "C" {

tbe_status tbe_workspace_size(const tbe_desc* d, int64_t n_max, uint32_t ws_flags,
                              size_t* bytes) {
  if (!bytes) return TBE_EINVAL;
  tbe_status st = check_desc(d);
  if (st != TBE_OK) return st;
  st = check_n(n_max);
  if (st != TBE_OK) return st;
  *bytes = make_layout(d, n_max, ws_flags).total;
  return TBE_OK;
}

tbe_status tbe_forward(const tbe_desc* d, const void* weights, const void* indices,
                       const void* offsets, int64_t n, const float* per_sample_weights,
                       float* out, void* workspace, size_t ws_bytes, void* stream,
                       uint32_t flags) {
  WsLayout W;
  // The plain forward needs only the status word and the repaired offsets,
  // but the workspace contract is the same for every entry point; after a
  // preprocess the layout must be the one the preprocess used.
  const bool pre = (flags & TBE_F_PREPROCESSED) != 0;
  tbe_status st = common_args(d, indices, offsets, n, workspace, ws_bytes,
                              pre && per_sample_weights != nullptr, &W);
  if (st != TBE_OK) return st;
  if (!weights || !out || !aligned16(weights) || !aligned16(out)) return TBE_EINVAL;
  const Launch L{d, n, static_cast<cudaStream_t>(stream), device_sms()};
  char* ws = static_cast<char*>(workspace);
  // The preprocessed path pays off when a bag holds enough lookups for its
  // hot rows to matter; shorter bags are pooled straight from the indices.
  const bool mean = (flags & TBE_F_MEAN) != 0;
  // fp32 weights are always pooled from the indices (no hot rows for them)
  if (pre && n >= static_cast<int64_t>(kHotFwdMinBagLen) * d->T * d->B &&
      d->weights_dtype != TBE_DT_F32) {
    if (mean) {
      st = from_cuda(launch_mean_factors(L, offsets, reinterpret_cast<float*>(ws + W.inv_len)));
      if (st != TBE_OK) return st;
    }
    return from_cuda(launch_forward_hot(L, W, ws, weights, per_sample_weights, out, mean));
  }
  const void* off_eff;
  int* status;
  st = run_checks(L, W, ws, offsets, flags, &off_eff, &status);
  if (st != TBE_OK) return st;
  if (!(flags & TBE_F_FORCE_GENERIC) && !mean &&
      small_table_eligible(d, n, per_sample_weights != nullptr))
    return from_cuda(launch_forward_small(L, weights, indices, off_eff, out, status,
                                          reinterpret_cast<int*>(ws + W.status)));
  return from_cuda(
      launch_forward_generic(L, weights, indices, off_eff, per_sample_weights, out, status, mean));
}

tbe_status tbe_preprocess(const tbe_desc* d, const void* indices, const void* offsets, int64_t n,
                          const float* per_sample_weights, void* workspace, size_t ws_bytes,
                          void* stream, uint32_t flags) {
  WsLayout W;
  tbe_status st = common_args(d, indices, offsets, n, workspace, ws_bytes,
                              per_sample_weights != nullptr, &W);
  if (st != TBE_OK) return st;
  const Launch L{d, n, static_cast<cudaStream_t>(stream), device_sms()};
  char* ws = static_cast<char*>(workspace);
  const void* off_eff;
  int* status;
  st = run_checks(L, W, ws, offsets, flags, &off_eff, &status);
  if (st != TBE_OK) return st;
  return from_cuda(launch_preprocess(L, W, ws, indices, off_eff, per_sample_weights,
                                     status != nullptr));
}

tbe_status tbe_backward_rowwise_adagrad(const tbe_desc* d, const float* grad_out,
                                        const void* indices, const void* offsets, int64_t n,
                                        const float* per_sample_weights, void* weights,
                                        float* momentum, float lr, float eps, void* workspace,
                                        size_t ws_bytes, void* stream, uint32_t flags) {
  WsLayout W;
  const bool mean = (flags & TBE_F_MEAN) != 0;
  tbe_status st = common_args(d, indices, offsets, n, workspace, ws_bytes,
                              per_sample_weights != nullptr, &W, mean);
  if (st != TBE_OK) return st;
  if (!grad_out || !weights || !momentum || !aligned16(grad_out) || !aligned16(weights))
    return TBE_EINVAL;
  const bool elementwise = (flags & TBE_F_ELEMENTWISE) != 0;
  if (elementwise && !aligned16(momentum)) return TBE_EINVAL;  // float4 accumulator rows
  const Launch L{d, n, static_cast<cudaStream_t>(stream), device_sms()};
  char* ws = static_cast<char*>(workspace);
  const void* off_eff = offsets;
  if (!(flags & TBE_F_PREPROCESSED)) {
    int* status;
    st = run_checks(L, W, ws, offsets, flags, &off_eff, &status);
    if (st != TBE_OK) return st;
    st = from_cuda(launch_preprocess(L, W, ws, indices, off_eff, per_sample_weights,
                                     status != nullptr));
    if (st != TBE_OK) return st;
  }
  if (mean) {
    // each bag's gradient row times its factor, as the bags' gradients
    float* inv_len = reinterpret_cast<float*>(ws + W.inv_len);
    float* scaled = reinterpret_cast<float*>(ws + W.grad_mean);
    st = from_cuda(launch_mean_factors(L, off_eff, inv_len));
    if (st != TBE_OK) return st;
    st = from_cuda(launch_scale_grad(L, grad_out, inv_len, scaled));
    if (st != TBE_OK) return st;
    grad_out = scaled;
  }
  return from_cuda(launch_update(L, W, ws, grad_out, weights, momentum, lr, eps,
                                 (flags & TBE_F_LONG_TWO_LAUNCH) != 0, elementwise));
}

tbe_status tbe_workspace_view(const tbe_desc* d, int64_t n, uint32_t ws_flags, void* workspace,
                              tbe_ws_view* view) {
  if (!view || !workspace) return TBE_EINVAL;
  tbe_status st = check_desc(d);
  if (st != TBE_OK) return st;
  st = check_n(n);
  if (st != TBE_OK) return st;
  const WsLayout W = make_layout(d, n, ws_flags);
  const char* ws = static_cast<const char*>(workspace);
  const int fin = radix_passes(d) & 1;
  view->sorted_keys = reinterpret_cast<const uint32_t*>(ws + W.keys[fin]);
  view->sorted_bags = reinterpret_cast<const uint32_t*>(ws + W.vals[fin]);
  view->sorted_psw = W.weighted ? reinterpret_cast<const float*>(ws + W.psw[fin]) : nullptr;
  view->unique_keys = reinterpret_cast<const uint32_t*>(ws + W.unique_keys);
  view->run_starts = reinterpret_cast<const uint32_t*>(ws + W.run_starts);
  view->counts = reinterpret_cast<const uint32_t*>(ws + W.counts);
  view->long_runs = reinterpret_cast<const uint32_t*>(ws + W.long_run);
  view->run_pairs = reinterpret_cast<const uint32_t*>(ws + W.run_pairs);
  view->pair_starts = reinterpret_cast<const uint32_t*>(ws + W.pair_starts);
  view->pair_bags = reinterpret_cast<const uint32_t*>(ws + W.pair_bags);
  view->hot_keys = reinterpret_cast<const uint32_t*>(ws + W.hot_keys(W.hot_next));
  view->hot_n = reinterpret_cast<const uint32_t*>(ws + W.hot_n(W.hot_next));
  view->hot_slots = kHot;
  view->long_threshold = kLongThreshold;
  view->medium_threshold = kMediumRun;
  view->chunk = kChunk;
  return TBE_OK;
}

tbe_status tbe_read_status(void* workspace, void* stream, int32_t* status_bits) {
  if (!workspace || !status_bits) return TBE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  // the workspace's side work (sort chain, hot-row gradient) may also set
  // bits: it is finished first
  cudaError_t e = cudaSuccess;
  if (SideFlow* f = find_side_flow(workspace)) e = cudaStreamSynchronize(f->side);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return TBE_ECUDA;
  *status_bits = v;
  return TBE_OK;
}

const char* tbe_version(void) { return "tbe-gb300 0.1 (sm_103a)"; }

tbe_status tbe_probe_set(uint32_t kernel) {
  if (kernel > TBE_PROBE_LAST) return TBE_EINVAL;
  std::lock_guard<std::mutex> lk(tbe::g_probe_mu);
  // events are kept for reuse; a new selection clears the record
  tbe::g_probe_used = 0;
  tbe::g_probe_open = false;
  tbe::g_probe_kernel.store(kernel, std::memory_order_relaxed);
  return TBE_OK;
}

tbe_status tbe_probe_read(uint32_t* launches, float* total_ms) {
  if (!launches || !total_ms) return TBE_EINVAL;
  std::lock_guard<std::mutex> lk(tbe::g_probe_mu);
  float sum = 0.f;
  for (int i = 0; i < tbe::g_probe_used; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(tbe::g_probe_ev[i][1]) != cudaSuccess) return TBE_ECUDA;
    if (cudaEventElapsedTime(&ms, tbe::g_probe_ev[i][0], tbe::g_probe_ev[i][1]) != cudaSuccess)
      return TBE_ECUDA;
    sum += ms;
  }
  *launches = static_cast<uint32_t>(tbe::g_probe_used);
  *total_ms = sum;
  return TBE_OK;
}

uint64_t tbe_kernel_launches(void) {
  return tbe::g_kernel_launches.load(std::memory_order_relaxed);
}

}  // extern "C"
