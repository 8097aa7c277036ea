// Backward with row-wise Adagrad for callers that cannot allocate device
// memory: the scratch lives in a fixed array inside the library instead of a
// caller-provided workspace.  The kernels are the ones tbe_backward_rowwise_
// adagrad runs; only where the scratch comes from differs.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace tbe {
namespace {

// Library-owned scratch for tbe_backward_rowwise_adagrad_noalloc.  Every GPU
// that loads the library holds this array until the process exits.  In host
// code the symbol is only a stand-in: its device address comes from
// cudaGetSymbolAddress, taken once per device in scratch_ptr().
static __device__ __align__(256) unsigned char g_noalloc_scratch[TBE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

}  // namespace
cudaError_t prepare_preprocess_kernels();
namespace {

// Set-up, per device and with that device current: the device address of
// the scratch, and the shared-memory attributes of the sort kernels.  Returns
// the scratch address on the current device, or nullptr on failure; a failed
// set-up is not remembered, so the next call on that device tries again.
char* scratch_ptr() {
  static char* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    if (prepare_preprocess_kernels() != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<char*>(p);
  }
  return ptrs[dev];
}

// Same checks as the workspace entry points, except that the workspace is the
// library's own array.
tbe_status check_args(const tbe_desc* d, const void* indices, const void* offsets, int64_t n) {
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
  if (n < 0) return TBE_EINVAL;
  if (n >= 0xfffffff0LL) return TBE_EUNSUPPORTED;
  if (!offsets || (n > 0 && !indices)) return TBE_EINVAL;
  return TBE_OK;
}

int sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
    return 148;
  return v;
}

}  // namespace
}  // namespace tbe

using namespace tbe;

extern "C" tbe_status tbe_backward_rowwise_adagrad_noalloc(
    const tbe_desc* d, const float* grad_out, const void* indices, const void* offsets, int64_t n,
    const float* per_sample_weights, void* weights, float* momentum, float lr, float eps,
    void* stream, uint32_t flags) {
  tbe_status st = check_args(d, indices, offsets, n);
  if (st != TBE_OK) return st;
  if (!grad_out || !weights || !momentum) return TBE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(grad_out) & 15u) || (reinterpret_cast<uintptr_t>(weights) & 15u))
    return TBE_EINVAL;
  if (flags & ~(TBE_F_LONG_TWO_LAUNCH | TBE_F_MEAN | TBE_F_ELEMENTWISE)) return TBE_EINVAL;
  const bool elementwise = (flags & TBE_F_ELEMENTWISE) != 0;
  if (elementwise && (reinterpret_cast<uintptr_t>(momentum) & 15u)) return TBE_EINVAL;
  const bool mean = (flags & TBE_F_MEAN) != 0;
  // The hot-row path is off here: its per-bag histograms would take most of
  // the fixed array, and without it no kernel of this call waits on
  // anything (every bounded wait of the library is in the hot-row and
  // small-table tensor-core kernels), so no call can end in a time-out.
  const WsLayout W = make_layout(d, n, (per_sample_weights ? TBE_WS_WEIGHTED : 0u) |
                                           (mean ? TBE_WS_MEAN : 0u), /*allow_hot=*/false);
  if (W.total > TBE_NOALLOC_SCRATCH_BYTES) return TBE_ETOO_LARGE;
  char* scratch = scratch_ptr();
  if (!scratch) return TBE_ECUDA;
  const Launch L{d, n, static_cast<cudaStream_t>(stream), sm_count()};
  // Each call stands alone: the hot-row set is cleared (the path is off, so
  // nothing reads it, but no stale set is kept), and everything else the
  // kernels read before writing is reset by launch_preprocess (counters,
  // first run and pair entries, band counts); the status word is not used
  // because bounds reporting is not offered here.
  if (cudaMemsetAsync(scratch + W.hot_n(W.hot_next), 0, static_cast<size_t>(d->T) * sizeof(uint32_t),
                      L.s) != cudaSuccess)
    return TBE_ECUDA;
  cudaError_t e = launch_preprocess(L, W, scratch, indices, offsets, per_sample_weights, false);
  if (e != cudaSuccess) return TBE_ECUDA;
  if (mean) {
    float* inv_len = reinterpret_cast<float*>(scratch + W.inv_len);
    float* scaled = reinterpret_cast<float*>(scratch + W.grad_mean);
    e = launch_mean_factors(L, offsets, inv_len);
    if (e != cudaSuccess) return TBE_ECUDA;
    e = launch_scale_grad(L, grad_out, inv_len, scaled);
    if (e != cudaSuccess) return TBE_ECUDA;
    grad_out = scaled;
  }
  e = launch_update(L, W, scratch, grad_out, weights, momentum, lr, eps,
                    (flags & TBE_F_LONG_TWO_LAUNCH) != 0, elementwise);
  return e == cudaSuccess ? TBE_OK : TBE_ECUDA;
}
