// Host-side interfaces between the translation units of the TBE library.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "tbe.h"

namespace tbe {

struct WsLayout;

// Counts one kernel launch (read back by tbe_kernel_launches).
void note_launch();

// Kernel probe (tbe_probe_set): events around launches of the selected kernel.
void probe_begin(uint32_t kernel, cudaStream_t s);
void probe_end(uint32_t kernel, cudaStream_t s);

// An event of the flow and the stream capture its latest record was made
// in (0: none).  A record made while a stream is captured into a CUDA graph
// is a dependency inside that graph, not a point in any stream: only the
// same capture may wait on it, and a capture may wait on no record made
// outside it.
struct FlowEvent {
  cudaEvent_t ev = nullptr;
  unsigned long long capture = 0;
};

// Side stream of one workspace (one per workspace and device, created at the
// workspace's first use): the preprocess runs its sort chain there,
// concurrently with the forward, and the backward its hot-row gradient,
// concurrently with the cold rows.  Events join the streams:
//   sorted  recorded on the side stream after the sort chain,
//   hot     recorded on it after the hot-row update,
//   done    recorded after every side segment (the latest side work),
//   fork    recorded on the caller's stream before a side segment.
// Because the flow belongs to the workspace, calls on different workspaces
// (other streams, other host threads) never wait on each other's events.
struct SideFlow {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr;
  FlowEvent sorted, hot, done;
};
// The flow of workspace `ws` on the current device, created on first use;
// nullptr if the stream or events could not be created (the next call
// tries again).
SideFlow* side_flow(const void* ws);
// The flow of `ws` if one exists, else nullptr (creates nothing).
SideFlow* find_side_flow(const void* ws);
// Makes `side` wait for everything enqueued on `s` so far.
cudaError_t fork_to(SideFlow* f, cudaStream_t s);
// Records e on s, noting the capture s is in.
cudaError_t flow_record(FlowEvent& e, cudaStream_t s);
// Makes s wait for e's latest record when both belong to the same capture
// (or to none); otherwise the wait is left out: a record made inside a
// graph is ordered by that graph's replays on the caller's stream, and one
// made before a capture by the synchronisation that precedes it.
cudaError_t flow_wait(cudaStream_t s, const FlowEvent& e);

// One call's launch context.
struct Launch {
  const tbe_desc* d;
  int64_t n;           // lookups
  cudaStream_t s;
  int num_sms;
};

// forward.cu
cudaError_t launch_forward_generic(const Launch& L, const void* weights, const void* indices,
                                   const void* offsets, const float* psw, float* out,
                                   int* status, bool mean);
// The generic kernel over tbe_preprocess's per-bag cold lists (linear keys);
// with hot_n, bags of tables with hot rows are added to out; with inv_len
// (mean pooling) every bag's result is scaled by its factor.
cudaError_t launch_forward_cold(const Launch& L, const void* weights, const uint32_t* cold_keys,
                                const uint32_t* cold_off, const float* cold_psw, float* out,
                                const uint32_t* hot_n, const float* inv_len);
// Mean pooling's per-bag factors (1/L for L > 1 lookups, else 1) into inv_len.
cudaError_t launch_mean_factors(const Launch& L, const void* offsets, float* inv_len);
cudaError_t launch_check_offsets(const Launch& L, const void* offsets, bool repair, void* fixed,
                                 int64_t* scratch, int* status);
int64_t repair_scratch_blocks(int64_t nb1);

// forward_small.cu: tensor-core histogram path for one small table.
bool small_table_eligible(const tbe_desc* d, int64_t n, bool weighted);
cudaError_t launch_forward_small(const Launch& L, const void* weights, const void* indices,
                                 const void* offsets, float* out, int* status, int* error_word);

// forward_hot.cu: forward from tbe_preprocess's results (hot rows on the
// tensor cores, cold lookups gathered).
cudaError_t launch_forward_hot(const Launch& L, const WsLayout& W, char* ws, const void* weights,
                               const float* psw, float* out, bool mean);

// preprocess.cu: expand, radix sort, run-length encode, classify.
cudaError_t launch_preprocess(const Launch& L, const WsLayout& W, char* ws, const void* indices,
                              const void* offsets, const float* psw, bool check);
// Sorted arrays end up in buffer (passes % 2); the layout needs to know which.
int radix_passes(const tbe_desc* d);

// hot_grad.cu: partial gradients of the hot rows (tensor cores).
cudaError_t launch_hot_grad(const Launch& L, const WsLayout& W, char* ws, const float* grad_out);

// update.cu: short-run and long-run row-wise Adagrad.
cudaError_t launch_update(const Launch& L, const WsLayout& W, char* ws, const float* grad_out,
                          void* weights, float* momentum, float lr, float eps, bool two_launch,
                          bool elementwise = false);
// The next call's hot set, chosen from this call's cold runs and hot-row
// counts (after the sort chain), written to the workspace's second set.
cudaError_t launch_hot_refresh(const Launch& L, const WsLayout& W, char* ws);
// Where the refresh runs: 0, at the end of the backward on the caller's
// stream; 1, at the end of the preprocess's sort chain on the side stream
// (beside the forward).
#ifndef TBE_REFRESH_IN_PREPROCESS
#define TBE_REFRESH_IN_PREPROCESS 1
#endif
// Mean pooling's backward input: out[b, D_off[t] + c] = grad_out[b, D_off[t] + c]
// times bag (t, b)'s factor from inv_len.
cudaError_t launch_scale_grad(const Launch& L, const float* grad_out, const float* inv_len,
                              float* out);

}  // namespace tbe
