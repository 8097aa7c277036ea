/*
 * tbe.h -- C ABI of the GB300 (sm_103a) Table Batched Embedding library.
 *
 * Table Batched Embedding (TBE) pools lookups from many embedding tables in
 * one launch and trains them with a backward that regroups lookups by row and
 * applies exactly one Adagrad update (row-wise, or element-wise) per touched
 * row.
 *
 * Sources (page titles and sections):
 *  - "Modernizing Table Batched Embeddings with FBTriton", sections
 *    "Why redesign a sparse operator?" (what TBE combines), "Forward: keep a
 *    narrowly specialized path beside the general one" (generic gather-pool,
 *    fp32 accumulation of fp16/bf16 weights, int32 index option, small-table
 *    histogram path and its eligibility, bounds checks off by default),
 *    "Backward: invert 'which rows did this sample use?'" (transpose, sort,
 *    run-length encoding into runs, short/long runs, fenced last-chunk
 *    update), "Fewer reads and synchronizations can beat more parallel work"
 *    (device-resident counts, no read-back), "Fusion boundaries are also
 *    engineering interfaces" (per-sample weights scale each contribution
 *    before grouping; the optimizer is the backward's epilogue).
 *  - "HugeCTR DistributedSlotSparseEmbeddingHash backward" (eqicode.com):
 *    CSR bags (row_offset / value), the sample-id expansion, radix sort by
 *    row with end_bit, run flags + prefix sum + run starts with a sentinel,
 *    and the Adagrad accumulator-then-weight order with eps outside the root
 *    (one accumulator per element there; row-wise here by default), and the
 *    sum/mean combiners with the mean backward's 1/L scaling.
 *
 * Data layout (all device buffers are owned by the caller):
 *  - T tables; table t has E_t rows of width D_t (D_t a multiple of 8, at
 *    most 1024).  Weights are fp16, bf16 or fp32 (weights_dtype), one flat
 *    buffer; table t starts at element weights_offsets[t], its rows are
 *    contiguous with stride D_t.
 *  - Momentum: fp32 [sum E_t], one value per row, row r of table t at
 *    hash_base[t] + r; with TBE_F_ELEMENTWISE fp32 [weights_offsets[T]], one
 *    value per weight element at the element's own position.
 *  - Bags are table-major: bag (t,b) has id t*B+b.  offsets: [T*B+1] of the
 *    index type, indices: [n], lookups of bag (t,b) at positions
 *    offsets[t*B+b] .. offsets[t*B+b+1]-1.  A lookup's row must lie in
 *    [0, E_t); any other value is skipped (contributes nothing), whether or
 *    not checks are enabled.
 *  - Pooled output and its gradient: fp32 row-major [B, sum D_t]; table t's
 *    pooled vector for bag b is at columns D_offsets[t] .. D_offsets[t+1]-1.
 *  - Optional per-sample weights: fp32 [n].
 *
 * Ordering and synchronisation: every call only enqueues work on the given
 * stream (a cudaStream_t passed as void*; NULL = legacy default stream) and
 * returns.  No call allocates device memory and no call on the hot path
 * synchronises with the host; tbe_read_status is the one explicit sync.
 *
 * Errors: argument problems are reported synchronously through tbe_status
 * before anything is enqueued.  Data problems found on the device (indices
 * out of range, malformed offsets) set bits in a status word that lives in
 * the workspace; tbe_read_status copies it to the host.  Without
 * TBE_F_REPAIR_OFFSETS, malformed offsets give unspecified results but every
 * kernel stays inside its buffers: each bag is read over its own offsets
 * clamped into [0, n] (bags may then overlap), and the backward keeps at
 * most n of the lookups such bags name.
 */
#ifndef TBE_H_
#define TBE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tbe_status {
  TBE_OK = 0,
  TBE_EINVAL = 1,       /* null pointer, negative size, dtype mismatch */
  TBE_EWORKSPACE = 2,   /* workspace null or smaller than tbe_workspace_size */
  TBE_EUNSUPPORTED = 3, /* well-formed but outside what the kernels cover */
  TBE_ECUDA = 4,        /* a CUDA call or launch returned an error */
  TBE_ETOO_LARGE = 5    /* the problem needs more scratch than the fixed array of
                           tbe_backward_rowwise_adagrad_noalloc holds */
} tbe_status;

/* element types */
enum { TBE_DT_F16 = 1, TBE_DT_I32 = 2, TBE_DT_I64 = 3, TBE_DT_BF16 = 4, TBE_DT_F32 = 5 };

/* call flags */
#define TBE_F_CHECK_BOUNDS (1u << 0)    /* validate offsets (separate kernel) and indices,
                                           report problems in the status word */
#define TBE_F_REPAIR_OFFSETS (1u << 1)  /* also repair offsets into a workspace copy:
                                           o'[0]=0, o'[i]=max(o'[i-1], clamp(o[i],0,n)) */
#define TBE_F_FORCE_GENERIC (1u << 2)   /* forward: never take the small-table path */
#define TBE_F_LONG_TWO_LAUNCH (1u << 3) /* backward: long runs write partial sums and a
                                           second kernel applies the update (instead of
                                           the fenced last-arriver update) */
#define TBE_F_PREPROCESSED (1u << 4)    /* forward and backward: the workspace already
                                           holds tbe_preprocess's results for these
                                           indices/offsets/per-sample weights (same
                                           stream); see tbe_forward for when the
                                           forward still reads the indices */
#define TBE_F_MEAN (1u << 5)            /* forward and backward: mean pooling (the HugeCTR
                                           page's mean combiner): a bag of L > 1 lookups
                                           (L by the offsets, rows out of range included)
                                           pools to its sum times 1/L, and its gradient
                                           row is scaled by 1/L before the regrouping
                                           (into the workspace: the backward needs one
                                           sized with TBE_WS_MEAN); bags of 0 or 1
                                           lookups are not scaled.  The small-table path
                                           is not taken. */
#define TBE_F_ELEMENTWISE (1u << 6)     /* backward: element-wise Adagrad (the HugeCTR
                                           page's Adagrad kernel, one accumulator per
                                           weight element): momentum is fp32 laid out
                                           like the weights (weights_offsets[T]
                                           entries, 16-byte aligned), and every element
                                           takes m_c <- m_c + g_c^2 and
                                           W[r, c] <- rn(W[r, c] - lr * g_c /
                                           (sqrt(m_c) + eps)).  The rows, runs, hot
                                           rows and summation are as in the row-wise
                                           update. */

/* workspace-size flags */
#define TBE_WS_WEIGHTED (1u << 0)       /* reserve room for per-sample weights */
#define TBE_WS_MEAN (1u << 1)           /* reserve room for the mean-scaled gradient
                                           (B x total_D floats, at the end of the
                                           layout): needed by a backward with
                                           TBE_F_MEAN */

/* device status bits (tbe_read_status) */
#define TBE_ERR_INDEX_RANGE (1 << 0)    /* a lookup's row was outside [0, E_t) */
#define TBE_ERR_OFFSETS (1 << 1)        /* offsets not 0 = o[0] <= ... <= o[T*B] <= n */
#define TBE_ERR_TIMEOUT (1 << 2)        /* a bounded device wait gave up: the call's results
                                           are incomplete (reported whatever the flags) */

/* Problem description.  The three int64 arrays are device pointers with T+1
 * entries each (cumulative sums starting at 0); the scalar totals are their
 * last entries, repeated here so that the host never reads device memory. */
typedef struct tbe_desc {
  int32_t T;                        /* number of tables, >= 1 */
  int32_t B;                        /* bags per table (batch size), >= 1 */
  int32_t weights_dtype;            /* TBE_DT_F16, TBE_DT_BF16 (accumulated in fp32
                                       like fp16; hot rows with bf16 tensor-core
                                       operands) or TBE_DT_F32 (the forward accumulates
                                       each output as a compensated two-float sum: as
                                       accurate as an fp64 accumulation rounded once to
                                       fp32, see tbe_forward).  The small-table path
                                       takes fp16 only, and fp32 tables take no hot
                                       rows: they take the gather paths there */
  int32_t index_dtype;              /* TBE_DT_I32 or TBE_DT_I64; offsets use it too */
  const int64_t* D_offsets;         /* device [T+1]: sum of D_t' for t' < t */
  const int64_t* hash_base;         /* device [T+1]: sum of E_t' for t' < t */
  const int64_t* weights_offsets;   /* device [T+1]: sum of E_t' * D_t' for t' < t */
  int64_t total_D;                  /* D_offsets[T] */
  int64_t total_E;                  /* hash_base[T]; must be < 2^32 - 1 */
  int32_t max_D;                    /* max_t D_t */
  int32_t min_D;                    /* min_t D_t */
} tbe_desc;

/* Device pointers into a workspace after tbe_preprocess, for inspection.
 * Counts marked (device) live in device memory and are never read back by the
 * library.  A run is the set of sorted lookups of one (table,row); inside a
 * run, a pair is the set of its lookups that come from one bag (they share
 * one gradient row, so the update gathers it once and scales it by the
 * pair's multiplicity or, with per-sample weights, by their sum). */
typedef struct tbe_ws_view {
  const uint32_t* sorted_keys;  /* [n] linear keys hash_base[t]+row, ascending; invalid
                                   lookups carry key total_E and sort last */
  const uint32_t* sorted_bags;  /* [n] bag b (within its table) of each sorted lookup;
                                   ascending within a run (the sort is stable) */
  const float* sorted_psw;      /* [n] per-sample weight of each sorted lookup, or NULL */
  const uint32_t* unique_keys;  /* [R] key of each run */
  const uint32_t* run_starts;   /* [R+1] first sorted position of each run; [R] = n_valid */
  const uint32_t* counts;       /* (device) [0] R runs, [1] n_valid lookups, [2] long runs,
                                   [3] long-run chunks, [6] P pairs */
  const uint32_t* long_runs;    /* [counts[2]] run id of each long run, in no set order */
  int32_t long_threshold;       /* pairs from which a run takes the chunked path */
  int32_t chunk;                /* pairs per chunk on the chunked path */
  const uint32_t* run_pairs;    /* [R+1] first pair of each run; [R] = P */
  const uint32_t* pair_starts;  /* [P+1] first sorted position of each pair; [P] = n_valid */
  const uint32_t* pair_bags;    /* [P] bag of each pair */
  const uint32_t* hot_keys;     /* [T][hot_slots] hot rows of each table (linear keys, the
                                   most looked-up first) */
  const uint32_t* hot_n;        /* [T] hot rows per table */
  int32_t hot_slots;            /* hot rows a table can have */
  int32_t medium_threshold;     /* pairs from which a run below long_threshold is updated
                                   by a whole warp (fewer pairs: several runs per warp) */
} tbe_ws_view;

/* Bytes of workspace needed for calls with at most n_max lookups.
 * ws_flags: TBE_WS_WEIGHTED if per-sample weights will be passed.
 * The caller allocates the workspace (16-byte aligned) and zero-fills it once
 * before its first use; the library keeps the status word at its start and
 * overwrites everything else on every call that needs it.
 * Errors: TBE_EINVAL (null desc/bytes, n_max < 0), TBE_EUNSUPPORTED
 * (n_max >= 2^32 or total_E >= 2^32 - 1). */
tbe_status tbe_workspace_size(const tbe_desc* d, int64_t n_max, uint32_t ws_flags,
                              size_t* bytes);

/* Pooled forward ("Forward: keep a narrowly specialized path beside the
 * general one"):
 *   out[b, D_offsets[t] + c] = sum over lookups i of bag (t,b) with a valid row
 *                              of psw_i * W_t[indices[i], c]   (psw_i = 1 if NULL)
 * accumulated in fp32 for 16-bit weights.  fp32 weights are accumulated as
 * an unevaluated sum hi + lo of two fp32 values (each addition an exact
 * two-sum, each weighted product exact through a fused multiply-add), rounded
 * once at the end; its error is the final rounding plus at most about
 * 4 n^2 2^-48 of the sum of |terms| for a bag of n lookups (about 1e-9 of
 * it at n = 200), as with the fp64 accumulation the pages name for fp32
 * weights.  An empty bag yields zeros.  One table with E <= 64,
 * 64 <= D <= 128, no per-sample weights and an average bag length >= 64 takes
 * the tensor-core histogram path (counts per bag times the table) unless
 * TBE_F_FORCE_GENERIC; every other problem takes the generic gather-pool.
 * With TBE_F_PREPROCESSED and bags of at least 64 lookups on average
 * (n >= 64 T B; shorter bags are pooled from the indices as without the
 * flag) the forward reads tbe_preprocess's results instead of the indices:
 * each table's hot rows are pooled as the per-bag histogram
 * times those rows on the tensor cores (fp16 MMAs: counts up to 255 are exact
 * fp16 values, larger or weighted counts are scaled per bag and split exactly
 * into three fp16 parts, so only the fp32 accumulation rounds; bf16 weights
 * take bf16 operands the same way: counts up to 255 are exact bf16 values and
 * three bf16 parts hold any fp32 value), the cold lookups are gathered from
 * the per-bag cold lists; the bounds/offsets flags are then ignored (the preprocess
 * checked them) and per_sample_weights must be NULL exactly when it was NULL
 * for the preprocess.  fp32 weights are always pooled from the indices, as
 * without the flag.
 * weights: device, weights_dtype; indices/offsets: device, index_dtype; n: lookups
 * (length of indices); per_sample_weights: fp32 device [n] or NULL;
 * out: fp32 device [B, total_D], fully overwritten.  Workspace: the status
 * word plus (TBE_F_REPAIR_OFFSETS) the repaired offsets; ws_bytes must be at
 * least tbe_workspace_size(d, n, ...).
 * Errors: TBE_EINVAL, TBE_EWORKSPACE, TBE_EUNSUPPORTED (dtype, D_t), TBE_ECUDA. */
tbe_status tbe_forward(const tbe_desc* d, const void* weights, const void* indices,
                       const void* offsets, int64_t n, const float* per_sample_weights,
                       float* out, void* workspace, size_t ws_bytes, void* stream,
                       uint32_t flags);

/* Backward preprocessing only ("Backward: invert ..." and the HugeCTR steps
 * 1-4): expand every lookup to (key = hash_base[t] + row, bag b, psw), radix
 * sort by key (stable, int32 keys), run-length encode into runs, and classify
 * runs into short and long with the long-run task list compacted on the
 * device.  Hot rows: the workspace keeps, per table, up to hot_slots rows
 * chosen by the previous backward on it (none at first); lookups of those
 * rows are not sorted but summed per bag into a histogram (counts, stored as
 * bytes for every 128-bag tile whose counts all fit one; otherwise, and for
 * sums of per-sample weights, fp32 with a per-bag power-of-two scale), and
 * the remaining (cold) lookups are also kept per bag in lookup order.  After
 * the sort the call chooses the next hot set from this batch: per table, the
 * most looked-up rows with at least max(B/64, 32) lookups (tables with D_t <=
 * 256 only, and only while the histograms, T * hot_slots * B * 5 bytes, stay
 * within 2 GiB; fp32 tables have none); the next preprocess on this
 * workspace takes it.  Results stay in the workspace (see tbe_workspace_view); a
 * later tbe_forward or tbe_backward_rowwise_adagrad with TBE_F_PREPROCESSED
 * consumes them.  The sort chain runs on a stream the library keeps for this
 * workspace (created at the workspace's first use, one per workspace and
 * device), so that a forward enqueued next runs concurrently with it; the
 * library's calls on this workspace order themselves against it (through
 * events), calls on other workspaces never wait on it, and reading the
 * sorted arrays directly needs a device synchronisation first.  Every
 * tbe_backward_rowwise_adagrad joins the workspace's side-stream work into
 * its stream before it returns, so whole training steps (preprocess,
 * forward, backward) can be captured into a CUDA graph and replayed; a
 * capture must end with a backward (a preprocess alone leaves its sort chain
 * unjoined), and the first call on a workspace, which creates its stream,
 * must come before any capture.
 * Errors as tbe_forward. */
tbe_status tbe_preprocess(const tbe_desc* d, const void* indices, const void* offsets, int64_t n,
                          const float* per_sample_weights, void* workspace, size_t ws_bytes,
                          void* stream, uint32_t flags);

/* Backward with exact row-wise Adagrad ("Backward: invert ...", "Fusion
 * boundaries ...", the HugeCTR Adagrad kernel in row-wise form).  For every
 * touched row r of table t, with the run of its lookups i:
 *   g_c   = sum_i psw_i * grad_out[b_i, D_offsets[t] + c]        (fp32)
 *   m_r  <- m_r + (1/D_t) * sum_c g_c^2
 *   W_t[r, c] <- fp16_rn(W_t[r, c] - lr * g_c / (sqrt(m_r) + eps))
 * exactly once per touched row; untouched rows are not written (fp16_rn is
 * bf16_rn for TBE_DT_BF16 weights, and the fp32 rounding of the step formed
 * in fp32 for TBE_DT_F32; TBE_F_ELEMENTWISE replaces the row accumulator by
 * one per element, see the flag).
 * grad_out: fp32 device [B, total_D]; weights (weights_dtype) and momentum (fp32
 * [total_E], or [weights_offsets[T]] with TBE_F_ELEMENTWISE) are updated in
 * place.  Without TBE_F_PREPROCESSED the call runs
 * tbe_preprocess first.  The gradient of a hot row (see tbe_preprocess) is
 * its histogram column times grad_out, summed over bag partitions in a fixed
 * order; every other row's gradient is summed over its sorted run.  Both are
 * fp32 sums whose rounding order differs, so a row's result can differ in the
 * last bits between a call where it is hot and one where it is cold (the hot
 * set comes from the previous preprocess on this workspace; see
 * tbe_preprocess).  No host synchronisation, no device-to-host copy.  Errors
 * as tbe_forward. */
tbe_status tbe_backward_rowwise_adagrad(const tbe_desc* d, const float* grad_out,
                                        const void* indices, const void* offsets, int64_t n,
                                        const float* per_sample_weights, void* weights,
                                        float* momentum, float lr, float eps, void* workspace,
                                        size_t ws_bytes, void* stream, uint32_t flags);

/* Fill *view with device pointers into a workspace sized for n lookups.
 * Errors: TBE_EINVAL. */
tbe_status tbe_workspace_view(const tbe_desc* d, int64_t n, uint32_t ws_flags, void* workspace,
                              tbe_ws_view* view);

/* Copy the device status word to *status_bits (a TBE_ERR_* mask) and clear it.
 * Synchronises the stream and the workspace's own side stream (see
 * tbe_preprocess): never call it inside a timed or captured region.
 * Errors: TBE_EINVAL, TBE_ECUDA. */
tbe_status tbe_read_status(void* workspace, void* stream, int32_t* status_bits);

/* Size of the library-owned scratch used by tbe_backward_rowwise_adagrad_noalloc. */
#define TBE_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Backward with exact row-wise Adagrad that allocates nothing, not even a
 * caller-provided workspace.  The pages have no counterpart: this entry point
 * exists for callers that must not allocate device memory when they call the
 * backward -- runtimes that hand out all device memory up front from their
 * own pools (a serving engine or a training loop with a static memory plan),
 * and code that cannot afford cudaMalloc/cudaFree, which may synchronise the
 * whole device and fragment such a plan.
 *
 * It computes what tbe_backward_rowwise_adagrad computes on a fresh
 * workspace, with the same sort and run kernels, but its scratch is a fixed
 * array of TBE_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library, held by
 * every GPU that loads the library until the process exits.  The hot-row
 * path is off here (its histograms would fill most of the array), so every
 * touched row is updated from its sorted run, and no kernel of this call
 * waits on anything: no call can end in a time-out.  Problems whose scratch
 * would be larger -- about 366k lookups of 128-wide rows (321k with
 * per-sample weights, 249k for 256-wide rows) -- are rejected with
 * TBE_ETOO_LARGE before anything is enqueued.  No cudaMalloc, cudaFree or
 * other allocating call is made.
 *
 * The first call on each device does the set-up (looks up the device address
 * of the array; a set-up that fails is tried again by the next call); make
 * that first call before any stream capture.  Every call shares the one
 * array and it keeps the previous call's contents; everything that must
 * start at zero is cleared by the call itself, so each call stands alone.
 * Calls whose work overlaps on the GPU (different streams, or several host
 * threads) race on the array: serialise them.
 *
 * Arguments as tbe_backward_rowwise_adagrad without workspace; flags may hold
 * TBE_F_LONG_TWO_LAUNCH, TBE_F_MEAN and TBE_F_ELEMENTWISE (no bounds reporting: the status word
 * lives in the caller's workspace elsewhere; invalid rows are still skipped).
 * Errors: TBE_EINVAL, TBE_EUNSUPPORTED, TBE_ETOO_LARGE, TBE_ECUDA. */
tbe_status tbe_backward_rowwise_adagrad_noalloc(const tbe_desc* d, const float* grad_out,
                                                const void* indices, const void* offsets,
                                                int64_t n, const float* per_sample_weights,
                                                void* weights, float* momentum, float lr,
                                                float eps, void* stream, uint32_t flags);

/* Library build identification: a static string. */
const char* tbe_version(void);

/* Number of CUDA kernels this library has launched in this process, over all
 * entry points, devices and threads (a relaxed atomic counter, never reset).
 * Memsets are not counted.  A measurement aid with no counterpart in the
 * method: the difference of two readings is the kernel count of the calls
 * made between them. */
uint64_t tbe_kernel_launches(void);

/* Kernel probe, a measurement aid with no counterpart in the method: times
 * every launch of one of the library's kernels with a pair of CUDA events
 * recorded on the launch's stream around it.
 * tbe_probe_set(kernel) selects the kernel (one of TBE_PROBE_*, or
 * TBE_PROBE_OFF) and clears the record; up to 256 launches are recorded
 * after that, later ones are not.  The events are created by the library
 * on the current device.  tbe_probe_read waits for the recorded events and
 * returns the number of recorded launches and their summed duration in
 * milliseconds.  Both are host calls for use outside timed work; probing
 * adds two event records per probed launch and nothing else.
 * Errors: TBE_EINVAL (unknown kernel, NULL pointers), TBE_ECUDA. */
#define TBE_PROBE_OFF 0u
#define TBE_PROBE_EXPAND_COUNT 1u
#define TBE_PROBE_RADIX_DOWNSWEEP 2u
#define TBE_PROBE_FORWARD_HOT 3u
#define TBE_PROBE_FORWARD_COLD 4u
#define TBE_PROBE_SHORT_RUNS 5u
#define TBE_PROBE_MEDIUM_RUNS 6u
#define TBE_PROBE_LONG_CHUNKS 7u
#define TBE_PROBE_HOT_GRAD 8u
#define TBE_PROBE_LAST 8u
tbe_status tbe_probe_set(uint32_t kernel);
tbe_status tbe_probe_read(uint32_t* launches, float* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* TBE_H_ */
