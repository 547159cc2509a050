/*
 * lp.h - C ABI of the deterministic linear-logp operator for GB300 (sm_103a).
 *
 * What the operator computes (page "feat(rl-kernel): add CUDA linear logp
 * provider integration", Motivation and Changes / Megatron integration): from
 * output-layer hidden states X[T,H], the local LM-head projection weight W and
 * bias b of each tensor-parallel vocabulary shard, the real/padded vocabulary
 * sizes and target ids y[T], it returns selected-token log probabilities and
 * optional entropy of softmax(z), z = (X W^T + b) / tau, without materialising
 * the logits. Temperature is applied exactly once (page "feat(rl-kernel): add
 * ROCm linear logp provider integration", Changes). Shards are reduced in rank
 * order and an empty shard gives zero probabilities, LSE = -inf, target logit 0
 * and logp = -inf, never NaN (page "Perf/cuda compact top p replay", Summary
 * and Walkthrough).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory. Scratch comes from the caller through
 *    `workspace`, sized by lp_workspace_size(). Host-side structs
 *    (lp_vocab_partition, lp_outputs, the shard range array and the arrays of
 *    per-shard pointers) are read during the call only.
 *  - bf16 tensors are row-major; rows of X, W and logits must start on a
 *    16-byte boundary (pointer % 16 == 0 and row stride % 8 elements == 0).
 *  - Vocabulary ids are GLOBAL ids. A partition lists n_shards (1..LP_MAX_SHARDS)
 *    contiguous ranges in ascending order that tile [0, vocab_padded) exactly, or,
 *    in a rank-local partition (local = 1), only this tensor-parallel rank's range
 *    [shards[0].vocab_start, shards[n_shards-1].vocab_end); ids in
 *    [vocab_real, vocab_padded) are padding and excluded from the softmax. A shard
 *    may be empty (vocab_start == vocab_end).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronises, except lp_get_device_error().
 *  - T = 0 (an empty batch) succeeds without work and without reading any tensor
 *    pointer; lp_backward then still writes zeros into dW and db.
 *  - Results are bitwise deterministic run to run and batch invariant: a row's
 *    outputs depend only on that row's inputs, never on T or on the row's
 *    position. Reductions over the vocabulary follow a fixed order that
 *    depends only on the partition and compile-time tile sizes.
 *  - Host-side validation errors are returned before anything is launched.
 *    Errors found on the device (a target or replay id out of range, a
 *    pipeline wait that timed out, a failed bounds check of a bounds-checked
 *    build) are recorded in a sticky per-device error word read by
 *    lp_get_device_error(); the affected rows get logp = -inf.
 *  - A call made while the current device is not sm_100-family (GB300 is
 *    sm_103) returns LP_ERR_UNSUPPORTED_DEVICE. There is no CPU fallback.
 */
#ifndef LP_H_
#define LP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LP_MAX_SHARDS 8     /* shards per call */
#define LP_REPLAY_SLOTS 64  /* replay id slots per row */
#define LP_NOALLOC_SCRATCH_BYTES (32u << 20) /* scratch of lp_forward_noalloc, per device */

#if defined(__GNUC__)
#define LP_API __attribute__((visibility("default")))
#else
#define LP_API
#endif

typedef struct CUstream_st* lp_stream_t; /* identical to cudaStream_t */

typedef enum {
  LP_OK = 0,
  LP_ERR_INVALID_ARG = 1,          /* null pointer, bad size, bad partition, tau not finite or <= 0 */
  LP_ERR_ALIGNMENT = 2,            /* a pointer or row stride breaks the 16-byte rule */
  LP_ERR_UNSUPPORTED_DEVICE = 3,   /* current device is not sm_100 family, or no device */
  LP_ERR_WORKSPACE_TOO_SMALL = 4,  /* ws_bytes < lp_workspace_size(...) */
  LP_ERR_TARGET_OUT_OF_RANGE = 5,  /* device: some y not in [0, vocab_real) */
  LP_ERR_REPLAY_ID_OUT_OF_RANGE = 6, /* device: a replay id not in {-1} U [0, vocab_real) */
  LP_ERR_DEVICE_TIMEOUT = 7,       /* device: a pipeline wait ran past its limit */
  LP_ERR_CUDA = 8,                 /* a CUDA runtime call failed */
  LP_ERR_REPLAY_TOO_MANY_IDS = 9,  /* device: a keep-mask row kept more than 64 ids (row fails closed) */
  LP_ERR_BOUNDS = 10               /* device, bounds-checked builds only: an index failed its check and
                                      the access was skipped (see lp_debug_bounds_build) */
} lp_status;

typedef enum {
  LP_OP_FORWARD = 0,
  LP_OP_FORWARD_FROM_LOGITS = 1,
  LP_OP_TOP_P_REPLAY = 2,
  LP_OP_BACKWARD = 3,
  LP_OP_TOP_P_REPLAY_DENSE_MASK = 4,
  LP_OP_BACKWARD_FROM_LOGITS = 5,  /* needs no workspace */
  LP_OP_FORWARD_HOST = 6
} lp_op;

/* Element type of an output buffer whose type the caller chooses. */
typedef enum {
  LP_DTYPE_F32 = 0,
  LP_DTYPE_BF16 = 1   /* the fp32 result rounded to nearest, ties to even */
} lp_dtype;

/* Global id range [vocab_start, vocab_end) of one shard. */
typedef struct {
  int64_t vocab_start;
  int64_t vocab_end;
} lp_shard_range;

/* Tensor-parallel vocabulary partition: the real and padded vocabulary sizes and
 * the shards in rank order (page "feat(rl-kernel): add CUDA linear logp provider
 * integration", Changes / Megatron integration: the provider is given the
 * tensor-parallel vocabulary range, and tensor parallelism is the vocabulary
 * reduction group). `shards` is a host array.
 *   local = 0  the shards tile [0, vocab_padded): every id of the vocabulary is here;
 *   local = 1  the shards tile only this rank's range [lo, hi) =
 *              [shards[0].vocab_start, shards[n_shards-1].vocab_end) within
 *              [0, vocab_padded). Every entry point then works on those ids alone:
 *              LSE and entropy are over the rank's real ids; a target outside [lo, hi)
 *              is another rank's (logp = -inf here, no error; a target outside
 *              [0, vocab_real) is still a device error); replay ids of other ranks are
 *              skipped; the backward takes the merged LSE and entropy and returns this
 *              rank's share of dX. The per-shard statistics (lp_outputs.shard_stats)
 *              are what the ranks exchange, merged by lp_merge_shard_stats.
 * A C caller that initialises the first four members leaves local = 0. */
typedef struct {
  int64_t vocab_real;
  int64_t vocab_padded;
  int32_t n_shards;
  const lp_shard_range* shards;
  int32_t local;
} lp_vocab_partition;

/* Per-row outputs, fp32 device arrays of length T.
 *   logp        z[y] - LSE (or -inf: target outside the support or device error)
 *   lse         log sum over the support of exp z (-inf when the support is empty)
 *   entropy     LSE - sum p z in nats; may be NULL; must be NULL for replay
 *   shard_stats optional [n_shards][3][T]: what each shard contributes to the
 *               rank-ordered reduction - its local LSE, its target logit (z[y] if y
 *               lies in the shard, else 0) and its own entropy
 *               -sum_{v in shard} p_v log p_v with p = softmax over the shard's ids
 *               (0 for replay). An empty shard reports (-inf, 0, 0). In replay, a
 *               target inside a shard that keeps other ids but not y is an excluded
 *               id: that shard's target logit is -inf. */
typedef struct {
  float* logp;
  float* lse;
  float* entropy;
  float* shard_stats;
} lp_outputs;

/* Bytes of device scratch the operation needs for these sizes (0 for none).
 * Returns 0 and is harmless for invalid arguments (the call itself reports them). */
LP_API size_t lp_workspace_size(lp_op op, int64_t T, int64_t H, const lp_vocab_partition* part);

/* Fused linear-logp forward (page "feat(rl-kernel): add CUDA linear logp provider
 * integration", Changes): logp, LSE and optional entropy of softmax((X W^T + b)/tau)
 * over the real vocabulary, computed by a tcgen05 GEMM whose epilogue folds each
 * vocabulary tile into per-row running statistics; logits never reach memory.
 *   X     bf16 [T, H], row-major, H % 8 == 0
 *   W     host array [n_shards] of device pointers, shard k bf16 [V_k, H] row-major
 *         (NULL allowed for an empty shard)
 *   bias  NULL, or host array [n_shards] of device pointers to bf16 [V_k] (entries may be NULL)
 *   y     int32 [T] global target ids in [0, vocab_real)
 *   tau   temperature, finite and > 0 */
LP_API lp_status lp_forward(const void* X, int64_t T, int64_t H,
                     const void* const* W, const void* const* bias,
                     const lp_vocab_partition* part, const int32_t* y, float tau,
                     const lp_outputs* out, void* workspace, size_t ws_bytes,
                     lp_stream_t stream);

/* lp_forward on host-resident rows: the whole call as a host program sees it. X_host
 * (bf16 [T, H]) and y_host (int32 [T]) are HOST memory, and so are the buffers in
 * out_host (logp, lse, and entropy / shard_stats when non-NULL); W and bias are device
 * memory as in lp_forward. On `stream` the call copies X and y into device staging held
 * in the workspace, runs lp_forward there and copies the requested outputs back, all
 * asynchronously: the host buffers hold the results once the stream has been
 * synchronised, and must stay valid until then. Page-locked host buffers make the copies
 * truly asynchronous; pageable ones also work. Results are bitwise those of lp_forward.
 * Batches of T >= 4096 rows run as two halves whose second half is copied in on an
 * auxiliary stream while the first half computes (a row's bits do not depend on its
 * batch); the first such call on a device creates that stream and three events, kept
 * until the process exits (make it before any stream capture). Calls from several host
 * threads may run at once: each call enqueues its uses of those events under a per-device
 * lock, which it holds only while enqueueing.
 * Workspace: lp_workspace_size(LP_OP_FORWARD_HOST, T, H, part) bytes of device memory. */
LP_API lp_status lp_forward_host(const void* X_host, int64_t T, int64_t H,
                                 const void* const* W, const void* const* bias,
                                 const lp_vocab_partition* part, const int32_t* y_host, float tau,
                                 const lp_outputs* out_host, void* workspace, size_t ws_bytes,
                                 lp_stream_t stream);

/* Logits-reuse forward (page "feat(rl-kernel): add CUDA linear logp provider
 * integration", Changes / Megatron integration: reuse local logits instead of a
 * second projection). logits[k] is shard k's UNSCALED bf16 logits (X W^T + b)
 * [T, V_k] with row stride ld[k] elements (ld[k] >= V_k, ld[k] % 8 == 0); the
 * temperature is applied once, here. Streams the logits once from HBM. */
LP_API lp_status lp_forward_from_logits(const void* const* logits, const int64_t* ld, int64_t T,
                                 const lp_vocab_partition* part, const int32_t* y, float tau,
                                 const lp_outputs* out, void* workspace, size_t ws_bytes,
                                 lp_stream_t stream);

/* Compact top-p replay (page "Perf/cuda compact top p replay", Summary and
 * Walkthrough "CUDA kernel and empty-shard handling"): per row, the up to 64 ids
 * in replay_ids[t][0..63] (-1 = unused slot; duplicates allowed) are validated,
 * sorted ascending and deduplicated; z_v = (x_t . W[v] + b[v]) / tau is scored
 * for those ids only (a gather GEMV, no full-vocabulary projection), and LSE is
 * taken over that set. logp = z[y] - LSE if y is in the set, else -inf.
 * Arguments as lp_forward, plus replay_ids int32 [T, 64]; out->entropy must be NULL. */
LP_API lp_status lp_top_p_replay(const void* X, int64_t T, int64_t H,
                          const void* const* W, const void* const* bias,
                          const lp_vocab_partition* part, const int32_t* replay_ids,
                          const int32_t* y, float tau, const lp_outputs* out,
                          void* workspace, size_t ws_bytes, lp_stream_t stream);

/* Compact top-p replay scored from reused local logits (page "Perf/cuda compact top p
 * replay", Walkthrough: the replay data travels with the local logits through the
 * tensor-parallel helper). Same id-set rules and outputs as lp_top_p_replay, but z_v
 * = logits[k][t, v - vocab_start_k] / tau: logits[k] is shard k's UNSCALED bf16 logits
 * [T, V_k] with row stride ld[k] elements (ld[k] >= V_k); temperature is applied once,
 * here. Reads only the logits of the replay ids. out->entropy must be NULL. */
LP_API lp_status lp_top_p_replay_from_logits(const void* const* logits, const int64_t* ld, int64_t T,
                                             const lp_vocab_partition* part, const int32_t* replay_ids,
                                             const int32_t* y, float tau, const lp_outputs* out,
                                             void* workspace, size_t ws_bytes, lp_stream_t stream);

/* The dense keep-mask route the compact replay replaces (page "Perf/cuda compact
 * top p replay", Validation: dense-mask and compact-support results are bitwise
 * equal). keep_mask[k] is uint8 [T, V_k] (nonzero = id kept, padded ids ignored).
 * Same outputs as lp_top_p_replay and bitwise equal to it for the same sets. */
LP_API lp_status lp_top_p_replay_dense_mask(const void* X, int64_t T, int64_t H,
                                     const void* const* W, const void* const* bias,
                                     const lp_vocab_partition* part,
                                     const uint8_t* const* keep_mask, const int32_t* y,
                                     float tau, const lp_outputs* out, void* workspace,
                                     size_t ws_bytes, lp_stream_t stream);

/* Backward of sum_t grad_logp[t] * logp[t] (+ sum_t grad_entropy[t] * entropy[t]),
 * the gradient the provider's autograd contract implies (page "feat(rl-kernel): add
 * CUDA linear logp provider integration", Summary: logp and optional entropy with
 * gradients attached). With p = softmax(z) over the real ids, lse and entropy the
 * merged outputs of lp_forward and mu = lse - entropy (= sum_v p_v z_v):
 *   G[t,v] = (grad_logp[t] (1[v == y_t] - p_tv) - grad_entropy[t] p_tv (z_tv - mu_t)) / tau
 *            (0 on padded ids)
 *   dX = sum_k G_k W_k (fp32 [T,H]),  dW_k = G_k^T X (fp32 [V_k,H]),  db_k = sum_t G_k (fp32 [V_k]).
 * entropy and grad_entropy are both NULL (logp term only) or both given. Rows whose
 * lse or grad_logp is not finite, or whose target is invalid, get no gradient.
 * dX, dW[k] and db[k] are overwritten. db may be NULL (then no bias gradient);
 * dW entries may be NULL only for empty shards. */
LP_API lp_status lp_backward(const void* X, int64_t T, int64_t H,
                      const void* const* W, const void* const* bias,
                      const lp_vocab_partition* part, const int32_t* y, float tau,
                      const float* lse, const float* grad_logp,
                      const float* entropy, const float* grad_entropy,
                      float* dX, float* const* dW, float* const* db,
                      void* workspace, size_t ws_bytes, lp_stream_t stream);

/* Output options of lp_backward_ex (page "feat(rl-kernel): add CUDA linear logp
 * provider integration", Changes / Megatron integration: the provider sits inside a
 * Megatron loss path, whose hidden-state gradients are bf16 and whose weight
 * gradients accumulate into fp32 buffers across micro-batches).
 *   dx_dtype    LP_DTYPE_F32: dX is float [T,H]; LP_DTYPE_BF16: dX is bf16 [T,H]
 *               holding the same fp32 sum rounded once to bf16.
 *   accumulate  0: dW[k] and db[k] are overwritten; 1: the gradient is added to what
 *               they hold (one fp32 add per element after the fixed-order sum, so the
 *               result is still deterministic); padded ids keep their old values and
 *               an empty batch leaves both untouched. dX is always overwritten.
 *   dw_dtype    LP_DTYPE_F32: dW[k] is float [V_k,H]; LP_DTYPE_BF16: bf16 [V_k,H], the
 *               same fp32 result rounded once to bf16 (half the largest write of the
 *               backward). Accumulation needs fp32 dW. db is always fp32. */
typedef struct {
  int32_t dx_dtype;
  int32_t accumulate;
  int32_t dw_dtype;
} lp_backward_options;

/* lp_backward with output options; opts NULL means {LP_DTYPE_F32, 0, LP_DTYPE_F32}, which
 * makes it identical to lp_backward. dX and the dW[k] point to float or bf16 per
 * opts->dx_dtype / opts->dw_dtype (16-byte aligned either way). Same workspace
 * (LP_OP_BACKWARD) and errors as lp_backward, plus LP_ERR_INVALID_ARG for an unknown
 * dtype, accumulate not 0/1, or accumulation into bf16 dW. */
LP_API lp_status lp_backward_ex(const void* X, int64_t T, int64_t H,
                                const void* const* W, const void* const* bias,
                                const lp_vocab_partition* part, const int32_t* y, float tau,
                                const float* lse, const float* grad_logp,
                                const float* entropy, const float* grad_entropy,
                                void* dX, void* const* dW, float* const* db,
                                const lp_backward_options* opts,
                                void* workspace, size_t ws_bytes, lp_stream_t stream);

/* Backward of the logits-reuse route (page "feat(rl-kernel): add CUDA linear logp
 * provider integration", Megatron integration: local logits are reused instead of a
 * second projection, so gradients flow back through them): the gradient of
 * sum_t grad_logp[t] logp[t] (+ sum_t grad_entropy[t] entropy[t]) of
 * lp_forward_from_logits with respect to the unscaled logits L_k. Since z = L / tau,
 *   dlogits[k][t, v - vocab_start_k] = G[t,v]
 *       = (grad_logp[t] (1[v == y_t] - p_tv) - grad_entropy[t] p_tv (z_tv - mu_t)) / tau
 * with p = exp(z - lse), mu = lse - entropy, and 0 on padded ids (the G of lp_backward).
 *   logits, ld  as lp_forward_from_logits (bf16, row stride ld[k] % 8 == 0)
 *   lse         the merged LSE of lp_forward_from_logits on the same logits
 *   entropy, grad_entropy   both NULL (logp term only) or both given
 *   dlogits     host array [n_shards] of device pointers: shard k [T, V_k] with row
 *               stride ld_out[k] elements, of type out_dtype (bf16: ld_out % 8 == 0;
 *               f32: ld_out % 4 == 0). dlogits[k] may be logits[k] itself (bf16,
 *               ld_out[k] == ld[k]): every element is read before it is overwritten
 *               by the same thread. Other overlaps are not allowed.
 * Rows whose lse or grad_logp is not finite, or whose target is out of range, get a
 * zero gradient (as in lp_backward; the forward has already reported a bad target).
 * Logits of -inf (entries a caller masked out) get a zero gradient. Streams the
 * logits once and writes the gradient once; needs no workspace. */
LP_API lp_status lp_backward_from_logits(const void* const* logits, const int64_t* ld, int64_t T,
                                         const lp_vocab_partition* part, const int32_t* y, float tau,
                                         const float* lse, const float* grad_logp,
                                         const float* entropy, const float* grad_entropy,
                                         void* const* dlogits, const int64_t* ld_out, lp_dtype out_dtype,
                                         lp_stream_t stream);

/* Fused forward that allocates nothing. The paper has no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory at all - a plugin
 * inside an engine whose memory manager owns every device byte, a runtime with a
 * memory budget fixed at start-up, a host language without a CUDA allocator - and so
 * cannot pass lp_forward a workspace.
 *
 * Same arguments, outputs and results as lp_forward, minus the workspace: the
 * scratch is one device array of LP_NOALLOC_SCRATCH_BYTES inside this library,
 * which every GPU that loads the library keeps until the process exits. Inputs and
 * outputs are still the caller's device memory. The call allocates nothing (no
 * cudaMalloc, no allocating library routine) and frees nothing.
 *  - Limit: lp_workspace_size(LP_OP_FORWARD, T, H, part) must not exceed
 *    LP_NOALLOC_SCRATCH_BYTES (32 MiB). That size is 3 * align256(4 T nb) +
 *    align256(4 T) bytes, nb = the number of 256-id vocabulary blocks (594 at
 *    V = 151936 in one shard), so at that vocabulary T <= 4704 rows fit and
 *    T = 4705 does not. Larger problems return LP_ERR_WORKSPACE_TOO_SMALL before
 *    any launch.
 *  - The first call on each device looks up that device's address of the array
 *    (with the device current); make that first call before any stream capture.
 *    The address is kept for the life of the process, so the device must not be
 *    reset (cudaDeviceReset) between calls: the array could move and later calls
 *    would write through a stale address.
 *  - Every call shares the one array and it keeps the previous call's contents.
 *    Nothing in it needs to start at zero (each call writes every slot it reads),
 *    but calls whose kernels overlap on the GPU - on different streams, or from
 *    different threads - race on it and give wrong results. */
LP_API lp_status lp_forward_noalloc(const void* X, int64_t T, int64_t H,
                                    const void* const* W, const void* const* bias,
                                    const lp_vocab_partition* part, const int32_t* y, float tau,
                                    const lp_outputs* out, lp_stream_t stream);

/* The rank-ordered reduction of per-shard statistics (page "Perf/cuda compact top p
 * replay", Summary: rank-ordered reductions, and tensor-parallel shards with no replay
 * candidates handled without NaN). After each tensor-parallel rank has run an entry
 * point on its own shards (a rank-local partition) with out->shard_stats, and the ranks
 * have gathered those statistics in rank order, every rank calls this to fold them:
 *   shard_stats  device fp32 [n_shards][3][T], the shards of `part` in ascending order,
 *                each (local LSE, target logit, own entropy) as lp_outputs describes
 *   part         the partition those shards form (usually the whole vocabulary)
 *   y            device int32 [T] global target ids in [0, vocab_real)
 *   out          logp and lse required, entropy optional, shard_stats must be NULL
 * Per row: LSE = log sum_k exp(lse_k); entropy = sum_k w_k (h_k + LSE - lse_k) with
 * w_k = exp(lse_k - LSE); logp = t_o - LSE for the shard o holding y, and -inf when no
 * shard of `part` holds y, when o is empty or when t_o is -inf. A row whose shards are
 * all empty gets LSE = -inf, logp = -inf, entropy = 0. The fold is the one every entry
 * point applies to its own shards, so merging the statistics of K rank-local calls gives
 * bit for bit what one call over all K shards returns (for replay statistics the
 * entropy output is meaningless: replay reports no entropy). A target outside
 * [0, vocab_real) records LP_ERR_TARGET_OUT_OF_RANGE. Needs no workspace. */
LP_API lp_status lp_merge_shard_stats(const float* shard_stats, int64_t T, const lp_vocab_partition* part,
                                      const int32_t* y, const lp_outputs* out, lp_stream_t stream);

#define LP_MAX_PARTS 64  /* partial sums per lp_sum_partials call */

/* out[i] = ((parts[0][i] + parts[1][i]) + parts[2][i]) + ... in exactly that order, for
 * i < count: the rank-ordered sum of per-rank partial results, such as each rank's share
 * of dX in the vocabulary-parallel backward (page "Perf/cuda compact top p replay",
 * Summary: rank-ordered reductions; a sum whose order varies would not be deterministic).
 *   parts     host array of n_parts (1..LP_MAX_PARTS) device pointers to fp32 [count],
 *             16-byte aligned
 *   out       device [count] fp32, or bf16 (the fp32 sum rounded once) per out_dtype,
 *             16-byte aligned; may be parts[0] itself (fp32), must not overlap any other
 * Needs no workspace. */
LP_API lp_status lp_sum_partials(const float* const* parts, int32_t n_parts, int64_t count, void* out,
                                 lp_dtype out_dtype, lp_stream_t stream);

/* Synchronises `stream`, returns the first device-side error recorded on the
 * current device since the last call (LP_OK if none) and clears it. */
LP_API lp_status lp_get_device_error(lp_stream_t stream);

/* Self-test of the bounded pipeline waits every kernel uses (failure detection): one
 * CTA waits on an mbarrier that nothing ever arrives on, with a limit of `limit_ns`
 * nanoseconds (1 us .. 2 s); the wait gives up, records LP_ERR_DEVICE_TIMEOUT in the
 * device error word and the kernel exits cleanly, leaving the context usable. Read the
 * result with lp_get_device_error(). Nothing hangs and nothing faults. */
LP_API lp_status lp_selftest_wait_timeout(uint64_t limit_ns, lp_stream_t stream);

/* The time limit of every pipeline wait of the GEMM kernels launched after this call, in
 * nanoseconds (1 us .. 10 s; 0 restores the default of 2 s), for the whole process. A wait
 * that runs past it gives up: the kernel records LP_ERR_DEVICE_TIMEOUT, lets the copies and
 * MMAs it already started finish, frees its tensor memory and returns, leaving the context
 * usable and the call's outputs undefined. Failure detection is tested by setting a limit
 * too short for any wait to be met. Returns LP_ERR_INVALID_ARG outside the range. */
LP_API lp_status lp_set_wait_limit(uint64_t limit_ns);

/* 1 if this library was built with device-side bounds checks (LP_DEBUG_BOUNDS=1), else 0.
 * The compute sanitizer is not available on every machine; such a build stands in for its
 * out-of-bounds checks: the index of every plain (non-TMA) load or store a kernel computes
 * from the grid, the partition, the targets or the replay ids - in the streaming, replay
 * and gradient kernels and in the epilogues of the tensor-core GEMMs (bias reads, the
 * forward's statistics, G, dW and dX stores) - is compared with the extent of its buffer
 * as the host computed it, before the access; a failed comparison records LP_ERR_BOUNDS in
 * the device error word and skips the access instead of touching memory. TMA copies are
 * bounded by their tensor maps. Results are otherwise bitwise those of the regular build,
 * which compiles the checks away. */
LP_API int lp_debug_bounds_build(void);

/* Self-test of the bounds checks: one thread checks an index equal to its extent. A
 * bounds-checked build records LP_ERR_BOUNDS (read it with lp_get_device_error()); the
 * regular build records nothing. No memory is accessed either way. */
LP_API lp_status lp_selftest_bounds(lp_stream_t stream);

/* Identity of this build: a hash of the sources and code flags it was compiled from (a
 * static string; "unknown" for a build made without the in-tree build script). Lets a
 * caller check that the library it loaded was built from the sources it expects. */
LP_API const char* lp_build_id(void);

/* 1 if the current device can run this library (sm_100 family, e.g. GB300), else 0. */
LP_API int lp_device_supported(void);

/* Static, human-readable name of a status code. */
LP_API const char* lp_status_string(lp_status s);

#ifdef __cplusplus
}
#endif

#endif /* LP_H_ */
