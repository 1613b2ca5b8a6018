/*
 * ep.h -- libep: MoE expert-parallel token dispatch / combine on one GPU
 * (NVIDIA GB300, sm_103a).  Plain C ABI: pointers, sizes, a CUDA stream.
 *
 * The calls mirror the per-step API of TransformerEngine PR #3034, "Expert
 * Parallelism: common C API + NCCL EP backend" (sections "Lifecycle
 * (host-only, eager)" and "Per-step (allocation-free, CUDA-graph
 * capturable)"): register_layer, prepare, dispatch, combine, dispatch_bwd and
 * combine_bwd.  On one GPU the expert-parallel ranks collapse into a single
 * expert-major receive buffer: there is no communicator, no symmetric-memory
 * window and no inter-GPU transfer, so those parameters are absent.
 *
 * Notation.  T tokens, H hidden (bf16 elements per row), E experts, K top-k,
 * A = dispatch_output_per_expert_alignment (given to ep_prepare).  A route is
 * a pair (t, k); route (t, k) picks expert topk_idx[t*K + k].  A value of -1
 * masks the route.  c_e = number of valid routes to expert e,
 * p_e = roundup(c_e, A) (0 when c_e = 0), off_e = p_0 + ... + p_{e-1},
 * P = off_E (receive rows in use), R = receive capacity in rows.
 * Receive row off_e + j holds the j-th route to expert e in ascending (t, k)
 * order; rows off_e + c_e .. off_e + p_e - 1 are padding.
 *
 * Ownership.  The caller allocates and owns every buffer: handle memory (size
 * from ep_register_layer) and all payloads.  libep allocates nothing per step.
 * All pointers passed to per-step calls are DEVICE pointers unless a
 * parameter says "host".  Per-step calls only enqueue work on `stream`: no
 * host-device synchronisation, no allocation, so they can be captured in a
 * CUDA graph.  The first call on a device also queries that device once
 * (compute capability, the kernel image, the largest thread-block cluster the
 * routing-map kernel may use there); make it before any stream capture.  Several handles (separate handle memories) may be in flight at
 * once; calls on one handle must be ordered (same stream or events).
 *
 * Layouts.  Row-major and contiguous.  Payload rows (tokens, receive rows,
 * expert outputs and their gradients) hold H elements of the layer's dtype:
 * bf16 (default), fp16 or fp32, passed as untyped pointers.  topk_idx is int64
 * [T, K]; weights are float32.  Payload pointers must be 16-byte aligned;
 * handle memory must be 256-byte aligned.
 *
 * Errors.  Every call returns an ep_status_t.  Host-detected problems (null
 * pointer, size out of range, unregistered layer, wrong GPU) return an error
 * code, enqueue nothing, and leave a message for ep_last_error() (per host
 * thread).  Problems only the GPU can see set sticky bits in the handle's
 * status word (EP_ST_*); ep_prepare rewrites that word, later calls add bits,
 * ep_read_info() reads it.  No kernel traps or waits on another kernel.
 */
#ifndef LIBEP_EP_H_
#define LIBEP_EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EP_ABI_VERSION 4u

typedef enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1,      /* null / misaligned pointer, bad value */
  EP_ERR_SHAPE = 2,            /* a size outside what the layer was registered for */
  EP_ERR_UNSUPPORTED_ARCH = 3, /* current device is not compute capability 10.3 */
  EP_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
  EP_ERR_NOT_REGISTERED = 5,   /* handle id unknown to this process */
  EP_ERR_LIMIT = 6             /* configuration beyond the library's limits */
} ep_status_t;

/* Sticky device status bits (handle status word). */
#define EP_ST_BAD_INDEX 1u       /* some topk_idx value outside [-1, E): treated as -1 */
#define EP_ST_OVERFLOW 2u        /* P > R: later row calls on the handle write nothing */
#define EP_ST_TOKENS_MISMATCH 4u /* a row call's num_tokens differs from the last prepare */
#define EP_ST_COUNTS_MISMATCH 16u /* sharded layers: the all-gathered counts given to
                                     ep_shard_prepare disagree with this rank's own
                                     routes; later row calls on the handle write nothing */
#define EP_ST_BAD_POINTER 32u    /* sharded layers: an address in a row call's pointer table
                                    was NULL or not 16-byte aligned; rows it would have
                                    addressed were skipped */
#define EP_ST_TIMEOUT 64u        /* reported by ep_read_info with EP_ST_NOT_PREPARED: the
                                    routing map's grid-wide wait gave up (its CTAs could not
                                    all run at once), nothing was prepared and the row calls
                                    write nothing; the grid-wide routing map (batches over
                                    65,536 routes) then does nothing on the handle until its
                                    memory is zero-filled again, while a smaller batch's
                                    prepare, which does not use the wait, rewrites it */
#define EP_ST_NOT_PREPARED 8u    /* reported by ep_read_info when no ep_prepare has
                                    written this handle memory; row calls then write nothing.
                                    Detected by a marker word in the handle header: zero-fill
                                    fresh handle memory so that stale contents of reused
                                    memory cannot carry the marker. */

/* Payload element types (TransformerEngine PR #3034 tests BF16, FP16 and FP32
 * payloads).  Sums accumulate in float32 and round once to the payload type
 * (round to nearest even; an fp32 payload receives the float32 sum itself). */
typedef enum { EP_DTYPE_BF16 = 0, EP_DTYPE_FP16 = 1, EP_DTYPE_FP32 = 2 } ep_dtype_t;

/* Library limits (checked at registration). */
#define EP_MAX_EXPERTS 1024
#define EP_MAX_TOPK 32

/* Per-layer configuration.  The pages name NVTEEpLayerConfig without listing
 * its fields; these are the ones a single-GPU expert-major layout needs. */
typedef struct {
  int64_t num_experts;   /* E, 1 .. EP_MAX_EXPERTS */
  int64_t top_k;         /* K, 1 .. EP_MAX_TOPK */
  int64_t hidden;        /* H, elements per payload row, > 0 and a multiple of 8 */
  int64_t max_tokens;    /* largest T any prepare will see, >= 0 */
  int64_t max_alignment; /* largest A any prepare will see, >= 1 */
  int64_t recv_capacity; /* R rows; 0 selects the worst case
                            max_tokens*K + min(E, max_tokens*K)*(max_alignment-1),
                            which no routing can overflow */
  int64_t dtype;         /* ep_dtype_t of every payload row (0 = bf16) */
} ep_layer_config_t;

/* Per-step handle: the registered layer id plus caller-owned device memory
 * holding the routing map (TransformerEngine's NVTEEpHandle {id, mem}). */
typedef struct {
  uint64_t id;
  void* mem;
} ep_handle_t;

/* What the last ep_prepare on a handle produced (read back by ep_read_info). */
typedef struct {
  uint32_t status;       /* EP_ST_* bits */
  int32_t num_tokens;    /* T of the last prepare */
  int32_t used_rows;     /* P */
  int32_t padding_rows;  /* P minus the number of valid routes */
} ep_info_t;

/* ABI version of the loaded library (EP_ABI_VERSION). */
uint32_t ep_abi_version(void);

/* Message of the last error returned on the calling host thread ("" if none). */
const char* ep_last_error(void);

/* Number of kernels libep has launched in this process (all threads). */
uint64_t ep_launch_count(void);

/* Register a layer (host only, eager, thread-safe).  Writes the new layer id
 * and the byte size of the handle memory each in-flight step needs.  Mirrors
 * nvte_ep_register_layer in "Lifecycle (host-only, eager)" of TransformerEngine
 * PR #3034.  Ids are never reused within a process. */
ep_status_t ep_register_layer(ep_layer_config_t config, uint64_t* id /* host, out */,
                              size_t* handle_mem_size /* host, out */);

/* Receive capacity R (rows) of a registered layer: recv_tokens, expert_out,
 * grad_expert_out and the grad rows given to ep_dispatch_bwd hold R rows
 * (only rows [0, P) are read or written). */
ep_status_t ep_recv_capacity(uint64_t id, int64_t* rows /* host, out */);

/* Build the routing map (TransformerEngine PR #3034, "Per-step", nvte_ep_prepare:
 * per-expert token counts and routing maps written to handle memory, each
 * expert block padded to dispatch_output_per_expert_alignment).
 *   topk_idx      int64 [T, K]  (T = num_tokens; may be NULL when T = 0)
 *   token_counts  int32 [E]     out: c_e, the raw count of valid routes
 *   alignment     A, 1 .. max_alignment
 * Rewrites the status word: EP_ST_BAD_INDEX, EP_ST_OVERFLOW. */
ep_status_t ep_prepare(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                       int32_t* token_counts, int64_t alignment, void* stream);

/* Same result as ep_prepare (same routing map, counts, offsets and status
 * bits), for callers that cannot allocate device memory themselves -- for
 * example a custom call inside a framework that owns all device memory (an
 * XLA-style runtime hands a custom call only the buffers it planned, so the
 * call cannot cudaMalloc a scratch buffer of its own), or a plug-in running
 * under a fixed memory budget.  The per-chunk counters that prepare needs
 * while it builds the map are kept in a fixed array compiled into libep: a
 * static __device__ array of 2^18 int32 (1 MiB) that every GPU which loads the
 * library holds until the process exits.  The pages have no counterpart: this
 * is a deployment variant of nvte_ep_prepare, not part of the method.
 *   - Arguments, ownership and results are those of ep_prepare; handle memory
 *     is still required (it receives the routing map); its scratch part is
 *     left untouched by this call.
 *   - Allocates nothing: no cudaMalloc / cudaFree, no library allocation.
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture on that device.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls that overlap on the GPU
 *     (two streams, or handles used without ordering) race on it: order them.
 *   - Returns EP_ERR_LIMIT, with a message and before any launch, when
 *     (num_experts + 1) x chunks exceeds the array's 2^18 ints, a chunk being
 *     at most 512 x W routes with W = max(1, min(16, 8192 / num_experts)):
 *     e.g. above 1,044,480 routes at 1024 experts, never below 2^24 routes at
 *     8 experts.  ep_prepare has no such limit. */
ep_status_t ep_prepare_static_scratch(ep_handle_t handle, const int64_t* topk_idx,
                                      int64_t num_tokens, int32_t* token_counts,
                                      int64_t alignment, void* stream);

/* Scatter token rows and routing weights to expert-major receive rows
 * (nvte_ep_dispatch): recv_tokens[slot(t,k)] = tokens[t],
 * recv_topk_weights[slot(t,k)] = topk_weights[t, k]; padding rows in [0, P)
 * get zeros.  topk_idx must be the array given to the last ep_prepare on this
 * handle (the slot map in handle memory is used; the pointer is only checked
 * for NULL when T > 0).
 *   tokens [T, H], topk_weights [T, K] f32,
 *   recv_tokens [R, H] out, recv_topk_weights [R] f32 out. */
ep_status_t ep_dispatch(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                        const void* tokens, const float* topk_weights,
                        void* recv_tokens, float* recv_topk_weights, void* stream);

/* Unweighted sum of expert outputs back to token order (nvte_ep_combine; the
 * caller has already multiplied by recv_topk_weights):
 *   result[t] = round( sum over k = 0..K-1 with a valid route of
 *                      float(expert_out[slot(t,k)]) ), sum from +0.0f in
 *                      ascending k, in float32, rounded once to the payload type.
 *   expert_out [R, H], result [T, H] out. */
ep_status_t ep_combine(ep_handle_t handle, const void* expert_out, int64_t num_tokens,
                       void* result, void* stream);

/* Backward of dispatch (nvte_ep_dispatch_bwd): token and weight gradients
 * returned to the source token.
 *   grad_tokens[t] = same float32 sum as ep_combine over grad rows;
 *   grad_topk_weights[t, k] = g_recv_topk_weights[slot(t,k)], 0 for a masked
 *   route, all 0 when g_recv_topk_weights is NULL (no weight gradient).
 *   grad [R, H], g_recv_topk_weights [R] f32 or NULL,
 *   grad_tokens [T, H] out, grad_topk_weights [T, K] f32 out. */
ep_status_t ep_dispatch_bwd(ep_handle_t handle, const void* grad,
                            const float* g_recv_topk_weights, int64_t num_tokens,
                            void* grad_tokens, float* grad_topk_weights, void* stream);

/* Backward of combine (nvte_ep_combine_bwd): grad_expert_out[slot(t,k)] = grad[t];
 * padding rows in [0, P) are zeroed.
 *   grad [T, H], grad_expert_out [R, H] out. */
ep_status_t ep_combine_bwd(ep_handle_t handle, const void* grad, int64_t num_tokens,
                           void* grad_expert_out, void* stream);

/* Weighted combine: the routing weight applied inside combine instead of by
 * the caller.  The pages' final combine is unweighted; in the TransformerEngine
 * PR #3035 review (thread on the weight multiply in combine) the fused multiply
 * is kept as an option for callers that do not fold the weight into the expert
 * MLP.
 *   result[t] = round( sum over valid k, ascending, from +0.0f, of
 *               float32( recv_topk_weights[slot] * float(expert_out[slot]) ) )
 *   expert_out [R, H], recv_topk_weights [R] f32, result [T, H] out. */
ep_status_t ep_combine_weighted(ep_handle_t handle, const void* expert_out,
                                const float* recv_topk_weights, int64_t num_tokens,
                                void* result, void* stream);

/* Backward of ep_combine_weighted:
 *   grad_expert_out[slot(t,k)] = round( float32(recv_topk_weights[slot] * float(grad[t])) ),
 *   g_recv_topk_weights[slot]  = sum over h of grad[t][h] * expert_out[slot][h]
 *                                (float32 fused multiply-adds; the order of the
 *                                sum is fixed by the kernel and does not vary
 *                                from run to run);
 *   padding rows in [0, P): zeros in both outputs.  Pass g_recv_topk_weights on
 *   to ep_dispatch_bwd to obtain grad_topk_weights.
 *   grad [T, H], expert_out [R, H], recv_topk_weights [R] f32,
 *   grad_expert_out [R, H] out, g_recv_topk_weights [R] f32 out. */
ep_status_t ep_combine_weighted_bwd(ep_handle_t handle, const void* grad,
                                    const void* expert_out, const float* recv_topk_weights,
                                    int64_t num_tokens, void* grad_expert_out,
                                    float* g_recv_topk_weights, void* stream);

/* Copy the padded expert offsets off_0 .. off_E (int32 [E+1], device) of the
 * last prepare, e.g. for a grouped GEMM over the receive buffer.  Sharded
 * layers: this rank's experts, int32 [E/N + 1].  Rank-major layers keep none
 * (EP_ERR_INVALID_ARG): the owner's single-buffer layer has them. */
ep_status_t ep_expert_offsets(ep_handle_t handle, int32_t* offsets, void* stream);

/* Copy the slot map of the last prepare: int32 [T, K], receive row of route
 * (t, k) or -1 (device). */
ep_status_t ep_token_slots(ep_handle_t handle, int32_t* slots, int64_t num_tokens, void* stream);

/* Read the handle's status word and the shape of the last prepare into host
 * memory.  Synchronises `stream`, so it cannot be captured in a graph. */
ep_status_t ep_read_info(ep_handle_t handle, ep_info_t* info /* host, out */, void* stream);

/* ------------------------------------------------------------------------
 * Sharded expert parallelism: N ranks, each holding its own tokens, rank q
 * owning the E/N experts [q*E/N, (q+1)*E/N) and their receive rows
 * (TransformerEngine PR #3035, "Sequence Diagram": prepare all-gathers the
 * routing table; dispatch pushes token rows to the owners of the chosen
 * experts; combine pulls the expert rows back; the backward pass runs the
 * reverse scatter and the reverse gather).
 *
 * Layout on owner q: expert-major blocks of q's experts starting at row 0,
 * each padded to a multiple of A; inside expert e's block the routes follow
 * (source rank, t, k) in ascending order.  Stacking the owners' buffers in
 * rank order therefore gives the single-buffer layout of all ranks' tokens
 * concatenated in rank order, and every output equals the matching slice of
 * the single-buffer step, bit for bit.
 *
 * Exchange.  libep holds no communicator (none of its calls talks to another
 * process).  Per step: ep_shard_count gives this rank's per-expert counts;
 * the caller all-gathers them over the ranks (int32 [N][E], rank-major: an
 * NCCL all-gather in a multi-GPU job); ep_shard_prepare takes the gathered
 * table.  Row calls address every rank's receive-side buffer through a
 * caller-owned DEVICE array of N pointers (entry r = rank r's buffer as this
 * rank's device can address it: its own memory for r = this rank, a peer
 * mapping otherwise); the kernels use plain vector loads and stores on
 * those addresses, no bulk copies or prefetches.  The caller orders the
 * ranks' calls: every rank's dispatch (or combine_bwd) must have completed
 * before an owner reads its receive rows, and an owner's expert outputs (or
 * gradient rows) must be written before any rank's combine (or
 * dispatch_bwd) reads them -- a barrier across the ranks between the
 * phases.
 *
 * Limits: 1 <= num_ranks <= EP_MAX_RANKS and N divides E (checked at
 * registration); max_tokens * top_k within the one-launch routing map,
 * C * W * 512 routes with W = the routing kernel's warps for E experts and C
 * = 16 CTAs where the device runs a 16-CTA cluster, else 8 (registration
 * checks C = 16; ep_shard_count and ep_shard_prepare return EP_ERR_LIMIT
 * before any launch when the batch exceeds what this device takes): 131,072
 * routes at E = 256 on a GB300.
 * ------------------------------------------------------------------------ */
#define EP_MAX_RANKS 64

/* Register a sharded layer for rank `rank` of `num_ranks`.  config holds the
 * global E, K, H, the largest T of any rank (max_tokens), max_alignment and
 * dtype; recv_capacity = 0 selects the owner's worst case
 * N*max_tokens*K + min(E/N, N*max_tokens*K)*(max_alignment-1). */
ep_status_t ep_register_layer_sharded(ep_layer_config_t config, int64_t num_ranks, int64_t rank,
                                      uint64_t* id /* host, out */,
                                      size_t* handle_mem_size /* host, out */);

/* This rank's histogram: local_counts[e] = valid routes of this rank's
 * topk_idx [T, K] to expert e, int32 [E] (device).  Writes nothing else. */
ep_status_t ep_shard_count(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                           int32_t* local_counts, void* stream);

/* Routing map of a sharded layer (nvte_ep_prepare with the all-gathered
 * table).  all_counts int32 [N][E] (device): row r = rank r's local_counts.
 * token_counts int32 [E/N] out: this rank's own experts' counts over all
 * ranks.  The handle then holds this rank's slot map (receive row of each
 * route on its owner) and owner map, and, as owner, its expert offsets
 * (ep_expert_offsets: int32 [E/N + 1]), P and padding rows.  Status:
 * EP_ST_BAD_INDEX (this rank's indices), EP_ST_OVERFLOW (any owner's
 * P > R), EP_ST_COUNTS_MISMATCH (row `rank` of all_counts is not this rank's
 * histogram). */
ep_status_t ep_shard_prepare(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                             const int32_t* all_counts, int32_t* token_counts,
                             int64_t alignment, void* stream);

/* Push (nvte_ep_dispatch over ranks): recv_tokens[owner][slot] = tokens[t],
 * recv_topk_weights[owner][slot] = topk_weights[t, k] for each route; this
 * rank's own padding rows are zeroed.  recv_tokens, recv_topk_weights:
 * device arrays of N device pointers. */
ep_status_t ep_shard_dispatch(ep_handle_t handle, int64_t num_tokens, const void* tokens,
                              const float* topk_weights, void* const* recv_tokens,
                              float* const* recv_topk_weights, void* stream);

/* Pull (nvte_ep_combine over ranks): result[t] = the float32 sum, k
 * ascending from +0.0f, of expert_out[owner][slot] over the token's valid
 * routes, rounded once to the payload type.  expert_out: device array of N
 * device pointers. */
ep_status_t ep_shard_combine(ep_handle_t handle, const void* const* expert_out,
                             int64_t num_tokens, void* result, void* stream);

/* Reverse scatter (nvte_ep_combine_bwd over ranks):
 * grad_expert_out[owner][slot] = grad[t]; this rank's own padding rows are
 * zeroed.  grad_expert_out: device array of N device pointers. */
ep_status_t ep_shard_combine_bwd(ep_handle_t handle, const void* grad, int64_t num_tokens,
                                 void* const* grad_expert_out, void* stream);

/* Reverse gather (nvte_ep_dispatch_bwd over ranks): grad_tokens[t] as in
 * ep_shard_combine over the grad rows; grad_topk_weights[t, k] =
 * g_recv_topk_weights[owner][slot], 0 for a masked route, all 0 when
 * g_recv_topk_weights is NULL.  grad, g_recv_topk_weights: device arrays of N
 * device pointers. */
ep_status_t ep_shard_dispatch_bwd(ep_handle_t handle, const void* const* grad,
                                  const float* const* g_recv_topk_weights, int64_t num_tokens,
                                  void* grad_tokens, float* grad_topk_weights, void* stream);

/* Owner map of the last ep_shard_prepare: int32 [T, K], the rank owning each
 * route's expert, or -1 (device). */
ep_status_t ep_shard_token_owners(ep_handle_t handle, int32_t* owners, int64_t num_tokens,
                                  void* stream);

/* ------------------------------------------------------------------------
 * Rank-major receive layout for sharded layers (TransformerEngine PR #3035,
 * review thread on the receive buffers: a rank-major buffer needs at most
 * max_tokens_per_rank x num_ranks rows per owner, the expert-major one up to
 * min(top_k, E) times that; the owner then permutes the received rows into
 * expert-major order itself).
 *
 * A token goes once to every rank owning one of its valid routes.  Owner q's
 * rows list the source ranks in order and each rank's tokens ascending, with
 * no gap between source blocks: M_q = sum over r of the tokens of rank r
 * that go to q, at most N * max_tokens.  With each row go the token's K
 * expert ids relative to q (int64, -1 where the route is masked, invalid or
 * owned by another rank) and its K routing weights (0.0f there): exactly the
 * topk_idx / topk_weights of a single-buffer layer of E/N experts on the
 * owner, whose ep_prepare / ep_dispatch do the local permutation and whose
 * ep_combine (or ep_dispatch_bwd) gives the owner's partial row per received
 * row.  ep_rank_major_combine then sums, per token, its owners' partial rows
 * in the order in which each owner first appears among the token's routes (k
 * ascending), in float32 from +0.0f, rounded once.  A token whose routes
 * share an owner is thus rounded twice, once on the owner and once here;
 * with one rank, or when a token's routes all have different owners, the
 * result equals the expert-major combine bit for bit.
 *
 * Exchange, tables and ordering as for the expert-major sharded layers
 * above: ep_rank_major_count gives this rank's counts per owner, the caller
 * all-gathers them (int32 [N][N]), ep_rank_major_prepare takes the table; row
 * calls address every rank's buffers through device arrays of N pointers,
 * each entry 16-byte aligned (NULL or misaligned entries: EP_ST_BAD_POINTER,
 * the rows they would address skipped).  The routing map runs over N
 * owners, so the batch limit is the sharded one for E = N (131,072 routes at
 * N <= 64 on a GB300).
 * ------------------------------------------------------------------------ */

/* Register a rank-major layer for rank `rank` of `num_ranks`.  config: global
 * E (divisible by num_ranks), K, H, the largest T of any rank (max_tokens)
 * and dtype; max_alignment is not used (the owner's local layer has its own);
 * recv_capacity = rows per owner, 0 selecting the worst case
 * num_ranks * max_tokens (no overflow possible). */
ep_status_t ep_register_layer_rank_major(ep_layer_config_t config, int64_t num_ranks, int64_t rank,
                                         uint64_t* id /* host, out */,
                                         size_t* handle_mem_size /* host, out */);

/* This rank's counts per owner: local_counts[q] = tokens of this rank's
 * topk_idx [T, K] with at least one valid route to an expert of rank q,
 * int32 [N] (device). */
ep_status_t ep_rank_major_count(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                                int32_t* local_counts, void* stream);

/* Rank-major routing map.  all_counts int32 [N][N] (device): row r = rank
 * r's local_counts.  recv_rows int32 [1] out (device): M_rank, the rows this
 * rank receives as owner.  The handle then holds, per route, the row of its
 * token on its owner at the owner's first route in the token (-1 at the
 * other routes; ep_token_slots reads it) and the owners.  Status as for
 * ep_shard_prepare: EP_ST_BAD_INDEX, EP_ST_OVERFLOW (some owner's M above
 * recv_capacity), EP_ST_COUNTS_MISMATCH. */
ep_status_t ep_rank_major_prepare(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                                  const int32_t* all_counts, int32_t* recv_rows, void* stream);

/* Push: for each token and each owner q of its routes,
 * recv_tokens[q][row] = tokens[t], recv_topk_idx[q][row*K + k] = the expert
 * of route k relative to q or -1, recv_topk_weights[q][row*K + k] = its
 * weight or 0.0f.  recv_topk_weights may be NULL (then topk_weights is not
 * read).  Tables: device arrays of N device pointers.  topk_idx must be the
 * table given to ep_rank_major_prepare (the rows come from the handle's map,
 * the ids from topk_idx). */
ep_status_t ep_rank_major_dispatch(ep_handle_t handle, const int64_t* topk_idx, int64_t num_tokens,
                                   const void* tokens, const float* topk_weights,
                                   void* const* recv_tokens, int64_t* const* recv_topk_idx,
                                   float* const* recv_topk_weights, void* stream);

/* Pull: result[t] = the float32 sum of partial[q][row of t on q] over the
 * token's owners q in first-route order, from +0.0f, rounded once to the
 * payload type (0 for a token without valid routes).  partial: device array
 * of N device pointers, each owner's [M_q, H] rows (its local ep_combine). */
ep_status_t ep_rank_major_combine(ep_handle_t handle, const void* const* partial, int64_t num_tokens,
                                  void* result, void* stream);

/* Reverse of ep_rank_major_combine: grad_recv[q][row of t on q] = grad[t] for
 * every owner q of the token (the input of the owner's local
 * ep_combine_bwd).  grad_recv: device array of N device pointers. */
ep_status_t ep_rank_major_combine_bwd(ep_handle_t handle, const void* grad, int64_t num_tokens,
                                      void* const* grad_recv, void* stream);

/* Reverse of ep_rank_major_dispatch: grad_tokens[t] as in
 * ep_rank_major_combine over the owners' [M_q, H] row gradients (their local
 * ep_dispatch_bwd); grad_topk_weights[t, k] = g_recv_topk_weights[q][row*K +
 * k] for route k's owner q and the token's row on q, 0 for a masked route,
 * all 0 when g_recv_topk_weights is NULL. */
ep_status_t ep_rank_major_dispatch_bwd(ep_handle_t handle, const void* const* grad_recv,
                                       const float* const* g_recv_topk_weights, int64_t num_tokens,
                                       void* grad_tokens, float* grad_topk_weights, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBEP_EP_H_ */
