/*
 * ring_attn.h -- C ABI of the GB300 ring-attention library (libring_attn.so).
 *
 * What it computes
 * ----------------
 * Ring attention for context parallelism.  The sequence (one document, or a
 * packed THD batch of documents described by cu_seqlens) is cut along the
 * token dimension into cp_size shards per document; the query shard of rank r
 * stays put while the key/value shards travel around a ring, and at every
 * ring step the rank computes attention of its queries against the key/value
 * shard it currently holds, merging the partial result into a running
 * (O, LSE).  Sources:
 *   - NVSHMEM/XLA page, "Paralelismo de contexto y atencion en anillo": each
 *     device processes its local part of the sequence, exchanges KV with its
 *     ring neighbours and computes attention incrementally as KV blocks
 *     circulate, keeping mathematical equivalence with standard attention.
 *   - Accelerate guide, "Detalhes tecnicos": Q, K, V sharded along the
 *     sequence (parts of size D//N), per-shard attention attn(Q_i, K_j, V_j)
 *     for every j, then a combine of the partials.
 *   - Accelerate guide: attention without a mask or with a causal mask only.
 *   - Dynamic-CP page, "Reprogramacion dinamica y empaquetado de datos": THD
 *     packing with cu_seqlens; a cp_size per document (per micro-batch).
 * On one GPU the ring is run as successive ring steps over key/value shards
 * that already sit in this GPU's memory; there is no communication.
 *
 * Readings taken where the pages are silent:
 *   - combine = exact log-sum-exp merge of normalised partials;
 *   - zigzag layout: 2*cp equal chunks per document (floor boundaries), rank r
 *     holds chunks r and 2*cp-1-r; contiguous layout: cp floor-boundary parts;
 *   - ring order: at step s rank r holds key/value shard (r - s) mod cp;
 *   - masks on global positions: a query sees a key iff both are in the same
 *     document and (not causal or key <= query);
 *   - GQA: query head h reads key/value head h / (Hq / Hkv);
 *   - LSE is the natural log of sum exp(scale * q.k), fp32, layout [Hq, T].
 *
 * Conventions
 * -----------
 * Tensors are dense, row-major THD in natural (global) token order:
 *   q, o, dout, dq : [T, Hq, head_dim]     k, v, dk, dv : [T, Hkv, head_dim]
 * bf16 unless a *_fp32 flag says fp32.  The layout only decides which token
 * ranges meet at which ring step; no permutation of the tensors is needed.
 * Every device pointer must be 16-byte aligned.  head_dim is 64 or 128.
 *
 * Ownership: the caller owns every device buffer, including the workspace.
 * The plan is host memory (its work lists are also kept in mapped pinned host
 * memory where a device is usable; see ra_plan_create).  ra_fwd/ra_bwd put the
 * plan's work lists into the workspace (a small kernel reading the pinned
 * copy, else cudaMemcpyAsync), enqueue kernels on `stream` (a cudaStream_t,
 * NULL = legacy default stream) and return without synchronising; nothing is
 * allocated on the device.
 *
 * Errors: every entry point validates its arguments on the host first and
 * returns RA_ERR_INVALID_ARG / RA_ERR_UNSUPPORTED / RA_ERR_WORKSPACE before
 * enqueuing anything; a CUDA launch or copy failure returns RA_ERR_CUDA.
 * ra_last_error() returns a thread-local message for the last non-OK status.
 * Kernels never trap: a pipeline wait that exceeds its time limit makes the
 * kernel record a code in the workspace header and return early;
 * ra_workspace_status() reads that code (RA_ERR_TIMEOUT).
 */
#ifndef RING_ATTN_H
#define RING_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1,
  RA_ERR_UNSUPPORTED = 2,
  RA_ERR_CUDA = 3,
  RA_ERR_WORKSPACE = 4,
  RA_ERR_TIMEOUT = 5
} ra_status;

typedef enum { RA_LAYOUT_CONTIGUOUS = 0, RA_LAYOUT_ZIGZAG = 1 } ra_layout;
typedef enum { RA_CP_DYNAMIC = 0, RA_CP_STATIC = 1 } ra_cp_mode;

typedef struct ra_plan ra_plan; /* opaque, host memory (work lists also pinned) */

/* Version of this ABI (bumped on any signature change). */
int32_t ra_abi_version(void);

/*
 * Build a plan: shard every document, pair shards per ring step and cut the
 * pairs into GPU work items.
 *   cu_seqlens      host int32[num_docs + 1], cu_seqlens[0] == 0, non-decreasing;
 *                   T = cu_seqlens[num_docs] (Dynamic-CP page, THD packing).
 *   cp_size_per_doc host int32[num_docs] ring size of each document, or NULL to
 *                   use cp_size for all (Dynamic-CP: cp chosen per micro-batch).
 *   layout          RA_LAYOUT_CONTIGUOUS or RA_LAYOUT_ZIGZAG.
 *   causal          1: key <= query within a document; 0: whole document.
 *   num_q_heads, num_kv_heads: Hq % Hkv == 0.
 *   softmax_scale   <= 0 selects 1/sqrt(head_dim).
 * The plan copies what it needs; the caller's arrays may be freed afterwards.
 * Where a CUDA device is usable, the plan also keeps its work lists in mapped
 * pinned host memory (cudaHostAlloc, a host allocation) so that each call
 * sets up its workspace with one small kernel instead of a copy from pageable
 * memory; without a device the plan is host-only and the calls copy.  The
 * environment variable RA_NO_PINNED_WORK_LISTS=1 selects the copies (tests).
 */
ra_status ra_plan_create(ra_plan** out, const int32_t* cu_seqlens, int32_t num_docs,
                         const int32_t* cp_size_per_doc, int32_t cp_size, int32_t layout,
                         int32_t causal, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, float softmax_scale);

/* Free a plan (NULL is ignored), including its pinned work-list copy. */
void ra_plan_destroy(ra_plan* plan);

/*
 * Run the plan's backward (ra_bwd, ra_bwd_ring_step, ra_bwd_ring_step_rank) on
 * CTA pairs: at head_dim 128 a cluster of two CTAs takes two neighbouring
 * 128-key tiles of one key/value head and issues its matrix products as
 * cta_group::2 tensor-core operations (M = 256 over the pair's keys for S, dP,
 * dV, dK; dQ of a 128-row query tile reduced over all 256 keys at once).  The
 * gradients are those of the one-CTA kernel (same formulas as ra_bwd, same
 * accumulation order within a key tile).  on = 0 (the default) or 1.  Changing
 * it rebuilds the plan's backward work lists (pairs of neighbouring key
 * tiles; a range with an odd number of tiles ends in an empty one), so it is
 * a host call to make between launches, not while work of this plan is in
 * flight.  RA_ERR_UNSUPPORTED for head_dim != 128, RA_ERR_INVALID_ARG for a
 * NULL plan or `on` outside {0, 1}.  This option is this library's own: the
 * pages describe no kernel design.
 */
ra_status ra_plan_set_bwd_cta_pairs(ra_plan* plan, int32_t on);

/*
 * Workspace sizes in bytes for ra_fwd (status header, work list and key-tile
 * table; the same for either output dtype, o_is_fp32 is accepted for
 * symmetry) and ra_bwd (given grads_fp32: bf16 gradients add their fp32
 * accumulators).  Either output pointer may be NULL.
 */
ra_status ra_plan_workspace_bytes(const ra_plan* plan, int32_t o_is_fp32, int32_t grads_fp32,
                                  size_t* fwd_bytes, size_t* bwd_bytes);

/*
 * Workspace bytes of the ring-step forward (ra_fwd_ring_steps, and
 * ra_fwd_prepare / ra_fwd_ring_step / ra_fwd_finish): status header, work
 * list and, for a bf16 output (o_is_fp32 == 0), the fp32 running output
 * [T, Hq, d] that the steps merge into.
 */
ra_status ra_plan_ring_step_workspace_bytes(const ra_plan* plan, int32_t o_is_fp32, size_t* fwd_bytes);

/*
 * Plan statistics: number of ring steps (max cp over documents), visible
 * (query, key) pairs summed over documents (per head), and the number of
 * forward / backward work items over all steps (backward items are per
 * key/value head).  Any pointer may be NULL.
 */
ra_status ra_plan_stats(const ra_plan* plan, int32_t* num_steps, int64_t* visible_pairs,
                        int64_t* fwd_items, int64_t* bwd_items);

/*
 * Copy the plan's GPU work items to host memory, for inspection and tests.
 * which = 0: forward items {q0, q1, kb0, ke0, kb1, ke1, flags, tiles};
 * which = 1: backward items {k0, k1, qb0, qe0, qb1, qe1, flags, tiles}
 * (8 int32 each, global token positions, ranges end-exclusive).  Forward
 * items cover all query heads; backward items are per key/value head, which
 * is flags >> 8 (bit 0 of flags marks ring step 0).
 * items: host int32[8 * capacity] or NULL; step_offsets: host
 * int64[num_steps + 1] or NULL (items of step s are [off[s], off[s+1])).
 * *count receives the total number of items; RA_ERR_INVALID_ARG if
 * capacity is too small for a non-NULL `items`.
 */
ra_status ra_plan_work_items(const ra_plan* plan, int32_t which, int32_t* items, int64_t capacity,
                             int64_t* step_offsets, int64_t* count);

/*
 * Token ranges of shard `rank` of document `doc` (global positions, end
 * exclusive): up to two ranges (zigzag: chunk rank and chunk 2*cp-1-rank).
 * begin2/end2 are host int32[2]; *count receives 1 or 2 (empty ranges are
 * still reported, with begin == end).  Accelerate guide, "Detalhes tecnicos".
 */
ra_status ra_shard_token_ranges(const ra_plan* plan, int32_t doc, int32_t rank,
                                int32_t* begin2, int32_t* end2, int32_t* count);

/*
 * Dynamic-CP sizing (host only; Dynamic-CP page, "Modelado del programador de
 * datos", "Necesidad de un enfoque dinamico", "Construccion de multiples
 * grupos de contexto paralelo por rango"): a context-parallel group size per
 * sequence and its place on num_ranks ranks, from the cost model
 *   time(L) = sec_per_pair * pairs(L) + sec_per_token * L,
 *   pairs(L) = L (L + 1) / 2 causal, L * L otherwise,
 * group sizes powers of two in [1, num_ranks] (num_ranks a power of two) and
 * at most max_tokens_per_rank tokens on a rank (a sequence of length L on a
 * group of size c puts ceil(L / c) tokens on each of its ranks).
 *   mode RA_CP_DYNAMIC: each sequence starts at the smallest size that fits
 *     the token limit and keeps its per-rank time <= sum(time) / num_ranks;
 *   mode RA_CP_STATIC: every sequence takes the size of the longest one.
 * Sequences are placed most expensive first on the aligned group
 * [g c, (g + 1) c) whose busiest rank ends least loaded (ties: lowest g),
 * within the token limit; one that fits no group moves to the next larger
 * size.  Outputs (host): cp_per_doc[num_docs] (usable as ra_plan_create's
 * cp_size_per_doc), first_rank[num_docs], and optionally rank_load[num_ranks]
 * (modelled seconds: sum of time(L)/c over the sequences a rank holds) and
 * rank_tokens[num_ranks].  RA_ERR_INVALID_ARG (with a message) for bad
 * arguments or a batch that does not fit.  No device work.
 */
ra_status ra_dynamic_cp(const int32_t* doc_lengths, int32_t num_docs, int32_t num_ranks,
                        int64_t max_tokens_per_rank, int32_t causal, double sec_per_pair, double sec_per_token,
                        int32_t mode, int32_t* cp_per_doc, int32_t* first_rank, double* rank_load,
                        int64_t* rank_tokens);

/*
 * ra_fwd_fused: the same call as ra_fwd (kept under this name).
 * ra_fwd: the forward in one launch over the whole ring.  Each
 * CTA keeps one 256-row query chunk's running (O, row max, row sums) on chip
 * and visits the key/value shards in ring order, s = 0 .. cp-1 (shard
 * (r - s) mod cp): the merge of step s into the running state is the online
 * softmax continuing over that shard's key tiles (NVSHMEM/XLA page,
 * "Paralelismo de contexto y atencion en anillo": attention is accumulated
 * incrementally as the KV blocks circulate; Accelerate guide, "Detalhes
 * tecnicos": `combine` of the per-shard results), so no running output goes
 * through HBM between steps and O is written once, in its final dtype.
 * Within a chunk the online softmax visits exactly the key tiles that the
 * ring steps would, in the same order, so the result equals the ring-step
 * forward (ra_fwd_ring_steps) up to fp32 rounding.
 *   q [T,Hq,d] bf16, k/v [T,Hkv,d] bf16 (device).
 *   o [T,Hq,d]: bf16, or fp32 when o_is_fp32 != 0 (device, written).
 *   lse [Hq,T] fp32 natural-log log-sum-exp (device, written).
 *   workspace: device, >= ra_plan_workspace_bytes(..).fwd.
 * The caller owns every buffer; RA_ERR_WORKSPACE when the workspace is too
 * small.
 */
ra_status ra_fwd(const ra_plan* plan, const void* q, const void* k, const void* v, void* o,
                 int32_t o_is_fp32, float* lse, void* workspace, size_t workspace_bytes,
                 void* stream);
ra_status ra_fwd_fused(const ra_plan* plan, const void* q, const void* k, const void* v, void* o,
                       int32_t o_is_fp32, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of ra_fwd / ra_fwd_fused (header, work list, key-tile table). */
ra_status ra_plan_fused_workspace_bytes(const ra_plan* plan, size_t* fwd_bytes);

/*
 * The single-launch forward's work list, for inspection and tests: items as
 * int32[8] each {q0, q1, first tile, tile count, active tiles of rows
 * [q0, q0+128), active tiles of rows [q0+128, q1), flags, tile count}, and
 * tiles as int32[2] each {tile start, end of its key range} (the tile covers
 * [start, min(start + 128, end))), ring step by ring step.  Either output may
 * be NULL; *num_items / *num_tiles receive the sizes; RA_ERR_INVALID_ARG if a
 * capacity is too small for a non-NULL output.
 */
ra_status ra_plan_fused_items(const ra_plan* plan, int32_t* items, int64_t item_capacity, int32_t* tiles,
                              int64_t tile_capacity, int64_t* num_items, int64_t* num_tiles);

/*
 * Forward, one launch per ring step: for s = 0 .. steps-1 every query shard r
 * attends to key/value shard (r - s) mod cp of its document (tcgen05
 * tensor-core block attention with online softmax); each step's partial
 * (O_s, LSE_s) is merged exactly into the running (O, LSE) in the step
 * kernel's epilogue.  Arguments as ra_fwd; workspace: device,
 * >= ra_plan_ring_step_workspace_bytes(.., o_is_fp32, ..).
 */
ra_status ra_fwd_ring_steps(const ra_plan* plan, const void* q, const void* k, const void* v, void* o,
                            int32_t o_is_fp32, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Backward from the saved LSE: Delta = rowsum(dout * o) (o as returned by
 * ra_fwd, dtype per o_is_fp32), then per ring step the probabilities are
 * recomputed as P = exp(scale q.k - LSE) and
 *   dV += P^T dO,  dS = P * (dO V^T - Delta),  dK += scale dS^T Q,  dQ += scale dS K,
 * with dK/dV summed over the query heads of each GQA group.
 *   dq [T,Hq,d], dk/dv [T,Hkv,d]: bf16, or fp32 when grads_fp32 != 0 (device, written).
 *   workspace: device, >= ra_plan_workspace_bytes(.., grads_fp32).bwd.
 */
ra_status ra_bwd(const ra_plan* plan, const void* q, const void* k, const void* v,
                 const void* o, int32_t o_is_fp32, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int32_t grads_fp32, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * The ring step as its own call.  ra_fwd_ring_steps is exactly
 *   ra_fwd_prepare; ra_fwd_ring_step(s) for s = 0 .. steps-1; ra_fwd_finish
 * (workspace >= ra_plan_ring_step_workspace_bytes) and ra_bwd is
 *   ra_bwd_prepare; ra_bwd_ring_step(s) for every s; ra_bwd_finish
 * on one workspace.  A multi-GPU driver would call the ring step after each
 * key/value exchange (NVSHMEM/XLA page, "Patrones de comunicacion en la
 * atencion en anillo": compute on the current KV block while the next one
 * is fetched).  Each ring-step call enqueues exactly one kernel.
 *
 * ra_fwd_prepare: reset the status word and copy the forward work list.
 * ra_fwd_ring_step: step in [0, steps); forward steps must run in order
 *   (step 0 initialises the running (O, LSE), later steps merge into it).
 * ra_fwd_finish: write the bf16 output from the fp32 running output (no-op
 *   when o_is_fp32).
 * ra_bwd_prepare: reset the status word, copy the backward work list,
 *   compute Delta = rowsum(dout * o) and LSE in log2 units, zero the fp32
 *   gradient accumulators (the gradients themselves when grads_fp32).
 *   dq/dk/dv may be NULL unless grads_fp32.
 * ra_bwd_ring_step: step in [0, steps), any order (accumulation only).
 * ra_bwd_finish: cast the fp32 accumulators to the bf16 gradients (no-op
 *   when grads_fp32).
 */
ra_status ra_fwd_prepare(const ra_plan* plan, int32_t o_is_fp32, void* workspace, size_t workspace_bytes,
                         void* stream);
ra_status ra_fwd_ring_step(const ra_plan* plan, int32_t step, const void* q, const void* k, const void* v,
                           void* o, int32_t o_is_fp32, float* lse, void* workspace, size_t workspace_bytes,
                           void* stream);
ra_status ra_fwd_finish(const ra_plan* plan, void* o, int32_t o_is_fp32, void* workspace,
                        size_t workspace_bytes, void* stream);
ra_status ra_bwd_prepare(const ra_plan* plan, const void* o, int32_t o_is_fp32, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int32_t grads_fp32,
                         void* workspace, size_t workspace_bytes, void* stream);
ra_status ra_bwd_ring_step(const ra_plan* plan, int32_t step, const void* q, const void* k, const void* v,
                           const void* dout, void* dq, void* dk, void* dv, int32_t grads_fp32,
                           void* workspace, size_t workspace_bytes, void* stream);
ra_status ra_bwd_finish(const ra_plan* plan, void* dq, void* dk, void* dv, int32_t grads_fp32,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * The ring step of one rank, for a multi-GPU ring (one process per GPU, rank
 * r keeps query shard r and holds key/value shard (r - s) mod cp at step s:
 * NVSHMEM/XLA page, "Patrones de comunicacion en la atencion en anillo";
 * Accelerate guide, "Detalhes tecnicos").  Same as ra_fwd_ring_step /
 * ra_bwd_ring_step, restricted to the work items of query shard `rank`
 * (rank in [0, steps)): the kernel reads only key/value rows of shard
 * (rank - step) mod cp and writes only the running output rows of shard rank
 * (forward), or dQ rows of shard rank and dK/dV rows of shard
 * (rank - step) mod cp (backward).  Tensors keep the global THD layout
 * [T, H, d]: a rank's buffers are full length and only the rows of the shards
 * it holds are used; every other row of q, k, v, o, dout and of the running
 * output must hold finite values (zeros), since 128-row tiles overhang a
 * shard's ranges and a masked probability of 0 times a NaN is not 0.
 * Workspaces and prepare/finish calls as for the all-ranks calls
 * (ra_fwd_prepare puts both work lists in place).
 */
ra_status ra_fwd_ring_step_rank(const ra_plan* plan, int32_t step, int32_t rank, const void* q, const void* k,
                                const void* v, void* o, int32_t o_is_fp32, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);
ra_status ra_bwd_ring_step_rank(const ra_plan* plan, int32_t step, int32_t rank, const void* q, const void* k,
                                const void* v, const void* dout, void* dq, void* dk, void* dv, int32_t grads_fp32,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * The per-rank work lists, for inspection and tests: items as in
 * ra_plan_work_items, grouped by (step, rank); offsets: host
 * int64[steps * steps + 1] or NULL (items of step s, rank r are
 * [off[s * steps + r], off[s * steps + r + 1])).
 */
ra_status ra_plan_rank_work_items(const ra_plan* plan, int32_t which, int32_t* items, int64_t capacity,
                                  int64_t* offsets, int64_t* count);

/*
 * Failure-detection self-test (no counterpart on the pages): enqueue one small
 * kernel that waits, through the same bounded mbarrier wait the ring kernels
 * use, on a barrier that nothing ever arrives on.  After limit_us microseconds
 * (1 .. 4000000) it gives up, writes site code 900 into the status word at the
 * start of `workspace` (device, >= 256 bytes, zeroed here first) and returns,
 * so ra_workspace_status() then reports RA_ERR_TIMEOUT and the CUDA context
 * stays usable.  No trap, no hang.  RA_ERR_INVALID_ARG for bad arguments.
 */
ra_status ra_selftest_wait_timeout(void* workspace, uint32_t limit_us, void* stream);

/*
 * Synchronise `stream` and read the status word that the last ra_fwd/ra_bwd
 * call on this workspace left in its header: RA_OK, or RA_ERR_TIMEOUT if a
 * kernel gave up on a pipeline wait (its outputs are then undefined).
 */
ra_status ra_workspace_status(const void* workspace, void* stream);

/*
 * Forward without any device allocation, for callers that cannot call
 * cudaMalloc or hand out a workspace: plugins whose host framework owns all
 * device memory and passes in only inputs and outputs, or serving loops that
 * must not allocate (an allocation can synchronise the device or overrun a
 * fixed memory budget).  (No counterpart on the pages; a library convenience.)
 * Same computation and arguments as ra_fwd, minus the workspace: the
 * workspace is a fixed 32 MiB device array inside this library, held on
 * every GPU that loads it until the process exits.
 *   - A plan whose forward workspace (ra_plan_workspace_bytes(..).fwd: the
 *     work list and key-tile table) exceeds 32 MiB is rejected with
 *     RA_ERR_WORKSPACE before any GPU work.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and so does the first
 *     call after the device's context was re-created (cudaDeviceReset); make
 *     those first calls before any stream capture.
 *   - All calls share the one array: calls that may overlap on the GPU (other
 *     streams, other host threads) race and must be serialised by the caller.
 *     Each call zeroes the array's status word and rewrites its work lists
 *     before the kernel reads them.
 */
ra_status ra_fwd_noalloc(const ra_plan* plan, const void* q, const void* k, const void* v, void* o,
                         int32_t o_is_fp32, float* lse, void* stream);

/*
 * Status of the last ra_fwd_noalloc call on the current device, read from
 * the fixed array's status word after synchronising `stream` (as
 * ra_workspace_status does for a caller's workspace): RA_OK, or
 * RA_ERR_TIMEOUT if its kernel gave up on a pipeline wait (the outputs are
 * then undefined).  Allocates nothing.
 */
ra_status ra_noalloc_status(void* stream);

/* Thread-local text for the last non-OK status returned on this thread. */
const char* ra_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RING_ATTN_H */
