/*
 * ccl.h -- ring-ordered collectives over p virtual ranks on one GB300 GPU.
 *
 * A "rank" is a buffer in this GPU's HBM.  Every collective takes HOST arrays
 * of p DEVICE pointers (one buffer per virtual rank), the element count, the
 * element type and the reduction, and enqueues its kernels on `stream`.
 *
 * Primitive semantics follow "Networks and Collective Communication"
 * (section 4.1, what each collective does; section 4.2, identities) and
 * "dist_train" (section "Collective Communication Primitives").  Reductions
 * follow the ring of "Networks and Collective Communication" section 5.1 and
 * "dist_train" section "Ring Algorithm": each chunk's partial sum walks the
 * ring once, and its fold order is fixed by that walk (see CHUNKS AND ORDER).
 *
 * CHUNKS AND ORDER.  A rank buffer of n elements is cut into p chunks; chunk c
 * has len(c) = floor(n/p) + (c < n mod p) elements and starts at
 * off(c) = c*floor(n/p) + min(c, n mod p)  (ccl_chunk_bounds).  Rank r passes
 * to rank r+1 (mod p).  Chunk c's partial starts at rank c+1 and visits ranks
 * c+2, ..., p-1, 0, ..., c, each adding its own value: for SUM the result is
 * ((x[c+1] + x[c+2]) + ...) + x[c], in fp32 for fp32 and bf16 data (bf16 is
 * widened exactly, summed in fp32 and rounded once, to nearest even) and in
 * wrapping two's-complement int32 for int32 data.  Rank k ends the
 * reduce-scatter phase owning chunk k.  Every entry point that reduces gives
 * results bit-identical to that walk.
 *
 * OWNERSHIP.  The caller owns every buffer.  The library keeps no state
 * between calls and allocates no device memory; pointer arrays are copied
 * into kernel parameters before a call returns, so they may be reused at
 * once.  Calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream); nothing synchronises unless the caller does.
 *
 * ERRORS.  Every entry point returns a ccl_status_t and never aborts.
 * Argument errors are detected on the host before anything is enqueued;
 * ccl_last_error() then gives a one-line reason (per calling thread).
 * Device pointers must be device-accessible and aligned to their element
 * size; 16-byte alignment of every pointer selects the vectorised kernels,
 * any other element-aligned pointer runs the element-wise kernels.
 */
#ifndef CCL_H_
#define CCL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CCL_ABI_VERSION 1
#define CCL_MAX_RANKS 128

typedef enum {
  CCL_OK = 0,
  CCL_ERR_INVALID_ARG = 1, /* bad p, pointer, size, alignment or aliasing */
  CCL_ERR_UNSUPPORTED = 2, /* valid arguments this library does not implement */
  CCL_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
  CCL_ERR_TIMEOUT = 4      /* a bounded device-side wait ran out (kernels run asynchronously,
                              so ccl_stream_check reports it); no kernel of this library waits
                              on a flag that another launch writes */
} ccl_status_t;

typedef enum { CCL_F32 = 0, CCL_BF16 = 1, CCL_I32 = 2 } ccl_dtype_t;

/* SUM is the pages' reduction.  MAX / MIN are extras: the receiving rank keeps
 * its own value when it is strictly greater (smaller) than the partial it got,
 * so ties and NaNs resolve in ring order too. */
typedef enum { CCL_SUM = 0, CCL_MAX = 1, CCL_MIN = 2 } ccl_op_t;

/* All-reduce schedules of "Networks and Collective Communication" section 5.2.
 * Each fixes the order in which an element's p values are added. */
typedef enum {
  CCL_SCHEDULE_RING = 0,               /* the ring (ccl_allreduce) */
  CCL_SCHEDULE_RECURSIVE_DOUBLING = 1, /* pairs at distance 1, 2, 4, ...; p a power of two */
  CCL_SCHEDULE_RABENSEIFNER = 2,       /* halving: pairs at distance p/2, p/4, ...; p a power of two */
  CCL_SCHEDULE_BINOMIAL_TREE = 3,      /* binomial reduce to rank 0 + broadcast; any p */
  CCL_SCHEDULE_NAIVE = 4               /* rank 0 adds ranks 1..p-1 in order, then broadcasts */
} ccl_schedule_t;

typedef enum {
  CCL_KIND_ALLREDUCE = 0,
  CCL_KIND_REDUCE_SCATTER = 1,
  CCL_KIND_ALL_GATHER = 2
} ccl_kind_t;

/* ------------------------------------------------------------- utilities */

/* CCL_ABI_VERSION of the loaded library. */
int ccl_abi_version(void);

/* Static text for a status code; never NULL. */
const char* ccl_status_string(ccl_status_t status);

/* One-line reason for the last non-OK status returned to this thread ("" if
 * none).  The pointer stays valid until this thread's next call. */
const char* ccl_last_error(void);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t ccl_kernel_launch_count(void);

/* The device error word: nonzero once a bounded device-side wait ran out (the
 * bulk-copy fan-out of ccl_all_gather / ccl_broadcast waits on its own copies
 * with a bound; no wait of this library depends on another launch or rank).
 * Synchronous (reads device memory); clear != 0 resets it to 0 afterwards.
 * Errors: flag NULL -> CCL_ERR_INVALID_ARG; a failed copy -> CCL_ERR_CUDA. */
ccl_status_t ccl_device_error_flag(unsigned int* flag, int clear);

/* Failure check after asynchronous work: synchronizes `stream`, then returns
 * CCL_ERR_TIMEOUT (and clears the word) if a bounded device-side wait ran out
 * since the last check, CCL_OK otherwise; the context stays usable either
 * way.  A failed synchronization -> CCL_ERR_CUDA. */
ccl_status_t ccl_stream_check(void* stream);

/* Self-test of that path: enqueues a one-thread kernel whose mbarrier wait
 * can never complete, so it gives up after a short bound (well under a
 * millisecond) and sets the error word; no copy is in flight and nothing
 * faults.  The next ccl_stream_check on `stream` returns CCL_ERR_TIMEOUT. */
ccl_status_t ccl_selftest_bounded_wait(void* stream);

/* Chunk c of an n-element buffer cut into p chunks (the rule under CHUNKS AND
 * ORDER; numpy's array_split).  Host only.  Errors: p outside 1..CCL_MAX_RANKS,
 * c outside 0..p-1, or a NULL output pointer -> CCL_ERR_INVALID_ARG. */
ccl_status_t ccl_chunk_bounds(int p, size_t n, int c, size_t* off, size_t* len);

/* Diagnostic (no counterpart on the pages): which fused fold kernel a call of
 * p ranks x n elements launches.  kind: the call (ccl_allreduce,
 * ccl_reduce_scatter, ccl_reduce with element type dt and reduction op, or
 * ccl_bucket_allreduce_scale_cast, whose dt must be CCL_F32 and op CCL_SUM).
 * aligned != 0: every pointer of the call is 16-byte aligned.  sm_count: the
 * device's SM count, or <= 0 for the current device's.  Returns *batch =
 * ranks whose loads one thread issues together and *vectors = 16-byte
 * vectors per thread of the small-p kernel, both 0 for the general kernel
 * (large p, MAX / MIN, unaligned buffers), or *batch = -1 for the kernel of
 * small chunks at p > 16 (every rank's part of a chunk segment loaded in one
 * round into shared memory; any op and alignment): at p = 17..32 while
 * p x (chunk + 1) <= 2048 elements, at p > 32 for chunks of at most 1536
 * elements while its grid (chunk segments of 4096 / p elements x p) holds at
 * most 4 CTAs per SM for every two of the 16-rank load rounds of the vector
 * kernels (ceil(p / 16)).  Host only; it enqueues nothing.
 * Errors: p outside 1..CCL_MAX_RANKS, an unknown kind / dt / op, a bucket
 * plan for another dt / op, NULL outputs -> CCL_ERR_INVALID_ARG. */
typedef enum {
  CCL_FOLD_ALLREDUCE = 0,
  CCL_FOLD_REDUCE_SCATTER = 1,
  CCL_FOLD_BUCKET = 2,
  CCL_FOLD_REDUCE = 3
} ccl_fold_kind_t;
ccl_status_t ccl_fold_plan(ccl_fold_kind_t kind, ccl_dtype_t dt, ccl_op_t op, int p, size_t n, int aligned,
                           int sm_count, int* batch, int* vectors);

/* -------------------------------------------------- fused single-pass kernels
 * One kernel reads every rank's element once, folds in ring order in fp32
 * (int32) registers and writes each output once.  Results are bit-identical
 * to the step-by-step ring. */

/* All-reduce ("Networks and Collective Communication" 4.1: everyone gets the
 * element-wise sum; 5.1: ring = reduce-scatter then all-gather).
 *   send[r]  p device pointers, each n elements of dt.
 *   recv[r]  p device pointers, each n elements of dt; recv[r] == send[r] is
 *            allowed (in place); any other overlap -> CCL_ERR_INVALID_ARG.
 * Every recv[r] receives the same ring-ordered reduction.  n == 0 is a no-op. */
ccl_status_t ccl_allreduce(const void* const* send, void* const* recv, int p, size_t n,
                           ccl_dtype_t dt, ccl_op_t op, void* stream);

/* All-reduce with the result another schedule would give, in one fused pass
 * (same buffers and aliasing rules as ccl_allreduce).  Recursive doubling and
 * the binomial tree add pairwise over ranks 0..p-1 (the same bits: IEEE
 * addition commutes, so only the pairing matters); Rabenseifner adds pairwise
 * over the ranks in bit-reversed order; naive adds in rank order from rank 0.
 * CCL_SCHEDULE_RING is ccl_allreduce.  Errors: recursive doubling or
 * Rabenseifner with p not a power of two -> CCL_ERR_INVALID_ARG; MAX / MIN
 * with a schedule other than the ring -> CCL_ERR_UNSUPPORTED. */
ccl_status_t ccl_allreduce_schedule(const void* const* send, void* const* recv, int p, size_t n,
                                    ccl_dtype_t dt, ccl_op_t op, ccl_schedule_t schedule,
                                    void* stream);

/* bf16 all-reduce / reduce-scatter with bf16 on the wire: the ring of
 * ccl_allreduce / ccl_reduce_scatter (same chunks, same order, same buffers
 * and aliasing rules, bf16 data, SUM), except that every hop rounds the new
 * partial to bf16 (nearest-even) before it travels on -- the partial a ring
 * sends when its messages are bf16 ("Networks and Collective Communication"
 * 5.1: each step moves one chunk; a bf16 chunk is half the bytes).  Chunk c
 * = bf16(...bf16(bf16(x_{c+1} + x_{c+2}) + x_{c+3})... + x_c), each add in
 * fp32.  For MAX / MIN rounding changes nothing: use ccl_allreduce. */
ccl_status_t ccl_allreduce_bf16_wire(const void* const* send, void* const* recv, int p, size_t n,
                                     void* stream);
ccl_status_t ccl_reduce_scatter_bf16_wire(const void* const* send, void* const* recv, int p, size_t n,
                                          void* stream);

/* All-reduce with the result of the hierarchical (two-level ring) all-reduce
 * ("Networks and Collective Communication" 6.3; 6.1's two-dimensional
 * all-reduce on an a x b grid folds the same way), in one fused pass (same
 * buffers and aliasing rules as ccl_allreduce).
 *   group   a, the ranks per group; groups are runs of consecutive ranks
 *           (group g = ranks g*a .. g*a + a - 1), b = p / a groups.
 * The buffer is cut into a chunks (chunk rule), chunk l into b sub-chunks; an
 * element of sub-chunk (l, m) is folded along every group's ring starting at
 * local rank l + 1, then along the ring over the groups starting at group
 * m + 1, in fp32 (int32), bf16 rounded once.  group == p or group == 1 gives
 * ccl_allreduce's bits.  Errors: group < 1 or not dividing p ->
 * CCL_ERR_INVALID_ARG; MAX / MIN -> CCL_ERR_UNSUPPORTED (order-free: use
 * ccl_allreduce). */
ccl_status_t ccl_allreduce_hierarchical(const void* const* send, void* const* recv, int p, int group,
                                        size_t n, ccl_dtype_t dt, ccl_op_t op, void* stream);

/* Reduce-scatter ("dist_train": process k gets sum_i x_i^(k); ZeRO's key op).
 *   send[r]  p device pointers, each n elements.
 *   recv[k]  p device pointers; recv[k] holds len(k) elements: chunk k of the
 *            ring-ordered reduction.  In place is allowed only as
 *            recv[k] == send[k] + off(k) elements; other overlaps are errors. */
ccl_status_t ccl_reduce_scatter(const void* const* send, void* const* recv, int p, size_t n,
                                ccl_dtype_t dt, ccl_op_t op, void* stream);

/* All-gather ("Networks and Collective Communication" 4.1: each device
 * contributes one block and everyone gets the whole concatenation).
 *   send[k]  p device pointers; send[k] holds len(k) elements (block k).
 *   recv[r]  p device pointers, each n elements; block k lands at off(k).
 *            In place is allowed only as send[k] == recv[k] + off(k)
 *            elements.  Pure copy: bit-exact for every dtype.  With the
 *            environment variable CCL_FORCE_VARIANT=tma, calls where p divides
 *            n, blocks are >= 1 MiB and every buffer is 16-byte aligned device
 *            memory run on the bulk-copy engine (one read into shared memory,
 *            p bulk stores) instead of the default thread stores. */
ccl_status_t ccl_all_gather(const void* const* send, void* const* recv, int p, size_t n,
                            ccl_dtype_t dt, void* stream);

/* Broadcast ("Networks and Collective Communication" 4.1: the root's data is
 * copied to everyone).  send: the root's n elements; recv[r]: p outputs of n
 * elements; recv[root] == send is allowed (in place).  One read of the root's
 * data, p writes (on the bulk-copy engine under the all-gather's opt-in and
 * conditions, with n * bytes >= 1 MiB). */
ccl_status_t ccl_broadcast(const void* send, void* const* recv, int p, size_t n, ccl_dtype_t dt,
                           int root, void* stream);

/* Reduce (4.1: element-wise reduction, result only on the root).  The pages
 * fix no order for it; it is the ring's reduce-scatter followed by a gather
 * of the shards to the root, so recv holds exactly the bits every rank gets
 * from ccl_allreduce.  send[r]: p inputs of n elements; recv: the root's n
 * outputs; recv == send[root] is allowed (in place). */
ccl_status_t ccl_reduce(const void* const* send, void* recv, int p, size_t n, ccl_dtype_t dt,
                        ccl_op_t op, int root, void* stream);

/* Scatter ("dist_train", Scatter: the root holds [x_1, ..., x_p] and rank k
 * receives x_k).  send: the root's n elements; recv[k]: len(k) elements, chunk
 * k by the CHUNKS rule; recv[root] == send + off(root) is allowed. */
ccl_status_t ccl_scatter(const void* send, void* const* recv, int p, size_t n, ccl_dtype_t dt,
                         int root, void* stream);

/* Gather ("dist_train", Gather: rank k holds x_k; the root receives
 * [x_1, ..., x_p]).  send[k]: len(k) elements; recv: the root's n elements,
 * block k at off(k); send[root] == recv + off(root) is allowed. */
ccl_status_t ccl_gather(const void* const* send, void* recv, int p, size_t n, ccl_dtype_t dt,
                        int root, void* stream);

/* DDP gradient-bucket all-reduce with the average and the cast fused in
 * ("dist_train", Communication-Computation Overlap: DDP cuts gradients into
 * buckets of bucket_cap_mb = 25 and all-reduces each finished bucket).
 *   grads[r]    p device pointers, n fp32 gradients each.
 *   out_bf16[r] p device pointers, n bf16 each; no overlap with any grads
 *               buffer or other output is allowed (the cast halves the width).
 * out = bf16_round_nearest_even( fp32(ring_sum) * scale ); pass scale = 1/p
 * for the DDP average. */
ccl_status_t ccl_bucket_allreduce_scale_cast(const float* const* grads, void* const* out_bf16,
                                             int p, size_t n, float scale, void* stream);

/* All-to-all ("Networks and Collective Communication" 4.1: device i's block j
 * goes to device j, a transpose).  send[i]: n elements cut into p blocks by
 * the chunk rule; recv[j]: p * len(j) elements, block j of every source in
 * source order (the all-to-allv with counts[s][d] = len(d) and one-element
 * rows); applying it twice restores the inputs when p divides n.  The block
 * geometry follows from p and n, so every call is one kernel launch. */
ccl_status_t ccl_all_to_all(const void* const* send, void* const* recv, int p, size_t n, ccl_dtype_t dt,
                            void* stream);

/* All-to-all with per-pair counts: the MoE dispatch / combine block transpose
 * ("Networks and Collective Communication" 4.1: device i's block j goes to
 * device j; 7.4: MoE dispatch and combine).
 *   counts     HOST array of p*p row counts, counts[s*p + d] = rows that
 *              source s sends to destination d.
 *   send[s]    sum_d counts[s][d] rows of row_elems elements; the block for d
 *              starts at row sum_{d' < d} counts[s][d'].
 *   recv[d]    sum_s counts[s][d] rows; the block from s lands at row
 *              sum_{s' < s} counts[s'][d].
 * Combine is the same call on the received buffers with counts transposed.
 * Buffers must not overlap.  Bit-exact copy for every dtype.  The counts
 * travel to the kernel as a table of row prefixes inside its parameter
 * block (nothing is allocated): one launch for p <= 85, else one launch per
 * group of destinations that fits (p = 128: three).  While some source has
 * 2^32 rows or more the table takes 64-bit entries and half as many
 * destinations per launch. */
ccl_status_t ccl_all_to_allv(const void* const* send, const size_t* counts, void* const* recv,
                             int p, size_t row_elems, ccl_dtype_t dt, void* stream);

/* Diagnostic (no counterpart on the pages): which all-to-all kernel a call
 * of ccl_all_to_all / ccl_all_to_allv with the same arguments launches.
 * The pointers are only read as addresses (their 16-byte phases decide);
 * nothing is dereferenced, checked against the device or enqueued.
 * sm_count: the device's SM count, or <= 0 for the current device's.
 *   form        where the block bounds come from: CCL_A2A_SMALL (p <= 16,
 *               4 KB parameter block), CCL_A2A_PLAIN (the chunk rule, p > 16),
 *               CCL_A2A_TABLE32 / CCL_A2A_TABLE64 (row-prefix tables of
 *               32- / 64-bit entries, p > 16 or a source of 2^32 rows or more)
 *   shift       some block's source and destination differ in 16-byte phase
 *   stage       the units that straddle blocks go through the small-block
 *               stage in shared memory
 *   launches    kernel launches of the call (0: nothing to move)
 *   tile_bytes  destination tile of the first launch (4096, 8192, 16384 or
 *               32768: by the launch's destination bytes per SM)
 * Errors: as the call's own argument checks (p, dt, NULL pointers, sizes)
 * -> CCL_ERR_INVALID_ARG. */
typedef enum { CCL_A2A_SMALL = 0, CCL_A2A_PLAIN = 1, CCL_A2A_TABLE32 = 2, CCL_A2A_TABLE64 = 3 } ccl_a2a_form_t;
typedef struct {
  ccl_a2a_form_t form;
  int shift;
  int stage;
  int launches;
  unsigned tile_bytes;
} ccl_a2a_plan_t;
ccl_status_t ccl_all_to_all_plan(const void* const* send, void* const* recv, int p, size_t n, ccl_dtype_t dt,
                                 int sm_count, ccl_a2a_plan_t* plan);
ccl_status_t ccl_all_to_allv_plan(const void* const* send, const size_t* counts, void* const* recv, int p,
                                  size_t row_elems, ccl_dtype_t dt, int sm_count, ccl_a2a_plan_t* plan);

/* DDP gradient bucketing ("dist_train", Communication-Computation Overlap:
 * with bucket_cap_mb = 25 the gradients are cut into buckets in the order
 * backprop produces them, and a bucket is all-reduced as soon as all of its
 * gradients are ready).  Host only; nothing is enqueued.
 *   numel[i]      element count of gradient i, in the order gradients become
 *                 ready (DDP: the reverse of parameter registration order).
 *   elem_bytes    bytes per gradient element (4 for fp32).
 *   cap_bytes     bucket capacity in bytes (25 MiB for bucket_cap_mb = 25).
 *   bucket_of     out, count entries: bucket index of gradient i.
 *   offset        out, count entries: element offset of gradient i in its
 *                 bucket (a bucket is the contiguous concatenation of its
 *                 gradients, in order).
 *   bucket_numel  out, capacity count entries (may be NULL): elements per bucket.
 *   num_buckets   out: number of buckets.
 * Rule: a gradient joins the current bucket while the bucket stays within
 * cap_bytes, else it starts the next bucket; a gradient larger than the cap
 * gets a bucket of its own.  Errors: NULL outputs, elem_bytes == 0 or
 * cap_bytes < elem_bytes -> CCL_ERR_INVALID_ARG. */
ccl_status_t ccl_plan_buckets(const size_t* numel, size_t count, size_t elem_bytes,
                              size_t cap_bytes, uint32_t* bucket_of, size_t* offset,
                              size_t* bucket_numel, size_t* num_buckets);

/* Head <-> sequence all-to-all of sequence-parallel attention ("LLM
 * Distributed Training Collectives", Sequence Parallelism / Ulysses).
 * Forward (inverse == 0): send[r] is sequence shard r with every head,
 * [seq_per_rank, heads, head_dim]; recv[r] gets the whole sequence of head
 * group r, [p * seq_per_rank, heads / p, head_dim]:
 *   recv[r][s*seq_per_rank + t][h][:] = send[s][t][r*heads/p + h][:].
 * Inverse (inverse != 0): the same arguments describe the way back (send[r]
 * is head group r, recv[s] gets sequence shard s).  heads must be a multiple
 * of p.  Buffers must not overlap.  Pure copy, bit-exact. */
ccl_status_t ccl_all_to_all_heads(const void* const* send, void* const* recv, int p,
                                  size_t seq_per_rank, size_t heads, size_t head_dim,
                                  ccl_dtype_t dt, int inverse, void* stream);

/* ------------------------------------------------- MoE expert parallelism
 * "Networks and Collective Communication" section 7.4: every MoE layer does an
 * all-to-all dispatch (each token to the ranks holding the k experts it chose)
 * and an all-to-all combine; DeepSeek-V3 dispatches in FP8 and combines in
 * BF16.  p <= 64 virtual ranks, 1 <= k <= 16, expert e on rank e / (E/p),
 * hidden a multiple of 128, tokens * k < 2^31.  Token t of source s sends one
 * row per choice j; destination d holds its rows grouped by source, then
 * token, then choice, at row sum_{s' < s} counts[s'][d] + slot.
 *
 * ccl_moe_route: expert_ids[s] (device, tokens*k int32, token-major) ->
 *   counts (device p*p int64, rows source -> destination) and slots[s]
 *   (device, tokens*k int32; -1 for an id outside [0, E)).  One launch.
 * ccl_moe_dispatch: x[s] (device, tokens x hidden bf16) -> recv[d] (rows x
 *   hidden bf16, or e4m3 bytes when fp8 != 0, with recv_scales[d] = rows x
 *   hidden/128 fp32: scale = amax/448 per 128-element block, code =
 *   e4m3(x/scale) round-to-nearest-even, saturating).  recv_rows (host, p) is
 *   the row capacity of each recv[d]; rows beyond it are not written (read
 *   counts back to size the buffers).  recv_expert (may be NULL) receives each
 *   row's expert id.
 * ccl_moe_combine: y[d] (rows x hidden bf16 in dispatch layout, y_rows rows)
 *   -> out[s] (tokens x hidden bf16) = bf16(sum_j weights[s][t*k+j] * y_j),
 *   fp32 products and sums in choice order.  With weights 1/k (k a power of
 *   two) combine(dispatch(x)) == x. */
ccl_status_t ccl_moe_route(const int32_t* const* expert_ids, int p, size_t tokens, int k,
                           int num_experts, int64_t* counts, int32_t* const* slots, void* stream);

ccl_status_t ccl_moe_dispatch(const void* const* x, const int32_t* const* expert_ids,
                              const int64_t* counts, const int32_t* const* slots, int p,
                              size_t tokens, int k, int num_experts, size_t hidden, int fp8,
                              void* const* recv, const size_t* recv_rows, float* const* recv_scales,
                              int32_t* const* recv_expert, void* stream);

ccl_status_t ccl_moe_combine(const void* const* y, const size_t* y_rows,
                             const int32_t* const* expert_ids, const float* const* weights,
                             const int64_t* counts, const int32_t* const* slots, int p,
                             size_t tokens, int k, int num_experts, size_t hidden, void* const* out,
                             void* stream);

/* ------------------------------------------------------- literal ring engine
 * Executes the ring schedule as written: the reduce-scatter phase's p-1 steps
 * (rank r sends its partial of chunk (r-s-1) mod p to rank r+1, which adds its
 * own) and the all-gather phase's p-1 steps (rank r sends chunk (r-s) mod p),
 * one kernel launch per step, and counts the bytes each rank sends
 * ("Networks and Collective Communication" 5.1 and 4.3; "dist_train", Ring
 * Algorithm).  Results equal the fused entry points bit for bit.
 *
 * bytes_sent  HOST array of p entries, overwritten with the bytes each rank
 *             sent in this call (reduce-scatter partials travel as 4-byte
 *             fp32/int32; all-gather chunks travel in dt).  May be NULL.
 * workspace   device scratch for the working buffers; its required size is
 *             ccl_ring_literal_workspace_bytes(kind, p, n, dt) (0 -> may be
 *             NULL).  It must not overlap any send or recv buffer.
 * Buffers follow the same layout and aliasing rules as the fused calls. */

/* Bytes of workspace a literal call needs: all-reduce p*n*4 for bf16 (fp32
 * partials), else 0; reduce-scatter p*n*4; all-gather 0.  Returns 0 for
 * invalid arguments. */
size_t ccl_ring_literal_workspace_bytes(ccl_kind_t kind, int p, size_t n, ccl_dtype_t dt);

ccl_status_t ccl_ring_allreduce_literal(const void* const* send, void* const* recv, int p,
                                        size_t n, ccl_dtype_t dt, ccl_op_t op,
                                        uint64_t* bytes_sent, void* workspace,
                                        size_t workspace_bytes, void* stream);

ccl_status_t ccl_ring_reduce_scatter_literal(const void* const* send, void* const* recv, int p,
                                             size_t n, ccl_dtype_t dt, ccl_op_t op,
                                             uint64_t* bytes_sent, void* workspace,
                                             size_t workspace_bytes, void* stream);

ccl_status_t ccl_ring_all_gather_literal(const void* const* send, void* const* recv, int p,
                                         size_t n, ccl_dtype_t dt, uint64_t* bytes_sent,
                                         void* stream);

/* ------------------------------------------- allocation-free reduce-scatter
 * The pages have no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory for the workspace that
 * ccl_ring_reduce_scatter_literal needs: code that runs inside a custom
 * allocator or memory-pool callback (allocating there would re-enter the
 * allocator), a host application that owns all device memory and does not let
 * libraries allocate, or a process that reserved its memory budget up front
 * and must not fail or fragment later.
 *
 * Same arguments, results and byte counts as ccl_ring_reduce_scatter_literal,
 * without the workspace: the p*n*4 bytes of working buffers come from a
 * scratch array built into the library (a file-scope static __device__ array
 * of CCL_STATIC_SCRATCH_BYTES).  Every GPU that loads the library holds that
 * array until the process exits.  The call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine).
 *   - p*n*4 > CCL_STATIC_SCRATCH_BYTES (p*n above 8,388,608 elements)
 *     -> CCL_ERR_INVALID_ARG, checked before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and looks it up again
 *     when the current context is no longer the one the address came from
 *     (after cudaDeviceReset re-creates the device's context).  Make that
 *     first call before any stream capture begins.
 *   - The array's memory is reserved when the library's device code is
 *     loaded into a context.  With the CUDA runtime's default lazy module
 *     loading that happens at the first call, and that first call can fail
 *     with CCL_ERR_CUDA if the device has no memory left at that moment.
 *     Callers that must not fail later make one small warm-up call (n >= 1)
 *     at initialisation; every later call on that context allocates nothing.
 *   - All calls share the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero: each call overwrites every byte
 *     it reads).  Calls whose GPU work overlaps -- on different streams, or
 *     from host threads that do not order their streams -- race on the array;
 *     the caller must serialise them. */
#define CCL_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

ccl_status_t ccl_ring_reduce_scatter_literal_noalloc(const void* const* send, void* const* recv,
                                                     int p, size_t n, ccl_dtype_t dt,
                                                     ccl_op_t op, uint64_t* bytes_sent,
                                                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CCL_H_ */
