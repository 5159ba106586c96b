/*
 * zipage.h — C ABI of the Compressed-PagedAttention compression pass (sm_103a).
 *
 * The operation is the compression step of Zipage ("Zipage: Maintain High Request Concurrency
 * for LLM Reasoning through Compressed PagedAttention", summaries on gist.science; zh page §2.1,
 * de page §2 "Methodik", es page §2 "Metodología", fr page §2.A–§2.E).  A request that holds
 * N_max blocks of b tokens and has filled its last block is compressed: every cached token of
 * every layer and KV head is scored, the top k = (N_max-1)*b per KV head are kept in their
 * original order and rewritten compactly into the first N_max-1 blocks (or into newly
 * allocated target blocks where the leading blocks are shared prefix blocks), and the last
 * block is released.
 *
 * Conventions
 *   - Every device buffer is allocated and owned by the caller; the library never frees
 *     caller memory.  "device" below means a pointer into GPU global memory, "host" a pointer
 *     into CPU memory.
 *   - Calls that launch work are asynchronous on the given stream and return as soon as the
 *     launch is queued.  Host-side argument errors are returned immediately and nothing is
 *     launched.  Errors that only the GPU can see (a block id outside the pool, a seq_len or
 *     query slot out of range, a wait that gave up) are written to the error word at the
 *     start of the caller's workspace; the unit concerned is skipped, never half-written.
 *     Read it with zp_read_error().
 *   - bf16 is passed as raw 16-bit storage (`uint16_t`): the library does not depend on any
 *     C++ bf16 type.
 *   - KV pool layout (bf16): [num_layers][num_blocks][2][num_kv_heads][block_size][head_dim],
 *     index 0 of the third dimension = K, 1 = V.  Each (layer, block, K|V, head) tile of
 *     block_size*head_dim values is contiguous.
 */
#ifndef ZIPAGE_H
#define ZIPAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t zp_status;
enum {
  ZP_OK = 0,
  ZP_ERR_INVALID_ARG = 1,  /* a host-side argument is out of range or inconsistent */
  ZP_ERR_NO_BLOCKS = 2,    /* the allocator cannot satisfy the request; nothing changed */
  ZP_ERR_BAD_TABLE = 3,    /* (device) a block id, seq_len or query slot is out of range */
  ZP_ERR_TIMEOUT = 4,      /* (device) a bounded wait inside a kernel gave up */
  ZP_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  ZP_ERR_UNSUPPORTED = 6,  /* valid arguments outside what the library implements */
  ZP_ERR_TOO_LARGE = 7     /* the call needs more scratch than zp_paged_decode_attn_static holds */
};

/* Opaque stream handle: a cudaStream_t (CUstream) passed through as a pointer, NULL = legacy
 * default stream. */
typedef void* zp_stream;

/* Method parameters.  The pages fix N_max, b and w; alpha, beta, decay and scale are readings
 * (the pages name the three scores but print no weights). */
typedef struct zp_params {
  int32_t num_layers;     /* layers in the pool */
  int32_t num_q_heads;    /* H_q */
  int32_t num_kv_heads;   /* H_kv; H_q % H_kv == 0, G_q = H_q / H_kv query heads per KV head */
  int32_t head_dim;       /* d: 64 or 128 */
  int32_t block_size;     /* b: 16 or 32 tokens per block */
  int32_t n_max;          /* N_max: block cap per request, >= 2 */
  int32_t window;         /* w: observation-window length, 1 <= w <= (n_max-1)*b */
  float alpha;            /* weight of the carried global score */
  float beta;             /* weight of the redundancy score (subtracted) */
  float decay;            /* global-score decay: G' = decay*G + attn */
  float scale;            /* logit scale, normally 1/sqrt(d) */
  int32_t protect_window; /* 1: the last w tokens are always kept */
  int32_t causal;         /* 1: window row i sees keys t <= L-w+i */
} zp_params;

typedef struct zp_kv_pool {
  void* base;             /* device, bf16, layout above; 16-byte aligned */
  int64_t num_blocks;     /* blocks per layer */
} zp_kv_pool;

typedef struct zp_seq_meta {
  int32_t num_requests;       /* R: requests compressed by this call */
  int32_t max_blocks;         /* row stride of the block tables (>= ceil(L_max / b)) */
  const int32_t* seq_len;     /* device [R]: cached tokens L of each request, k < L <= L_max
                                 (L = n_max*b at the decode trigger; a request that left a long
                                 prefill may hold more, zh §2.1) */
  const int32_t* qslot;       /* device [R]: query slot of each request, 0 <= qslot < num_qslots */
  const int32_t* dst_tables;  /* device [R][max_blocks]: where survivors go; equals the source
                                 table except at target blocks (zp_plan_compress) */
  int32_t max_seq_len;        /* L_max: the longest seq_len of the call (<= 16384), or 0 for
                                 n_max*b.  It is also the row length of global_scores and of
                                 the zp_debug arrays. */
  const int32_t* n_max_per_req; /* device [R] or NULL: per-request block budgets
                                   2 <= N_max_r <= params.n_max (the pages' per-request dynamic
                                   budgets, de §5); request r keeps k_r = (N_max_r-1)*b tokens per
                                   head.  NULL: every request uses params.n_max. */
  int32_t layer_begin;        /* the call compresses layers [layer_begin, layer_begin +
                                 layer_count) of every request; layer_count 0 means all layers
                                 (then layer_begin must be 0).  Layer indices into the pool,
                                 obs_q, global_scores and the zp_debug arrays stay absolute, so a
                                 caller can compress a model layer by layer (for instance while
                                 the next layer's blocks are still being copied in). */
  int32_t layer_count;
} zp_seq_meta;

/* Optional per-token outputs, each device [R][num_layers][num_kv_heads][L_max] (row-major),
 * any field may be NULL.  attn = window attention score, redund = Lightning redundancy,
 * score = combined score S (+inf on protected tokens), keep = 1 if kept else 0. */
typedef struct zp_debug {
  float* attn;
  float* redund;
  float* score;
  int32_t* keep;
} zp_debug;

/* ---------------------------------------------------------------------------------------
 * Compression pass (zh §2.1 core mechanism; zh §2.3 cross-layer parallel compression).
 *
 * One launch covers every (request, layer, kv head) unit.  For unit (r, l, h) with
 * L = seq_len[r] cached tokens read through block_tables[r]:
 *   attn[t]  = mean over the w*G_q window rows (i, g) of softmax_t(scale*<q_{i,g}, k_t>),
 *              row i being the query of position L-w+i (causal if params.causal);
 *   R[t]     = mean cosine similarity of k_t to the other keys of its block (Lightning);
 *   S[t]     = attn[t] + alpha*G[t] - beta*R[t]  (+inf for the last w if protect_window);
 *   keep the k = (n_max-1)*b tokens first in (S desc, t asc); survivor j (ascending t) is
 *   copied bit for bit to logical slot j of dst_tables[r]; G'[j] = decay*G[src_j] + attn[src_j]
 *   for j < k and 0 for k <= j < L.
 * Arguments
 *   pool          device KV pool, read through block_tables and written through dst_tables.
 *   block_tables  device [R][max_blocks] int32, physical block of each logical block.
 *   meta          host struct with device pointers (see zp_seq_meta).
 *   obs_q         device bf16 [num_qslots][num_layers][w][H_q][d]: the window queries;
 *                 16-byte aligned.
 *   num_qslots    M, number of query slots in obs_q and global_scores.
 *   global_scores device fp32 [num_qslots][num_layers][H_kv][L_max], updated in place.
 *   params        host.
 *   dbg           host struct or NULL.
 *   workspace     device, >= zp_compress_workspace_size() bytes, 256-byte aligned; holds the
 *                 error word (cleared by the call before any kernel runs), the unit counters,
 *                 and the request order grouped by length that the call builds when the
 *                 requests' lengths may need clusters of different sizes (max_seq_len above
 *                 n_max*b, or per-request budgets): each group then runs in a launch of its
 *                 own cluster size.  One workspace serves one call in flight at a time.
 *   stream        stream to launch on.
 * Source and destination blocks of different requests must not overlap (shared prefix
 * blocks are only read).  Returns ZP_OK once queued.
 * A unit with bad metadata (ZP_ERR_BAD_TABLE) is skipped whole and every other unit is
 * compressed.  ZP_ERR_TIMEOUT (a wait inside the kernel gave up after 2 s, which only a broken
 * device or driver state produces) means the call failed: the pool and the global scores of
 * the units the stalled cluster went on to process are undefined.
 * --------------------------------------------------------------------------------------- */
zp_status zp_compress(const zp_kv_pool* pool, const int32_t* block_tables, const zp_seq_meta* meta,
                      const uint16_t* obs_q, int32_t num_qslots, float* global_scores,
                      const zp_params* params, const zp_debug* dbg, void* workspace,
                      size_t workspace_bytes, zp_stream stream);

/* Bytes of workspace zp_compress needs.  max_seq_len 0 means n_max*b.  Up to 4096 tokens: a
 * 512-byte header (error word, unit counters, length groups) and 4 bytes per request (the
 * grouped request order), rounded up to 256.  Above 4096: 256 bytes and the scratch of the
 * multi-pass form (per unit: 1 KB per 256-token chunk and 16 bytes per token). */
size_t zp_compress_workspace_size(const zp_params* params, int32_t num_requests, int32_t max_seq_len);

/* Kernel launches one zp_compress call makes for this max_seq_len (0 means n_max*b) and
 * budget form (per_request_budgets != 0 when meta->n_max_per_req is given): 1 when every
 * request fits one cluster size, 1 + G when the call groups the requests by length into G
 * cluster sizes (the grouping kernel and one launch per size, empty groups included), 4 for
 * the multi-pass form (max_seq_len above 4096).  0 for arguments zp_compress rejects on its
 * sizes.  Host only; launches nothing. */
int32_t zp_compress_kernel_launches(const zp_params* params, int32_t max_seq_len, int32_t per_request_budgets);

/* ---------------------------------------------------------------------------------------
 * Original (all-pairs) redundancy score — the ablation of the Lightning Redundancy Score
 * (zh §2.1 and es §2: the original compares every pair of the N*b cached tokens, O(N^2 b^2),
 * where Lightning compares the b^2 pairs of each block, O(N b^2); de §2: the original needs
 * the full similarity matrix).  Not used by zp_compress: it exists to measure what Lightning
 * saves.
 *   redund[r][l][h][t] = (1/(L-1)) * sum over j < L, j != t of cos(k_t, k_j),
 * cosine with norms clamped at 1e-12, for t < L = seq_len[r]; 0 for t >= L and when L < 2.
 * Arguments
 *   pool          device KV pool, read through block_tables (only K is read).
 *   block_tables  device [R][max_blocks] int32.
 *   meta          host struct: num_requests, max_blocks, seq_len (device [R]) and
 *                 max_seq_len (the row length L_max of redund; n_max*b when 0).  The other
 *                 fields are ignored.  L_max <= 4096.
 *   params        host; num_layers, num_kv_heads, head_dim (64 or 128), block_size (16 or
 *                 32) and n_max are used.
 *   redund        device fp32 [R][num_layers][H_kv][L_max], written.
 *   workspace     device, >= zp_redundancy_workspace_size(params, R, max_seq_len) bytes,
 *                 256-byte aligned: the error word (a block id outside the pool or a seq_len
 *                 above L_max: ZP_ERR_BAD_TABLE; a wait that gave up: ZP_ERR_TIMEOUT), then
 *                 the squared key norms that a pre-pass computes.
 * Returns ZP_OK once queued.
 * --------------------------------------------------------------------------------------- */
zp_status zp_redundancy_all_pairs(const zp_kv_pool* pool, const int32_t* block_tables, const zp_seq_meta* meta,
                                  const zp_params* params, float* redund, void* workspace,
                                  size_t workspace_bytes, zp_stream stream);

/* Bytes of workspace zp_redundancy_all_pairs needs: the error word and one fp32 squared key
 * norm per (request, layer, kv head, token < L_max). */
size_t zp_redundancy_workspace_size(const zp_params* params, int32_t num_requests, int32_t max_seq_len);

/* ---------------------------------------------------------------------------------------
 * Paged decode attention over the (compacted) cache — the consumer that runs on the main
 * stream while compression runs on a side stream (zh §2.1 asynchronous compression and
 * decoding; fr §2.D).
 *   out[r][qh] = softmax_t(scale*<q[r][qh], k_t>) . v_t over t < seq_lens[r], with keys and
 *   values of kv head qh / G_q of `layer`, read through block_tables[r].
 * q, out: device bf16 [B][H_q][d]; block_tables device [B][max_blocks]; seq_lens device [B]
 * (1 <= seq_len <= max_blocks*b).  workspace >= zp_paged_decode_workspace_size() bytes,
 * 256-byte aligned (split-KV partials + error word).
 * --------------------------------------------------------------------------------------- */
zp_status zp_paged_decode_attn(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                               const int32_t* block_tables, const int32_t* seq_lens, int32_t B,
                               int32_t max_blocks, uint16_t* out, const zp_params* params,
                               void* workspace, size_t workspace_bytes, zp_stream stream);

size_t zp_paged_decode_workspace_size(const zp_params* params, int32_t B, int32_t max_blocks);

/* Kernel launches one zp_paged_decode_attn call with these sizes makes on the current device:
 * 1 when every request fits one split (the split size is chosen per call from B, H_kv,
 * max_blocks and the device's SM count), 2 with the kernel that merges the splits.  0 for
 * invalid arguments.  Host only; launches nothing. */
int32_t zp_paged_decode_kernel_launches(const zp_params* params, int32_t B, int32_t max_blocks);

/* ---------------------------------------------------------------------------------------
 * zp_paged_decode_attn without any device allocation by anyone.  The paper has no
 * counterpart: this is a convenience of this library.
 *
 * For callers that cannot allocate device memory: a host runtime that owns every device
 * buffer through its own pool and hands this library no allocator, a serving loop that must
 * not call cudaMalloc (which can synchronise the whole device) in its hot path, or a process
 * that must know its complete device footprint when the library is loaded.
 *
 * Same operation and arguments as zp_paged_decode_attn, except that the split-KV partials
 * live in a fixed 16 MiB array inside the library (held by every GPU that loads it until the
 * process exits), so no workspace is passed.  A call needs
 * B * H_q * ceil(max_blocks / 32) * (head_dim + 2) * 4 bytes of it, at most 16 MiB - 256 B;
 * larger calls return ZP_ERR_TOO_LARGE and launch nothing.
 *   dev_status  device int32 written with the call's device-side status (0, or
 *               ZP_ERR_BAD_TABLE for a block id outside the pool or a bad seq_len); it is
 *               cleared on the stream before the kernel runs.  May be NULL, in which case
 *               device-side errors are not reported.
 * The first call on a device looks up the array's device address for that device (with the
 * device current); make that first call before any stream capture.  The address is kept for
 * the life of the process: after cudaDeviceReset, or anything else that destroys the device's
 * primary context, do not call this entry point on that device again in the same process (the
 * library would be reloaded at an address it does not know).  Every call shares the
 * one array: calls whose kernels may overlap on the GPU (different streams without an
 * ordering between them) race on it and must be serialised by the caller.  The call
 * allocates and frees nothing.
 * --------------------------------------------------------------------------------------- */
zp_status zp_paged_decode_attn_static(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                                      const int32_t* block_tables, const int32_t* seq_lens, int32_t B,
                                      int32_t max_blocks, uint16_t* out, const zp_params* params,
                                      int32_t* dev_status, zp_stream stream);

/* Test hook of the device-side failure detection (bounded waits).  Not for production use.
 * Same operation, arguments and workspace as zp_paged_decode_attn, plus stall_limit_ns
 * (1 .. 10^9).  Before its first chunk of K/V, every warp of the decode kernel first waits, for
 * at most stall_limit_ns, on a shared-memory barrier that nothing ever completes.  That wait
 * runs out, and the kernel then takes the path of any wait that gives up: it waits (bounded,
 * 2 s) for the copies it has already issued, writes its outputs from the keys it has folded in
 * (none: zeros) and records ZP_ERR_TIMEOUT in the workspace's error word, which
 * zp_read_error() returns.  Nothing faults or hangs, and the context stays usable.  Returns
 * ZP_OK once queued. */
zp_status zp_test_decode_stalled(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                                 const int32_t* block_tables, const int32_t* seq_lens, int32_t B,
                                 int32_t max_blocks, uint16_t* out, const zp_params* params,
                                 void* workspace, size_t workspace_bytes, int64_t stall_limit_ns,
                                 zp_stream stream);

/* Test hook of the same kind for the compression pass.  Not for production use.  Same
 * operation, arguments and workspace as zp_compress (no debug outputs), plus stall_limit_ns
 * (1 .. 10^9); meta->max_seq_len must exceed 4096, so that the call takes the multi-pass form,
 * whose CTAs exchange nothing with one another (ZP_ERR_INVALID_ARG otherwise).  Before its first
 * chunk, thread 0 of every CTA of the statistics launch first waits, for at most stall_limit_ns,
 * on a shared-memory barrier that nothing ever completes.  That wait runs out, and the CTA then
 * takes the path of any wait that gives up: its chunks get empty row statistics, it waits
 * (bounded, 2 s) for the copy it has in flight and records ZP_ERR_TIMEOUT in the error word.
 * The later launches of the call run as usual, so, as for any ZP_ERR_TIMEOUT, the pool rows and
 * global scores of the call's units are undefined afterwards; nothing is written outside the
 * call's buffers.  Nothing faults or hangs, and the context stays usable.  Returns ZP_OK once
 * queued. */
zp_status zp_test_compress_stalled(const zp_kv_pool* pool, const int32_t* block_tables, const zp_seq_meta* meta,
                                   const uint16_t* obs_q, int32_t num_qslots, float* global_scores,
                                   const zp_params* params, void* workspace, size_t workspace_bytes,
                                   int64_t stall_limit_ns, zp_stream stream);

/* Synchronises `stream`, copies the error word at the start of `workspace` to *out_status and
 * clears it.  Returns ZP_ERR_CUDA if the copy fails. */
zp_status zp_read_error(void* workspace, zp_stream stream, zp_status* out_status);

/* ---------------------------------------------------------------------------------------
 * Block allocator with reference counts (the PagedAttention block manager with prefix
 * sharing: zh §2.2, de §2 "Prefix Caching", fr §2.C).  Host only.  Free ids are handed out
 * lowest first so that plans are deterministic.  Every call is all-or-nothing.
 * --------------------------------------------------------------------------------------- */
typedef struct zp_alloc zp_alloc;

zp_status zp_alloc_create(int64_t num_blocks, zp_alloc** out);
void zp_alloc_destroy(zp_alloc* a);
/* n fresh blocks (refcount 1) into ids[n]; ZP_ERR_NO_BLOCKS if fewer than n are free. */
zp_status zp_alloc_blocks(zp_alloc* a, int32_t n, int32_t* ids);
/* Marks the given free ids as allocated (refcount 1), e.g. to restore a saved state;
 * ZP_ERR_INVALID_ARG if any is out of range, repeated or not free. */
zp_status zp_alloc_reserve(zp_alloc* a, const int32_t* ids, int32_t n);
zp_status zp_incref(zp_alloc* a, const int32_t* ids, int32_t n);
/* A block whose refcount reaches 0 becomes free.  ZP_ERR_INVALID_ARG on a free id. */
zp_status zp_decref(zp_alloc* a, const int32_t* ids, int32_t n);
/* Deferred decref: applied once all work queued on `stream` before this call has finished
 * (the library records its own event).  stream may be NULL only if no CUDA work reads the
 * blocks; then the decref is applied at once. */
zp_status zp_decref_after(zp_alloc* a, const int32_t* ids, int32_t n, zp_stream stream);
/* Applies the deferred decrefs whose work has finished (non-blocking). */
zp_status zp_alloc_poll(zp_alloc* a);
/* Waits for all deferred decrefs and applies them. */
zp_status zp_alloc_drain(zp_alloc* a);
/* Test hook (host-side fault injection): the nth_call-th allocating call from now returns
 * ZP_ERR_NO_BLOCKS without changing anything; 0 disables. */
zp_status zp_alloc_inject_failure(zp_alloc* a, int64_t nth_call);
int32_t zp_refcount(const zp_alloc* a, int32_t id);   /* -1 if id out of range */
int64_t zp_num_free(const zp_alloc* a);
int64_t zp_num_pending(const zp_alloc* a);           /* blocks waiting in deferred decrefs */

/* Plan of one compression (zh §2.2 / fr §2.C target blocks).  host_tables, host_dst_tables:
 * host [R][max_blocks].  For each request and each logical block i < n_max-1 the destination
 * is the same physical block unless its refcount is > 1 (shared prefix block), in which case
 * it is a freshly allocated target block.  Entries i >= n_max-1 are copied unchanged.
 * Transactional: ZP_ERR_NO_BLOCKS leaves the allocator unchanged. */
zp_status zp_plan_compress(zp_alloc* a, const int32_t* host_tables, int32_t R, int32_t max_blocks,
                           int32_t n_max, int32_t* host_dst_tables);
/* As zp_plan_compress with a per-request budget host_n_max[R] (2 <= N_max_r <= max_blocks). */
zp_status zp_plan_compress_budgets(zp_alloc* a, const int32_t* host_tables, int32_t R, int32_t max_blocks,
                                   const int32_t* host_n_max, int32_t* host_dst_tables);

/* After the compression launched on `stream`: for each request, decref every replaced shared
 * block (old != new for i < n_max-1) and every old block past the first n_max-1
 * (old[n_max-1 .. ceil(seq_len/b)) — the last block at the decode trigger, more after a
 * prefill), deferred until the work queued on `stream` has finished (the kernel still reads
 * those blocks).  host_seq_len: host [R], or NULL when every request holds n_max blocks. */
zp_status zp_commit_compress(zp_alloc* a, const int32_t* old_tables, const int32_t* new_tables,
                             int32_t R, int32_t max_blocks, int32_t n_max, int32_t block_size,
                             const int32_t* host_seq_len, zp_stream stream);
/* As zp_commit_compress with a per-request budget host_n_max[R] (NULL: n_max for all). */
zp_status zp_commit_compress_budgets(zp_alloc* a, const int32_t* old_tables, const int32_t* new_tables,
                                     int32_t R, int32_t max_blocks, const int32_t* host_n_max, int32_t n_max,
                                     int32_t block_size, const int32_t* host_seq_len, zp_stream stream);

/* ---------------------------------------------------------------------------------------
 * Hybrid scheduler (zh §2.2, de §2 "Hybrid Scheduling", es §2, fr §2.B).  Host only.
 *
 * Plans engine steps around the compression pass: only the first num_slots running requests
 * (admission order) hold a query slot; requests below n_max blocks, or whose last block still
 * has room, decode without one; a request at n_max blocks with a full last block (or longer,
 * after a prefill) compresses if it holds a slot and waits otherwise; when a block cannot be
 * allocated the most recently admitted request without a slot is preempted (it returns to the
 * front of the queue and recomputes); with none left the step runs in restricted mode (only
 * slot holders grow).  Blocks come from the given allocator; compressions keep the first
 * n_max-1 blocks and release the rest when the next step applies them.
 * --------------------------------------------------------------------------------------- */
typedef struct zp_sched zp_sched;

typedef struct zp_sched_config {
  int32_t n_max;        /* block cap per request */
  int32_t block_size;   /* b */
  int32_t num_slots;    /* M query slots */
  int32_t max_running;  /* cap on running requests, 0 = none */
} zp_sched_config;

/* The plan of one step; the arrays belong to the scheduler and stay valid until the next
 * zp_sched_step or zp_sched_destroy. */
typedef struct zp_sched_plan {
  int32_t num_decode;           /* requests that decode one token */
  const int32_t* decode_ids;
  int32_t num_compress;         /* requests whose compression runs this step (async) */
  const int32_t* compress_ids;
  int32_t num_prefill;          /* requests admitted this step */
  const int32_t* prefill_ids;
  int32_t num_preempted;        /* requests preempted this step */
  const int32_t* preempted_ids;
  int32_t restricted;           /* 1: this step ran in restricted mode */
} zp_sched_plan;

typedef struct zp_sched_request_info {
  int32_t state;                /* 0 waiting, 1 running, 2 finished */
  int32_t seq_len;              /* cached tokens */
  int32_t generated;            /* tokens decoded so far */
  int32_t num_blocks;
  const int32_t* table;         /* host [num_blocks], valid until the next step */
  int32_t has_slot;
  int32_t preemptions;
} zp_sched_request_info;

typedef struct zp_sched_stats {
  int64_t steps, submitted, admitted, finished, decoded_tokens, compressions, preemptions, slot_waits,
      restricted_steps, blocks_in_use;
  int32_t running;
} zp_sched_stats;

zp_status zp_sched_create(zp_alloc* alloc, const zp_sched_config* cfg, zp_sched** out);
void zp_sched_destroy(zp_sched* s);
/* Queues a request of prompt_len tokens that will decode gen_len tokens; *req_id = its id. */
zp_status zp_sched_submit(zp_sched* s, int32_t prompt_len, int32_t gen_len, int32_t* req_id);
/* Applies the previous step's plan (decoded tokens, compressions, finished requests) and
 * plans the next one. */
zp_status zp_sched_step(zp_sched* s, zp_sched_plan* plan);
zp_status zp_sched_request(const zp_sched* s, int32_t req_id, zp_sched_request_info* info);
zp_status zp_sched_get_stats(const zp_sched* s, zp_sched_stats* out);

/* Library version, for the binding's sanity check. */
int32_t zp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZIPAGE_H */
