/*
 * msa.h -- C ABI of libmsa.so: Multi-Segment Attention (MSA) on one B300 (sm_103a).
 *
 * Source: "Multi-Segment Attention: Enabling Efficient KV-Cache Management for
 * Faster Large Language Model Serving" (Shi, Chen, Chen, Miao, Cui), abstract,
 * Fig. 1 / Eq. 1 (attention), Fig. 4 / section 4.1 (non-contiguous cache segments
 * are disjoint KV regions), Fig. 5 (MSA).
 *
 * What MSA computes.  A query chunk -- recomputed evicted KV blocks plus new tokens,
 * each at its ORIGINAL position -- attends exactly (Eq. 1, scale 1/sqrt(d)) over a
 * KV context that is the union of many non-contiguous segments: cached paged blocks
 * plus the chunk's own freshly computed K/V, with a causal mask by original position
 * (key position <= query position, the query itself included).  Query head h reads
 * KV head h / (Hq/Hkv).  Outputs are O (bf16) and LSE = ln(sum_j exp(scale*q.k_j))
 * (fp32, natural log).  Decode: the newest token of each sequence (its own K/V
 * already in the pool) attends over every KV token of its sequence.
 *
 * Conventions.
 *  - All tensors named "device" are device pointers owned by the caller.  The
 *    library allocates no device memory at run time; it owns the opaque host plan
 *    object and, for msa_decode_no_alloc only, one fixed 8 MiB device array that is
 *    part of the loaded module.
 *  - Launch functions are asynchronous on the given stream; they return argument and
 *    launch errors at once.  Errors found on the device (a bounded wait that ran out)
 *    are written to the workspace status word and read by msa_get_status.
 *  - bf16 tensors are raw IEEE bfloat16 (uint16) arrays, row-major, densely packed.
 *  - All validation of the layout happens in msa_plan_create.
 *  - Plans are immutable after creation and may be used from several threads.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = -1,   /* null pointer, bad count, unsorted q_pos, inconsistent run */
  MSA_ERR_UNSUPPORTED = -2,   /* head_dim not in {64,128}, block_size != 16, Hq % Hkv != 0 */
  MSA_ERR_POS_OVERLAP = -3,   /* two KV tokens of one sequence share an original position */
  MSA_ERR_BLOCK_OOB = -4,     /* block id outside [0, num_pool_blocks) or logical block outside the row */
  MSA_ERR_WORKSPACE = -5,     /* workspace or output buffer too small / misaligned */
  MSA_ERR_CUDA = -6,          /* a CUDA runtime call failed (launch, copy, tensor map) */
  MSA_ERR_TIMEOUT = -7,       /* a device wait ran past its bound; the kernel gave up */
  MSA_ERR_MODE = -8           /* plan built for the other mode */
} msa_status_t;

typedef enum { MSA_PREFILL = 0, MSA_DECODE = 1 } msa_mode_t;

/* One segment: a run of `num_blocks` logical blocks of row `seq` of the block table,
 * starting at logical block `first_logical_block`, whose original positions are
 * consecutive: block_pos[bt[k+1]] == block_pos[bt[k]] + 16, and only the last block
 * of a run may hold fewer than 16 tokens (section 4.1: a cache segment is one
 * disjoint KV region; the paged block layout follows the paged KV cache the paper
 * builds on). */
typedef struct {
  int32_t seq;
  int32_t first_logical_block;
  int32_t num_blocks;
} msa_segment_t;

typedef struct {
  int32_t num_heads_q;        /* Hq */
  int32_t num_heads_kv;       /* Hkv, Hq % Hkv == 0 */
  int32_t head_dim;           /* d, 64 or 128 */
  int32_t block_size;         /* tokens per pool block, must be 16 */
  int32_t decode_split_blocks;/* decode: pool blocks per split-KV work unit, 0 = automatic */
  int32_t decode_min_ctas;    /* decode: target number of CTAs when automatic, 0 = 16 x SMs */
  int32_t prefill_ctas;       /* prefill: CTAs of the persistent launch the work is balanced
                                 over (one per SM), 0 = 148 (the B300's SM count) */
  int32_t chunk_queries_only; /* prefill: 0 = the chunk's rows are queries AND keys (MSA);
                                 1 = queries only: the KV context is the pool segments alone
                                 (partial attention over a subset of the context, e.g. one
                                 segment, for a log-sum-exp merge; a query that sees no key
                                 gets O = 0 and LSE = -inf) */
  int32_t reserved[2];        /* must be 0 */
} msa_plan_opts_t;

typedef struct msa_plan msa_plan_t;

typedef struct {
  int64_t useful_flops;       /* 4 * d * Hq * number of visible (query, key) pairs */
  int64_t kv_tokens;          /* KV tokens over all sequences (pool + chunk) */
  int64_t algorithmic_bytes;  /* decode: K/V + Q + O + LSE + block metadata bytes read/written once */
  int32_t num_kv_tiles;
  int32_t num_q_tiles;
  int32_t num_work_items;     /* prefill CTA work items, or decode split units x Hkv */
  int32_t num_tile_pairs;     /* prefill: non-skipped (query tile, KV tile) pairs x heads/2 */
  int32_t num_partial_pairs;
  int32_t num_splits;         /* decode split units (before x Hkv) */
  int32_t num_prefill_ctas;   /* prefill: CTAs of the launch */
  int32_t num_split_items;    /* prefill: work items cut into several pieces (merged on device) */
} msa_plan_stats_t;

/* Build a plan on the host (no CUDA call).  Inputs are host arrays, copied.
 *   segs[num_segs]                      segment descriptors, any order
 *   block_table[num_seqs * max_blocks_per_seq]  physical block of each logical block
 *   block_pos[num_pool_blocks]          original position of token 0 of each block
 *   block_fill[num_pool_blocks]         valid tokens of each block (1..16 when referenced)
 *   cu_q[num_seqs+1], q_pos[cu_q[num_seqs]]  prefill: query rows of each sequence and
 *                                       their original positions, strictly ascending per
 *                                       sequence; decode: cu_q must be 0..num_seqs (one
 *                                       query per sequence), q_pos may be NULL.
 * Errors: INVALID_ARG, UNSUPPORTED (also: num_pool_blocks * Hkv * 16 or, in prefill,
 * total query rows * Hkv above 2^31 - 1, since the kernels address the pool and the chunk
 * by 32-bit TMA row coordinates), POS_OVERLAP (pool and chunk positions of one sequence
 * repeat), BLOCK_OOB.  On error *out is NULL. */
msa_status_t msa_plan_create(const msa_plan_opts_t* opts, msa_mode_t mode, int32_t num_seqs,
                             const msa_segment_t* segs, int32_t num_segs,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* block_pos, const int32_t* block_fill,
                             int32_t num_pool_blocks,
                             const int32_t* cu_q, const int32_t* q_pos,
                             msa_plan_t** out);
void msa_plan_destroy(msa_plan_t* plan);

/* Bytes of the plan's device image; the caller allocates a device buffer of at least
 * this size (16-byte aligned) and fills it with msa_plan_upload (async copy on
 * `stream`; the plan must outlive the copy). */
size_t msa_plan_device_bytes(const msa_plan_t* plan);
msa_status_t msa_plan_upload(const msa_plan_t* plan, void* plan_dev, size_t bytes, cudaStream_t stream);

/* Workspace: status word, merge counters and partial results (decode split-KV units;
 * prefill work items cut into pieces).  The caller
 * allocates msa_workspace_bytes (256-byte aligned) and calls msa_workspace_init once
 * before first use (it zeroes the buffer on `stream`); the kernels leave it re-usable.
 * A workspace must not be shared by launches that may overlap. */
size_t msa_workspace_bytes(const msa_plan_t* plan);
msa_status_t msa_workspace_init(void* workspace, size_t bytes, cudaStream_t stream);

/* Canonical plan as int32 (the bit-exact indexing contract):
 *   header  [mode, num_seqs, n_tok, n_kt, n_qt, n_cls]
 *   n_tok x (src, id, offset, pos)     canonical KV order, each sequence in turn;
 *                                      src 0 = pool (id = physical block, offset = slot),
 *                                      src 1 = chunk (id = global query row, offset 0)
 *   n_kt  x (seq, src, tok_begin, n_tok, minpos, maxpos)   prefill KV tiles: the
 *                                      sequence's keys in position order as units of <= 16
 *                                      keys (a pool block, or <= 16 chunk rows that follow
 *                                      each other with no pool block between them), 8 units
 *                                      per tile; src 0 / 1 = all units pool / chunk,
 *                                      2 = mixed
 *   n_qt  x (seq, row0, nrows, minpos, maxpos)             query tiles of 128 rows
 *   n_cls x class (0 SKIP, 1 FULL, 2 PARTIAL), per query tile, per KV tile of its sequence
 * Decode plans export the tokens only (n_kt = n_qt = n_cls = 0).
 * With out == NULL only *n (int32 count) is written.  WORKSPACE if capacity < *n. */
msa_status_t msa_plan_export(const msa_plan_t* plan, int32_t* out, size_t capacity, size_t* n);

/* Decode split units as int32 triples (seq, first canonical block, number of blocks). */
msa_status_t msa_plan_export_splits(const msa_plan_t* plan, int32_t* out, size_t capacity, size_t* n);

/* Prefill schedule as int32 records of 9 words, one per piece, grouped by CTA in the
 * order each CTA runs them: (cta, query tile, KV head, first query head, first list entry,
 * list entries, pieces of the work item, first partial slot of the item, own slot).  The
 * list of a query tile is its non-skipped KV tiles, full ones first, each group in
 * position order.  A work item is (query tile, KV head, first query head); its pieces
 * cover its list exactly once.  Decode plans export nothing. */
msa_status_t msa_plan_export_schedule(const msa_plan_t* plan, int32_t* out, size_t capacity, size_t* n);

msa_status_t msa_plan_get_stats(const msa_plan_t* plan, msa_plan_stats_t* stats);

/* Adaptive chunk tiler (abstract: an adaptive chunking scheduler keeps the hardware
 * busy; the pages give no rule, this is the library's rule): for R recompute tokens
 * take n = ceil(R/max_chunk) chunks of near-equal size rounded up to the 128-token
 * tile, c = min(R, roundup(ceil(R/n),128)); cut front to back into ceil(R/c) chunks,
 * the last taking the remainder; R < min_chunk gives one chunk.  max_chunk must be a
 * positive multiple of 128.  Writes *n sizes (capacity permitting). */
msa_status_t msa_chunk_sizes(int32_t R, int32_t min_chunk, int32_t max_chunk,
                             int32_t* sizes, int32_t capacity, int32_t* n);

/* MSA prefill (TTFT path), one launch for all sequences of the plan.
 *   q        device bf16 [total_q][Hq][d]
 *   k_chunk  device bf16 [total_q][Hkv][d], v_chunk likewise (the chunk's fresh K/V)
 *   k_pool   device bf16 [num_pool_blocks][Hkv][16][d], v_pool likewise; slots past a
 *            block's fill may hold anything (NaN and Inf included): they never reach a result
 *   out      device bf16 [total_q][Hq][d]; lse device fp32 [total_q][Hq]
 *   scale    softmax scale (1/sqrt(d) for Eq. 1)
 * All device pointers 16-byte aligned.  Errors: INVALID_ARG, MODE, WORKSPACE, CUDA. */
msa_status_t msa_prefill(const msa_plan_t* plan, const void* plan_dev,
                         const void* q, const void* k_chunk, const void* v_chunk,
                         const void* k_pool, const void* v_pool,
                         void* out, float* lse, float scale,
                         void* workspace, size_t ws_bytes, cudaStream_t stream);

/* MSA decode (TPOT path): split-KV over the segments with the LSE merge fused in.
 *   q   device bf16 [num_seqs][Hq][d]; out bf16 [num_seqs][Hq][d]; lse fp32 [num_seqs][Hq]
 *   k_pool, v_pool as for msa_prefill (slots past a block's fill may hold anything)
 * Errors: INVALID_ARG, MODE, WORKSPACE, CUDA. */
msa_status_t msa_decode(const msa_plan_t* plan, const void* plan_dev, const void* q,
                        const void* k_pool, const void* v_pool,
                        void* out, float* lse, float scale,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Decode without any device allocation.  The paper has no counterpart: this is a
 * convenience of this library for callers that cannot allocate device memory -- e.g. a
 * serving engine that reserves almost all of HBM for its KV-cache pool when it starts and
 * hands out nothing afterwards, or a latency-critical loop that must not call cudaMalloc or
 * cudaFree because they can synchronise the whole device.  Same inputs, outputs and result
 * as msa_decode, but no workspace argument: the split-KV scratch lives in one fixed 8 MiB
 * device array owned by the library (every GPU that loads libmsa.so holds it until the
 * process exits).  Plans whose msa_workspace_bytes exceed 8 MiB are rejected with
 * MSA_ERR_WORKSPACE.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture.  The address is kept for the life of the process: do not use this entry point
 * after a cudaDeviceReset (or anything else that destroys and re-creates the device's
 * primary context), since the array is then re-loaded at another address.  Each call
 * clears the scratch's status word and merge counters on `stream` (cudaMemsetAsync) and
 * allocates nothing.  All calls share the one array, so calls that may overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller.  Its bounded
 * waits use the limit of msa_set_wait_limit, like every other launch; a device-side error
 * of this variant (a wait that ran out) is read with msa_get_status_no_alloc.
 * Errors: INVALID_ARG, MODE, WORKSPACE, CUDA. */
msa_status_t msa_decode_no_alloc(const msa_plan_t* plan, const void* plan_dev, const void* q,
                                 const void* k_pool, const void* v_pool,
                                 void* out, float* lse, float scale, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the device status word that the last
 * msa_decode_no_alloc call on the current device left in the library's scratch array.
 * Returns MSA_OK or the device-side error (e.g. MSA_ERR_TIMEOUT); allocates nothing. */
msa_status_t msa_get_status_no_alloc(cudaStream_t stream);

/* Merge two partial attention results over disjoint key sets (elementwise over
 * rows x heads): m = max(lse_a, lse_b), w = exp(lse - m), O = (w_a O_a + w_b O_b)/(w_a + w_b),
 * LSE = m + ln(w_a + w_b); a part with lse = -inf weighs 0; both -inf give O = 0, LSE = -inf.
 *   o_a, o_b  device fp32 [rows][heads][head_dim]; lse_a, lse_b fp32 [rows][heads]
 *   o         device bf16 [rows][heads][head_dim]; lse fp32 [rows][heads]
 * head_dim % 4 == 0.  Errors: INVALID_ARG, CUDA. */
msa_status_t msa_merge_lse(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                           void* o, float* lse, int32_t rows, int32_t heads, int32_t head_dim,
                           cudaStream_t stream);

/* Gather the KV context of every sequence in canonical (position) order, bit-exact:
 *   k_out, v_out device bf16 [n_tok][Hkv][d] in export order; pos_out int32 [n_tok] (nullable).
 * k_chunk / v_chunk may be NULL for decode plans.  Errors: INVALID_ARG, WORKSPACE, CUDA. */
msa_status_t msa_gather(const msa_plan_t* plan, const void* plan_dev,
                        const void* k_chunk, const void* v_chunk,
                        const void* k_pool, const void* v_pool,
                        void* k_out, void* v_out, int32_t* pos_out, size_t out_tokens,
                        cudaStream_t stream);

/* Write-back of a chunk's fresh K/V into the paged pool (the step after prefill: the
 * abstract's recomputed evicted blocks, and the new tokens, go back into pool blocks at
 * their original positions so later chunks and decode find them).  Host-only planning:
 *   q_pos[n]            original positions of ONE sequence's chunk rows, strictly ascending
 *   free_blocks[n_free] physical pool blocks the caller hands out, taken in order
 *   seq_blocks[n_seq_blocks]  the sequence's blocks already in the pool (any order; may be
 *                       NULL when 0): a position block that a chunk row continues part-way
 *                       (e.g. a new turn's suffix after a partial last block) is found here
 *   block_pos, block_fill [num_pool_blocks]  in/out: set for every block written
 *   dst_slot[n]         out: pool slot of each row, physical_block * 16 + offset
 *   new_blocks[n_free]  out: the blocks taken from free_blocks, in position order; *n_new
 * Rows are grouped by position block (pos / 16) and go to one pool block each, at offset
 * pos % 16.  A group that starts at offset 0 takes the next free block; one that starts at
 * offset f > 0 continues the sequence's block whose block_pos is the group's position block
 * and whose fill is f.  Either way the group must extend its block without a hole.  Errors:
 * INVALID_ARG (unsorted positions, a hole, no block to continue), WORKSPACE (free_blocks too
 * short), BLOCK_OOB (a block id outside [0, num_pool_blocks)).  On error nothing is written. */
msa_status_t msa_append_plan(const int32_t* q_pos, int32_t n, const int32_t* free_blocks, int32_t n_free,
                             const int32_t* seq_blocks, int32_t n_seq_blocks, int32_t* block_pos,
                             int32_t* block_fill, int32_t num_pool_blocks, int32_t* dst_slot,
                             int32_t* new_blocks, int32_t* n_new);

/* Copy rows of the chunk's K and V into their pool slots (bit-exact; asynchronous on
 * `stream`):  k_pool[dst / 16][g][dst % 16][:] = k_chunk[row][g][:] for every KV head g, and
 * likewise for V.  dst_slot device int32 [n] (a negative slot skips the row; a slot past the
 * pool is ignored), k_chunk / v_chunk device bf16 [n][Hkv][d], k_pool / v_pool device bf16
 * [num_pool_blocks][Hkv][16][d]; 16-byte aligned.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
msa_status_t msa_kv_append(const int32_t* dst_slot, const void* k_chunk, const void* v_chunk,
                           void* k_pool, void* v_pool, int32_t n, int32_t num_heads_kv, int32_t head_dim,
                           int32_t num_pool_blocks, cudaStream_t stream);

/* Synchronise `stream`, read and clear the workspace status word.  Returns MSA_OK or
 * the device-side error (e.g. MSA_ERR_TIMEOUT). */
msa_status_t msa_get_status(void* workspace, cudaStream_t stream);

/* Device-wait bound: nanoseconds (global timer) that each mbarrier wait of a kernel may
 * spin before the kernel gives up with MSA_ERR_TIMEOUT; <= 0 restores the default of
 * 2 s.  Applies to later launches. */
void msa_set_wait_limit(int64_t ns);

/* Test hook for the give-up path (the paper has no counterpart).  Later launches of
 * `kernel` leave out one of their copies, so that the bounded wait for it runs out and the
 * kernel gives up exactly as it would on a copy that never completes: it records
 * MSA_ERR_TIMEOUT in the status word, lets every copy and MMA it did start land, frees its
 * tensor memory and returns.  kernel 0 = msa_prefill: CTA `cta` leaves out the K tile it
 * would load as its `index`-th (counting from 0 over all its work); kernel 1 = msa_decode
 * and msa_decode_no_alloc: warp 0 of CTA (split unit `cta`, head group 0) leaves out its
 * `index`-th block.  Nothing faults and nothing waits past the wait limit.  Results of such
 * a launch are undefined, and it may leave merge counters set: re-initialise the workspace
 * (msa_workspace_init) before its next use.  A negative argument turns the hook off (the
 * default). */
void msa_set_test_drop(int32_t kernel, int32_t cta, int32_t index);

/* ------------------------------------------------------------------ eviction policy
 * Host-side KV-block eviction policy (abstract: eviction that jointly weighs hit rate and
 * position-aware recompute cost; Fig. 6 / Eq. 5: the marginal recompute latency of a
 * block; Fig. 7 / Fig. 8: reuse-time distribution and a piecewise exponential reuse model
 * in an O(log n) structure; Fig. 10 / Eq. 10: the lambda update from the mean block
 * lifespan; appendix A.1: only an exponential keeps the order of blocks not accessed).
 * No GPU is involved.  Score of a cached block b at time t, the smallest evicted first:
 *   S_b(t) = C_b * min(1, lambda * F_b * exp(-(t - t_b) / beta)),
 *   C_b = k5 * p_b + k_const   (Eq. 5 with l1 + 2 q1 approximated by p_b, the number of
 *                               blocks before b in its sequence; k_const = k2 - k3 + k5),
 *   F_b = accesses of b while cached, t_b = its last access,
 *   lambda = exp((tau - tau0) / beta - tau / alpha)   (Eq. 10), tau = the mean lifespan
 *   (eviction time - insertion time) of the last `window` evicted blocks, refreshed every
 *   `period` evictions (period 0: lambda stays lambda0).
 * Ties go to the smaller block id.  Times are any increasing unit (e.g. request count). */
typedef enum {
  MSA_EVICT_COST = 0,       /* the score above, ordered sets: O(log n) per operation */
  MSA_EVICT_COST_SCAN = 1,  /* the same score by a linear scan per eviction: O(n) */
  MSA_EVICT_LRU = 2,        /* baseline: least recently accessed first */
  MSA_EVICT_PREFIX = 3      /* baseline, prefix caching: largest position first (then LRU) */
} msa_evict_policy_t;

typedef struct {
  double k5;         /* Eq. 5 coefficient of (l1 + 2 q1), per block, > = 0 */
  double k_const;    /* k2 - k3 + k5, > 0 (so every C_b > 0) */
  double beta;       /* time scale of the exponential (and of Eq. 10), > 0 */
  double alpha;      /* Eq. 10, > 0 */
  double tau0;       /* Eq. 10 */
  double lambda0;    /* lambda before the first update, > 0 */
  int32_t window;    /* lifespans in the sliding window (> 0 when period > 0) */
  int32_t period;    /* evictions between lambda updates, 0 = never */
  int32_t policy;    /* msa_evict_policy_t */
  int32_t reserved;  /* must be 0 */
} msa_evict_opts_t;

typedef struct msa_evict msa_evict_t;  /* opaque, host-owned */

/* Errors: INVALID_ARG (a bad option, an unknown or duplicate block, an empty cache on
 * victim, a non-finite time).  Block ids are any non-negative int32. */
msa_status_t msa_evict_create(const msa_evict_opts_t* opts, msa_evict_t** out);
void msa_evict_destroy(msa_evict_t* policy);
/* A block enters the cache (its first access) at time `now`; pos_block = p_b. */
msa_status_t msa_evict_insert(msa_evict_t* policy, int32_t block, int32_t pos_block, double now);
/* A cached block is accessed again (a hit). */
msa_status_t msa_evict_access(msa_evict_t* policy, int32_t block, double now);
/* A block leaves the cache without being evicted (e.g. its sequence ended). */
msa_status_t msa_evict_remove(msa_evict_t* policy, int32_t block);
/* Choose the block to evict at time `now`, remove it and record its lifespan. */
msa_status_t msa_evict_victim(msa_evict_t* policy, double now, int32_t* block);
/* S_b(now) of a cached block (cost-aware definition, whatever the policy). */
msa_status_t msa_evict_score(const msa_evict_t* policy, int32_t block, double now, double* score);
msa_status_t msa_evict_get_lambda(const msa_evict_t* policy, double* lambda);
int32_t msa_evict_size(const msa_evict_t* policy);
/* Consistency check of the policy's internal ordered sets (for tests). */
msa_status_t msa_evict_check(const msa_evict_t* policy, double now);

const char* msa_status_string(msa_status_t status);
int32_t msa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H_ */
