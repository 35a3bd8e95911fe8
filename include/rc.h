/*
 * rc.h -- C ABI of the prefix-cached paged attention library (librc).
 *
 * The library implements the data path of RadixAttention (SGLang, "Efficient Execution of
 * Structured Language Model Programs", arXiv 2312.07104): KV caches of all requests live in one
 * pool of token-sized pages; a radix tree over token sequences finds each request's longest
 * cached prefix, whose KV is reused, so only the unmatched suffix is computed; finished
 * sequences are inserted back; unreferenced leaves are evicted in LRU order when the pool runs
 * short.
 *
 * Conventions
 *   - Every function returns an int status: RC_OK (0) or a negative RC_ERR_* code. The message
 *     of the last failure on the calling thread is available from rc_last_error().
 *   - The caller owns every buffer. Pointers documented as "device" point to GPU memory of the
 *     current CUDA device; "host" pointers to CPU memory. The library allocates no device memory;
 *     decode attention takes an explicit caller-provided workspace.
 *   - Device entry points are asynchronous on the given stream (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream), never synchronise, and report launch failures as
 *     RC_ERR_CUDA. Kernels that detect bad data (a slot index out of range, a length beyond the
 *     slot-table row, an expired wait) set a device status word and skip the access instead of
 *     trapping; rc_device_status() reads and clears it.
 *   - Pool and tree objects are not thread-safe: one scheduler thread drives them.
 *   - Layouts are row-major and contiguous. T = total new tokens of an extend batch, B = requests,
 *     Hq / Hkv = query / KV heads (Hq % Hkv == 0; query head h reads KV head h / (Hq / Hkv)),
 *     d = head_dim.
 *   - KV pool of one layer: K and V each [num_slots, Hkv, d]; slot s holds the KV of one token
 *     for all KV heads. The slot table req_to_token is [max_reqs, max_ctx] int32: row r lists
 *     the slots of request r's tokens in order.
 */
#ifndef RC_H
#define RC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RC_OK 0
#define RC_ERR_INVALID -1     /* bad argument, stale node handle, double free */
#define RC_ERR_OOM -2         /* fewer free slots than requested; nothing allocated */
#define RC_ERR_INSUFFICIENT -3 /* eviction freed fewer tokens than requested */
#define RC_ERR_CUDA -4        /* a CUDA runtime call failed */
#define RC_ERR_DEVICE -5      /* a kernel reported bad data through the device status word */

#define RC_DTYPE_BF16 0
#define RC_DTYPE_F32 1

typedef struct rc_pool rc_pool;
typedef struct rc_radix rc_radix;
/* Node handle. 0 is the root. A handle goes stale when its node is evicted; a stale handle is
 * rejected with RC_ERR_INVALID. A split keeps the handle of the lower (deeper) part, so a handle
 * always names the node that ends where it ended when it was returned. */
typedef uint64_t rc_node;

/* Thread-local message of the last failure (empty string if none). Never NULL. */
const char* rc_last_error(void);
/* Number of kernels this library has launched in this process (all device entry points). */
uint64_t rc_launch_count(void);

/* ---------------------------------------------------------------------------------------- */
/* Token pool (paper digest Sec. 3: KV stored in pages of one token; cached and running       */
/* requests share one pool). Slots are the page indices 0 .. num_slots-1.                     */
/* ---------------------------------------------------------------------------------------- */

/* Create a pool of num_slots free slots. initial_order (host, num_slots int32, a permutation of
 * 0..num_slots-1, may be NULL for 0,1,2,...) is the initial free-list order. */
int rc_pool_create(int64_t num_slots, const int32_t* initial_order, rc_pool** out);
void rc_pool_destroy(rc_pool* pool);
/* Take n slots from the head of the free list into out_slots (host, n int32). All or nothing:
 * RC_ERR_OOM and no change when fewer than n are free. */
int rc_kv_pool_alloc(rc_pool* pool, int64_t n, int32_t* out_slots);
/* Return n slots (host) to the tail of the free list in the given order. RC_ERR_INVALID and no
 * change if any slot is out of range, already free, or repeated. */
int rc_kv_pool_free(rc_pool* pool, const int32_t* slots, int64_t n);
int rc_kv_pool_available(const rc_pool* pool, int64_t* out);
/* Host fault injection, for testing callers' failure paths without a real shortage (the pages
 * describe no failure handling; this is a test hook of the library's own). After `after_calls`
 * further successful rc_kv_pool_alloc calls on this pool, the next one fails with RC_ERR_OOM
 * and changes nothing; the hook then disarms itself. Slots the radix tree takes internally
 * (host-tier spills and loads) are not affected. after_calls = -1 disarms it; any other
 * negative value is RC_ERR_INVALID. */
int rc_pool_inject_alloc_failure(rc_pool* pool, int64_t after_calls);

/* ---------------------------------------------------------------------------------------- */
/* Radix tree (paper digest Sec. 3 and Fig. 3; SGLang blog Sec. 2.3; RadixAttention explainer */
/* "insert / match / split / evict"). Edges are token sequences; a node holds the slots of    */
/* its edge's tokens. The tree frees evicted slots into the pool it was created with.         */
/* ---------------------------------------------------------------------------------------- */

int rc_radix_create(rc_pool* pool, rc_radix** out);
/* Destroys the tree; slots it still holds are NOT returned to the pool. */
void rc_radix_destroy(rc_radix* tree);

/* Longest cached prefix of tokens[0:n] (host). Writes its length to *out_len, its slots to
 * out_slots[0:*out_len] (host, capacity n) and the node where it ends to *out_node (0 if
 * nothing matched). When the match ends inside an edge the edge is split there, so that
 * locking *out_node protects exactly the matched tokens. Marks the path as most recently
 * used (nodes stamped root to leaf with a logical clock). */
int rc_radix_match_prefix(rc_radix* tree, const int32_t* tokens, int64_t n, int32_t* out_slots,
                          int64_t* out_len, rc_node* out_node);
/* Insert tokens[0:n] with their slots (host). Tokens already present keep the tree's slots;
 * *out_existing = number of leading tokens that were present (the caller owns and should free
 * its own slots[P:*out_existing] where P is what it matched). The sequence end becomes a node
 * boundary (splitting an edge if needed); *out_node = that node. Marks the path as used. */
int rc_radix_insert(rc_radix* tree, const int32_t* tokens, const int32_t* slots, int64_t n,
                    int64_t* out_existing, rc_node* out_node);
/* Reference counts: +1 / -1 on node and every ancestor (the root excluded). A node with a
 * nonzero count is never evicted. Unlocking a node whose count is zero is RC_ERR_INVALID. */
int rc_radix_lock(rc_radix* tree, rc_node node);
int rc_radix_unlock(rc_radix* tree, rc_node node);
/* Evict least-recently-used leaves with reference count 0, whole nodes at a time, smallest
 * (stamp, node id) first, until at least n_tokens are freed; a parent that becomes such a leaf
 * joins the candidates. Freed slots go to the pool tail, node by node, in token order.
 * *out_freed = tokens freed (may exceed n_tokens). RC_ERR_INSUFFICIENT if fewer than n_tokens
 * could be freed (what could be freed is freed). */
int rc_radix_evict_lru(rc_radix* tree, int64_t n_tokens, int64_t* out_freed);

typedef struct rc_stats {
  int64_t nodes;             /* excluding the root */
  int64_t cached_tokens;     /* tokens held by the tree */
  int64_t evictable_tokens;  /* tokens in nodes with reference count 0 */
  int64_t protected_tokens;  /* tokens in nodes with reference count > 0 */
  int64_t splits;
  int64_t evicted_nodes;
  int64_t evicted_tokens;
  int64_t matched_tokens;    /* sum of match lengths (prefill tokens skipped) */
  int64_t match_queries;     /* sum of query lengths given to match */
  int64_t host_tokens;       /* tokens held in the host tier */
  int64_t spilled_tokens;    /* evicted device tokens moved to the host tier */
  int64_t loaded_tokens;     /* host-tier tokens moved back to the device */
  int64_t dropped_tokens;    /* tokens that left a tree with a host tier altogether */
} rc_stats;
int rc_radix_stats(const rc_radix* tree, rc_stats* out);

/* Canonical dump for tests: depth first, children in ascending order of their first token; per
 * node (root excluded): id, parent id, reference count, stamp, edge length L, L tokens, L slots
 * (int64 each). Node ids count creations from 1 (root 0); a split's new upper node takes the
 * next id. Returns the number of int64 written, or minus the number needed if cap is short. */
int64_t rc_radix_dump(const rc_radix* tree, int64_t* buf, int64_t cap);

/* Batched host steps for a scheduler step (host pointers). Sequence b is
 * tokens[indptr[b] : indptr[b+1]]; rows is a [B, row_stride] int32 host array of slot rows.
 *
 * rc_radix_match_batch: for b in order, match the first match_len[b] tokens of sequence b
 * (match_len may be NULL = whole sequence), lock the node where the match ends, write the
 * matched slots to rows[b, 0:prefix_len[b]] and the node to nodes[b]. */
int rc_radix_match_batch(rc_radix* tree, const int32_t* tokens, const int64_t* indptr, int32_t B,
                         const int32_t* match_len, int32_t* rows, int64_t row_stride,
                         int32_t* prefix_len, rc_node* nodes);
/* rc_radix_insert_batch: for b in order, insert sequence b with slots rows[b, 0:len_b]; free the
 * caller's duplicate slots rows[b, prefix_len[b] : existing_b] to the pool; if keep_locked,
 * lock the inserted sequence's end node (written to end_nodes[b] if end_nodes is not NULL);
 * then unlock unlock_nodes[b] (skipped when unlock_nodes is NULL). *out_freed = duplicates
 * freed (may be NULL). */
int rc_radix_insert_batch(rc_radix* tree, const int32_t* tokens, const int64_t* indptr, int32_t B,
                          const int32_t* rows, int64_t row_stride, const int32_t* prefix_len,
                          const rc_node* unlock_nodes, int32_t keep_locked, rc_node* end_nodes,
                          int64_t* out_freed);

/* Host tier (SGLang blog Sec. 6.1 HiCache: GPU memory holds the hottest KV, host memory the next
 * tier). With a host pool attached, rc_radix_evict_lru moves each least-recently-used device
 * leaf to host slots instead of freeing it: the node keeps its place in the tree and becomes
 * host-resident. Device-resident nodes always form the part of the tree that contains the root
 * (a device leaf = device-resident, unreferenced, no device-resident child). To make room in the
 * host pool, unreferenced host nodes without children are dropped, least recently used first
 * (smallest (stamp, node id)); a victim the host tier cannot take even then is freed. Host slots
 * index the caller's host KV planes exactly as device slots index the device planes.
 *
 * The tree records the copies this implies and the caller performs them before any later device
 * work writes a recycled slot: spills (device slot -> host slot) first, then loads (host slot ->
 * device slot), in one stream. rc_radix_pending_copies counts them; rc_radix_drain_copies hands
 * them out (buffers sized by the counts) and forgets them. Eviction is refused (RC_ERR_INVALID)
 * while loads are pending.
 *
 * The single-sequence match, rc_radix_match_batch and rc_schedule_batch see device-resident
 * tokens only (a walk stops at the first host-resident node). rc_radix_match_batch_tiered
 * continues through host-resident nodes: prefix_len[b] = the device-resident part (its slots in
 * rows), host_len[b] = the host-resident tokens after it; the lock covers both. After making
 * room for sum(host_len) device slots, rc_radix_load_batch moves those nodes back to the device
 * (device slots from the pool in request and token order; the host slots return to the host
 * pool when the copies are drained), writes their slots to rows[b, prefix_len[b]:...] and adds
 * host_len[b] to prefix_len[b]. RC_ERR_OOM if fewer device slots are free than sum(host_len).
 * An insert through host-resident tokens gives them the caller's slots (the node returns to the
 * device) and counts only the leading device-resident tokens as already present.
 * rc_radix_tiers writes (node id, 1 if host-resident) per node in the dump's order. */
int rc_radix_attach_host_tier(rc_radix* tree, rc_pool* host_pool);
int rc_radix_match_batch_tiered(rc_radix* tree, const int32_t* tokens, const int64_t* indptr,
                                int32_t B, const int32_t* match_len, int32_t* rows,
                                int64_t row_stride, int32_t* prefix_len, rc_node* nodes,
                                int32_t* host_len);
int rc_radix_load_batch(rc_radix* tree, const int32_t* tokens, const int64_t* indptr, int32_t B,
                        int32_t* rows, int64_t row_stride, int32_t* prefix_len,
                        const int32_t* host_len);
int rc_radix_pending_copies(const rc_radix* tree, int64_t* n_spill, int64_t* n_load);
int rc_radix_drain_copies(rc_radix* tree, int32_t* spill_dev, int32_t* spill_host,
                          int32_t* load_host, int32_t* load_dev);
int64_t rc_radix_tiers(const rc_radix* tree, int64_t* buf, int64_t cap);

/* Cache-aware batch formation (paper digest Sec. 3 "cache-aware scheduling": order the waiting
 * requests longest shared prefix first rather than first come first served; its Theorem 3.1
 * says that order is the radix tree's depth-first order, which computes every edge once when
 * the cache holds the longest request; App. A.2 pseudocode: match every waiting request, sort
 * by match length, admit into the batch while memory allows, evicting as needed). Reads the
 * tree and the pool; changes nothing (no split, no stamp, no lock).
 *
 * Waiting sequence w is tokens[indptr[w] : indptr[w+1]] (host arrays, w in queue order); its
 * match is the longest cached prefix of its first match_len[w] tokens (match_len NULL = the
 * whole sequence), written to out_match[w]. out_order[0:B] = the waiting sequences in
 * scheduling order: RC_SCHED_LSPF by descending match, ties in queue order; RC_SCHED_FCFS in
 * queue order. Admission walks that order and stops at the first sequence that does not fit:
 *   - at most max_batch sequences;
 *   - at most max_new_tokens computed tokens, sum of (length - match) (max_new_tokens < 0: no
 *     limit);
 *   - room: free slots + cached tokens in nodes with reference count 0 - reserve_slots must cover
 *     the computed tokens plus the unreferenced cached tokens that the admitted matches would
 *     lock (each cached token counted once).
 * *out_admitted = the admitted count; the batch is out_order[0 : *out_admitted]. Matching the
 * admitted sequences in that order (rc_radix_match_batch with the same match_len) and evicting
 * the shortfall then always succeeds. RC_ERR_INVALID on a NULL or inconsistent argument. */
enum { RC_SCHED_LSPF = 0, RC_SCHED_FCFS = 1 };
int rc_schedule_batch(const rc_radix* tree, const int32_t* tokens, const int64_t* indptr,
                      int32_t B, const int32_t* match_len, int32_t policy, int32_t max_batch,
                      int64_t max_new_tokens, int64_t reserve_slots, int32_t* out_order,
                      int32_t* out_match, int32_t* out_admitted);
/* The same batch formation over W waiting sequences given as ranges of one token buffer:
 * sequence w is tokens[starts[w], starts[w] + lengths[w]) (host int64 arrays of W entries;
 * ranges may be in any order, with gaps). Outputs, order and admission exactly as
 * rc_schedule_batch over the same sequences. A caller that keeps its whole queue in one buffer
 * passes the waiting entries' ranges instead of repacking the queue for every call. */
int rc_schedule_batch_ranges(const rc_radix* tree, const int32_t* tokens, const int64_t* starts,
                             const int64_t* lengths, int32_t W, const int32_t* match_len,
                             int32_t policy, int32_t max_batch, int64_t max_new_tokens,
                             int64_t reserve_slots, int32_t* out_order, int32_t* out_match,
                             int32_t* out_admitted);

/* ---------------------------------------------------------------------------------------- */
/* Device entry points                                                                       */
/* ---------------------------------------------------------------------------------------- */

/* Slot-table write: req_to_token[seg_row[i], seg_col[i] + j] = values[seg_indptr[i] + j] for
 * j < seg_indptr[i+1] - seg_indptr[i]. All arrays device int32. A segment outside the table
 * sets the device status word and is skipped. */
typedef struct rc_slot_write_args {
  int32_t num_segments;
  int32_t max_reqs;          /* rows of req_to_token */
  int32_t max_ctx;           /* columns of req_to_token */
  int64_t total_values;      /* seg_indptr[num_segments] (host-known) */
  const int32_t* seg_row;
  const int32_t* seg_col;
  const int32_t* seg_indptr; /* [num_segments + 1] */
  const int32_t* values;
  int32_t* req_to_token;
} rc_slot_write_args;
int rc_slot_table_write(const rc_slot_write_args* args, void* stream);

/* KV row copies between two pools (the host tier's spills and loads; SGLang blog Sec. 6.1):
 * for i < n and every layer, the K row and the V row of slot src_slots[i] in the source planes
 * are copied to slot dst_slots[i] in the destination planes. Planes are [layers][num_slots][row]
 * with row = row_bytes (Hkv x d x element size, a multiple of 16), 16-byte aligned, in device
 * memory or in pinned host memory that the GPU can address (on Grace-Blackwell the kernel reads
 * and writes it directly). src_slots / dst_slots are device int32 arrays. Destination slots
 * must be distinct; rows are copied in no particular order. A slot outside its pool sets the
 * device status word (rc_device_status) and that row is skipped. Asynchronous on `stream`. */
typedef struct rc_kv_copy_args {
  int64_t n;
  int32_t layers;
  int64_t row_bytes;
  const int32_t* src_slots;
  const int32_t* dst_slots;
  const void* src_k;
  const void* src_v;
  int64_t src_num_slots;
  void* dst_k;
  void* dst_v;
  int64_t dst_num_slots;
} rc_kv_copy_args;
int rc_kv_copy(const rc_kv_copy_args* args, void* stream);

/* Extend attention (SGLang blog Sec. 2.3 "compute only the unmatched tokens"; paper digest
 * App. A.1). For request b with matched prefix P = prefix_len[b] and S = qo_indptr[b+1] -
 * qo_indptr[b] new tokens at positions P .. P+S-1, each new token's query attends to the P
 * cached keys, gathered through req_to_token[req_idx[b], 0:P], and causally to the new keys of
 * positions <= its own, which are read from k_new / v_new:
 *   O[t,h] = sum_{j <= P+i} softmax_j(sm_scale * <q_t,h , k_j,h/g>) v_j,h/g,  t = qo_indptr[b]+i
 * and the new K/V rows are scattered: k_pool[out_loc[t]] = k_new[t], v_pool likewise.
 *   q [T, Hq, d], k_new / v_new [T, Hkv, d], o [T, Hq, d] in dtype; lse [T, Hq] fp32 natural log
 *   of the softmax denominator of the scaled scores (optional, NULL to skip); out_loc [T],
 *   qo_indptr [B+1], prefix_len [B], req_idx [B] device int32. bf16 requires head_dim 128
 *   (tensor-core path); f32 takes head_dim 64 or 128. Requests may have S = 0. q, k_new,
 *   v_new, o and the pool planes are 16-byte aligned (RC_ERR_INVALID otherwise). */
typedef struct rc_extend_args {
  int32_t dtype;
  int32_t num_reqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t max_reqs;          /* rows of req_to_token; every req_idx must be below it */
  int32_t max_ctx;           /* columns of req_to_token, multiple of 4 */
  int32_t max_q_len;         /* >= every S (host-known; sizes the grid) */
  int32_t max_prefix_len;    /* >= every P (host-known) */
  int64_t num_tokens;        /* T */
  int64_t num_slots;
  float sm_scale;
  const void* q;
  const void* k_new;
  const void* v_new;
  const int32_t* out_loc;
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  const int32_t* req_idx;
  const int32_t* req_to_token;
  void* k_pool;              /* this layer's K plane [num_slots, Hkv, d] */
  void* v_pool;
  void* o;
  float* lse;
  /* Optional prefix stacking (the shared-prefix query stacking of the paper digest's related
   * work, Sec. 7; num_groups = 0 disables it). Group g is the run of consecutive requests
   * [group_range[2g], group_range[2g+1]) whose req_to_token rows hold the same slots at
   * positions [0, group_shared[g]), a prefix they all matched. A first pass attends the
   * members' new-token queries, stacked, to those keys -- each K/V tile gathered once for the
   * whole group -- and keeps every row's partial result (normalised O in o, its log-sum-exp in
   * the workspace); the per-request pass then covers the keys from group_shared[g] on and
   * merges the two with log-sum-exp weights. Outputs are those of the definition above.
   * Contract: ranges ascending and disjoint; group_shared[g] >= 1 and <= prefix_len[b] of
   * every member; max_group_rows >= the new tokens of every group. Breaches are reported
   * through the device status word and never leave the given buffers. bf16 only (the fp32 path
   * ignores the groups). Device int32 arrays; workspace >= rc_extend_workspace_bytes bytes,
   * 16-byte aligned, used only when num_groups > 0. */
  int32_t num_groups;
  int32_t max_group_rows;
  const int32_t* group_range;   /* [2 * num_groups] */
  const int32_t* group_shared;  /* [num_groups] */
  void* workspace;
  size_t workspace_bytes;
  /* Optional cascade over the levels of the radix tree (num_levels <= 1: the single level
   * above). Groups are listed level by level: level l holds groups [level_indptr[l],
   * level_indptr[l+1]) (HOST int32 array of num_levels + 1 entries, level_indptr[0] = 0,
   * level_indptr[num_levels] = num_groups, at most RC_MAX_STACK_LEVELS levels). Within a level
   * the contract above holds. A group of level l > 0 lies inside one group of level l - 1 and
   * group_start[g] (device int32 [num_groups]; NULL = all 0) is that parent's group_shared: its
   * stacked pass covers keys [group_start[g], group_shared[g]) only and merges its result into
   * the partial the levels above left (levels run in order). A request's per-request pass
   * starts at the largest group_shared of the groups holding it. group_start[g] >= 0 and
   * < group_shared[g], else reported through the status word. */
  int32_t num_levels;
  const int32_t* level_indptr;
  const int32_t* group_start;
  /* Optional folding of short remainders into the stacked pass. group_fold[g] = 1 (device int32
   * [num_groups], NULL = none) marks a group that no deeper group lies inside and whose every
   * member b has at most 128 keys left after the shared prefix (prefix_len[b] - group_shared[g]
   * + its new tokens <= 128): its stacked pass then also attends each member's rows to that
   * remainder (one 128-key tile per member: its own cached tokens after the shared prefix, then
   * its new tokens, causally), writes the final outputs and scatters the new K/V, and the
   * per-request pass leaves its members alone. skip_request_pass = 1 (host flag) when every
   * request is in a folded group: the per-request pass is not launched. A folded member whose
   * remainder exceeds 128 keys is reported through the status word. */
  const int32_t* group_fold;
  int32_t skip_request_pass;
} rc_extend_args;
#define RC_MAX_STACK_LEVELS 4
int rc_extend_workspace_bytes(const rc_extend_args* args, size_t* out_bytes);
int rc_extend_attention(const rc_extend_args* args, void* stream);

/* Planner of the extend call's prefix stacking (the shared-prefix query stacking of the paper
 * digest's related work, Sec. 7; host only). From the batch's host slot rows (rows[b] the slots
 * of request b, its prefix_len[b] matched tokens first; row_stride int32 per row) it finds, level
 * by level of the radix tree, runs of consecutive requests whose rows hold the same slots over
 * at least min_shared positions past their parent's shared length (level 0: from 0); a run's
 * shared length is its members' smallest agreement with its first member. Under RC_STACK_COST a
 * run is kept where a cost model of the extend kernel (calibrated on GB300) estimates stacking
 * to save 10% or more; a run not kept is not searched further. An innermost kept group folds
 * (takes its members' remainders in its own pass) under RC_FOLD_ALL, or under RC_FOLD_COST where
 * the model estimates the folded pass at no more than the stacked pass plus the members' own;
 * a group folds only if each CTA of its pass has at most 512 remainder key tiles and 256
 * members. group_size = query heads per KV head. The outputs fill rc_extend_args: group_range,
 * group_shared, group_start, group_fold (capacity entries; num_reqs * max_levels suffice),
 * level_indptr (num_levels + 1 entries used), max_group_rows, skip_request_pass = all_folded.
 * RC_ERR_INVALID if an argument is out of range or more groups than capacity are found. */
enum { RC_STACK_COST = 0, RC_STACK_ALL = 1 };
enum { RC_FOLD_NONE = 0, RC_FOLD_COST = 1, RC_FOLD_ALL = 2 };
typedef struct rc_stack_plan_args {
  int32_t num_reqs;
  const int32_t* rows;           /* host [num_reqs, row_stride] */
  int64_t row_stride;
  const int32_t* prefix_len;     /* host [num_reqs] matched tokens, <= row_stride */
  const int32_t* new_len;        /* host [num_reqs] new tokens */
  int32_t min_shared;            /* >= 1 */
  int32_t group_size;            /* >= 1 */
  int32_t max_levels;            /* 1 .. RC_MAX_STACK_LEVELS */
  int32_t policy;                /* RC_STACK_COST or RC_STACK_ALL */
  int32_t fold;                  /* RC_FOLD_NONE, RC_FOLD_COST or RC_FOLD_ALL */
} rc_stack_plan_args;
typedef struct rc_stack_plan {
  int32_t capacity;              /* in: entries of the four arrays below */
  int32_t* group_range;          /* out: [2 capacity] host */
  int32_t* group_shared;         /* out: [capacity] */
  int32_t* group_start;          /* out: [capacity] */
  int32_t* group_fold;           /* out: [capacity] */
  int32_t level_indptr[RC_MAX_STACK_LEVELS + 1];   /* out; entries past num_levels = num_groups */
  int32_t num_groups, num_levels, max_group_rows, all_folded;   /* out */
} rc_stack_plan;
int rc_plan_extend_stacking(const rc_stack_plan_args* args, rc_stack_plan* out);

/* Decode attention (paper digest App. A.1; RadixAttention explainer: each generated token
 * attends to the KV of all previous tokens). Request b has seq_len[b] tokens including its new
 * one, whose slot is out_loc[b] == req_to_token[req_idx[b], seq_len[b]-1]. Its query q[b]
 * attends to all seq_len[b] keys: the first seq_len[b]-1 gathered from the pool, the last read
 * from k_new[b] / v_new[b], which are also scattered to the pool at out_loc[b]. The context is
 * cut into chunks of kv_chunk tokens processed in parallel (split-K); each chunk's partial
 * state goes to the workspace and a merge kernel combines them with log-sum-exp weights.
 *   q [B, Hq, d], k_new / v_new [B, Hkv, d], o [B, Hq, d] in dtype; lse [B, Hq] fp32 optional;
 *   out_loc, seq_len, req_idx [B] device int32. head_dim 64 or 128. */
typedef struct rc_decode_args {
  int32_t dtype;
  int32_t num_reqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t max_reqs;          /* rows of req_to_token; every req_idx must be below it */
  int32_t max_ctx;           /* columns of req_to_token */
  int32_t kv_chunk;          /* tokens per split, multiple of 64; 0 = library default (512) */
  int64_t max_total_tokens;  /* >= sum of seq_len (host-known; sizes workspace and grid) */
  int64_t num_slots;
  float sm_scale;
  const void* q;
  const void* k_new;
  const void* v_new;
  const int32_t* out_loc;
  const int32_t* seq_len;
  const int32_t* req_idx;
  const int32_t* req_to_token;
  void* k_pool;
  void* v_pool;
  void* o;
  float* lse;
  /* Optional shared-context groups; num_groups = 0 computes every request on its own. Group g
   * lists the requests group_members[group_indptr[g] .. group_indptr[g+1]), the first being the
   * leader, whose req_to_token rows hold the same slots at positions [0, group_shared[g]) -- the
   * KV of a prefix they share in the radix tree. The chunks wholly inside that range are read once
   * for the whole group, the members' queries stacked next to each other (the shared-prefix
   * stacking of the paper digest's related work, Sec. 7, applied to decode); every member still
   * gets its own partial state per chunk, so the outputs are those of the per-request definition.
   * Contract: each request is in at most one group; a group has at most 8 / (Hq / Hkv) members;
   * group_shared[g] <= seq_len[m] - 1 for every member m. Breaking it is reported through the
   * device status word (RC_ERR_DEVICE at the next check); slots that differ inside the shared
   * range give the non-leading members the leader's KV there, never an out-of-range access.
   * Stacking applies to bf16; the fp32 path ignores the groups. Device int32 arrays. */
  int32_t num_groups;
  const int32_t* group_indptr;   /* [num_groups + 1] */
  const int32_t* group_members;  /* [group_indptr[num_groups]] request indices */
  const int32_t* group_shared;   /* [num_groups] tokens of shared context */
  /* 1: skip the plan (the job list in the workspace) and reuse the one the previous call on this
   * workspace made -- the layers of one decode step share it. The caller guarantees that call had
   * the same num_reqs, seq_len, req_idx contents, groups, kv_chunk and max_total_tokens, and that
   * it completed without a status error. bf16 only; the fp32 path always plans. */
  int32_t reuse_plan;
} rc_decode_args;
/* Workspace bytes rc_decode_attention needs for these arguments (device memory, 256-B aligned,
 * no initialisation needed). */
/* Planner of decode's shared-context groups (host only): requests whose host slot rows
 * (rows[b], lengths[b] context tokens, row_stride int32 per row) start with the same slot share
 * that prefix's KV. Greedy, bucket by bucket in order of first appearance of the first slot: the
 * bucket's first request leads; the others with the longest common slot prefix join (ties: the
 * later request first), up to group_size members in all, while that prefix is at least
 * min_shared tokens; the group's shared length is its members' smallest common prefix. Requests
 * shorter than max(min_shared, 1) take part in none. Outputs (host; num_reqs + 1, num_reqs and
 * num_reqs entries suffice) fill rc_decode_args' group_indptr, group_members and group_shared.
 * group_size < 2 or fewer than two requests: no group. */
int rc_plan_decode_groups(const int32_t* rows, int64_t row_stride, const int64_t* lengths,
                          int32_t num_reqs, int32_t group_size, int64_t min_shared,
                          int32_t* out_indptr, int32_t* out_members, int32_t* out_shared,
                          int32_t* out_num_groups);
int rc_decode_workspace_bytes(const rc_decode_args* args, size_t* out_bytes);
int rc_decode_attention(const rc_decode_args* args, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Decode attention for callers that cannot allocate device memory. Some callers have no way
 * to provide a workspace: a plugin interface that hands an operator only its input and output
 * buffers, or a serving loop that forbids device allocation once it is running (an allocation
 * can stall the whole device). This entry point takes the same arguments as
 * rc_decode_attention but no workspace: its scratch lives in one fixed area of
 * RC_DECODE_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 * keeps until the process exits. It calls no allocator of any kind. The paper has no
 * counterpart; this is a deployment convenience.
 *   - Arguments whose scratch need (rc_decode_workspace_bytes) exceeds the area are rejected
 *     with RC_ERR_INVALID; a larger kv_chunk needs less scratch.
 *   - The first call on a device looks up the area's device address (once per device, with
 *     that device current); make that first call before any stream capture.
 *   - All calls on a device share the area and it keeps the last call's contents (everything
 *     that must start at zero is reset by the call itself). Calls whose kernels overlap on the
 *     GPU -- on different streams without ordering between them -- race on the area.
 *   - reuse_plan is ignored: the job list in the shared area may belong to any earlier call on
 *     the device (another caller's, or one with other arguments), so every call plans afresh. */
#define RC_DECODE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
int rc_decode_attention_noalloc(const rc_decode_args* args, void* stream);

/* Test hook; the pages have no counterpart. Bound, in nanoseconds, of every wait inside the
 * extend kernel (0 restores the default, 2 s). With a short bound waits give up: the kernel
 * records code 3 in the device status word, stops issuing work and returns without hanging; its
 * outputs are then not written. The wait that guards the release of tensor memory keeps the
 * default. Applies to launches made after the call, on every device. */
int rc_debug_set_wait_limit_ns(uint64_t ns);

/* Read and clear the device status word of the current device (synchronises `stream`).
 * *out_code = 0 if no kernel reported bad data since the last call, else the first code seen:
 * 1 slot out of range, 2 position beyond the slot-table row, 3 a wait expired. */
int rc_device_status(int32_t* out_code, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RC_H */
