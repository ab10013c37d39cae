/*
 * rx.h -- C ABI of librx: the RadixAttention hot path on one GB300 (sm_103a).
 *
 * A host radix cache over a token-granular KV pool decides which KV slots
 * every request reads; CUDA kernels store new K/V into the pool and compute
 * extend (suffix prefill) and decode attention over the slots the cache hands
 * out.  Sources, by page title and section:
 *
 *   [T]  "SGLang: the tree, and the language nobody remembers"
 *        - "A tree, not a map": TreeNode fields, lock_ref accounting, heap
 *          eviction cascading to childless unlocked parents, node split at
 *          divergence, children keyed on the first token at page_size 1 and
 *          on the first page otherwise; keys truncated to whole pages and
 *          matches rounded down to a page (page_aligned).
 *        - "What the C++ tree is actually for": match_prefix returns the
 *          matched KV indices and a node handle.
 *        - "Speculative decoding puts a tree inside the tree": a tree node
 *          maps a token run to a vector of KV indices in the pool.
 *   [B]  "SGLang" (bibekananda.in) - "One tree for everybody" (walk from the
 *          root as far as tokens match; matched state is pointed at, not
 *          recomputed; the divergent part becomes a new branch), "Eviction on
 *          a tree" (leaves first, a parent only after its children).
 *   [L]  "SGLang: Structured LLM Programs for Efficient Inference"
 *        - "A quick recap of how an LLM generates text": decode attends over
 *          the KV cache and appends its own keys and values.
 *        - "How RadixAttention reuses past work": match, lock, prefill only
 *          the rest attending to the reused KV as if just computed, decode and
 *          insert, release.
 *        - "Worked example, step by step": a node is evicted whole; locked
 *          nodes are never evicted; with nothing evictable the request waits.
 *
 * Conventions
 *   - Every call returns an rx_status; nothing throws across the ABI.  On an
 *     error rx_last_error() returns a text for the calling thread.
 *   - The library owns the tree (opaque rx_cache).  The caller owns every host
 *     array and every device buffer (raw pointers, e.g. from torch tensors)
 *     and the CUDA stream.  The library never allocates device memory and
 *     creates no streams; it creates events only when asked to
 *     (rx_events_create).  Every kernel runs on the caller's stream, in call
 *     order.
 *   - Host calls are synchronous and not thread-safe for one cache.  Device
 *     calls only enqueue work on the given stream (cudaStream_t passed as
 *     rx_stream_t; NULL is the legacy default stream) and return RX_ERR_CUDA
 *     if the launch itself fails.  They may be made from several threads and
 *     on several devices at once (the library's per-device and per-thread
 *     state is set up safely); rx_decode_attention_static is the exception
 *     (one scratch array per device).
 *   - Token ids and slots are int32.  Slot 0 is a pad slot that the allocator
 *     never hands out; kernels read it for out-of-range keys only as a
 *     harmless address and mask the value.
 *   - Pages: the pool is cut into pages of page_size consecutive slots (page
 *     p = slots p*page_size .. p*page_size+page_size-1); page 0 is the pad
 *     page.  The cache hands out and takes back whole pages, keys in the tree
 *     are whole pages, and a request's positions [k*page_size,
 *     (k+1)*page_size) always lie in one page, in slot order.  At page_size 1
 *     a page is a slot and every rule below reduces to token granularity.
 *     The kernels read slot tables and are the same at every page size.
 *   - KV pool layout (device, bf16): K and V each [num_layers][num_kv_heads]
 *     [num_slots][head_dim], row-major; one slot row of one head is head_dim
 *     contiguous bf16 (256 B at d=128, 512 B at d=256).  Pool base pointers
 *     must be 16-byte aligned.  head_dim must be 128 or 256.
 */
#ifndef RX_H
#define RX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rx_status {
  RX_OK = 0,
  RX_ERR_INVALID = 1,  /* bad argument, shape, alignment or unknown node   */
  RX_ERR_NO_SPACE = 2, /* allocation impossible even after eviction        */
  RX_ERR_STATE = 3,    /* lock misuse or a rule the caller had to keep     */
  RX_ERR_CUDA = 4      /* a CUDA launch or copy returned an error          */
} rx_status;

typedef struct CUstream_st* rx_stream_t; /* identical to cudaStream_t */
typedef struct CUevent_st* rx_event_t;   /* identical to cudaEvent_t  */

/* A node handle is the node's id: 0 is the root, every created node (new
 * leaf, or the upper half of a split) takes the next id.  A handle stays valid
 * while its node is in the tree; a split keeps the lower half's id, so a held
 * handle keeps naming exactly the prefix it was returned for. */
typedef int64_t rx_node;

typedef struct rx_cache rx_cache;

typedef struct rx_config {
  int64_t num_slots; /* pool slots including the pad page; a multiple of
                        page_size                                        */
  int32_t page_size; /* slots per page, >= 1 (1 = token granularity)     */
  int32_t reserved;  /* must be 0                                         */
  int64_t host_slots;/* slots of the host tier including its pad page; 0
                        = one tier; else a multiple of page_size          */
} rx_config;

typedef struct rx_stats_t {
  int64_t cached_tokens;    /* tokens held by tree nodes                   */
  int64_t evictable_tokens; /* cached tokens with lock_ref == 0            */
  int64_t protected_tokens; /* cached tokens with lock_ref > 0             */
  int64_t free_slots;       /* slots on the free list                      */
  int64_t num_nodes;        /* nodes excluding the root                    */
  int64_t evicted_nodes;    /* since creation                              */
  int64_t evicted_tokens;   /* since creation                              */
  int64_t clock;            /* logical access clock                        */
  int64_t host_cached_tokens; /* tokens resident on the host tier          */
  int64_t host_free_slots;    /* slots on the host free list               */
  int64_t host_evicted_nodes; /* nodes evicted from the host tier          */
} rx_stats_t;

typedef struct rx_evict_rec {
  int64_t node_id;
  int64_t num_tokens;
} rx_evict_rec;

/* ------------------------------------------------------------------------
 * Cache lifecycle
 * ---------------------------------------------------------------------- */

/* Create an empty tree and a FIFO free list holding pages 1 ..
 * num_slots/page_size - 1 (reading: the pages do not fix the allocator
 * order).  Errors: RX_ERR_INVALID if page_size < 1, num_slots is not a
 * positive multiple of page_size, or out == NULL. */
rx_status rx_cache_create(const rx_config* cfg, rx_cache** out);
rx_status rx_cache_destroy(rx_cache* cache);

/* Copy the calling thread's last error text (NUL-terminated, truncated to
 * cap).  Returns the full length of the text. */
size_t rx_last_error(char* buf, size_t cap);

/* ------------------------------------------------------------------------
 * S1 match  ([T] "A tree, not a map", [B] "One tree for everybody")
 * ---------------------------------------------------------------------- */

/* Longest cached prefix of tokens[0..n) in whole pages, without side
 * effects (no split, no access-time update).  Used by the in-batch prefix
 * rule. */
rx_status rx_match_length(const rx_cache* cache, const int32_t* tokens,
                          int64_t n, int64_t* out_len);

/* Walk from the root as far as tokens[0..n) match, in whole pages (n is
 * truncated to whole pages, a match inside an edge rounded down to one).
 * Writes the matched prefix's slots to out_slots (caller capacity >= n), its
 * length to *out_len and the node whose root path is exactly that prefix to
 * *out_node (0 when nothing matched).  A match ending inside an edge splits
 * the edge there
 * (reading: so the returned node covers exactly the matched prefix).  The
 * access clock advances by one and every node on the matched path takes it.
 * Errors: RX_ERR_INVALID on NULL pointers or n < 0. */
rx_status rx_match_prefix(rx_cache* cache, const int32_t* tokens, int64_t n,
                          int32_t* out_slots, int64_t* out_len,
                          rx_node* out_node);

/* ------------------------------------------------------------------------
 * S2 lock  ([T] inc_lock_ref / dec_lock_ref, [L] step 2 and step 5)
 * ---------------------------------------------------------------------- */

/* lock_ref += 1 on the node and every ancestor (root excluded); a node whose
 * lock_ref goes 0 -> 1 moves its length from the evictable to the protected
 * count.  Locking the root is a no-op.
 * Errors: RX_ERR_INVALID for an unknown or evicted node. */
rx_status rx_lock(rx_cache* cache, rx_node node);

/* lock_ref -= 1 along the same path; 1 -> 0 moves the length back.
 * Errors: RX_ERR_INVALID unknown node; RX_ERR_STATE if any lock_ref on the
 * path is already 0 (nothing is changed then). */
rx_status rx_unlock(rx_cache* cache, rx_node node);

/* ------------------------------------------------------------------------
 * S3 allocate / evict  ([T] heap eviction, [L] "Worked example")
 * ---------------------------------------------------------------------- */

/* Take ceil(k / page_size) pages from the head of the free list and write
 * their first k slots, page after page, to out_slots[0..k) (the rest of the
 * last page belongs to the caller too).  If too few pages are free, first
 * evict (rx_evict) the shortfall.  If still short: RX_ERR_NO_SPACE, nothing
 * is allocated, and nodes evicted during the attempt stay evicted ("D would
 * have to wait"). */
rx_status rx_alloc(rx_cache* cache, int64_t k, int32_t* out_slots);

/* Evict unlocked leaves, least recent first (key: priority 0,
 * last_access_time, node id), each node whole; its pages join the free-list
 * tail in stored order; a parent that becomes childless and unlocked joins
 * the candidates.  Stops once >= k slots were freed or no candidate is left.
 * *out_freed = slots freed (may exceed k). */
rx_status rx_evict(rx_cache* cache, int64_t k, int64_t* out_freed);

/* Return the pages of the given slots to the free-list tail, each page once,
 * in the order of its first slot.  The caller must own those whole pages
 * (allocated and not held by the tree).  Errors: RX_ERR_INVALID for a slot in
 * the pad page or beyond the pool. */
rx_status rx_free(rx_cache* cache, const int32_t* slots, int64_t k);

/* ------------------------------------------------------------------------
 * S10 insert  ([B] "the divergent part becomes a new branch", [L] step 4)
 * ---------------------------------------------------------------------- */

/* Insert the whole pages of tokens[0..n) with their slots (n truncated to
 * whole pages).  Walks and splits as rx_match_prefix; the uncached remainder
 * becomes one new leaf holding slots of that part.
 * *out_already = tokens that were already cached (the caller still owns its
 * own slots for that part and frees those beyond what it had locked);
 * *out_node = node ending exactly at n.  The access clock advances by one and
 * the whole path takes it. */
rx_status rx_insert(rx_cache* cache, const int32_t* tokens,
                    const int32_t* slots, int64_t n, int64_t* out_already,
                    rx_node* out_node);

/* ------------------------------------------------------------------------
 * Introspection
 * ---------------------------------------------------------------------- */
rx_status rx_stats(const rx_cache* cache, rx_stats_t* out);

/* Copy eviction records [start, start+cap) (in eviction order) to out;
 * *out_total = number of records since creation. */
rx_status rx_eviction_log(const rx_cache* cache, int64_t start,
                          rx_evict_rec* out, int64_t cap, int64_t* out_total);

/* Number of tokens on the root path of a node (its depth in tokens). */
rx_status rx_node_depth(const rx_cache* cache, rx_node node,
                        int64_t* out_depth);

/* ------------------------------------------------------------------------
 * Batch steps of the request flow ([L] "How RadixAttention reuses past
 * work"), composed from the calls above so one batch costs one call.
 * ---------------------------------------------------------------------- */

/* S1+S2+S3+S4 for an extend batch of R requests.  tokens holds the prompts
 * back to back, request r at [tok_indptr[r], tok_indptr[r+1]) (offsets need
 * not start at 0: a batch of a wave may pass the wave's tokens and its slice
 * of the wave's offsets; the same holds for rx_extend_end).  In request
 * order: rx_match_prefix on the prompt without its last token (the last prompt
 * token is always recomputed) and rx_lock of the matched node; then ONE
 * allocation of every request's ceil(new tokens / page_size) pages, handed
 * out in request order (a request's new tokens fill its own pages).  Writes
 *   req_to_token[r*row_stride + 0 .. n_r)  = matched slots ++ new slots,
 *   out_prefix_len[r], out_match_node[r],
 *   out_new_slots[0 .. total_new) = the new slots in request order (the K/V
 *   of the batch's new tokens are stored there), *out_total_new.
 * On RX_ERR_NO_SPACE every lock taken is released again (evictions stay).
 * Errors: RX_ERR_INVALID if a prompt is empty or longer than row_stride. */
rx_status rx_extend_begin(rx_cache* cache, int32_t R, const int32_t* tokens,
                          const int64_t* tok_indptr, int32_t* req_to_token,
                          int64_t row_stride, int32_t* out_prefix_len,
                          rx_node* out_match_node, int32_t* out_new_slots,
                          int64_t* out_total_new);

/* S10 after an extend batch: for each request in order rx_insert(prompt,
 * row) (its whole pages; a partly filled last page stays the request's),
 * rx_lock(prompt node), rx_unlock(matched node).  Writes
 * out_prompt_node[r].  If a prompt finds more of itself cached than its
 * match (an identical prompt was inserted by an earlier batch), the
 * request's own pages for that part go back to the free list and its row is
 * rewritten in place with the tree's slots (same tokens after the same
 * predecessors, so the same K/V); *out_rewritten (may be NULL) counts the
 * requests whose row changed, so the caller can refresh device rows. */
rx_status rx_extend_end(rx_cache* cache, int32_t R, const int32_t* tokens,
                        const int64_t* tok_indptr, int32_t* req_to_token,
                        int64_t row_stride, const int32_t* prefix_len,
                        const rx_node* match_node, rx_node* out_prompt_node,
                        int64_t* out_rewritten);

/* Finish (S10): for each request, rx_insert(prompt ++ outputs, row) where
 * tokens/tok_indptr hold prompt ++ outputs and the row holds their slots;
 * the request's pages past the prompt's whole pages that another request
 * had already inserted, and its partly filled last page, are freed; then
 * rx_unlock(prompt_node[r]).  out_already[r] and out_full_node[r] (the node
 * ending at the inserted sequence's last whole page) may be NULL. */
rx_status rx_finish(rx_cache* cache, int32_t R, const int32_t* tokens,
                    const int64_t* tok_indptr, const int32_t* req_to_token,
                    int64_t row_stride, const int64_t* prompt_len,
                    const rx_node* prompt_node, int64_t* out_already,
                    rx_node* out_full_node);

/* In-batch prefix rule ([T] "The scheduler is where the cache is won or
 * lost") at token granularity: *out_conflict = 1 if the common prefix of
 * tokens[0..n) with any of the R member prompts (concatenated as in
 * rx_extend_begin) is longer than match_len, else 0.  (rx_batch_end applies
 * the rule in whole pages of its cache.) */
rx_status rx_batch_conflict(const int32_t* tokens, int64_t n,
                            int64_t match_len, int32_t R,
                            const int32_t* member_tokens,
                            const int64_t* member_indptr,
                            int32_t* out_conflict);

/* The batch that starts at request `start` of a wave, under the same rule:
 * requests start, start+1, ... join it while request j's prompt shares no
 * more than m_j = rx_match_length(prompt_j minus its last token) tokens,
 * counted in whole pages, with every earlier member; *out_end = the first j
 * that would share more (it
 * starts the next batch), or R.  The cache is only read.  tokens/indptr hold
 * the wave's R prompts concatenated.  Errors: RX_ERR_INVALID (start not in
 * [0, R), an empty prompt). */
rx_status rx_batch_end(const rx_cache* cache, const int32_t* tokens,
                       const int64_t* indptr, int32_t start, int32_t R,
                       int32_t* out_end);

/* ------------------------------------------------------------------------
 * Two tiers: device pool + host pool ([T] "What the C++ tree is actually
 * for": match_prefix returns the device indices, the host-matched length
 * and a node per tier; writing_through / commit_writing_through; loading
 * onboard).  With rx_config.host_slots > 0 a node holds device slots, host
 * slots or both; the device-resident nodes hang from the root as a subtree,
 * and so do the host-resident ones.  Device eviction (rx_evict, and every
 * allocation) takes unlocked device leaves (no child on the device), least
 * recent first: a node backed up on the host gives up its device slots and
 * stays, a device-only node leaves the tree; the parent joins the
 * candidates once it has no child on the device.  A backup that needs host
 * pages evicts host-only childless nodes, least recent first.  The calls
 * only decide slots; the caller copies KV between the pools (rx_kv_copy)
 * in stream order before anything reads the destination.  With one tier
 * every call below finds nothing to move.
 * ---------------------------------------------------------------------- */

/* Walk every tier as rx_match_prefix does (split, touch).  Writes the slots
 * of the leading device-resident part of the match to out_slots, its length
 * to *out_device_len and its last node to *out_device_node; *out_host_len =
 * the tokens matched past it on the host only, *out_host_node = the last
 * node matched (== device node when *out_host_len is 0). */
rx_status rx_match_prefix_tiers(rx_cache* cache, const int32_t* tokens,
                                int64_t n, int32_t* out_slots,
                                int64_t* out_device_len, int64_t* out_host_len,
                                rx_node* out_device_node,
                                rx_node* out_host_node);

/* Bring the host-only nodes of node's root path to the device: device pages
 * are allocated for them (evicting as rx_alloc does, with the path's device
 * part locked meanwhile) and they become resident on both tiers.  Writes
 * the copies to make, host slot -> device slot, to out_host_slots /
 * out_device_slots (capacity cap), *out_n = their number (0: nothing to
 * load).  RX_ERR_NO_SPACE (nothing loaded) if the device cannot hold them. */
rx_status rx_load_onboard(rx_cache* cache, rx_node node,
                          int32_t* out_host_slots, int32_t* out_device_slots,
                          int64_t cap, int64_t* out_n);

/* Back up the device-only nodes of node's root path (which must be on the
 * device) to the host: host pages are allocated for them (evicting host-only
 * leaves if needed), node is locked until the commit, and the copies to
 * make, device slot -> host slot, are written (capacity cap); *out_n = their
 * number, *out_ticket = the ticket to commit.  *out_ticket = 0 and *out_n =
 * 0 when there is nothing to copy or a backup of a node on the path is
 * still in flight (retry after its commit).  RX_ERR_NO_SPACE if the host
 * tier cannot hold the path (nothing changes). */
rx_status rx_write_through(rx_cache* cache, rx_node node,
                           int32_t* out_device_slots, int32_t* out_host_slots,
                           int64_t cap, int64_t* out_n, int64_t* out_ticket);

/* Resolve a write-through: success != 0 makes the path resident on both
 * tiers; 0 returns its host pages.  The node is unlocked either way. */
rx_status rx_commit_write_through(rx_cache* cache, int64_t ticket,
                                  int32_t success);

/* Batch step before rx_extend_begin: for each request in order, match its
 * prompt without the last token across tiers and load a host-only remainder
 * (rx_load_onboard; a load the device cannot hold is skipped and that part
 * is prefilled).  Prompts as in rx_extend_begin.  Copies host slot ->
 * device slot of every load, request after request, to out_host_slots /
 * out_device_slots (capacity cap); *out_n = their number, out_counts[r] =
 * request r's share. */
rx_status rx_load_batch(rx_cache* cache, int32_t R, const int32_t* tokens,
                        const int64_t* indptr, int32_t* out_host_slots,
                        int32_t* out_device_slots, int64_t cap, int64_t* out_n,
                        int64_t* out_counts);

/* Batch step after rx_finish: rx_write_through of every node (in order,
 * e.g. rx_finish's out_full_node), each committed with success at once (the
 * caller's copies are stream-ordered before any later load); a backup the
 * host tier cannot hold is skipped.  Copies device slot -> host slot to
 * the output arrays (capacity cap); *out_n = their number, out_counts[r] =
 * node r's share. */
rx_status rx_write_through_batch(rx_cache* cache, int32_t R,
                                 const rx_node* nodes,
                                 int32_t* out_device_slots,
                                 int32_t* out_host_slots, int64_t cap,
                                 int64_t* out_n, int64_t* out_counts);

/* Host-tier eviction records [start, start+cap); *out_total = their count. */
rx_status rx_host_eviction_log(const rx_cache* cache, int64_t start,
                               rx_evict_rec* out, int64_t cap,
                               int64_t* out_total);

/* ------------------------------------------------------------------------
 * Cache-aware scheduling ([T] "The scheduler is where the cache is won or
 * lost"); host, reads the cache only.
 * ---------------------------------------------------------------------- */

#define RX_POLICY_FCFS 0       /* arrival order                              */
#define RX_POLICY_LPM 1        /* longest prefix match first                 */
#define RX_POLICY_DFS_WEIGHT 2 /* weighted depth-first order of the tree     */

/* Order in which a waiting queue of R prompts (concatenated, request r at
 * [indptr[r], indptr[r+1]), each non-empty) is served: out_order[k] = queue
 * position of the k-th request to serve.  Each request's match, against the
 * tree and against the queue tree below, is taken on its prompt without the
 * last token, in whole pages; sorts are stable (equal keys keep queue order).
 *   RX_POLICY_LPM: requests sorted by decreasing tree match.  A request
 *     whose tree match is at most 32 tokens is also matched against a radix
 *     tree over the waiting queue: sharing at least 32 tokens with a prompt
 *     already in it sends the request to the back (its sibling runs first
 *     and populates the tree), otherwise its prompt joins that queue tree.
 *     With more than 128 waiting requests LPM falls back to arrival order.
 *   RX_POLICY_DFS_WEIGHT: a request hangs off the deepest node whose whole
 *     root path its prompt matches; each node weighs the requests hanging in
 *     its subtree; the order is depth first from the root, a node's own
 *     requests (in queue order) before its children, heavier children first,
 *     ties by the queue position of the child subtree's earliest request.
 * Errors: RX_ERR_INVALID (unknown policy, empty prompt). */
rx_status rx_schedule(const rx_cache* cache, int32_t policy, int32_t R,
                      const int32_t* tokens, const int64_t* indptr,
                      int32_t* out_order);

/* A whole wave's extend bookkeeping in one call: starting at request 0,
 * each batch is found by rx_batch_end and run through rx_extend_begin and
 * rx_extend_end, exactly as those calls made batch by batch would (so the
 * slots, nodes and eviction order are the same).  tokens/indptr hold the
 * wave's R prompts; req_to_token rows 0 .. R-1 (row_stride) receive the
 * rows, as rx_extend_end leaves them.  Writes out_batch_end[b] (the request
 * that ends batch b, exclusive) for b < *out_n_batches, out_prefix_len[r],
 * out_prompt_node[r], out_new_slots (every batch's new slots, batch after
 * batch, request order within a batch: request r's new tokens' slots) and
 * out_batch_rewritten[b] (rows of batch b that rx_extend_end rewrote with
 * tree slots: the row a batch's kernels use is then its matched slots
 * followed by its new slots).  A failing batch returns its error with
 * *out_n_batches = the batches done before it (their effects kept, the
 * failing batch's locks released). */
rx_status rx_extend_wave(rx_cache* cache, int32_t R, const int32_t* tokens,
                         const int64_t* indptr, int32_t* req_to_token,
                         int64_t row_stride, int32_t* out_batch_end,
                         int32_t* out_n_batches, int32_t* out_prefix_len,
                         rx_node* out_prompt_node, int32_t* out_new_slots,
                         int64_t* out_batch_rewritten);

/* ------------------------------------------------------------------------
 * Decode plan (S7/S8 split; host)
 * ---------------------------------------------------------------------- */

/* Layout of the int32 plan written by rx_plan_decode (all offsets in int32
 * words from the start of the plan):
 *   work[n_work][RX_WORK_WORDS]: {req_to_token row, kv_begin, kv_end,
 *       member_off, n_members, part_base, n_rows (= n_members*G), 0}
 *       -- one CTA per work item and KV head attends the member requests'
 *       query heads of that KV head over keys row[kv_begin .. kv_end);
 *   members[n_member_entries]: decode batch index of each member;
 *   req_part_indptr[B+1], req_parts[n_parts]: partial results of request b
 *       are entries req_parts[req_part_indptr[b] .. req_part_indptr[b+1]).
 * Partial entry p of work item w's member i is part_base(w) + i.  Word 7 of a
 * work item is 0, or for a request's private tail the end of that tail at
 * step 0 of a multi-step plan: at step t the item's keys end at
 * min(kv_end, word7 + t) (an item left empty writes a zero partial with
 * lse = -inf, which the merge weighs 0). */
#define RX_WORK_WORDS 8
typedef struct rx_decode_plan_info {
  int64_t plan_words;     /* int32 words used                             */
  int64_t n_work;         /* work items (grid = n_work x num_kv_heads)    */
  int64_t n_parts;        /* partial (o, lse) entries                     */
  int64_t n_member_entries;
  int64_t off_work, off_members, off_req_part_indptr, off_req_parts;
  int64_t n_shared_segments; /* tree segments read by >= 2 requests       */
  int64_t workspace_bytes;   /* device scratch rx_decode_attention needs  */
  int64_t distinct_kv_tokens;/* distinct context tokens of the batch      */
  int64_t n_work_tc;      /* the last n_work_tc items have more than 16 rows
                             and run on the tensor-core tile role        */
  int64_t tails_private;  /* 1: at every step of the plan each request's
                             newest token lies in a private tail run by the
                             warp role (group <= 16), so
                             rx_decode_steps stores it inside that kernel */
} rx_decode_plan_info;

/* Plan one decode step for a batch of B requests.  prompt_node[b] is the
 * locked node ending at request b's cached path; ctx_len[b] is the request's
 * whole context length this step (cached path + decode tokens, the current
 * token included); req_rows[b] is its row in the device req_to_token table,
 * whose first ctx_len[b] entries must hold the context's slots.
 * A tree node on the path of >= 2 requests becomes a shared segment read once
 * for all of them as a multi-query tile; the rest of each context is that
 * request's private segment.  Any partition of a context into segments gives
 * the same attention after the log-sum-exp merge, so the plan affects speed
 * only.  Errors: RX_ERR_INVALID (unknown node, ctx_len shorter than the node
 * depth, plan_cap too small -- *out_info still reports plan_words). */
rx_status rx_plan_decode(const rx_cache* cache, int32_t B,
                         const rx_node* prompt_node, const int32_t* ctx_len,
                         const int32_t* req_rows, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim,
                         int32_t* plan, int64_t plan_cap,
                         rx_decode_plan_info* out_info);

/* One plan for n_steps consecutive decode steps of the same batch: the tree
 * does not change while the batch decodes (decode tokens stay outside it
 * until finish), so the shared segments stay the same and only each private
 * tail grows by one token per step.  ctx_len[b] is request b's context at
 * the first step (its token included); at step t it is ctx_len[b] + t, and
 * req_to_token rows must hold the slots of all n_steps tokens before the last
 * step runs.  distinct_kv_tokens counts step 0.  The kernels take the step
 * index through rx_decode_step.step. */
rx_status rx_plan_decode_steps(const rx_cache* cache, int32_t B, int32_t n_steps,
                               const rx_node* prompt_node, const int32_t* ctx_len,
                               const int32_t* req_rows, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t* plan, int64_t plan_cap,
                               rx_decode_plan_info* out_info);

/* n_steps consecutive rx_alloc(k) calls (one decode slot per request and
 * step), written to out_slots[t*k .. t*k+k).  RX_ERR_NO_SPACE at the first
 * step that cannot be served (earlier steps stay allocated).  Page size 1
 * only (RX_ERR_INVALID otherwise; use rx_alloc_decode_steps). */
rx_status rx_alloc_steps(rx_cache* cache, int64_t k, int32_t n_steps,
                         int32_t* out_slots);

/* Decode slots of n_steps steps for B requests at any page size.  Request
 * b's first decode token is at position pos0[b], right after the slot
 * last_slot[b] (the slot of position pos0[b]-1).  At step t, in request
 * order, a token whose position starts a page takes a new page (one
 * allocation per step of the pages that step needs, handed out in request
 * order, evicting as rx_alloc does) and gets its first slot; any other token
 * gets the slot after the request's previous one.  Writes
 * out_slots[t*B + b].  At page size 1 this equals rx_alloc_steps(B,
 * n_steps).  RX_ERR_NO_SPACE at the first step that cannot be served
 * (earlier steps stay allocated). */
rx_status rx_alloc_decode_steps(rx_cache* cache, int32_t B, int32_t n_steps,
                                const int32_t* pos0, const int32_t* last_slot,
                                int32_t* out_slots);

/* ------------------------------------------------------------------------
 * Device calls
 * ---------------------------------------------------------------------- */

/* A KV pool, owned by the caller.  Every device call checks it first:
 * both pointers non-NULL and 16-byte aligned, head_dim 128 or 256,
 * num_slots >= 2, L and Hkv > 0, and L * Hkv * num_slots < 2^31 (the
 * kernels address pool rows with 32-bit TMA coordinates); RX_ERR_INVALID
 * otherwise. */
typedef struct rx_pool_desc {
  void* k_pool;          /* device bf16 [L][Hkv][num_slots][head_dim]      */
  void* v_pool;          /* same layout                                    */
  int64_t num_slots;
  int32_t num_layers;
  int32_t num_kv_heads;
  int32_t head_dim;      /* 128 or 256                                     */
  int32_t reserved;
} rx_pool_desc;

/* S5 ([L] "A quick recap": a token's keys and values are stored in the
 * cache): K_pool[layer][h][d_slots[i]][:] = d_k[i][h][:], same for V, for
 * i < T.  d_k, d_v: device bf16 [T][Hkv][head_dim], 16-byte aligned.
 * Slots must be distinct.  A slot outside [1, num_slots) is skipped on the
 * device and reported by rx_device_check (bit 0).  Errors: RX_ERR_INVALID
 * (the pool, T < 0, NULL or misaligned inputs); T = 0 launches nothing. */
rx_status rx_kv_store(const rx_pool_desc* pool, int32_t layer,
                      const int32_t* d_slots, const void* d_k,
                      const void* d_v, int64_t T, rx_stream_t stream);

/* Device req_to_token append: d_table[d_rows[i]*row_stride + d_pos[i]] =
 * d_slots[i] for i < n (used to add decode tokens to device rows).  d_table
 * is device int32 [num_rows][row_stride]; d_rows, d_pos, d_slots device
 * int32 [n].  An entry whose row is outside [0, num_rows) or whose position
 * is outside [0, row_stride) is skipped on the device and reported by
 * rx_device_check (bit 4).  Errors: RX_ERR_INVALID (n < 0, num_rows < 0,
 * row_stride <= 0, a NULL array when n > 0); n = 0 launches nothing. */
rx_status rx_req_to_token_write(int32_t* d_table, int64_t num_rows,
                                int64_t row_stride, const int32_t* d_rows,
                                const int32_t* d_pos, const int32_t* d_slots,
                                int64_t n, rx_stream_t stream);

/* Host tile schedule for rx_extend_attention: tile_indptr[R+1] = prefix sums
 * of the query-row tiles of each request (request r has
 * (qo_indptr[r+1]-qo_indptr[r]) * Hq/Hkv rows per KV head, in tiles of 128
 * rows; an empty suffix has none).  Errors: RX_ERR_INVALID (NULL arrays,
 * R < 0, Hq % Hkv != 0, head_dim not 128 or 256, qo_indptr decreasing, 2^31
 * tiles or more). */
rx_status rx_extend_plan(const int32_t* qo_indptr, int32_t R,
                         int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t* tile_indptr,
                         int64_t* out_num_tiles);

/* S6 extend attention ([L] step 3: only the unmatched suffix is prefilled,
 * attending to the reused KV as if it had just been computed).
 * For request r (r < R) with prefix p = d_prefix_len[r] and suffix queries
 * i in [0, s_r), s_r = qo_indptr[r+1]-qo_indptr[r], query head h:
 *   o = softmax(scale * q . K[j]) V over keys j = 0 .. p+i of the request,
 * key j's K/V read from pool slot d_req_to_token[d_req_rows[r]*row_stride+j],
 * KV head h / (Hq/Hkv).  Inputs: d_q bf16 [total_q][Hq][head_dim] (request
 * r's queries at rows qo_indptr[r] ..), d_qo_indptr/d_tile_indptr [R+1],
 * d_prefix_len/d_req_rows [R] (all device int32), num_tiles from
 * rx_extend_plan.  Outputs: d_out fp32 [total_q][Hq][head_dim], d_lse fp32
 * [total_q][Hq] (natural log of the sum of exp of scaled scores).
 * Errors: RX_ERR_INVALID for head_dim not in {128, 256}, Hq % Hkv != 0,
 * layer out of range, misaligned pointers. */
rx_status rx_extend_attention(const rx_pool_desc* pool, int32_t layer,
                              const void* d_q, int32_t num_q_heads,
                              const int32_t* d_req_to_token,
                              int64_t row_stride, const int32_t* d_req_rows,
                              const int32_t* d_prefix_len,
                              const int32_t* d_qo_indptr,
                              const int32_t* d_tile_indptr, int32_t R,
                              int64_t num_tiles, float scale, float* d_out,
                              float* d_lse, rx_stream_t stream);

/* The extend batches of one wave for one layer, launched in order on one
 * stream: for batch i, rx_kv_store of its new tokens' K/V, then
 * rx_extend_attention of its requests (each with the arguments those calls
 * document).  Batch i + 1 may read KV that batch i stored, which the single
 * stream orders.  A batch's d_q, d_k, d_v hold its n_new suffix tokens
 * (n_new = d_qo_indptr[R]) and d_new_slots their slots; d_req_to_token with
 * row_stride holds the rows d_req_rows names.  events: NULL, or 4 events per
 * batch (rx_events_create) recorded before and after the store and before
 * and after the attention, for rx_event_elapsed_ms.  Stops at the first
 * error, with the batches before it launched. */
typedef struct rx_extend_batch {
  const void* d_q;               /* bf16 [n_new][Hq][head_dim]              */
  const void* d_k;               /* bf16 [n_new][Hkv][head_dim]             */
  const void* d_v;               /* bf16 [n_new][Hkv][head_dim]             */
  const int32_t* d_new_slots;    /* device int32 [n_new]                    */
  const int32_t* d_req_to_token; /* device int32 rows, row_stride apart     */
  const int32_t* d_req_rows;     /* device int32 [R]                        */
  const int32_t* d_prefix_len;   /* device int32 [R]                        */
  const int32_t* d_qo_indptr;    /* device int32 [R+1]                      */
  const int32_t* d_tile_indptr;  /* device int32 [R+1], from rx_extend_plan */
  float* d_out;                  /* fp32 [n_new][Hq][head_dim]              */
  float* d_lse;                  /* fp32 [n_new][Hq]                        */
  int64_t n_new;
  int64_t num_tiles;
  int64_t row_stride;
  int32_t R;
  int32_t reserved;
} rx_extend_batch;

rx_status rx_extend_batches(const rx_pool_desc* pool, int32_t layer,
                            int32_t num_q_heads, const rx_extend_batch* batches,
                            int32_t n, float scale, const rx_event_t* events,
                            rx_stream_t stream);

/* n timing events (cudaEventCreate) written to out[0 .. n); destroyed by
 * rx_events_destroy.  rx_event_elapsed_ms: milliseconds between two
 * recorded events (RX_ERR_CUDA while either is not complete). */
rx_status rx_events_create(int32_t n, rx_event_t* out);
rx_status rx_events_destroy(int32_t n, const rx_event_t* events);
rx_status rx_event_elapsed_ms(rx_event_t start, rx_event_t end, float* out_ms);

/* S7+S8+S9 decode attention ([L] "A quick recap": each new token attends
 * over the KV cache, its own K/V already stored).  For request b < B, query
 * head h: o = softmax(scale * q . K) V over its whole context, computed per
 * plan segment into partial (o, lse) entries of d_workspace and merged by
 * log-sum-exp: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
 * d_q bf16 [B][Hq][head_dim]; d_plan = device copy of the rx_plan_decode
 * plan; info = its host info.  d_workspace: caller-owned device scratch of at
 * least info->workspace_bytes, 16-byte aligned.  Outputs d_out fp32
 * [B][Hq][head_dim], d_lse fp32 [B][Hq]. */
rx_status rx_decode_attention(const rx_pool_desc* pool, int32_t layer,
                              const void* d_q, int32_t num_q_heads,
                              const int32_t* d_req_to_token,
                              int64_t row_stride, const int32_t* d_plan,
                              const rx_decode_plan_info* info, int32_t B,
                              float scale, float* d_out, float* d_lse,
                              void* d_workspace, size_t workspace_bytes,
                              rx_stream_t stream);

/* A run of decode steps planned ahead ([T] "The overlap that pays for
 * itself": the next batch is built from slot numbers, never from sampled
 * values, so allocation and planning run ahead of the GPU).  For each step
 * s < n_steps, in order on the stream: rx_kv_store of that step's new tokens
 * (steps[s].d_k / d_v at steps[s].d_slots, B tokens), then
 * rx_decode_attention with steps[s]'s plan, queries and outputs.  When the
 * plan's tails_private is 1 the store is not a launch of its own: the warp
 * that reads the chunk holding request b's newest token (position
 * ctx_len[b] + step - 1) first writes that token's K/V row to
 * steps[s].d_slots[b], then reads the chunk; the result is the same.  The
 * req_to_token rows must already hold every step's slots (a token's position
 * beyond a step's context is never read by that step).  d_workspace must hold
 * the largest steps[s].info->workspace_bytes.  Stops at the first error.
 * Errors: RX_ERR_INVALID (n_steps < 0, steps NULL, the pool, Hq % Hkv != 0,
 * and each step's as in rx_decode_attention). */
typedef struct rx_decode_step {
  const void* d_q;          /* bf16 [B][Hq][head_dim]                     */
  const void* d_k;          /* bf16 [B][Hkv][head_dim] new tokens' K      */
  const void* d_v;          /* bf16 [B][Hkv][head_dim] new tokens' V      */
  const int32_t* d_slots;   /* device int32 [B] new tokens' slots         */
  const int32_t* d_plan;    /* device copy of this step's plan            */
  const rx_decode_plan_info* info; /* host info of that plan             */
  float* d_out;             /* fp32 [B][Hq][head_dim]                     */
  float* d_lse;             /* fp32 [B][Hq]                               */
  int32_t step;             /* step index within a multi-step plan        */
  int32_t reserved;
} rx_decode_step;

rx_status rx_decode_steps(const rx_pool_desc* pool, int32_t layer,
                          int32_t num_q_heads, const int32_t* d_req_to_token,
                          int64_t row_stride, const rx_decode_step* steps,
                          int32_t n_steps, int32_t B, float scale,
                          void* d_workspace, size_t workspace_bytes,
                          rx_stream_t stream);

/* Decode attention that allocates nothing and takes no scratch buffer.  The
 * pages have no counterpart of this call; it exists for callers that cannot
 * supply device memory -- e.g. a host whose device memory is all reserved up
 * front by its own pool, or a plugin handed a stream and tensors but no
 * allocator.  Arguments and results are those of rx_decode_attention without
 * d_workspace / workspace_bytes; the partial results go to a fixed array of
 * RX_DECODE_STATIC_SCRATCH_BYTES inside the library's device image, which
 * every GPU that loads the library holds until the process exits.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 *   - A plan whose info->workspace_bytes exceeds the limit is rejected with
 *     RX_ERR_INVALID and a message; nothing is launched.
 *   - Every call shares the one array.  Calls that overlap on the GPU (other
 *     streams, or other threads) race on it; serialise them.  Nothing in the
 *     array needs to start at zero: each partial result is written before the
 *     merge reads it. */
#define RX_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
rx_status rx_decode_attention_static(const rx_pool_desc* pool, int32_t layer,
                                     const void* d_q, int32_t num_q_heads,
                                     const int32_t* d_req_to_token,
                                     int64_t row_stride, const int32_t* d_plan,
                                     const rx_decode_plan_info* info, int32_t B,
                                     float scale, float* d_out, float* d_lse,
                                     rx_stream_t stream);

/* ------------------------------------------------------------------------
 * Draft-tree verification and KV moves ([T] "Speculative decoding puts a
 * tree inside the tree")
 * ---------------------------------------------------------------------- */

/* Host: slot-table rows of the draft tokens of R requests.  Request r's
 * context before its draft tree is prefix_len[r] tokens whose slots are
 * prefix_rows[r*prefix_stride .. +prefix_len[r]); its drafts are
 * i in [draft_indptr[r], draft_indptr[r+1]) with parents[i] the index, local
 * to the request, of the draft that i continues (-1: i continues the last
 * verified token; a parent precedes its child) and draft_slots[i] the slot
 * its K/V is stored in.  Writes, per draft i: out_rows[i*out_stride ..] =
 * context slots ++ the slots of i's root path, root first, ending with i's
 * own; out_ctx_len[i] = prefix_len[r] + depth(i) + 1; out_positions[i] (may
 * be NULL) = prefix_len[r] + depth(i), the draft's sequence position.
 * Errors: RX_ERR_INVALID (a parent not before its child, a row longer than
 * out_stride). */
rx_status rx_verify_rows(int32_t R, const int32_t* prefix_len,
                         const int32_t* prefix_rows, int64_t prefix_stride,
                         const int64_t* draft_indptr, const int32_t* parents,
                         const int32_t* draft_slots, int32_t* out_rows,
                         int64_t out_stride, int32_t* out_ctx_len,
                         int32_t* out_positions);

/* Tree-masked attention of N draft tokens over the pool: draft i (query
 * d_q[i], bf16 [N][Hq][head_dim]) attends, with softmax, to the keys of its
 * row of d_req_to_token (its request's context, then its ancestors and
 * itself: exactly the tree mask).  The plan is rx_plan_decode over the
 * drafts with prompt_node = each draft's request's locked node, ctx_len =
 * out_ctx_len of rx_verify_rows and req_rows = the drafts' rows: the
 * context a request's drafts share is read once for all of them as a
 * multi-query tile.  The drafts' K/V must be stored first (rx_kv_store).
 * Arguments, outputs and errors as rx_decode_attention with B = N. */
rx_status rx_verify_attention(const rx_pool_desc* pool, int32_t layer,
                              const void* d_q, int32_t num_q_heads,
                              const int32_t* d_req_to_token,
                              int64_t row_stride, const int32_t* d_plan,
                              const rx_decode_plan_info* info, int32_t N,
                              float scale, float* d_out, float* d_lse,
                              void* d_workspace, size_t workspace_bytes,
                              rx_stream_t stream);

/* dst->k/v_pool[l][h][d_dst_slots[i]] = src->k/v_pool[l][h][d_src_slots[i]]
 * for i < n, every layer l and KV head h (device int32 slot lists).  With
 * src == dst it moves KV within the pool (the accepted path of a draft tree
 * to the slots the request's next positions use, move_kv_cache); with two
 * pools of the same shape it copies between them (e.g. the device pool and
 * a page-locked host pool the device reads and writes directly).  Within
 * one pool no target slot may be another entry's source.  A slot outside
 * [1, num_slots) of its pool skips the entry on the device and is reported
 * by rx_device_check (bit 5).  Errors: RX_ERR_INVALID (pools of different
 * shape, NULL or misaligned pools). */
rx_status rx_kv_copy(const rx_pool_desc* src, const rx_pool_desc* dst,
                     const int32_t* d_src_slots, const int32_t* d_dst_slots,
                     int64_t n, rx_stream_t stream);

/* Page-locked host memory of exactly `bytes` bytes, mapped into the device
 * address space and usable from every device (cudaHostAlloc, portable and
 * mapped): for a host pool that rx_kv_copy reads and writes directly, and
 * for host buffers that copies to and from the device run asynchronously
 * with.  Released with rx_host_free.  This is host memory: the library still
 * allocates no device memory.  Errors: RX_ERR_INVALID (bytes 0, out NULL),
 * RX_ERR_CUDA (the allocation failed; *out = NULL).  rx_host_free(NULL)
 * does nothing; freeing anything but a pointer from rx_host_alloc is
 * RX_ERR_CUDA. */
rx_status rx_host_alloc(size_t bytes, void** out);
rx_status rx_host_free(void* p);

/* Synchronise the current device and read the kernels' error words (then
 * clear them).  *out_flags (may be NULL): bit 0 = rx_kv_store met a slot
 * outside [1, num_slots) and skipped that write; bit 1 = an attention kernel
 * read a slot outside [0, num_slots) from req_to_token and used slot 0
 * instead; bit 2 = a tensor-core kernel gave up a barrier wait after its
 * time limit (about 2 s) and returned without results (every output of
 * that launch is void; its CTAs still wait, bounded, for the loads and
 * tensor-core operations they had issued before they exit); bit 3 = a
 * tensor-core tile found its dynamic shared memory off a 1024-byte boundary
 * and returned without results; bit 4 = rx_req_to_token_write met a row or
 * position outside the table and skipped that entry; bit 5 = rx_kv_copy met
 * a slot outside its pool and skipped that entry.  Returns RX_ERR_CUDA
 * if a flag was set or the device reported an error. */
rx_status rx_device_check(int32_t* out_flags);

/* Test hook (host fault injection): the k-th page allocation from now, on
 * the device or the host pool (counted together, k >= 1), fails with
 * RX_ERR_NO_SPACE after the evictions it would do anyway, exactly as if the
 * pool were still short; every call then takes its documented failure path
 * (locks released, nothing allocated, evictions kept).  k = 0 turns the
 * hook off.  Not for production use. */
rx_status rx_debug_fail_alloc(rx_cache* cache, int64_t k);

/* Library build information (kernel variant names, compiled arch). */
const char* rx_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* RX_H */
