/*
 * rx.h -- C ABI of the prefix-shared KV attention library (librx.so).
 *
 * What the library does.  "SGLang: Efficient Execution of Structured Language
 * Model Programs" (unite.ai, es), section "Introducción a SGLang", describes
 * RadixAttention: the KV cache of finished generation calls is kept, as an
 * LRU cache inside a radix tree with matching, insertion and eviction, so that
 * calls sharing a prefix reuse its KV instead of recomputing it.  This library
 * is the data-parallel hot path under that cache:
 *
 *   - a token-slot KV pool on the GPU: K and V are separate bf16 arrays of
 *     shape [num_slots, num_kv_heads, head_dim], row-major, one row per token;
 *   - per-request slot lists (req_to_token): row r of an int32 matrix with
 *     leading dimension rtt_stride lists the pool slots of request r's tokens
 *     in position order; requests that share a prefix list the same slots;
 *   - rx_kv_store: scatter of new K/V rows into the pool;
 *   - rx_attn_extend: new tokens attend causally to their cached prefix plus
 *     themselves;
 *   - rx_attn_decode: one query per request over its whole slotted context,
 *     reading KV shared by several requests once per group when a decode plan
 *     says which requests share which positions;
 *   - a host radix tree (rx_match_prefix / rx_insert / rx_evict_lru) and a
 *     slot free list, which only produce slot ids and prefix lengths.
 *
 * Around that path:
 *   - cache-aware scheduling over the tree (rx_prefix_len, rx_schedule);
 *   - radix keys for an image's tokens (rx_image_keys);
 *   - the rotary position embedding, in place and fused into the scatter
 *     (rx_rope, rx_kv_store_rope);
 *   - FP8 (E4M3) pools and their scatter (rx_kv_store_fp8);
 *   - the compressed finite-state machine of constrained decoding
 *     (rx_fsm_compress on the host, rx_fsm_step on the device).
 *
 * Attention definition (all attention entry points).  For a query row of
 * request b at absolute position p, q-head h, with G = num_q_heads /
 * num_kv_heads and kv-head g = h / G:
 *     s_j = sm_scale * sum_c q[c] * K[req_to_token[b][j]][g][c],  j = 0 .. p
 *     o   = sum_j softmax(s)_j * V[req_to_token[b][j]][g]
 *     lse = log(sum_j exp(s_j))            (natural log)
 * Inputs are bf16; products, sums and the softmax run in fp32; o is rounded
 * to bf16 (round to nearest even).  The causal mask is the "j <= p" bound.
 *
 * Conventions.
 *   - Every function returns an int status: RX_OK (0) or a negative RX_ERR_*.
 *     rx_last_error() returns a thread-local message for the last failure.
 *   - No exception, abort or device trap crosses this ABI.
 *   - "device" pointers are CUDA global memory on the current device; "host"
 *     pointers are ordinary process memory.  The caller owns every buffer;
 *     the library allocates no device memory.  bf16 tensors (pools, q, o, new
 *     K/V) must start on a 16-byte boundary (RX_ERR_INVALID otherwise).
 *   - GPU entry points are asynchronous on `stream` (a cudaStream_t passed as
 *     void*, NULL = legacy default stream) and return after validation and
 *     launch.  Errors found by kernels (an out-of-range slot id or length) are OR-ed as
 *     RX_DEV_* bits into *dev_status, a device int32 the caller zeroes; a row
 *     with a bad slot reads as zeros and nothing outside the buffers is
 *     touched.  dev_status may be NULL (bad slots are then skipped silently).
 *   - Host tree functions are not thread-safe per tree; distinct trees are
 *     independent.
 */
#ifndef RX_H
#define RX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status ------------------------------------------------------------ */

#define RX_OK 0
#define RX_ERR_INVALID (-1)     /* null pointer, bad size or shape            */
#define RX_ERR_CAPACITY (-2)    /* caller's output array too small            */
#define RX_ERR_NOMEM (-3)       /* host allocation failed                      */
#define RX_ERR_NOT_ENOUGH (-4)  /* fewer slots/tokens available than asked     */
#define RX_ERR_CUDA (-5)        /* a CUDA runtime call failed                  */
#define RX_ERR_UNSUPPORTED (-6) /* shape the kernels are not built for         */

#define RX_DEV_BAD_SLOT 1       /* a kernel met a slot id outside the pool     */
#define RX_DEV_BAD_LEN 2        /* a device length exceeded its host bound or
                                   the req_to_token stride; rows left unwritten */
#define RX_DEV_TIMEOUT 4        /* a pipeline wait gave up (never expected; the
                                   kernel stopped early, outputs incomplete)   */
#define RX_DEV_FSM_DONE 8       /* rx_fsm_step: a request's state allows no
                                   token (its constrained text is complete)    */
#define RX_DEV_BAD_STATE 16     /* rx_fsm_step: a state id outside the machine,
                                   or a mask bit with no matching edge          */

/* Message for the last failed call on this thread ("" if none). */
const char *rx_last_error(void);

/* ABI version (bumped on any change of a signature or of a buffer
 * contract, such as a workspace size). */
int rx_version(void);

/* ---- radix tree (host) --------------------------------------------------
 * Source: "SGLang: Efficient Execution of Structured Language Model
 * Programs" (unite.ai, es), "Introducción a SGLang" (RadixAttention bullet:
 * LRU cache of KV inside a radix tree with matching, insertion, eviction) and
 * "SGLang: Modelo de programación y metodología" (nine-step walkthrough:
 * edges labelled with token sequences; an extension becomes a new node; a
 * partial share splits a node; least recently used nodes are evicted).
 *
 * Keys are int64 token ids; values are int32 pool slots, one per token.
 * Node boundaries follow the history of inserts: an insert that extends a
 * cached sequence adds its new tokens as one new leaf node; an insert that
 * leaves a node strictly inside it splits the node there; nodes are never
 * merged.  A logical clock advances once per rx_match_prefix / rx_insert /
 * rx_lock_prefix call, and every node holding at least one token of that
 * call's matched path takes the new value.  rx_evict_lru removes whole leaf
 * nodes with no lock, least recently used first.
 */
typedef struct rx_tree rx_tree;

int rx_tree_create(rx_tree **out);
void rx_tree_destroy(rx_tree *tree);

/* Longest cached prefix of tokens[0..n).  Writes its slot ids to
 * out_slots[0..prefix_len) (host, capacity out_cap) and its length to
 * *out_prefix_len.  Touches the LRU clock on the matched path; never changes
 * the tree's shape.  RX_ERR_CAPACITY if out_cap < prefix_len (nothing written
 * to out_slots, *out_prefix_len still set). */
int rx_match_prefix(rx_tree *tree, const int64_t *tokens, int64_t n, int32_t *out_slots,
                    int64_t out_cap, int64_t *out_prefix_len);

/* Cache tokens[0..n) with slots[0..n).  *out_already_cached = length of the
 * leading part that was cached before the call; that part keeps the tree's
 * slots and the caller owns (and should free) its own slots[0..already). */
int rx_insert(rx_tree *tree, const int64_t *tokens, const int32_t *slots, int64_t n,
              int64_t *out_already_cached);

/* Evict leaf nodes, least recently used first, until at least num_tokens
 * slots are freed or nothing unlocked is left.  Freed slot ids go to
 * out_freed (host, capacity out_cap), node by node, each node in token
 * order; *out_num_freed is their count.  The last node may overshoot
 * num_tokens.  Returns RX_ERR_NOT_ENOUGH when fewer than num_tokens could be
 * freed (what was freed is still reported) and RX_ERR_CAPACITY when the next
 * node would not fit in out_cap (the nodes before it are evicted and
 * reported; call again with room). */
int rx_evict_lru(rx_tree *tree, int64_t num_tokens, int32_t *out_freed, int64_t out_cap,
                 int64_t *out_num_freed);

/* Lock (delta = +1) or unlock (delta = -1) the cached prefix of
 * tokens[0..n): each of its tokens gets its lock count changed by delta, and a
 * node holding any locked token is never evicted.  Locking touches the LRU
 * clock like a match; unlocking does not.  *out_len gets the prefix length.
 * Unlock with exactly the tokens a lock reported (n = its *out_len): more may
 * be cached by then.  RX_ERR_INVALID (nothing changed) when unlocking a token
 * whose count is zero. */
int rx_lock_prefix(rx_tree *tree, const int64_t *tokens, int64_t n, int32_t delta,
                   int64_t *out_len);

/* Cached token count, node count (root excluded) and evictable token count. */
int rx_tree_stats(rx_tree *tree, int64_t *cached_tokens, int64_t *num_nodes,
                  int64_t *evictable_tokens);

/* Structure dump for tests and tools: for every node in depth-first order
 * (children by ascending first token) writes the int64 record
 *   [node_id, parent_id (-1 under the root), last_access, n_tokens,
 *    tokens[n_tokens], slots[n_tokens], lock_counts[n_tokens]]
 * to out (host, capacity out_cap words).  *out_len = words written, or needed
 * when RX_ERR_CAPACITY is returned. */
int rx_tree_dump(rx_tree *tree, int64_t *out, int64_t out_cap, int64_t *out_len);

/* ---- slot free list (host) ----------------------------------------------
 * Hands out pool slots in the order given at creation, takes freed slots back
 * at the tail (first in, first out). */
typedef struct rx_slot_alloc rx_slot_alloc;

/* free_order: host int32 [n], distinct values in [0, num_slots). */
int rx_slot_alloc_create(const int32_t *free_order, int64_t n, int64_t num_slots,
                         rx_slot_alloc **out);
void rx_slot_alloc_destroy(rx_slot_alloc *a);
/* Takes n slots into out (host).  RX_ERR_NOT_ENOUGH (nothing taken) if fewer are free. */
int rx_slot_alloc_take(rx_slot_alloc *a, int64_t n, int32_t *out);
/* Returns n slots.  RX_ERR_INVALID (nothing returned) on an out-of-range id. */
int rx_slot_alloc_give(rx_slot_alloc *a, const int32_t *slots, int64_t n);
int64_t rx_slot_alloc_free_count(const rx_slot_alloc *a);

/* ---- request admission (host) -------------------------------------------
 * Prefix match and slot assignment for one request, in one call:
 * matches tokens[0..n), locks the matched path, takes n - prefix_len fresh
 * slots from `alloc` (first evicting least recently used unlocked nodes into
 * `alloc` when it is short) and writes the request's full slot list to
 * out_row[0..n) (host): cached slots first, then the fresh ones.
 * *out_prefix_len = cached length, *out_evicted = tokens evicted.
 * RX_ERR_NOT_ENOUGH (lock released, nothing taken) if the pool cannot hold
 * the request. */
int rx_admit(rx_tree *tree, rx_slot_alloc *alloc, const int64_t *tokens, int64_t n,
             int32_t *out_row, int64_t *out_prefix_len, int64_t *out_evicted);

/* After the request's KV is in the pool: unlocks the path locked by rx_admit
 * (prefix_len tokens), inserts tokens[0..n) with row[0..n), and returns to
 * `alloc` the fresh slots whose tokens turned out to be cached already. */
int rx_commit(rx_tree *tree, rx_slot_alloc *alloc, const int64_t *tokens, const int32_t *row,
              int64_t n, int64_t prefix_len);

/* ---- cache-aware scheduling (host) ---------------------------------------
 * Source: "SGLang: Efficient Execution of Structured Language Model
 * Programs" (unite.ai, es), "SGLang: Evaluación y resultados": SGLang's
 * cache-aware scheduling reaches about 96 % of the optimal cache hit rate on
 * average.  The pages do not spell the policy out; the reading taken is the
 * plain one: among the waiting requests, those with the longest cached prefix
 * run first (they reuse it while it is resident), ties in arrival order.
 * The hit rate is the share of prompt tokens found cached at admission; the
 * optimum computes every distinct prefix token once. */
#define RX_SCHED_FCFS 0   /* arrival order                                 */
#define RX_SCHED_LPM 1    /* longest cached prefix first, ties by arrival  */

/* Length of the longest cached prefix of tokens[0..n) (host) in *out_len.  A
 * probe: the LRU clock is not touched. */
int rx_prefix_len(rx_tree *tree, const int64_t *tokens, int64_t n, int64_t *out_len);

/* Orders n_req waiting requests.  Request i's tokens are tokens[offsets[i] ..
 * offsets[i+1]) (host int64; offsets has n_req + 1 entries, offsets[0] = 0,
 * non-decreasing).  Writes request i's cached prefix length (a probe, as in
 * rx_prefix_len) to out_prefix_len[i] and the order to run them in to
 * out_order[0..n_req), a permutation of 0 .. n_req-1 (host int32).  policy:
 * RX_SCHED_FCFS or RX_SCHED_LPM.  RX_ERR_INVALID (nothing written) on bad
 * offsets or policy. */
int rx_schedule(rx_tree *tree, const int64_t *tokens, const int64_t *offsets, int32_t n_req, int32_t policy,
                int32_t *out_order, int64_t *out_prefix_len);

/* ---- multimodal keys (host) ---------------------------------------------
 * Source: "SGLang: Efficient Execution of Structured Language Model
 * Programs" (unite.ai, es), "SGLang: Evaluación y resultados", multimodal
 * results: RadixAttention computes the hash of each input image and uses it
 * as the key in the radix tree, so requests about the same image reuse the
 * KV of its tokens.  rx_image_keys gives the keys of the n_tokens positions an
 * image occupies in a request's key sequence: key i (0-based) is output i + 1
 * of the SplitMix64 generator seeded with the 64-bit FNV-1a hash of the
 * image's bytes, with the top bit set -- negative as int64, so no image key
 * equals a text token id (those are >= 0).  Identical bytes give identical
 * keys; other bytes give other keys except with probability about
 * n_tokens^2 / 2^63.  out_keys: host int64 [n_tokens]. */
int rx_image_keys(const uint8_t *data, int64_t nbytes, int64_t n_tokens, int64_t *out_keys);

/* ---- KV pool (device) ----------------------------------------------------
 * K and V of one layer, or of a model's L layers in one allocation each.
 * With num_layers L > 1, k and v point to [L, num_slots, num_kv_heads,
 * head_dim] arrays and a call reads or writes layer `layer` only: the
 * layer's rows start layer * num_slots * num_kv_heads * head_dim elements
 * after k (v alike).  A slot id names the same token in every layer, so one
 * radix tree, one slot list per request and one decode plan serve all
 * layers.  num_layers 0 or 1 is a one-layer pool (layer must be 0); a layer
 * outside [0, L) is RX_ERR_INVALID. */
typedef struct {
    void *k;              /* device bf16 [num_layers,] num_slots, num_kv_heads, head_dim */
    void *v;              /* device bf16, same shape                                     */
    int64_t num_slots;
    int32_t num_kv_heads;
    int32_t head_dim;     /* 64 or 128                                                   */
    int32_t num_layers;   /* 0 or 1: one layer; L > 1: k and v hold L layers             */
    int32_t layer;        /* the layer this call reads or writes                         */
} rx_kv_pool;

/* KV slot scatter: K[slots[i]] = k_new[i], V[slots[i]] = v_new[i] for i < n.
 * k_new, v_new: device bf16 [n, num_kv_heads, head_dim]; slots: device int32
 * [n], distinct (duplicates race: one of the rows wins).  16-byte aligned
 * pointers required.  Source: the reuse of stored KV across calls,
 * "SGLang: Efficient Execution of Structured Language Model Programs",
 * "Introducción a SGLang", RadixAttention bullet. */
int rx_kv_store(const rx_kv_pool *pool, const void *k_new, const void *v_new, const int32_t *slots,
                int64_t n, int32_t *dev_status, void *stream);

/* ---- FP8 key/value pools (device) ---------------------------------------
 * Not from the pages, which do not speak of reduced-precision KV: a pool of
 * OCP FP8 E4M3 codes ("fn": bias 7, subnormals m/8 * 2^-6, no infinities,
 * largest finite 448), one byte per value in the [S, Hkv, d] layout, with
 * one fp32 scale per pool.  The value a code stands for is E4M3(code) *
 * scale, half the bytes of a bf16 pool.
 *
 * rx_kv_store_fp8: for each i < n, K[slots[i]] = E4M3(k_new[i] / k_scale)
 * and the same for V, where the division is a correctly rounded fp32
 * division of the bf16 value, the code is the nearest (ties to the even
 * mantissa), magnitudes past 448 saturate to 448 and NaN stays NaN.
 * k_new, v_new: device bf16 [n, Hkv, d], 16-byte aligned; pools 8-byte
 * aligned; Hkv * d a multiple of 8.  A slot id outside the pool sets
 * RX_DEV_BAD_SLOT and its row is not written.  rx_attn_decode_fp8 and
 * rx_attn_extend_fp8 read such pools. */
typedef struct {
    void *k;          /* device uint8 [num_layers,] num_slots, num_kv_heads, head_dim */
    void *v;
    int64_t num_slots;
    int32_t num_kv_heads;
    int32_t head_dim;
    float k_scale;    /* > 0 */
    float v_scale;    /* > 0 */
    int32_t num_layers;   /* as in rx_kv_pool */
    int32_t layer;
} rx_kv_pool_fp8;

int rx_kv_store_fp8(const rx_kv_pool_fp8 *pool, const void *k_new, const void *v_new, const int32_t *slots,
                    int64_t n, int32_t *dev_status, void *stream);


/* ---- rotary position embedding (device) --------------------------------
 * Not from the pages, which do not reach inside the model: the position
 * encoding that the Llama-family models whose attention shapes the workloads
 * take apply to q and k before attention, in its rotate-half form.  For a
 * token at position p, every head, and c < head_dim / 2, with
 * theta_c = base^(-2c / head_dim) and a = p * theta_c:
 *     x'[c]                = x[c] cos a - x[c + head_dim/2] sin a
 *     x'[c + head_dim / 2] = x[c + head_dim/2] cos a + x[c] sin a
 * theta_c / (2 pi) is tabulated on the host as a 64-bit fraction of a turn,
 * so p * theta_c is reduced modulo 2 pi exactly in integer arithmetic (to the
 * table's 2^-53 relative rounding) at any position; sine and cosine, and the
 * rotation, in fp32; results rounded to bf16.
 * head_dim 64 or 128; base > 1 (10000 and 500000 are usual). */

/* In place on x: device bf16 [n, heads, head_dim], 16-byte aligned; pos:
 * device int32 [n], the tokens' positions. */
int rx_rope(void *x, const int32_t *pos, int64_t n, int32_t heads, int32_t head_dim, double base,
            void *stream);

/* rx_kv_store with K rotated on the way into the pool: K[slots[i]] =
 * rope(k_new[i], pos[i]) as rx_rope computes it, V[slots[i]] = v_new[i].
 * Same buffers and errors as rx_kv_store, plus pos: device int32 [n]. */
int rx_kv_store_rope(const rx_kv_pool *pool, const void *k_new, const void *v_new, const int32_t *slots,
                     const int32_t *pos, int64_t n, double base, int32_t *dev_status, void *stream);

/* rx_kv_store_rope into FP8 pools: K[slots[i]] = the codes rx_kv_store_fp8
 * stores for rope(k_new[i], pos[i]) as rx_rope computes it (rotated, rounded
 * to bf16), V[slots[i]] = the codes of v_new[i].  Same buffers and errors as
 * rx_kv_store_fp8, plus pos and base as in rx_kv_store_rope. */
int rx_kv_store_rope_fp8(const rx_kv_pool_fp8 *pool, const void *k_new, const void *v_new,
                         const int32_t *slots, const int32_t *pos, int64_t n, double base, int32_t *dev_status,
                         void *stream);

/* Extend attention.  Request b (b < batch) has prefix_len[b] cached tokens and
 * extend_len[b] new ones whose K/V are already in the pool; the slot list is
 * req_to_token row req_idx[b], positions 0 .. prefix_len[b]+extend_len[b]-1.
 * New token i of request b sits at position prefix_len[b] + i and attends to
 * positions 0 .. prefix_len[b] + i (the extend pass over a reused prefix:
 * "SGLang: Efficient Execution of Structured Language Model Programs",
 * "Introducción a SGLang", RadixAttention bullet).
 *   q:  device bf16 [sum(extend_len), num_q_heads, head_dim], request b's
 *       tokens at rows qo_indptr[b] .. qo_indptr[b+1]-1;
 *   o:  device bf16, same shape as q;  lse_or_null: device fp32
 *       [sum(extend_len), num_q_heads] or NULL;
 *   qo_indptr: device int32 [batch+1]; req_idx, prefix_len, extend_len:
 *       device int32 [batch]; req_to_token: device int32, row stride
 *       rtt_stride;
 *   max_extend_len: host bound on extend_len[b] (sizes the grid; larger
 *       device values are an error that leaves rows unwritten);
 *   workspace, ws_bytes: NULL / 0, or device memory of at least
 *       rx_attn_extend_workspace(...) bytes, 256-byte aligned, owned by the
 *       caller and not used by anything else until the call's work on
 *       `stream` is done.  With a workspace the call first copies every
 *       request's context rows out of the pool into it, packed per request,
 *       and the attention kernel then streams them with tiled TMA loads;
 *       without one the attention kernel gathers rows through the slot list
 *       itself.  Both give the same result.  Contexts that sum to more rows
 *       than the workspace was sized for set RX_DEV_BAD_LEN and leave every
 *       output row unwritten.
 * Requires head_dim 64 or 128, num_q_heads % num_kv_heads == 0 and
 * 128 % (num_q_heads / num_kv_heads) == 0. */
int rx_attn_extend(const rx_kv_pool *pool, const void *q, void *o, float *lse_or_null,
                   int32_t num_q_heads, const int32_t *qo_indptr, const int32_t *req_idx,
                   const int32_t *prefix_len, const int32_t *extend_len,
                   const int32_t *req_to_token, int64_t rtt_stride, int32_t batch,
                   int32_t max_extend_len, void *workspace, size_t ws_bytes, float sm_scale,
                   int32_t *dev_status, void *stream);

/* Workspace bytes for rx_attn_extend over `batch` requests whose contexts
 * (prefix_len[b] + extend_len[b]) sum to at most total_ctx_tokens; 0 on an
 * invalid argument (rx_last_error says which). */
size_t rx_attn_extend_workspace(int64_t total_ctx_tokens, int32_t batch, int32_t num_kv_heads,
                                int32_t head_dim);

/* ---- decode -------------------------------------------------------------
 * Source: "SGLang: Efficient Execution of Structured Language Model
 * Programs" (unite.ai, es), "Introducción a SGLang", RadixAttention bullet:
 * later calls reuse the KV cache of the prefixes they share.  Reading a
 * shared prefix's KV from HBM once for all the requests below it, by way of
 * a plan that groups those requests, is this library's design, not the
 * pages'.
 *
 * Decode plan: which requests of the batch share which positions, so that a
 * shared segment's KV is read once for all of them.  Built on the host by
 * rx_decode_plan_build from the host copy of req_to_token; the caller copies
 * the packed buffer to the device and fills this struct with device pointers
 * into that copy (see rx_decode_plan_build for the layout).
 *
 * A plan outlives the step it was built for.  A request's last position is
 * never part of a shared segment, so every request ends in a piece of its
 * own, and that piece's pos_end is RX_PLAN_OPEN_END: the kernels end it at
 * the request's seq_len when the plan is used.  The same plan therefore
 * serves every later decode step of the batch -- each request one token
 * longer, its earlier slot ids unchanged -- with no host work; rebuild it
 * when the batch's requests change.  (Later steps reuse the split of the
 * first: a request's last piece grows by one position per step.)
 */
#define RX_PLAN_OPEN_END (-1)

typedef struct {
    const int32_t *order;   /* device int32 [batch]: batch index of each plan row   */
    const int32_t *nparts;  /* device int32 [batch]: partial results per request    */
    const int32_t *items;   /* device int32 [n_items * 8]: work items               */
    int32_t n_items;
    int32_t max_parts;      /* largest nparts[b]                                     */
    int32_t n_wide;         /* the last n_wide items are all-heads items (from
                               rx_decode_plan_info.n_wide; 0 is always valid)   */
} rx_decode_plan;

typedef struct {
    int32_t n_items;
    int32_t max_parts;
    int32_t n_segments;     /* shared segments found (groups of >= 2 requests)  */
    int32_t kv_chunk;       /* positions per work item that the plan used       */
    int64_t shared_tokens;  /* positions inside shared segments, counted once   */
    int64_t tokens_read;    /* KV token rows the plan reads per kv head: shared
                               segments once, everything else once per request */
    int64_t buf_words;      /* int32 words of the packed buffer                 */
    int32_t n_wide;         /* all-heads items at the end of the list, read
                               across all kv heads at once (whole slot rows).
                               With one q head per kv head: the items that
                               hold a single request.  With 8 kv heads and
                               G = 2, 4, 8 or 16 q heads each: those, and the
                               items of shared segments cut into groups of up
                               to 16 / G requests (16 query rows per kv head)
                               when a chunk makes at most 16 such groups.
                               Otherwise 0.                                   */
} rx_decode_plan_info;

/* Builds a decode plan.  Inputs (host): req_to_token (row stride rtt_stride),
 * req_idx [batch], seq_len [batch] (> 0); num_q_heads, num_kv_heads;
 * kv_chunk = positions per work item (multiple of 64, <= 4096; 0 picks one:
 * about 1216 work items over all kv heads; with all-heads items, shared
 * chunks for about 76 per-head items -- or 152 (chunk, kv head) pairs when
 * they go to the all-heads kernel in request groups -- and private pieces
 * of about 1/304 of the batch's private positions); min_shared =
 * shortest shared segment worth grouping (>= 1).  Requests whose slot lists
 * agree on positions [a, b) (same slot at every position, from position 0 on)
 * form a segment; segments nest like the radix tree the slots came from.
 * Packed output (host int32, capacity out_cap words): order [batch], nparts
 * [batch], then items [n_items][8] = {first plan row, row count, pos_begin,
 * pos_end, part index, is_final, req_to_token row of the first request (its
 * req_idx), batch index of the first request}.  Per-head items come first,
 * then the info->n_wide all-heads items; within each part, items holding
 * several requests come before single-request ones, each ordered longest
 * first.  RX_ERR_CAPACITY (info->buf_words set) if out_cap is too small.
 * rx_attn_decode flags RX_DEV_BAD_LEN for an all-heads item with more
 * requests than its kernel takes (and reads it as its first request). */
int rx_decode_plan_build(const int32_t *req_to_token, int64_t rtt_stride, const int32_t *req_idx,
                         const int32_t *seq_len, int32_t batch, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t kv_chunk, int32_t min_shared,
                         int32_t *out_buf, int64_t out_cap, rx_decode_plan_info *info);

/* Workspace bytes rx_attn_decode needs: fp32 partial results when a request
 * is split over several work items, plus 256 bytes for a work counter when
 * the plan has single-request ("wide") items that run on the all-heads
 * kernel; 0 when neither applies.  With plan == NULL the split is chosen
 * from batch and max_seq_len. */
size_t rx_attn_decode_workspace(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_seq_len,
                                const rx_decode_plan *plan_or_null);

/* Decode attention: one query per request b at position seq_len[b]-1 over
 * positions 0 .. seq_len[b]-1 of req_to_token row req_idx[b] (its own new K/V
 * must already be in the pool).
 *   q, o: device bf16 [batch, num_q_heads, head_dim]; lse_or_null: device fp32
 *   [batch, num_q_heads] or NULL; req_idx, seq_len: device int32 [batch];
 *   max_seq_len: host bound on seq_len (sizes the grid without a plan);
 *   plan_or_null: device plan from rx_decode_plan_build for this batch, or
 *   NULL for one work split per request;
 *   workspace: device, >= rx_attn_decode_workspace(...) bytes, 256-byte
 *   aligned, contents ignored on entry and undefined after the call
 *   (partial results of split work, whose cache lines the merge discards
 *   once read).
 * Requires head_dim in {64, 128}, num_q_heads % num_kv_heads == 0 and
 * 64 % (num_q_heads / num_kv_heads) == 0. */
int rx_attn_decode(const rx_kv_pool *pool, const void *q, void *o, float *lse_or_null,
                   int32_t num_q_heads, const int32_t *req_idx, const int32_t *seq_len,
                   const int32_t *req_to_token, int64_t rtt_stride, int32_t batch,
                   int32_t max_seq_len, const rx_decode_plan *plan_or_null, void *workspace,
                   size_t ws_bytes, float sm_scale, int32_t *dev_status, void *stream);

/* ---- decode without a caller workspace ----------------------------------
 * The pages have no counterpart to this entry point; it exists for callers of
 * this library that cannot give it device scratch memory -- for example an
 * engine that commits all device memory at start-up (most of it to the KV
 * pool) and allows no allocator calls while serving, or a host program that
 * only lends its own buffers for inputs and outputs.
 *
 * Same arguments and results as rx_attn_decode, without workspace/ws_bytes:
 * the partial results of split work go to a fixed device array of
 * RX_DECODE_STATIC_SCRATCH_BYTES owned by the library (every GPU that loads
 * the library holds one until the process exits).  The call allocates
 * nothing.  Its first call with a given device current looks up that
 * device's array address (cudaGetSymbolAddress) and keeps it; make that
 * first call before any stream capture.  Every call shares the one array,
 * so calls that overlap on the GPU (different streams, or different host
 * threads without ordering) race; calls ordered on one stream are safe.
 * Nothing needs clearing by the caller: every partial result a call reads
 * from the array it has written earlier in the same call, and the call
 * zeroes the one counter it keeps there before its kernels start.  A device
 * reset (cudaDeviceReset, or anything else that destroys the device's
 * primary context) makes the kept address stale: do not call this entry
 * point on that device afterwards.  The arguments are checked as
 * rx_attn_decode checks them (RX_ERR_INVALID / RX_ERR_UNSUPPORTED), then
 * RX_ERR_CAPACITY is returned when rx_attn_decode_workspace(...) for the
 * batch exceeds the array. */
#define RX_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
int rx_attn_decode_static(const rx_kv_pool *pool, const void *q, void *o, float *lse,
                          int32_t num_q_heads, const int32_t *req_idx, const int32_t *seq_len,
                          const int32_t *req_to_token, int64_t rtt_stride, int32_t batch,
                          int32_t max_seq_len, const rx_decode_plan *plan_or_null, float sm_scale,
                          int32_t *dev_status, void *stream);

/* ---- attention over FP8 pools --------------------------------------------- */

/* Decode attention over FP8 pools: rx_attn_decode's definition applied to the
 * values E4M3(code) * scale of each pool, with the same arguments (q, o, lse,
 * the plan or NULL, and a workspace of rx_attn_decode_workspace(...) bytes
 * as there) and the same head counts and head dims.  The work goes to the
 * same kernels as over a bf16 pool, each reading code rows (num_kv_heads *
 * head_dim bytes, half a bf16 row's): the per-head kernel and the all-heads
 * kernel for one q head per kv head widen codes exactly (to bf16 tiles, to
 * fp32) and compute as on a bf16 pool holding E4M3(code) -- with both scales
 * 1, bit for bit rx_attn_decode's result on such a pool -- while the
 * all-heads kernel for 8 kv heads with 2 to 16 q heads each runs its products
 * in f16 with fp32 sums: codes widen to f16 exactly, q is converted to f16
 * (exact for |q| within f16's range, which q must respect; values below
 * 2^-14 round to f16 subnormals), and the softmax weights are rounded to f16
 * rather than bf16.  K's scale multiplies the scores, V's the output. */
int rx_attn_decode_fp8(const rx_kv_pool_fp8 *pool, const void *q, void *o, float *lse, int32_t num_q_heads,
                       const int32_t *req_idx, const int32_t *seq_len, const int32_t *req_to_token,
                       int64_t rtt_stride, int32_t batch, int32_t max_seq_len, const rx_decode_plan *plan,
                       void *workspace, size_t ws_bytes, float sm_scale, int32_t *dev_status, void *stream);

/* Extend attention over FP8 pools: rx_attn_extend's definition applied to
 * the values E4M3(code) * scale of each pool, with the same arguments (q, o,
 * lse, qo_indptr, req_idx, prefix_len, extend_len, req_to_token and
 * max_extend_len, and the workspace or NULL, as there).  Both paths read
 * the code rows (num_kv_heads * head_dim bytes each, half a bf16 pool's) and
 * widen them to bf16 -- exactly, since every E4M3 value is a bf16 value --
 * the staged path in its staging copy, the gather path in the attention
 * kernel's producer warps; the attention then runs as on a bf16 pool holding
 * E4M3(code), with K's scale folded into the score scale and V's into the
 * output, and both paths give the same result.  With both scales 1 the result is bit for
 * bit rx_attn_extend's on such a pool.  Pools 8-byte aligned; head_dim 64 or
 * 128 and the head counts rx_attn_extend takes. */
int rx_attn_extend_fp8(const rx_kv_pool_fp8 *pool, const void *q, void *o, float *lse_or_null,
                       int32_t num_q_heads, const int32_t *qo_indptr, const int32_t *req_idx,
                       const int32_t *prefix_len, const int32_t *extend_len, const int32_t *req_to_token,
                       int64_t rtt_stride, int32_t batch, int32_t max_extend_len, void *workspace,
                       size_t ws_bytes, float sm_scale, int32_t *dev_status, void *stream);

/* ---- compressed finite-state machine (constrained decoding) -------------
 * Source: "SGLang: Efficient Execution of Structured Language Model
 * Programs" (unite.ai, es), "Introducción a SGLang", compressed-FSM bullet.
 * Systems that follow an output constraint look only at the next token, so
 * they decode one token per step; the runtime instead builds a compressed
 * finite-state machine of the constraint and decodes a path of several
 * tokens in one step wherever the constraint fixes them.
 *
 * The constraint is a deterministic automaton over token ids (how it is
 * derived from a regular expression and a tokenizer is outside this
 * library): states 0 .. n_states-1, and for state s the edges
 * e in [row_ptr[s], row_ptr[s+1]) with token tok[e] (strictly increasing
 * within a state, < vocab) leading to state nxt[e].  A state without edges
 * is terminal.  A state with exactly one edge fixes the next token.
 *
 * rx_fsm_compress (host): the jump of every state s -- the tokens fixed along
 * the path of single-edge states from s, and the state where it stops (the
 * first state with zero or several edges, a state the path already passed,
 * or after max_jump tokens) -- packed as jump_len [S], jump_off [S] (int64,
 * state order), jump_end [S] and jump_tok [sum of jump_len]; the
 * allowed-token mask: bit t % 32 of word t / 32 of row s is set when state s
 * has an edge with token t, uint32 [S][W] with W = ceil(vocab / 128) * 4
 * (rows padded to 16 bytes with zero words); and its word ranks:
 * rank[s][w] = the number of edges of state s with a token below 32 w,
 * int32 [S][W] (so that the edge of an allowed token t
 * is row_ptr[s] + rank[s][t / 32] + the set bits of its mask word below
 * t % 32, found without a search).  Any output may be
 * NULL; info (required) gets the sizes, so a first call with NULL outputs
 * sizes jump_tok.  RX_ERR_INVALID (nothing written) for arrays that break
 * the rules above; RX_ERR_CAPACITY when out_jump_tok is given and
 * jump_tok_cap < info->jump_tokens. */
typedef struct {
    int64_t n_edges;
    int64_t jump_tokens;   /* tokens over all jumps                        */
    int32_t n_singular;    /* states with exactly one edge                 */
    int32_t n_looped;      /* states whose jump stopped on a repeated state */
    int32_t longest_jump;
} rx_fsm_info;

int rx_fsm_compress(int32_t n_states, int32_t vocab, const int64_t *row_ptr, const int32_t *tok,
                    const int32_t *nxt, int32_t max_jump, uint32_t *out_mask, int32_t *out_rank,
                    int32_t *out_jump_len, int64_t *out_jump_off, int32_t *out_jump_end,
                    int32_t *out_jump_tok, int64_t jump_tok_cap, rx_fsm_info *info);

/* The compressed machine on the device: copies of the automaton's arrays and
 * of rx_fsm_compress's outputs (for the same max_jump), owned by the caller. */
typedef struct {
    const int64_t *row_ptr;
    const int32_t *tok;
    const int32_t *nxt;
    const uint32_t *mask;
    const int32_t *rank;
    const int32_t *jump_len;
    const int64_t *jump_off;
    const int32_t *jump_end;
    const int32_t *jump_tok;
    int32_t n_states, vocab, max_jump;
} rx_fsm;

/* One constrained decoding step for `batch` requests (device, asynchronous
 * on `stream`).  For request b in state s = state[b]:
 *   t  = argmax over the tokens s allows of logits[b][t] (NaN counts as
 *        -inf; equal values go to the smallest id),
 *   s1 = the state edge (s, t) leads to,
 * then out_tokens[b][0] = t, out_tokens[b][1 .. 1+L) = the jump of s1
 * (L = jump_len[s1] <= max_jump), out_count[b] = 1 + L and
 * state[b] = jump_end[s1].  A terminal state sets RX_DEV_FSM_DONE, a state
 * id out of range (or a mask bit without its edge) RX_DEV_BAD_STATE; such a
 * request gets out_count[b] = 0 and keeps its state.
 *   logits: device fp32 rows of logits_stride floats (>= vocab, a multiple
 *   of 4, rows 16-byte aligned); state: device int32 [batch], updated in
 *   place; out_tokens: device int32 [batch][1 + max_jump]; out_count: device
 *   int32 [batch]; workspace: device uint64 [batch + 1], 8-byte aligned,
 *   all zero before the first call -- every call leaves it zero (the
 *   per-request best candidate, and a count of the scan's finished CTAs,
 *   while the call runs).  Rows are read once, as 16-byte vectors.  Up to
 *   512 requests, one kernel on `stream`: the scan, whose last CTA to finish
 *   follows every request's chosen edge; larger batches, the scan and then a
 *   finish kernel as its programmatic dependent. */
int rx_fsm_step(const rx_fsm *fsm, const float *logits, int64_t logits_stride, int32_t batch,
                int32_t *state, int32_t *out_tokens, int32_t *out_count, uint64_t *workspace,
                int32_t *dev_status, void *stream);

/* ---- failure paths, for tests -------------------------------------------
 * Not from the pages.  Two switches that let a test drive the library's
 * error paths without a failing allocator or a stuck GPU.
 *
 * rx_test_fail_alloc: the n-th next radix-tree node allocation (counting
 * from 1, over every tree in the process) fails as a failing host allocator
 * would; the call that needed it returns RX_ERR_NOMEM and leaves the tree
 * and the free list exactly as they were.  n = 0 switches it off;
 * RX_ERR_INVALID for n < 0.
 *
 * rx_decode_set_wait_limit: the bound, in SM clock cycles, on each pipeline
 * wait of the decode kernels launched from then on (process-wide);
 * cycles <= 0 restores the default of 2^31 cycles (about one second).  A
 * wait that runs out ORs RX_DEV_TIMEOUT into the call's status word and
 * stops its CTA: the other warps leave at their next wait, and the copies
 * already in flight are waited for (with the default bound) before the CTA
 * exits, so the context stays usable.  The outputs of that call are then
 * incomplete. */
int rx_test_fail_alloc(int64_t n);
int rx_decode_set_wait_limit(int64_t cycles);

#ifdef __cplusplus
}
#endif

#endif /* RX_H */
