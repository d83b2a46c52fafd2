// rx_internal.h -- declarations shared by the translation units of librx.
#pragma once

#include <stdint.h>

#define RX_ABI_VERSION 3

// Longest position range one decode work item covers (the plan builder and
// the no-plan split both stay at or below it).
#define RX_MAX_KV_CHUNK 4096

// Work items an automatic decode split aims for: about four waves of two
// CTAs on each of 152 SMs.
#define RX_DECODE_TARGET_ITEMS 1216
// automatic plans with single-request ("wide") items: pieces of the private
// positions over the whole batch (two per SM of a 152-SM GPU, handed out
// first come first served) and their shortest length; (kv head, shared
// chunk) items for the per-head kernel, which runs beside the all-heads
// kernel (half an SM wave: each item pays a fixed start-up, so fewer,
// longer ones take less SM time); and, when shared chunks go to the
// all-heads kernel in request groups, the chunk size that gives about one
// wave of (kv head, chunk) pairs.  Measured on few-shot decode: 304 / 152
// beats 608 / 304 by 7 %, and 76 per-head items beat 152 by 6 %.
#define RX_DECODE_TARGET_WIDE_ITEMS 304
// When every shared chunk goes to the all-heads kernel as request groups (no
// per-head kernel beside it), the short group items, handed out last, fill
// the end of the schedule, and fewer, longer private pieces do better:
// measured on the long-chat decode (16 requests of 24,577 private
// positions), 228 / 190 / 152 targets take 0.273 / 0.315 / 0.369 ms against
// 0.281 for 304; tree-of-thought decode keeps its private ranges whole
// either way.
#define RX_DECODE_TARGET_WIDE_ITEMS_GROUPED 228
#define RX_DECODE_MIN_WIDE_CHUNK 16
#define RX_DECODE_TARGET_SHARED_ITEMS 76
#define RX_DECODE_TARGET_GROUP_CHUNKS 152
// With 8 kv heads and G q heads each (G >= 2), the all-heads kernel also
// takes items of up to 16 / G requests that share their positions (16 query
// rows per kv head).  A shared chunk whose requests make at most this many
// such groups goes to it, one item per group (read as whole slot rows; the
// groups of one chunk are claimed together, so all but the first mostly hit
// L2); a chunk shared more widely stays with the per-head kernel.  Measured
// on tree-of-thought decode (1, 4 and 16 groups per segment): limits of 4,
// 8 and 16 give 0.093, 0.093 and 0.088 ms; on the long-chat decode (8
// groups) 8 beats 4 by 1.5 %.
#define RX_DECODE_MAX_GROUPS 16

// Head counts whose single-request decode items have an all-heads kernel
// with several q heads per kv head: 8 kv heads, G = 2, 4, 8 or 16.
static inline bool rx_gqa_heads(int32_t hq, int32_t hkv)
{
    if (hkv != 8 || hq % hkv != 0) return false;
    const int32_t G = hq / hkv;
    return G == 2 || G == 4 || G == 8 || G == 16;
}

// Sets the thread-local message returned by rx_last_error and returns code.
int rx_set_error(int code, const char *fmt, ...);

// The one-layer view of a pool: for a layered pool, k and v advanced to the
// call's layer (num_layers and layer of the result are 0).  RX_ERR_INVALID
// (message naming `who`) for a layer outside the pool.  A null `in` is
// passed through for the caller's own checks.
int rx_pool_layer(const void *in, void *out, int fp8, const char *who);

// Host entry points that allocate wrap their body in RX_TRY ... RX_CATCH so
// that no exception crosses the C ABI.
#ifdef __cplusplus
#include <new>
#define RX_TRY try {
#define RX_CATCH                                                                   \
    }                                                                              \
    catch (const std::bad_alloc &) {                                               \
        return rx_set_error(RX_ERR_NOMEM, "%s: host allocation failed", __func__); \
    }                                                                              \
    catch (...) {                                                                  \
        return rx_set_error(RX_ERR_INVALID, "%s: unexpected exception", __func__); \
    }
#endif

// Positions per decode work item when no plan is given, and the resulting
// number of partial results per request.  Chosen from the batch shape only,
// so rx_attn_decode_workspace and rx_attn_decode agree.
int32_t rx_decode_default_chunk(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len);
