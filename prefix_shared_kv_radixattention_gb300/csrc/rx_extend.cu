// rx_extend.cu -- extend attention on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM).
//
// What is computed: the new tokens of a request attend to its cached prefix
// plus themselves, causally -- the extend pass under RadixAttention, where a
// request that shares a cached prefix reuses that prefix's KV instead of
// recomputing it ("SGLang: Efficient Execution of Structured Language Model
// Programs", unite.ai, es, section "Introducción a SGLang", RadixAttention
// bullet).  For new token i of request b (absolute position p = P_b + i),
// q-head h and kv-head g = h / G:
//     o = softmax_j<=p( sm_scale * q . K[slot_j] ) V[slot_j],
// slot_j = req_to_token[req_idx[b]][j].  Both products are real GEMMs, so
// they run on tcgen05:
//
//   - a CTA owns 256 query rows: 256 / G new tokens of one request times the
//     G q-heads of one kv head (rows token-major), as two 128-row tensor-core
//     tiles that share every K/V tile of 128 keys;
//   - K and V reach shared memory, in the 128-byte-swizzled layout the tensor
//     core reads, by one of two producers: with a workspace, a staging kernel
//     first packs each request's context rows and one thread streams them with
//     tiled TMA loads; without one, three warps gather rows through the slot
//     list with 16-byte cp.async (slot ids prefetched into a small ring).  K
//     and V have rings of their own: a K stage frees as soon as S has read it;
//   - per Q tile t, S_t = Q_t K^T (M = 128, N = 128 keys) lands in 128 TMEM
//     columns; the softmax overwrites them with P_t as bf16 pairs, and O_t +=
//     P_t V (A operand read from TMEM, V MN-major) accumulates in another 128
//     columns -- P never touches shared memory.  S_t(j + 1) may reuse the
//     columns only after O_t += P_t(j) V_j has read them, so the MMA thread
//     staggers the two tiles by half a step (S_0, PV_1, S_1, PV_0, ...): each
//     tile's softmax overlaps the other tile's tensor-core work;
//   - eight softmax warps (four per Q tile, one TMEM lane quadrant and one
//     row per thread) read the row's scores 64 at a time (tcgen05.ld), take
//     the row max (three-input max), then write P = 2^(s - m) back over the
//     scores;
//     the causal test runs only on warps holding a row that crosses its
//     bound, and O is rescaled in TMEM only when the row max grew by more
//     than 2^8.
// Every mbarrier wait is bounded in time: a wait that gives up sets
// RX_DEV_TIMEOUT and raises an abort flag; every role then runs to the common
// exit, where the MMA thread waits for its last tensor-core work and TMEM is
// freed.  Warp-collective TMEM accesses always sit on warp-uniform paths.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <climits>

#include <mutex>
#include <type_traits>

#include "rx_common.cuh"

namespace {

using bf16 = __nv_bfloat16;

constexpr int kQT = 2;              // Q tiles per CTA
constexpr int kRows = 128;          // query rows per Q tile (MMA M)
constexpr int kCtaRows = kQT * kRows;
constexpr int kBN = 128;            // keys per K/V tile (MMA N of S, MMA K of P V)
constexpr int kStages = 2;          // K ring and V ring depth
constexpr int kLag = kStages - 1;   // slot-id prefetch distance (tiles)
constexpr int kNSL = kLag + 1;      // slot-id ring (tiles)
constexpr int kProducer0 = 256;     // producer threads: warps 8-10
constexpr int kProducers = 96;
constexpr int kMmaWarp = 11;
constexpr int kThreads = 32 * 12;   // no register reallocation: every warp keeps the launch count
// staged path (contexts copied into a workspace first): one TMA thread feeds
// the ring, so the CTA is 8 softmax warps + a producer warp + the MMA warp
constexpr int kStagedThreads = 32 * 10;
constexpr int kStagedProducerWarp = 8;
constexpr int kStagedMmaWarp = 9;
constexpr int kStageBlock = 4;     // rows per copy unit of the staging kernel
constexpr uint32_t kTmemCols = 512;  // per Q tile t: S (then P as bf16) [256t, +128), O [256t + 128, +128)
constexpr float kRescale = 8.f;      // log2 units the running max may lag

template <int D>
struct XL {
    static constexpr int NB = D / 64;            // 128-byte column blocks of one row
    static constexpr int QBLK = kRows * 128;     // bytes of one column block of a Q tile
    static constexpr int KBLK = kBN * 128;       // bytes of one column block of a K or V tile
    static constexpr int OFF_Q = 0;              // kQT tiles x NB blocks
    static constexpr int OFF_K = OFF_Q + kQT * NB * QBLK;
    static constexpr int OFF_V = OFF_K + kStages * NB * KBLK;
    static constexpr int OFF_SLOT = OFF_V + kStages * NB * KBLK;  // slot-id ring
    static constexpr int OFF_BAR = OFF_SLOT + kNSL * kBN * 4;
    // per Q tile: q_full; per stage: k_full, v_full, k_empty (S read it),
    // v_empty (O += P V read it); per Q tile: s_full (S in TMEM), p_full
    // (P written over S), pv_done (O += P V finished, S/P columns free)
    static constexpr int B_QFULL = 0, B_KFULL = kQT, B_VFULL = B_KFULL + kStages,
                         B_KEMPTY = B_VFULL + kStages, B_VEMPTY = B_KEMPTY + kStages,
                         B_SFULL = B_VEMPTY + kStages, B_PFULL = B_SFULL + kQT,
                         B_PVDONE = B_PFULL + kQT, B_FINAL = B_PVDONE + kQT, N_BAR = B_FINAL + 1;
    static constexpr int OFF_TMEM = OFF_BAR + N_BAR * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 8;
    static constexpr int BYTES = OFF_ABORT + 8 + 1024;  // + room to align the base to 1024
};
static_assert(XL<128>::BYTES <= 227 * 1024, "shared memory budget");
static_assert(XL<128>::OFF_BAR % 8 == 0 && XL<64>::OFF_BAR % 8 == 0, "mbarrier alignment");

struct XParams {  // 64-byte aligned through its tensor maps
    // staged path: the packed context rows as [row][kv head][head_dim], box
    // 64 x 1 x 64 (128-byte rows, 128-byte swizzle)
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    const int64_t *stage_offs;  // first packed row of request b; [batch] = rows used
    const int32_t *stage_src;   // request whose packed rows hold b's leading shared tiles
    const int32_t *stage_share; // leading prefix tiles of b read from stage_src[b]'s rows
    int64_t stage_cap;          // rows the workspace holds
    const bf16 *q;
    bf16 *o;
    float *lse;
    const bf16 *k_pool;
    const bf16 *v_pool;
    const unsigned char *k8;   // FP8 pools (gather path): E4M3 codes, else null
    const unsigned char *v8;
    int64_t num_slots;
    int hq, hkv, G;
    const int32_t *qo_indptr;
    const int32_t *req_idx;
    const int32_t *prefix_len;
    const int32_t *extend_len;
    const int32_t *rtt;
    int64_t rtt_stride;
    float scale_log2;       // sm_scale log2(e), times K's scale for an FP8 pool
    float v_scale;          // V's scale for an FP8 pool (multiplies o); 1 otherwise
    int32_t *status;
};

struct Tile {
    int M;             // valid query rows (<= 256)
    int nqt;           // Q tiles with valid rows (1 or 2)
    int64_t qbase;     // packed token index of row group 0
    int row0_pos;      // absolute position of row group 0
    int kv_end;        // keys [0, kv_end)
    int ntiles;
    int stage_row0;    // staged path: first packed row of this request's own tiles
    int share_tiles;   // staged path: leading tiles read from another request's rows
    int share_row0;    // ... which start at this packed row
    const int32_t *slots;
    int g;
};

// Bounded wait of one thread; false when it gave up (or another role did).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status)
{
    if (rx::mbar_test_wait(bar, parity)) return true;  // already flipped: no suspend
    const long long t0 = clock64();
    do {
        if (rx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    } while (clock64() - t0 < rx::kWaitCycles);
    *abort_flag = 1;
    if (status) atomicOr(status, RX_DEV_TIMEOUT);
    return false;
}
// The same for a whole warp, with one answer for all its lanes (the warp-wide
// tcgen05.ld / st that follow need every lane).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status)
{
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag, status));
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major
// tile whose 128-byte column blocks are blk bytes apart
__device__ __forceinline__ uint32_t sw128(int r, int c, int blk)
{
    return (uint32_t)((c >> 3) * blk + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// Bounded wait that ignores the abort flag: used only to let copies already
// issued finish landing before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t *status)
{
    const long long t0 = clock64();
    do {
        if (rx::mbar_try_wait(bar, parity)) return;
    } while (clock64() - t0 < rx::kWaitCycles);
    if (status) atomicOr(status, RX_DEV_TIMEOUT);
}

// Eight E4M3 codes (element 0 in the low byte) as eight bf16: every E4M3
// value, subnormals included, is exact in f16 and in bf16, so the widening
// through f16 is exact.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 c)
{
    const uint32_t w[2] = {c.x, c.y};
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t h = rx::e4m3x2_to_f16x2((uint16_t)(w[k >> 1] >> (16 * (k & 1))));
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
        r[k] = rx::pack_bf16(f.x, f.y);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// ---------------------------------------------------------------------------
// producer warps: K and V tiles through the slot list
// ---------------------------------------------------------------------------

// F8: the pools hold E4M3 codes (p.k8, p.v8), widened here to the bf16 tiles.
template <int D, bool F8>
__device__ void producer(const XParams &p, const Tile &T, unsigned char *smem, uint32_t sbase)
{
    using L = XL<D>;
    constexpr int CPR = D / 8;            // 16-byte chunks per row
    const uint32_t bar = sbase + L::OFF_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    const int32_t *sbuf = reinterpret_cast<const int32_t *>(smem + L::OFF_SLOT);
    const int pt = threadIdx.x - kProducer0;

    // slot ids of tile j -> slot ring entry j % kNSL (4-byte async copies)
    auto fetch_slots = [&](int j) {
        if (j >= T.ntiles) return;
        for (int r = pt; r < kBN; r += kProducers) {
            const int pos = j * kBN + r;
            rx::cp_async_4(sbase + L::OFF_SLOT + ((j % kNSL) * kBN + r) * 4,
                           T.slots + (pos < T.kv_end ? pos : 0), pos < T.kv_end ? 4 : 0);
        }
    };
    for (int j = 0; j < kLag; ++j) fetch_slots(j);
    rx::cp_async_commit();

    // one cp.async group per tile j: its K and V rows and the slot ids of
    // tile j + kLag.  K and V have their own stage barriers (a K stage frees
    // as soon as S has read it, a V stage only after O += P V); each gets a
    // producer thread's arrival as soon as that thread's copies have landed
    // (cp.async.mbarrier.arrive), so handing a tile over never waits for the
    // producer loop; the MMA thread fences the landed rows into the async
    // proxy before reading them.
    for (int j = 0; j < T.ntiles; ++j) {
        const int st = j % kStages;
        if (j < kLag)
            rx::cp_async_wait<0>();                 // the first slot ids
        else
            rx::cp_async_wait<kLag - 1>();          // group of tile j - kLag: slot ids of tile j
        rx::named_bar_sync(1, kProducers);          // every producer sees the slot ids
        const int32_t *sl = sbuf + (j % kNSL) * kBN;
        // one pass per matrix: K (w = 0) into its stage, then V (w = 1)
        bool stop = false;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            if (j >= kStages) {
                const bool ok = wait_or_abort(bar + 8 * ((w ? L::B_VEMPTY : L::B_KEMPTY) + st),
                                              ((j / kStages) - 1) & 1, abort_flag, p.status);
                if (rx::named_bar_or(1, kProducers, !ok)) {  // every producer leaves together
                    stop = true;
                    break;
                }
            }
            const uint32_t dst = sbase + (w ? L::OFF_V : L::OFF_K) + st * L::NB * L::KBLK;
            if constexpr (F8) {
                // FP8 pools: 16 codes a chunk, loaded (two 8-byte loads,
                // four chunks in flight), widened exactly to bf16 and stored
                // as the tile's two 16-byte chunks; then this thread's arrival
                constexpr int CPR8 = D / 16;
                const unsigned char *pool8 = w ? p.v8 : p.k8;
                unsigned char *tile = smem + (dst - sbase);
                for (int i0 = pt; i0 < kBN * CPR8; i0 += 4 * kProducers) {
                    uint2 lo[4], hi[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int idx = i0 + u * kProducers;
                        lo[u] = hi[u] = make_uint2(0u, 0u);
                        if (idx < kBN * CPR8) {
                            const int r = idx / CPR8, c = idx % CPR8;
                            const int pos = j * kBN + r;
                            const int32_t s = sl[r];
                            const bool inside = pos < T.kv_end;
                            const bool ok = inside && s >= 0 && (int64_t)s < p.num_slots;
                            if (w == 0 && inside && !ok && c == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_SLOT);
                            if (ok) {
                                const uint2 *src = reinterpret_cast<const uint2 *>(
                                    pool8 + ((int64_t)s * p.hkv + T.g) * D + c * 16);
                                lo[u] = __ldg(src);
                                hi[u] = __ldg(src + 1);
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int idx = i0 + u * kProducers;
                        if (idx < kBN * CPR8) {
                            const int r = idx / CPR8, c = idx % CPR8;
                            *reinterpret_cast<uint4 *>(tile + sw128(r, 2 * c, L::KBLK)) =
                                e4m3x8_to_bf16x8(lo[u]);
                            *reinterpret_cast<uint4 *>(tile + sw128(r, 2 * c + 1, L::KBLK)) =
                                e4m3x8_to_bf16x8(hi[u]);
                        }
                    }
                }
                rx::mbar_arrive(bar + 8 * ((w ? L::B_VFULL : L::B_KFULL) + st));
            } else {
                const bf16 *pool = w ? p.v_pool : p.k_pool;
                for (int idx = pt; idx < kBN * CPR; idx += kProducers) {
                    const int r = idx / CPR, c = idx % CPR;
                    const int pos = j * kBN + r;
                    const int32_t s = sl[r];
                    const bool inside = pos < T.kv_end;
                    const bool ok = inside && s >= 0 && (int64_t)s < p.num_slots;
                    if (w == 0 && inside && !ok && c == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_SLOT);
                    const int64_t off = ok ? (((int64_t)s * p.hkv + T.g) * D + c * 8) : 0;
                    rx::cp_async_16(dst + sw128(r, c, L::KBLK), pool + off, ok ? 16 : 0);
                }
                rx::cp_async_mbar_arrive(bar + 8 * ((w ? L::B_VFULL : L::B_KFULL) + st));
            }
        }
        if (stop) break;
        rx::named_bar_sync(1, kProducers);          // slot entry j % kNSL is read: refill allowed
        fetch_slots(j + kLag);
        rx::cp_async_commit();
    }
    rx::cp_async_wait<0>();
}

// Staged path: one thread streams tile j of the request's packed context with
// four (D = 128) or two (D = 64) TMA box loads -- K and V, one box per
// 128-byte column block, each box kBN rows of one kv head.  Every packed
// region is a whole number of kBN-row tiles with zeroed padding, so the boxes
// never leave the request's region.
template <int D>
__device__ void tma_producer(const XParams &p, const Tile &T, unsigned char *smem, uint32_t sbase)
{
    using L = XL<D>;
    const uint32_t bar = sbase + L::OFF_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    int issued[2] = {0, 0};  // tiles of K, of V
    for (int j = 0; j < T.ntiles; ++j) {
        const int st = j % kStages;
        // leading tiles shared with an earlier request come from its rows
        const int row = j < T.share_tiles ? T.share_row0 + j * kBN : T.stage_row0 + (j - T.share_tiles) * kBN;
        bool stop = false;
#pragma unroll
        for (int w = 0; w < 2; ++w) {  // K into its stage once S freed it, then V
            if (j >= kStages && !wait_or_abort(bar + 8 * ((w ? L::B_VEMPTY : L::B_KEMPTY) + st),
                                               ((j / kStages) - 1) & 1, abort_flag, p.status)) {
                stop = true;
                break;
            }
            const uint32_t full = bar + 8 * ((w ? L::B_VFULL : L::B_KFULL) + st);
            rx::mbar_arrive_expect_tx(full, kBN * D * 2);
            const uint32_t dst = sbase + (w ? L::OFF_V : L::OFF_K) + st * L::NB * L::KBLK;
#pragma unroll
            for (int cb = 0; cb < L::NB; ++cb)
                rx::tma_load_3d(dst + cb * L::KBLK, w ? &p.tm_v : &p.tm_k, cb * 64, T.g, row, full);
            issued[w] = j + 1;
        }
        if (stop) break;
    }
    // no copy may still be landing when the CTA exits (normally every stage
    // was consumed already; after an abort the last ones may not have been)
    for (int w = 0; w < 2; ++w)
        for (int jj = issued[w] > kStages ? issued[w] - kStages : 0; jj < issued[w]; ++jj)
            drain_wait(bar + 8 * ((w ? L::B_VFULL : L::B_KFULL) + jj % kStages), (jj / kStages) & 1, p.status);
}

// ---------------------------------------------------------------------------
// MMA thread
// ---------------------------------------------------------------------------

template <int D, bool kStaged>
__device__ void mma_issuer(const XParams &p, const Tile &T, unsigned char *smem, uint32_t sbase,
                           uint32_t tmem)
{
    using L = XL<D>;
    const uint32_t bar = sbase + L::OFF_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    constexpr uint32_t idesc_qk = rx::idesc_bf16(kRows, kBN, false, false);
    constexpr uint32_t idesc_pv = rx::idesc_bf16(kRows, D, false, true);
    auto wait = [&](int b, uint32_t parity) { return wait_or_abort(bar + 8 * b, parity, abort_flag, p.status); };
    // shared-memory descriptors built once: every operand block is the
    // region base plus a byte offset, i.e. the descriptor plus offset / 16
    const uint64_t dq = rx::sdesc_sw128(sbase + L::OFF_Q, 16, 1024);
    const uint64_t dk = rx::sdesc_sw128(sbase + L::OFF_K, 16, 1024);
    const uint64_t dv = rx::sdesc_sw128(sbase + L::OFF_V, L::KBLK, 1024);

    // Per Q tile t the work is a chain: S_t(j) = Q_t K_j^T into its TMEM
    // columns, the softmax overwrites them with P_t(j) (bf16), O_t +=
    // P_t(j) V_j reads P from TMEM, and only then may S_t(j + 1) reuse the
    // columns.  The two tiles are staggered by half a step, so each tile's
    // softmax overlaps tensor-core work of the other tile and the two
    // softmaxes do not contend for the exp unit:
    //   S_0(0) | P V_1(j - 1), S_1(j), P V_0(j), S_0(j + 1) | ... | P V_1(n - 1)
    auto issue_s = [&](int t, int j) -> bool {
        const int st = j % kStages;
        if (!wait(L::B_KFULL + st, (j / kStages) & 1)) return false;
        if (j == 0 ? !wait(L::B_QFULL + t, 0) : !wait(L::B_PVDONE + t, (j - 1) & 1)) return false;
        if (!kStaged) rx::fence_proxy_async_smem();  // K rows landed by cp.async -> async proxy
        rx::tc_fence_after();
        const uint64_t dks = dk + (uint64_t)((st * L::NB * L::KBLK) >> 4);
        const uint64_t dqt = dq + (uint64_t)((t * L::NB * L::QBLK) >> 4);
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb)
            rx::tc_mma(tmem + t * 256, dqt + (uint64_t)(((kb >> 2) * L::QBLK + (kb & 3) * 32) >> 4),
                       dks + (uint64_t)(((kb >> 2) * L::KBLK + (kb & 3) * 32) >> 4), idesc_qk, kb > 0);
        rx::tc_commit(bar + 8 * (L::B_SFULL + t));
        // the last tile to read K_j releases its stage
        if (t == T.nqt - 1) rx::tc_commit(bar + 8 * (L::B_KEMPTY + st));
        return true;
    };
    auto issue_pv = [&](int t, int j) -> bool {
        const int st = j % kStages;
        if (!wait(L::B_PFULL + t, j & 1)) return false;
        if (!wait(L::B_VFULL + st, (j / kStages) & 1)) return false;
        if (!kStaged) rx::fence_proxy_async_smem();  // V rows landed by cp.async
        rx::tc_fence_after();
        const uint64_t dvs = dv + (uint64_t)((st * L::NB * L::KBLK) >> 4);
        // A = P_t(j) in TMEM: 16 keys per MMA = 8 columns of bf16 pairs
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
            rx::tc_mma_ts(tmem + t * 256 + 128, tmem + t * 256 + ks * 8, dvs + (uint64_t)((ks * 16 * 128) >> 4),
                          idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        rx::tc_commit(bar + 8 * (L::B_PVDONE + t));
        if (t == T.nqt - 1) rx::tc_commit(bar + 8 * (L::B_VEMPTY + st));
        return true;
    };
    const bool two = T.nqt == 2;
    bool ok = issue_s(0, 0);
    for (int j = 0; j < T.ntiles && ok; ++j) {
        if (two) {
            if (j > 0 && !(ok = issue_pv(1, j - 1))) break;
            if (!(ok = issue_s(1, j))) break;
        }
        if (!(ok = issue_pv(0, j))) break;
        if (j + 1 < T.ntiles && !(ok = issue_s(0, j + 1))) break;
    }
    if (ok && two) issue_pv(1, T.ntiles - 1);
    // everything issued has finished before TMEM is released
    rx::tc_commit(bar + 8 * L::B_FINAL);
    drain_wait(bar + 8 * L::B_FINAL, 0, p.status);
}

// ---------------------------------------------------------------------------
// softmax warps: one query row per thread
// ---------------------------------------------------------------------------

template <int D>
__device__ void softmax_rows(const XParams &p, const Tile &T, unsigned char *smem, uint32_t sbase,
                             uint32_t tmem)
{
    using L = XL<D>;
    const int warp = threadIdx.x >> 5;
    const int t = warp >> 2;                      // Q tile
    if (t >= T.nqt) return;
    const uint32_t bar = sbase + L::OFF_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    const int rl = threadIdx.x & (kRows - 1);     // row in the Q tile = TMEM lane
    const int row = t * kRows + rl;
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tbase = tmem + t * 256 + lanes;
    const uint32_t tO = tbase + 128;
    const int row_lim = T.row0_pos + row / p.G;   // keys at positions <= row_lim are visible
    const float sl2 = p.scale_log2;
    {
        // this tile's Q rows (CTA row r: token r / G, q head g G + r % G) with
        // coalesced 16-byte copies by the tile's four warps, zeros past the
        // last row; fenced into the async proxy before the tensor core reads
        constexpr int CPR = D / 8;
        const int G = p.G;
        const uint32_t qd = sbase + L::OFF_Q + t * L::NB * L::QBLK;
        for (int idx = rl; idx < kRows * CPR; idx += kRows) {
            const int r = idx / CPR, c = idx % CPR;
            const int qr = t * kRows + r;
            const bool ok = qr < T.M;
            const bf16 *src = ok ? p.q + ((T.qbase + qr / G) * p.hq + (int64_t)T.g * G + qr % G) * D + c * 8 : p.q;
            rx::cp_async_16(qd + sw128(r, c, L::QBLK), src, ok ? 16 : 0);
        }
        rx::cp_async_commit();
        rx::cp_async_wait<0>();
        rx::fence_proxy_async_smem();
        rx::mbar_arrive(bar + 8 * (L::B_QFULL + t));
    }
    float m_used = -INFINITY, l = 0.f;
    const uint32_t tS = tbase;  // S_t(j), then P_t(j) over its first kBN / 2 columns
    for (int j = 0; j < T.ntiles; ++j) {
        if (!warp_wait(bar + 8 * (L::B_SFULL + t), j & 1, abort_flag, p.status)) return;
        rx::tc_fence_after();
        const int kbase = j * kBN;
        // one answer per warp: the masked and unmasked passes below hold
        // different warp-collective tcgen05.ld instructions, so all lanes of
        // a warp must take the same one (the masked pass is exact for every row)
        const bool need_mask = __any_sync(0xffffffffu, kbase + kBN - 1 > row_lim);
        // the tile's kBN scores of this row, loaded once (four loads in
        // flight) and kept in registers for the max and the exponentials;
        // the causal test only on tiles that cross the row's bound
        uint32_t sv[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
            rx::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
        rx::tmem_wait_ld();
        if (need_mask) {
#pragma unroll
            for (int k = 0; k < kBN; ++k)
                if (kbase + k > row_lim) sv[k] = __float_as_uint(-INFINITY);
        }
        // the row max: four running three-input maxima (few live registers
        // next to the kBN scores)
        float mx;
        {
            float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
            for (int k = 0; k < kBN / 8; ++k) {
                a0 = rx::fmax3(a0, u2f(sv[8 * k]), u2f(sv[8 * k + 1]));
                a1 = rx::fmax3(a1, u2f(sv[8 * k + 2]), u2f(sv[8 * k + 3]));
                a2 = rx::fmax3(a2, u2f(sv[8 * k + 4]), u2f(sv[8 * k + 5]));
                a3 = rx::fmax3(a3, u2f(sv[8 * k + 6]), u2f(sv[8 * k + 7]));
            }
            mx = rx::fmax3(fmaxf(a0, a1), a2, a3);
        }
        const float m_new = fmaxf(m_used, mx * sl2);
        const bool need = (m_used == -INFINITY) || (m_new > m_used + kRescale);
        const float alpha = (need && m_used != -INFINITY) ? rx::fast_exp2(m_used - m_new) : 1.f;
        if (need) {
            l *= alpha;
            m_used = m_new;
        }
        // pass 2: P = 2^(s sl2 - m) as bf16 pairs written back over the S
        // columns already read (64 scores -> 32 columns at a time), the row
        // sum in four packed accumulators.  (Measured: moving a share of the
        // exponentials to a polynomial on the FMA pipe is slower here, since
        // the softmax is bound by issue and the ALU pipe, not the exp unit.)
        const float mu = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t scale2 = rx::f2(sl2, sl2), negm2 = rx::f2(-mu, -mu);
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c2 = 0; c2 < kBN / 64; ++c2) {
            uint32_t pk[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                float x0, x1;
                rx::f2_split(rx::f2_fma(rx::f2(u2f(sv[c2 * 64 + 2 * k]), u2f(sv[c2 * 64 + 2 * k + 1])), scale2, negm2),
                             x0, x1);
                const float e0 = rx::fast_exp2(x0), e1 = rx::fast_exp2(x1);  // -inf -> 0
                acc[k & 3] = rx::f2_add(acc[k & 3], rx::f2(e0, e1));
                pk[k] = rx::pack_bf16(e0, e1);
            }
            // P over the first kBN / 2 columns: every score is in registers
            rx::tmem_st32(tS + c2 * 32, pk);
        }
        if (j > 0 && __any_sync(0xffffffffu, need)) {
            // rescale the O rows in TMEM (after the exponentials, when the
            // scores no longer hold registers): O += P V of tile j - 1
            // finished before S_t(j) was issued, and the next one waits for
            // p_full
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t r[32];
                rx::tmem_ld32(tO + c4 * 32, r);
                rx::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(u2f(r[k]) * alpha);
                rx::tmem_st32(tO + c4 * 32, r);
            }
            rx::tmem_wait_st();
        }
        rx::tmem_wait_st();
        {
            float a0, a1;
            rx::f2_split(rx::f2_add(rx::f2_add(acc[0], acc[1]), rx::f2_add(acc[2], acc[3])), a0, a1);
            l += a0 + a1;
        }
        rx::tc_fence_before();
        rx::mbar_arrive(bar + 8 * (L::B_PFULL + t));
    }
    const int jl = T.ntiles - 1;
    if (!warp_wait(bar + 8 * (L::B_PVDONE + t), jl & 1, abort_flag, p.status)) return;
    rx::tc_fence_after();
    const bool valid = row < T.M;
    const int G = p.G;
    const int64_t orow = (T.qbase + row / G) * p.hq + (int64_t)T.g * G + row % G;
    const float inv = p.v_scale / l;
#pragma unroll
    for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t r[32];
        rx::tmem_ld32(tO + c4 * 32, r);
        rx::tmem_wait_ld();
        if (valid) {
            bf16 *dst = p.o + orow * D + c4 * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 v;
                v.x = rx::pack_bf16(u2f(r[8 * q + 0]) * inv, u2f(r[8 * q + 1]) * inv);
                v.y = rx::pack_bf16(u2f(r[8 * q + 2]) * inv, u2f(r[8 * q + 3]) * inv);
                v.z = rx::pack_bf16(u2f(r[8 * q + 4]) * inv, u2f(r[8 * q + 5]) * inv);
                v.w = rx::pack_bf16(u2f(r[8 * q + 6]) * inv, u2f(r[8 * q + 7]) * inv);
                *reinterpret_cast<uint4 *>(dst + 8 * q) = v;
            }
        }
    }
    if (valid && p.lse) p.lse[orow] = (m_used + log2f(l)) * rx::kLn2;
}

template <int D, bool kStaged, bool F8 = false>
__global__ void __launch_bounds__(kStaged ? kStagedThreads : kThreads, 1)
    extend_kernel(const __grid_constant__ XParams p)
{
    using L = XL<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = rx::smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned swizzle atoms
    const uint32_t sbase = rx::smem_u32(smem);

    // staged: launched as a programmatic dependent of the copy; every CTA
    // waits for the staging kernels (so this grid completes after them)
    // before anything else
    if (kStaged) rx::pdl_wait();

    // which rows: 256 / G tokens of request b times the G q-heads of kv head g
    Tile T;
    const int b = blockIdx.z;
    T.g = blockIdx.y;
    const int tb = kCtaRows / p.G;
    const int E = __ldg(p.extend_len + b);
    if (E > (int)gridDim.x * tb) {  // past max_extend_len
        if (p.status && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            atomicOr(p.status, RX_DEV_BAD_LEN);
        return;
    }
    const int t0 = ((int)gridDim.x - 1 - (int)blockIdx.x) * tb;  // longest rows first
    if (t0 >= E) return;
    const int ntok = min(tb, E - t0);
    const int64_t P = __ldg(p.prefix_len + b);
    if (P < 0 || P + E > p.rtt_stride) {
        if (p.status && threadIdx.x == 0) atomicOr(p.status, RX_DEV_BAD_LEN);
        return;
    }
    if (kStaged) {
        // contexts larger than the workspace: nothing was staged (flagged there)
        if (p.stage_offs[gridDim.z] > p.stage_cap) return;
        T.stage_row0 = (int)p.stage_offs[b];
        T.share_tiles = p.stage_share[b];
        T.share_row0 = (int)p.stage_offs[p.stage_src[b]];
    }
    T.M = ntok * p.G;
    T.nqt = T.M > kRows ? 2 : 1;
    T.qbase = (int64_t)__ldg(p.qo_indptr + b) + t0;
    T.row0_pos = (int)(P + t0);
    T.kv_end = (int)(P + t0 + ntok);
    T.ntiles = (T.kv_end + kBN - 1) / kBN;
    T.slots = p.rtt + (int64_t)__ldg(p.req_idx + b) * p.rtt_stride;

    const uint32_t bar = sbase + L::OFF_BAR;
    const int warp = threadIdx.x >> 5;
    constexpr int mma_warp = kStaged ? kStagedMmaWarp : kMmaWarp;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kQT; ++i) rx::mbar_init(bar + 8 * (L::B_QFULL + i), 128);  // softmax threads
        for (int i = 0; i < kStages; ++i) {
            // gather path: every producer thread's copies; staged: the TMA thread's
            // arrival plus the boxes' bytes
            rx::mbar_init(bar + 8 * (L::B_KFULL + i), kStaged ? 1 : kProducers);
            rx::mbar_init(bar + 8 * (L::B_VFULL + i), kStaged ? 1 : kProducers);
            rx::mbar_init(bar + 8 * (L::B_KEMPTY + i), 1);  // MMA commits
            rx::mbar_init(bar + 8 * (L::B_VEMPTY + i), 1);
        }
        for (int i = 0; i < kQT; ++i) {
            rx::mbar_init(bar + 8 * (L::B_SFULL + i), 1);     // MMA commit
            rx::mbar_init(bar + 8 * (L::B_PFULL + i), 128);   // the tile's softmax threads
            rx::mbar_init(bar + 8 * (L::B_PVDONE + i), 1);    // MMA commit
        }
        rx::mbar_init(bar + 8 * L::B_FINAL, 1);
        *reinterpret_cast<volatile int *>(smem + L::OFF_ABORT) = 0;
        rx::fence_mbar_init();
    }
    if (warp == mma_warp) rx::tmem_alloc(sbase + L::OFF_TMEM, kTmemCols);
    rx::tc_fence_before();
    __syncthreads();
    rx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::OFF_TMEM);

    if (warp < 8) {
        softmax_rows<D>(p, T, smem, sbase, tmem);
    } else {
        if (warp < mma_warp) {
            if (!kStaged) {
                producer<D, F8>(p, T, smem, sbase);
            } else if (warp == kStagedProducerWarp) {
                if ((threadIdx.x & 31) == 0) tma_producer<D>(p, T, smem, sbase);
                __syncwarp();
            }
        } else {
            if ((threadIdx.x & 31) == 0) mma_issuer<D, kStaged>(p, T, smem, sbase, tmem);
            __syncwarp();  // the whole warp reaches the exit barrier together
        }
    }

    rx::tc_fence_before();
    __syncthreads();
    if (warp == mma_warp) {
        rx::tc_fence_after();
        rx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// staging: the contexts copied out of the pool, packed per request
// ---------------------------------------------------------------------------

// Packed rows of request b: its context (prefix + extend tokens) rounded up
// to whole kBN-row tiles; none for lengths the attention kernel rejects.
__device__ __forceinline__ int64_t staged_rows(const int32_t *prefix_len, const int32_t *extend_len, int b,
                                               int64_t rtt_stride)
{
    const int64_t P = __ldg(prefix_len + b), E = __ldg(extend_len + b);
    if (P < 0 || E < 0 || P + E > rtt_stride) return 0;
    return (P + E + kBN - 1) / kBN * kBN;
}

// Requests of one batch that share a cached prefix (their slot lists agree
// on it) need its rows staged once.  For request b: src[b] = the first
// request r < b whose slot list agrees with b's on position 0, both
// prefixes covering the first kBN-row tile, and share[b] = the leading
// tiles, inside both prefixes, on which b and r agree (0 when even the first
// differs: then src[b] = b).  Such an r stages every tile of its own (an
// earlier request agreeing with it on position 0 would be b's candidate
// instead), so b stages only tiles share[b] .. and reads the others from r's
// rows.  One CTA per request, in a few rounds of loads issued together:
// the first slot id of every earlier request (a thread per candidate), then
// every position of the shared tiles (a thread per position of a tile).
__global__ void __launch_bounds__(kBN) stage_share_kernel(const int32_t *__restrict__ rtt, int64_t rtt_stride,
                                                         const int32_t *__restrict__ req_idx,
                                                         const int32_t *__restrict__ prefix_len,
                                                         const int32_t *__restrict__ extend_len, int32_t *src,
                                                         int32_t *share)
{
    __shared__ int first, diff;
    const int b = blockIdx.x, t = threadIdx.x;
    rx::pdl_launch_dependents();  // the offsets kernel may launch and wait on the device
    auto covers = [&](int i) {
        const int64_t P = __ldg(prefix_len + i), E = __ldg(extend_len + i);
        return P >= kBN && E >= 0 && P + E <= rtt_stride;
    };
    if (t == 0) {
        first = b;
        diff = INT_MAX;
    }
    __syncthreads();
    const bool b_ok = covers(b);
    const int32_t *rb = rtt + (int64_t)__ldg(req_idx + b) * rtt_stride;
    if (b_ok) {
        const int32_t s0 = __ldg(rb);
        for (int r = t; r < b; r += kBN)
            if (covers(r) && __ldg(rtt + (int64_t)__ldg(req_idx + r) * rtt_stride) == s0) {
                atomicMin(&first, r);
                break;
            }
    }
    __syncthreads();
    const int r = first;
    int tiles = 0;
    if (r != b) {
        const int32_t *rr = rtt + (int64_t)__ldg(req_idx + r) * rtt_stride;
        const int ntile = (int)(min(__ldg(prefix_len + b), __ldg(prefix_len + r)) / kBN);
        int local = ntile;
#pragma unroll 8
        for (int j = 0; j < ntile; ++j)
            if (__ldg(rr + (int64_t)j * kBN + t) != __ldg(rb + (int64_t)j * kBN + t)) local = min(local, j);
        if (local < ntile) atomicMin(&diff, local);
        __syncthreads();
        tiles = min(ntile, diff);
    }
    if (t == 0) {
        src[b] = tiles > 0 ? r : b;
        share[b] = tiles;
    }
}

// offs[b] = first packed row of request b's own tiles (exclusive prefix sum
// of the packed row counts: its context rounded up to whole kBN-row tiles,
// less the tiles it shares), offs[batch] = rows used; more than `cap` rows
// is flagged, and then neither the copy nor the attention kernel does
// anything.
__global__ void __launch_bounds__(1024) ctx_offsets_kernel(const int32_t *prefix_len, const int32_t *extend_len,
                                                           const int32_t *share, int batch, int64_t rtt_stride,
                                                           int64_t cap, int64_t *offs, int32_t *status)
{
    __shared__ int64_t warp_tot[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    rx::pdl_launch_dependents();
    rx::pdl_wait();  // the share counts are written by the kernel before this one
    const int per = (batch + 1023) / 1024;
    const int b0 = threadIdx.x * per;
    int64_t local = 0;
    for (int i = 0; i < per && b0 + i < batch; ++i)
        local += staged_rows(prefix_len, extend_len, b0 + i, rtt_stride) - (int64_t)share[b0 + i] * kBN;
    // inclusive scan over the block: within each warp, then over warp totals
    int64_t x = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = warp_tot[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int64_t run = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);  // exclusive
    for (int i = 0; i < per && b0 + i < batch; ++i) {
        offs[b0 + i] = run;
        run += staged_rows(prefix_len, extend_len, b0 + i, rtt_stride) - (int64_t)share[b0 + i] * kBN;
    }
    if (threadIdx.x == 1023) {
        const int64_t total = warp_tot[31];
        offs[batch] = total;
        if (total > cap && status) atomicOr(status, RX_DEV_BAD_LEN);
    }
}

// Packed row offs[b] + i = pool row req_to_token[req_idx[b]][share[b] kBN + i]
// for K and V (all kv heads: one contiguous row of the pool each), zeros from
// the end of the context to the kBN-row boundary and for slot ids outside the
// pool (flagged).  One warp per block of kStageBlock rows; every request's
// region is a multiple of kBN rows, so a block never straddles two requests.
// F8: the pools hold E4M3 codes (a byte a value), widened to bf16 on the way
// (their scales are applied by the attention kernel).
template <bool F8>
__global__ void __launch_bounds__(256) stage_rows_kernel(
    const void *__restrict__ k_pool, const void *__restrict__ v_pool, int64_t num_slots,
    const int32_t *__restrict__ rtt, int64_t rtt_stride, const int32_t *__restrict__ req_idx,
    const int32_t *__restrict__ prefix_len, const int32_t *__restrict__ extend_len,
    const int32_t *__restrict__ share, int batch, const int64_t *__restrict__ offs, int64_t cap,
    bf16 *__restrict__ ks, bf16 *__restrict__ vs, int row_elems, int32_t *status)
{
    rx::pdl_launch_dependents();
    rx::pdl_wait();  // the packed-row offsets are written by the kernel before this one
    const int64_t total = offs[batch];
    if (total > cap) return;
    const int lane = threadIdx.x & 31;
    const int row_vecs = row_elems / 8;
    const int64_t nblk = total / kStageBlock;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; blk < nblk; blk += nwarps) {
        const int64_t row0 = blk * kStageBlock;
        int lo = 0, hi = batch - 1;  // last request whose region starts at or before row0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (offs[mid] <= row0) lo = mid; else hi = mid - 1;
        }
        // a request that shares all its tiles has an empty region: the
        // search above lands on the last request starting at row0, which
        // owns it
        const int b = lo;
        const int64_t ctx = (int64_t)__ldg(prefix_len + b) + __ldg(extend_len + b);
        const int64_t pos0 = row0 - offs[b] + (int64_t)share[b] * kBN;
        int32_t my_slot = -1;
        if (lane < kStageBlock && pos0 + lane < ctx) {
            const int32_t sl = __ldg(rtt + (int64_t)__ldg(req_idx + b) * rtt_stride + pos0 + lane);
            if (sl >= 0 && (int64_t)sl < num_slots) my_slot = sl;
            else if (status) atomicOr(status, RX_DEV_BAD_SLOT);
        }
#pragma unroll 4
        for (int r = 0; r < kStageBlock; ++r) {
            const int32_t sl = __shfl_sync(0xffffffffu, my_slot, r);
            // source row: row_elems values of 2 bytes (bf16) or 1 (codes)
            const int64_t src_off = (int64_t)(sl < 0 ? 0 : sl) * row_elems * (F8 ? 1 : 2);
            const unsigned char *ksrc = static_cast<const unsigned char *>(k_pool) + src_off;
            const unsigned char *vsrc = static_cast<const unsigned char *>(v_pool) + src_off;
            uint4 *kdst = reinterpret_cast<uint4 *>(ks + (row0 + r) * row_elems);
            uint4 *vdst = reinterpret_cast<uint4 *>(vs + (row0 + r) * row_elems);
            for (int v = lane; v < row_vecs; v += 32) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                uint4 kv = z, vv = z;
                if (sl >= 0) {
                    if constexpr (F8) {
                        kv = e4m3x8_to_bf16x8(__ldg(reinterpret_cast<const uint2 *>(ksrc) + v));
                        vv = e4m3x8_to_bf16x8(__ldg(reinterpret_cast<const uint2 *>(vsrc) + v));
                    } else {
                        kv = __ldg(reinterpret_cast<const uint4 *>(ksrc) + v);
                        vv = __ldg(reinterpret_cast<const uint4 *>(vsrc) + v);
                    }
                }
                kdst[v] = kv;
                vdst[v] = vv;
            }
        }
    }
}

int check_pool(const rx_kv_pool *pool)
{
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0)
        return rx_set_error(RX_ERR_INVALID, "rx_attn_extend: invalid pool");
    if (pool->head_dim != 64 && pool->head_dim != 128)
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_attn_extend: head_dim %d (supported: 64, 128)",
                            pool->head_dim);
    return RX_OK;
}

// Workspace of the staged path: int64 packed-row offsets [batch + 1], int32
// share sources [batch] and shared tile counts [batch], then the packed K
// rows and the packed V rows, [cap][kv heads][head_dim] bf16 each, every
// part 256-byte aligned.
struct StageLayout {
    size_t off_src, off_share, off_k, off_v, bytes;
};
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t stage_head(int32_t batch)
{
    return align256((size_t)(batch + 1) * sizeof(int64_t)) + 2 * align256((size_t)batch * sizeof(int32_t));
}
StageLayout stage_layout(int64_t cap, int32_t batch, int64_t row_bytes)
{
    StageLayout l;
    l.off_src = align256((size_t)(batch + 1) * sizeof(int64_t));
    l.off_share = l.off_src + align256((size_t)batch * sizeof(int32_t));
    l.off_k = stage_head(batch);
    const size_t region = align256((size_t)cap * (size_t)row_bytes);
    l.off_v = l.off_k + region;
    l.bytes = l.off_v + region;
    return l;
}
// largest row count a workspace of ws_bytes holds (TMA row coordinates are int32)
int64_t stage_cap_for(size_t ws_bytes, int32_t batch, int64_t row_bytes)
{
    const size_t head = stage_head(batch);
    if (ws_bytes <= head) return 0;
    int64_t cap = (int64_t)((ws_bytes - head) / 2 / (size_t)row_bytes);
    cap = cap < (int64_t)INT32_MAX - 2 * kBN ? cap : (int64_t)INT32_MAX - 2 * kBN;
    while (cap > 0 && stage_layout(cap, batch, row_bytes).bytes > ws_bytes) --cap;
    return cap;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); looked up once per process.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Packed rows [cap][hkv][D] bf16 as a 3-D map whose box is 64 elements (128
// bytes, the swizzle span) of one kv head over 64 consecutive rows.
int encode_stage_map(CUtensorMap *m, void *base, int64_t cap, int hkv, int D)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
    if (!fn) return rx_set_error(RX_ERR_CUDA, "rx_attn_extend: cuTensorMapEncodeTiled not available");
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)cap};
    const cuuint64_t strides[2] = {(cuuint64_t)D * sizeof(bf16), (cuuint64_t)hkv * D * sizeof(bf16)};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBN};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return rx_set_error(RX_ERR_CUDA, "rx_attn_extend: tensor map encode failed (%d)", (int)r);
    return RX_OK;
}

// Launches `kernel` on `st` as a programmatic dependent of the kernel
// enqueued just before it: it may start while that one runs and orders
// itself with pdl_wait.
template <typename... KArgs, typename... Args>
int launch_dependent(void (*kernel)(KArgs...), dim3 grid, unsigned block, size_t smem, cudaStream_t st,
                     Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    RX_CUDA_CHECK(cudaLaunchKernelEx(&cfg, kernel, args...));
    return RX_OK;
}

template <int D, bool kStaged, bool F8 = false>
int launch_extend(const XParams &p, dim3 grid, cudaStream_t st)
{
    static bool configured = false;
    if (!configured) {
        RX_CUDA_CHECK(cudaFuncSetAttribute(extend_kernel<D, kStaged, F8>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, XL<D>::BYTES));
        configured = true;
    }
    // staged: a programmatic dependent of the staging copy
    if (kStaged)
        return launch_dependent(extend_kernel<D, kStaged, F8>, grid, kStagedThreads, XL<D>::BYTES, st, p);
    extend_kernel<D, kStaged, F8><<<grid, kThreads, XL<D>::BYTES, st>>>(p);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}

}  // namespace

namespace {

// One layer of the pool an extend call reads: bf16 rows, or E4M3 codes with
// a scale per pool.
struct ExtendPool {
    const void *k, *v;
    int64_t num_slots;
    int hkv, D;
    bool f8;
    float k_scale, v_scale;
};

// rx_attn_extend and rx_attn_extend_fp8 after their pool checks (`who`
// names the entry point in messages).
int extend_call(const char *who, const ExtendPool &pool, const void *q, void *o, float *lse, int32_t hq,
                const int32_t *qo_indptr, const int32_t *req_idx, const int32_t *prefix_len,
                const int32_t *extend_len, const int32_t *rtt, int64_t rtt_stride, int32_t batch,
                int32_t max_extend_len, void *workspace, size_t ws_bytes, float sm_scale, int32_t *dev_status,
                void *stream)
{
    if (!q || !o || !qo_indptr || !req_idx || !prefix_len || !extend_len || !rtt ||
        rtt_stride <= 0 || rtt_stride > INT32_MAX || batch < 0 || hq <= 0 || max_extend_len < 0 ||
        !(sm_scale > 0.f))
        return rx_set_error(RX_ERR_INVALID, "%s: invalid argument", who);
    if (hq % pool.hkv != 0 || kRows % (hq / pool.hkv) != 0)
        return rx_set_error(RX_ERR_UNSUPPORTED, "%s: %d q heads over %d kv heads (need G | 128)", who, hq,
                            pool.hkv);
    // bf16 rows move in 16-byte pieces; code rows in 8-byte ones
    const uintptr_t pool_align = pool.f8 ? 7 : 15;
    if (rx_misaligned16(q) || rx_misaligned16(o) || (reinterpret_cast<uintptr_t>(pool.k) & pool_align) != 0 ||
        (reinterpret_cast<uintptr_t>(pool.v) & pool_align) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3) != 0)
        return rx_set_error(RX_ERR_INVALID, "%s: q and o must be 16-byte aligned, the pools %d-byte aligned", who,
                            (int)pool_align + 1);
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return rx_set_error(RX_ERR_INVALID, "%s: workspace must be 256-byte aligned", who);
    if (batch == 0 || max_extend_len == 0) return RX_OK;
    if (batch > 65535 || pool.hkv > 65535)
        return rx_set_error(RX_ERR_UNSUPPORTED, "%s: batch or kv heads above 65535", who);
    XParams p{};
    p.q = (const bf16 *)q;
    p.o = (bf16 *)o;
    p.lse = lse;
    p.k_pool = pool.f8 ? nullptr : (const bf16 *)pool.k;
    p.v_pool = pool.f8 ? nullptr : (const bf16 *)pool.v;
    p.k8 = pool.f8 ? (const unsigned char *)pool.k : nullptr;
    p.v8 = pool.f8 ? (const unsigned char *)pool.v : nullptr;
    p.num_slots = pool.num_slots;
    p.hq = hq;
    p.hkv = pool.hkv;
    p.G = hq / pool.hkv;
    p.qo_indptr = qo_indptr;
    p.req_idx = req_idx;
    p.prefix_len = prefix_len;
    p.extend_len = extend_len;
    p.rtt = rtt;
    p.rtt_stride = rtt_stride;
    p.scale_log2 = sm_scale * pool.k_scale * rx::kLog2e;
    p.v_scale = pool.v_scale;
    p.status = dev_status;
    const int tb = kCtaRows / p.G;
    dim3 grid((unsigned)((max_extend_len + tb - 1) / tb), (unsigned)p.hkv, (unsigned)batch);
    cudaStream_t st = (cudaStream_t)stream;
    const int D = pool.D;
    int rc = RX_OK;
    if (!workspace) {
        if (pool.f8)
            return D == 128 ? launch_extend<128, false, true>(p, grid, st) : launch_extend<64, false, true>(p, grid, st);
        return D == 128 ? launch_extend<128, false>(p, grid, st) : launch_extend<64, false>(p, grid, st);
    }

    // staged path: offsets, packed copy of every context, then attention
    const int64_t row_bytes = (int64_t)p.hkv * D * (int64_t)sizeof(bf16);
    const int64_t cap = stage_cap_for(ws_bytes, batch, row_bytes);
    if (cap < kBN) return rx_set_error(RX_ERR_CAPACITY, "%s: workspace of %zu bytes too small", who, ws_bytes);
    const StageLayout lay = stage_layout(cap, batch, row_bytes);
    int64_t *offs = static_cast<int64_t *>(workspace);
    bf16 *ks = reinterpret_cast<bf16 *>(static_cast<char *>(workspace) + lay.off_k);
    bf16 *vs = reinterpret_cast<bf16 *>(static_cast<char *>(workspace) + lay.off_v);
    if ((rc = encode_stage_map(&p.tm_k, ks, cap, p.hkv, D)) != RX_OK) return rc;
    if ((rc = encode_stage_map(&p.tm_v, vs, cap, p.hkv, D)) != RX_OK) return rc;
    int32_t *src = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + lay.off_src);
    int32_t *share = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + lay.off_share);
    p.stage_offs = offs;
    p.stage_src = src;
    p.stage_share = share;
    p.stage_cap = cap;
    int dev = 0, sms = 0;
    RX_CUDA_CHECK(cudaGetDevice(&dev));
    RX_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    stage_share_kernel<<<batch, kBN, 0, st>>>(rtt, rtt_stride, req_idx, prefix_len, extend_len, src, share);
    RX_CUDA_CHECK(cudaGetLastError());
    // the offsets, the copy and the attention kernel are each a programmatic
    // dependent of the kernel before: each waits on the device for what it reads
    if ((rc = launch_dependent(ctx_offsets_kernel, dim3(1), 1024, 0, st, prefix_len, extend_len,
                               (const int32_t *)share, batch, rtt_stride, cap, offs, dev_status)) != RX_OK)
        return rc;
    auto stage = pool.f8 ? stage_rows_kernel<true> : stage_rows_kernel<false>;
    if ((rc = launch_dependent(stage, dim3(sms * 8), 256, 0, st, pool.k, pool.v, p.num_slots, rtt, rtt_stride,
                               req_idx, prefix_len, extend_len, (const int32_t *)share, batch,
                               (const int64_t *)offs, cap, ks, vs, p.hkv * D, dev_status)) != RX_OK)
        return rc;
    return D == 128 ? launch_extend<128, true>(p, grid, st) : launch_extend<64, true>(p, grid, st);
}

}  // namespace

extern "C" int rx_attn_extend(const rx_kv_pool *pool_in, const void *q, void *o, float *lse,
                              int32_t hq, const int32_t *qo_indptr, const int32_t *req_idx,
                              const int32_t *prefix_len, const int32_t *extend_len,
                              const int32_t *rtt, int64_t rtt_stride, int32_t batch,
                              int32_t max_extend_len, void *workspace, size_t ws_bytes, float sm_scale,
                              int32_t *dev_status, void *stream)
{
    rx_kv_pool layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 0, "rx_attn_extend")) return rc;
    const rx_kv_pool *pool = pool_in ? &layer_view : nullptr;
    if (const int rc = check_pool(pool)) return rc;
    const ExtendPool ep{pool->k, pool->v, pool->num_slots, pool->num_kv_heads, pool->head_dim, false, 1.f, 1.f};
    return extend_call("rx_attn_extend", ep, q, o, lse, hq, qo_indptr, req_idx, prefix_len, extend_len, rtt,
                       rtt_stride, batch, max_extend_len, workspace, ws_bytes, sm_scale, dev_status, stream);
}

extern "C" int rx_attn_extend_fp8(const rx_kv_pool_fp8 *pool_in, const void *q, void *o, float *lse,
                                  int32_t hq, const int32_t *qo_indptr, const int32_t *req_idx,
                                  const int32_t *prefix_len, const int32_t *extend_len, const int32_t *rtt,
                                  int64_t rtt_stride, int32_t batch, int32_t max_extend_len, void *workspace,
                                  size_t ws_bytes, float sm_scale, int32_t *dev_status, void *stream)
{
    rx_kv_pool_fp8 layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 1, "rx_attn_extend_fp8")) return rc;
    const rx_kv_pool_fp8 *pool = pool_in ? &layer_view : nullptr;
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0 ||
        !(pool->k_scale > 0.f) || !(pool->v_scale > 0.f))
        return rx_set_error(RX_ERR_INVALID, "rx_attn_extend_fp8: invalid pool");
    if (pool->head_dim != 64 && pool->head_dim != 128)
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_attn_extend_fp8: head_dim %d (supported: 64, 128)",
                            pool->head_dim);
    const ExtendPool ep{pool->k, pool->v, pool->num_slots, pool->num_kv_heads, pool->head_dim, true,
                        pool->k_scale, pool->v_scale};
    return extend_call("rx_attn_extend_fp8", ep, q, o, lse, hq, qo_indptr, req_idx, prefix_len, extend_len, rtt,
                       rtt_stride, batch, max_extend_len, workspace, ws_bytes, sm_scale, dev_status, stream);
}

extern "C" size_t rx_attn_extend_workspace(int64_t total_ctx_tokens, int32_t batch, int32_t num_kv_heads,
                                           int32_t head_dim)
{
    if (total_ctx_tokens < 0 || batch <= 0 || batch > 65535 || num_kv_heads <= 0 ||
        (head_dim != 64 && head_dim != 128)) {
        rx_set_error(RX_ERR_INVALID, "rx_attn_extend_workspace: invalid argument");
        return 0;
    }
    const int64_t cap = total_ctx_tokens + (int64_t)(kBN - 1) * batch;  // each context rounded up to kBN rows
    if (cap > (int64_t)INT32_MAX - 2 * kBN) {
        rx_set_error(RX_ERR_UNSUPPORTED, "rx_attn_extend_workspace: %lld context rows", (long long)cap);
        return 0;
    }
    return stage_layout(cap < kBN ? kBN : cap, batch, (int64_t)num_kv_heads * head_dim * 2).bytes;
}
