// rx_decode.cu -- decode attention over the token-slot pool: a persistent,
// warp-specialised split-KV kernel plus the log-sum-exp merge of split
// results.
//
// What is computed: for each request b (one query at position L_b - 1) and
// q-head h, o = softmax(sm_scale * q K^T) V over the pool rows listed in
// req_to_token[b][0 .. L_b-1], kv-head g = h / G.  Work is cut into items:
// a set of query rows that read the same positions [p0, p1) of the same
// slot list -- the requests below one shared radix node, times the G q-heads
// of one kv head -- so the KV of a shared prefix is read from HBM once per
// group ("SGLang: Efficient Execution of Structured Language Model Programs",
// unite.ai, es, section "SGLang: Modelo de programación y metodología":
// requests that share a prefix share its KV).  Items come from a host-built
// decode plan, or, without one, from a fixed split of every request.
//
// The kernel is HBM-bound (about 4 flops per KV byte), so it is built to keep
// bytes in flight:
//   - one persistent CTA per SM walks a static round-robin share of the
//     (item, kv head) list, longest items first;
//   - a scheduler warp decodes the CTA's items 32 at a time (lane-parallel
//     loads), publishes each as a descriptor in a 4-deep ring, and prefetches
//     the slot ids of every 64-key stage with 4-byte cp.async into a 16-deep
//     slot ring -- so no copy ever waits on a dependent index load;
//   - seven copier warps gather K and V rows (head_dim * 2 contiguous bytes
//     per row and kv head, 16-byte cp.async, a seventh of every stage each)
//     into a ring of 64-key stages, and the query rows into a double-buffered
//     Q slot; every ring entry is an mbarrier that the copies themselves
//     complete (cp.async.mbarrier.arrive), so the ring streams across item
//     boundaries with no per-item fill or drain.  Several issuing warps are
//     needed: measured on GB300, one warp issuing either 16-byte cp.async or
//     256-byte bulk copies keeps only a few KB in flight (about 1 TB/s);
//   - four consumer warps run S = Q K^T and O += P V on mma.sync m16n8k16
//     (bf16 in, fp32 accumulators; the contraction is small, so the legacy
//     tensor path is ample) with the online softmax in the exp2 domain; they
//     split the rows 16 per warp when an item has many rows and split each
//     stage's keys when it has few, combining key-split partials through
//     shared memory;
//   - rows sit at a padded stride of head_dim * 2 + 16 bytes, so the eight
//     rows an ldmatrix reads fall in distinct banks; stage rows past an
//     item's end are zero-filled by the copy and their scores masked.
// Single-request items of a plan with one q head per kv head go instead to
// decode_wide_kernel (below), which reads whole slot rows across all kv heads
// and runs alongside this kernel.
// An item that covers a row's whole context writes bf16 o directly;
// otherwise it writes a normalised fp32 partial and its log2-sum-exp, and
// merge_kernel combines them: o = sum_s w_s o_s / sum_s w_s with
// w_s = 2^(lse_s - max lse).
//
// Every mbarrier wait is bounded; a wait that gives up sets RX_DEV_TIMEOUT,
// raises a shared abort flag so the other warps stop too, and each copying
// warp waits for its own copies before the CTA exits.
#include <math.h>

#include <mutex>

#include <atomic>
#include <type_traits>

#include "rx_common.cuh"

namespace {

using bf16 = __nv_bfloat16;

constexpr int kBN = 64;                      // keys per stage
constexpr int kCopiers = 7;                  // copier warps
constexpr int kConsumers = 4;                // consumer warps
constexpr int kThreads = 32 * (1 + kCopiers + kConsumers);  // scheduler, copiers, consumers
constexpr int kConsumer0 = 32 * (1 + kCopiers);  // first consumer thread
constexpr int kMaxRows = 64;                 // query rows per item
constexpr int kNIT = 4;                      // item descriptor ring
constexpr int kNSL = 16;                     // slot-id ring (stages)

// Item descriptor published by the scheduler warp.  M == 0 ends the stream.
struct Desc {
    int M, p0, p1, part, final_, g, rtt_row, pad;
    int qrow[kMaxRows];                      // q/o row of each request of the item
};

// F8: the pools hold E4M3 codes; the ring's tiles stay bf16 (codes widened on
// the way in), with one stage fewer at d 128 to make room for two buffers of
// a stage's codes.
template <int D, bool F8 = false>
struct Layout {
    static constexpr int NST = (D == 128) ? (F8 ? 3 : 4) : 8;  // K/V ring stages
    static constexpr int RS = D + 8;                    // padded row stride (elements)
    static constexpr int TILE = kBN * RS;               // elements of one K (or V) stage
    static constexpr int QSLOT = kMaxRows * RS;         // elements of one Q slot
    static constexpr int RED_FLOATS = 2 * 4 * 16 + 4 * 16 * D;  // m, l and O of 4 key splits
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NST * TILE * 2;
    static constexpr int OFF_Q = OFF_V + NST * TILE * 2;
    static constexpr int OFF_RED = OFF_Q + 2 * QSLOT * 2;
    static constexpr int OFF_SLOT = OFF_RED + RED_FLOATS * 4;
    static constexpr int OFF_DESC = OFF_SLOT + kNSL * kBN * 4;
    static constexpr int OFF_BAR = OFF_DESC + kNIT * (int)sizeof(Desc);
    // barrier indices
    static constexpr int B_FULL = 0, B_EMPTY = NST, B_QFULL = 2 * NST, B_QEMPTY = 2 * NST + 2,
                         B_SLFULL = 2 * NST + 4, B_SLEMPTY = B_SLFULL + kNSL,
                         B_ITFULL = B_SLEMPTY + kNSL, B_ITEMPTY = B_ITFULL + kNIT,
                         B_RED = B_ITEMPTY + kNIT, N_BAR = B_RED + 1;
    static constexpr int OFF_ABORT = OFF_BAR + N_BAR * 8;
    // FP8: two buffers of one stage's codes, K then V (kBN rows of D bytes)
    static constexpr int CODE_STAGE = 2 * kBN * D;
    static constexpr int OFF_CODE = (OFF_ABORT + 16 + 127) / 128 * 128;
    static constexpr int BYTES = F8 ? OFF_CODE + 2 * CODE_STAGE : OFF_ABORT + 16;
};
static_assert(Layout<128>::BYTES <= 227 * 1024, "shared memory budget");
static_assert(Layout<64>::BYTES <= 227 * 1024, "shared memory budget");
static_assert(Layout<128, true>::BYTES <= 227 * 1024, "shared memory budget");
static_assert(Layout<64, true>::BYTES <= 227 * 1024, "shared memory budget");

struct Params {
    const bf16 *q;
    bf16 *o;
    float *lse;
    const bf16 *k_pool;
    const bf16 *v_pool;
    int64_t num_slots;
    int hq, hkv, G;
    int head_dim;
    const int32_t *req_idx;
    const int32_t *seq_len;
    const int32_t *rtt;
    int64_t rtt_stride;
    const int32_t *order;   // plan
    const int32_t *nparts;  // plan
    const int32_t *items;   // plan
    int batch;
    int chunk;              // no plan: positions per item
    int n_chunks;           // no plan: items per request
    int total_work;         // items x kv heads
    int max_parts;          // partial-result stride per row
    float *ws_o;
    float *ws_lse;
    float scale_log2;
    int32_t *status;
    int wide0, n_wide;      // plan: single-request items for the wide kernel
    int *wide_counter;      // next wide item to hand out (zeroed before the launch)
    long long wait_cycles;  // bound on each pipeline wait (rx_decode_set_wait_limit)
    // the pools as bytes, for the all-heads kernels' whole-row copies: bf16
    // pools (row_bytes = hkv * d * 2) or FP8 code pools (hkv * d)
    const unsigned char *kb;
    const unsigned char *vb;
    int64_t row_bytes;
    float v_scale;          // FP8 pools: scale of V (K's is folded into scale_log2); 1 otherwise
};

struct Item {
    int M, p0, p1, part, final_, g, rtt_row, qrow0, r0;
};

// End of a plan item whose pos_end is RX_PLAN_OPEN_END: the length of its
// request (batch index b) now.  A length past the slot-list stride, or not
// past the item's start, is an error: flagged (by `report` lanes), and the
// item is read as its first position alone, so that nothing outside the
// buffers is touched and no row is left without keys.
__device__ __forceinline__ int open_end(const Params &p, int b, int p0, bool report)
{
    const int64_t L = __ldg(p.seq_len + b);
    if (L > p0 && L <= p.rtt_stride) return (int)L;
    if (report && p.status) atomicOr(p.status, RX_DEV_BAD_LEN);
    return p0 + 1;
}

// Decodes work index w (one per lane); false when the item is empty.
template <bool PLAN>
__device__ __forceinline__ bool get_item(const Params &p, int w, Item &it)
{
    it.g = w % p.hkv;
    const int i = w / p.hkv;
    if (PLAN) {
        // scalar loads: the items array is only 4-byte aligned
        const int32_t *v = p.items + 8 * (int64_t)i;
        it.r0 = __ldg(v + 0);
        it.M = __ldg(v + 1) * p.G;
        it.p0 = __ldg(v + 2);
        it.p1 = __ldg(v + 3);
        it.part = __ldg(v + 4);
        it.final_ = __ldg(v + 5);
        it.rtt_row = __ldg(v + 6);
        it.qrow0 = __ldg(v + 7);
        if (it.p1 == RX_PLAN_OPEN_END) it.p1 = open_end(p, it.qrow0, it.p0, it.g == 0);
        return it.M > 0 && it.p1 > it.p0;
    }
    const int b = i / p.n_chunks, c = i % p.n_chunks;
    const int64_t L = __ldg(p.seq_len + b);
    if (L > (int64_t)p.n_chunks * p.chunk || L > p.rtt_stride) {  // past max_seq_len
        if (c == 0 && it.g == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_LEN);
        return false;
    }
    const int p0 = c * p.chunk;
    if (p0 >= L) return false;
    it.r0 = 0;
    it.M = p.G;
    it.p0 = p0;
    it.p1 = (int)min(L, (int64_t)p0 + p.chunk);
    it.part = c;
    it.final_ = L <= p.chunk;
    it.rtt_row = __ldg(p.req_idx + b);
    it.qrow0 = b;
    return true;
}

// Bounded wait by a whole warp, with one answer for all its lanes (the warp
// then runs warp-wide shuffles, ldmatrix and barriers).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status, long long limit)
{
    // already complete: no suspend; otherwise blocking tries while the
    // limit lasts (the clock is read before each try, since one try may
    // itself suspend for longer than a small limit)
    bool ok = rx::mbar_test_wait(bar, parity);
    if (!ok) {
        const long long t0 = clock64();
        while (clock64() - t0 < limit) {
            if (rx::mbar_try_wait(bar, parity)) {
                ok = true;
                break;
            }
            if (*abort_flag) break;
        }
    }
    if (!ok && !*abort_flag) {
        *abort_flag = 1;
        if (status) atomicOr(status, RX_DEV_TIMEOUT);
    }
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int mpad_of(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

__device__ __forceinline__ int shfl(int v, int src) { return __shfl_sync(0xffffffffu, v, src); }

// ---------------------------------------------------------------------------
// scheduler warp: descriptors and slot ids
// ---------------------------------------------------------------------------

template <int D, bool PLAN, bool F8>
__device__ void scheduler(const Params &p, unsigned char *smem)
{
    using L = Layout<D, F8>;
    Desc *descs = reinterpret_cast<Desc *>(smem + L::OFF_DESC);
    int32_t *slotbuf = reinterpret_cast<int32_t *>(smem + L::OFF_SLOT);
    const uint32_t bar = rx::smem_u32(smem + L::OFF_BAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    const int lane = threadIdx.x & 31;
    uint32_t n_it = 0, n_tile = 0;
    bool alive = true;
    auto publish = [&](const Item &it, bool end) -> bool {
        const uint32_t di = n_it % kNIT;
        if (!wait_or_abort(bar + 8 * (L::B_ITEMPTY + di), ((n_it / kNIT) & 1) ^ 1, abort_flag, p.status, p.wait_cycles))
            return false;
        Desc *d = descs + di;
        if (lane == 0) {
            d->M = end ? 0 : it.M;
            d->p0 = it.p0;
            d->p1 = it.p1;
            d->part = it.part;
            d->final_ = it.final_;
            d->g = it.g;
            d->rtt_row = it.rtt_row;
            d->qrow[0] = it.qrow0;
        }
        if (!end && PLAN) {
            const int nreq = it.M / p.G;
            for (int i = 1 + lane; i < nreq; i += 32) d->qrow[i] = __ldg(p.order + it.r0 + i);
        }
        __syncwarp();
        if (lane == 0) rx::mbar_arrive(bar + 8 * (L::B_ITFULL + di));
        ++n_it;
        return true;
    };
    for (int base = 0; alive && blockIdx.x + base * (int)gridDim.x < p.total_work; base += 32) {
        const int wl = blockIdx.x + (base + lane) * (int)gridDim.x;
        Item mine{};
        const bool vl = wl < p.total_work && get_item<PLAN>(p, wl, mine);
        for (int j = 0; j < 32; ++j) {
            if (blockIdx.x + (base + j) * (int)gridDim.x >= p.total_work) break;
            if (!__shfl_sync(0xffffffffu, vl, j)) continue;
            Item it;
            it.M = shfl(mine.M, j);
            it.p0 = shfl(mine.p0, j);
            it.p1 = shfl(mine.p1, j);
            it.part = shfl(mine.part, j);
            it.final_ = shfl(mine.final_, j);
            it.g = shfl(mine.g, j);
            it.rtt_row = shfl(mine.rtt_row, j);
            it.qrow0 = shfl(mine.qrow0, j);
            it.r0 = shfl(mine.r0, j);
            if (!publish(it, false)) {
                alive = false;
                break;
            }
            const int32_t *row = p.rtt + (int64_t)it.rtt_row * p.rtt_stride;
            const int ntiles = (it.p1 - it.p0 + kBN - 1) / kBN;
            for (int t = 0; t < ntiles; ++t, ++n_tile) {
                const uint32_t sb = n_tile % kNSL;
                if (!wait_or_abort(bar + 8 * (L::B_SLEMPTY + sb), ((n_tile / kNSL) & 1) ^ 1, abort_flag,
                                   p.status, p.wait_cycles)) {
                    alive = false;
                    break;
                }
                int32_t *dst = slotbuf + sb * kBN;
                const int pos = it.p0 + t * kBN + lane;
                rx::cp_async_4(rx::smem_u32(dst + lane), row + (pos < it.p1 ? pos : 0), pos < it.p1 ? 4 : 0);
                rx::cp_async_4(rx::smem_u32(dst + lane + 32), row + (pos + 32 < it.p1 ? pos + 32 : 0),
                               pos + 32 < it.p1 ? 4 : 0);
                rx::cp_async_mbar_arrive(bar + 8 * (L::B_SLFULL + sb));
            }
            if (!alive) break;
        }
    }
    if (alive) publish(Item{}, true);
    rx::cp_async_wait_all();
}

// ---------------------------------------------------------------------------
// copier warp: Q rows and K/V stages
// ---------------------------------------------------------------------------

// Eight E4M3 codes (element 0 in the low byte) as eight bf16: every E4M3
// value, subnormals included, is exact in f16 and in bf16.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint32_t lo, uint32_t hi)
{
    const uint32_t w[2] = {lo, hi};
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t h = rx::e4m3x2_to_f16x2((uint16_t)(w[k >> 1] >> (16 * (k & 1))));
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
        r[k] = rx::pack_bf16(f.x, f.y);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// F8: each copier thread lands its 16-byte chunks of a tile's codes in code
// buffer (tile & 1) with cp.async, and once they are in (one tile later, or
// at the item's end) widens exactly those chunks into the tile's bf16 rows
// and arrives on its full barrier itself -- no thread reads codes another
// copied, so nothing but the thread's own cp.async groups orders the steps.
template <int D, bool F8>
__device__ void copier(const Params &p, unsigned char *smem)
{
    using L = Layout<D, F8>;
    constexpr int CPR = F8 ? D / 16 : D / 8;            // 16-byte chunks per row (codes or bf16)
    constexpr int QCPR = D / 8;                         // 16-byte chunks per query row
    constexpr int NCT = 32 * kCopiers;                  // copier threads
    bf16 *Ks = reinterpret_cast<bf16 *>(smem + L::OFF_K);
    bf16 *Vs = reinterpret_cast<bf16 *>(smem + L::OFF_V);
    bf16 *Qs = reinterpret_cast<bf16 *>(smem + L::OFF_Q);
    const Desc *descs = reinterpret_cast<const Desc *>(smem + L::OFF_DESC);
    const int32_t *slotbuf = reinterpret_cast<const int32_t *>(smem + L::OFF_SLOT);
    const uint32_t bar = rx::smem_u32(smem + L::OFF_BAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    const int lane = threadIdx.x & 31, ct = threadIdx.x - 32;
    uint32_t n_it = 0, n_tile = 0, qi = 0;
    for (;; ++n_it) {
        const uint32_t di = n_it % kNIT;
        if (!wait_or_abort(bar + 8 * (L::B_ITFULL + di), (n_it / kNIT) & 1, abort_flag, p.status, p.wait_cycles)) break;
        const Desc *d = descs + di;
        const int M = d->M, p0 = d->p0, p1 = d->p1, g = d->g;
        if (M == 0) break;
        {  // query rows -> Q slot (rows past M zero-filled), by every copier thread
            const uint32_t qs = qi & 1;
            if (!wait_or_abort(bar + 8 * (L::B_QEMPTY + qs), ((qi >> 1) & 1) ^ 1, abort_flag, p.status, p.wait_cycles))
                break;
            const int Mpad = mpad_of(M);
            bf16 *qd = Qs + qs * L::QSLOT;
            for (int idx = ct; idx < Mpad * QCPR; idx += NCT) {
                const int m = idx / QCPR, c = idx % QCPR;
                const uint32_t dst = rx::smem_u32(qd + m * L::RS + c * 8);
                if (m < M) {
                    const int64_t qr = d->qrow[m / p.G];
                    rx::cp_async_16(dst, p.q + ((qr * p.hq + (int64_t)g * p.G + m % p.G) * D + c * 8), 16);
                } else {
                    rx::cp_async_16(dst, p.q, 0);
                }
            }
            rx::cp_async_mbar_arrive(bar + 8 * (L::B_QFULL + qs));
            ++qi;
        }
        __syncwarp();
        if (lane == 0) rx::mbar_arrive(bar + 8 * (L::B_ITEMPTY + di));
        // K/V stages: the copier threads stride over the stage's 16-byte chunks
        const int ntiles = (p1 - p0 + kBN - 1) / kBN;
        bool ok_all = true;
        int64_t pend = -1;  // F8: the tile whose codes this thread has in flight
        // F8: this thread's chunks of tile nt's codes -> the tile's bf16 rows,
        // once the ring stage is free; then its arrival on the stage's full barrier
        auto widen = [&](uint32_t nt) -> bool {
            const uint32_t s = nt % L::NST;
            if (!wait_or_abort(bar + 8 * (L::B_EMPTY + s), ((nt / L::NST) & 1) ^ 1, abort_flag, p.status,
                               p.wait_cycles))
                return false;
            const unsigned char *cb = smem + L::OFF_CODE + (nt & 1) * L::CODE_STAGE;
            bf16 *kd = Ks + s * L::TILE;
            bf16 *vd = Vs + s * L::TILE;
            for (int idx = ct; idx < kBN * CPR; idx += NCT) {
                const int r = idx / CPR, c = idx % CPR;
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(cb + kv * kBN * D + r * D + c * 16);
                    uint4 *dst = reinterpret_cast<uint4 *>((kv ? vd : kd) + r * L::RS + c * 16);
                    dst[0] = e4m3x8_to_bf16x8(w.x, w.y);
                    dst[1] = e4m3x8_to_bf16x8(w.z, w.w);
                }
            }
            rx::mbar_arrive(bar + 8 * (L::B_FULL + s));
            return true;
        };
        for (int t = 0; t < ntiles; ++t, ++n_tile) {
            const uint32_t sb = n_tile % kNSL, s = n_tile % L::NST;
            if (!wait_or_abort(bar + 8 * (L::B_SLFULL + sb), (n_tile / kNSL) & 1, abort_flag, p.status, p.wait_cycles) ||
                (!F8 && !wait_or_abort(bar + 8 * (L::B_EMPTY + s), ((n_tile / L::NST) & 1) ^ 1, abort_flag,
                                       p.status, p.wait_cycles))) {
                ok_all = false;
                break;
            }
            const int base = p0 + t * kBN;
            const int32_t *sl = slotbuf + sb * kBN;
            if constexpr (F8) {
                unsigned char *cb = smem + L::OFF_CODE + (n_tile & 1) * L::CODE_STAGE;
#pragma unroll 4
                for (int idx = ct; idx < kBN * CPR; idx += NCT) {
                    const int r = idx / CPR, c = idx % CPR;
                    const int32_t slot = sl[r];
                    const bool inside = base + r < p1;
                    const bool ok = inside && slot >= 0 && (int64_t)slot < p.num_slots;
                    if (inside && !ok && c == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_SLOT);
                    const int64_t off = ok ? (((int64_t)slot * p.hkv + g) * D + c * 16) : 0;
                    rx::cp_async_16(rx::smem_u32(cb + r * D + c * 16), p.kb + off, ok ? 16 : 0);
                    rx::cp_async_16(rx::smem_u32(cb + kBN * D + r * D + c * 16), p.vb + off, ok ? 16 : 0);
                }
                rx::cp_async_commit();
            } else {
                bf16 *kd = Ks + s * L::TILE;
                bf16 *vd = Vs + s * L::TILE;
#pragma unroll 4
                for (int idx = ct; idx < kBN * CPR; idx += NCT) {
                    const int r = idx / CPR, c = idx % CPR;
                    const int32_t slot = sl[r];
                    const bool inside = base + r < p1;
                    const bool ok = inside && slot >= 0 && (int64_t)slot < p.num_slots;
                    if (inside && !ok && c == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_SLOT);
                    const int64_t off = ok ? (((int64_t)slot * p.hkv + g) * D + c * 8) : 0;
                    const int dsto = r * L::RS + c * 8;
                    rx::cp_async_16(rx::smem_u32(kd + dsto), p.k_pool + off, ok ? 16 : 0);
                    rx::cp_async_16(rx::smem_u32(vd + dsto), p.v_pool + off, ok ? 16 : 0);
                }
            }
            __syncwarp();
            if (lane == 0) rx::mbar_arrive(bar + 8 * (L::B_SLEMPTY + sb));
            if constexpr (F8) {
                // the previous tile's codes are in once only this tile's group
                // may still be pending
                if (pend >= 0) {
                    rx::cp_async_wait<1>();
                    if (!widen((uint32_t)pend)) {
                        ok_all = false;
                        break;
                    }
                }
                pend = n_tile;
            } else {
                rx::cp_async_mbar_arrive(bar + 8 * (L::B_FULL + s));
            }
        }
        // F8: the item's last tile, before anything that waits on the consumers
        if (F8 && ok_all && pend >= 0) {
            rx::cp_async_wait<0>();
            ok_all = widen((uint32_t)pend);
        }
        if (!ok_all) break;
    }
    rx::cp_async_wait_all();
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------

template <int D, int WM, bool F8>
__device__ bool consume(const Params &p, const Desc *d, unsigned char *smem, uint32_t &n_tile,
                        uint32_t &qi, uint32_t &n_red)
{
    using L = Layout<D, F8>;
    constexpr int WK = kConsumers / WM;   // warps along keys
    constexpr int KW = kBN / WK;          // keys per warp per stage
    constexpr int NT = KW / 8;            // S n-tiles per warp
    constexpr int KT = KW / 16;           // PV k-steps per warp
    constexpr int DT = D / 8;             // O n-tiles
    constexpr int Mpad = WM * 16;
    const bf16 *Ks = reinterpret_cast<const bf16 *>(smem + L::OFF_K);
    const bf16 *Vs = reinterpret_cast<const bf16 *>(smem + L::OFF_V);
    const bf16 *Qs = reinterpret_cast<const bf16 *>(smem + L::OFF_Q);
    const uint32_t bar = rx::smem_u32(smem + L::OFF_BAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    const int cw = (threadIdx.x - kConsumer0) >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int wm = cw % WM, wk = cw / WM;
    const int G = p.G;
    const int M = d->M, p0 = d->p0, p1 = d->p1, g = d->g, part = d->part;
    const bool fin = d->final_ != 0;

    // Q fragments
    const uint32_t qs = qi & 1;
    if (!wait_or_abort(bar + 8 * (L::B_QFULL + qs), (qi >> 1) & 1, abort_flag, p.status, p.wait_cycles)) return false;
    uint32_t qf[D / 16][4];
    {
        const bf16 *qb = Qs + qs * L::QSLOT;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int row = wm * 16 + (lane & 15);
            const int ch = ks * 2 + (lane >> 4);
            rx::ldmatrix_x4(rx::smem_u32(qb + row * L::RS + ch * 8), qf[ks][0], qf[ks][1], qf[ks][2],
                            qf[ks][3]);
        }
    }
    __syncwarp();
    if (lane == 0) rx::mbar_arrive(bar + 8 * (L::B_QEMPTY + qs));
    ++qi;

    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};
    float oacc[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    const int ntiles = (p1 - p0 + kBN - 1) / kBN;
    for (int t = 0; t < ntiles; ++t, ++n_tile) {
        const uint32_t s = n_tile % L::NST;
        if (!wait_or_abort(bar + 8 * (L::B_FULL + s), (n_tile / L::NST) & 1, abort_flag, p.status, p.wait_cycles))
            return false;
        const bf16 *kt = Ks + s * L::TILE;
        const bf16 *vt = Vs + s * L::TILE;
        float sc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const int key = wk * KW + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4(rx::smem_u32(kt + key * L::RS + ch * 8), b0, b1, b2, b3);
                rx::mma_bf16_16816(sc[2 * np], qf[ks], b0, b1);
                rx::mma_bf16_16816(sc[2 * np + 1], qf[ks], b2, b3);
            }
        }
        const int kpos0 = p0 + t * kBN + wk * KW;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int pos = kpos0 + nt * 8 + tig * 2 + (j & 1);
                sc[nt][j] = (pos < p1) ? sc[nt][j] * p.scale_log2 : -INFINITY;
            }
            mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        if (mn0 != m_r[0] || mn1 != m_r[1]) {
            const float a0 = rx::fast_exp2(m_r[0] - mu0), a1 = rx::fast_exp2(m_r[1] - mu1);
            l_r[0] *= a0;
            l_r[1] *= a1;
#pragma unroll
            for (int i = 0; i < DT; ++i) {
                oacc[i][0] *= a0;
                oacc[i][1] *= a0;
                oacc[i][2] *= a1;
                oacc[i][3] *= a1;
            }
            m_r[0] = mn0;
            m_r[1] = mn1;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            sc[nt][0] = rx::fast_exp2(sc[nt][0] - mu0);
            sc[nt][1] = rx::fast_exp2(sc[nt][1] - mu0);
            sc[nt][2] = rx::fast_exp2(sc[nt][2] - mu1);
            sc[nt][3] = rx::fast_exp2(sc[nt][3] - mu1);
            l_r[0] += sc[nt][0] + sc[nt][1];
            l_r[1] += sc[nt][2] + sc[nt][3];
        }
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            uint32_t a[4];
            a[0] = rx::pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
            a[1] = rx::pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
            a[2] = rx::pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            a[3] = rx::pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int key = wk * KW + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4_trans(rx::smem_u32(vt + key * L::RS + ch * 8), b0, b1, b2, b3);
                rx::mma_bf16_16816(oacc[2 * dp], a, b0, b1);
                rx::mma_bf16_16816(oacc[2 * dp + 1], a, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) rx::mbar_arrive(bar + 8 * (L::B_EMPTY + s));
    }

    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 1);
    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 2);
    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 1);
    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 2);

    auto out_row = [&](int m) -> int64_t {
        return (int64_t)d->qrow[m / G] * p.hq + (int64_t)g * G + m % G;
    };
    if constexpr (WK == 1) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = wm * 16 + gid + half * 8;
            if (r >= M) continue;
            const int64_t orow = out_row(r);
            const float inv = p.v_scale / l_r[half];  // V's scale: 1 for a bf16 pool
            if (fin) {
                bf16 *dst = p.o + orow * D;
#pragma unroll
                for (int dt = 0; dt < DT; ++dt)
                    *reinterpret_cast<uint32_t *>(dst + dt * 8 + tig * 2) =
                        rx::pack_bf16(oacc[dt][2 * half] * inv, oacc[dt][2 * half + 1] * inv);
                if (p.lse && tig == 0) p.lse[orow] = (m_r[half] + log2f(l_r[half])) * rx::kLn2;
            } else {
                const int64_t prow = orow * p.max_parts + part;
                float *dst = p.ws_o + prow * D;
                const uint64_t keep = rx::l2_evict_last();  // the merge reads them back, then discards the lines
#pragma unroll
                for (int dt = 0; dt < DT; ++dt)
                    rx::st_hint(dst + dt * 8 + tig * 2, oacc[dt][2 * half] * inv, oacc[dt][2 * half + 1] * inv, keep);
                if (tig == 0) p.ws_lse[prow] = m_r[half] + log2f(l_r[half]);
            }
        }
    } else {
        float *red_m = reinterpret_cast<float *>(smem + L::OFF_RED);
        float *red_l = red_m + WK * Mpad;
        float *red_o = red_l + WK * Mpad;  // [WK][Mpad][D]
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = wm * 16 + gid + half * 8;
            if (tig == 0) {
                red_m[wk * Mpad + r] = m_r[half];
                red_l[wk * Mpad + r] = l_r[half];
            }
#pragma unroll
            for (int dt = 0; dt < DT; ++dt)
                *reinterpret_cast<float2 *>(red_o + (wk * Mpad + r) * D + dt * 8 + tig * 2) =
                    make_float2(oacc[dt][2 * half], oacc[dt][2 * half + 1]);
        }
        // consumer-only barrier: one arrival per warp, bounded wait
        __syncwarp();
        if (lane == 0) rx::mbar_arrive(bar + 8 * L::B_RED);
        if (!wait_or_abort(bar + 8 * L::B_RED, n_red & 1, abort_flag, p.status, p.wait_cycles)) return false;
        ++n_red;
        const int ct = threadIdx.x - kConsumer0;
        for (int e = ct; e < Mpad * D; e += 32 * kConsumers) {
            const int r = e / D, c = e % D;
            if (r >= M) continue;
            float mt = -INFINITY;
#pragma unroll
            for (int k = 0; k < WK; ++k) mt = fmaxf(mt, red_m[k * Mpad + r]);
            const float mu = (mt == -INFINITY) ? 0.f : mt;
            float lt = 0.f, ot = 0.f;
#pragma unroll
            for (int k = 0; k < WK; ++k) {
                const float f = rx::fast_exp2(red_m[k * Mpad + r] - mu);
                lt += red_l[k * Mpad + r] * f;
                ot += red_o[(k * Mpad + r) * D + c] * f;
            }
            const int64_t orow = out_row(r);
            ot *= p.v_scale;  // V's scale: 1 for a bf16 pool
            if (fin) {
                p.o[orow * D + c] = __float2bfloat16_rn(ot / lt);
                if (p.lse && c == 0) p.lse[orow] = (mt + log2f(lt)) * rx::kLn2;
            } else {
                const int64_t prow = orow * p.max_parts + part;
                const uint64_t keep = rx::l2_evict_last();  // the merge reads them back, then discards the lines
                rx::st_hint(p.ws_o + prow * D + c, ot / lt, keep);
                if (c == 0) p.ws_lse[prow] = mt + log2f(lt);
            }
        }
        __syncwarp();  // the next item may overwrite the buffer once every warp is here
        if (lane == 0) rx::mbar_arrive(bar + 8 * L::B_RED);
        if (!wait_or_abort(bar + 8 * L::B_RED, n_red & 1, abort_flag, p.status, p.wait_cycles)) return false;
        ++n_red;
    }
    return true;
}

template <int D, bool PLAN, bool F8>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const Params p)
{
    using L = Layout<D, F8>;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t bar = rx::smem_u32(smem + L::OFF_BAR);
    // the kernels after this one in the call do not wait for it to start
    // (the all-heads kernel) or wait for it in their own code (the merge)
    rx::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::NST; ++s) {
            rx::mbar_init(bar + 8 * (L::B_FULL + s), 32 * kCopiers);  // copier lanes' copies
            rx::mbar_init(bar + 8 * (L::B_EMPTY + s), kConsumers);
        }
        for (int q = 0; q < 2; ++q) {
            rx::mbar_init(bar + 8 * (L::B_QFULL + q), 32 * kCopiers);  // every copier lane's copies
            rx::mbar_init(bar + 8 * (L::B_QEMPTY + q), kConsumers);
        }
        for (int s = 0; s < kNSL; ++s) {
            rx::mbar_init(bar + 8 * (L::B_SLFULL + s), 32);       // scheduler lanes' copies
            rx::mbar_init(bar + 8 * (L::B_SLEMPTY + s), kCopiers);
        }
        for (int i = 0; i < kNIT; ++i) {
            rx::mbar_init(bar + 8 * (L::B_ITFULL + i), 1);        // scheduler
            rx::mbar_init(bar + 8 * (L::B_ITEMPTY + i), kCopiers + kConsumers);
        }
        rx::mbar_init(bar + 8 * L::B_RED, kConsumers);            // consumer-only barrier
        *reinterpret_cast<volatile int *>(smem + L::OFF_ABORT) = 0;
        rx::fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        scheduler<D, PLAN, F8>(p, smem);
        return;
    }
    if (warp <= kCopiers) {
        copier<D, F8>(p, smem);
        return;
    }
    const Desc *descs = reinterpret_cast<const Desc *>(smem + L::OFF_DESC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_ABORT);
    const int lane = threadIdx.x & 31;
    uint32_t n_it = 0, n_tile = 0, qi = 0, n_red = 0;
    for (;; ++n_it) {
        const uint32_t di = n_it % kNIT;
        if (!wait_or_abort(bar + 8 * (L::B_ITFULL + di), (n_it / kNIT) & 1, abort_flag, p.status, p.wait_cycles)) return;
        const Desc *d = descs + di;
        const int M = d->M;
        if (M == 0) return;
        bool ok;
        if (M <= 16)
            ok = consume<D, 1, F8>(p, d, smem, n_tile, qi, n_red);
        else if (M <= 32)
            ok = consume<D, 2, F8>(p, d, smem, n_tile, qi, n_red);
        else
            ok = consume<D, 4, F8>(p, d, smem, n_tile, qi, n_red);
        if (!ok) return;
        __syncwarp();
        if (lane == 0) rx::mbar_arrive(bar + 8 * (L::B_ITEMPTY + di));
    }
}

constexpr int kMergeFew = 12;    // parts up to which a row's partials are loaded in one go
constexpr int kMergeBatch = 16;  // rows a batch above that (up to 64 parts)

// FEW (4, 8 or kMergeFew): the parts a row may have for the one-round-trip
// path, the call's max_parts rounded up; MANY: rows may have more than
// kMergeFew parts, and only then is the batched path built.  Registers grow
// with both, and a merge of many rows with few parts each (thousands of
// warps) wants them small, so that its CTAs fit the GPU in one wave.
template <int D, int FEW, bool MANY>
__global__ void __launch_bounds__(128) merge_kernel(const Params p, int use_plan)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;
    const bool live = row < (int64_t)p.batch * p.hq;
    int np = 0;
    if (live) {  // the plan and the lengths are inputs: read before the wait
        const int b = (int)(row / p.hq);
        np = use_plan ? __ldg(p.nparts + b) : (int)((__ldg(p.seq_len + b) + p.chunk - 1) / p.chunk);
    }
    // the partials are written by the decode kernels just before this one
    rx::pdl_wait();
    // > max_parts: flagged by the decode kernel; > FEW without MANY: not
    // launched for such rows (FEW is at least max_parts then)
    if (!live || np <= 1 || np > p.max_parts || (!MANY && np > FEW)) return;
    const float *lp = p.ws_lse + row * p.max_parts;
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] = 0.f;
    float m = -INFINITY, wsum = 0.f;
    if (np <= FEW) {
        // few parts: their rows and log2-sum-exps are loaded together (one
        // round trip to L2), then weighted
        const float *src0 = p.ws_o + row * p.max_parts * D + lane * PER;
        float v[FEW][PER];
#pragma unroll
        for (int k = 0; k < FEW; ++k) {
            if (k < np) {
                if constexpr (PER == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(src0 + (int64_t)k * D);
                    v[k][0] = t.x;
                    v[k][1] = t.y;
                    v[k][2] = t.z;
                    v[k][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2 *>(src0 + (int64_t)k * D);
                    v[k][0] = t.x;
                    v[k][1] = t.y;
                }
            }
        }
        const float ll = lane < np ? lp[lane] : -INFINITY;
        m = ll;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float wl = lane < np ? rx::fast_exp2(ll - m) : 0.f;
        wsum = wl;
#pragma unroll
        for (int k = 0; k < FEW; ++k) {
            const float wgt = __shfl_sync(0xffffffffu, wl, k);
            if (k < np)
#pragma unroll
                for (int j = 0; j < PER; ++j) acc[j] = fmaf(wgt, v[k][j], acc[j]);
        }
    } else if constexpr (!MANY) {
        // not reached: np <= FEW above
    } else if (np <= 2 * 32) {
        // up to 64 parts: every log2-sum-exp (two a lane) and the first 16
        // rows are loaded together; each later batch of 16 rows is loaded
        // before the previous one is weighted, so about np / 16 round trips
        // to L2 remain
        constexpr int NB = kMergeBatch;
        const float *src0 = p.ws_o + row * p.max_parts * D + lane * PER;
        auto load = [&](float (&v)[NB][PER], int base) {
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                if (base + k < np) {
                    const float *src = src0 + (int64_t)(base + k) * D;
                    if constexpr (PER == 4) {
                        const float4 t = *reinterpret_cast<const float4 *>(src);
                        v[k][0] = t.x;
                        v[k][1] = t.y;
                        v[k][2] = t.z;
                        v[k][3] = t.w;
                    } else {
                        const float2 t = *reinterpret_cast<const float2 *>(src);
                        v[k][0] = t.x;
                        v[k][1] = t.y;
                    }
                }
            }
        };
        float va[NB][PER], vb[NB][PER];
        const float l0 = lane < np ? lp[lane] : -INFINITY;
        const float l1 = lane + 32 < np ? lp[lane + 32] : -INFINITY;
        load(va, 0);
        m = fmaxf(l0, l1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float w0 = lane < np ? rx::fast_exp2(l0 - m) : 0.f;
        const float w1 = lane + 32 < np ? rx::fast_exp2(l1 - m) : 0.f;
        wsum = w0 + w1;
        auto weigh = [&](const float (&v)[NB][PER], int base) {
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                const int i = base + k;  // warp-uniform
                const float wgt = __shfl_sync(0xffffffffu, i < 32 ? w0 : w1, i & 31);
                if (i < np)
#pragma unroll
                    for (int j = 0; j < PER; ++j) acc[j] = fmaf(wgt, v[k][j], acc[j]);
            }
        };
        for (int base = 0; base < np; base += 2 * NB) {
            if (base + NB < np) load(vb, base + NB);
            weigh(va, base);
            if (base + NB >= np) break;
            if (base + 2 * NB < np) load(va, base + 2 * NB);
            weigh(vb, base + NB);
        }
    } else {
        for (int i = lane; i < np; i += 32) m = fmaxf(m, lp[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        // part weights computed lane-parallel (lane k: part base + k), then the
        // parts' rows read eight at a time so their loads are in flight together
        for (int base = 0; base < np; base += 32) {
            const int cnt = min(32, np - base);
            const float wl = lane < cnt ? rx::fast_exp2(lp[base + lane] - m) : 0.f;
            wsum += wl;
            const float *src0 = p.ws_o + (row * p.max_parts + base) * D + lane * PER;
#pragma unroll 8
            for (int k = 0; k < cnt; ++k) {
                const float wgt = __shfl_sync(0xffffffffu, wl, k);
                const float *src = src0 + (int64_t)k * D;
                if constexpr (PER == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    acc[0] = fmaf(wgt, v.x, acc[0]);
                    acc[1] = fmaf(wgt, v.y, acc[1]);
                    acc[2] = fmaf(wgt, v.z, acc[2]);
                    acc[3] = fmaf(wgt, v.w, acc[3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[0] = fmaf(wgt, v.x, acc[0]);
                    acc[1] = fmaf(wgt, v.y, acc[1]);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    // every lane's loads of the parts have been used: their L2 lines (whole
    // 128-byte lines, D * 4 bytes a part) are dropped without a write-back
    __syncwarp();
    {
        constexpr int LPP = D * 4 / 128;  // lines a part
        const char *base = reinterpret_cast<const char *>(p.ws_o + row * p.max_parts * D);
        for (int li = lane; li < np * LPP; li += 32) rx::discard_l2(base + (int64_t)li * 128);
    }
    const float inv = 1.f / wsum;
    bf16 *dst = p.o + row * D + lane * PER;
#pragma unroll
    for (int j = 0; j < PER; j += 2)
        *reinterpret_cast<uint32_t *>(dst + j) = rx::pack_bf16(acc[j] * inv, acc[j + 1] * inv);
    if (p.lse && lane == 0) p.lse[row] = (m + log2f(wsum)) * rx::kLn2;
}

int num_sms()
{
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 148;
    }
    return sms;
}

// ---------------------------------------------------------------------------
// wide items: one request, every kv head at once
// ---------------------------------------------------------------------------
//
// A plan item that holds a single request covers positions nobody else reads
// (a private tail), with one query row per q head.  Its K (and V) rows for all
// kv heads of a slot are contiguous in the pool (num_kv_heads * head_dim * 2
// bytes: 8 KiB for 32 x 128), and on GB300 a random gather of whole slot rows
// streams at HBM speed where a gather of 256-byte rows per kv head does not
// (measured: 8 KiB rows 6.8 TB/s, 2 KiB rows 4.4 TB/s, 256-byte rows 2.9
// TB/s).  So these items go to this kernel:
//   - one producer warp moves whole slot rows, one bulk copy (TMA engine) per
//     row, into a ring of stages whose full barrier counts the bytes;
//   - eight consumer warps each own hq / 8 q heads, with q (pre-scaled into
//     the exp2 domain) and the running o in registers, D / 32 values per
//     lane; one query row per head makes the work a matrix-vector product,
//     about one flop per byte, so it runs on the CUDA cores: per head and
//     position a lane-split dot product, a warp all-reduce and an online
//     softmax step.

constexpr int kWideStages = 3;
constexpr int kWideStageBytes = 32768;  // K bytes per stage (as many again for V)
constexpr int kWideMaxPos = 32;         // positions per stage at most (one producer lane each)

// Shared-memory layout of an all-heads kernel: STAGES ring entries of K
// (and as many of V) rows, per-stage row flags, slot ids and headers, NQ
// query-row slots, then the barriers: full [STAGES], empty [STAGES], q_empty
// [NQ], desc [STAGES] (a stage's slot ids are written: the copy warps may
// start).
template <int STAGES_, int STAGE_BYTES_, int NQ_, int QBYTES_>
struct WideLayoutT {
    static constexpr int STAGES = STAGES_, STAGE_BYTES = STAGE_BYTES_, NQ = NQ_;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = STAGES * STAGE_BYTES;
    static constexpr int OFF_OK = 2 * STAGES * STAGE_BYTES;               // int [stage][pos]: row valid
    static constexpr int OFF_SLOT = OFF_OK + STAGES * kWideMaxPos * 4;    // int [stage][pos]: slot id or -1
    static constexpr int OFF_HDR = OFF_SLOT + STAGES * kWideMaxPos * 4;   // int4 [stage]: item, first
                                                                          // position, item end, requests
    static constexpr int OFF_Q = (OFF_HDR + STAGES * 16 + 127) / 128 * 128;  // NQ x the item's query rows
    static constexpr int QBYTES = QBYTES_;                                // bytes of one q slot
    static constexpr int OFF_BAR = OFF_Q + NQ * QBYTES;
    static constexpr int OFF_ABORT = OFF_BAR + (3 * STAGES + NQ) * 8;
    static constexpr int B_DESC = 2 * STAGES + NQ;  // first desc barrier
    static constexpr int BYTES = OFF_ABORT + 16 + 128;  // + room to align the base to 128
    static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
    static_assert(BYTES <= 227 * 1024, "shared memory budget");
    // bulk copies land on 16-byte boundaries: stage bases, rows (16-byte
    // multiples from a stage base) and the q slots
    static_assert(STAGE_BYTES % 128 == 0 && OFF_V % 128 == 0 && OFF_Q % 128 == 0 && QBYTES % 128 == 0,
                  "bulk-copy destination alignment");
};
// one q head per kv head: slot rows packed (32 KB of K a stage), two q slots
// of one request's query row (hq * D * 2 bytes, 16 KB at most)
using WideLayout = WideLayoutT<kWideStages, kWideStageBytes, 2, 16384>;

// bounded single-thread wait that ignores the abort flag: lets copies already
// issued land before the CTA exits
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t *status)
{
    const long long t0 = clock64();
    do {
        if (rx::mbar_try_wait(bar, parity)) return;
    } while (clock64() - t0 < rx::kWaitCycles);
    if (status) atomicOr(status, RX_DEV_TIMEOUT);
}

// E consecutive bf16 of shared memory as floats (E = 2, 4, 8 or 16: one 4-,
// 8- or 16-byte load, or two 16-byte loads)
template <int E>
__device__ __forceinline__ void load_bf16(const unsigned char *src, float (&out)[E])
{
    if constexpr (E == 8 || E == 16) {
#pragma unroll
        for (int c = 0; c < E / 8; ++c) {
            const uint4 r = *reinterpret_cast<const uint4 *>(src + 16 * c);
            const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
                out[8 * c + 2 * k] = f.x;
                out[8 * c + 2 * k + 1] = f.y;
            }
        }
    } else if constexpr (E == 4) {
        const uint2 r = *reinterpret_cast<const uint2 *>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
        out[0] = a.x;
        out[1] = a.y;
        out[2] = b.x;
        out[3] = b.y;
    } else {
        const uint32_t r = *reinterpret_cast<const uint32_t *>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r));
        out[0] = a.x;
        out[1] = a.y;
    }
}

// E consecutive E4M3 codes of shared memory as floats (E = 2, 4, 8 or 16:
// one 2-, 4-, 8- or 16-byte load); exact, through f16.
template <int E>
__device__ __forceinline__ void load_e4m3(const unsigned char *src, float (&out)[E])
{
    uint32_t w[E >= 4 ? E / 4 : 1];
    if constexpr (E == 16) {
        const uint4 r = *reinterpret_cast<const uint4 *>(src);
        w[0] = r.x;
        w[1] = r.y;
        w[2] = r.z;
        w[3] = r.w;
    } else if constexpr (E == 8) {
        const uint2 r = *reinterpret_cast<const uint2 *>(src);
        w[0] = r.x;
        w[1] = r.y;
    } else if constexpr (E == 4) {
        w[0] = *reinterpret_cast<const uint32_t *>(src);
    } else {
        w[0] = *reinterpret_cast<const uint16_t *>(src);
    }
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        const uint32_t h = rx::e4m3x2_to_f16x2((uint16_t)(w[k >> 1] >> (16 * (k & 1))));
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
        out[2 * k] = f.x;
        out[2 * k + 1] = f.y;
    }
}

// Producer warp of an all-heads kernel (layout WL, NP positions a stage,
// one lane per position; GROUPS: items may hold up to 16 / G requests,
// else one).  Items come from a global counter, first come
// first served, so a CTA that starts late (behind the per-head kernel
// running alongside) takes fewer of them.  Each stage's header names its
// item; a last header with item -1 tells the consumers to stop.  A stage's
// rows sit row_stride bytes apart (row bytes RB = hkv * head_dim * 2).
template <class WL, int NP, int NH, bool GROUPS>
__device__ void wide_producer(const Params &p, unsigned char *smem, uint32_t sbase, volatile int *abort_flag,
                              int row_stride)
{
    const uint32_t bar = sbase + WL::OFF_BAR;
    int *okf = reinterpret_cast<int *>(smem + WL::OFF_OK);
    int *slotf = reinterpret_cast<int *>(smem + WL::OFF_SLOT);
    const int lane = threadIdx.x & 31;
    const int RB = (int)p.row_bytes;
    // Under load a global load takes microseconds, so nothing on the copy
    // path waits for one: a cursor runs three stages ahead of the stage
    // being issued, and its loads (at an item boundary: the claim, the
    // item's fields, then slot ids) are made before the wait for a free
    // stage.  Claims stay only a few stages ahead of their first copy, so
    // the queue still hands the last items to the CTAs that free up first.
    struct Cursor {
        int it, q0, p1, nr, qb;   // qb: batch index of the item's request `lane`
        const int32_t *slots;
    };
    auto fetch = [&]() -> int {
        int it = 0;
        if (lane == 0) it = atomicAdd(p.wide_counter, 1);
        return __shfl_sync(0xffffffffu, it, 0);
    };
    auto open_item = [&](Cursor &c, int it) {
        c.it = it;
        if (it < p.n_wide) {
            const int32_t *v = p.items + 8 * (int64_t)(p.wide0 + it);
            c.q0 = __ldg(v + 2);
            c.p1 = __ldg(v + 3);
            if (c.p1 == RX_PLAN_OPEN_END) c.p1 = open_end(p, __ldg(v + 7), c.q0, lane == 0);
            c.slots = p.rtt + (int64_t)__ldg(v + 6) * p.rtt_stride;
            int nr = __ldg(v + 1);
            // a malformed item (more requests than the kernel's rows, or
            // none) is flagged and read as its first request alone
            if (nr < 1 || (GROUPS ? nr * p.G > 16 : nr != 1)) {
                if (lane == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_LEN);
                nr = 1;
            }
            c.nr = nr;
            c.qb = lane == 0 ? __ldg(v + 7) : (lane < nr ? __ldg(p.order + __ldg(v) + lane) : 0);
        }
    };
    auto advance = [&](Cursor &c) {
        if (c.it >= p.n_wide) return;  // past the end: stays there
        c.q0 += NP;
        if (c.q0 >= c.p1) open_item(c, fetch());
    };
    auto slot_of = [&](const Cursor &c) -> int32_t {
        const int pos = c.q0 + lane;
        return (c.it < p.n_wide && lane < NP && pos < c.p1) ? __ldg(c.slots + pos) : -1;
    };
    int4 *hdr = reinterpret_cast<int4 *>(smem + WL::OFF_HDR);
    const uint32_t qbytes = (uint32_t)(p.hq * p.head_dim * 2);
    Cursor c0{}, c1, c2, c3;
    open_item(c0, fetch());
    int32_t s0 = slot_of(c0);
    c1 = c0;
    advance(c1);
    int32_t s1 = slot_of(c1);
    c2 = c1;
    advance(c2);
    int32_t s2 = slot_of(c2);
    c3 = c2;
    advance(c3);
    int32_t s3 = slot_of(c3);
    int j = 0, n_items = 0;   // items opened so far; item k uses q slot k % NQ
    int prev_it = -1;
    for (;; ++j) {
        const bool end = c0.it >= p.n_wide;
        const int st = j % WL::STAGES;
        if (j >= WL::STAGES &&
            !wait_or_abort(bar + 8 * (WL::STAGES + st), ((j / WL::STAGES) - 1) & 1, abort_flag, p.status, p.wait_cycles))
            break;
        // an item's first stage also brings its query row into q slot
        // k % NQ, once the consumers have read item k - NQ's out of it
        const bool with_q = !end && c0.it != prev_it;
        const int qb = n_items % WL::NQ;
        if (with_q && n_items >= WL::NQ &&
            !wait_or_abort(bar + 8 * (2 * WL::STAGES + qb), ((n_items / WL::NQ) - 1) & 1, abort_flag,
                           p.status, p.wait_cycles))
            break;
        const bool inside = !end && lane < NP && c0.q0 + lane < c0.p1;
        const bool ok = inside && s0 >= 0 && (int64_t)s0 < p.num_slots;
        if (inside && !ok && p.status) atomicOr(p.status, RX_DEV_BAD_SLOT);
        if (lane < NP) {
            okf[st * kWideMaxPos + lane] = ok ? 1 : 0;
            slotf[st * kWideMaxPos + lane] = ok ? s0 : -1;
        }
        if (lane == 0) hdr[st] = make_int4(end ? -1 : c0.it, c0.q0, c0.p1, end ? 0 : c0.nr);
        const int nok = __popc(__ballot_sync(0xffffffffu, ok));
        __syncwarp();  // flags and header are written before lane 0's arrive releases them
        if (lane == 0)
            rx::mbar_arrive_expect_tx(bar + 8 * st,
                                      (uint32_t)(2 * nok * RB) + (with_q ? (uint32_t)c0.nr * qbytes : 0u));
        __syncwarp();
        // the query rows of the item's requests, one after another in the slot
        if (with_q && lane < c0.nr)
            rx::bulk_g2s(sbase + WL::OFF_Q + qb * WL::QBYTES + lane * qbytes,
                         p.q + (int64_t)c0.qb * p.hq * p.head_dim, qbytes, bar + 8 * st);
        if (with_q) ++n_items;
        if constexpr (NH > 0) {
            // the copy warps issue this stage's row copies (issuing bulk
            // copies costs each warp tens of nanoseconds apiece)
            if (lane == 0) rx::mbar_arrive(bar + 8 * (WL::B_DESC + st));
        } else if (ok) {
            // a single request's rows are read once: first out of L2
            const uint64_t pol = c0.nr == 1 ? rx::l2_evict_first() : rx::l2_evict_normal();
            const uint32_t off = (uint32_t)(st * WL::STAGE_BYTES + lane * row_stride);
            rx::bulk_g2s_hint(sbase + WL::OFF_K + off, p.kb + (int64_t)s0 * p.row_bytes, (uint32_t)RB, bar + 8 * st,
                              pol);
            rx::bulk_g2s_hint(sbase + WL::OFF_V + off, p.vb + (int64_t)s0 * p.row_bytes, (uint32_t)RB, bar + 8 * st,
                              pol);
        }
        if (end) {
            ++j;
            break;
        }
        prev_it = c0.it;
        // shift the lookahead; the new far cursor's loads are in flight
        // while the next stage waits to be free
        c0 = c1;
        s0 = s1;
        c1 = c2;
        s1 = s2;
        c2 = c3;
        s2 = s3;
        advance(c3);
        s3 = slot_of(c3);
    }
    // no copy may still be landing when the CTA exits
    if (lane == 0)
        for (int jj = j > WL::STAGES ? j - WL::STAGES : 0; jj < j; ++jj)
            drain_wait(bar + 8 * (jj % WL::STAGES), (jj / WL::STAGES) & 1, p.status);
    __syncwarp();
}

// Copy warp h of NH of an all-heads kernel: for every stage the producer
// described, issues the K and V row copies of positions h, h + NH, ... (one
// lane each) onto the stage's full barrier.  It stops at the stage whose
// header holds no item; the producer's drain covers its copies.  Rows of a
// single-request item (a request's own positions, read by nothing else in
// the call) are fetched evict-first, so that they do not push out of L2 the
// rows a request group re-reads or the partial results the merge reads back.
template <class WL, int NP, int NH>
__device__ void wide_copier(const Params &p, unsigned char *smem, uint32_t sbase, volatile int *abort_flag,
                            int row_stride, int h)
{
    const uint32_t bar = sbase + WL::OFF_BAR;
    const int *slotf = reinterpret_cast<const int *>(smem + WL::OFF_SLOT);
    const int4 *hdr = reinterpret_cast<const int4 *>(smem + WL::OFF_HDR);
    const int lane = threadIdx.x & 31;
    const uint32_t RB = (uint32_t)p.row_bytes;
    const int pos = lane * NH + h;
    const uint64_t once = rx::l2_evict_first(), shared = rx::l2_evict_normal();
    for (int j = 0;; ++j) {
        const int st = j % WL::STAGES;
        if (!wait_or_abort(bar + 8 * (WL::B_DESC + st), (j / WL::STAGES) & 1, abort_flag, p.status, p.wait_cycles)) return;
        const int4 h4 = hdr[st];
        if (h4.x < 0) return;
        const int s = pos < NP ? slotf[st * kWideMaxPos + pos] : -1;
        if (s >= 0) {
            const uint64_t pol = h4.w == 1 ? once : shared;
            const uint32_t off = (uint32_t)(st * WL::STAGE_BYTES + pos * row_stride);
            rx::bulk_g2s_hint(sbase + WL::OFF_K + off, p.kb + (int64_t)s * p.row_bytes, RB, bar + 8 * st, pol);
            rx::bulk_g2s_hint(sbase + WL::OFF_V + off, p.vb + (int64_t)s * p.row_bytes, RB, bar + 8 * st, pol);
        }
    }
}

constexpr int kWideCopyWarps = 2;  // copy warps of the one-q-head-per-kv-head kernel

// F8: the pools hold E4M3 codes (one byte a value, so twice the positions a
// stage); the consumers widen them to floats exactly as they load them, K's
// scale is in scale_log2 and V's multiplies the output.
template <int D, int LOG_NP, int HPW, int CW, bool F8>
__global__ void __launch_bounds__(32 * (1 + kWideCopyWarps + CW), 1) decode_wide_kernel(const Params p)
{
    using WL = WideLayout;
    constexpr int NP = 1 << LOG_NP;  // positions per stage
    extern __shared__ __align__(128) unsigned char wraw[];
    const uint32_t raw = rx::smem_u32(wraw);
    unsigned char *smem = wraw + (((raw + 127u) & ~127u) - raw);
    const uint32_t sbase = rx::smem_u32(smem);
    const uint32_t bar = sbase + WL::OFF_BAR;  // full: [0, S), empty: [S, 2S)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + WL::OFF_ABORT);
    int *okf = reinterpret_cast<int *>(smem + WL::OFF_OK);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = (int)p.row_bytes;       // bytes of one slot row (hkv * D values)
    constexpr int EB = F8 ? 1 : 2;         // bytes a value
    // runs beside the per-head kernel (it reads none of that kernel's
    // results) and ends after it; the merge may be launched at once
    rx::PdlWaitOnExit ends_after_per_head;
    rx::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kWideStages; ++i) {
            rx::mbar_init(bar + 8 * i, 1);                                  // producer + bytes
            rx::mbar_init(bar + 8 * (kWideStages + i), CW);                 // consumer warps
        }
        for (int i = 0; i < 2; ++i) rx::mbar_init(bar + 8 * (2 * kWideStages + i), CW);  // q slot read
        for (int i = 0; i < kWideStages; ++i) rx::mbar_init(bar + 8 * (WL::B_DESC + i), 1);  // producer
        *abort_flag = 0;
        rx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        wide_producer<WL, NP, kWideCopyWarps, false>(p, smem, sbase, abort_flag, RB);
    } else if (warp <= kWideCopyWarps) {
        wide_copier<WL, NP, kWideCopyWarps>(p, smem, sbase, abort_flag, RB, warp - 1);
    } else {
        // consumers: warp cw owns q heads (= kv heads, G == 1) h0 .. h0 + HPW - 1.
        // A stage is taken in sub-stages of NPS positions: eight (head,
        // position) pairs, four lanes each.  Lane l serves pair x = l / 4
        // (head hh = x / NPS, position pi = x % NPS) and quarter qd = l % 4 of
        // its dot product, DQ dims; the quarters meet in two shuffles, and max
        // and sum over a head's positions take LOG_NPS shuffles each, so the
        // chain of dependent shuffles per sub-stage stays short.  For P.V the
        // 32 / HPW lanes of a head each own DO consecutive output dims.
        constexpr int LOG_HPW = HPW == 1 ? 0 : HPW == 2 ? 1 : 2;
        constexpr int LOG_NPS = LOG_NP + LOG_HPW <= 3 ? LOG_NP : 3 - LOG_HPW;
        constexpr int NPS = 1 << LOG_NPS;
        static_assert(HPW * NPS == 8 && NP % NPS == 0, "eight (head, position) pairs per sub-stage");
        constexpr int DQ = D / 4;          // dims of a lane's quarter of a dot product
        constexpr int NCH = DQ / 8;        // its 16-byte chunks (4 at d 128, 2 at d 64)
        constexpr int DO = D * HPW / 32;   // output dims per lane
        static_assert(NCH == 2 || NCH == 4, "quarter of 2 or 4 chunks");
        static_assert(DO % 2 == 0, "output dims stored in pairs");
        const int cw = warp - 1 - kWideCopyWarps;
        const int h0 = cw * HPW;
        const int x = lane >> 2, qd = lane & 3;
        const int hh = x >> LOG_NPS, pi = x & (NPS - 1);
        const int hl = lane & (32 / HPW - 1);  // lane within its head's lanes
        const int head = h0 + hh;
        // chunk c of a quarter is read at rotated position cc(c), so that the
        // eight lanes of each 16-byte load phase hit distinct bank groups
        auto chunk_at = [&](int c) -> int {
            return NCH == 4 ? ((c + (qd >> 1) + 2 * (x & 1)) & 3) : ((c + (x & 1)) & 1);
        };
        const int4 *hdr = reinterpret_cast<const int4 *>(smem + WL::OFF_HDR);
        float q[NCH][8], o[DO], m = -INFINITY, l = 0.f;
        int cur = -1, p1 = 0, part_idx = 0, b = 0, n_items = 0;
        bool fin = false;
        // the current item's result for this lane's head
        auto write_out = [&]() {
            const int64_t orow = (int64_t)b * p.hq + head;
            const float inv = p.v_scale / l;  // V's scale: 1 for a bf16 pool
            if (fin) {
                bf16 *dst = p.o + orow * D + hl * DO;
#pragma unroll
                for (int e = 0; e < DO; e += 2)
                    *reinterpret_cast<uint32_t *>(dst + e) = rx::pack_bf16(o[e] * inv, o[e + 1] * inv);
                if (p.lse && hl == 0) p.lse[orow] = (m + log2f(l)) * rx::kLn2;
            } else {
                const int64_t prow = orow * p.max_parts + part_idx;
                float *dst = p.ws_o + prow * D + hl * DO;
                const uint64_t keep = rx::l2_evict_last();  // the merge reads them back, then discards the lines
#pragma unroll
                for (int e = 0; e < DO; e += 2) rx::st_hint(dst + e, o[e] * inv, o[e + 1] * inv, keep);
                if (hl == 0) p.ws_lse[prow] = m + log2f(l);
            }
        };
        for (int j = 0;; ++j) {
            const int st = j % kWideStages;
            if (!wait_or_abort(bar + 8 * st, (j / kWideStages) & 1, abort_flag, p.status, p.wait_cycles)) return;
            const int4 h = hdr[st];
            // a new item starts, or (item -1) none is left -- possibly before
            // this CTA got any, when the other CTAs drained the queue first
            if (h.x != cur || h.x < 0) {
                if (cur >= 0) write_out();
                if (h.x < 0) break;
                cur = h.x;
                const int32_t *v = p.items + 8 * (int64_t)(p.wide0 + cur);
                p1 = h.z;   // the item's end as the producer resolved it
                part_idx = __ldg(v + 4);
                fin = __ldg(v + 5) != 0;
                b = __ldg(v + 7);
                // the query row came with this stage: read this lane's quarter
                // of its head (in the rotated chunk order), then hand the q
                // slot back
                const int qb = n_items & 1;
                const unsigned char *qs = smem + WL::OFF_Q + qb * WL::QBYTES + head * D * 2 + qd * DQ * 2;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    load_bf16<8>(qs + 16 * chunk_at(c), q[c]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) q[c][e] *= p.scale_log2;
                }
#pragma unroll
                for (int e = 0; e < DO; ++e) o[e] = 0.f;
                m = -INFINITY;
                l = 0.f;
                __syncwarp();
                if (lane == 0) rx::mbar_arrive(bar + 8 * (2 * kWideStages + qb));
                ++n_items;
            }
            const int n = min(NP, p1 - h.y);  // positions of the item in this stage
            const int *okp = okf + st * kWideMaxPos;
            for (int sub = 0; sub * NPS < n; ++sub) {
                const int ns = min(NPS, n - sub * NPS);
                const unsigned char *kst = smem + WL::OFF_K + st * kWideStageBytes + sub * NPS * RB;
                const unsigned char *vst = smem + WL::OFF_V + st * kWideStageBytes + sub * NPS * RB;
                // bit i: position i of the sub-stage holds a valid row
                uint32_t vmask = 0;
#pragma unroll
                for (int i = 0; i < NPS; ++i) vmask |= (i < ns && okp[sub * NPS + i] != 0) ? (1u << i) : 0u;
                // this lane's quarter of the dot product of its pair
                const unsigned char *kr = kst + pi * RB + head * D * EB + qd * DQ * EB;
                float sc = 0.f;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    float kf[8];
                    if constexpr (F8)
                        load_e4m3<8>(kr + 8 * chunk_at(c), kf);
                    else
                        load_bf16<8>(kr + 16 * chunk_at(c), kf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) sc = fmaf(q[c][e], kf[e], sc);
                }
                sc += __shfl_xor_sync(0xffffffffu, sc, 1);
                sc += __shfl_xor_sync(0xffffffffu, sc, 2);
                // a position past the item is out; a row with an invalid slot reads as zeros
                const bool okx = (vmask >> pi) & 1u;
                sc = pi < ns ? (okx ? sc : 0.f) : -INFINITY;
                float smax = sc;
#pragma unroll
                for (int k = 0; k < LOG_NPS; ++k) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 4 << k));
                const float mn = fmaxf(m, smax);
                const float pw = rx::fast_exp2(sc - mn);  // 0 past the item
                float ps = pw;
#pragma unroll
                for (int k = 0; k < LOG_NPS; ++k) ps += __shfl_xor_sync(0xffffffffu, ps, 4 << k);
                const float al = rx::fast_exp2(m - mn);   // 0 on the item's first sub-stage
                m = mn;
                l = fmaf(l, al, ps);
#pragma unroll
                for (int e = 0; e < DO; ++e) o[e] *= al;
                const float pv = okx ? pw : 0.f;  // weight of this lane's pair for V
                const unsigned char *vr = vst + head * D * EB + hl * DO * EB;
#pragma unroll
                for (int i = 0; i < NPS; ++i) {
                    const float w = __shfl_sync(0xffffffffu, pv, ((hh << LOG_NPS) + i) << 2);
                    // rows past the item or with an invalid slot were never
                    // written in this stage: skip them (0 * stale NaN is NaN)
                    if (!((vmask >> i) & 1u)) continue;
                    float vf[DO];
                    if constexpr (F8)
                        load_e4m3<DO>(vr + i * RB, vf);
                    else
                        load_bf16<DO>(vr + i * RB, vf);
#pragma unroll
                    for (int e = 0; e < DO; ++e) o[e] = fmaf(w, vf[e], o[e]);
                }
            }
            __syncwarp();
            if (lane == 0) rx::mbar_arrive(bar + 8 * (kWideStages + st));
        }
    }
}

// ---------------------------------------------------------------------------
// single-request items with several q heads per kv head
// ---------------------------------------------------------------------------
//
// With G = hq / hkv > 1 a kv head's K row meets G query rows, so the work per
// byte is G times that of G == 1 and belongs on the tensor cores.  This
// kernel keeps the all-heads data path (whole slot rows, 2 KiB at 8 x 128,
// one bulk copy each, from the same producer) and gives each of the eight kv
// heads one consumer warp that runs mma.sync m16n8k16 on them: the G query
// rows of the kv head, padded to 16, against 16 positions a stage.
//   - rows sit at a stride of 2048 + 16 bytes, so the eight rows an ldmatrix
//     reads fall in distinct banks;
//   - bulk copies cannot zero-fill, so V rows of positions past the item or
//     with an invalid slot id are zeroed in the mma operands instead (a
//     probability of 0 times a stale NaN would still be NaN); their scores
//     are -inf past the item and 0 for an invalid slot (a zero K row).

constexpr int kGqaNP = 16;                         // positions per stage
constexpr int kGqaRowStride = 2048 + 16;           // slot row (8 kv heads x 128 x 2 at most) + pad
// one q slot: the query rows of an item's requests (up to 16 / G of them,
// 16 * 8 * D * 2 bytes at most)
using GqaLayout = WideLayoutT<3, kGqaNP * kGqaRowStride, 1, 32768>;
constexpr int kGqaWarps = 8;                       // one consumer warp per kv head
constexpr int kGqaCopyWarps = 2;                   // copy warps: 32 row copies a stage
// FP8 (E4M3) pools: slot rows of one byte a value (1 KiB at 8 x 128), the
// same q slot, and per consumer warp an f16 copy of its kv head's V rows of
// the stage (16 rows of D halves + a 16-byte pad, for conflict-free
// ldmatrix), placed after the layout
constexpr int kGqaRowStride8 = 1024 + 16;
using GqaLayout8 = WideLayoutT<3, kGqaNP * kGqaRowStride8, 1, 32768>;
__host__ __device__ constexpr int gqa8_scratch_off() { return (GqaLayout8::OFF_ABORT + 16 + 127) / 128 * 128; }
template <int D>
__host__ __device__ constexpr int gqa8_scratch_rs() { return D * 2 + 16; }
template <int D>
__host__ __device__ constexpr int gqa8_bytes()
{
    return gqa8_scratch_off() + kGqaWarps * kGqaNP * gqa8_scratch_rs<D>() + 128;
}
static_assert(gqa8_bytes<128>() <= 227 * 1024, "shared memory budget");

// F8: the pools hold E4M3 codes (rx_attn_decode_fp8).  The MMAs then run on
// f16 operands: codes widen to f16 exactly, q converts exactly within f16's
// range, and P rounds to f16.  K fragments are built straight from the code
// rows: with the 16 dims of a k-step permuted so that lane group tig takes
// dims 4 tig .. 4 tig + 3 (a dot product does not depend on the order of
// its terms; q's fragments use the same order), one 4-byte load gives both
// B registers.  V rows are widened into the warp's f16 scratch first, then
// read with ldmatrix.trans as on the bf16 path.  K's scale is in
// scale_log2, V's multiplies the output.
template <int D, bool F8>
__global__ void __launch_bounds__(32 * (1 + kGqaCopyWarps + kGqaWarps), 1) decode_gqa_kernel(const Params p)
{
    using WL = std::conditional_t<F8, GqaLayout8, GqaLayout>;
    constexpr int RS = F8 ? kGqaRowStride8 : kGqaRowStride;  // slot row stride in a stage
    constexpr int KS = D / 16;   // k-steps of S = Q K^T
    constexpr int DT = D / 8;    // n-tiles of O
    extern __shared__ __align__(128) unsigned char graw[];
    const uint32_t raw = rx::smem_u32(graw);
    unsigned char *smem = graw + (((raw + 127u) & ~127u) - raw);
    const uint32_t sbase = rx::smem_u32(smem);
    const uint32_t bar = sbase + WL::OFF_BAR;  // full: [0, S), empty: [S, 2S), q_empty: [2S]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + WL::OFF_ABORT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    rx::PdlWaitOnExit ends_after_per_head;  // as in the one-q-head kernel
    rx::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < WL::STAGES; ++i) {
            rx::mbar_init(bar + 8 * i, 1);                          // producer + bytes
            rx::mbar_init(bar + 8 * (WL::STAGES + i), kGqaWarps);   // consumer warps
        }
        rx::mbar_init(bar + 8 * (2 * WL::STAGES), kGqaWarps);       // q slot read
        for (int i = 0; i < WL::STAGES; ++i) rx::mbar_init(bar + 8 * (WL::B_DESC + i), 1);  // producer
        *abort_flag = 0;
        rx::fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        wide_producer<WL, kGqaNP, kGqaCopyWarps, true>(p, smem, sbase, abort_flag, RS);
        return;
    }
    if (warp <= kGqaCopyWarps) {
        wide_copier<WL, kGqaNP, kGqaCopyWarps>(p, smem, sbase, abort_flag, RS, warp - 1);
        return;
    }
    // consumer warp: kv head g.  Row m = i * G + j of its m16 tile is q head
    // g * G + j of the item's request i (M = requests x G rows, 16 at most).
    const int g = warp - 1 - kGqaCopyWarps;
    const int G = p.G;
    const int gid = lane >> 2, tig = lane & 3;
    const int4 *hdr = reinterpret_cast<const int4 *>(smem + WL::OFF_HDR);
    const int *okf = reinterpret_cast<const int *>(smem + WL::OFF_OK);
    uint32_t qf[KS][4];
    float oacc[DT][4], m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    int cur = -1, p1 = 0, part_idx = 0, M = 0;
    int ob[2] = {0, 0};  // batch index of this thread's output rows gid, gid + 8
    bool fin = false;
    auto write_out = [&]() {
        float l0 = l_r[0], l1 = l_r[1];
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        const float ls[2] = {l0, l1};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = gid + half * 8;
            if (r >= M) continue;
            const int64_t orow = (int64_t)ob[half] * p.hq + (int64_t)g * G + r % G;
            const float inv = F8 ? p.v_scale / ls[half] : 1.f / ls[half];
            if (fin) {
                bf16 *dst = p.o + orow * D;
#pragma unroll
                for (int dt = 0; dt < DT; ++dt)
                    *reinterpret_cast<uint32_t *>(dst + dt * 8 + tig * 2) =
                        rx::pack_bf16(oacc[dt][2 * half] * inv, oacc[dt][2 * half + 1] * inv);
                if (p.lse && tig == 0) p.lse[orow] = (m_r[half] + log2f(ls[half])) * rx::kLn2;
            } else {
                const int64_t prow = orow * p.max_parts + part_idx;
                float *dst = p.ws_o + prow * D;
                const uint64_t keep = rx::l2_evict_last();  // the merge reads them back, then discards the lines
#pragma unroll
                for (int dt = 0; dt < DT; ++dt)
                    rx::st_hint(dst + dt * 8 + tig * 2, oacc[dt][2 * half] * inv, oacc[dt][2 * half + 1] * inv, keep);
                if (tig == 0) p.ws_lse[prow] = m_r[half] + log2f(ls[half]);
            }
        }
    };
    for (int j = 0;; ++j) {
        const int st = j % WL::STAGES;
        if (!wait_or_abort(bar + 8 * st, (j / WL::STAGES) & 1, abort_flag, p.status, p.wait_cycles)) return;
        const int4 h = hdr[st];
        // a new item starts, or (item -1) none is left -- possibly before
        // this CTA got any, when the other CTAs drained the queue first
        if (h.x != cur || h.x < 0) {
            if (cur >= 0) write_out();
            if (h.x < 0) break;
            cur = h.x;
            const int32_t *v = p.items + 8 * (int64_t)(p.wide0 + cur);
            const int r0 = __ldg(v + 0);
            int nr = __ldg(v + 1);
            if (nr < 1 || nr * G > 16) nr = 1;  // flagged by the producer, which copied one row
            M = nr * G;
            p1 = h.z;   // the item's end as the producer resolved it
            part_idx = __ldg(v + 4);
            fin = __ldg(v + 5) != 0;
            const int b0 = __ldg(v + 7);
            // batch indices of the two output rows: loaded now, used when
            // the item's last stage is done
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int i = (gid + half * 8) / G;
                ob[half] = (i == 0 || i >= nr) ? b0 : __ldg(p.order + r0 + i);
            }
            // the query rows came with this stage: A fragments of rows
            // 0 .. M - 1 (rows past M read row 0 and are zeroed), then hand
            // the q slot back
            if constexpr (F8) {
                // rows gid and gid + 8, dims 4 tig .. 4 tig + 3 of every
                // k-step (the permuted order), bf16 -> f16
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = gid + half * 8;
                    const int qm = r < M ? r : 0;
                    const unsigned char *qs =
                        smem + WL::OFF_Q + (size_t)(qm / G) * p.hq * D * 2 + (size_t)(g * G + qm % G) * D * 2;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(qs + (ks * 16 + 4 * tig) * 2);
                        const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
                        const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
                        qf[ks][half] = r < M ? rx::pack_f16(x01.x, x01.y) : 0u;
                        qf[ks][half + 2] = r < M ? rx::pack_f16(x23.x, x23.y) : 0u;
                    }
                }
            } else {
                const int qm = (lane & 15) < M ? (lane & 15) : 0;
                const unsigned char *qs =
                    smem + WL::OFF_Q + (size_t)(qm / G) * p.hq * D * 2 + (size_t)(g * G + qm % G) * D * 2;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int ch = ks * 2 + (lane >> 4);
                    rx::ldmatrix_x4(rx::smem_u32(qs + ch * 16), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
                    if (gid >= M) qf[ks][0] = qf[ks][2] = 0u;
                    if (gid + 8 >= M) qf[ks][1] = qf[ks][3] = 0u;
                }
            }
            __syncwarp();
            if (lane == 0) rx::mbar_arrive(bar + 8 * (2 * WL::STAGES));
            m_r[0] = m_r[1] = -INFINITY;
            l_r[0] = l_r[1] = 0.f;
#pragma unroll
            for (int dt = 0; dt < DT; ++dt) oacc[dt][0] = oacc[dt][1] = oacc[dt][2] = oacc[dt][3] = 0.f;
        }
        const int n = min(kGqaNP, p1 - h.y);  // positions of the item in this stage
        const int *okp = okf + st * kWideMaxPos;
        uint32_t vmask = 0;  // bit i: position i holds a valid row
#pragma unroll
        for (int i = 0; i < kGqaNP; ++i) vmask |= (i < n && okp[i] != 0) ? (1u << i) : 0u;
        constexpr int EB = F8 ? 1 : 2;  // bytes a value in the pools
        const unsigned char *kt = smem + WL::OFF_K + st * WL::STAGE_BYTES + g * D * EB;
        const unsigned char *vt = smem + WL::OFF_V + st * WL::STAGE_BYTES + g * D * EB;
        // S = Q K^T over the stage's 16 positions (two n-tiles)
        float sc[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
        if constexpr (F8) {
            // B of n-tile nt: position nt * 8 + gid, dims 4 tig .. 4 tig + 3
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t c4 = *reinterpret_cast<const uint32_t *>(kt + (nt * 8 + gid) * RS + ks * 16 + 4 * tig);
                    rx::mma_f16_16816(sc[nt], qf[ks], rx::e4m3x2_to_f16x2((uint16_t)(c4 & 0xffffu)),
                                      rx::e4m3x2_to_f16x2((uint16_t)(c4 >> 16)));
                }
        } else {
            const int key = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int ch = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4(rx::smem_u32(kt + key * kGqaRowStride + ch * 16), b0, b1, b2, b3);
                rx::mma_bf16_16816(sc[0], qf[ks], b0, b1);
                rx::mma_bf16_16816(sc[1], qf[ks], b2, b3);
            }
        }
        // scale into the exp2 domain; -inf past the item, 0 for an invalid slot
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int pos = nt * 8 + tig * 2 + (jj & 1);
                const float x = pos < n ? (((vmask >> pos) & 1u) ? sc[nt][jj] * p.scale_log2 : 0.f) : -INFINITY;
                sc[nt][jj] = x;
                if (jj < 2) mx0 = fmaxf(mx0, x);
                else mx1 = fmaxf(mx1, x);
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);  // finite: n >= 1
        const float a0 = rx::fast_exp2(m_r[0] - mn0), a1 = rx::fast_exp2(m_r[1] - mn1);
        m_r[0] = mn0;
        m_r[1] = mn1;
        l_r[0] *= a0;
        l_r[1] *= a1;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            oacc[dt][0] *= a0;
            oacc[dt][1] *= a0;
            oacc[dt][2] *= a1;
            oacc[dt][3] *= a1;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            sc[nt][0] = rx::fast_exp2(sc[nt][0] - mn0);
            sc[nt][1] = rx::fast_exp2(sc[nt][1] - mn0);
            sc[nt][2] = rx::fast_exp2(sc[nt][2] - mn1);
            sc[nt][3] = rx::fast_exp2(sc[nt][3] - mn1);
            l_r[0] += sc[nt][0] + sc[nt][1];
            l_r[1] += sc[nt][2] + sc[nt][3];
        }
        uint32_t a[4];
        if constexpr (F8) {
            a[0] = rx::pack_f16(sc[0][0], sc[0][1]);
            a[1] = rx::pack_f16(sc[0][2], sc[0][3]);
            a[2] = rx::pack_f16(sc[1][0], sc[1][1]);
            a[3] = rx::pack_f16(sc[1][2], sc[1][3]);
        } else {
            a[0] = rx::pack_bf16(sc[0][0], sc[0][1]);
            a[1] = rx::pack_bf16(sc[0][2], sc[0][3]);
            a[2] = rx::pack_bf16(sc[1][0], sc[1][1]);
            a[3] = rx::pack_bf16(sc[1][2], sc[1][3]);
        }
        // V rows of positions tig*2, tig*2+1 (b0, b2) and tig*2+8, +9 (b1, b3):
        // zero the ones that were never written in this stage
        const uint32_t vz0 = (((vmask >> (tig * 2)) & 1u) ? 0x0000ffffu : 0u) |
                             (((vmask >> (tig * 2 + 1)) & 1u) ? 0xffff0000u : 0u);
        const uint32_t vz1 = (((vmask >> (tig * 2 + 8)) & 1u) ? 0x0000ffffu : 0u) |
                             (((vmask >> (tig * 2 + 9)) & 1u) ? 0xffff0000u : 0u);
        if constexpr (F8) {
            // widen this kv head's 16 V rows into the warp's f16 scratch:
            // lane l takes half l & 1 of row l / 2 (D / 2 codes)
            unsigned char *scr = smem + gqa8_scratch_off() + (warp - 1 - kGqaCopyWarps) * kGqaNP * gqa8_scratch_rs<D>();
            {
                const int r = lane >> 1, c0 = (lane & 1) * (D / 2);
#pragma unroll
                for (int c = 0; c < D / 2; c += 16) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(vt + r * RS + c0 + c);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    uint32_t h[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        h[2 * k] = rx::e4m3x2_to_f16x2((uint16_t)(ws[k] & 0xffffu));
                        h[2 * k + 1] = rx::e4m3x2_to_f16x2((uint16_t)(ws[k] >> 16));
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(scr + r * gqa8_scratch_rs<D>() + (c0 + c) * 2);
                    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
                    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
            __syncwarp();
            const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int ch = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4_trans(rx::smem_u32(scr + key * gqa8_scratch_rs<D>() + ch * 16), b0, b1, b2, b3);
                b0 &= vz0;
                b1 &= vz1;
                b2 &= vz0;
                b3 &= vz1;
                rx::mma_f16_16816(oacc[2 * dp], a, b0, b1);
                rx::mma_f16_16816(oacc[2 * dp + 1], a, b2, b3);
            }
        } else {
            const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int ch = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4_trans(rx::smem_u32(vt + key * kGqaRowStride + ch * 16), b0, b1, b2, b3);
                b0 &= vz0;
                b1 &= vz1;
                b2 &= vz0;
                b3 &= vz1;
                rx::mma_bf16_16816(oacc[2 * dp], a, b0, b1);
                rx::mma_bf16_16816(oacc[2 * dp + 1], a, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) rx::mbar_arrive(bar + 8 * (WL::STAGES + st));
    }
}

// All-heads items with G > 1 (one request, or a group of up to 16 / G
// requests) go to decode_gqa_kernel for 8 kv heads and G = 2, 4, 8 or 16: a
// kv head's 16 query rows fit one m16 tile, and a group's query rows the q
// slot.
bool gqa_supported(int hq, int hkv, int D)
{
    return rx_gqa_heads(hq, hkv) && (D == 64 || D == 128) && 16 * hkv * D * 2 <= GqaLayout::QBYTES;
}

// Launches `kernel` on `st`.  With `dependent`, it is launched as a
// programmatic dependent of the kernel enqueued just before it on `st`: it
// may start while that kernel runs, and orders itself with pdl_wait (see
// rx_common.cuh).  One stream carries the whole call, so its kernels need no
// events between them.
template <typename... KArgs, typename... Args>
int launch_on(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
              bool dependent, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    RX_CUDA_CHECK(cudaLaunchKernelEx(&cfg, kernel, args...));
    return RX_OK;
}

template <int D, bool F8 = false>
int launch_decode_gqa(const Params &p, cudaStream_t st, bool dependent)
{
    constexpr int bytes = F8 ? gqa8_bytes<D>() : GqaLayout::BYTES;
    static bool configured = false;
    if (!configured) {
        RX_CUDA_CHECK(cudaFuncSetAttribute(decode_gqa_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           bytes));
        configured = true;
    }
    const int grid = p.n_wide < num_sms() ? p.n_wide : num_sms();
    return launch_on(decode_gqa_kernel<D, F8>, grid, 32 * (1 + kGqaCopyWarps + kGqaWarps), bytes, st, dependent, p);
}

template <int D, int LOG_NP, int HPW, int CW, bool F8>
int launch_decode_wide_cfg(const Params &p, cudaStream_t st, bool dependent)
{
    static bool configured = false;
    if (!configured) {
        RX_CUDA_CHECK(cudaFuncSetAttribute(decode_wide_kernel<D, LOG_NP, HPW, CW, F8>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, WideLayout::BYTES));
        configured = true;
    }
    const int grid = p.n_wide < num_sms() ? p.n_wide : num_sms();
    return launch_on(decode_wide_kernel<D, LOG_NP, HPW, CW, F8>, grid, 32 * (1 + kWideCopyWarps + CW),
                     WideLayout::BYTES, st, dependent, p);
}

// Wide items need one q head per kv head and 8, 16, 32 or 64 heads: the
// consumer warps (16, or 8 for 8 heads) each own hq / 16 (or one) heads, and
// a stage holds at most one (head, position) pair per lane for each of them.
bool wide_supported(int hq, int hkv, int D)
{
    return hq == hkv && (hq == 8 || hq == 16 || hq == 32 || hq == 64) && (D == 64 || D == 128);
}

template <int D, bool F8>
int launch_decode_wide(const Params &p, cudaStream_t st, bool dependent)
{
    // log2 positions per stage at 8 heads: a stage holds 32 KB of K rows
    // (twice the positions for code rows), at most kWideMaxPos positions (one
    // producer lane each)
    constexpr int L0r = (D == 128 ? 4 : 5) + (F8 ? 1 : 0);
    constexpr int L0 = L0r > 5 ? 5 : L0r;
    static_assert((1 << L0) <= kWideMaxPos, "one producer lane a position");
    switch (p.hq) {
    case 8: return launch_decode_wide_cfg<D, L0, 1, 8, F8>(p, st, dependent);
    case 16: return launch_decode_wide_cfg<D, L0 - 1, 1, 16, F8>(p, st, dependent);
    case 32: return launch_decode_wide_cfg<D, L0 - 2, 2, 16, F8>(p, st, dependent);
    default: return launch_decode_wide_cfg<D, L0 - 3, 4, 16, F8>(p, st, dependent);
    }
}

// the all-heads kernel for the plan's single-request items
template <bool F8>
int launch_all_heads(const Params &p, int D, cudaStream_t st, bool dependent)
{
    if (p.G == 1)
        return D == 128 ? launch_decode_wide<128, F8>(p, st, dependent)
                        : launch_decode_wide<64, F8>(p, st, dependent);
    return D == 128 ? launch_decode_gqa<128, F8>(p, st, dependent) : launch_decode_gqa<64, F8>(p, st, dependent);
}

template <int D, bool PLAN, bool F8>
int launch_decode(const Params &p, cudaStream_t st)
{
    static bool configured = false;
    if (!configured) {
        RX_CUDA_CHECK(cudaFuncSetAttribute(decode_kernel<D, PLAN, F8>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Layout<D, F8>::BYTES));
        configured = true;
    }
    const int grid = p.total_work < num_sms() ? p.total_work : num_sms();
    return launch_on(decode_kernel<D, PLAN, F8>, grid, kThreads, Layout<D, F8>::BYTES, st, false, p);
}

template <int D>
int launch_merge(const Params &p, int use_plan, cudaStream_t st)
{
    const int64_t rows = (int64_t)p.batch * p.hq;
    const unsigned grid = (unsigned)((rows + 3) / 4);
    if (p.max_parts > kMergeFew)
        return launch_on(merge_kernel<D, kMergeFew, true>, grid, 128, 0, st, true, p, use_plan);
    if (p.max_parts > 8) return launch_on(merge_kernel<D, kMergeFew, false>, grid, 128, 0, st, true, p, use_plan);
    if (p.max_parts > 4) return launch_on(merge_kernel<D, 8, false>, grid, 128, 0, st, true, p, use_plan);
    return launch_on(merge_kernel<D, 4, false>, grid, 128, 0, st, true, p, use_plan);
}

}  // namespace

int32_t rx_decode_default_chunk(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len)
{
    const int64_t total = (int64_t)batch * num_kv_heads * (int64_t)max_seq_len;
    int64_t c = (total + RX_DECODE_TARGET_ITEMS - 1) / RX_DECODE_TARGET_ITEMS;
    c = (c + 63) / 64 * 64;
    if (c < 64) c = 64;
    if (c > RX_MAX_KV_CHUNK) c = RX_MAX_KV_CHUNK;
    return (int32_t)c;
}

extern "C" size_t rx_attn_decode_workspace(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t max_seq_len,
                                           const rx_decode_plan *plan)
{
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_seq_len <= 0)
        return 0;
    int64_t parts;
    if (plan) {
        parts = plan->max_parts;
    } else {
        const int64_t c = rx_decode_default_chunk(batch, num_kv_heads, max_seq_len);
        parts = (max_seq_len + c - 1) / c;
    }
    // partials (o and log2-sum-exp) when a request is split, then 256 bytes
    // for the wide kernel's item counter when it runs
    const int64_t rows = parts > 1 ? (int64_t)batch * num_q_heads * parts : 0;
    const int64_t bytes = (rows * (head_dim + 1) * 4 + 255) / 256 * 256;
    const bool wide = plan && plan->n_wide > 0 && (wide_supported(num_q_heads, num_kv_heads, head_dim) ||
                                                   gqa_supported(num_q_heads, num_kv_heads, head_dim));
    return (size_t)(bytes + (wide ? 256 : 0));
}

// Bound on each pipeline wait of the decode kernels (0: rx::kWaitCycles).
static std::atomic<long long> g_decode_wait_cycles{0};

extern "C" int rx_decode_set_wait_limit(int64_t cycles)
{
    g_decode_wait_cycles.store(cycles > 0 ? (long long)cycles : 0);
    return RX_OK;
}

namespace {

// One layer of the pool a decode call reads: bf16 rows, or E4M3 codes with a
// scale per pool.
struct DecodePool {
    const void *k, *v;
    int64_t num_slots;
    int hkv, D;
    bool f8;
    float k_scale, v_scale;
};

// Argument checks shared by the decode entry points (`who` names the entry
// point in the message), after each has checked its pool struct.
int check_decode_args(const char *who, const DecodePool &pool, const void *q, const void *o, const float *lse,
                      int32_t hq, const int32_t *req_idx, const int32_t *seq_len, const int32_t *rtt,
                      int64_t rtt_stride, int32_t batch, int32_t max_seq_len, const rx_decode_plan *plan,
                      float sm_scale)
{
    if (pool.D != 64 && pool.D != 128)
        return rx_set_error(RX_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 64, 128)", who, pool.D);
    if (!q || !o || !req_idx || !seq_len || !rtt || rtt_stride <= 0 || rtt_stride > INT32_MAX ||
        batch < 0 || hq <= 0 || max_seq_len <= 0 || max_seq_len > rtt_stride || !(sm_scale > 0.f))
        return rx_set_error(RX_ERR_INVALID, "%s: invalid argument", who);
    if (hq % pool.hkv != 0 || 64 % (hq / pool.hkv) != 0)
        return rx_set_error(RX_ERR_UNSUPPORTED, "%s: %d q heads over %d kv heads (need G | 64)", who, hq,
                            pool.hkv);
    if (rx_misaligned16(q) || rx_misaligned16(o) || rx_misaligned16(pool.k) ||
        rx_misaligned16(pool.v) || (reinterpret_cast<uintptr_t>(lse) & 3) != 0)
        return rx_set_error(RX_ERR_INVALID, "%s: q, o and the pools must be 16-byte aligned", who);
    if (plan && (!plan->order || !plan->nparts || !plan->items || plan->n_items < 0 ||
                 plan->max_parts < 1 || plan->n_wide < 0 || plan->n_wide > plan->n_items))
        return rx_set_error(RX_ERR_INVALID, "%s: invalid plan", who);
    return RX_OK;
}

int bf16_pool(const char *who, const rx_kv_pool *pool, DecodePool &out)
{
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0)
        return rx_set_error(RX_ERR_INVALID, "%s: invalid pool", who);
    out = DecodePool{pool->k, pool->v, pool->num_slots, pool->num_kv_heads, pool->head_dim, false, 1.f, 1.f};
    return RX_OK;
}

// The decode call on either pool type, after the checks: the per-head
// kernel takes the plan's items of several requests (or, without a plan,
// the fixed split of every request), the all-heads kernel the plan's
// single-request items where it has a variant for the head counts, and the
// merge combines split rows.
int decode_call(const char *who, const DecodePool &pool, const void *q, void *o, float *lse, int32_t hq,
                const int32_t *req_idx, const int32_t *seq_len, const int32_t *rtt, int64_t rtt_stride,
                int32_t batch, int32_t max_seq_len, const rx_decode_plan *plan, void *workspace, size_t ws_bytes,
                float sm_scale, int32_t *dev_status, void *stream)
{
    if (batch == 0) return RX_OK;
    const int D = pool.D;
    Params p{};
    p.q = (const bf16 *)q;
    p.o = (bf16 *)o;
    p.lse = lse;
    p.k_pool = pool.f8 ? nullptr : (const bf16 *)pool.k;
    p.v_pool = pool.f8 ? nullptr : (const bf16 *)pool.v;
    p.kb = (const unsigned char *)pool.k;
    p.vb = (const unsigned char *)pool.v;
    p.row_bytes = (int64_t)pool.hkv * D * (pool.f8 ? 1 : 2);
    p.v_scale = pool.v_scale;
    p.num_slots = pool.num_slots;
    p.hq = hq;
    p.hkv = pool.hkv;
    p.G = hq / pool.hkv;
    p.head_dim = D;
    p.req_idx = req_idx;
    p.seq_len = seq_len;
    p.rtt = rtt;
    p.rtt_stride = rtt_stride;
    p.batch = batch;
    p.scale_log2 = sm_scale * pool.k_scale * rx::kLog2e;
    p.status = dev_status;
    const long long limit = g_decode_wait_cycles.load();
    p.wait_cycles = limit > 0 ? limit : rx::kWaitCycles;
    int64_t total;
    if (plan) {
        p.order = plan->order;
        p.nparts = plan->nparts;
        p.items = plan->items;
        p.max_parts = plan->max_parts;
        // the plan's last n_wide items hold one request each; they go to the
        // all-heads kernel for the head counts it is built for (else to the
        // per-head kernel with the rest)
        p.n_wide = (wide_supported(hq, p.hkv, D) || gqa_supported(hq, p.hkv, D)) ? plan->n_wide : 0;
        p.wide0 = plan->n_items - p.n_wide;
        total = (int64_t)p.wide0 * p.hkv;
    } else {
        p.chunk = rx_decode_default_chunk(batch, p.hkv, max_seq_len);
        p.n_chunks = (max_seq_len + p.chunk - 1) / p.chunk;
        p.max_parts = p.n_chunks;
        total = (int64_t)batch * p.n_chunks * p.hkv;
    }
    if (total > INT32_MAX) return rx_set_error(RX_ERR_UNSUPPORTED, "%s: %lld work items", who, (long long)total);
    if (total == 0 && p.n_wide == 0) return RX_OK;
    p.total_work = (int)total;
    const size_t need = rx_attn_decode_workspace(batch, hq, p.hkv, D, max_seq_len, plan);
    const bool merge = p.max_parts > 1;
    if (need > 0) {
        if (!workspace || ws_bytes < need)
            return rx_set_error(RX_ERR_CAPACITY, "%s: workspace needs %zu bytes, got %zu", who, need, ws_bytes);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
            return rx_set_error(RX_ERR_INVALID, "%s: workspace must be 256-byte aligned", who);
        if (merge) {
            p.ws_o = (float *)workspace;
            p.ws_lse = p.ws_o + (int64_t)batch * hq * p.max_parts * D;
        }
        if (p.n_wide > 0) p.wide_counter = reinterpret_cast<int *>(static_cast<char *>(workspace) + need - 256);
    }
    cudaStream_t st = (cudaStream_t)stream;
    int rc = RX_OK;
    auto per_head = [&](cudaStream_t s) {
        if (pool.f8) {
            if (D == 128) return plan ? launch_decode<128, true, true>(p, s) : launch_decode<128, false, true>(p, s);
            return plan ? launch_decode<64, true, true>(p, s) : launch_decode<64, false, true>(p, s);
        }
        if (D == 128) return plan ? launch_decode<128, true, false>(p, s) : launch_decode<128, false, false>(p, s);
        return plan ? launch_decode<64, true, false>(p, s) : launch_decode<64, false, false>(p, s);
    };
    // One stream, up to three kernels.  The per-head items (shared segments)
    // and the single-request items run side by side: the all-heads kernel is
    // a programmatic dependent of the per-head kernel, which lets it start at
    // once; it reads nothing the per-head kernel writes and ends after it.
    // The merge is a dependent of the last of them and waits for it (and so
    // for both) before it reads their partial results.
    if (p.n_wide > 0) RX_CUDA_CHECK(cudaMemsetAsync(p.wide_counter, 0, sizeof(int), st));
    if (p.total_work > 0) rc = per_head(st);
    if (rc == RX_OK && p.n_wide > 0)
        rc = pool.f8 ? launch_all_heads<true>(p, D, st, p.total_work > 0)
                     : launch_all_heads<false>(p, D, st, p.total_work > 0);
    if (rc != RX_OK || !merge) return rc;
    return D == 128 ? launch_merge<128>(p, plan != nullptr, st) : launch_merge<64>(p, plan != nullptr, st);
}

}  // namespace

extern "C" int rx_attn_decode(const rx_kv_pool *pool_in, const void *q, void *o, float *lse,
                              int32_t hq, const int32_t *req_idx, const int32_t *seq_len,
                              const int32_t *rtt, int64_t rtt_stride, int32_t batch,
                              int32_t max_seq_len, const rx_decode_plan *plan, void *workspace,
                              size_t ws_bytes, float sm_scale, int32_t *dev_status, void *stream)
{
    rx_kv_pool layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 0, "rx_attn_decode")) return rc;
    DecodePool pool;
    if (const int rc = bf16_pool("rx_attn_decode", pool_in ? &layer_view : nullptr, pool)) return rc;
    if (const int rc = check_decode_args("rx_attn_decode", pool, q, o, lse, hq, req_idx, seq_len, rtt, rtt_stride,
                                         batch, max_seq_len, plan, sm_scale))
        return rc;
    return decode_call("rx_attn_decode", pool, q, o, lse, hq, req_idx, seq_len, rtt, rtt_stride, batch,
                       max_seq_len, plan, workspace, ws_bytes, sm_scale, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Decode over FP8 (E4M3) pools
// ---------------------------------------------------------------------------
//
// The same items and kernels as over a bf16 pool, each in an FP8 variant:
// the per-head kernel's copiers widen the code rows into its bf16 tiles, the
// one-q-head all-heads kernel widens codes to floats as it loads them, and
// the GQA all-heads kernel reads whole code rows and widens them to f16 on
// the way to the tensor cores.  K's scale joins the score scale, V's the
// output; split rows merge as usual.

extern "C" int rx_attn_decode_fp8(const rx_kv_pool_fp8 *pool_in, const void *q, void *o, float *lse,
                                  int32_t hq, const int32_t *req_idx, const int32_t *seq_len,
                                  const int32_t *rtt, int64_t rtt_stride, int32_t batch, int32_t max_seq_len,
                                  const rx_decode_plan *plan, void *workspace, size_t ws_bytes, float sm_scale,
                                  int32_t *dev_status, void *stream)
{
    rx_kv_pool_fp8 layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 1, "rx_attn_decode_fp8")) return rc;
    const rx_kv_pool_fp8 *pool = pool_in ? &layer_view : nullptr;
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0 ||
        !(pool->k_scale > 0.f) || !(pool->v_scale > 0.f))
        return rx_set_error(RX_ERR_INVALID, "rx_attn_decode_fp8: invalid pool");
    const DecodePool dp{pool->k, pool->v, pool->num_slots, pool->num_kv_heads, pool->head_dim, true,
                        pool->k_scale, pool->v_scale};
    if (const int rc = check_decode_args("rx_attn_decode_fp8", dp, q, o, lse, hq, req_idx, seq_len, rtt,
                                         rtt_stride, batch, max_seq_len, plan, sm_scale))
        return rc;
    return decode_call("rx_attn_decode_fp8", dp, q, o, lse, hq, req_idx, seq_len, rtt, rtt_stride, batch,
                       max_seq_len, plan, workspace, ws_bytes, sm_scale, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Decode without a caller workspace
// ---------------------------------------------------------------------------
//
// Some callers cannot hand this library device scratch memory: an engine
// whose device memory is all committed at start-up (most of it to the KV
// pool) and that forbids allocator calls while serving, or a host program
// that only lends its own buffers for inputs and outputs.  For them the
// partial results of split work live in the fixed array below instead of a
// workspace.  It is a file-scope device array, so every GPU that loads this
// library holds RX_DECODE_STATIC_SCRATCH_BYTES of it until the process
// exits.  In host code its name is only a stand-in for the symbol, never a
// device address: the address is looked up once per device with
// cudaGetSymbolAddress (on the first call made with that device current) and
// kept.  A device reset (cudaDeviceReset, or anything else that destroys the
// device's primary context) unloads the module and makes the kept address
// stale: this entry point must not be called on that device afterwards.

static __device__ __align__(256) unsigned char g_decode_scratch[RX_DECODE_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
}  // namespace

extern "C" int rx_attn_decode_static(const rx_kv_pool *pool_in, const void *q, void *o, float *lse,
                                     int32_t num_q_heads, const int32_t *req_idx,
                                     const int32_t *seq_len, const int32_t *req_to_token,
                                     int64_t rtt_stride, int32_t batch, int32_t max_seq_len,
                                     const rx_decode_plan *plan_or_null, float sm_scale,
                                     int32_t *dev_status, void *stream)
{
    rx_kv_pool layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 0, "rx_attn_decode_static")) return rc;
    const rx_kv_pool *pool = pool_in ? &layer_view : nullptr;
    // the same checks as rx_attn_decode first, so that a malformed call is
    // reported as such rather than as a batch too big for the array
    DecodePool dp;
    if (const int rc = bf16_pool("rx_attn_decode_static", pool, dp)) return rc;
    const int chk = check_decode_args("rx_attn_decode_static", dp, q, o, lse, num_q_heads, req_idx, seq_len,
                                      req_to_token, rtt_stride, batch, max_seq_len, plan_or_null, sm_scale);
    if (chk != RX_OK) return chk;
    if (batch == 0) return RX_OK;
    const size_t need = rx_attn_decode_workspace(batch, num_q_heads, pool->num_kv_heads,
                                                 pool->head_dim, max_seq_len, plan_or_null);
    if (need > (size_t)RX_DECODE_STATIC_SCRATCH_BYTES)
        return rx_set_error(RX_ERR_CAPACITY,
                            "rx_attn_decode_static: this batch needs %zu bytes of partial results, "
                            "above the fixed %u-byte scratch array; use rx_attn_decode with a workspace",
                            need, (unsigned)RX_DECODE_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    if (need > 0) {
        int dev = 0;
        RX_CUDA_CHECK(cudaGetDevice(&dev));
        if (dev < 0 || dev >= kMaxDevices)
            return rx_set_error(RX_ERR_UNSUPPORTED, "rx_attn_decode_static: device %d", dev);
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev]) {
            void *addr = nullptr;
            RX_CUDA_CHECK(cudaGetSymbolAddress(&addr, g_decode_scratch));
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    // Every partial read from the scratch array is written earlier in the
    // same call, and rx_attn_decode zeroes the work counter it keeps at the
    // array's end before each launch, so nothing carries over between calls.
    return rx_attn_decode(pool, q, o, lse, num_q_heads, req_idx, seq_len, req_to_token, rtt_stride,
                          batch, max_seq_len, plan_or_null, scratch, need, sm_scale, dev_status,
                          stream);
}
