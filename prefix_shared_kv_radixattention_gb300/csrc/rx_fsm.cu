// rx_fsm.cu -- compressed finite-state machine for constrained decoding.
//
// "SGLang: Efficient Execution of Structured Language Model Programs"
// (unite.ai, es), "Introducción a SGLang", compressed-FSM bullet: instead of
// following an output constraint one next token at a time, the runtime
// analyses the constraint, builds a compressed finite-state machine, and
// turns a path of several tokens into one step wherever it can.
//
// Reading taken here (the pages give no algorithm):
//   * the constraint is a deterministic automaton over token ids (CSR per
//     state, tokens ascending); a state without edges is terminal;
//   * a state with exactly one edge fixes the next token; the jump of a state
//     is the run of fixed tokens along such states, stopping at the first
//     state with another edge count, on coming back to a state, or after
//     max_jump tokens (rx_fsm_compress, on the host);
//   * a decoding step takes the masked argmax of the request's logits over
//     the tokens its state allows (NaN as -inf, ties to the smallest id),
//     follows that edge, and emits the jump of the state it reaches in the
//     same step (rx_fsm_step, on the device).
//
// The step is a streaming pass over each request's logits row (HBM-bound):
// a cluster of C CTAs shares a row and each CTA takes one slice.  In a CTA
// one thread streams the slice into a ring of shared-memory stages with bulk
// copies (cp.async.bulk onto mbarriers: 96 KB in flight per CTA, no
// registers held) together with the matching words of the request state's
// allowed-token mask, and fifteen warps scan each landed stage from shared
// memory alone.  The CTAs' best (value, id) pairs meet
// in CTA 0 through distributed shared memory, and one warp of CTA 0 follows
// the edge and writes the jump.
#include <algorithm>
#include <climits>
#include <cmath>
#include <limits>
#include <vector>

#include "rx_common.cuh"

namespace {

constexpr int kFsmThreads = 512;                  // warp 0 copies, warps 1 .. 15 scan
constexpr int kFsmScanWarps = kFsmThreads / 32 - 1;
constexpr int kFsmScanThreads = 32 * kFsmScanWarps;
constexpr int kFsmMaxCluster = 8;
constexpr int kFsmStages = 3;                     // ring of logits stages per CTA
constexpr int kFsmStageIds = 8192;                // 32 KB of fp32 logits a stage
constexpr int kFsmGroups = kFsmStageIds / 4;      // 16-byte groups of four ids a stage
constexpr int kFsmCopyBytes = 8192;               // largest single bulk copy
constexpr int kFsmGroupsPerThread = (kFsmGroups + kFsmScanThreads - 1) / kFsmScanThreads;
constexpr int kFsmOffMask = kFsmStages * kFsmStageIds * 4;         // mask words [S][ids / 32]
constexpr int kFsmOffBar = kFsmOffMask + kFsmStages * (kFsmStageIds / 32) * 4;  // full [S], empty [S]
constexpr int kFsmOffAbort = kFsmOffBar + 2 * kFsmStages * 8;
constexpr int kFsmSmem = kFsmOffAbort + 16 + 128;  // + room to align the base to 128

struct FsmParams {
    const int64_t *row_ptr;
    const int32_t *tok;
    const int32_t *nxt;
    const uint32_t *mask;
    const int32_t *rank;
    const int32_t *jump_len;
    const int64_t *jump_off;
    const int32_t *jump_end;
    const int32_t *jump_tok;
    const float *logits;
    int64_t stride;
    int32_t *state;
    int32_t *out_tokens;
    int32_t *out_count;
    int32_t *status;
    int32_t n_states, vocab, max_jump, words, chunk;
};

// candidate (v, i) beats (bv, bi): larger value, or equal value and smaller id
__device__ __forceinline__ bool beats(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void take(float v, int i, float &bv, int &bi)
{
    v = (v != v) ? -INFINITY : v;  // NaN counts as -inf
    if (beats(v, i, bv, bi)) {
        bv = v;
        bi = i;
    }
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// value at the same shared-memory offset in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t dsmem_ld_u32(const void *local, uint32_t rank)
{
    uint32_t addr = rx::smem_u32(local), remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(addr), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// bounded wait of one thread (the copying lane); false on timeout or abort
__device__ __forceinline__ bool fsm_wait1(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status)
{
    const long long t0 = clock64();
    do {
        if (rx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    } while (clock64() - t0 < rx::kWaitCycles);
    if (!*abort_flag) {
        *abort_flag = 1;
        if (status) atomicOr(status, RX_DEV_TIMEOUT);
    }
    return false;
}

// bounded wait of a whole warp; false (for every lane) on timeout or abort
__device__ __forceinline__ bool fsm_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status)
{
    bool ok = false;
    const long long t0 = clock64();
    do {
        if (rx::mbar_try_wait(bar, parity)) {
            ok = true;
            break;
        }
        if (*abort_flag) break;
    } while (clock64() - t0 < rx::kWaitCycles);
    if (!ok && !*abort_flag) {
        *abort_flag = 1;
        if (status) atomicOr(status, RX_DEV_TIMEOUT);
    }
    return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kFsmThreads) fsm_step_kernel(const FsmParams p)
{
    extern __shared__ __align__(128) unsigned char fraw[];
    __shared__ float wv[kFsmThreads / 32];
    __shared__ int wi[kFsmThreads / 32];
    __shared__ float cta_v;
    __shared__ int cta_i;
    const uint32_t raw = rx::smem_u32(fraw);
    unsigned char *smem = fraw + (((raw + 127u) & ~127u) - raw);
    const float *buf = reinterpret_cast<const float *>(smem);
    const uint32_t *mbuf = reinterpret_cast<const uint32_t *>(smem + kFsmOffMask);
    const uint32_t bar = rx::smem_u32(smem + kFsmOffBar);  // full [S], empty [S]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kFsmOffAbort);
    const uint32_t rank = cluster_rank();
    uint32_t nrank;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(nrank));
    const int b = (int)(blockIdx.x / nrank);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kFsmStages; ++i) {
            rx::mbar_init(bar + 8 * i, 1);                                 // the copying lane + bytes
            rx::mbar_init(bar + 8 * (kFsmStages + i), kFsmScanWarps);      // scanning warps
        }
        *abort_flag = 0;
        rx::fence_mbar_init();
    }
    __syncthreads();
    const int s = __ldg(p.state + b);
    const bool good = s >= 0 && s < p.n_states;
    const int lo = (int)rank * p.chunk;
    const int hi = min(p.vocab, lo + p.chunk);
    const int n_stages = (good && hi > lo) ? (hi - lo + kFsmStageIds - 1) / kFsmStageIds : 0;
    // requests start their rows at different stages (taken round the row):
    // the rows' streams then do not walk the same offsets in step
    const int rot = n_stages ? b % n_stages : 0;
    auto stage_at = [&](int j) { return j + rot < n_stages ? j + rot : j + rot - n_stages; };

    float bv = -INFINITY;
    int bi = INT_MAX;
    if (warp == 0) {
        if (lane == 0) {
            // whole 16-byte groups: a row holds at least vocab rounded up to
            // four ids, and ids past vocab have no mask bit; mask rows are
            // padded to 16 bytes, and a stage starts on a 128-id boundary
            const float *row = p.logits + (int64_t)b * p.stride;
            const uint32_t *mrow = p.mask + (int64_t)s * p.words;
            int j = 0;
            for (; j < n_stages; ++j) {
                const int st = j % kFsmStages;
                if (j >= kFsmStages &&
                    !fsm_wait1(bar + 8 * (kFsmStages + st), ((j / kFsmStages) - 1) & 1, abort_flag, p.status))
                    break;
                const int i0 = lo + stage_at(j) * kFsmStageIds;
                const int cnt = min(kFsmStageIds, hi - i0);
                const uint32_t bytes = (uint32_t)((cnt + 3) / 4) * 16u;
                const uint32_t mbytes = (uint32_t)((cnt + 127) / 128) * 16u;
                rx::mbar_arrive_expect_tx(bar + 8 * st, bytes + mbytes);
                // the stage in copies of at most 8 KB, so that it streams in
                // as several requests at once
                for (uint32_t c = 0; c < bytes; c += kFsmCopyBytes)
                    rx::bulk_g2s(rx::smem_u32(buf + st * kFsmStageIds) + c,
                                 reinterpret_cast<const unsigned char *>(row + i0) + c,
                                 min((uint32_t)kFsmCopyBytes, bytes - c), bar + 8 * st);
                rx::bulk_g2s(rx::smem_u32(mbuf + st * (kFsmStageIds / 32)), mrow + i0 / 32, mbytes, bar + 8 * st);
            }
            // no copy may still be landing when the CTA exits
            for (int jj = j > kFsmStages ? j - kFsmStages : 0; jj < j; ++jj) {
                const long long t0 = clock64();
                while (!rx::mbar_try_wait(bar + 8 * (jj % kFsmStages), (jj / kFsmStages) & 1))
                    if (clock64() - t0 >= rx::kWaitCycles) {
                        if (p.status) atomicOr(p.status, RX_DEV_TIMEOUT);
                        break;
                    }
            }
        }
        __syncwarp();
    } else {
        const int ct = (int)threadIdx.x - 32;
        for (int j = 0; j < n_stages; ++j) {
            const int st = j % kFsmStages;
            const int i0 = lo + stage_at(j) * kFsmStageIds;       // a multiple of 128: groups sit in mask words
            const int ng = (min(kFsmStageIds, hi - i0) + 3) / 4;
            if (!fsm_wait_warp(bar + 8 * st, (j / kFsmStages) & 1, abort_flag, p.status)) break;
            const float4 *sb = reinterpret_cast<const float4 *>(buf + st * kFsmStageIds);
            const uint32_t *sm = mbuf + st * (kFsmStageIds / 32);
            uint32_t mb[kFsmGroupsPerThread];
#pragma unroll
            for (int u = 0; u < kFsmGroupsPerThread; ++u) {
                const int g = ct + u * kFsmScanThreads;
                mb[u] = g < ng ? (sm[g >> 3] >> ((4 * g) & 31)) & 0xFu : 0u;
            }
#pragma unroll
            for (int u = 0; u < kFsmGroupsPerThread; ++u) {
                if (!mb[u]) continue;
                const int g = ct + u * kFsmScanThreads;
                const float4 x = sb[g];
                const int i = i0 + 4 * g;
                if (mb[u] & 1u) take(x.x, i, bv, bi);
                if (mb[u] & 2u) take(x.y, i + 1, bv, bi);
                if (mb[u] & 4u) take(x.z, i + 2, bv, bi);
                if (mb[u] & 8u) take(x.w, i + 3, bv, bi);
            }
            __syncwarp();
            if (lane == 0) rx::mbar_arrive(bar + 8 * (kFsmStages + st));
        }
    }
    // warp, then CTA
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (beats(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if (lane == 0) {
        wv[warp] = bv;
        wi[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kFsmThreads / 32; ++w)
            if (beats(wv[w], wi[w], bv, bi)) {
                bv = wv[w];
                bi = wi[w];
            }
        cta_v = bv;
        cta_i = bi;
    }
    // the cluster's CTAs meet in CTA 0 (both barriers are reached by every
    // thread of every CTA; the second keeps each CTA's shared memory alive
    // until CTA 0 has read it)
    cluster_sync();
    if (rank == 0 && warp == 0) {
        float v = -INFINITY;
        int i = INT_MAX;
        if (lane < (int)nrank) {
            v = __uint_as_float(dsmem_ld_u32(&cta_v, (uint32_t)lane));
            i = (int)dsmem_ld_u32(&cta_i, (uint32_t)lane);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            if (beats(ov, oi, v, i)) {
                v = ov;
                i = oi;
            }
        }
        bv = v;
        bi = i;
    }
    cluster_sync();
    if (rank != 0 || warp != 0) return;

    // follow the chosen edge, then the jump of the state it reaches
    int32_t *out = p.out_tokens + (int64_t)b * (1 + p.max_jump);
    if (!good) {
        if (lane == 0) {
            p.out_count[b] = 0;
            if (p.status) atomicOr(p.status, RX_DEV_BAD_STATE);
        }
        return;
    }
    if (bi == INT_MAX) {  // no token allowed: the constrained text is complete
        if (lane == 0) {
            p.out_count[b] = 0;
            if (p.status) atomicOr(p.status, RX_DEV_FSM_DONE);
        }
        return;
    }
    int s1 = -1, jl = 0;
    int64_t off = 0;
    if (lane == 0) {
        // the chosen token's edge: the state's edges below its mask word,
        // plus the allowed ids below it within the word (three independent
        // loads, then the edge)
        const int64_t wrd = (int64_t)s * p.words + (bi >> 5);
        const int64_t e = __ldg(p.row_ptr + s) + __ldg(p.rank + wrd) +
                          __popc(__ldg(p.mask + wrd) & ((1u << (bi & 31)) - 1u));
        if (e < __ldg(p.row_ptr + s + 1) && __ldg(p.tok + e) == bi) s1 = __ldg(p.nxt + e);
        if (s1 >= 0 && s1 < p.n_states) {
            jl = __ldg(p.jump_len + s1);
            off = __ldg(p.jump_off + s1);
            if (jl < 0 || jl > p.max_jump) s1 = -1;
        } else {
            s1 = -1;
        }
    }
    s1 = __shfl_sync(0xffffffffu, s1, 0);
    jl = __shfl_sync(0xffffffffu, jl, 0);
    off = __shfl_sync(0xffffffffu, off, 0);
    if (s1 < 0) {  // mask and edge list disagree, or a malformed jump
        if (lane == 0) {
            p.out_count[b] = 0;
            if (p.status) atomicOr(p.status, RX_DEV_BAD_STATE);
        }
        return;
    }
    for (int k = lane; k < jl; k += 32) out[1 + k] = __ldg(p.jump_tok + off + k);
    if (lane == 0) {
        out[0] = bi;
        p.out_count[b] = 1 + jl;
        p.state[b] = __ldg(p.jump_end + s1);
    }
}

int fsm_num_sms()
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

}  // namespace

extern "C" int rx_fsm_compress(int32_t n_states, int32_t vocab, const int64_t *row_ptr, const int32_t *tok,
                               const int32_t *nxt, int32_t max_jump, uint32_t *out_mask, int32_t *out_rank,
                               int32_t *out_jump_len, int64_t *out_jump_off, int32_t *out_jump_end,
                               int32_t *out_jump_tok, int64_t jump_tok_cap, rx_fsm_info *info)
{
    RX_TRY
    if (n_states < 1 || vocab < 1 || max_jump < 0 || !row_ptr || !info)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_compress: invalid argument");
    if (row_ptr[0] != 0) return rx_set_error(RX_ERR_INVALID, "rx_fsm_compress: row_ptr[0] != 0");
    for (int32_t s = 0; s < n_states; ++s)
        if (row_ptr[s + 1] < row_ptr[s])
            return rx_set_error(RX_ERR_INVALID, "rx_fsm_compress: row_ptr decreases at state %d", s);
    const int64_t E = row_ptr[n_states];
    if (E > 0 && (!tok || !nxt)) return rx_set_error(RX_ERR_INVALID, "rx_fsm_compress: null edge arrays");
    for (int32_t s = 0; s < n_states; ++s)
        for (int64_t e = row_ptr[s]; e < row_ptr[s + 1]; ++e) {
            if (tok[e] < 0 || tok[e] >= vocab || nxt[e] < 0 || nxt[e] >= n_states)
                return rx_set_error(RX_ERR_INVALID, "rx_fsm_compress: edge %lld out of range", (long long)e);
            if (e > row_ptr[s] && tok[e] <= tok[e - 1])
                return rx_set_error(RX_ERR_INVALID, "rx_fsm_compress: tokens of state %d not increasing", s);
        }
    // jumps: follow single-edge states from every state
    std::vector<int32_t> len((size_t)n_states), end((size_t)n_states);
    std::vector<char> looped((size_t)n_states, 0);
    std::vector<int32_t> seen((size_t)n_states, -1);  // state -> start state of the walk that passed it
    int64_t total = 0;
    int32_t longest = 0, n_single = 0, n_loop = 0;
    for (int32_t s = 0; s < n_states; ++s) {
        n_single += row_ptr[s + 1] - row_ptr[s] == 1;
        int32_t u = s, k = 0;
        while (k < max_jump && row_ptr[u + 1] - row_ptr[u] == 1) {
            if (seen[(size_t)u] == s) {
                looped[(size_t)s] = 1;
                break;
            }
            seen[(size_t)u] = s;
            u = nxt[row_ptr[u]];
            ++k;
        }
        len[(size_t)s] = k;
        end[(size_t)s] = u;
        total += k;
        longest = std::max(longest, k);
        n_loop += looped[(size_t)s];
    }
    info->n_edges = E;
    info->jump_tokens = total;
    info->n_singular = n_single;
    info->n_looped = n_loop;
    info->longest_jump = longest;
    if (out_jump_tok && jump_tok_cap < total)
        return rx_set_error(RX_ERR_CAPACITY, "rx_fsm_compress: jumps need %lld tokens", (long long)total);
    int64_t off = 0;
    for (int32_t s = 0; s < n_states; ++s) {
        if (out_jump_len) out_jump_len[s] = len[(size_t)s];
        if (out_jump_off) out_jump_off[s] = off;
        if (out_jump_end) out_jump_end[s] = end[(size_t)s];
        if (out_jump_tok) {
            int32_t u = s;
            for (int32_t k = 0; k < len[(size_t)s]; ++k) {
                out_jump_tok[off + k] = tok[row_ptr[u]];
                u = nxt[row_ptr[u]];
            }
        }
        off += len[(size_t)s];
    }
    const int64_t W = ((int64_t)vocab + 127) / 128 * 4;  // words per row, padded to 16 bytes
    if (out_mask) {
        std::fill(out_mask, out_mask + (int64_t)n_states * W, 0u);
        for (int32_t s = 0; s < n_states; ++s)
            for (int64_t e = row_ptr[s]; e < row_ptr[s + 1]; ++e)
                out_mask[(int64_t)s * W + tok[e] / 32] |= 1u << (tok[e] % 32);
    }
    if (out_rank) {
        for (int32_t s = 0; s < n_states; ++s) {
            int64_t e = row_ptr[s];
            for (int64_t w = 0; w < W; ++w) {
                while (e < row_ptr[s + 1] && tok[e] < 32 * w) ++e;
                out_rank[(int64_t)s * W + w] = (int32_t)(e - row_ptr[s]);
            }
        }
    }
    return RX_OK;
    RX_CATCH
}

extern "C" int rx_fsm_step(const rx_fsm *fsm, const float *logits, int64_t logits_stride, int32_t batch,
                           int32_t *state, int32_t *out_tokens, int32_t *out_count, int32_t *dev_status,
                           void *stream)
{
    if (!fsm || batch < 0 || fsm->n_states < 1 || fsm->vocab < 1 || fsm->max_jump < 0)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_step: invalid argument");
    if (batch == 0) return RX_OK;
    if (!logits || !state || !out_tokens || !out_count || !fsm->row_ptr || !fsm->tok || !fsm->nxt ||
        !fsm->mask || !fsm->rank || !fsm->jump_len || !fsm->jump_off || !fsm->jump_end || !fsm->jump_tok)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_step: null pointer");
    if ((reinterpret_cast<uintptr_t>(fsm->mask) & 15) != 0)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_step: the mask must be 16-byte aligned");
    if (logits_stride < fsm->vocab || logits_stride % 4 != 0 ||
        (reinterpret_cast<uintptr_t>(logits) & 15) != 0)
        return rx_set_error(RX_ERR_INVALID,
                            "rx_fsm_step: logits rows must be 16-byte aligned (stride %lld >= vocab, multiple of 4)",
                            (long long)logits_stride);
    FsmParams p{};
    p.row_ptr = fsm->row_ptr;
    p.tok = fsm->tok;
    p.nxt = fsm->nxt;
    p.mask = fsm->mask;
    p.rank = fsm->rank;
    p.jump_len = fsm->jump_len;
    p.jump_off = fsm->jump_off;
    p.jump_end = fsm->jump_end;
    p.jump_tok = fsm->jump_tok;
    p.logits = logits;
    p.stride = logits_stride;
    p.state = state;
    p.out_tokens = out_tokens;
    p.out_count = out_count;
    p.status = dev_status;
    p.n_states = fsm->n_states;
    p.vocab = fsm->vocab;
    p.max_jump = fsm->max_jump;
    p.words = (fsm->vocab + 127) / 128 * 4;
    // CTAs per request: as many as keep the grid to one wave of two
    // 512-thread CTAs per SM (registers allow two), at most a portable
    // cluster of 8, and slices of at least 2048 ids
    const int want = 2 * fsm_num_sms() / batch;
    const int by_size = std::max(1, fsm->vocab / 2048);
    const int C = std::max(1, std::min(std::min(want, by_size), kFsmMaxCluster));
    p.chunk = (int)(((int64_t)fsm->vocab + C - 1) / C);
    p.chunk = (p.chunk + 127) / 128 * 128;  // slices start on a mask word
    if ((int64_t)batch * C > INT32_MAX) return rx_set_error(RX_ERR_UNSUPPORTED, "rx_fsm_step: batch too large");
    static bool configured = false;
    if (!configured) {
        RX_CUDA_CHECK(cudaFuncSetAttribute(fsm_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFsmSmem));
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(batch * C));
    cfg.blockDim = dim3(kFsmThreads);
    cfg.dynamicSmemBytes = kFsmSmem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    RX_CUDA_CHECK(cudaLaunchKernelEx(&cfg, fsm_step_kernel, p));
    return RX_OK;
}
