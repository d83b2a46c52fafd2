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
// The step is a streaming pass over each request's logits row (HBM-bound).
// The scan kernel's CTAs (one resident wave) walk (request, 16384-id tile)
// pairs with 16-byte loads of logits and of the 32-bit allowed-token mask
// words of the request's state, and fold each tile's allowed candidates into
// the request's best (value, id) key with a 64-bit atomicMax.  Then each
// request follows the chosen edge without a search (a per-word prefix count
// of the state's edges), writes the jump, and sets its key back to zero for
// the next call.  For up to kScanThreads requests that finish runs in the
// scan kernel itself: every CTA counts itself done on a counter once its
// warps' key updates are fenced, and the CTA that completes the count -- the
// last one, which then sees every key -- finishes all requests, one a
// thread, and re-arms the counter.  Larger batches use a second kernel, a
// programmatic dependent of the scan, with a warp per request.
#include <algorithm>
#include <climits>
#include <cmath>
#include <limits>
#include <vector>

#include "rx_common.cuh"

namespace {

constexpr int kScanThreads = 512;
constexpr int kTileIds = 16384;          // ids of one scan tile (64 KB of fp32 logits)
constexpr int kScanUnroll = 4;           // 16-byte groups each thread has in flight
constexpr int kScanCtasPerSm = 3;        // resident scan CTAs per SM (registers allow three)
constexpr int kFinishThreads = 256;      // one warp per request

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
    unsigned long long *best;
    unsigned long long *done;   // CTAs of the scan done (the finish in the scan)
    int32_t *status;
    int32_t n_states, vocab, max_jump, words, batch, tiles_per_row;
    int32_t fused;              // the last scan CTA finishes every request
};

// Order-preserving key of a candidate (value v, id i): a larger value, then
// a smaller id, gives a larger key.  NaN counts as -inf and -0 as +0 (equal
// values tie); every candidate's key is above 0, which means "none".  The
// value's half: fmaxf returns its other operand for a NaN, and -0 + 0 is
// +0; then the sign-magnitude bits are made to order as unsigned integers.
__device__ __forceinline__ uint32_t value_key(float v)
{
    v = fmaxf(v, -INFINITY) + 0.f;
    const uint32_t u = __float_as_uint(v);
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}
__device__ __forceinline__ unsigned long long key_of(uint32_t vk, int i)
{
    return ((unsigned long long)vk << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
}

// The edge of state s for token bi, and the jump of the state it leads to:
// s1 = -1 when the mask and the edge list disagree or the jump is malformed.
__device__ __forceinline__ void follow_edge(const FsmParams &p, int s, int bi, int &s1, int &jl, int64_t &off)
{
    s1 = -1;
    jl = 0;
    off = 0;
    if (bi < 0 || bi >= p.vocab) return;
    // the state's edges below bi's mask word, plus the allowed ids below it
    // within the word (no search)
    const int64_t wrd = (int64_t)s * p.words + (bi >> 5);
    const int64_t e = __ldg(p.row_ptr + s) + __ldg(p.rank + wrd) + __popc(__ldg(p.mask + wrd) & ((1u << (bi & 31)) - 1u));
    if (e < __ldg(p.row_ptr + s + 1) && __ldg(p.tok + e) == bi) s1 = __ldg(p.nxt + e);
    if (s1 >= 0 && s1 < p.n_states) {
        jl = __ldg(p.jump_len + s1);
        off = __ldg(p.jump_off + s1);
        if (jl < 0 || jl > p.max_jump) s1 = -1;
    } else {
        s1 = -1;
    }
}

// Finish of request b by one thread, given its best key (0: no token allowed).
__device__ void finish_request(const FsmParams &p, int b, unsigned long long key)
{
    const int s = p.state[b];
    const bool good = s >= 0 && s < p.n_states;
    if (!good || key == 0ull) {  // a bad state, or no token allowed (the text is complete)
        p.out_count[b] = 0;
        if (p.status) atomicOr(p.status, good ? RX_DEV_FSM_DONE : RX_DEV_BAD_STATE);
        return;
    }
    const int bi = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    int s1, jl;
    int64_t off;
    follow_edge(p, s, bi, s1, jl, off);
    if (s1 < 0) {  // mask and edge list disagree, or a malformed jump
        p.out_count[b] = 0;
        if (p.status) atomicOr(p.status, RX_DEV_BAD_STATE);
        return;
    }
    int32_t *out = p.out_tokens + (int64_t)b * (1 + p.max_jump);
    out[0] = bi;
    for (int k = 0; k < jl; ++k) out[1 + k] = __ldg(p.jump_tok + off + k);
    p.out_count[b] = 1 + jl;
    p.state[b] = __ldg(p.jump_end + s1);
}

// Scan: CTAs walk (request, tile) pairs and fold each tile's allowed
// candidates into the request's best key with a 64-bit atomicMax, one per
// warp and tile.  16-byte loads of logits and of the state's mask words,
// four groups in flight per thread.  A thread keeps its best value key and
// id in 32-bit registers (it visits ids in increasing order, so a strict
// comparison keeps the smaller id of a tie) and forms the 64-bit key once
// per tile.
__global__ void __launch_bounds__(kScanThreads, kScanCtasPerSm) fsm_scan_kernel(const FsmParams p)
{
    rx::pdl_launch_dependents();  // the finish kernel may launch now and wait on the device
    const int lane = threadIdx.x & 31;
    const int total = p.batch * p.tiles_per_row;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int b = tile / p.tiles_per_row;
        const int lo = (tile - b * p.tiles_per_row) * kTileIds;
        const int hi = min(p.vocab, lo + kTileIds);
        const int s = __ldg(p.state + b);
        if (s < 0 || s >= p.n_states) continue;  // flagged by the finish kernel
        const float4 *row = reinterpret_cast<const float4 *>(p.logits + (int64_t)b * p.stride);
        const uint32_t *mrow = p.mask + (int64_t)s * p.words;
        // whole 16-byte groups: a row holds at least vocab rounded up to four
        // ids, and ids past vocab have no mask bit; a tile starts on a word
        const int g1 = (hi + 3) / 4;
        uint32_t bv = 0u;  // best value key so far (0: none)
        int bi = 0;        // its id
        for (int g = lo / 4 + (int)threadIdx.x; g < g1; g += kScanThreads * kScanUnroll) {
            float4 x[kScanUnroll];
            uint32_t mw[kScanUnroll];  // the mask word of each group, its 4 bits at 4 * (gg % 8)
#pragma unroll
            for (int u = 0; u < kScanUnroll; ++u) {
                const int gg = g + u * kScanThreads;
                mw[u] = 0u;
                if (gg < g1) {
                    mw[u] = __ldg(mrow + (gg >> 3));
                    x[u] = __ldg(row + gg);
                }
            }
            // every group of one pass sits at the same place in its word (the
            // groups are kScanThreads apart, a multiple of 8)
            static_assert(kScanThreads % 8 == 0, "groups of a pass share their bit position");
            const int sh = (4 * g) & 31;
#pragma unroll
            for (int u = 0; u < kScanUnroll; ++u) {
                const uint32_t mu = (mw[u] >> sh) & 0xFu;
                if (!mu) continue;
                const int i = 4 * (g + u * kScanThreads);
                auto consider = [&](float v, int id) {
                    const uint32_t k = value_key(v);
                    if (k > bv) {
                        bv = k;
                        bi = id;
                    }
                };
                if (mu & 1u) consider(x[u].x, i);
                if (mu & 2u) consider(x[u].y, i + 1);
                if (mu & 4u) consider(x[u].z, i + 2);
                if (mu & 8u) consider(x[u].w, i + 3);
            }
        }
        unsigned long long best = bv ? key_of(bv, bi) : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (lane == 0 && best) atomicMax(p.best + b, best);
    }
    if (!p.fused) return;
    // this CTA's key updates (made by each warp's lane 0) are visible device
    // wide before it counts itself done
    __shared__ int is_last;
    if (lane == 0) __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(p.done, 1ull) == (unsigned long long)gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    // the last CTA: every other CTA's keys are in; read them past L1
    __threadfence();
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
        const unsigned long long key = __ldcg(p.best + b);
        p.best[b] = 0ull;
        finish_request(p, b, key);
    }
    if (threadIdx.x == 0) *p.done = 0ull;  // re-armed for the next call
}

// Finish: one warp per request follows the chosen edge and writes the jump,
// then re-arms the request's key for the next call.
__global__ void __launch_bounds__(kFinishThreads) fsm_finish_kernel(const FsmParams p)
{
    const int b = (int)((blockIdx.x * (unsigned)kFinishThreads + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    // the state is an input (the scan does not write it): read before the wait
    const int s = b < p.batch ? __ldg(p.state + b) : 0;
    rx::pdl_wait();  // the scan kernel's keys are complete and visible
    if (b >= p.batch) return;
    unsigned long long key = 0;
    if (lane == 0) {
        key = p.best[b];
        p.best[b] = 0ull;
    }
    key = __shfl_sync(0xffffffffu, key, 0);
    const bool good = s >= 0 && s < p.n_states;
    if (!good || key == 0ull) {  // a bad state, or no token allowed (the text is complete)
        if (lane == 0) {
            p.out_count[b] = 0;
            if (p.status) atomicOr(p.status, good ? RX_DEV_FSM_DONE : RX_DEV_BAD_STATE);
        }
        return;
    }
    const int bi = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    int s1 = -1, jl = 0;
    int64_t off = 0;
    if (lane == 0) follow_edge(p, s, bi, s1, jl, off);
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
    int32_t *out = p.out_tokens + (int64_t)b * (1 + p.max_jump);
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
                           int32_t *state, int32_t *out_tokens, int32_t *out_count, uint64_t *workspace,
                           int32_t *dev_status, void *stream)
{
    if (!fsm || batch < 0 || fsm->n_states < 1 || fsm->vocab < 1 || fsm->max_jump < 0)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_step: invalid argument");
    if (batch == 0) return RX_OK;
    if (!logits || !state || !out_tokens || !out_count || !workspace || !fsm->row_ptr || !fsm->tok ||
        !fsm->nxt || !fsm->mask || !fsm->rank || !fsm->jump_len || !fsm->jump_off || !fsm->jump_end ||
        !fsm->jump_tok)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_step: null pointer");
    if ((reinterpret_cast<uintptr_t>(workspace) & 7) != 0)
        return rx_set_error(RX_ERR_INVALID, "rx_fsm_step: the workspace must be 8-byte aligned");
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
    p.best = reinterpret_cast<unsigned long long *>(workspace);
    p.done = p.best + batch;
    p.status = dev_status;
    p.n_states = fsm->n_states;
    p.vocab = fsm->vocab;
    p.max_jump = fsm->max_jump;
    p.words = (fsm->vocab + 127) / 128 * 4;
    p.batch = batch;
    p.tiles_per_row = (fsm->vocab + kTileIds - 1) / kTileIds;
    const int64_t tiles = (int64_t)batch * p.tiles_per_row;
    if (tiles > INT32_MAX) return rx_set_error(RX_ERR_UNSUPPORTED, "rx_fsm_step: batch too large");
    p.fused = batch <= kScanThreads;
    cudaStream_t st = (cudaStream_t)stream;
    // scan: one resident wave of CTAs walking the (request, tile) pairs
    const int64_t resident = (int64_t)kScanCtasPerSm * fsm_num_sms();
    const unsigned grid = (unsigned)std::min<int64_t>(tiles, resident);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kScanThreads);
    cfg.stream = st;
    RX_CUDA_CHECK(cudaLaunchKernelEx(&cfg, fsm_scan_kernel, p));
    if (p.fused) return RX_OK;  // the last scan CTA finished every request
    // finish: a programmatic dependent of the scan, waiting on the device
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(((int64_t)batch * 32 + kFinishThreads - 1) / kFinishThreads));
    cfg.blockDim = dim3(kFinishThreads);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    RX_CUDA_CHECK(cudaLaunchKernelEx(&cfg, fsm_finish_kernel, p));
    return RX_OK;
}
