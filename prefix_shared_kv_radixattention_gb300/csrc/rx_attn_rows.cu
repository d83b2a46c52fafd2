// rx_attn_rows.cu -- extend attention on the mma.sync tensor path: up to 64
// query rows (64 / G new tokens of one request times the G q-heads of one kv
// head) per CTA against the slot-gathered keys 0 .. prefix + last token, each
// row masked at its own causal bound j <= p.
//
// What is computed: o = softmax(sm_scale * q K^T + causal mask) V over the
// pool rows listed in req_to_token[b][0..p] (kv-head g = h / G), the extend
// pass of RadixAttention: new tokens attend to their cached prefix plus
// themselves ("SGLang: Efficient Execution of Structured Language Model
// Programs", unite.ai, es, section "Introducción a SGLang": KV of a shared
// prefix is reused, not recomputed).
//
// Data path: slot ids prefetched one pipeline step ahead into registers; K
// and V rows gathered with 16-byte cp.async into a 3-stage shared-memory ring
// of 64-key tiles (16-byte chunks XOR-swizzled for conflict-free ldmatrix);
// S = Q K^T and O += P V on mma.sync m16n8k16 with fp32 accumulators; online
// softmax in the exp2 domain.
#include <math.h>

#include "rx_common.cuh"

namespace {

using bf16 = __nv_bfloat16;

constexpr int kBN = 64;       // keys per tile
constexpr int kStages = 3;    // cp.async ring depth
constexpr int kThreads = 128; // 4 warps
constexpr int kMaxRows = 64;  // query rows per CTA

enum Mode { kExtend = 2 };

struct Params {
    const bf16 *q;
    bf16 *o;
    float *lse;
    const bf16 *k_pool;
    const bf16 *v_pool;
    int64_t num_slots;
    int hq, hkv, G;
    const int32_t *req_idx;
    const int32_t *seq_len;
    const int32_t *qo_indptr;   // extend
    const int32_t *prefix_len;  // extend
    const int32_t *extend_len;  // extend
    const int32_t *rtt;
    int64_t rtt_stride;
    const int32_t *order;
    const int32_t *nparts;
    const int32_t *items;
    int batch;
    int chunk;      // grid mode: positions per item
    int max_parts;  // partial-result stride per row
    float *ws_o;
    float *ws_lse;
    float scale_log2;
    int32_t *status;
};

struct Work {
    int M;                 // query rows
    int64_t p0, p1;        // key positions [p0, p1)
    const int32_t *slots;  // slot list shared by every row of the item
    int part;
    bool final_;
    int r0;                // plan mode: first plan row
    int b;                 // grid mode: batch index
    int64_t qbase;         // extend: packed token index of row group 0
    int64_t cbase;         // extend: position of row group 0
};

template <int MODE>
__device__ __forceinline__ int64_t qrow_of(const Params &p, const Work &w, int m)
{
    return w.qbase + m / p.G;
}

template <int D, int WM, int MODE>
__device__ __forceinline__ void attn_rows_body(const Params &p, const Work &w, int g,
                                               unsigned char *smem)
{
    constexpr int WK = 4 / WM;          // warps along keys
    constexpr int KW = kBN / WK;        // keys per warp per tile
    constexpr int NT = KW / 8;          // S n-tiles per warp
    constexpr int KT = KW / 16;         // PV k-steps per warp
    constexpr int DT = D / 8;           // O n-tiles
    constexpr int CPR = D / 8;          // 16-byte chunks per K/V row
    constexpr int ROW_STEP = kThreads / CPR;
    constexpr int RPT = kBN / ROW_STEP; // K/V rows per thread per tile
    constexpr int Mpad = WM * 16;

    bf16 *Qs = reinterpret_cast<bf16 *>(smem);
    bf16 *Ks = Qs + kMaxRows * D;
    bf16 *Vs = Ks + kStages * kBN * D;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int wm = warp % WM, wk = warp / WM;
    const int G = p.G;

    // ---- Q rows -> shared (cp.async group 0) ----
    for (int idx = tid; idx < Mpad * CPR; idx += kThreads) {
        const int m = idx / CPR, c = idx % CPR;
        const uint32_t dst = rx::smem_u32(Qs + m * D + ((c ^ (m & 7)) * 8));
        if (m < w.M) {
            const int64_t qr = qrow_of<MODE>(p, w, m);
            const bf16 *src = p.q + ((qr * p.hq + (int64_t)g * G + m % G) * D + c * 8);
            rx::cp_async_16(dst, src, 16);
        } else {
            rx::cp_async_16(dst, p.q, 0);
        }
    }

    const int64_t len = w.p1 - w.p0;
    const int n_tiles = (int)((len + kBN - 1) / kBN);
    const int c_ld = tid % CPR, r_ld = tid / CPR;

    int32_t sl[RPT];
    auto load_slots = [&](int tile) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int64_t pos = w.p0 + (int64_t)tile * kBN + r_ld + i * ROW_STEP;
            sl[i] = (pos < w.p1) ? __ldg(w.slots + pos) : -1;
        }
    };
    auto issue = [&](int tile, int stage) {
        bf16 *kd = Ks + stage * kBN * D;
        bf16 *vd = Vs + stage * kBN * D;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = r_ld + i * ROW_STEP;
            const int64_t pos = w.p0 + (int64_t)tile * kBN + r;
            const int32_t s = sl[i];
            const bool inside = pos < w.p1;
            const bool ok = inside && s >= 0 && (int64_t)s < p.num_slots;
            if (inside && !ok && c_ld == 0 && p.status) atomicOr(p.status, RX_DEV_BAD_SLOT);
            const int64_t off = ok ? (((int64_t)s * p.hkv + g) * D + c_ld * 8) : 0;
            const int dsto = r * D + ((c_ld ^ (r & 7)) * 8);
            rx::cp_async_16(rx::smem_u32(kd + dsto), p.k_pool + off, ok ? 16 : 0);
            rx::cp_async_16(rx::smem_u32(vd + dsto), p.v_pool + off, ok ? 16 : 0);
        }
    };

    load_slots(0);
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < n_tiles) issue(s, s);
        rx::cp_async_commit();
        load_slots(s + 1);
    }

    // keys at positions >= lim are masked: the item's end, and for extend rows
    // the causal bound of the row's own token
    int64_t lim0 = w.p1, lim1 = w.p1;
    if (MODE == kExtend) {
        const int r = wm * 16 + gid;
        lim0 = min(w.p1, w.cbase + r / G + 1);
        lim1 = min(w.p1, w.cbase + (r + 8) / G + 1);
    }
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};
    float oacc[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i)
        oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    uint32_t qf[D / 16][4];

    for (int t = 0; t < n_tiles; ++t) {
        rx::cp_async_wait<kStages - 2>();
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int row = wm * 16 + (lane & 15);
                const int ch = ks * 2 + (lane >> 4);
                rx::ldmatrix_x4(rx::smem_u32(Qs + row * D + ((ch ^ (row & 7)) * 8)), qf[ks][0],
                                qf[ks][1], qf[ks][2], qf[ks][3]);
            }
        }
        {
            const int tn = t + kStages - 1;
            if (tn < n_tiles) issue(tn, tn % kStages);
            rx::cp_async_commit();
            load_slots(tn + 1);
        }
        const bf16 *kt = Ks + (t % kStages) * kBN * D;
        const bf16 *vt = Vs + (t % kStages) * kBN * D;

        // S = Q K^T over this warp's KW keys
        float s[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const int key = wk * KW + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4(rx::smem_u32(kt + key * D + ((ch ^ (key & 7)) * 8)), b0, b1, b2, b3);
                rx::mma_bf16_16816(s[2 * np], qf[ks], b0, b1);
                rx::mma_bf16_16816(s[2 * np + 1], qf[ks], b2, b3);
            }
        }
        // scale into the log2 domain; mask keys past each row's bound
        const int64_t kpos0 = w.p0 + (int64_t)t * kBN + wk * KW;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t pos = kpos0 + nt * 8 + tig * 2 + (j & 1);
                const int64_t lim = (j < 2) ? lim0 : lim1;
                s[nt][j] = (pos < lim) ? s[nt][j] * p.scale_log2 : -INFINITY;
            }
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float a0 = rx::fast_exp2(m_r[0] - mu0), a1 = rx::fast_exp2(m_r[1] - mu1);
        m_r[0] = mn0;
        m_r[1] = mn1;
        l_r[0] *= a0;
        l_r[1] *= a1;
#pragma unroll
        for (int i = 0; i < DT; ++i) {
            oacc[i][0] *= a0;
            oacc[i][1] *= a0;
            oacc[i][2] *= a1;
            oacc[i][3] *= a1;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            s[nt][0] = rx::fast_exp2(s[nt][0] - mu0);
            s[nt][1] = rx::fast_exp2(s[nt][1] - mu0);
            s[nt][2] = rx::fast_exp2(s[nt][2] - mu1);
            s[nt][3] = rx::fast_exp2(s[nt][3] - mu1);
            l_r[0] += s[nt][0] + s[nt][1];
            l_r[1] += s[nt][2] + s[nt][3];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            uint32_t a[4];
            a[0] = rx::pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            a[1] = rx::pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            a[2] = rx::pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = rx::pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int key = wk * KW + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                rx::ldmatrix_x4_trans(rx::smem_u32(vt + key * D + ((ch ^ (key & 7)) * 8)), b0, b1,
                                      b2, b3);
                rx::mma_bf16_16816(oacc[2 * dp], a, b0, b1);
                rx::mma_bf16_16816(oacc[2 * dp + 1], a, b2, b3);
            }
        }
    }
    rx::cp_async_wait<0>();
    __syncthreads();

    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 1);
    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 2);
    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 1);
    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 2);

    auto out_offset = [&](int m) -> int64_t {
        return qrow_of<MODE>(p, w, m) * p.hq + (int64_t)g * G + m % G;
    };

    if constexpr (WK == 1) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = wm * 16 + gid + half * 8;
            if (r >= w.M) continue;
            const int64_t orow = out_offset(r);
            const float inv = 1.f / l_r[half];
            if (w.final_) {
                bf16 *dst = p.o + orow * D;
#pragma unroll
                for (int dt = 0; dt < DT; ++dt)
                    *reinterpret_cast<uint32_t *>(dst + dt * 8 + tig * 2) =
                        rx::pack_bf16(oacc[dt][2 * half] * inv, oacc[dt][2 * half + 1] * inv);
                if (p.lse && tig == 0) p.lse[orow] = (m_r[half] + log2f(l_r[half])) * rx::kLn2;
            } else {
                const int64_t prow = orow * p.max_parts + w.part;
                float *dst = p.ws_o + prow * D;
#pragma unroll
                for (int dt = 0; dt < DT; ++dt)
                    *reinterpret_cast<float2 *>(dst + dt * 8 + tig * 2) =
                        make_float2(oacc[dt][2 * half] * inv, oacc[dt][2 * half + 1] * inv);
                if (tig == 0) p.ws_lse[prow] = m_r[half] + log2f(l_r[half]);
            }
        }
    } else {
        // combine the WK key-split partials of each row through shared memory
        float *red_m = reinterpret_cast<float *>(smem);
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
        __syncthreads();
        for (int e = tid; e < Mpad * D; e += kThreads) {
            const int r = e / D, c = e % D;
            if (r >= w.M) continue;
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
            const int64_t orow = out_offset(r);
            if (w.final_) {
                p.o[orow * D + c] = __float2bfloat16_rn(ot / lt);
                if (p.lse && c == 0) p.lse[orow] = (mt + log2f(lt)) * rx::kLn2;
            } else {
                const int64_t prow = orow * p.max_parts + w.part;
                p.ws_o[prow * D + c] = ot / lt;
                if (c == 0) p.ws_lse[prow] = mt + log2f(lt);
            }
        }
    }
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 2) attn_rows_kernel(const Params p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    Work w;
    const int g = blockIdx.y;
    {
        const int b = blockIdx.z;
        const int tb = kMaxRows / p.G;  // tokens per CTA
        const int E = __ldg(p.extend_len + b);
        if (E > (int)gridDim.x * tb) {  // past max_extend_len
            if (p.status && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
                atomicOr(p.status, RX_DEV_BAD_LEN);
            return;
        }
        const int xb = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest rows first
        const int t0 = xb * tb;
        if (t0 >= E) return;
        const int ntok = min(tb, E - t0);
        const int64_t P = __ldg(p.prefix_len + b);
        if (P < 0 || P + E > p.rtt_stride) {  // the slot list cannot hold the context
            if (p.status && threadIdx.x == 0) atomicOr(p.status, RX_DEV_BAD_LEN);
            return;
        }
        w.b = b;
        w.r0 = 0;
        w.M = ntok * p.G;
        w.p0 = 0;
        w.p1 = P + t0 + ntok;
        w.part = 0;
        w.final_ = true;
        w.qbase = (int64_t)__ldg(p.qo_indptr + b) + t0;
        w.cbase = P + t0;
        w.slots = p.rtt + (int64_t)__ldg(p.req_idx + b) * p.rtt_stride;
    }
    if (w.M <= 0 || w.p1 <= w.p0) return;
    if (w.M <= 16)
        attn_rows_body<D, 1, MODE>(p, w, g, smem);
    else if (w.M <= 32)
        attn_rows_body<D, 2, MODE>(p, w, g, smem);
    else
        attn_rows_body<D, 4, MODE>(p, w, g, smem);
}

constexpr size_t smem_bytes(int D) { return (size_t)(kMaxRows + 2 * kStages * kBN) * D * 2; }

template <int D, int MODE>
int launch_rows(const Params &p, dim3 grid, cudaStream_t st)
{
    static bool configured = false;
    if (!configured) {
        RX_CUDA_CHECK(cudaFuncSetAttribute(attn_rows_kernel<D, MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem_bytes(D)));
        configured = true;
    }
    attn_rows_kernel<D, MODE><<<grid, kThreads, smem_bytes(D), st>>>(p);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}

int check_pool(const rx_kv_pool *pool, const char *fn)
{
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0)
        return rx_set_error(RX_ERR_INVALID, "%s: invalid pool", fn);
    if (pool->head_dim != 64 && pool->head_dim != 128)
        return rx_set_error(RX_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 64, 128)", fn,
                            pool->head_dim);
    return RX_OK;
}

}  // namespace

extern "C" int rx_attn_extend(const rx_kv_pool *pool, const void *q, void *o, float *lse,
                              int32_t hq, const int32_t *qo_indptr, const int32_t *req_idx,
                              const int32_t *prefix_len, const int32_t *extend_len,
                              const int32_t *rtt, int64_t rtt_stride, int32_t batch,
                              int32_t max_extend_len, float sm_scale, int32_t *dev_status,
                              void *stream)
{
    int rc = check_pool(pool, "rx_attn_extend");
    if (rc != RX_OK) return rc;
    if (!q || !o || !qo_indptr || !req_idx || !prefix_len || !extend_len || !rtt ||
        rtt_stride <= 0 || batch < 0 || hq <= 0 || max_extend_len < 0 || !(sm_scale > 0.f))
        return rx_set_error(RX_ERR_INVALID, "rx_attn_extend: invalid argument");
    if (hq % pool->num_kv_heads != 0 || 64 % (hq / pool->num_kv_heads) != 0)
        return rx_set_error(RX_ERR_UNSUPPORTED,
                            "rx_attn_extend: %d q heads over %d kv heads (need G | 64)", hq,
                            pool->num_kv_heads);
    if (rx_misaligned16(q) || rx_misaligned16(o) || rx_misaligned16(pool->k) ||
        rx_misaligned16(pool->v) || (reinterpret_cast<uintptr_t>(lse) & 3) != 0)
        return rx_set_error(RX_ERR_INVALID, "rx_attn_extend: q, o and the pools must be 16-byte aligned");
    if (batch == 0 || max_extend_len == 0) return RX_OK;
    const int D = pool->head_dim;
    Params p{};
    p.q = (const bf16 *)q;
    p.o = (bf16 *)o;
    p.lse = lse;
    p.k_pool = (const bf16 *)pool->k;
    p.v_pool = (const bf16 *)pool->v;
    p.num_slots = pool->num_slots;
    p.hq = hq;
    p.hkv = pool->num_kv_heads;
    p.G = hq / pool->num_kv_heads;
    p.req_idx = req_idx;
    p.qo_indptr = qo_indptr;
    p.prefix_len = prefix_len;
    p.extend_len = extend_len;
    p.rtt = rtt;
    p.rtt_stride = rtt_stride;
    p.batch = batch;
    p.scale_log2 = sm_scale * rx::kLog2e;
    p.status = dev_status;
    const int tb = kMaxRows / p.G;
    dim3 grid((unsigned)((max_extend_len + tb - 1) / tb), (unsigned)p.hkv, (unsigned)batch);
    cudaStream_t st = (cudaStream_t)stream;
    return D == 128 ? launch_rows<128, kExtend>(p, grid, st) : launch_rows<64, kExtend>(p, grid, st);
}
