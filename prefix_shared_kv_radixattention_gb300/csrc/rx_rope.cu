// rx_rope.cu -- rotary position embedding: in place on query rows, and
// fused into the K side of the slot scatter.
//
// Not from the pages, which do not reach inside the model: it is the
// position encoding that the Llama-family models whose attention shapes the
// workloads take apply to q and k before attention, in its rotate-half
// form.  For a token at position p and c < d/2, with theta_c = base^(-2c/d)
// and a = p * theta_c:
//     x'[c]       = x[c] cos a - x[c + d/2] sin a
//     x'[c + d/2] = x[c + d/2] cos a + x[c] sin a
//
// The work is a copy with a few flops per element, so it is laid out for
// HBM.  A thread takes one token, one group of eight pairs and a run of
// `cpt` chunks of four heads: it forms the eight angles once and for each
// chunk issues all its 16-byte loads (both halves of four heads) before
// rotating and storing them.  Consecutive threads take consecutive groups of
// one head, so the accesses coalesce.
//
// Angles: the host tabulates f_c = theta_c / (2 pi) as a 64-bit binary
// fraction of a turn, F_c = f_c 2^64 (f_c < 1).  Then p F_c mod 2^64 is
// p f_c mod 1 in units of 2^-64 turn, exactly as integer arithmetic wraps,
// so the reduction modulo 2 pi is exact up to the table's rounding (about
// 2^-53 of f_c) at any int32 position; its top 32 bits, read as a signed
// number, are the angle in [-pi, pi) in units of 2^-31 pi, which sincosf
// then takes.  Two integer multiplies a pair -- this GPU runs double
// precision at a small fraction of its fp32 and integer rates.
#include <math.h>

#include <type_traits>

#include "rx_common.cuh"

namespace {

using bf16 = __nv_bfloat16;

constexpr int kMaxHalf = 64;  // head_dim 128

struct RopeTab {
    uint32_t f_hi[kMaxHalf];  // theta_c / (2 pi) as a 64-bit fraction of a turn: high word
    uint32_t f_lo[kMaxHalf];  // low word
};

struct Rot8 {
    float c[8], s[8];
};

__device__ __forceinline__ Rot8 angles(const RopeTab &tab, int32_t pos, int c0)
{
    // |p|, and the sine's sign: a rotation by -a is the one by a with sin negated
    const uint32_t up = pos < 0 ? 0u - (uint32_t)pos : (uint32_t)pos;
    const float sgn = pos < 0 ? -1.f : 1.f;
    constexpr float kTurn = 1.4629180792671596e-9f;  // 2 pi / 2^32
    Rot8 r;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        // bits 32 .. 63 of |p| F_c: the high word of |p| f_lo plus the low
        // word of |p| f_hi (the higher words are whole turns)
        const uint32_t t = __umulhi(up, tab.f_lo[c0 + k]) + up * tab.f_hi[c0 + k];
        const float ar = (float)(int32_t)t * kTurn;  // in [-pi, pi)
        sincosf(ar, &r.s[k], &r.c[k]);
        r.s[k] *= sgn;
    }
    return r;
}

constexpr int kHeadsPerThread = 4;

// rotates eight pairs: lo holds x[c0 .. c0 + 7], hi holds x[c0 + d/2 .. + 7]
__device__ __forceinline__ void rotate(const Rot8 &r, uint4 &lo, uint4 &hi)
{
    uint32_t *pl = reinterpret_cast<uint32_t *>(&lo), *ph = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pl + k));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(ph + k));
        const int e = 2 * k;
        const float l0 = a.x * r.c[e] - b.x * r.s[e], h0 = b.x * r.c[e] + a.x * r.s[e];
        const float l1 = a.y * r.c[e + 1] - b.y * r.s[e + 1], h1 = b.y * r.c[e + 1] + a.y * r.s[e + 1];
        pl[k] = rx::pack_bf16(l0, l1);
        ph[k] = rx::pack_bf16(h0, h1);
    }
}

__global__ void __launch_bounds__(256) rope_kernel(uint4 *__restrict__ x, const int32_t *__restrict__ pos,
                                                   int64_t n, int heads, int D, int cpt, const RopeTab tab)
{
    const int groups = D / 16;          // groups of eight pairs per head
    const int64_t cpr = (int64_t)D / 8;  // 16-byte chunks per head row
    const int hchunks = (heads + kHeadsPerThread - 1) / kHeadsPerThread;
    const int runs = (hchunks + cpt - 1) / cpt;
    const int64_t per_tok = (int64_t)runs * groups;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < n * per_tok; w += step) {
        const int64_t i = w / per_tok;
        const int rem = (int)(w - i * per_tok);
        const int run = rem / groups, gi = rem - run * groups;
        const Rot8 r = angles(tab, __ldg(pos + i), gi * 8);
        uint4 *row = x + i * heads * cpr;
        for (int hc = run * cpt; hc < min(hchunks, (run + 1) * cpt); ++hc) {
        uint4 lo[kHeadsPerThread], hi[kHeadsPerThread];
#pragma unroll
        for (int k = 0; k < kHeadsPerThread; ++k) {
            const int h = hc * kHeadsPerThread + k;
            if (h < heads) {
                lo[k] = row[h * cpr + gi];
                hi[k] = row[h * cpr + groups + gi];
            }
        }
#pragma unroll
        for (int k = 0; k < kHeadsPerThread; ++k) {
            const int h = hc * kHeadsPerThread + k;
            if (h < heads) {
                rotate(r, lo[k], hi[k]);
                row[h * cpr + gi] = lo[k];
                row[h * cpr + groups + gi] = hi[k];
            }
        }
        }
    }
}

// F8: the pools hold E4M3 codes; the rotated K row (rounded to bf16 as
// above) and the V row are stored as rx_kv_store_fp8 stores rows: value /
// scale, correctly rounded, to the nearest code (8 codes per 8 values).
template <bool F8>
__global__ void __launch_bounds__(256) kv_store_rope_kernel(const uint4 *__restrict__ k_new,
                                                            const uint4 *__restrict__ v_new,
                                                            const int32_t *__restrict__ slots,
                                                            const int32_t *__restrict__ pos, int64_t n,
                                                            int hkv, int D, void *__restrict__ k_pool_,
                                                            void *__restrict__ v_pool_, int64_t num_slots,
                                                            int32_t *status, int cpt, const RopeTab tab,
                                                            float k_scale, float v_scale)
{
    using Chunk = std::conditional_t<F8, uint2, uint4>;  // 8 values of the pool
    Chunk *k_pool = static_cast<Chunk *>(k_pool_);
    Chunk *v_pool = static_cast<Chunk *>(v_pool_);
    const int groups = D / 16;
    const int64_t cpr = (int64_t)D / 8;
    const int64_t row_chunks = hkv * cpr;  // one slot row: every kv head
    const int hchunks = (hkv + kHeadsPerThread - 1) / kHeadsPerThread;
    const int runs = (hchunks + cpt - 1) / cpt;
    const int64_t per_tok = (int64_t)runs * groups;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < n * per_tok; w += step) {
        const int64_t i = w / per_tok;
        const int rem = (int)(w - i * per_tok);
        const int run = rem / groups, gi = rem - run * groups;
        const int32_t s = __ldg(slots + i);
        if (s < 0 || (int64_t)s >= num_slots) {
            if (status && rem == 0) atomicOr(status, RX_DEV_BAD_SLOT);
            continue;
        }
        const Rot8 r = angles(tab, __ldg(pos + i), gi * 8);
        const uint4 *ks = k_new + i * row_chunks;
        const uint4 *vs = v_new + i * row_chunks;
        Chunk *kd = k_pool + (int64_t)s * row_chunks;
        Chunk *vd = v_pool + (int64_t)s * row_chunks;
        for (int hc = run * cpt; hc < min(hchunks, (run + 1) * cpt); ++hc) {
        uint4 klo[kHeadsPerThread], khi[kHeadsPerThread], vlo[kHeadsPerThread], vhi[kHeadsPerThread];
#pragma unroll
        for (int k = 0; k < kHeadsPerThread; ++k) {
            const int h = hc * kHeadsPerThread + k;
            if (h < hkv) {
                klo[k] = __ldg(ks + h * cpr + gi);
                khi[k] = __ldg(ks + h * cpr + groups + gi);
                vlo[k] = __ldg(vs + h * cpr + gi);
                vhi[k] = __ldg(vs + h * cpr + groups + gi);
            }
        }
#pragma unroll
        for (int k = 0; k < kHeadsPerThread; ++k) {
            const int h = hc * kHeadsPerThread + k;
            if (h < hkv) {
                rotate(r, klo[k], khi[k]);
                if constexpr (F8) {
                    kd[h * cpr + gi] = rx::e4m3x8_from_bf16x8(klo[k], k_scale);
                    kd[h * cpr + groups + gi] = rx::e4m3x8_from_bf16x8(khi[k], k_scale);
                    vd[h * cpr + gi] = rx::e4m3x8_from_bf16x8(vlo[k], v_scale);
                    vd[h * cpr + groups + gi] = rx::e4m3x8_from_bf16x8(vhi[k], v_scale);
                } else {
                    kd[h * cpr + gi] = klo[k];
                    kd[h * cpr + groups + gi] = khi[k];
                    vd[h * cpr + gi] = vlo[k];
                    vd[h * cpr + groups + gi] = vhi[k];
                }
            }
        }
        }
    }
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

bool make_tab(int D, double base, RopeTab &tab)
{
    if ((D != 64 && D != 128) || !(base > 1.0)) return false;
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    for (int c = 0; c < D / 2; ++c) {
        // f_c < 1 / (2 pi): f_c 2^64 < 2^62, converted exactly from the double
        const double f = pow(base, -2.0 * c / D) / kTwoPi;
        const uint64_t F = (uint64_t)ldexp(f, 64);
        tab.f_hi[c] = (uint32_t)(F >> 32);
        tab.f_lo[c] = (uint32_t)F;
    }
    return true;
}

unsigned grid_for(int64_t work)
{
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    return (unsigned)(blocks > cap ? cap : (blocks < 1 ? 1 : blocks));
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

// head chunks a thread walks: one while that leaves fewer threads than about
// 1024 a SM, else as many as keep that many threads
int chunks_per_thread(int64_t n, int heads, int D)
{
    const int hchunks = (heads + kHeadsPerThread - 1) / kHeadsPerThread;
    const int64_t target = (int64_t)num_sms() * 1024;
    const int64_t one = n * (D / 16) * hchunks;  // threads at one chunk each
    int64_t cpt = (one + target - 1) / target;
    if (cpt < 1) cpt = 1;
    if (cpt > hchunks) cpt = hchunks;
    return (int)cpt;
}

}  // namespace

extern "C" int rx_rope(void *x, const int32_t *pos, int64_t n, int32_t heads, int32_t head_dim, double base,
                       void *stream)
{
    RopeTab tab;
    if (n < 0 || heads <= 0 || (n > 0 && (!x || !pos)))
        return rx_set_error(RX_ERR_INVALID, "rx_rope: invalid argument");
    if (!make_tab(head_dim, base, tab))
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_rope: head_dim %d, base %g (need 64 or 128, base > 1)",
                            head_dim, base);
    if (misaligned(x)) return rx_set_error(RX_ERR_INVALID, "rx_rope: x must be 16-byte aligned");
    if (n == 0) return RX_OK;
    const int cpt = chunks_per_thread(n, heads, head_dim);
    const int hchunks = (heads + kHeadsPerThread - 1) / kHeadsPerThread;
    const int64_t work = n * ((hchunks + cpt - 1) / cpt) * (head_dim / 16);
    rope_kernel<<<grid_for(work), 256, 0, (cudaStream_t)stream>>>((uint4 *)x, pos, n, heads, head_dim, cpt, tab);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}

extern "C" int rx_kv_store_rope(const rx_kv_pool *pool_in, const void *k_new, const void *v_new,
                                const int32_t *slots, const int32_t *pos, int64_t n, double base,
                                int32_t *dev_status, void *stream)
{
    rx_kv_pool layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 0, "rx_kv_store_rope")) return rc;
    const rx_kv_pool *pool = pool_in ? &layer_view : nullptr;
    RopeTab tab;
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0 || n < 0 ||
        (n > 0 && (!k_new || !v_new || !slots || !pos)))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store_rope: invalid argument");
    if (!make_tab(pool->head_dim, base, tab))
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_kv_store_rope: head_dim %d, base %g (need 64 or 128, base > 1)",
                            pool->head_dim, base);
    if (misaligned(pool->k) || misaligned(pool->v) || misaligned(k_new) || misaligned(v_new))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store_rope: pointers must be 16-byte aligned");
    if (n == 0) return RX_OK;
    const int cpt = chunks_per_thread(n, pool->num_kv_heads, pool->head_dim);
    const int hchunks = (pool->num_kv_heads + kHeadsPerThread - 1) / kHeadsPerThread;
    const int64_t work = n * ((hchunks + cpt - 1) / cpt) * (pool->head_dim / 16);
    kv_store_rope_kernel<false><<<grid_for(work), 256, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, slots, pos, n, pool->num_kv_heads, pool->head_dim,
        pool->k, pool->v, pool->num_slots, dev_status, cpt, tab, 1.f, 1.f);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}

extern "C" int rx_kv_store_rope_fp8(const rx_kv_pool_fp8 *pool_in, const void *k_new, const void *v_new,
                                    const int32_t *slots, const int32_t *pos, int64_t n, double base,
                                    int32_t *dev_status, void *stream)
{
    rx_kv_pool_fp8 layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 1, "rx_kv_store_rope_fp8")) return rc;
    const rx_kv_pool_fp8 *pool = pool_in ? &layer_view : nullptr;
    RopeTab tab;
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0 || n < 0 ||
        !(pool->k_scale > 0.f) || !(pool->v_scale > 0.f) || (n > 0 && (!k_new || !v_new || !slots || !pos)))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store_rope_fp8: invalid argument");
    if (!make_tab(pool->head_dim, base, tab))
        return rx_set_error(RX_ERR_UNSUPPORTED,
                            "rx_kv_store_rope_fp8: head_dim %d, base %g (need 64 or 128, base > 1)",
                            pool->head_dim, base);
    if ((reinterpret_cast<uintptr_t>(pool->k) & 7) != 0 || (reinterpret_cast<uintptr_t>(pool->v) & 7) != 0 ||
        misaligned(k_new) || misaligned(v_new))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store_rope_fp8: pools must be 8-byte and new rows 16-byte aligned");
    if (n == 0) return RX_OK;
    const int cpt = chunks_per_thread(n, pool->num_kv_heads, pool->head_dim);
    const int hchunks = (pool->num_kv_heads + kHeadsPerThread - 1) / kHeadsPerThread;
    const int64_t work = n * ((hchunks + cpt - 1) / cpt) * (pool->head_dim / 16);
    kv_store_rope_kernel<true><<<grid_for(work), 256, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, slots, pos, n, pool->num_kv_heads, pool->head_dim,
        pool->k, pool->v, pool->num_slots, dev_status, cpt, tab, pool->k_scale, pool->v_scale);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}
