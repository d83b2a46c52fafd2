// rx_kv_store.cu -- scatter of new K/V rows into the token-slot pool.
//
// The pool keeps every finished call's KV so later calls reuse it instead of
// recomputing it ("SGLang: Efficient Execution of Structured Language Model
// Programs", unite.ai, es, section "Introducción a SGLang", RadixAttention
// bullet).  This kernel is the write side: K[slot[i]] = k_new[i] and the same
// for V.  It is a pure HBM copy (read 2*n*row bytes, write as many), so it is
// written as a grid-stride loop of 16-byte vector loads and stores: each
// 16-byte chunk of a row is one thread's work, consecutive threads walk
// consecutive chunks of a row (coalesced on both sides), and the grid is a
// multiple of the SM count.
#include "rx_common.cuh"

namespace {

__global__ void __launch_bounds__(256) kv_store_kernel(const uint4 *__restrict__ k_new,
                                                       const uint4 *__restrict__ v_new,
                                                       const int32_t *__restrict__ slots,
                                                       int64_t n_rows, int64_t chunks_per_row,
                                                       uint4 *__restrict__ k_pool,
                                                       uint4 *__restrict__ v_pool,
                                                       int64_t num_slots, int32_t *status)
{
    const int64_t total = n_rows * chunks_per_row;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * total; i += step) {
        const bool is_v = i >= total;
        const int64_t j = is_v ? i - total : i;
        const int64_t row = j / chunks_per_row;
        const int64_t c = j - row * chunks_per_row;
        const int32_t s = __ldg(slots + row);
        if (s < 0 || (int64_t)s >= num_slots) {
            if (status && c == 0 && !is_v) atomicOr(status, RX_DEV_BAD_SLOT);
            continue;
        }
        const uint4 val = is_v ? __ldg(v_new + j) : __ldg(k_new + j);
        (is_v ? v_pool : k_pool)[(int64_t)s * chunks_per_row + c] = val;
    }
}

// FP8 store: each thread takes 8 bf16 values (16 bytes) of a new row, divides
// them by the pool's scale (correctly rounded fp32 division) and writes their
// E4M3 codes (8 bytes): round to nearest even, magnitudes past 448 saturate.
__global__ void __launch_bounds__(256) kv_store_fp8_kernel(const uint4 *__restrict__ k_new,
                                                           const uint4 *__restrict__ v_new,
                                                           const int32_t *__restrict__ slots,
                                                           int64_t n_rows, int64_t chunks_per_row,
                                                           uint2 *__restrict__ k_pool, uint2 *__restrict__ v_pool,
                                                           int64_t num_slots, float k_scale, float v_scale,
                                                           int32_t *status)
{
    const int64_t total = n_rows * chunks_per_row;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * total; i += step) {
        const bool is_v = i >= total;
        const int64_t j = is_v ? i - total : i;
        const int64_t row = j / chunks_per_row;
        const int64_t c = j - row * chunks_per_row;
        const int32_t s = __ldg(slots + row);
        if (s < 0 || (int64_t)s >= num_slots) {
            if (status && c == 0 && !is_v) atomicOr(status, RX_DEV_BAD_SLOT);
            continue;
        }
        const uint4 val = is_v ? __ldg(v_new + j) : __ldg(k_new + j);
        (is_v ? v_pool : k_pool)[(int64_t)s * chunks_per_row + c] =
            rx::e4m3x8_from_bf16x8(val, is_v ? v_scale : k_scale);
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

}  // namespace

extern "C" int rx_kv_store(const rx_kv_pool *pool_in, const void *k_new, const void *v_new,
                           const int32_t *slots, int64_t n, int32_t *dev_status, void *stream)
{
    rx_kv_pool layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 0, "rx_kv_store")) return rc;
    const rx_kv_pool *pool = pool_in ? &layer_view : nullptr;
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0 ||
        pool->head_dim <= 0 || n < 0 || (n > 0 && (!k_new || !v_new || !slots)))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store: invalid argument");
    const int64_t row_bytes = (int64_t)pool->num_kv_heads * pool->head_dim * 2;
    if (row_bytes % 16 != 0)
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_kv_store: row of %lld bytes is not a multiple of 16",
                            (long long)row_bytes);
    auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
    if (misaligned(pool->k) || misaligned(pool->v) || misaligned(k_new) || misaligned(v_new))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store: pointers must be 16-byte aligned");
    if (n == 0) return RX_OK;
    const int64_t cpr = row_bytes / 16;
    const int64_t work = 2 * n * cpr;
    const int threads = 256;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    kv_store_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, slots, n, cpr, (uint4 *)pool->k,
        (uint4 *)pool->v, pool->num_slots, dev_status);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}

extern "C" int rx_kv_store_fp8(const rx_kv_pool_fp8 *pool_in, const void *k_new, const void *v_new,
                               const int32_t *slots, int64_t n, int32_t *dev_status, void *stream)
{
    rx_kv_pool_fp8 layer_view;
    if (const int rc = rx_pool_layer(pool_in, &layer_view, 1, "rx_kv_store_fp8")) return rc;
    const rx_kv_pool_fp8 *pool = pool_in ? &layer_view : nullptr;
    if (!pool || !pool->k || !pool->v || pool->num_slots <= 0 || pool->num_kv_heads <= 0 ||
        pool->head_dim <= 0 || n < 0 || (n > 0 && (!k_new || !v_new || !slots)) ||
        !(pool->k_scale > 0.f) || !(pool->v_scale > 0.f))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store_fp8: invalid argument");
    const int64_t row_elems = (int64_t)pool->num_kv_heads * pool->head_dim;
    if (row_elems % 8 != 0)
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_kv_store_fp8: a row of %lld values is not a multiple of 8",
                            (long long)row_elems);
    auto misaligned = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
    if (misaligned(pool->k, 8) || misaligned(pool->v, 8) || misaligned(k_new, 16) || misaligned(v_new, 16))
        return rx_set_error(RX_ERR_INVALID, "rx_kv_store_fp8: pools must be 8-byte and new rows 16-byte aligned");
    if (n == 0) return RX_OK;
    const int64_t cpr = row_elems / 8;
    const int64_t work = 2 * n * cpr;
    const int threads = 256;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    kv_store_fp8_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, slots, n, cpr, (uint2 *)pool->k, (uint2 *)pool->v,
        pool->num_slots, pool->k_scale, pool->v_scale, dev_status);
    RX_CUDA_CHECK(cudaGetLastError());
    return RX_OK;
}
