/*
 * oracle/attn_fp64.c -- fp64 CPU oracle for slot-indexed attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py may load this library.  It shares no code,
 * header, table or helper with the CUDA path and includes nothing from it.
 *
 * What it computes is the plain definition, in fp64, from bf16 inputs widened
 * exactly:
 *
 *   KV store  -- the step that places a request's new K/V into the shared pool
 *                so that later calls reuse it ("SGLang: Efficient Execution of
 *                Structured Language Model Programs", unite.ai, section
 *                "Introducción a SGLang", RadixAttention bullet: the KV cache of
 *                finished calls is kept and reused instead of discarded).
 *                pool'[slot[i]] = new[i]; every other slot is unchanged.
 *
 *   Attention -- o = softmax(q K^T * sm_scale + causal mask) V, where row j of
 *                K and V is the pool row named by req_to_token[row][j], for
 *                keys j = kbeg .. kend-1 (the full causal range is 0 .. p for
 *                a query at absolute position p).  For q-head h the kv-head is
 *                h / (Hq / Hkv).  Steps, in this order and nothing else:
 *                  1. g = h / G
 *                  2. s_j = (sum_c q[c] * K[slot_j][g][c]) * sm_scale
 *                  3. m = max_j s_j
 *                  4. w_j = exp(s_j - m)
 *                  5. o[c] = (sum_j w_j * V[slot_j][g][c]) / (sum_j w_j)
 *                  6. lse = m + log(sum_j w_j)
 *                Loops run in ascending j, so the result is deterministic.
 *
 * Parity of every function here is pinned in tests/test_oracle_pins.py
 * (library attention routine, closed forms, invariants, mutation checks).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen_bf16(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* KV store definition.  Returns 0, or -1 when a slot id is out of range
 * (nothing is written then), or -2 when two rows name the same slot. */
int oracle_kv_store(uint16_t *k_pool, uint16_t *v_pool, int64_t num_slots, int hkv, int d,
                    const uint16_t *k_new, const uint16_t *v_new, const int32_t *slots, int64_t n)
{
    int64_t row = (int64_t)hkv * d;
    for (int64_t i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= num_slots)
            return -1;
        for (int64_t j = 0; j < i; ++j)
            if (slots[j] == slots[i])
                return -2;
    }
    for (int64_t i = 0; i < n; ++i) {
        memcpy(k_pool + (int64_t)slots[i] * row, k_new + i * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_pool + (int64_t)slots[i] * row, v_new + i * row, (size_t)row * sizeof(uint16_t));
    }
    return 0;
}

typedef struct {
    const uint16_t *q;
    int hq, hkv, d;
    const uint16_t *k_pool, *v_pool;
    int64_t num_slots;
    const int32_t *rtt;
    int64_t rtt_stride;
    const int32_t *q_row, *kbeg, *kend;
    double sm_scale;
    double *o, *lse;
    int64_t first, last; /* range of (query, head) items for one thread */
    int status;
} job_t;

/* One (query, q-head) item, following steps 1..6 above. */
static int one_item(const job_t *J, int64_t item, double *s, double *acc)
{
    int64_t t = item / J->hq;
    int h = (int)(item % J->hq);
    int G = J->hq / J->hkv;
    int g = h / G;                                           /* step 1 */
    const uint16_t *q = J->q + (t * J->hq + h) * (int64_t)J->d;
    const int32_t *row = J->rtt + (int64_t)J->q_row[t] * J->rtt_stride;
    int64_t j0 = J->kbeg[t], j1 = J->kend[t];
    if (j1 <= j0)
        return -3;
    for (int64_t j = j0; j < j1; ++j) {                      /* step 2 */
        int32_t slot = row[j];
        if (slot < 0 || slot >= J->num_slots)
            return -1;
        const uint16_t *k = J->k_pool + ((int64_t)slot * J->hkv + g) * J->d;
        double dot = 0.0;
        for (int c = 0; c < J->d; ++c)
            dot += widen_bf16(q[c]) * widen_bf16(k[c]);
        s[j - j0] = dot * J->sm_scale;
    }
    double m = s[0];                                         /* step 3 */
    for (int64_t j = j0 + 1; j < j1; ++j)
        if (s[j - j0] > m)
            m = s[j - j0];
    double wsum = 0.0;
    for (int c = 0; c < J->d; ++c)
        acc[c] = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        double w = exp(s[j - j0] - m);                       /* step 4 */
        wsum += w;
        const uint16_t *v = J->v_pool + ((int64_t)row[j] * J->hkv + g) * J->d;
        for (int c = 0; c < J->d; ++c)
            acc[c] += w * widen_bf16(v[c]);
    }
    double *o = J->o + item * (int64_t)J->d;
    for (int c = 0; c < J->d; ++c)                           /* step 5 */
        o[c] = acc[c] / wsum;
    if (J->lse)
        J->lse[item] = m + log(wsum);                        /* step 6 */
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int64_t max_len = 0;
    for (int64_t it = J->first; it < J->last; ++it) {
        int64_t t = it / J->hq;
        if (J->kend[t] - J->kbeg[t] > max_len)
            max_len = J->kend[t] - J->kbeg[t];
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)J->d);
    J->status = (s && acc) ? 0 : -4;
    for (int64_t it = J->first; it < J->last && J->status == 0; ++it)
        J->status = one_item(J, it, s, acc);
    free(s);
    free(acc);
    return NULL;
}

/* Attention over explicit key ranges.
 *   q        bf16 [n_q, hq, d]
 *   q_row    int32 [n_q]  req_to_token row of each query
 *   kbeg/kend int32 [n_q] keys kbeg .. kend-1 of that row (causal: 0 .. p+1)
 *   o        fp64 [n_q, hq, d], lse fp64 [n_q, hq] (may be NULL)
 * Returns 0, -1 (slot out of range), -3 (empty key range), -4 (no memory),
 * -5 (bad head counts). */
int oracle_attention(const uint16_t *q, int64_t n_q, int hq, const uint16_t *k_pool,
                     const uint16_t *v_pool, int64_t num_slots, int hkv, int d,
                     const int32_t *rtt, int64_t rtt_stride, const int32_t *q_row,
                     const int32_t *kbeg, const int32_t *kend, double sm_scale, double *o,
                     double *lse, int n_threads)
{
    if (hkv <= 0 || hq <= 0 || hq % hkv != 0 || d <= 0)
        return -5;
    int64_t items = n_q * hq;
    if (items == 0)
        return 0;
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > items)
        n_threads = (int)items;
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -4;
    }
    for (int i = 0; i < n_threads; ++i) {
        job_t *J = &jobs[i];
        J->q = q;
        J->hq = hq;
        J->hkv = hkv;
        J->d = d;
        J->k_pool = k_pool;
        J->v_pool = v_pool;
        J->num_slots = num_slots;
        J->rtt = rtt;
        J->rtt_stride = rtt_stride;
        J->q_row = q_row;
        J->kbeg = kbeg;
        J->kend = kend;
        J->sm_scale = sm_scale;
        J->o = o;
        J->lse = lse;
        J->first = items * i / n_threads;
        J->last = items * (i + 1) / n_threads;
    }
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[i], NULL, worker, &jobs[i]) == 0)
            started = i;
        else
            break;
    worker(&jobs[0]);
    for (int i = 1; i <= started; ++i)
        pthread_join(th[i], NULL);
    int status = 0;
    for (int i = started + 1; i < n_threads; ++i) /* threads that failed to start run here */
        worker(&jobs[i]);
    for (int i = 0; i < n_threads; ++i)
        if (jobs[i].status != 0)
            status = jobs[i].status;
    free(jobs);
    free(th);
    return status;
}
