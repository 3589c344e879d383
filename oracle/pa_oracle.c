/*
 * CPU fp64 oracle for the paged-attention path.  TEST INFRASTRUCTURE ONLY:
 * see pa_oracle.h for the citations and the rule on who may call it.
 *
 * Plain loops, no blocking, no fusion, no reordering beyond the definitions.
 * Compiled with -ffp-contract=off so that x86 and Arm give identical bits.
 */
#include "pa_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ sizes */

int64_t orc_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int elem_bytes)
{
    /* the leading 2: one K and one V vector per KV head per layer */
    return (int64_t)2 * n_layers * n_kv_heads * head_dim * elem_bytes;
}

int64_t orc_blocks_for_tokens(int64_t tokens, int block_size)
{
    return (tokens + block_size - 1) / block_size;
}

int64_t orc_pool_blocks(int64_t pool_bytes, int block_size, int64_t bytes_per_token)
{
    return pool_bytes / ((int64_t)block_size * bytes_per_token);
}

/* -------------------------------------------------------------- allocator */

struct orc_alloc {
    int n;          /* physical blocks in the pool */
    int *queue;     /* ring buffer of free block ids, head first */
    int head;
    int count;
    int *ref;       /* reference count per block; 0 = free */
};

orc_alloc* orc_alloc_create(int num_blocks, const int32_t* initial_order)
{
    orc_alloc* a = (orc_alloc*)calloc(1, sizeof(orc_alloc));
    a->n = num_blocks;
    a->queue = (int*)malloc(sizeof(int) * (size_t)(num_blocks > 0 ? num_blocks : 1));
    a->ref = (int*)calloc((size_t)(num_blocks > 0 ? num_blocks : 1), sizeof(int));
    for (int i = 0; i < num_blocks; ++i)
        a->queue[i] = initial_order ? initial_order[i] : i;
    a->head = 0;
    a->count = num_blocks;
    return a;
}

int orc_alloc_take(orc_alloc* a, int n, int32_t* out)
{
    if (n > a->count) return -1;
    for (int i = 0; i < n; ++i) {
        int id = a->queue[a->head];
        a->head = (a->head + 1) % a->n;
        a->count -= 1;
        a->ref[id] = 1;
        out[i] = id;
    }
    return 0;
}

void orc_alloc_share(orc_alloc* a, const int32_t* ids, int n)
{
    for (int i = 0; i < n; ++i) a->ref[ids[i]] += 1;
}

void orc_alloc_release(orc_alloc* a, const int32_t* ids, int n)
{
    for (int i = 0; i < n; ++i) {
        int id = ids[i];
        a->ref[id] -= 1;
        if (a->ref[id] == 0) {          /* back to the tail of the queue, at once */
            a->queue[(a->head + a->count) % a->n] = id;
            a->count += 1;
        }
    }
}

int orc_alloc_num_free(const orc_alloc* a) { return a->count; }
int orc_alloc_refcount(const orc_alloc* a, int id) { return a->ref[id]; }

void orc_alloc_destroy(orc_alloc* a)
{
    if (!a) return;
    free(a->queue);
    free(a->ref);
    free(a);
}

int orc_build_tables(orc_alloc* a, int B, const int32_t* lens, const uint8_t* sharer,
                     int prefix_tokens, int block_size, int max_blocks, int32_t* tables)
{
    int n_prefix = 0, any_sharer = 0;
    int32_t* prefix = NULL;
    for (int s = 0; s < B; ++s)
        if (sharer && sharer[s]) any_sharer = 1;
    for (int64_t i = 0; i < (int64_t)B * max_blocks; ++i) tables[i] = -1;
    if (any_sharer && prefix_tokens > 0) {
        n_prefix = prefix_tokens / block_size;   /* the prefix is whole blocks */
        prefix = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_prefix);
        if (orc_alloc_take(a, n_prefix, prefix) != 0) { free(prefix); return -1; }
    }
    int first_sharer = 1;
    for (int s = 0; s < B; ++s) {
        int need = (int)orc_blocks_for_tokens(lens[s], block_size);
        int32_t* row = tables + (int64_t)s * max_blocks;
        int own_from = 0;
        if (prefix && sharer[s]) {
            for (int j = 0; j < n_prefix; ++j) row[j] = prefix[j];
            if (!first_sharer) orc_alloc_share(a, prefix, n_prefix);
            first_sharer = 0;
            own_from = n_prefix;
        }
        if (need > max_blocks) { free(prefix); return -1; }
        if (need > own_from && orc_alloc_take(a, need - own_from, row + own_from) != 0) {
            free(prefix);
            return -1;
        }
    }
    free(prefix);
    return 0;
}

void orc_slot_mapping(const int32_t* tables, int max_blocks, int block_size,
                      const int32_t* seq, const int32_t* pos, int T, int64_t* slots)
{
    for (int t = 0; t < T; ++t) {
        int32_t phys = tables[(int64_t)seq[t] * max_blocks + pos[t] / block_size];
        slots[t] = (int64_t)phys * block_size + pos[t] % block_size;
    }
}

/* ------------------------------------------------------ cache write, gather */

void orc_cache_write(uint8_t* k_cache, uint8_t* v_cache, const uint8_t* k, const uint8_t* v,
                     const int64_t* slots, int T, int num_blocks, int n_kv, int block_size,
                     int head_dim, int elem_bytes)
{
    size_t row = (size_t)head_dim * elem_bytes;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        int64_t b = slot / block_size, o = slot % block_size;
        if (b >= num_blocks) continue;
        for (int h = 0; h < n_kv; ++h) {
            size_t dst = (((size_t)b * n_kv + h) * block_size + (size_t)o) * row;
            size_t src = ((size_t)t * n_kv + h) * row;
            memcpy(k_cache + dst, k + src, row);
            memcpy(v_cache + dst, v + src, row);
        }
    }
}

void orc_cache_write_vt(uint8_t* v_cache, const uint8_t* v, const int64_t* slots, int T,
                        int num_blocks, int n_kv, int block_size, int head_dim, int elem_bytes,
                        int piece)
{
    const int pieces = block_size / piece;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        int64_t b = slot / block_size, o = slot % block_size;
        if (b >= num_blocks) continue;
        for (int h = 0; h < n_kv; ++h)
            for (int i = 0; i < head_dim; ++i) {
                size_t dst = (((((size_t)b * n_kv + h) * pieces + (size_t)(o / piece)) * head_dim +
                               (size_t)i) * piece + (size_t)(o % piece)) * elem_bytes;
                size_t src = (((size_t)t * n_kv + h) * head_dim + (size_t)i) * elem_bytes;
                memcpy(v_cache + dst, v + src, (size_t)elem_bytes);
            }
    }
}

void orc_copy_blocks(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k, uint8_t* dst_v,
                     const int32_t* map, int n, int64_t block_bytes)
{
    for (int i = 0; i < n; ++i) {
        int64_t s = map[2 * i], d = map[2 * i + 1];
        memmove(dst_k + d * block_bytes, src_k + s * block_bytes, (size_t)block_bytes);
        memmove(dst_v + d * block_bytes, src_v + s * block_bytes, (size_t)block_bytes);
    }
}

void orc_gather(const uint8_t* cache, const int32_t* table, int L, int n_kv, int block_size,
                int head_dim, int elem_bytes, uint8_t* out)
{
    size_t row = (size_t)head_dim * elem_bytes;
    for (int p = 0; p < L; ++p) {
        int64_t b = table[p / block_size];
        int o = p % block_size;
        for (int h = 0; h < n_kv; ++h)
            memcpy(out + ((size_t)p * n_kv + h) * row,
                   cache + (((size_t)b * n_kv + h) * block_size + (size_t)o) * row, row);
    }
}

/* ------------------------------------------------------------ fp8 e4m3 */

double orc_fp8_e4m3_decode(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 0xF, m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);          /* subnormal: m/8 * 2^(1-7) */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The 127 non-negative finite code values, in code order (strictly
 * increasing; a pin checks it), built once from the decoder. */
static double g_fp8_vals[0x7F];
static pthread_once_t g_fp8_once = PTHREAD_ONCE_INIT;

static void fp8_build_table(void)
{
    for (int c = 0; c <= 0x7E; ++c) g_fp8_vals[c] = orc_fp8_e4m3_decode((uint8_t)c);
}

uint8_t orc_fp8_e4m3_encode(float xf)
{
    double x = (double)xf;
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;           /* the sign bit, so -0.0 -> 0x80 */
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);        /* saturate */
    /* nearest of the 127 non-negative finite codes, ties to the even code:
     * the two codes around a (vals[lo] <= a < vals[lo + 1]) by bisection over
     * the increasing values, then the nearer of the two */
    pthread_once(&g_fp8_once, fp8_build_table);
    int lo = 0, hi = 0x7E;                                /* vals[lo] <= a < vals[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_fp8_vals[mid] <= a) lo = mid; else hi = mid;
    }
    double d_lo = a - g_fp8_vals[lo], d_hi = g_fp8_vals[hi] - a;
    int best = d_lo < d_hi ? lo : (d_hi < d_lo ? hi : ((lo & 1) == 0 ? lo : hi));
    return (uint8_t)(sign | best);
}

typedef struct { const float* x; int64_t b, e; float scale; uint8_t* out; } q_job_t;

static void* quantize_worker(void* arg)
{
    q_job_t* j = (q_job_t*)arg;
    for (int64_t i = j->b; i < j->e; ++i) {
        float q = j->x[i] / j->scale;                      /* fp32 division */
        j->out[i] = orc_fp8_e4m3_encode(q);
    }
    return NULL;
}

void orc_quantize_fp8(const float* x, int64_t n, float scale, uint8_t* out)
{
    /* element-wise, so the work is split in contiguous ranges over threads */
    int nt = n >= (1 << 20) ? 16 : 1;
    pthread_t th[16];
    q_job_t jobs[16];
    for (int t = 0; t < nt; ++t) {
        jobs[t].x = x; jobs[t].scale = scale; jobs[t].out = out;
        jobs[t].b = n * t / nt; jobs[t].e = n * (t + 1) / nt;
        if (nt == 1) quantize_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, quantize_worker, &jobs[t]);
    }
    if (nt > 1)
        for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
}

void orc_dequantize_fp8(const uint8_t* code, int64_t n, double scale, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_e4m3_decode(code[i]) * scale;
}

/* -------------------------------------------------------------- attention */

/* One query row against rows 0..n-1 of one K/V head:
 *   z_p = scale * sum_i q_i K_p,i ;  w = exp(z - max z) / sum exp(z - max z) ;
 *   out = sum_p w_p V_p
 * K_p,i = K[(p * kv_stride) + i], likewise V. */
static void attend_row(double* out, const double* q, const double* K, const double* V,
                       size_t kv_stride, int n, int d, double scale, double* z)
{
    double m = -INFINITY;
    for (int p = 0; p < n; ++p) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += q[i] * K[(size_t)p * kv_stride + i];
        z[p] = scale * acc;
        if (z[p] > m) m = z[p];
    }
    double denom = 0.0;
    for (int p = 0; p < n; ++p) {
        z[p] = exp(z[p] - m);
        denom += z[p];
    }
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    for (int p = 0; p < n; ++p) {
        double w = z[p] / denom;
        for (int i = 0; i < d; ++i) out[i] += w * V[(size_t)p * kv_stride + i];
    }
}

typedef struct {
    /* shared */
    double* out; const double* q; const double* K; const double* V;
    const int64_t* q_start; const int32_t* chunk;
    const int64_t* kv_start; const int32_t* lens;
    int n_seq, n_q, n_kv, d; double scale;
    int prefill;
    /* work split */
    int64_t n_items; int nthreads; int tid;
} job_t;

static void* worker(void* arg)
{
    job_t* j = (job_t*)arg;
    int g = j->n_q / j->n_kv;
    size_t kv_stride = (size_t)j->n_kv * j->d;
    int max_len = 0;
    for (int s = 0; s < j->n_seq; ++s) if (j->lens[s] > max_len) max_len = j->lens[s];
    double* z = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    for (int64_t it = j->tid; it < j->n_items; it += j->nthreads) {
        if (!j->prefill) {
            int s = (int)(it / j->n_q), h = (int)(it % j->n_q), kvh = h / g;
            const double* Ks = j->K + (size_t)j->kv_start[s] * kv_stride + (size_t)kvh * j->d;
            const double* Vs = j->V + (size_t)j->kv_start[s] * kv_stride + (size_t)kvh * j->d;
            size_t qo = ((size_t)s * j->n_q + h) * j->d;
            attend_row(j->out + qo, j->q + qo, Ks, Vs, kv_stride, j->lens[s], j->d, j->scale, z);
        } else {
            /* items: (request, query row within its chunk, head) flattened per request */
            int64_t rem = it;
            int r = 0;
            while (rem >= (int64_t)j->chunk[r] * j->n_q) { rem -= (int64_t)j->chunk[r] * j->n_q; ++r; }
            int i = (int)(rem / j->n_q), h = (int)(rem % j->n_q), kvh = h / g;
            int pos = j->lens[r] - j->chunk[r] + i;       /* absolute position of the query */
            const double* Ks = j->K + (size_t)j->kv_start[r] * kv_stride + (size_t)kvh * j->d;
            const double* Vs = j->V + (size_t)j->kv_start[r] * kv_stride + (size_t)kvh * j->d;
            size_t qo = ((size_t)(j->q_start[r] + i) * j->n_q + h) * j->d;
            attend_row(j->out + qo, j->q + qo, Ks, Vs, kv_stride, pos + 1, j->d, j->scale, z);
        }
    }
    free(z);
    return NULL;
}

static void run_jobs(job_t base, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        pthread_create(&th[t], NULL, worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
}

void orc_decode(double* out, const double* q, const double* K, const double* V,
                const int64_t* kv_start, const int32_t* lens, int B, int n_q, int n_kv,
                int head_dim, double scale, int nthreads)
{
    job_t j;
    memset(&j, 0, sizeof(j));
    j.out = out; j.q = q; j.K = K; j.V = V; j.kv_start = kv_start; j.lens = lens;
    j.n_seq = B; j.n_q = n_q; j.n_kv = n_kv; j.d = head_dim; j.scale = scale;
    j.prefill = 0;
    j.n_items = (int64_t)B * n_q;
    run_jobs(j, nthreads);
}

void orc_prefill(double* out, const double* q, const int64_t* q_start, const int32_t* chunk,
                 const double* K, const double* V, const int64_t* kv_start, const int32_t* lens,
                 int R, int n_q, int n_kv, int head_dim, double scale, int nthreads)
{
    job_t j;
    memset(&j, 0, sizeof(j));
    j.out = out; j.q = q; j.K = K; j.V = V; j.q_start = q_start; j.chunk = chunk;
    j.kv_start = kv_start; j.lens = lens;
    j.n_seq = R; j.n_q = n_q; j.n_kv = n_kv; j.d = head_dim; j.scale = scale;
    j.prefill = 1;
    int64_t rows = 0;
    for (int r = 0; r < R; ++r) rows += chunk[r];
    j.n_items = rows * n_q;
    run_jobs(j, nthreads);
}
