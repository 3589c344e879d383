/*
 * CPU fp64 oracle for the paged-attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path includes, links or
 * calls this code; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no source, header, table or helper with the
 * CUDA library.
 *
 * Each function restates one definition from the pages, cited by page title
 * and section:
 *   [KVsize]   "vLLM Serving - PagedAttention, Continuous Batching, and
 *              Production Tuning", section "How big is the KV cache?"
 *   [Blocks]   same page, "PagedAttention in depth" (block table diagram,
 *              30-token example) and "Worked memory example"
 *   [Queue]    "Life of a prompt", section "Back to the queue, and into vLLM
 *              proper" (free block queue, page table, a new block every 16
 *              tokens, blocks returned immediately)
 *   [Sharing]  "vLLM Serving ...", "Sharing and copy-on-write" (several
 *              block tables point at one physical block; reference counts;
 *              a sharer that diverges gets a copy of that one block) and
 *              "The scheduler: waiting, running, swapped" (blocks of preempted
 *              sequences move to CPU memory and back)
 *   [Detour]   "Life of a prompt", sections "The detour, what really happens
 *              inside one forward pass" and "The decode stage" (softmax of
 *              Q K^T, times V; one query row per decode step; K/V appended)
 *   [Kernel]   "vLLM Serving ...", "How the attention kernel actually reads
 *              paged blocks" (block table lookup per block; result is the same
 *              attention as over a contiguous tensor)
 *   [Chunked]  "The hands-on guide to LLM Inference with vLLM", chunked
 *              prefill: each chunk attends to every earlier cached token
 *   [Quant]    same guide, KV cache footprint ("1 if you quantize the cache
 *              to FP8") and "vLLM Serving ...", quantization (--kv-cache-dtype
 *              fp8 roughly doubles KV capacity)
 *
 * Values are read as their stored numbers converted exactly to double.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* [KVsize] bytes/token = 2 * n_layers * n_kv_heads * d_head * dtype_bytes */
int64_t orc_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int elem_bytes);
/* [Blocks] a sequence of L tokens occupies ceil(L / block_size) blocks */
int64_t orc_blocks_for_tokens(int64_t tokens, int block_size);
/* [Blocks] free pool bytes / bytes per block, rounded down */
int64_t orc_pool_blocks(int64_t pool_bytes, int block_size, int64_t bytes_per_token);

/* [Queue]+[Sharing] FIFO free-block queue with per-block reference counts. */
typedef struct orc_alloc orc_alloc;
orc_alloc* orc_alloc_create(int num_blocks, const int32_t* initial_order);
int  orc_alloc_take(orc_alloc* a, int n, int32_t* out);        /* 0 ok, -1 not enough */
void orc_alloc_share(orc_alloc* a, const int32_t* ids, int n);  /* refcount += 1 */
void orc_alloc_release(orc_alloc* a, const int32_t* ids, int n);/* refcount -= 1; at 0 back to the tail */
int  orc_alloc_num_free(const orc_alloc* a);
int  orc_alloc_refcount(const orc_alloc* a, int id);
void orc_alloc_destroy(orc_alloc* a);

/* Block tables for a batch, taken from the queue in sequence order.  The first
 * `prefix_tokens` tokens of every sequence flagged in `sharer` map to one set of
 * prefix blocks taken once (before any sequence) and shared by all sharers.
 * Unused table entries hold -1.  Returns 0, or -1 if the pool ran out. */
int orc_build_tables(orc_alloc* a, int B, const int32_t* lens, const uint8_t* sharer,
                     int prefix_tokens, int block_size, int max_blocks, int32_t* tables);

/* [Queue]/[Blocks] slot of logical position pos of sequence seq:
 * physical block * block_size + offset within the block. */
void orc_slot_mapping(const int32_t* tables, int max_blocks, int block_size,
                      const int32_t* seq, const int32_t* pos, int T, int64_t* slots);

/* [Detour] append: copy the bytes of each token's K and V row into its slot of
 * the [num_blocks][n_kv][block_size][d] pools; a negative slot is skipped. */
void orc_cache_write(uint8_t* k_cache, uint8_t* v_cache, const uint8_t* k, const uint8_t* v,
                     const int64_t* slots, int T, int num_blocks, int n_kv, int block_size,
                     int head_dim, int elem_bytes);

/* Same append for a V pool stored transposed per piece of `piece` tokens of
 * a (block, head): [num_blocks][n_kv][block_size / piece][head_dim][piece],
 * i.e. element i of the row that goes to slot (b, o) lands at
 * [b][h][o / piece][i][o % piece].  piece divides block_size; piece =
 * block_size is the whole block transposed. */
void orc_cache_write_vt(uint8_t* v_cache, const uint8_t* v, const int64_t* slots, int T,
                        int num_blocks, int n_kv, int block_size, int head_dim, int elem_bytes,
                        int piece);

/* [Sharing] copy-on-write / swap: for i < n, copy the whole physical block
 * map[i][0] of the source pools (all KV heads, all rows, K and V) over block
 * map[i][1] of the destination pools.  Every source block is read as it was
 * before the call (callers pass copies of the source pools), so the order of
 * the pairs does not matter; a destination must not also be a source of the
 * same call when the pools are the same.
 * block_bytes = n_kv * block_size * head_dim * elem_bytes. */
void orc_copy_blocks(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k, uint8_t* dst_v,
                     const int32_t* map, int n, int64_t block_bytes);

/* [Quant] FP8 E4M3 cache: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits, subnormals, largest finite 448, no infinities, NaN = all exponent and
 * mantissa bits set.  Encoding rounds the magnitude to nearest, ties to even,
 * saturates it to 448, and copies the sign bit of x: -0.0, and a negative
 * value whose magnitude rounds to zero, give the negative-zero code 0x80, as
 * IEEE rounding of a signed value does.  NaN gives 0x7F (the pages fix no NaN
 * code; the tests never write one).  A cache value is encode(x / scale) with
 * the division in fp32; its meaning is decode(code) * scale. */
uint8_t orc_fp8_e4m3_encode(float x);
double  orc_fp8_e4m3_decode(uint8_t code);
void    orc_quantize_fp8(const float* x, int64_t n, float scale, uint8_t* out);
void    orc_dequantize_fp8(const uint8_t* code, int64_t n, double scale, double* out);

/* [Kernel] logical row p of a sequence lives in block table[p / bs], offset
 * p % bs; copy rows 0..L-1 out as a contiguous [L][n_kv][d] array. */
void orc_gather(const uint8_t* cache, const int32_t* table, int L, int n_kv, int block_size,
                int head_dim, int elem_bytes, uint8_t* out);

/* [Detour] decode: out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s over the
 * L_s logical rows of sequence s, K/V head = h / (n_q / n_kv).
 * q [B][n_q][d]; K, V packed [sum L][n_kv][d] with sequence s at row kv_start[s];
 * out [B][n_q][d]. */
void orc_decode(double* out, const double* q, const double* K, const double* V,
                const int64_t* kv_start, const int32_t* lens, int B, int n_q, int n_kv,
                int head_dim, double scale, int nthreads);

/* [Chunked] query row i of request r sits at absolute position
 * L_r - C_r + i and attends logical rows 0..that position.
 * q packed [sum C][n_q][d] (request r at row q_start[r]); K, V packed
 * [sum L][n_kv][d] (request r at row kv_start[r]); out like q. */
void orc_prefill(double* out, const double* q, const int64_t* q_start, const int32_t* chunk,
                 const double* K, const double* V, const int64_t* kv_start, const int32_t* lens,
                 int R, int n_q, int n_kv, int head_dim, double scale, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
