/*
 * pa.h - C ABI of the GB300 paged-attention library (libpa.so).
 *
 * The operations follow the pages' statement of the problem:
 *   "vLLM Serving - PagedAttention, Continuous Batching, and Production
 *   Tuning", sections "PagedAttention in depth" (fixed-size KV blocks in one
 *   pool, a per-sequence block table mapping logical to physical blocks) and
 *   "How the attention kernel actually reads paged blocks" (the kernel takes
 *   the block table as input, looks a block up once per block, computes q.k
 *   against the keys of that block and accumulates the softmax-weighted sum of
 *   the values of the same block);
 *   "Life of a prompt", section "Back to the queue, and into vLLM proper"
 *   (each decode step appends one K and one V row into the next free slot, a
 *   fresh block every block_size tokens, a FIFO free-block queue);
 *   "The hands-on guide to LLM Inference with vLLM", chunked prefill (each
 *   chunk attends over every earlier cached token plus itself).
 *
 * Conventions for every call below:
 *   - Device pointers are owned by the caller; the library allocates nothing
 *     on the device.  Scratch space ("workspace") is passed in by the caller and
 *     sized with the *_workspace_size queries.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All device work is enqueued asynchronously on it.
 *   - Argument checks happen on the host before any launch.  A failed check
 *     returns a status other than PA_OK and launches nothing;
 *     pa_last_error_message() then describes it.
 *   - Data errors only visible on the device (a block id outside [0,
 *     num_blocks), a slot beyond the pool) set a sticky device error word and
 *     skip the affected unit of work (its outputs are then unspecified).  No
 *     kernel traps or asserts.  Read and clear the word with
 *     pa_get_device_error().
 *   - Every wait inside a kernel is bounded in time; a wait that runs out sets
 *     PA_ERR_TIMEOUT in the device error word and the kernel returns.
 *
 * KV cache layout (one transformer layer, K and V in separate tensors):
 *   k_cache, v_cache : [num_blocks][n_kv_heads][block_size][head_dim], row-major.
 *   The token at logical position p of sequence s lives in physical block
 *   block_tables[s][p / block_size], row p % block_size.  Its slot number is
 *   physical_block * block_size + p % block_size.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* a pointer, size or shape check failed          */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim, block size) */
    PA_ERR_OUT_OF_RANGE = 3,  /* device: block id or slot outside the pool       */
    PA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required      */
    PA_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out                  */
    PA_ERR_CUDA = 6           /* a CUDA runtime call failed                      */
} pa_status;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* Shape of one layer's paged K/V pool.  head_dim in {64, 128} and block_size
 * in {16, 32} run on the tensor-core paths; fp32 pools run on a CUDA-core
 * path.  n_kv_heads >= 1.
 * FP8 pools ("The hands-on guide to LLM Inference with vLLM", KV footprint:
 * 1 byte per element if the cache is quantized to FP8; head_dim 64 or 128):
 * dtype PA_FP8_E4M3,
 * each stored code c means decode_e4m3(c) * k_scale for K (v_scale for V);
 * act_dtype (PA_BF16 or PA_F16) is the dtype of q and of the K/V rows given
 * to pa_reshape_and_cache_quant.  The three fields are ignored otherwise.
 * In FP8 pools the V codes of each 16-token piece of a (block, KV head) are
 * stored transposed, v_cache [num_blocks][n_kv_heads][block_size / 16]
 * [head_dim][16]: the code of slot offset o, element i sits at
 * [b][h][o / 16][i][o % 16].  A piece (head_dim x 16 codes) is contiguous, so
 * the kernels fetch it with one bulk copy, and a 16-byte row holds the 16
 * tokens of one head-dim element, the order the P.V fragments use; K keeps
 * the layout above. */
typedef struct {
    int num_blocks;
    int block_size;
    int n_kv_heads;
    int head_dim;
    pa_dtype dtype;
    float k_scale;
    float v_scale;
    pa_dtype act_dtype;
} pa_cache_desc;

/* ---------------------------------------------------------------- cache write
 * Append K/V rows into their slots ("Life of a prompt": one new K and V
 * vector per token go into the next free slot of the sequence's blocks).
 *   k, v          : [num_tokens][n_kv_heads][head_dim], contiguous, cache dtype
 *                   (for FP8 pools: E4M3 codes, copied as they are; the V codes
 *                   land in the pool's transposed V layout described above).
 *   k_cache/v_cache: pools as in the layout above; written in place.
 *   slot_mapping  : int64 [num_tokens] on the device.  slot < 0 means "skip this
 *                   token" (padding).  slot >= num_blocks*block_size sets
 *                   PA_ERR_OUT_OF_RANGE on the device and the token is skipped.
 *                   Two tokens with one slot: the winner is unspecified.
 * Only the addressed rows of the pools change, bit for bit.  Pointers must be
 * 16-byte aligned.  num_tokens == 0 is a no-op. */
pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens,
                               const pa_cache_desc* cache, void* stream);

/* Cache write with conversion: k, v are [num_tokens][n_kv_heads][head_dim] in
 * in_dtype (PA_F32, PA_F16 or PA_BF16).  Into an FP8 pool each element is
 * stored as the E4M3 code of fp32(x) / k_scale (v_scale for V), the division
 * IEEE-rounded in fp32, the code rounded to nearest even and saturated to
 * +-448.  Into a pool of in_dtype it is pa_reshape_and_cache.  Other pairs
 * return PA_ERR_UNSUPPORTED.  Slot rules as for pa_reshape_and_cache. */
pa_status pa_reshape_and_cache_quant(const void* k, const void* v, pa_dtype in_dtype,
                                     void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens,
                                     const pa_cache_desc* cache, void* stream);

/* ---------------------------------------------------------------- decode
 * One query row per sequence ("Life of a prompt", "The decode stage"):
 *   out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s
 * over the context_lens[s] logical rows of sequence s, read through its block
 * table ("How the attention kernel actually reads paged blocks").  Query head
 * h reads KV head h / (n_q_heads / n_kv_heads) (grouped-query attention).
 *   out          : [num_seqs][n_q_heads][head_dim] in out_dtype.
 *   q            : [num_seqs][n_q_heads][head_dim], cache dtype.
 *   block_tables : int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(len / block_size) are never read.
 *   context_lens : int32 [num_seqs]; the count includes the newest token
 *                  (append it with pa_reshape_and_cache first).  Each must be in
 *                  [1, max_blocks_per_seq * block_size]: the host cannot check
 *                  device values, so a length outside that range is a caller
 *                  error (rows past the table are clamped away; length 0 gives
 *                  undefined output for that sequence).
 *   block_size   : must equal cache->block_size.
 *   workspace    : device scratch of at least pa_decode_workspace_size(...)
 *                  bytes for the same shapes, 256-byte aligned; its contents
 *                  need no initialisation.  It holds the work counter of the
 *                  persistent decode kernel (reset on the stream by each call
 *                  that uses one; batches of a few units per resident thread
 *                  block are dealt round robin and use none) and, for long
 *                  contexts split over several thread blocks,
 *                  the partial results the second kernel combines.  Calls that
 *                  overlap on the GPU must not share one workspace.
 * n_q_heads must be a multiple of n_kv_heads.  Accumulation is fp32.
 * FP8 pools: q is in cache->act_dtype; K/V codes are widened exactly to fp16
 * and q is rounded to fp16 for the tensor-core products (exact for bf16 q of
 * magnitude in [2^-14, 65504]); the scales multiply the scores and the output. */
pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q,
                    const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int n_q_heads,
                    float scale, int block_size,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace pa_decode needs for sequences of at most max_context_len
 * tokens (pass max_blocks_per_seq * block_size of the tables you will pass);
 * at least 256. */
size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                                int block_size, int max_context_len);

/* ---------------------------------------------------------------- multi-query decode
 * Verification of k drafted tokens in one pass ("vLLM Serving ...",
 * "Speculative decoding"; "Inference engineering", Trick 5: the target model
 * checks all k guesses in one forward pass): every sequence brings q_per_seq
 * = k + 1 query rows whose K/V rows were appended first, so
 *   out[s][i][h] = softmax(scale * q[s][i][h] . K_s[0..p]^T) V_s[0..p],
 *   p = context_lens[s] - q_per_seq + i      (causal among the new rows).
 * The g query heads of a KV head and the q_per_seq rows form (head, query)
 * rows of one tensor-core tile, so each K/V slab is still read once for all
 * of them.
 *   out, q       : [num_seqs][q_per_seq][n_q_heads][head_dim] (out in out_dtype,
 *                  q in the cache dtype, or cache->act_dtype for FP8 pools).
 *   context_lens : include the q_per_seq new rows; a length below q_per_seq
 *                  flags PA_ERR_OUT_OF_RANGE in the device error word and the
 *                  sequence's rows are not written.
 *   workspace    : pa_decode_verify_workspace_size(...) bytes, as for pa_decode.
 * q_per_seq in [1, 16]; q_per_seq = 1 is pa_decode.  bf16/fp16/FP8 pools with
 * head_dim 64 or 128 (else PA_ERR_UNSUPPORTED); other rules as pa_decode. */
pa_status pa_decode_verify(void* out, pa_dtype out_dtype, const void* q,
                           const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int q_per_seq,
                           int n_q_heads, float scale, int block_size,
                           void* workspace, size_t workspace_bytes, void* stream);
size_t pa_decode_verify_workspace_size(int num_seqs, int q_per_seq, int n_q_heads,
                                       int n_kv_heads, int head_dim, int block_size,
                                       int max_context_len);

/* ---------------------------------------------------------------- decode, no allocation
 * The paper has no counterpart to this call.  It is pa_decode for callers that
 * cannot allocate device memory: a host runtime that gives all free HBM to its
 * KV block pool at start-up and offers plugins no allocator, or a
 * latency-critical loop that cannot pay for cudaMalloc's device-wide
 * synchronisation.  Inputs and outputs are exactly those of pa_decode; the
 * split-K scratch is a fixed array of PA_DECODE_NO_ALLOC_SCRATCH_BYTES inside
 * the library, present on every GPU that loads it until the process exits.
 *   - Allocates nothing (no cudaMalloc/cudaFree, no allocating library call).
 *   - A batch whose pa_decode_workspace_size(...) exceeds the fixed size is
 *     rejected with PA_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device looks up the array's device address (a
 *     one-time set-up per device); make that first call before any stream
 *     capture.
 *   - All calls share the array and it keeps the last call's contents; what
 *     must start at zero (the work counter, when the batch uses one) is
 *     cleared on the stream by every call that uses it.  Calls that overlap on
 *     the GPU (other streams, other host threads) race on it: serialise them. */
#define PA_DECODE_NO_ALLOC_SCRATCH_BYTES (16u << 20)
pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype, const void* q,
                             const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int num_seqs, int n_q_heads,
                             float scale, int block_size, void* stream);

/* ---------------------------------------------------------------- chunked prefill
 * A chunk of C_r new query rows of request r attends causally over the paged
 * context ("The hands-on guide ...", chunked prefill): query row i sits at
 * absolute position context_lens[r] - C_r + i and attends logical rows
 * 0 .. that position.  The chunk's own K/V must already be in the pool
 * (pa_reshape_and_cache).  With no earlier context it is ordinary causal
 * prefill of the whole prompt.
 *   out, q          : [total_q][n_q_heads][head_dim], request r's rows start at
 *                     query_start_loc[r]; out in out_dtype, q in the cache
 *                     dtype (FP8 pools: in cache->act_dtype).
 *   query_start_loc : int32 [num_reqs + 1] on the device, non-decreasing,
 *                     query_start_loc[0] = 0; C_r = difference of neighbours.
 *   context_lens    : int32 [num_reqs] on the device: total tokens L_r of
 *                     request r including the chunk (C_r <= L_r).
 *   max_query_len   : host value >= every C_r (sizes the grid).  A request
 *                     with C_r > max_query_len sets PA_ERR_OUT_OF_RANGE in the
 *                     device error word (its rows past max_query_len are not
 *                     written).
 *   workspace       : reserved; pass NULL / 0 (pa_prefill_workspace_size is 0).
 * bf16, fp16 and FP8 E4M3 pools (f32 pools return PA_ERR_UNSUPPORTED).  FP8
 * pools keep V transposed per 16-token piece as for decode; their codes are
 * widened exactly to fp16 on chip (every E4M3 value is an fp16 value) and the
 * scales are folded into the softmax scale (k_scale) and the output (v_scale). */
pa_status pa_prefill_chunk(void* out, pa_dtype out_dtype, const void* q,
                           const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* query_start_loc, const int32_t* context_lens,
                           int num_reqs, int max_query_len, int n_q_heads,
                           float scale, int block_size,
                           void* workspace, size_t workspace_bytes, void* stream);

size_t pa_prefill_workspace_size(int num_reqs, int n_q_heads, int head_dim, int total_q);

/* ---------------------------------------------------------------- block copies
 * Copy-on-write ("vLLM Serving ...", "Sharing and copy-on-write": a sharer
 * that diverges gets a copy of the one shared block it writes to, then its
 * block table points at the copy).  For i < num_pairs, every K and V row of
 * physical block block_mapping[2i] (all KV heads) is copied over block
 * block_mapping[2i+1] of the same pools.
 *   block_mapping : int32 [num_pairs][2] (source, destination), device-readable.
 * Every source block is read as it was before the call; a destination must not
 * also be a source in the same call (the copies run in parallel).  An id
 * outside [0, num_blocks) sets PA_ERR_OUT_OF_RANGE on the device and that pair
 * is skipped. */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc* cache,
                         const int32_t* block_mapping, int num_pairs, void* stream);

/* Swap ("vLLM Serving ...", "The scheduler: waiting, running, swapped": the
 * blocks of a preempted sequence move to a pool in CPU memory and come back
 * when it resumes).  Copies whole blocks from one pool pair to another of the
 * same layout (layout->num_blocks is ignored; the two sizes are given).  Either
 * side may be device memory or page-locked host memory mapped into the GPU's
 * address space (cudaHostAlloc / cudaMallocHost, or registered as mapped), so
 * one call moves many blocks with no per-block cudaMemcpy.  Same mapping rules
 * as pa_copy_blocks; ids are checked against each side's block count. */
pa_status pa_swap_blocks(const void* src_k, const void* src_v, int src_num_blocks,
                         void* dst_k, void* dst_v, int dst_num_blocks,
                         const pa_cache_desc* layout, const int32_t* block_mapping,
                         int num_pairs, void* stream);

/* ---------------------------------------------------------------- errors
 * Synchronizes `stream`, returns the device error word (PA_OK if clean) and
 * clears it.  The word is per device and shared by every stream. */
pa_status pa_get_device_error(void* stream);
const char* pa_status_string(pa_status status);
/* Text of the last host-side failure on the calling thread ("" if none). */
const char* pa_last_error_message(void);

/* Self-test of the bounded waits: launches one thread that waits on an
 * mbarrier nothing ever completes.  After limit_us (1 .. 2e6) the wait gives up,
 * PA_ERR_TIMEOUT is recorded in the device error word and the kernel writes 2
 * to *scratch (a device word) and returns; the context stays usable.  Read the
 * outcome with pa_get_device_error. */
pa_status pa_selftest_bounded_wait(unsigned limit_us, void* scratch, void* stream);

/* Measurement hook: when both are non-NULL, pa_decode records `start` right
 * before its main attention kernel and `stop` right after it on the call's
 * stream (cudaEvent_t passed as void*).  Pass NULL, NULL to turn it off. */
void pa_set_profile_events(void* start, void* stop);

/* ---------------------------------------------------------------- host allocator
 * The free-block queue and page tables of "Life of a prompt" ("Back to the
 * queue, and into vLLM proper"): a FIFO queue of free physical block ids, a
 * reference count per block for sharing ("Sharing and copy-on-write"), blocks
 * returned to the tail of the queue the moment their count reaches zero.
 * Host memory only; not thread-safe (one owner thread). */
typedef struct pa_alloc pa_alloc;
/* initial_order: the queue's starting order (a permutation of 0..n-1), or NULL
 * for 0..n-1.  Returns NULL on bad arguments. */
pa_alloc* pa_alloc_create(int num_blocks, const int32_t* initial_order);
/* Takes n blocks from the head of the queue into out (refcount 1 each).
 * Returns 0, or -1 (nothing taken) if fewer than n are free. */
int  pa_alloc_blocks(pa_alloc* a, int n, int32_t* out);
/* Adds one reference to each listed block (another table points at it). */
void pa_alloc_share(pa_alloc* a, const int32_t* ids, int n);
/* Drops one reference from each listed block; a block reaching zero goes back
 * to the tail of the queue. */
void pa_alloc_free(pa_alloc* a, const int32_t* ids, int n);
int  pa_alloc_num_free(const pa_alloc* a);
int  pa_alloc_refcount(const pa_alloc* a, int block_id);
void pa_alloc_destroy(pa_alloc* a);

/* Builds block tables for a batch, sequences in order, ceil(len/block_size)
 * blocks each.  Sequences flagged in `sharer` (may be NULL) point their first
 * prefix_tokens/block_size entries at one set of prefix blocks taken once,
 * before any sequence, and shared (refcount = number of sharers);
 * prefix_tokens must be a multiple of block_size.  Unused entries are -1.
 * tables: int32 [num_seqs][max_blocks_per_seq] host memory. */
pa_status pa_alloc_build_tables(pa_alloc* a, int num_seqs, const int32_t* lens,
                                const uint8_t* sharer, int prefix_tokens, int block_size,
                                int max_blocks_per_seq, int32_t* tables);

/* Host: slots[t] = tables[seq[t]][pos[t] / block_size] * block_size
 *                  + pos[t] % block_size.  Returns PA_ERR_INVALID_ARG if a
 * position falls outside the table or on an unused (-1) entry. */
pa_status pa_slot_mapping(const int32_t* tables, int max_blocks_per_seq, int block_size,
                          const int32_t* seq, const int32_t* pos, int num_tokens,
                          int64_t* slots);

/* ---------------------------------------------------------------- prefix cache
 * Automatic reuse of computed K/V blocks across requests ("The hands-on guide
 * to LLM Inference with vLLM", Automatic Prefix Caching; "vLLM Serving ...",
 * "Prefix caching (automatic KV reuse)"; "Inference engineering", Trick 3):
 *  - only full blocks are cached; a block's fingerprint chains the fingerprint
 *    of the block before it (0 for the first) with its block_size token ids:
 *    FNV-1a 64 over the parent (8 bytes, little endian), then each token id
 *    (4 bytes, little endian).  An entry also keeps the parent fingerprint and
 *    the tokens, so a hit always means equal contents;
 *  - a request reuses the leading run of its full blocks that hit; every block
 *    counts the requests using it;
 *  - a block whose count drops to zero keeps its entry on an LRU list; new
 *    blocks come from the free queue first and, only when it is empty, by
 *    evicting the least recently released cached block (blocks released in
 *    one call count as released deepest first).
 * Host memory only; not thread-safe (one owner thread).  Block ids are the
 * pool's physical blocks, the same ids pa_decode's tables hold. */
typedef struct pa_prefix pa_prefix;
/* free_order: the free queue's starting order (a permutation of
 * 0..num_blocks-1) or NULL.  Returns NULL on bad arguments. */
pa_prefix* pa_prefix_create(int num_blocks, int block_size, const int32_t* free_order);
void pa_prefix_destroy(pa_prefix* p);
/* Fingerprint of one full block of block_size tokens after `parent`. */
uint64_t pa_prefix_block_hash(uint64_t parent, const int32_t* tokens, int block_size);
/* Number of leading full blocks of tokens[0..n_tokens) already cached (no
 * change to the cache), or -1 on bad arguments. */
int pa_prefix_lookup(const pa_prefix* p, const int32_t* tokens, int n_tokens);
/* Block table for a request of n_tokens >= 1 tokens: its hitting leading full
 * blocks (one more reference each), then ceil(n_tokens / block_size) - hits
 * new blocks; entries past those up to table_len are set to -1.  Returns the
 * number of hit blocks (their K/V need not be recomputed), -1 when the pool
 * cannot supply the new blocks (nothing taken), -2 on bad arguments. */
int pa_prefix_acquire(pa_prefix* p, const int32_t* tokens, int n_tokens, int32_t* table,
                      int table_len);
/* n more blocks for growing sequences (reference count 1 each).  Returns 0,
 * -1 when the pool cannot supply them (nothing taken), -2 on bad arguments. */
int pa_prefix_alloc(pa_prefix* p, int n, int32_t* out);
/* Registers the full blocks of a request whose K/V have been written: for
 * block i < n_tokens / block_size, table[i] is entered unless the same
 * contents are cached already (then table[i] stays private).  Every listed
 * full block must be held (count > 0).  Returns the number of blocks entered,
 * or -2 on bad arguments (nothing entered). */
int pa_prefix_commit(pa_prefix* p, const int32_t* tokens, int n_tokens, const int32_t* table);
/* Drops one reference from each listed block (-1 entries skipped).  Returns 0,
 * or -2 (nothing changed) on an id out of range or a block without enough
 * references. */
int pa_prefix_release(pa_prefix* p, const int32_t* table, int n_blocks);
int pa_prefix_num_free(const pa_prefix* p);       /* free, not cached */
int pa_prefix_num_evictable(const pa_prefix* p);  /* cached, count 0 */
int pa_prefix_num_cached(const pa_prefix* p);     /* entries in the table */
int pa_prefix_refcount(const pa_prefix* p, int block);

/* Sizing ("vLLM Serving ...", "How big is the KV cache?"):
 * 2 * n_layers * n_kv_heads * head_dim * elem_bytes, and the number of whole
 * blocks of block_size tokens that fit in pool_bytes. */
int64_t pa_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int elem_bytes);
int64_t pa_pool_blocks(int64_t pool_bytes, int block_size, int64_t bytes_per_token);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
