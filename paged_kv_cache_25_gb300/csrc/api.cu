// C-ABI entry points: argument checks, workspace carving, tensor maps, the
// device error word and launches.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// ------------------------------------------------------------------ messages
static thread_local char g_msg[512] = "";

pa_status fail(pa_status st, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

pa_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static pa_status ok()
{
    g_msg[0] = '\0';
    return PA_OK;
}

// ------------------------------------------------------------------ error word
__device__ unsigned g_device_error;

static constexpr int kMaxDevices = 64;

unsigned* device_error_word()
{
    static std::mutex mu;
    static unsigned* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned*>(p);
    }
    return addr[dev];
}

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

pa_status encode_pool_map(CUtensorMap* map, const void* base, pa_dtype dt, int head_dim,
                          uint64_t rows, int box_x, int box_y, int swizzle)
{
    auto fn = encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const CUtensorMapDataType t =
        dt == PA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                     : (dt == PA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * elem_bytes(dt)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, t, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                         : (swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                          : CU_TENSOR_MAP_SWIZZLE_NONE),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

// ------------------------------------------------------------------ profiling hook
static std::atomic<cudaEvent_t> g_prof_start{nullptr}, g_prof_stop{nullptr};

void profile_events(cudaEvent_t* start, cudaEvent_t* stop)
{
    *start = g_prof_start.load();
    *stop = g_prof_stop.load();
    if (!*start || !*stop) *start = *stop = nullptr;
}

// ------------------------------------------------------------------ partition policy
int decode_partition_tokens(int64_t seq_groups, int block_size, int max_context_len)
{
    // 1024 tokens (64 or 32 blocks) per partition spreads the fixed cost of a
    // unit (block ids, q fragments, the first TMA round trip, the cross-warp
    // combine) over 16 stages per warp and keeps the split-K bytes below 1 %;
    // halve it (down to 128) while the batch would offer fewer than ~300 units
    // (about one per resident CTA at 2 per SM on 152 SMs): smaller units cost
    // more in per-unit overhead and split-K traffic than they win in balance
    // (a 64-sequence TinyLlama-shaped batch, 3 CTAs per SM: the decode kernel
    // at 0.378 of the copy peak with a bound of 608 units, 0.394 with 300,
    // 0.340 with 1216).
    int p = 1024;
    while (p > 128 && p > block_size &&
           seq_groups * ((max_context_len + p - 1) / p) < 300)
        p /= 2;
    return p;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// need_act: the call reads q in act_dtype (decode); a cache write names its
// input dtype itself and ignores act_dtype.
static pa_status check_cache(const pa_cache_desc* c, bool need_act = true)
{
    if (!c) return fail(PA_ERR_INVALID_ARG, "cache descriptor is NULL");
    if (c->dtype != PA_F32 && c->dtype != PA_F16 && c->dtype != PA_BF16 && c->dtype != PA_FP8_E4M3)
        return fail(PA_ERR_INVALID_ARG, "unknown cache dtype %d", (int)c->dtype);
    if (c->dtype == PA_FP8_E4M3) {
        if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || !std::isfinite(c->k_scale) ||
            !std::isfinite(c->v_scale))
            return fail(PA_ERR_INVALID_ARG, "FP8 pools need finite positive k_scale and v_scale");
        if (need_act && c->act_dtype != PA_BF16 && c->act_dtype != PA_F16)
            return fail(PA_ERR_INVALID_ARG, "FP8 pools need act_dtype PA_BF16 or PA_F16");
    }
    if (c->num_blocks <= 0 || c->n_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "num_blocks and n_kv_heads must be positive");
    if (c->block_size != 16 && c->block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d not supported (16 or 32)", c->block_size);
    if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 96 && c->head_dim != 128 &&
        c->head_dim != 256)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not supported (32/64/96/128/256)", c->head_dim);
    if (static_cast<int64_t>(c->num_blocks) * c->n_kv_heads * c->block_size >= (1ll << 31))
        return fail(PA_ERR_UNSUPPORTED, "pool has 2^31 or more rows");
    return PA_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace: a 256-byte control area (the decode's work counter), then, when
// some sequence can span several partitions, (m, l) [B][n_q][J][2] and the
// partial outputs [B][n_q][J][D], all fp32.
static constexpr size_t kControlBytes = 256;

static size_t decode_ws_bytes(int B, int nq, int n_q, int n_kv, int D, int BS, int max_ctx,
                              int* part, int* parts)
{
    // work units per partition index: (sequence, KV head, 8-row sub-group)
    const int64_t groups = static_cast<int64_t>(B) * n_kv * ((n_q / n_kv * nq + 7) / 8);
    int p = decode_partition_tokens(groups, BS, max_ctx);
    // several query rows a sequence (16-row units): each unit's combine and
    // partials cost more, so large batches take 2048-token partitions
    // (Llama-3-8B batch verifying 3 drafts: 0.837 -> 0.906 of the copy peak)
    if (nq > 1 && p == 1024 && groups * ((max_ctx + 2047) / 2048) >= 300) p = 2048;
    const int J = (max_ctx + p - 1) / p;
    if (part) *part = p;
    if (parts) *parts = J < 1 ? 1 : J;
    if (J <= 1) return kControlBytes;
    const size_t units = static_cast<size_t>(B) * nq * n_q * J;
    return kControlBytes + align256(units * 2 * sizeof(float)) + units * D * sizeof(float);
}

// One thread waits on an mbarrier that nothing ever completes: the bounded
// wait gives up after limit_ns, records PA_ERR_TIMEOUT and the kernel returns.
__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned* err, unsigned* reached)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const bool ok = mbar_wait(b, 0, err, limit_ns);
    *reached = ok ? 1u : 2u;   // 2: the wait ran out and the kernel went on
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_last_error_message(void) { return g_msg; }

const char* pa_status_string(pa_status st)
{
    switch (st) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
    }
    return "PA_ERR_UNKNOWN";
}

void pa_set_profile_events(void* start, void* stop)
{
    g_prof_start.store(static_cast<cudaEvent_t>(start));
    g_prof_stop.store(static_cast<cudaEvent_t>(stop));
}

pa_status pa_selftest_bounded_wait(unsigned limit_us, void* scratch, void* stream)
{
    if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 3u) != 0)
        return fail(PA_ERR_INVALID_ARG, "scratch must be a 4-byte aligned device word");
    if (limit_us == 0 || limit_us > 2000000u)
        return fail(PA_ERR_INVALID_ARG, "limit_us must be in [1, 2e6]");
    unsigned* err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot locate the device error word");
    selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint64_t>(limit_us) * 1000u, err, static_cast<unsigned*>(scratch));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return ok();
}

pa_status pa_get_device_error(void* stream)
{
    unsigned* w = device_error_word();
    if (!w) return fail(PA_ERR_CUDA, "cannot locate the device error word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned v = 0;
    e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (v != 0) {
        e = cudaMemset(w, 0, sizeof v);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    }
    return static_cast<pa_status>(v);
}

pa_status pa_reshape_and_cache_quant(const void* k, const void* v, pa_dtype in_dtype,
                                     void* k_cache, void* v_cache, const int64_t* slot_mapping,
                                     int num_tokens, const pa_cache_desc* cache, void* stream)
{
    pa_status st = check_cache(cache, false);
    if (st != PA_OK) return st;
    if (in_dtype == cache->dtype)
        return pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_tokens, cache, stream);
    if (cache->dtype != PA_FP8_E4M3 ||
        (in_dtype != PA_F32 && in_dtype != PA_F16 && in_dtype != PA_BF16))
        return fail(PA_ERR_UNSUPPORTED, "cache write from dtype %d into dtype %d", (int)in_dtype,
                    (int)cache->dtype);
    if (cache->head_dim != 64 && cache->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "FP8 pools take head_dim 64 or 128");
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return ok();
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "k, v and the pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
    unsigned* err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot locate the device error word");
    cudaError_t e = launch_cache_write_fp8(k, v, in_dtype, k_cache, v_cache, slot_mapping,
                                           num_tokens, *cache, err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cache write launch");
    return ok();
}

pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens,
                               const pa_cache_desc* cache, void* stream)
{
    pa_status st = check_cache(cache, false);
    if (st != PA_OK) return st;
    if (cache->dtype == PA_FP8_E4M3 && cache->head_dim != 64 && cache->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "FP8 pools take head_dim 64 or 128");
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return ok();
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "k, v and the pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
    unsigned* err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot locate the device error word");
    // FP8 pools keep V transposed per 16-token piece of a block: the rows
    // (codes already) go through the FP8 writer, which copies them and lays V
    // out that way
    cudaError_t e = cache->dtype == PA_FP8_E4M3
                        ? launch_cache_write_fp8(k, v, PA_FP8_E4M3, k_cache, v_cache, slot_mapping,
                                                 num_tokens, *cache, err,
                                                 static_cast<cudaStream_t>(stream))
                        : launch_cache_write(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                             *cache, err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cache write launch");
    return ok();
}

pa_status pa_swap_blocks(const void* src_k, const void* src_v, int src_num_blocks, void* dst_k,
                         void* dst_v, int dst_num_blocks, const pa_cache_desc* layout,
                         const int32_t* block_mapping, int num_pairs, void* stream)
{
    if (!layout) return fail(PA_ERR_INVALID_ARG, "layout descriptor is NULL");
    pa_cache_desc c = *layout;
    c.num_blocks = src_num_blocks > 0 ? src_num_blocks : 1;
    pa_status st = check_cache(&c);
    if (st != PA_OK) return st;
    if (num_pairs < 0 || src_num_blocks < 0 || dst_num_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_pairs == 0) return ok();
    if (num_pairs > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 block pairs per call");
    if (!src_k || !src_v || !dst_k || !dst_v || !block_mapping)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v) ||
        (reinterpret_cast<uintptr_t>(block_mapping) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARG, "pools must be 16-byte and the mapping 8-byte aligned");
    unsigned* err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot locate the device error word");
    cudaError_t e = launch_copy_blocks(src_k, src_v, src_num_blocks, dst_k, dst_v, dst_num_blocks,
                                       *layout, block_mapping, num_pairs, err,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block copy launch");
    return ok();
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc* cache,
                         const int32_t* block_mapping, int num_pairs, void* stream)
{
    if (!cache) return fail(PA_ERR_INVALID_ARG, "cache descriptor is NULL");
    return pa_swap_blocks(k_cache, v_cache, cache->num_blocks, k_cache, v_cache, cache->num_blocks,
                          cache, block_mapping, num_pairs, stream);
}

size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                                int block_size, int max_context_len)
{
    if (num_seqs <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_context_len <= 0)
        return 0;
    if (n_q_heads % n_kv_heads != 0) return 0;
    return decode_ws_bytes(num_seqs, 1, n_q_heads, n_kv_heads, head_dim, block_size,
                           max_context_len, nullptr, nullptr);
}

size_t pa_decode_verify_workspace_size(int num_seqs, int q_per_seq, int n_q_heads, int n_kv_heads,
                                       int head_dim, int block_size, int max_context_len)
{
    if (num_seqs <= 0 || q_per_seq <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_context_len <= 0 || n_q_heads % n_kv_heads != 0)
        return 0;
    return decode_ws_bytes(num_seqs, q_per_seq, n_q_heads, n_kv_heads, head_dim, block_size,
                           max_context_len, nullptr, nullptr);
}

static pa_status decode_common(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                               const void* v_cache, const pa_cache_desc* cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int q_per_seq,
                               int n_q_heads, float scale, int block_size, void* workspace,
                               size_t workspace_bytes, void* stream)
{
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (num_seqs == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences per call");
    if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16)
        return fail(PA_ERR_INVALID_ARG, "unknown out_dtype %d", (int)out_dtype);
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(block_tables) || !aligned16(context_lens))
        return fail(PA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    if (block_size != cache->block_size)
        return fail(PA_ERR_INVALID_ARG, "block_size %d != cache block_size %d", block_size,
                    cache->block_size);
    if (n_q_heads <= 0 || n_q_heads % cache->n_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "n_q_heads %d is not a positive multiple of n_kv_heads %d",
                    n_q_heads, cache->n_kv_heads);
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be > 0");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size > (1 << 30))
        return fail(PA_ERR_UNSUPPORTED, "max context above 2^30 tokens");
    if (cache->dtype == PA_FP8_E4M3 && cache->head_dim != 64 && cache->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "FP8 pools decode with head_dim 64 or 128");

    const int max_ctx = max_blocks_per_seq * block_size;
    int part = 0, parts = 0;
    const size_t need = decode_ws_bytes(num_seqs, q_per_seq, n_q_heads, cache->n_kv_heads,
                                        cache->head_dim, block_size, max_ctx, &part, &parts);
    if (parts > 65535) return fail(PA_ERR_UNSUPPORTED, "too many partitions per sequence");
    if (!workspace || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(PA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    unsigned* err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot locate the device error word");

    DecodeArgs a{};
    a.out = out; a.out_dtype = out_dtype; a.q = q;
    a.k_cache = k_cache; a.v_cache = v_cache; a.cache = *cache;
    a.block_tables = block_tables; a.max_blocks = max_blocks_per_seq;
    a.context_lens = context_lens; a.num_seqs = num_seqs; a.n_q = n_q_heads; a.scale = scale;
    a.q_per_seq = q_per_seq;
    a.part_tokens = part; a.max_parts = parts; a.err = err;
    a.ticket = static_cast<unsigned*>(workspace);
    if (need > kControlBytes) {
        const size_t units = static_cast<size_t>(num_seqs) * q_per_seq * n_q_heads * parts;
        char* base = static_cast<char*>(workspace) + kControlBytes;
        a.ws_ml = reinterpret_cast<float*>(base);
        a.ws_acc = reinterpret_cast<float*>(base + align256(units * 2 * sizeof(float)));
    }
    cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ok();
}

pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                    const void* v_cache, const pa_cache_desc* cache, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                    int n_q_heads, float scale, int block_size, void* workspace,
                    size_t workspace_bytes, void* stream)
{
    return decode_common(out, out_dtype, q, k_cache, v_cache, cache, block_tables,
                         max_blocks_per_seq, context_lens, num_seqs, 1, n_q_heads, scale,
                         block_size, workspace, workspace_bytes, stream);
}

pa_status pa_decode_verify(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                           const void* v_cache, const pa_cache_desc* cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int q_per_seq,
                           int n_q_heads, float scale, int block_size, void* workspace,
                           size_t workspace_bytes, void* stream)
{
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (q_per_seq < 1 || q_per_seq > 16)
        return fail(PA_ERR_INVALID_ARG, "q_per_seq %d outside [1, 16]", q_per_seq);
    if (cache->dtype == PA_F32 || (cache->head_dim != 64 && cache->head_dim != 128))
        return fail(PA_ERR_UNSUPPORTED,
                    "multi-query decode runs on bf16/fp16/FP8 pools with head_dim 64 or 128");
    return decode_common(out, out_dtype, q, k_cache, v_cache, cache, block_tables,
                         max_blocks_per_seq, context_lens, num_seqs, q_per_seq, n_q_heads, scale,
                         block_size, workspace, workspace_bytes, stream);
}

size_t pa_prefill_workspace_size(int num_reqs, int n_q_heads, int head_dim, int total_q)
{
    (void)num_reqs; (void)n_q_heads; (void)head_dim; (void)total_q;
    return 0;
}

pa_status pa_prefill_chunk(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                           const void* v_cache, const pa_cache_desc* cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* query_start_loc, const int32_t* context_lens,
                           int num_reqs, int max_query_len, int n_q_heads, float scale,
                           int block_size, void* workspace, size_t workspace_bytes, void* stream)
{
    (void)workspace; (void)workspace_bytes;
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (num_reqs < 0 || max_query_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_reqs == 0 || max_query_len == 0) return ok();
    if (cache->dtype == PA_F32)
        return fail(PA_ERR_UNSUPPORTED, "chunked prefill runs on bf16/fp16/FP8 pools only");
    if (cache->head_dim != 64 && cache->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "chunked prefill supports head_dim 64 and 128");
    if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16)
        return fail(PA_ERR_INVALID_ARG, "unknown out_dtype %d", (int)out_dtype);
    if (!out || !q || !k_cache || !v_cache || !block_tables || !query_start_loc || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(block_tables) || !aligned16(query_start_loc) || !aligned16(context_lens))
        return fail(PA_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
    if (block_size != cache->block_size)
        return fail(PA_ERR_INVALID_ARG, "block_size %d != cache block_size %d", block_size,
                    cache->block_size);
    if (n_q_heads <= 0 || n_q_heads % cache->n_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "n_q_heads %d is not a positive multiple of n_kv_heads %d",
                    n_q_heads, cache->n_kv_heads);
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be > 0");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
    if (num_reqs > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 requests per call");
    unsigned* err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot locate the device error word");
    PrefillArgs a{};
    a.out = out; a.out_dtype = out_dtype; a.q = q;
    a.k_cache = k_cache; a.v_cache = v_cache; a.cache = *cache;
    a.block_tables = block_tables; a.max_blocks = max_blocks_per_seq;
    a.q_start = query_start_loc; a.context_lens = context_lens;
    a.num_reqs = num_reqs; a.max_q = max_query_len; a.n_q = n_q_heads; a.scale = scale;
    a.err = err;
    cudaError_t e = launch_prefill_tc(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

}  // extern "C"
