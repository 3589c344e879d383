// pa_decode_no_alloc: decode with the split-K scratch held inside the library.
//
// Some callers cannot allocate device memory for the decode's workspace: a
// host runtime that hands all free HBM to its KV block pool at start-up and
// gives plugins no allocator, or a latency-critical loop that cannot afford
// cudaMalloc's device-wide synchronisation.  This entry point takes the same
// inputs and outputs as pa_decode but keeps the scratch in one fixed-size
// device array declared below, so it allocates nothing.
//
// The array lives on every GPU that loads the library, until the process
// exits.  All calls share it and it keeps the previous call's contents; the
// one word that must start at zero (the decode's work counter, for batches
// large enough to use one) is cleared on the stream by every call that uses
// it, and every partial the reduce reads is written earlier in the same call.  Calls whose work overlaps on the GPU (different
// streams, or several host threads) race on it.
#include <mutex>

#include "pa_internal.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device.  Host code only
// sees a host-side stand-in under the array's name, so the real address is
// looked up once per device, with that device current.
pa_status scratch_address(void** out)
{
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pa::cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return pa::fail(PA_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return pa::cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
        addr[dev] = p;
    }
    *out = addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype, const void* q,
                                        const void* k_cache, const void* v_cache,
                                        const pa_cache_desc* cache, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* context_lens,
                                        int num_seqs, int n_q_heads, float scale, int block_size,
                                        void* stream)
{
    if (!cache) return pa::fail(PA_ERR_INVALID_ARG, "cache descriptor is NULL");
    if (num_seqs > 0 && max_blocks_per_seq > 0 && block_size > 0) {
        const int64_t max_ctx = static_cast<int64_t>(max_blocks_per_seq) * block_size;
        if (max_ctx <= (1 << 30)) {
            const size_t need = pa_decode_workspace_size(num_seqs, n_q_heads, cache->n_kv_heads,
                                                         cache->head_dim, block_size,
                                                         static_cast<int>(max_ctx));
            if (need > PA_DECODE_NO_ALLOC_SCRATCH_BYTES)
                return pa::fail(PA_ERR_WORKSPACE,
                                "this batch needs %zu bytes of scratch; the library's fixed "
                                "scratch holds %zu (use pa_decode with a caller workspace)",
                                need, (size_t)PA_DECODE_NO_ALLOC_SCRATCH_BYTES);
        }
    }
    void* scratch = nullptr;
    const pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    return pa_decode(out, out_dtype, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, n_q_heads, scale, block_size, scratch,
                     PA_DECODE_NO_ALLOC_SCRATCH_BYTES, stream);
}
