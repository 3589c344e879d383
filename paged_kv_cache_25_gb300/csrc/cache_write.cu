// Slot-mapped cache write ("Life of a prompt", "Back to the queue, and into
// vLLM proper": every new token's K and V vector is appended into the next
// free slot of its sequence's blocks).
//
// One thread moves one 16-byte chunk of one (token, kv head) row for both K
// and V: consecutive threads cover consecutive chunks of a row, so the reads
// of k/v and the writes into the pool are fully coalesced 16-byte accesses.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                   uint4* __restrict__ kc, uint4* __restrict__ vc,
                   const int64_t* __restrict__ slots, int64_t total, int n_kv, int block_size,
                   int chunks_per_row, int64_t num_slots, unsigned* err)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t row = i / chunks_per_row;       // (token, head) row
    const int c = static_cast<int>(i - row * chunks_per_row);
    const int64_t t = row / n_kv;
    const int h = static_cast<int>(row - t * n_kv);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return;                          // padding token
    if (slot >= num_slots) {
        set_error(err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int64_t b = slot / block_size, o = slot - b * block_size;
    const int64_t dst = ((b * n_kv + h) * block_size + o) * chunks_per_row + c;
    const uint4 kx = __ldcs(k + i);               // read once: streaming
    const uint4 vx = __ldcs(v + i);
    kc[dst] = kx;
    vc[dst] = vx;
}

cudaError_t launch_cache_write(const void* k, const void* v, void* kc, void* vc,
                               const int64_t* slots, int T, const pa_cache_desc& c,
                               unsigned* err, cudaStream_t s)
{
    const int cpr = c.head_dim * elem_bytes(c.dtype) / 16;
    const int64_t total = static_cast<int64_t>(T) * c.n_kv_heads * cpr;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    cache_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(kc),
        static_cast<uint4*>(vc), slots, total, c.n_kv_heads, c.block_size, cpr,
        static_cast<int64_t>(c.num_blocks) * c.block_size, err);
    return cudaGetLastError();
}

}  // namespace pa
