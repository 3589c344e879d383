// Whole-block copies between block pools ("vLLM Serving - PagedAttention,
// Continuous Batching, and Production Tuning": copy-on-write copies the one
// shared block a diverging sequence writes to; the scheduler swaps the blocks
// of preempted sequences to CPU memory and back).
//
// One thread block per (pair, slice): a block of n_kv * block_size * head_dim
// elements is contiguous in the [num_blocks][n_kv][block_size][head_dim]
// layout, so each pair is two flat copies (K and V) of 16-byte vectors.  The
// pools may live in device memory or in page-locked host memory that the GPU
// reaches through the unified address space.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
copy_blocks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                   int src_blocks, uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                   int dst_blocks, const int32_t* __restrict__ mapping, int64_t vec_per_block,
                   unsigned* err)
{
    const int pair = blockIdx.y;
    const int32_t s = __ldg(mapping + 2 * pair), d = __ldg(mapping + 2 * pair + 1);
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_error(err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const uint4* sk = src_k + static_cast<int64_t>(s) * vec_per_block;
    const uint4* sv = src_v + static_cast<int64_t>(s) * vec_per_block;
    uint4* dk = dst_k + static_cast<int64_t>(d) * vec_per_block;
    uint4* dv = dst_v + static_cast<int64_t>(d) * vec_per_block;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < vec_per_block;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 a = sk[i], b = sv[i];
        dk[i] = a;
        dv[i] = b;
    }
}

cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, int src_blocks, void* dst_k,
                               void* dst_v, int dst_blocks, const pa_cache_desc& layout,
                               const int32_t* mapping, int pairs, unsigned* err, cudaStream_t s)
{
    const int64_t bytes = static_cast<int64_t>(layout.n_kv_heads) * layout.block_size *
                          layout.head_dim * elem_bytes(layout.dtype);
    const int64_t vecs = bytes / 16;
    const int threads = 256;
    const int64_t slices = (vecs + threads * 4 - 1) / (threads * 4);   // ~64 KB per thread block
    dim3 grid(static_cast<unsigned>(slices < 1 ? 1 : slices), static_cast<unsigned>(pairs));
    copy_blocks_kernel<<<grid, threads, 0, s>>>(
        static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v), src_blocks,
        static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), dst_blocks, mapping, vecs, err);
    return cudaGetLastError();
}

}  // namespace pa
