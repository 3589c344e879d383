// Multi-query decode: the tensor-core decode kernel instantiated for several
// query rows per sequence (verification of drafted tokens, "vLLM Serving ...",
// "Speculative decoding").  A KV head's g query heads times q_per_seq queries
// form (head, query) rows of the MMA tiles, 8 rows per work unit, so each K/V
// slab still serves all of them; query i of a sequence of L rows sees keys
// 0..L - q_per_seq + i.  Kept in its own translation unit so the plain decode
// kernels carry none of the extra row arithmetic and compile in parallel.
#include "decode_mma.cuh"

namespace pa {

cudaError_t launch_decode_mq(const DecodeArgs& a, cudaStream_t s, float scale_log2)
{
    return run_mma_any<true>(a, s, scale_log2);
}

}  // namespace pa
