// Slot-mapped cache write ("Life of a prompt", "Back to the queue, and into
// vLLM proper": every new token's K and V vector is appended into the next
// free slot of its sequence's blocks).
//
// One thread moves one 16-byte chunk of one (token, kv head) row for both K
// and V: consecutive threads cover consecutive chunks of a row, so the reads
// of k/v and the writes into the pool are fully coalesced 16-byte accesses.
#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                   uint4* __restrict__ kc, uint4* __restrict__ vc,
                   const int64_t* __restrict__ slots, int64_t total, int n_kv, int block_size,
                   int chunks_per_row, int64_t num_slots, unsigned* err)
{
    // the decode launched next (a programmatic dependent) may be scheduled at
    // once; it waits for this grid to complete before it reads the pool
    allow_dependent_launch();
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

// Write into an FP8 E4M3 pool: one thread turns 16 input elements of one
// (token, head) row into 16 codes: code = e4m3_rn_satfinite(x / scale) with
// x / scale an IEEE fp32 division (or, for rows given as codes, the codes
// themselves).  K codes are one 16-byte store; V codes go to the transposed V
// slab, one column of [head_dim][block_size].
template <typename TI>
__device__ __forceinline__ float load_as_float(const TI* p, int i);
template <> __device__ __forceinline__ float load_as_float<float>(const float* p, int i) { return p[i]; }
template <> __device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p, int i)
{
    return __bfloat162float(p[i]);
}
template <> __device__ __forceinline__ float load_as_float<__half>(const __half* p, int i)
{
    return __half2float(p[i]);
}

template <typename TI>
__device__ __forceinline__ uint4 quant16(const TI* src, float scale)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = __fdiv_rn(load_as_float(src, 4 * i + 0), scale);
        const float b = __fdiv_rn(load_as_float(src, 4 * i + 1), scale);
        const float c = __fdiv_rn(load_as_float(src, 4 * i + 2), scale);
        const float d = __fdiv_rn(load_as_float(src, 4 * i + 3), scale);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
        w[i] = (lo & 0xFFFFu) | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sixteen elements of a row as E4M3 codes: quantized from fp32/fp16/bf16, or,
// for rows that already hold codes (TI = uint8_t), the 16 bytes themselves.
template <typename TI>
__device__ __forceinline__ uint4 codes16(const TI* src, float scale)
{
    return quant16(src, scale);
}
template <>
__device__ __forceinline__ uint4 codes16<uint8_t>(const uint8_t* src, float)
{
    return __ldcs(reinterpret_cast<const uint4*>(src));
}

template <typename TI>
__global__ void __launch_bounds__(256)
cache_write_fp8_kernel(const TI* __restrict__ k, const TI* __restrict__ v, uint4* __restrict__ kc,
                       uint4* __restrict__ vc, const int64_t* __restrict__ slots, int64_t total,
                       int n_kv, int block_size, int pieces_per_row, int64_t num_slots,
                       float k_scale, float v_scale, unsigned* err)
{
    allow_dependent_launch();   // as in cache_write_kernel
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t row = i / pieces_per_row;       // (token, head) row
    const int c = static_cast<int>(i - row * pieces_per_row);
    const int64_t t = row / n_kv;
    const int h = static_cast<int>(row - t * n_kv);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return;
    if (slot >= num_slots) {
        set_error(err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int64_t b = slot / block_size, o = slot - b * block_size;
    const int64_t dst = ((b * n_kv + h) * block_size + o) * pieces_per_row + c;
    const int64_t src = i * 16;                   // element offset of this piece
    kc[dst] = codes16(k + src, k_scale);
    // V codes are stored transposed per (block, head): [head_dim][block_size]
    const uint4 vq = codes16(v + src, v_scale);
    uint8_t* vcol = reinterpret_cast<uint8_t*>(vc) +
                    ((b * n_kv + h) * (pieces_per_row * 16) + c * 16) * block_size + o;
    const uint32_t w[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) vcol[e * block_size] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
}

cudaError_t launch_cache_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* kc,
                                   void* vc, const int64_t* slots, int T, const pa_cache_desc& c,
                                   unsigned* err, cudaStream_t s)
{
    const int ppr = c.head_dim / 16;
    const int64_t total = static_cast<int64_t>(T) * c.n_kv_heads * ppr;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = static_cast<unsigned>((total + threads - 1) / threads);
    const int64_t ns = static_cast<int64_t>(c.num_blocks) * c.block_size;
#define PA_QW(TI)                                                                              \
    cache_write_fp8_kernel<TI><<<blocks, threads, 0, s>>>(                                     \
        static_cast<const TI*>(k), static_cast<const TI*>(v), static_cast<uint4*>(kc),         \
        static_cast<uint4*>(vc), slots, total, c.n_kv_heads, c.block_size, ppr, ns, c.k_scale, \
        c.v_scale, err)
    if (in_dtype == PA_BF16) PA_QW(__nv_bfloat16);
    else if (in_dtype == PA_F16) PA_QW(__half);
    else if (in_dtype == PA_FP8_E4M3) PA_QW(uint8_t);   // codes already: copied, V transposed
    else PA_QW(float);
#undef PA_QW
    return cudaGetLastError();
}

}  // namespace pa
