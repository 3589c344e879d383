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

// Write into an FP8 E4M3 pool: 16 input elements of one (token, head) row
// become 16 codes: code = e4m3_rn_satfinite(x / scale) with x / scale an IEEE
// fp32 division (or, for rows given as codes, the codes themselves).  K keeps
// the row layout; V codes go to the transposed slab of their 16-token piece of
// the block, [block_size / 16][head_dim][16].
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

// A CTA takes 16 consecutive tokens and kHpc KV heads (128 threads: one per
// 16-element piece of a (token, head) row).  K codes go straight to the pool,
// 16 bytes per thread (a row's pieces are neighbours: coalesced).  V codes are
// transposed through shared memory, [head][d][16 tokens], and then written one
// (head, d) row of the slab per thread: 16 bytes when the 16 tokens fill 16
// aligned consecutive slots (one whole 16-token piece: a chunk of a prompt),
// 4 bytes for each aligned run of 4 consecutive slots, single bytes otherwise
// (one decode token per sequence lands in 16 different blocks).
constexpr int kFp8Tok = 16;

template <typename TI, int D>
__global__ void __launch_bounds__(128)
cache_write_fp8_kernel(const TI* __restrict__ k, const TI* __restrict__ v, uint8_t* __restrict__ kc,
                       uint8_t* __restrict__ vc, const int64_t* __restrict__ slots, int T, int n_kv,
                       int block_size, int64_t num_slots, float k_scale, float v_scale,
                       unsigned* err)
{
    constexpr int kPpr = D / 16;                  // 16-element pieces per row
    constexpr int kHpc = 128 / (kFp8Tok * kPpr);  // heads per CTA (1 at d 128, 2 at d 64)
    __shared__ __align__(16) uint8_t vt[kHpc][D][kFp8Tok];
    __shared__ int64_t s_slot[kFp8Tok];
    __shared__ int s_run16;                       // the 16 slots: aligned and consecutive
    __shared__ int s_run4[kFp8Tok / 4];           // each quad: aligned and consecutive
    allow_dependent_launch();                     // as in cache_write_kernel

    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * kFp8Tok;
    const int hh = tid / (kFp8Tok * kPpr), rem = tid % (kFp8Tok * kPpr);
    const int tt = rem / kPpr, c = rem % kPpr;
    const int h = blockIdx.y * kHpc + hh;
    if (tid < kFp8Tok) s_slot[tid] = t0 + tid < T ? __ldg(slots + t0 + tid) : -1;
    __syncthreads();
    if (tid == 0) {
        const int64_t s0 = s_slot[0];
        int run16 = s0 >= 0 && s0 + kFp8Tok <= num_slots && s0 % kFp8Tok == 0;
        for (int i = 1; i < kFp8Tok; ++i) run16 = run16 && s_slot[i] == s0 + i;
        s_run16 = run16;
        for (int q4 = 0; q4 < kFp8Tok / 4; ++q4) {
            const int64_t a = s_slot[4 * q4];
            int run = a >= 0 && a + 4 <= num_slots && a % 4 == 0;
            for (int i = 1; i < 4; ++i) run = run && s_slot[4 * q4 + i] == a + i;
            s_run4[q4] = run;
        }
    }

    // this thread's piece: K codes to the pool, V codes to the transpose tile
    const int t = t0 + tt;
    const int64_t slot = s_slot[tt];
    uint4 vq = make_uint4(0u, 0u, 0u, 0u);
    if (h < n_kv && t < T && slot >= 0) {
        const int64_t src = (static_cast<int64_t>(t) * n_kv + h) * D + c * 16;
        if (slot >= num_slots) {
            set_error(err, PA_ERR_OUT_OF_RANGE);
        } else {
            const int64_t b = slot / block_size, o = slot - b * block_size;
            reinterpret_cast<uint4*>(kc)[((b * n_kv + h) * block_size + o) * kPpr + c] =
                codes16(k + src, k_scale);
        }
        vq = codes16(v + src, v_scale);
    }
    const uint32_t w[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) vt[hh][c * 16 + e][tt] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
    __syncthreads();

    // one (head, d) row of the transposed V slab per thread
    const int rh = tid / D, d = tid % D;
    const int vh = blockIdx.y * kHpc + rh;
    if (vh >= n_kv) return;
    const uint8_t* row = vt[rh][d];
    auto dst = [&](int64_t sl) {   // byte address of slot sl's code in row d of head vh
        const int64_t b = sl / block_size, o = sl - b * block_size;
        return vc + (((b * n_kv + vh) * (block_size / 16) + o / 16) * D + d) * 16 + (o & 15);
    };
    if (s_run16) {
        *reinterpret_cast<uint4*>(dst(s_slot[0])) = *reinterpret_cast<const uint4*>(row);
        return;
    }
#pragma unroll
    for (int q4 = 0; q4 < kFp8Tok / 4; ++q4) {
        if (s_run4[q4]) {
            *reinterpret_cast<uint32_t*>(dst(s_slot[4 * q4])) = *reinterpret_cast<const uint32_t*>(row + 4 * q4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t sl = s_slot[4 * q4 + i];
                if (sl >= 0 && sl < num_slots) *dst(sl) = row[4 * q4 + i];
            }
        }
    }
}

cudaError_t launch_cache_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* kc,
                                   void* vc, const int64_t* slots, int T, const pa_cache_desc& c,
                                   unsigned* err, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const int64_t ns = static_cast<int64_t>(c.num_blocks) * c.block_size;
    const int hpc = c.head_dim == 128 ? 1 : (c.head_dim == 64 ? 2 : 0);
    if (!hpc) return cudaErrorInvalidValue;   // FP8 pools: head_dim 64 or 128 (checked by the caller)
    const dim3 grid(static_cast<unsigned>((T + kFp8Tok - 1) / kFp8Tok),
                    static_cast<unsigned>((c.n_kv_heads + hpc - 1) / hpc));
#define PA_QW(TI, DD)                                                                           \
    cache_write_fp8_kernel<TI, DD><<<grid, 128, 0, s>>>(                                        \
        static_cast<const TI*>(k), static_cast<const TI*>(v), static_cast<uint8_t*>(kc),        \
        static_cast<uint8_t*>(vc), slots, T, c.n_kv_heads, c.block_size, ns, c.k_scale,         \
        c.v_scale, err)
#define PA_QW_D(TI) \
    if (c.head_dim == 128) PA_QW(TI, 128); else PA_QW(TI, 64)
    if (in_dtype == PA_BF16) PA_QW_D(__nv_bfloat16);
    else if (in_dtype == PA_F16) PA_QW_D(__half);
    else if (in_dtype == PA_FP8_E4M3) PA_QW_D(uint8_t);   // codes already: copied, V transposed
    else PA_QW_D(float);
#undef PA_QW_D
#undef PA_QW
    return cudaGetLastError();
}

}  // namespace pa
