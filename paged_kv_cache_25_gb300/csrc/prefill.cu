// Chunked-prefill attention over a paged context ("The hands-on guide to LLM
// Inference with vLLM", chunked prefill: a chunk's queries attend over every
// earlier cached token plus the chunk itself; the chunk's K/V are already in
// the pool).  Query row i of request r sits at position L_r - C_r + i and
// attends logical rows 0 .. that position.
//
// CTA = (128 query rows, KV head, request).  The 128 M rows are (position,
// head) pairs of one GQA group, position-major, so one pass over the K/V
// blocks serves every query head that shares the KV head.  A producer warp
// streams (block, kv head) slabs of K and V into an NS-stage ring with 2-D TMA
// tile loads; eight consumer warps each own 16 rows and run m16n8k16 MMAs
// with an online softmax in registers.  P is applied as hi + lo halves of the
// input type (two MMAs) so P keeps ~16 bits.
#include "pa_device.cuh"
#include "pa_internal.h"

#include <math.h>

namespace pa {

constexpr int kPfConsumers = 8;
constexpr int kPfRows = kPfConsumers * 16;

__device__ __forceinline__ void store_any_pf(void* out, int64_t idx, float v, pa_dtype dt)
{
    if (dt == PA_F32)
        static_cast<float*>(out)[idx] = v;
    else if (dt == PA_BF16)
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

template <typename T, int D, int BS, int NS>
__global__ void __launch_bounds__((kPfConsumers + 1) * 32)
prefill_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   void* __restrict__ out, pa_dtype out_dtype, const T* __restrict__ q,
                   const int32_t* __restrict__ block_tables, int max_blocks,
                   const int32_t* __restrict__ q_start, const int32_t* __restrict__ context_lens,
                   int n_q, int n_kv, int group, int num_blocks, float scale_log2, unsigned* err)
{
    constexpr int kSlab = BS * D * static_cast<int>(sizeof(T));
    constexpr int kStage = 2 * kSlab;
    constexpr int kHalf = 64;
    constexpr int kHalves = D / kHalf;
    constexpr int kHalfTile = BS * 128;

    const int tile = blockIdx.x, kvh = blockIdx.y, r = blockIdx.z;
    const int qs = __ldg(q_start + r);
    const int C = __ldg(q_start + r + 1) - qs;
    const int L = __ldg(context_lens + r);
    const int rows_total = C * group;
    const int row0 = tile * kPfRows;
    if (row0 >= rows_total) return;
    if (C > L) {
        if (threadIdx.x == 0) set_error(err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int ctx0 = L - C;
    const int last_row = min(rows_total, row0 + kPfRows) - 1;
    const int max_pos = ctx0 + last_row / group;
    const int n_blocks = max_pos / BS + 1;

    __shared__ __align__(8) uint64_t full_bar[NS];
    __shared__ __align__(8) uint64_t empty_bar[NS];
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t ring = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < NS) {
        mbar_init(smem_u32(&full_bar[tid]), 1);
        mbar_init(smem_u32(&empty_bar[tid]), kPfConsumers);
    }
    fence_mbar_init();
    __syncthreads();

    if (warp == kPfConsumers) {
        // ---------------- producer warp ----------------
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            for (int k = 0; k < n_blocks; ++k) {
                const int st = k % NS;
                if (k >= NS && !mbar_wait(smem_u32(&empty_bar[st]), ((k / NS) - 1) & 1, err)) break;
                int b = k < max_blocks ? __ldg(block_tables + static_cast<int64_t>(r) * max_blocks + k) : -1;
                if (b < 0 || b >= num_blocks) {
                    set_error(err, PA_ERR_OUT_OF_RANGE);
                    b = 0;   // keep the ring moving; the outputs are flagged as invalid
                }
                const uint32_t bar = smem_u32(&full_bar[st]);
                const uint32_t kdst = ring + st * kStage, vdst = kdst + kSlab;
                const int row = (b * n_kv + kvh) * BS;
                mbar_arrive_expect_tx(bar, kStage);
#pragma unroll
                for (int hx = 0; hx < kHalves; ++hx) {
                    tma_load_2d(kdst + hx * kHalfTile, &kmap, hx * kHalf, row, bar);
                    tma_load_2d(vdst + hx * kHalfTile, &vmap, hx * kHalf, row, bar);
                }
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int g = lane >> 2, t4 = lane & 3;
    const int wrow0 = row0 + warp * 16;
    const bool warp_live = wrow0 < rows_total;
    const int ra = wrow0 + g, rb = ra + 8;
    const bool va = ra < rows_total, vb = rb < rows_total;
    const int pos_a = va ? ctx0 + ra / group : ctx0;     // absolute position of row a
    const int pos_b = vb ? ctx0 + rb / group : ctx0;
    const int pw_lo = ctx0 + wrow0 / group;
    const int pw_hi = ctx0 + min(wrow0 + 15, rows_total - 1) / group;

    uint32_t qa[D / 16][4];
    {
        const T* qpa = q + (static_cast<int64_t>(qs) + (va ? ra / group : 0)) * n_q * D +
                       static_cast<int64_t>(kvh * group + (va ? ra % group : 0)) * D;
        const T* qpb = q + (static_cast<int64_t>(qs) + (vb ? rb / group : 0)) * n_q * D +
                       static_cast<int64_t>(kvh * group + (vb ? rb % group : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c = kk * 16 + 2 * t4;
            qa[kk][0] = va ? __ldg(reinterpret_cast<const unsigned*>(qpa + c)) : 0u;
            qa[kk][1] = vb ? __ldg(reinterpret_cast<const unsigned*>(qpb + c)) : 0u;
            qa[kk][2] = va ? __ldg(reinterpret_cast<const unsigned*>(qpa + c + 8)) : 0u;
            qa[kk][3] = vb ? __ldg(reinterpret_cast<const unsigned*>(qpb + c + 8)) : 0u;
        }
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int k = 0; k < n_blocks; ++k) {
        const int st = k % NS;
        const bool ok = mbar_wait(smem_u32(&full_bar[st]), (k / NS) & 1, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int t0 = k * BS;
        const uint32_t kbase = ring + st * kStage, vbase = kbase + kSlab;
        if (t0 + BS > L) {
            // the request's last block: rows at or past L may hold anything
            // (even NaN).  Every consumer warp writes the same zeros over them in
            // V before it reads the slab, so no cross-warp barrier is needed:
            // each warp reads either its own zeros or another warp's.
            uint8_t* vgen = smem + st * kStage + kSlab;
            const int valid = L - t0;
            const int nbytes = (BS - valid) * 128;
            for (int hx = 0; hx < kHalves; ++hx)
                for (int off = lane * 16; off < nbytes; off += 32 * 16)
                    *reinterpret_cast<uint4*>(vgen + hx * kHalfTile + valid * 128 + off) =
                        make_uint4(0, 0, 0, 0);
            __syncwarp();
        }
        if (warp_live && t0 <= pw_hi) {
            float sc[BS / 8][4];
#pragma unroll
            for (int nt = 0; nt < BS / 8; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int kc = 0; kc < D / 16; kc += 2) {
                    const int rr = nt * 8 + (lane & 7);
                    const int chunk = kc * 2 + (lane >> 3);
                    const uint32_t addr = kbase + (chunk >> 3) * kHalfTile + rr * 128 +
                                          (((chunk & 7) ^ (rr & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    MmaOp<T>::run(sc[nt], qa[kc], b0, b1);
                    MmaOp<T>::run(sc[nt], qa[kc + 1], b2, b3);
                }
            }
            const bool need_mask = t0 + BS - 1 > pw_lo;
            float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = t0 + nt * 8 + 2 * t4 + e;
                    const float za = (!need_mask || t <= pos_a) ? sc[nt][e] * scale_log2 : -INFINITY;
                    const float zb = (!need_mask || t <= pos_b) ? sc[nt][2 + e] * scale_log2 : -INFINITY;
                    sc[nt][e] = za;
                    sc[nt][2 + e] = zb;
                    mxa = fmaxf(mxa, za);
                    mxb = fmaxf(mxb, zb);
                }
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
            const float ala = exp2f(m_a - mna), alb = exp2f(m_b - mnb);
            m_a = mna;
            m_b = mnb;
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pa = exp2f(sc[nt][e] - mna);
                    const float pb = exp2f(sc[nt][2 + e] - mnb);
                    sc[nt][e] = pa;
                    sc[nt][2 + e] = pb;
                    sa += pa;
                    sb += pb;
                }
            l_a = l_a * ala + sa;
            l_b = l_b * alb + sb;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= ala; o[i][1] *= ala; o[i][2] *= alb; o[i][3] *= alb;
            }
#pragma unroll
            for (int ks = 0; ks < BS / 16; ++ks) {
                uint32_t ph[4], pl[4];
                split_pair<T>(sc[2 * ks][0], sc[2 * ks][1], ph[0], pl[0]);
                split_pair<T>(sc[2 * ks][2], sc[2 * ks][3], ph[1], pl[1]);
                split_pair<T>(sc[2 * ks + 1][0], sc[2 * ks + 1][1], ph[2], pl[2]);
                split_pair<T>(sc[2 * ks + 1][2], sc[2 * ks + 1][3], ph[3], pl[3]);
#pragma unroll
                for (int nt = 0; nt < D / 8; nt += 2) {
                    const int mi = lane >> 3;
                    const int rr = ks * 16 + (mi & 1) * 8 + (lane & 7);
                    const int chunk = nt + (mi >> 1);
                    const uint32_t addr = vbase + (chunk >> 3) * kHalfTile + rr * 128 +
                                          (((chunk & 7) ^ (rr & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    MmaOp<T>::run(o[nt], ph, b0, b1);
                    MmaOp<T>::run(o[nt], pl, b0, b1);
                    MmaOp<T>::run(o[nt + 1], ph, b2, b3);
                    MmaOp<T>::run(o[nt + 1], pl, b2, b3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }

    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    if (!warp_live) return;
    const float ia = 1.f / l_a, ib = 1.f / l_b;
    const int64_t oa = ((static_cast<int64_t>(qs) + (va ? ra / group : 0)) * n_q + kvh * group +
                        (va ? ra % group : 0)) * D;
    const int64_t ob = ((static_cast<int64_t>(qs) + (vb ? rb / group : 0)) * n_q + kvh * group +
                        (vb ? rb % group : 0)) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        const int c = nt * 8 + 2 * t4;
        if (va) {
            store_any_pf(out, oa + c, o[nt][0] * ia, out_dtype);
            store_any_pf(out, oa + c + 1, o[nt][1] * ia, out_dtype);
        }
        if (vb) {
            store_any_pf(out, ob + c, o[nt][2] * ib, out_dtype);
            store_any_pf(out, ob + c + 1, o[nt][3] * ib, out_dtype);
        }
    }
}

template <typename T, int D, int BS>
static cudaError_t run_prefill(const PrefillArgs& a, cudaStream_t s, float sl2)
{
    constexpr int kStage = 2 * BS * D * static_cast<int>(sizeof(T));
    constexpr int NS = 65536 / kStage > 2 ? 65536 / kStage : 2;
    constexpr int kDyn = NS * kStage + 1024;
    auto kern = prefill_mma_kernel<T, D, BS, NS>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    CUtensorMap kmap, vmap;
    const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * a.cache.n_kv_heads * BS;
    if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, 64, BS) != PA_OK ||
        encode_pool_map(&vmap, a.v_cache, a.cache.dtype, D, rows, 64, BS) != PA_OK)
        return cudaErrorInvalidValue;
    const int group = a.n_q / a.cache.n_kv_heads;
    const int64_t tiles = (static_cast<int64_t>(a.max_q) * group + kPfRows - 1) / kPfRows;
    dim3 grid(static_cast<unsigned>(tiles), a.cache.n_kv_heads, a.num_reqs);
    kern<<<grid, (kPfConsumers + 1) * 32, kDyn, s>>>(
        kmap, vmap, a.out, a.out_dtype, static_cast<const T*>(a.q), a.block_tables, a.max_blocks,
        a.q_start, a.context_lens, a.n_q, a.cache.n_kv_heads, group, a.cache.num_blocks, sl2, a.err);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t run_prefill_dt(const PrefillArgs& a, cudaStream_t s, float sl2)
{
    const int D = a.cache.head_dim, BS = a.cache.block_size;
    if (D == 64 && BS == 16) return run_prefill<T, 64, 16>(a, s, sl2);
    if (D == 64 && BS == 32) return run_prefill<T, 64, 32>(a, s, sl2);
    if (D == 128 && BS == 16) return run_prefill<T, 128, 16>(a, s, sl2);
    if (D == 128 && BS == 32) return run_prefill<T, 128, 32>(a, s, sl2);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s)
{
    const float sl2 = a.scale * 1.4426950408889634f;
    if (a.cache.dtype == PA_BF16) return run_prefill_dt<__nv_bfloat16>(a, s, sl2);
    if (a.cache.dtype == PA_F16) return run_prefill_dt<__half>(a, s, sl2);
    return cudaErrorInvalidValue;
}

}  // namespace pa
