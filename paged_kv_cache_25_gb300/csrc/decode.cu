// Paged decode attention: one query row per (sequence, query head) against
// the sequence's K/V read through its block table ("How the attention kernel
// actually reads paged blocks": look the block up once, q.k against its keys,
// softmax-weighted sum of its values).
//
// Work unit = (sequence s, KV head, partition j of part_tokens tokens).  Long
// contexts are split into partitions whose (max, sum, unnormalised output)
// are combined by decode_reduce_kernel; a sequence that fits in one
// partition is finished by the partition kernel itself.
//
// Tensor-core path (bf16/fp16, head_dim 64/128, block 16/32):
//   - the g query heads sharing one KV head form the M rows of an m16n8k16
//     MMA, so each K/V slab is read from HBM once for the whole group;
//   - each warp owns a ring of NS stages; lane 0 streams whole
//     (block, kv head) slabs of K and V into it with 2-D TMA tile loads
//     (128-byte swizzle, so ldmatrix reads are bank-conflict free);
//   - online softmax in registers with quad shuffles;
//   - P is split into hi + lo halves of the input type and placed in rows
//     0-7 and 8-15 of the A operand, so P.V costs one MMA yet keeps ~16 bits
//     of P (rows 8-15 would otherwise be padding).  Groups of more than 8 heads
//     are handled as several 8-head sub-groups.
// CUDA-core path (fp32, or shapes the tensor path does not cover): one warp
// per query head, plain loads, fp32 FMA.
#include "pa_device.cuh"
#include "pa_internal.h"

#include <math.h>

namespace pa {

constexpr int kDecWarps = 4;
constexpr int kMaxPartBlocks = 64;

__device__ __forceinline__ void store_any(void* out, int64_t idx, float v, pa_dtype dt)
{
    if (dt == PA_F32)
        static_cast<float*>(out)[idx] = v;
    else if (dt == PA_BF16)
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

template <typename T, int D, int BS, int NS>
struct DecodeCfg {
    static constexpr int kSlabBytes = BS * D * static_cast<int>(sizeof(T));  // one K (or V) slab
    static constexpr int kStageBytes = 2 * kSlabBytes;
    static constexpr int kWarpBytes = NS * kStageBytes;
    static constexpr int kRingBytes = kDecWarps * kWarpBytes;
    static constexpr int kReduceBytes = kDecWarps * 8 * (D + 2) * 4;
    static constexpr int kDynBytes = (kRingBytes > kReduceBytes ? kRingBytes : kReduceBytes) + 1024;
    static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
    static_assert(BS % 16 == 0, "block_size must be a multiple of 16");
};

template <typename T, int D, int BS, int NS>
__global__ void __launch_bounds__(kDecWarps * 32)
decode_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  void* __restrict__ out, pa_dtype out_dtype, const T* __restrict__ q,
                  const int32_t* __restrict__ block_tables, int max_blocks,
                  const int32_t* __restrict__ context_lens, int n_q, int n_kv, int group,
                  int num_blocks, float scale_log2, float* __restrict__ ws_ml,
                  float* __restrict__ ws_acc, int part_tokens, int max_parts, unsigned* err)
{
    using Cfg = DecodeCfg<T, D, BS, NS>;
    constexpr int kHalf = 64;              // elements per 128-byte swizzled row
    constexpr int kHalves = D / kHalf;
    constexpr int kHalfTileBytes = BS * 128;

    const int j = blockIdx.x;
    const int n_sub = (group + 7) >> 3;
    const int kvh = blockIdx.y / n_sub;
    const int sub = blockIdx.y - kvh * n_sub;
    const int s = blockIdx.z;
    const int h0 = kvh * group + sub * 8;
    const int nh = min(8, group - sub * 8);

    const int L = __ldg(context_lens + s);
    const int tok0 = j * part_tokens;
    if (tok0 >= L) return;
    const int tok1 = min(L, tok0 + part_tokens);
    const int nblk = (tok1 - tok0 + BS - 1) / BS;
    const int blk0 = tok0 / BS;
    const int nparts = min((L + part_tokens - 1) / part_tokens, max_parts);

    __shared__ int s_blk[kMaxPartBlocks];
    __shared__ int s_bad;
    __shared__ __align__(8) uint64_t s_bar[kDecWarps * NS];
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                               ~static_cast<uintptr_t>(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    for (int i = tid; i < nblk; i += blockDim.x) {
        const int lb = blk0 + i;
        int b = -1;
        if (lb < max_blocks) b = __ldg(block_tables + static_cast<int64_t>(s) * max_blocks + lb);
        if (b < 0 || b >= num_blocks) {
            s_bad = 1;
            set_error(err, PA_ERR_OUT_OF_RANGE);
        }
        s_blk[i] = b;
    }
    if (tid < kDecWarps * NS) mbar_init(smem_u32(&s_bar[tid]), 1);
    fence_mbar_init();
    __syncthreads();
    if (s_bad) return;

    // ---- per-warp TMA ring --------------------------------------------
    const uint32_t ring = smem_u32(smem) + warp * Cfg::kWarpBytes;
    const uint32_t bar0 = smem_u32(&s_bar[warp * NS]);
    const int my_n = nblk > warp ? (nblk - warp + kDecWarps - 1) / kDecWarps : 0;

    auto issue = [&](int k) {
        const int b = s_blk[warp + k * kDecWarps];
        const int st = k % NS;
        const uint32_t kdst = ring + st * Cfg::kStageBytes;
        const uint32_t vdst = kdst + Cfg::kSlabBytes;
        const uint32_t bar = bar0 + st * 8;
        const int row = (b * n_kv + kvh) * BS;
        mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
#pragma unroll
        for (int hx = 0; hx < kHalves; ++hx) {
            tma_load_2d(kdst + hx * kHalfTileBytes, &kmap, hx * kHalf, row, bar);
            tma_load_2d(vdst + hx * kHalfTileBytes, &vmap, hx * kHalf, row, bar);
        }
    };
    if (lane == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        for (int k = 0; k < min(NS, my_n); ++k) issue(k);
    }

    // ---- query fragments: rows 0-7 = heads of the sub-group, rows 8-15 zero
    const int g = lane >> 2, t4 = lane & 3;
    uint32_t qa[D / 16][2];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        if (g < nh) {
            const T* qp = q + (static_cast<int64_t>(s) * n_q + h0 + g) * D + kk * 16 + 2 * t4;
            qa[kk][0] = __ldg(reinterpret_cast<const unsigned int*>(qp));
            qa[kk][1] = __ldg(reinterpret_cast<const unsigned int*>(qp + 8));
        } else {
            qa[kk][0] = 0u;
            qa[kk][1] = 0u;
        }
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    for (int k = 0; k < my_n; ++k) {
        const int st = k % NS;
        const bool ok = mbar_wait(bar0 + st * 8, (k / NS) & 1, err);
        if (!__all_sync(0xffffffffu, ok)) break;   // leave together: shuffles follow
        const int pos0 = tok0 + (warp + k * kDecWarps) * BS;
        const int valid = min(BS, L - pos0);
        const uint32_t kbase = ring + st * Cfg::kStageBytes;
        const uint32_t vbase = kbase + Cfg::kSlabBytes;

        if (valid < BS) {
            // rows past the sequence may hold anything (even NaN): zero them in
            // V so that 0 * row stays 0 inside the MMA
            uint8_t* vgen = smem + (vbase - smem_u32(smem));
            const int nbytes = (BS - valid) * 128;
            for (int hx = 0; hx < kHalves; ++hx)
                for (int off = lane * 16; off < nbytes; off += 32 * 16)
                    *reinterpret_cast<uint4*>(vgen + hx * kHalfTileBytes + valid * 128 + off) =
                        make_uint4(0, 0, 0, 0);
            __syncwarp();
        }

        // S = Q K^T for the BS tokens of the block
        float sc[BS / 8][4];
#pragma unroll
        for (int nt = 0; nt < BS / 8; ++nt) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kc = 0; kc < D / 16; kc += 2) {
                const int r = nt * 8 + (lane & 7);
                const int chunk = kc * 2 + (lane >> 3);
                const uint32_t addr = kbase + (chunk >> 3) * kHalfTileBytes + r * 128 +
                                      (((chunk & 7) ^ (r & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                const uint32_t a0[4] = {qa[kc][0], 0u, qa[kc][1], 0u};
                const uint32_t a1[4] = {qa[kc + 1][0], 0u, qa[kc + 1][1], 0u};
                MmaOp<T>::run(sc[nt], a0, b0, b1);
                MmaOp<T>::run(sc[nt], a1, b2, b3);
            }
        }

        // online softmax on row g (log2 domain)
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int p = pos0 + nt * 8 + 2 * t4 + e;
                const float z = p < L ? sc[nt][e] * scale_log2 : -INFINITY;
                sc[nt][e] = z;
                mx = fmaxf(mx, z);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = exp2f(m_run - m_new);
        m_run = m_new;
        float psum = 0.f;
#pragma unroll
        for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float p = exp2f(sc[nt][e] - m_new);
                sc[nt][e] = p;
                psum += p;
            }
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= alpha; o[i][1] *= alpha; o[i][2] *= alpha; o[i][3] *= alpha;
        }

        // O += P V, P as hi (rows 0-7) + lo (rows 8-15)
#pragma unroll
        for (int ks = 0; ks < BS / 16; ++ks) {
            uint32_t pa[4];
            split_pair<T>(sc[2 * ks][0], sc[2 * ks][1], pa[0], pa[1]);
            split_pair<T>(sc[2 * ks + 1][0], sc[2 * ks + 1][1], pa[2], pa[3]);
#pragma unroll
            for (int nt = 0; nt < D / 8; nt += 2) {
                const int mi = lane >> 3;
                const int r = ks * 16 + (mi & 1) * 8 + (lane & 7);
                const int chunk = nt + (mi >> 1);
                const uint32_t addr = vbase + (chunk >> 3) * kHalfTileBytes + r * 128 +
                                      (((chunk & 7) ^ (r & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(addr, b0, b1, b2, b3);
                MmaOp<T>::run(o[nt], pa, b0, b1);
                MmaOp<T>::run(o[nt + 1], pa, b2, b3);
            }
        }

        __syncwarp();
        if (lane == 0 && k + NS < my_n) {
            fence_proxy_async_smem();
            issue(k + NS);
        }
    }

    // ---- combine the warps ------------------------------------------------
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    __syncthreads();  // every warp is done with its ring: reuse it
    float* red_o = reinterpret_cast<float*>(smem);              // [warps][8][D]
    float* red_m = red_o + kDecWarps * 8 * D;                   // [warps][8]
    float* red_l = red_m + kDecWarps * 8;                       // [warps][8]
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        float* dst = red_o + (warp * 8 + g) * D + nt * 8 + 2 * t4;
        dst[0] = o[nt][0] + o[nt][2];
        dst[1] = o[nt][1] + o[nt][3];
    }
    if (t4 == 0) {
        red_m[warp * 8 + g] = m_run;
        red_l[warp * 8 + g] = l_run;
    }
    __syncthreads();
    for (int idx = tid; idx < nh * D; idx += blockDim.x) {
        const int hh = idx / D, dd = idx - hh * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red_m[w * 8 + hh]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float f = exp2f(red_m[w * 8 + hh] - M);
            lsum += f * red_l[w * 8 + hh];
            acc += f * red_o[(w * 8 + hh) * D + dd];
        }
        const int64_t sh = static_cast<int64_t>(s) * n_q + h0 + hh;
        if (nparts == 1) {
            store_any(out, sh * D + dd, acc / lsum, out_dtype);
        } else {
            const int64_t u = sh * max_parts + j;
            ws_acc[u * D + dd] = acc;
            if (dd == 0) {
                ws_ml[2 * u] = M;
                ws_ml[2 * u + 1] = lsum;
            }
        }
    }
}

// CUDA-core path: one warp per (partition, query head, sequence).
template <typename T, int DPL>
__global__ void __launch_bounds__(128)
decode_simt_kernel(void* __restrict__ out, pa_dtype out_dtype, const T* __restrict__ q,
                   const T* __restrict__ kc, const T* __restrict__ vc,
                   const int32_t* __restrict__ block_tables, int max_blocks,
                   const int32_t* __restrict__ context_lens, int n_q, int n_kv, int group,
                   int num_blocks, int block_size, float scale_log2, float* __restrict__ ws_ml,
                   float* __restrict__ ws_acc, int part_tokens, int max_parts, unsigned* err)
{
    constexpr int D = DPL * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x;
    const int h = blockIdx.y * 4 + warp;
    const int s = blockIdx.z;
    if (h >= n_q) return;
    const int kvh = h / group;
    const int L = __ldg(context_lens + s);
    const int tok0 = j * part_tokens;
    if (tok0 >= L) return;
    const int tok1 = min(L, tok0 + part_tokens);
    const int nparts = min((L + part_tokens - 1) / part_tokens, max_parts);

    float qv[DPL], acc[DPL];
    const T* qp = q + (static_cast<int64_t>(s) * n_q + h) * D;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
        qv[i] = Cvt<T>::to_f(qp[lane + 32 * i]);
        acc[i] = 0.f;
    }
    float m_run = -INFINITY, l_run = 0.f;
    int64_t base = 0;
    for (int p = tok0; p < tok1; ++p) {
        const int off = p % block_size;
        if (off == 0 || p == tok0) {
            const int lb = p / block_size;
            int b = lb < max_blocks ? __ldg(block_tables + static_cast<int64_t>(s) * max_blocks + lb) : -1;
            if (b < 0 || b >= num_blocks) {
                set_error(err, PA_ERR_OUT_OF_RANGE);
                return;
            }
            base = (static_cast<int64_t>(b) * n_kv + kvh) * block_size;
        }
        const T* kr = kc + (base + off) * D;
        const T* vr = vc + (base + off) * D;
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) dot = fmaf(qv[i], Cvt<T>::to_f(kr[lane + 32 * i]), dot);
#pragma unroll
        for (int w = 16; w > 0; w >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
        const float z = dot * scale_log2;
        const float m_new = fmaxf(m_run, z);
        const float alpha = exp2f(m_run - m_new);
        const float pz = exp2f(z - m_new);
        l_run = l_run * alpha + pz;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(pz, Cvt<T>::to_f(vr[lane + 32 * i]), acc[i] * alpha);
        m_run = m_new;
    }
    const int64_t sh = static_cast<int64_t>(s) * n_q + h;
    if (nparts == 1) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) store_any(out, sh * D + lane + 32 * i, acc[i] / l_run, out_dtype);
    } else {
        const int64_t u = sh * max_parts + j;
#pragma unroll
        for (int i = 0; i < DPL; ++i) ws_acc[u * D + lane + 32 * i] = acc[i];
        if (lane == 0) {
            ws_ml[2 * u] = m_run;
            ws_ml[2 * u + 1] = l_run;
        }
    }
}

// Second pass: out = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j.
__global__ void __launch_bounds__(128)
decode_reduce_kernel(void* __restrict__ out, pa_dtype out_dtype,
                     const int32_t* __restrict__ context_lens, const float* __restrict__ ws_ml,
                     const float* __restrict__ ws_acc, int n_q, int head_dim, int part_tokens,
                     int max_parts)
{
    const int h = blockIdx.x, s = blockIdx.y;
    const int L = __ldg(context_lens + s);
    const int J = min((L + part_tokens - 1) / part_tokens, max_parts);
    if (J <= 1) return;
    const int64_t sh = static_cast<int64_t>(s) * n_q + h;
    const float* ml = ws_ml + 2 * sh * max_parts;
    float M = -INFINITY;
    for (int jj = 0; jj < J; ++jj) M = fmaxf(M, ml[2 * jj]);
    float lsum = 0.f;
    for (int jj = 0; jj < J; ++jj) lsum += exp2f(ml[2 * jj] - M) * ml[2 * jj + 1];
    const float inv = 1.f / lsum;
    for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
        float acc = 0.f;
        for (int jj = 0; jj < J; ++jj)
            acc += exp2f(ml[2 * jj] - M) * ws_acc[(sh * max_parts + jj) * head_dim + d];
        store_any(out, sh * head_dim + d, acc * inv, out_dtype);
    }
}

// ------------------------------------------------------------------ launch

template <typename T, int D, int BS>
static cudaError_t run_mma(const DecodeArgs& a, cudaStream_t s, float scale_log2)
{
    // ring depth per warp: about 24 KB of K+V in flight per warp, at least 2 stages
    constexpr int kStage = 2 * BS * D * static_cast<int>(sizeof(T));
    constexpr int NS = 24576 / kStage > 2 ? 24576 / kStage : 2;
    using Cfg = DecodeCfg<T, D, BS, NS>;
    auto kern = decode_mma_kernel<T, D, BS, NS>;
    static bool attr_done = false;   // per process; the attribute is per function
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::kDynBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    CUtensorMap kmap, vmap;
    const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * a.cache.n_kv_heads * BS;
    if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, 64, BS) != PA_OK ||
        encode_pool_map(&vmap, a.v_cache, a.cache.dtype, D, rows, 64, BS) != PA_OK)
        return cudaErrorInvalidValue;
    const int group = a.n_q / a.cache.n_kv_heads;
    dim3 grid(a.max_parts, a.cache.n_kv_heads * ((group + 7) / 8), a.num_seqs);
    kern<<<grid, kDecWarps * 32, Cfg::kDynBytes, s>>>(
        kmap, vmap, a.out, a.out_dtype, static_cast<const T*>(a.q), a.block_tables, a.max_blocks,
        a.context_lens, a.n_q, a.cache.n_kv_heads, group, a.cache.num_blocks, scale_log2, a.ws_ml,
        a.ws_acc, a.part_tokens, a.max_parts, a.err);
    return cudaGetLastError();
}

template <typename T, int DPL>
static cudaError_t run_simt(const DecodeArgs& a, cudaStream_t s, float scale_log2)
{
    dim3 grid(a.max_parts, (a.n_q + 3) / 4, a.num_seqs);
    decode_simt_kernel<T, DPL><<<grid, 128, 0, s>>>(
        a.out, a.out_dtype, static_cast<const T*>(a.q), static_cast<const T*>(a.k_cache),
        static_cast<const T*>(a.v_cache), a.block_tables, a.max_blocks, a.context_lens, a.n_q,
        a.cache.n_kv_heads, a.n_q / a.cache.n_kv_heads, a.cache.num_blocks, a.cache.block_size,
        scale_log2, a.ws_ml, a.ws_acc, a.part_tokens, a.max_parts, a.err);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t run_simt_dt(const DecodeArgs& a, cudaStream_t s, float sl2)
{
    switch (a.cache.head_dim) {
        case 32: return run_simt<T, 1>(a, s, sl2);
        case 64: return run_simt<T, 2>(a, s, sl2);
        case 96: return run_simt<T, 3>(a, s, sl2);
        case 128: return run_simt<T, 4>(a, s, sl2);
        case 256: return run_simt<T, 8>(a, s, sl2);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
static cudaError_t run_mma_dt(const DecodeArgs& a, cudaStream_t s, float sl2)
{
    const int D = a.cache.head_dim, BS = a.cache.block_size;
    if (D == 64 && BS == 16) return run_mma<T, 64, 16>(a, s, sl2);
    if (D == 64 && BS == 32) return run_mma<T, 64, 32>(a, s, sl2);
    if (D == 128 && BS == 16) return run_mma<T, 128, 16>(a, s, sl2);
    if (D == 128 && BS == 32) return run_mma<T, 128, 32>(a, s, sl2);
    return run_simt_dt<T>(a, s, sl2);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s)
{
    const float sl2 = a.scale * 1.4426950408889634f;   // softmax in base 2
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    profile_events(&ev0, &ev1);
    if (ev0) cudaEventRecord(ev0, s);
    cudaError_t e;
    switch (a.cache.dtype) {
        case PA_BF16: e = run_mma_dt<__nv_bfloat16>(a, s, sl2); break;
        case PA_F16: e = run_mma_dt<__half>(a, s, sl2); break;
        default: e = run_simt_dt<float>(a, s, sl2); break;
    }
    if (ev1) cudaEventRecord(ev1, s);
    if (e != cudaSuccess) return e;
    if (a.max_parts > 1) {
        dim3 grid(a.n_q, a.num_seqs);
        decode_reduce_kernel<<<grid, 128, 0, s>>>(a.out, a.out_dtype, a.context_lens, a.ws_ml,
                                                  a.ws_acc, a.n_q, a.cache.head_dim,
                                                  a.part_tokens, a.max_parts);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace pa
