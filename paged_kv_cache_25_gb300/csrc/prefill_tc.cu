// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05).
//
// Semantics ("The hands-on guide to LLM Inference with vLLM", chunked
// prefill): query row i of request r's chunk of C_r rows sits at absolute
// position L_r - C_r + i and attends logical K/V rows 0 .. that position,
// read through the request's block table; the chunk's own K/V are already in
// the pool.
//
// CTA = (128 M rows, KV head, request).  The M rows are (position, head) pairs
// of one GQA group, position-major, so one pass over the keys serves all the
// query heads that share the KV head.  Keys go in tiles of 64.
//   warp 4  : TMA producer: 16-row K and V slabs of each 64-key tile into a
//             3-stage ring (128-byte swizzle), one block-table lookup per block;
//   warp 5  : one thread issues the MMAs: S = Q K^T (M 128, N 64, K = d) into a
//             double-buffered TMEM tile, then O += P V (M 128, N = d, K 64)
//             into TMEM, signalling completion with tcgen05.commit;
//   warps 0-3: one thread per M row: read S from TMEM, causal mask on absolute
//             positions, online softmax in base 2 with lazy rescaling (O in TMEM
//             is rescaled only when the running max grows by more than 2^8),
//             P written to shared memory as hi + lo bf16/fp16 halves so that P V
//             keeps ~16 bits of P, final O / l written to global memory.
// All waits are bounded; the kernel never traps.
#include "pa_device.cuh"
#include "pa_internal.h"

#include <math.h>

#include <mutex>
#include <type_traits>

namespace pa {

constexpr int kTcRows = 128;      // M rows per CTA
constexpr int kTcKeys = 64;       // keys per tile
constexpr int kTcStages = 3;      // K/V ring depth
constexpr int kTcThreads = 192;   // 4 softmax warps + producer + MMA issuer
constexpr uint32_t kTmemCols = 256;   // S0 [0,64) S1 [64,128) O [128, 128 + d)

template <typename T, int D>
struct PfLayout {
    static constexpr int kHalves = D / 64;
    static constexpr uint32_t kQBytes = kTcRows * D * 2;          // Q tile
    static constexpr uint32_t kPBytes = kTcRows * kTcKeys * 2;    // one of P hi / P lo
    static constexpr uint32_t kKBytes = kTcKeys * D * 2;          // K (or V) of one tile
    static constexpr uint32_t kStageBytes = 2 * kKBytes;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffPh = kOffQ + kQBytes;
    static constexpr uint32_t kOffPl = kOffPh + kPBytes;
    static constexpr uint32_t kOffKV = kOffPl + kPBytes;
    static constexpr uint32_t kDynBytes = kOffKV + kTcStages * kStageBytes + 1024;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

template <typename T>
__device__ __forceinline__ void store_row(void* out, int64_t base, int col, const float* v, int n,
                                          pa_dtype dt)
{
    if (dt == PA_F32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + base + col);
        for (int i = 0; i < n; i += 4) p[i / 4] = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else if (dt == PA_BF16) {
        uint4* p = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + base + col);
        for (int i = 0; i < n; i += 8)
            p[i / 8] = make_uint4(Cvt<__nv_bfloat16>::pack(v[i], v[i + 1]),
                                  Cvt<__nv_bfloat16>::pack(v[i + 2], v[i + 3]),
                                  Cvt<__nv_bfloat16>::pack(v[i + 4], v[i + 5]),
                                  Cvt<__nv_bfloat16>::pack(v[i + 6], v[i + 7]));
    } else {
        uint4* p = reinterpret_cast<uint4*>(static_cast<__half*>(out) + base + col);
        for (int i = 0; i < n; i += 8)
            p[i / 8] = make_uint4(Cvt<__half>::pack(v[i], v[i + 1]), Cvt<__half>::pack(v[i + 2], v[i + 3]),
                                  Cvt<__half>::pack(v[i + 4], v[i + 5]),
                                  Cvt<__half>::pack(v[i + 6], v[i + 7]));
    }
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  void* __restrict__ out, pa_dtype out_dtype, const T* __restrict__ q,
                  const int32_t* __restrict__ block_tables, int max_blocks,
                  const int32_t* __restrict__ q_start, const int32_t* __restrict__ context_lens,
                  int n_q, int n_kv, int group, int num_blocks, float scale_log2, unsigned* err)
{
    using Ly = PfLayout<T, D>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdescQK = idesc_f16(kBf16, false, false, kTcRows, kTcKeys);
    constexpr uint32_t kIdescPV = idesc_f16(kBf16, false, true, kTcRows, D);
    static_assert(BS % 16 == 0 && kTcKeys % BS == 0, "block size must divide the key tile");

    // tiles with more keys first: the last position tiles are the heaviest
    const int tile = gridDim.x - 1 - blockIdx.x;
    const int kvh = blockIdx.y, r = blockIdx.z;
    const int qs = __ldg(q_start + r);
    const int C = __ldg(q_start + r + 1) - qs;
    const int L = __ldg(context_lens + r);
    const int rows_total = C * group;
    const int row0 = tile * kTcRows;
    if (row0 >= rows_total) return;
    if (C > L || C < 0) {
        if (threadIdx.x == 0) set_error(err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int ctx0 = L - C;
    const int last_row = min(rows_total, row0 + kTcRows) - 1;
    const int n_tiles = (ctx0 + last_row / group) / kTcKeys + 1;

    __shared__ __align__(8) uint64_t kv_full[kTcStages], kv_empty[kTcStages];
    __shared__ __align__(8) uint64_t s_full[2], s_empty[2], p_full, pv_done, q_ready;
    __shared__ uint32_t s_tmem;
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(smem_u32(&kv_full[i]), 1);
            mbar_init(smem_u32(&kv_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&s_empty[i]), 4);
        }
        mbar_init(smem_u32(&p_full), 4);
        mbar_init(smem_u32(&pv_done), 1);
        mbar_init(smem_u32(&q_ready), 4);
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kTcStages;
                if (j >= kTcStages &&
                    !mbar_wait(smem_u32(&kv_empty[st]), ((j / kTcStages) - 1) & 1, err))
                    break;
                const uint32_t full = smem_u32(&kv_full[st]);
                const uint32_t kdst = sbase + Ly::kOffKV + st * Ly::kStageBytes;
                const uint32_t vdst = kdst + Ly::kKBytes;
                mbar_arrive_expect_tx(full, Ly::kStageBytes);
                int b = 0;
#pragma unroll
                for (int c = 0; c < kTcKeys / 16; ++c) {
                    const int key0 = j * kTcKeys + c * 16;
                    if (key0 < L) {   // past L the tile's rows are masked: reuse the last block
                        const int lb = key0 / BS;
                        b = lb < max_blocks ? __ldg(block_tables + static_cast<int64_t>(r) * max_blocks + lb) : -1;
                        if (b < 0 || b >= num_blocks) {
                            set_error(err, PA_ERR_OUT_OF_RANGE);
                            b = 0;   // keep the ring moving; the outputs are flagged invalid
                        }
                    }
                    const int row = (b * n_kv + kvh) * BS + (key0 % BS);
#pragma unroll
                    for (int hx = 0; hx < Ly::kHalves; ++hx) {
                        tma_load_2d(kdst + hx * (kTcKeys * 128) + c * 2048, &kmap, hx * 64, row, full);
                        tma_load_2d(vdst + hx * (kTcKeys * 128) + c * 2048, &vmap, hx * 64, row, full);
                    }
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&q_ready), 0, err);
            tc_fence_after();
            for (int j = 0; ok && j <= n_tiles; ++j) {
                if (j < n_tiles) {
                    const int st = j % kTcStages, sb = j & 1;
                    if (!mbar_wait(smem_u32(&kv_full[st]), (j / kTcStages) & 1, err)) break;
                    if (j >= 2 && !mbar_wait(smem_u32(&s_empty[sb]), ((j >> 1) - 1) & 1, err)) break;
                    tc_fence_after();
                    const uint32_t kbase = sbase + Ly::kOffKV + st * Ly::kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32u;   // 16 columns = 32 bytes
                        const uint64_t a = sdesc_sw128(sbase + Ly::kOffQ + (kk >> 2) * (kTcRows * 128) + off, 16, 1024);
                        const uint64_t b = sdesc_sw128(kbase + (kk >> 2) * (kTcKeys * 128) + off, 16, 1024);
                        umma_f16(tmem + sb * kTcKeys, a, b, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&s_full[sb]));
                }
                if (j >= 1) {
                    const int jp = j - 1, stp = jp % kTcStages;
                    if (!mbar_wait(smem_u32(&p_full), jp & 1, err)) break;
                    tc_fence_after();
                    const uint32_t vbase = sbase + Ly::kOffKV + stp * Ly::kStageBytes + Ly::kKBytes;
#pragma unroll
                    for (int ks = 0; ks < kTcKeys / 16; ++ks) {
                        const uint64_t ah = sdesc_sw128(sbase + Ly::kOffPh + ks * 32, 16, 1024);
                        const uint64_t al = sdesc_sw128(sbase + Ly::kOffPl + ks * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(vbase + ks * 2048, kTcKeys * 128, 1024);
                        umma_f16(tmem + 128, ah, b, kIdescPV, (jp > 0 || ks > 0) ? 1u : 0u);
                        umma_f16(tmem + 128, al, b, kIdescPV, 1u);
                    }
                    umma_commit(smem_u32(&pv_done));
                    umma_commit(smem_u32(&kv_empty[stp]));
                }
            }
        }
    } else {
        // ------------------------------------------------ softmax warps 0-3
        const int rr = tid;                           // M row = TMEM lane
        const int grow = row0 + rr;
        const bool valid = grow < rows_total;
        const int pos_local = valid ? grow / group : 0;
        const int head = kvh * group + (valid ? grow - (grow / group) * group : 0);
        const int p_abs = valid ? ctx0 + pos_local : L - 1;   // padding rows see every key
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);

        // Q row -> shared memory, 128-byte swizzled rows, one 64-column half at a time
        {
            const uint4* qp = reinterpret_cast<const uint4*>(
                q + (static_cast<int64_t>(qs + pos_local) * n_q + head) * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = valid ? __ldg(qp + c) : make_uint4(0, 0, 0, 0);
                const uint32_t addr = sbase + Ly::kOffQ + (c >> 3) * (kTcRows * 128) + rr * 128 +
                                      (((c & 7) ^ (rr & 7)) << 4);
                st_shared_v4(addr, v.x, v.y, v.z, v.w);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&q_ready));
        }

        float m_used = -INFINITY, l = 0.f;
        bool broken = false;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            const bool ok = mbar_wait(smem_u32(&s_full[sb]), (j >> 1) & 1, err);
            if (!__all_sync(0xffffffffu, ok)) {
                broken = true;
                break;
            }
            tc_fence_after();
            uint32_t sr[64];
            {
                uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
                uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
                tmem_ld32(lane_addr + sb * kTcKeys, lo);
                tmem_ld32(lane_addr + sb * kTcKeys + 32, hi);
                tmem_ld_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_empty[sb]));

            const int key0 = j * kTcKeys;
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kTcKeys; ++i) {
                const float z = (key0 + i <= p_abs) ? __uint_as_float(sr[i]) * scale_log2 : -INFINITY;
                sr[i] = __float_as_uint(z);
                mx = fmaxf(mx, z);
            }
            const bool resc = mx > m_used + 8.f;      // lazy: only when the max grew a lot
            float fac = 1.f;
            if (resc) {
                fac = exp2f(m_used - mx);
                m_used = mx;
                l *= fac;
            }
            uint32_t ph[kTcKeys / 2], pl[kTcKeys / 2];
            float ps = 0.f;
#pragma unroll
            for (int i = 0; i < kTcKeys / 2; ++i) {
                const float p0 = exp2f(__uint_as_float(sr[2 * i]) - m_used);
                const float p1 = exp2f(__uint_as_float(sr[2 * i + 1]) - m_used);
                ps += p0 + p1;
                split_pair<T>(p0, p1, ph[i], pl[i]);
            }
            l += ps;

            if (j >= 1) {   // the previous P V is done: P buffer free, O stable
                const bool ok2 = mbar_wait(smem_u32(&pv_done), (j - 1) & 1, err);
                if (!__all_sync(0xffffffffu, ok2)) {
                    broken = true;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, resc)) {   // TMEM access is warp-wide
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(lane_addr + 128 + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac);
                        tmem_st32(lane_addr + 128 + c0, o);
                    }
                    tmem_st_wait();
                }
            }
#pragma unroll
            for (int c = 0; c < kTcKeys / 8; ++c) {
                const uint32_t sw = ((c ^ (rr & 7)) << 4);
                st_shared_v4(sbase + Ly::kOffPh + rr * 128 + sw, ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
                st_shared_v4(sbase + Ly::kOffPl + rr * 128 + sw, pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
            }
            if (key0 + kTcKeys > L) {
                // keys at or past L (only in the request's last tile) may hold
                // anything, even NaN: zero those V rows so P = 0 keeps them out
                const int valid_rows = max(0, L - key0);
                const int n16 = (kTcKeys - valid_rows) * 8 * Ly::kHalves;   // 16-byte pieces
                const uint32_t vb = sbase + Ly::kOffKV + (j % kTcStages) * Ly::kStageBytes + Ly::kKBytes;
                for (int i = tid; i < n16; i += 128) {
                    const int hx = i / ((kTcKeys - valid_rows) * 8);
                    const int rem = i - hx * ((kTcKeys - valid_rows) * 8);
                    st_shared_v4(vb + hx * (kTcKeys * 128) + valid_rows * 128 + rem * 16, 0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_full));
        }

        // ------------------------------------------------ epilogue: O / l
        if (!broken) {
            const bool ok = mbar_wait(smem_u32(&pv_done), (n_tiles - 1) & 1, err);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float inv = 1.f / l;
                const int64_t obase = (static_cast<int64_t>(qs + pos_local) * n_q + head) * D;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + 128 + c0, o);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * inv;
                    if (valid) store_row<T>(out, obase, c0, v, 32, out_dtype);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int D, int BS>
static cudaError_t run_prefill_tc(const PrefillArgs& a, cudaStream_t s, float sl2)
{
    using Ly = PfLayout<T, D>;
    auto kern = prefill_tc_kernel<T, D, BS>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(Ly::kDynBytes));
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap kmap, vmap;
    const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * a.cache.n_kv_heads * BS;
    if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, 64, 16) != PA_OK ||
        encode_pool_map(&vmap, a.v_cache, a.cache.dtype, D, rows, 64, 16) != PA_OK)
        return cudaErrorInvalidValue;
    const int group = a.n_q / a.cache.n_kv_heads;
    const int64_t tiles = (static_cast<int64_t>(a.max_q) * group + kTcRows - 1) / kTcRows;
    dim3 grid(static_cast<unsigned>(tiles), a.cache.n_kv_heads, a.num_reqs);
    kern<<<grid, kTcThreads, Ly::kDynBytes, s>>>(
        kmap, vmap, a.out, a.out_dtype, static_cast<const T*>(a.q), a.block_tables, a.max_blocks,
        a.q_start, a.context_lens, a.n_q, a.cache.n_kv_heads, group, a.cache.num_blocks, sl2, a.err);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t run_prefill_tc_dt(const PrefillArgs& a, cudaStream_t s, float sl2)
{
    const int D = a.cache.head_dim, BS = a.cache.block_size;
    if (D == 64 && BS == 16) return run_prefill_tc<T, 64, 16>(a, s, sl2);
    if (D == 64 && BS == 32) return run_prefill_tc<T, 64, 32>(a, s, sl2);
    if (D == 128 && BS == 16) return run_prefill_tc<T, 128, 16>(a, s, sl2);
    if (D == 128 && BS == 32) return run_prefill_tc<T, 128, 32>(a, s, sl2);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s)
{
    const float sl2 = a.scale * 1.4426950408889634f;
    if (a.cache.dtype == PA_BF16) return run_prefill_tc_dt<__nv_bfloat16>(a, s, sl2);
    if (a.cache.dtype == PA_F16) return run_prefill_tc_dt<__half>(a, s, sl2);
    return cudaErrorInvalidValue;
}

}  // namespace pa
