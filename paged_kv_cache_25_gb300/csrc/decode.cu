// Paged decode attention: one query row per (sequence, query head) against
// the sequence's K/V read through its block table ("How the attention kernel
// actually reads paged blocks": look the block up once, q.k against its keys,
// softmax-weighted sum of its values).  The tensor-core kernel lives in
// decode_mma.cuh; this file holds the CUDA-core kernel (fp32 pools and other
// head dims), the split-K reduce and the launch.
#include "decode_mma.cuh"

namespace pa {

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
    // tokens in groups of kTok: their K/V rows are loaded before any of them is
    // used, so the loads of a group overlap (one token at a time left every
    // warp waiting on one row's latency per token)
    constexpr int kTok = 4;
    const int32_t* table = block_tables + static_cast<int64_t>(s) * max_blocks;
    for (int p0 = tok0; p0 < tok1; p0 += kTok) {
        float kf[kTok][DPL], vf[kTok][DPL];
        bool bad = false;
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            const int p = p0 + u;
            if (p < tok1) {
                const int lb = p / block_size;
                const int b = lb < max_blocks ? __ldg(table + lb) : -1;
                bad = bad || b < 0 || b >= num_blocks;
                const int64_t row = (static_cast<int64_t>(b < 0 ? 0 : b) * n_kv + kvh) * block_size +
                                    p % block_size;
                const T* kr = kc + row * D;
                const T* vr = vc + row * D;
#pragma unroll
                for (int i = 0; i < DPL; ++i) {
                    kf[u][i] = b < 0 || b >= num_blocks ? 0.f : Cvt<T>::to_f(kr[lane + 32 * i]);
                    vf[u][i] = b < 0 || b >= num_blocks ? 0.f : Cvt<T>::to_f(vr[lane + 32 * i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < DPL; ++i) kf[u][i] = vf[u][i] = 0.f;
            }
        }
        if (bad) {                 // the same block ids in every lane: uniform
            set_error(err, PA_ERR_OUT_OF_RANGE);
            return;
        }
        float z[kTok];
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) dot = fmaf(qv[i], kf[u][i], dot);
            z[u] = dot;
        }
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
#pragma unroll
            for (int u = 0; u < kTok; ++u) z[u] += __shfl_xor_sync(0xffffffffu, z[u], w);
        float m_new = m_run;
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            z[u] = p0 + u < tok1 ? z[u] * scale_log2 : -INFINITY;
            m_new = fmaxf(m_new, z[u]);
        }
        const float alpha = exp2f(m_run - m_new);   // 0 on the first group (m_run = -inf)
        float pz[kTok], psum = 0.f;
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            pz[u] = p0 + u < tok1 ? exp2f(z[u] - m_new) : 0.f;
            psum += pz[u];
        }
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            float a = acc[i] * alpha;
#pragma unroll
            for (int u = 0; u < kTok; ++u) a = fmaf(pz[u], vf[u][i], a);
            acc[i] = a;
        }
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

// Second pass, one warp per (sequence, query head):
//   out = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j.
template <int DPL>
__global__ void __launch_bounds__(128)
decode_reduce_kernel(void* __restrict__ out, pa_dtype out_dtype,
                     const int32_t* __restrict__ context_lens, const float* __restrict__ ws_ml,
                     const float* __restrict__ ws_acc, int num_seqs, int n_q, int nq,
                     int part_tokens, int max_parts)
{
    constexpr int D = DPL * 32;
    const int lane = threadIdx.x & 31;
    grid_dependency_wait();   // launched as a programmatic dependent of the partial kernel
    // one warp per output row ((sequence, query) x head)
    const int64_t sh = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    if (sh >= static_cast<int64_t>(num_seqs) * nq * n_q) return;
    const int s = static_cast<int>(sh / (static_cast<int64_t>(nq) * n_q));
    const int L = __ldg(context_lens + s);
    const int J = min((L + part_tokens - 1) / part_tokens, max_parts);
    if (J <= 1) return;
    const float* ml = ws_ml + 2 * sh * max_parts;
    float M = -INFINITY;
    for (int jj = lane; jj < J; jj += 32) M = fmaxf(M, ml[2 * jj]);
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, w));
    float lsum = 0.f;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    const float* a = ws_acc + sh * max_parts * D;
    for (int jj = 0; jj < J; ++jj) {
        const float w = exp2f(ml[2 * jj] - M);
        lsum += w * ml[2 * jj + 1];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(w, a[jj * D + lane + 32 * i], acc[i]);
    }
    const float inv = 1.f / lsum;
#pragma unroll
    for (int i = 0; i < DPL; ++i) store_any(out, sh * D + lane + 32 * i, acc[i] * inv, out_dtype);
}

// ------------------------------------------------------------------ launch

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

static cudaError_t run_reduce(const DecodeArgs& a, cudaStream_t s)
{
    const int64_t pairs = static_cast<int64_t>(a.num_seqs) * a.q_per_seq * a.n_q;
    const unsigned grid = static_cast<unsigned>((pairs + 3) / 4);
    // a programmatic dependent of the partial kernel: its launch overlaps that
    // kernel's tail, and it waits for the partials before reading them
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define PA_REDUCE(DPL)                                                                            \
    cudaLaunchKernelEx(&cfg, decode_reduce_kernel<DPL>, a.out, a.out_dtype, a.context_lens,       \
                       static_cast<const float*>(a.ws_ml), static_cast<const float*>(a.ws_acc),  \
                       a.num_seqs, a.n_q, a.q_per_seq, a.part_tokens, a.max_parts)
    switch (a.cache.head_dim) {
        case 32: return PA_REDUCE(1);
        case 64: return PA_REDUCE(2);
        case 96: return PA_REDUCE(3);
        case 128: return PA_REDUCE(4);
        case 256: return PA_REDUCE(8);
        default: return cudaErrorInvalidValue;
    }
#undef PA_REDUCE
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s)
{
    const float sl2 = a.scale * 1.4426950408889634f;   // softmax in base 2
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    profile_events(&ev0, &ev1);
    if (ev0) cudaEventRecord(ev0, s);
    cudaError_t e;
    if (a.q_per_seq > 1) {
        e = launch_decode_mq(a, s, sl2);
    } else {
        e = run_mma_any<false>(a, s, sl2);
        if (e == cudaErrorNotSupported) {        // fp32 pools, other head dims
            switch (a.cache.dtype) {
                case PA_BF16: e = run_simt_dt<__nv_bfloat16>(a, s, sl2); break;
                case PA_F16: e = run_simt_dt<__half>(a, s, sl2); break;
                default: e = run_simt_dt<float>(a, s, sl2); break;
            }
        }
    }
    if (ev1) cudaEventRecord(ev1, s);
    if (e != cudaSuccess) return e;
    if (a.max_parts > 1) e = run_reduce(a, s);
    return e;
}

}  // namespace pa
