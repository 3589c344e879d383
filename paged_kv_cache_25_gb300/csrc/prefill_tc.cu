// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05).
//
// Semantics ("The hands-on guide to LLM Inference with vLLM", chunked
// prefill): query row i of request r's chunk of C_r rows sits at absolute
// position L_r - C_r + i and attends logical K/V rows 0 .. that position,
// read through the request's block table; the chunk's own K/V are already in
// the pool.
//
// CTA = (256 M rows, KV head, request) as two 128-row tiles A and B that share
// one stream of K/V.  The M rows are (position, head) pairs of one GQA group,
// position-major, so one pass over the keys serves all the query heads that
// share the KV head.  Keys go in tiles of 128.
//   warps 16, 17: TMA producers: 16-row K (warp 16) and V (warp 17) slabs of
//             each 128-key tile into their own 2-stage rings (128-byte swizzle),
//             one block-table lookup per block (FP8 pools: see below);
//   last warp: the MMA issuer, a warp-wide loop in which one elected lane
//             issues S_t = Q_t K^T (M 128, N 128, K = d) into TMEM and
//             O_t += P_t V (M 128, N = d, K 128) into TMEM, in the order
//             P_A(j) V, S_A(j+1), P_B(j) V, S_B(j+1): while one tile's rows run
//             their softmax the tensor cores work on the other tile;
//   warps 0-15: two threads per M row of a tile (warps 0-3 and 8-11 tile A,
//             4-7 and 12-15 tile B), each with 64 of a key tile's 128 keys and
//             half of O's columns; the pair swaps partial row maxima through
//             shared memory and a named barrier.  A row reads its scores from
//             TMEM, applies the causal mask on absolute positions,
//             runs the online softmax in base 2 with lazy rescaling (O in TMEM
//             is rescaled only when the running max grows by more than 2^8),
//             and writes P back over its scores in TMEM: as hi + lo bf16
//             halves with bf16 operands (P V keeps ~16 bits of P), as one fp16
//             part with fp16 operands (11 bits); the P V MMA takes P straight
//             from TMEM.  At the end O / l goes to global memory.
// FP8 (E4M3) pools: converter warps replace the two producers; they copy the
// codes chunk by chunk into staging buffers and widen them exactly to fp16 in
// the same rings (V kept in the pool's transposed [d][keys] pieces, a K-major
// operand of P V); keys at or past the context are written as zeros.  The
// MMAs run on fp16 operands (bf16 queries are scaled into fp16 per row), except
// that with head_dim 128 and bf16 queries the score MMAs read the K codes
// themselves (a K-loader warp TMAs them; two converters widen V alone).
// k_scale is folded into the softmax scale and v_scale into the output.
// All waits are bounded; the kernel never traps.
#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"

#include <math.h>

#include <mutex>
#include <type_traits>

namespace pa {

// Four MMAs into one accumulator from a converged warp, under one election:
// D (+)= A_i B_i for i = 0..3 in that order, the first accumulating only if
// `acc`, the others always.  Next to the busy softmax warps the issuing warp
// gets few issue slots, so fewer instructions per MMA issue faster.
// A and B from shared memory (kind::f16, or kind::f8f6f4 with E4M3 codes):
template <bool kF8>
__device__ __forceinline__ void umma4_ss(uint32_t d, uint64_t a0, uint64_t b0, uint64_t a1, uint64_t b1,
                                         uint64_t a2, uint64_t b2, uint64_t a3, uint64_t b3,
                                         uint32_t idesc, uint32_t acc)
{
    if constexpr (kF8) {
        asm volatile(
            "{\n\t.reg .pred e, p, q;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %10, 0;\n\t"
            "setp.eq.b32 q, %9, %9;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %9, p;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %4, %9, q;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %5, %6, %9, q;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %7, %8, %9, q;\n\t}" ::"r"(d),
            "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc),
            "r"(acc)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred e, p, q;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %10, 0;\n\t"
            "setp.eq.b32 q, %9, %9;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %9, p;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %9, q;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %9, q;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %9, q;\n\t}" ::"r"(d),
            "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc),
            "r"(acc)
            : "memory");
    }
}

// the same with A from tensor memory (kind::f16)
__device__ __forceinline__ void umma4_ts(uint32_t d, uint32_t a0, uint64_t b0, uint32_t a1, uint64_t b1,
                                         uint32_t a2, uint64_t b2, uint32_t a3, uint64_t b3,
                                         uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred e, p, q;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 q, %9, %9;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %9, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %9, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %9, q;\n\t}" ::"r"(d),
        "r"(a0), "l"(b0), "r"(a1), "l"(b1), "r"(a2), "l"(b2), "r"(a3), "l"(b3), "r"(idesc),
        "r"(acc)
        : "memory");
}

constexpr int kTcRows = 128;      // M rows per tile
constexpr int kTcTiles = 2;       // tiles per CTA (A, B)
constexpr int kTcKeys = 128;      // keys per key tile
constexpr int kTcStages = 2;      // K/V ring depth
constexpr int kRankedReqs = 64;   // requests ordered by context length, at most
constexpr int kSoftmaxWarps = 8 * kTcTiles;   // two threads per row of each tile
constexpr int kKWarp = kSoftmaxWarps, kVWarp = kSoftmaxWarps + 1;
// FP8 pools: converter warps widen codes into the rings.  In general a key
// tile is 2 x (128 / kF8ChunkKeys) chunks (K's, then V's) for three converters
// and chunk g of the whole sequence goes to converter g % 3.  With head_dim 128
// and bf16 queries the score MMA reads the K codes as they are (kind::f8f6f4;
// each q row, scaled by a power of two, is exactly the sum of two E4M3 parts):
// a loader warp of its own TMAs the codes into the K ring and two converters
// widen V alone (three measured 2 % slower).  (An fp16 query has 11
// significant bits, more than two E4M3 parts carry.)
constexpr int kF8ChunkKeys = 32;   // keys per staged chunk of codes (16 or 32)
constexpr int kF8MaxConverters = 3;
constexpr int kF8MaxDepth = 2;     // staging buffers per converter
template <bool F8, int D, bool BQ>
struct PfMode {
    static constexpr bool kDirectK = F8 && D == 128 && BQ;   // K codes straight into the score MMA
    static constexpr int kConverters = F8 ? (kDirectK ? 2 : 3) : 0;
    static constexpr int kKLoaders = kDirectK ? 1 : 0;   // direct K: a warp TMAs the K codes
    static constexpr int kDepth = 2;
};
// Warps after the softmax ones: the K and V producers (or the FP8
// converters, and with direct K the K-code loader), then the MMA issuer.
template <bool F8, int D, bool BQ>
struct PfWarps {
    using Mode = PfMode<F8, D, BQ>;
    static constexpr int kProducers = F8 ? Mode::kConverters + Mode::kKLoaders : 2;
    static constexpr int kFirstConverter = kSoftmaxWarps;
    static constexpr int kKLoader = kFirstConverter + Mode::kConverters;   // (direct K only)
    static constexpr int kMma = kSoftmaxWarps + kProducers;
    static constexpr int kThreads = (kMma + 1) * 32;
    // the register file is split per SM sub-partition: 20 warps (5 on each)
    // keep 96 registers a thread, 21 would leave 80 and spill the softmax
    static_assert(kMma + 1 <= 20, "at most 20 warps");
};
constexpr uint32_t kTmemCols = 512;   // S/P_A [0,128) S/P_B [128,256) O_A, O_B from 256

template <typename T, int D, bool F8, bool BQ>
struct PfLayout {
    static constexpr bool kDirectK = PfMode<F8, D, BQ>::kDirectK;
    static constexpr int kHalves = D / 64;
    // one Q tile: 16-bit rows, or (direct K) the E4M3 hi part then the lo part
    static constexpr uint32_t kQBytes = kTcRows * D * 2;
    static constexpr uint32_t kQLo = kTcRows * D;                 // direct K: offset of the lo part
    static constexpr uint32_t kKBytes = kTcKeys * D * (kDirectK ? 1 : 2);   // K of one key tile
    static constexpr uint32_t kVBytes = kTcKeys * D * 2;          // V of one key tile (16-bit)
    static constexpr uint32_t kCodeBytes = kF8ChunkKeys * D;      // FP8: codes of one staged chunk
    static constexpr uint32_t kOffQ = 0;                          // Q_A, Q_B
    static constexpr uint32_t kOffK = kOffQ + kTcTiles * kQBytes; // K ring
    static constexpr uint32_t kOffV = kOffK + kTcStages * kKBytes;   // V ring
    static constexpr uint32_t kOffCS = kOffV + kTcStages * kVBytes;  // FP8: 2 code buffers per converter
    static constexpr uint32_t kDynBytes =
        kOffCS + PfMode<F8, D, BQ>::kConverters * PfMode<F8, D, BQ>::kDepth * kCodeBytes + 1024;
    // S_t at t * 128; P_t overwrites it, keys 32c .. 32c+31 as hi in columns
    // 32c .. 32c+15 and (bf16 operands) lo in 32c+16 .. 32c+31 (two 16-bit
    // values per column)
    static constexpr uint32_t kTmemS = 0;
    static constexpr uint32_t kTmemO = 256;                       // + t * D
    static_assert(kDynBytes <= 232448, "shared memory per CTA");
    static_assert(kTmemO + kTcTiles * D <= kTmemCols, "tensor memory columns");
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

// Four E4M3 codes -> four fp16 values (exact: every E4M3 value is an fp16
// normal or zero), as two packed pairs, by the hardware pair conversion.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Sixteen codes of k-order positions i (low byte first) with the ones at or
// past `keep` replaced by zeros.
__device__ __forceinline__ uint4 keep_codes(uint4 c, int keep)
{
    uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int k = min(4, max(0, keep - 4 * e));
        w[e] &= k >= 4 ? 0xFFFFFFFFu : ((1u << (8 * k)) - 1u);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// T: the MMA operand type (P, K, V and the staged Q); QT: the type q arrives
// in.  They differ only for FP8 pools with bf16 activations, which run on fp16
// operands (the codes widen to fp16 in one instruction a pair): each q row is
// scaled by a power of two 2^-e into fp16 (exact for bf16 values down to 2^-28
// of the row's largest) and 2^e goes into that row's softmax scale.
template <typename T, typename QT, int D, int BS, bool F8 = false>
__global__ void __launch_bounds__(PfWarps<F8, D, std::is_same<QT, __nv_bfloat16>::value>::kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const uint8_t* __restrict__ k_codes, const uint8_t* __restrict__ v_codes,
                  void* __restrict__ out, pa_dtype out_dtype, const QT* __restrict__ q,
                  const int32_t* __restrict__ block_tables, int max_blocks,
                  const int32_t* __restrict__ q_start, const int32_t* __restrict__ context_lens,
                  int max_q, int n_q, int n_kv, int group, int num_blocks, float scale_log2,
                  float v_scale, unsigned* err)
{
    constexpr bool kBq = std::is_same<QT, __nv_bfloat16>::value;
    using Ly = PfLayout<T, D, F8, kBq>;
    using Wp = PfWarps<F8, D, kBq>;
    constexpr bool kDirectK = Ly::kDirectK;
    constexpr int kMmaWarp = Wp::kMma;
    constexpr int kFirstConv = Wp::kFirstConverter;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    // P for P V: fp16 operands (fp16 and FP8 pools) take P as one fp16 part,
    // 11 significant bits, so each output moves by at most 2^-12 of the
    // largest |v| it averages; bf16 operands take P as hi + lo bf16 parts
    // (8 significant bits each, ~16 together)
    constexpr bool kOneP = !kBf16;
    constexpr uint32_t kIdescQK = idesc_f16(kBf16, false, false, kTcRows, kTcKeys);
    // kind::f8f6f4 with E4M3 A and B (type code 0 in both fields), fp32 accumulate
    constexpr uint32_t kIdescQK8 = idesc_f16(false, false, false, kTcRows, kTcKeys);
    // P V: V as [keys][d] (MN-major) from 16-bit pools, as [d][keys] (K-major) from FP8
    constexpr uint32_t kIdescPV = idesc_f16(kBf16, false, !F8, kTcRows, D);
    static_assert(BS % 16 == 0 && kTcKeys % BS == 0, "block size must divide the key tile");

    // heavier CTAs first, as the grid is scheduled in index order: the z index
    // is the request's rank by context length (longest first, ties by index;
    // up to kRankedReqs requests, else request order), and within a request
    // the last position blocks, which see the most keys, come first
    static_assert(kRankedReqs <= Wp::kThreads, "one thread per ranked request");
    int r = blockIdx.z;
    if (gridDim.z > 1 && gridDim.z <= kRankedReqs) {
        __shared__ int s_req;
        const int R = gridDim.z, i = threadIdx.x;
        if (i < R) {
            const int Li = __ldg(context_lens + i);
            int rank = 0;
            for (int k = 0; k < R; ++k) {
                const int Lk = __ldg(context_lens + k);
                rank += (Lk > Li || (Lk == Li && k < i)) ? 1 : 0;
            }
            if (rank == static_cast<int>(blockIdx.z)) s_req = i;
        }
        __syncthreads();
        r = s_req;
    }
    const int blk = gridDim.x - 1 - blockIdx.x;
    const int kvh = blockIdx.y;
    const int qs = __ldg(q_start + r);
    const int C = __ldg(q_start + r + 1) - qs;
    const int L = __ldg(context_lens + r);
    const int rows_total = C * group;
    const int row0 = blk * (kTcTiles * kTcRows);
    // the grid covers max_q rows per request: a longer chunk would leave its
    // last rows unwritten, so it is flagged (once, by the request's first CTA)
    if (C > max_q && blk == 0 && threadIdx.x == 0) set_error(err, PA_ERR_OUT_OF_RANGE);
    if (row0 >= rows_total) return;
    if (C > L || C < 0) {
        if (threadIdx.x == 0) set_error(err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int ctx0 = L - C;
    // key tiles each tile's rows need (0: the tile has no rows); when both
    // tiles have rows, n_t[0] <= n_t[1]
    int n_t[kTcTiles];
#pragma unroll
    for (int t = 0; t < kTcTiles; ++t) {
        const int first = row0 + t * kTcRows;
        const int last = min(rows_total, first + kTcRows) - 1;
        n_t[t] = first < rows_total ? (ctx0 + last / group) / kTcKeys + 1 : 0;
    }
    const int n_tiles = max(n_t[0], n_t[1]);

    // Every barrier below is waited on in completion order and its waiter is
    // never two phases behind: S_t(j + 1) is issued after P_t(j) V, which
    // waits for P_t(j), which needs S_t(j).
    __shared__ __align__(8) uint64_t k_full[kTcStages], k_empty[kTcStages];
    __shared__ __align__(8) uint64_t v_full[kTcStages], v_empty[kTcStages];
    __shared__ __align__(8) uint64_t s_full[kTcTiles], p_full[kTcTiles], pv_done[kTcTiles], q_ready;
    __shared__ __align__(8) uint64_t code_full[kF8MaxConverters][kF8MaxDepth];   // FP8: codes landed, per converter and buffer
    __shared__ uint32_t s_tmem;
    // partial row maxima of the two threads of a row (double-buffered by key
    // tile), a "stop" flag beside each, and the partial row sums at the end
    __shared__ float xmax[2][kTcTiles][2][kTcRows];
    __shared__ uint8_t xstop[2][kTcTiles][2][kTcRows];
    __shared__ float xsum[kTcTiles][2][kTcRows];
    __shared__ uint8_t xstop_end[kTcTiles][2][kTcRows];
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            // FP8: one arrival per widened chunk; 16-bit pools and the direct
            // K codes: the TMA's
            mbar_init(smem_u32(&k_full[i]), F8 && !kDirectK ? kTcKeys / kF8ChunkKeys : 1);
            mbar_init(smem_u32(&k_empty[i]), 1);
            mbar_init(smem_u32(&v_full[i]), F8 ? kTcKeys / kF8ChunkKeys : 1);
            mbar_init(smem_u32(&v_empty[i]), 1);
        }
        for (int t = 0; t < kTcTiles; ++t) {
            mbar_init(smem_u32(&s_full[t]), 1);
            mbar_init(smem_u32(&p_full[t]), 8);
            mbar_init(smem_u32(&pv_done[t]), 1);
        }
        mbar_init(smem_u32(&q_ready), kSoftmaxWarps);
        for (int i = 0; i < kF8MaxDepth * kF8MaxConverters; ++i)
            mbar_init(smem_u32(&code_full[i / kF8MaxDepth][i % kF8MaxDepth]), 1);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    static_assert(!F8 || std::is_same<T, __half>::value, "FP8 codes widen to fp16 operands");
    if (F8 && warp >= kFirstConv && warp < kFirstConv + Wp::Mode::kConverters) {
        // ------------------------------------------------ FP8 converters
        // Chunk g (tile g / kPerTile; K chunks first, then V) is widened by
        // converter g % kNc into its ring stage, which then gets
        // one arrival on its full barrier.  Each converter's chunks pass
        // through kDepth staging buffers: while it widens its chunk n, chunks
        // n + 1 .. n + kDepth - 1 are in flight, and lane 0 requests chunk
        // n + kDepth into the same buffer once the warp has read it (the chunk
        // is at most two key tiles ahead).  The block ids of a tile's 16-key pieces
        // (one per lane) are loaded a tile ahead.
        // (direct K: V chunks only)
        constexpr int kCK = kF8ChunkKeys, kChunks = kTcKeys / kCK, kBoxes = kCK / 16;
        constexpr int kKChunks = kDirectK ? 0 : kChunks;       // K chunks per tile
        constexpr int kPerTile = kKChunks + kChunks;
        constexpr int kNc = F8 ? Wp::Mode::kConverters : 1;     // (16-bit pools never get here)
        constexpr int kDepth = Wp::Mode::kDepth;
        const int pw = warp - kFirstConv;
        const int total = (kPerTile * n_tiles - pw + kNc - 1) / kNc;   // this warp's chunks
        const uint32_t stage = sbase + Ly::kOffCS + pw * kDepth * Ly::kCodeBytes;
        const uint8_t* stage_ptr = smem + Ly::kOffCS + pw * kDepth * Ly::kCodeBytes;
        const uint64_t* cbars = code_full[pw];
        const int32_t* table = block_tables + static_cast<int64_t>(r) * max_blocks;
        // lane c < 8: raw block id of 16-key piece c of tile t (-1: past the
        // table; 0 for pieces at or past L, whose codes become zeros)
        auto piece_ids = [&](int t) -> int {
            const int key0 = t * kTcKeys + (lane & 7) * 16;
            if (lane >= 8 || t >= n_tiles || key0 >= L) return 0;
            return key0 / BS < max_blocks ? __ldg(table + key0 / BS) : -1;
        };
        // ids[0] / ids[1]: pieces of tiles id_tile and id_tile + 1
        int id_tile = 0;
        int ids[2] = {piece_ids(0), piece_ids(1)};
        auto request = [&](int n) {   // whole warp: this warp's chunk n
            const int g = pw + kNc * n, j = g / kPerTile, item = g % kPerTile;
            const bool k_chunk = item < kKChunks;
            const int e = k_chunk ? item : item - kKChunks;
            const int src_ids = j == id_tile ? ids[0] : ids[1];   // j <= id_tile + 1
            int bb[kBoxes];
#pragma unroll
            for (int x = 0; x < kBoxes; ++x) bb[x] = __shfl_sync(0xffffffffu, src_ids, e * kBoxes + x);
            if (lane == 0) {
                const uint32_t bar = smem_u32(&cbars[n % kDepth]);
                const uint32_t buf = stage + (n % kDepth) * Ly::kCodeBytes;
                mbar_arrive_expect_tx(bar, Ly::kCodeBytes);
#pragma unroll
                for (int x = 0; x < kBoxes; ++x) {
                    const int key0 = j * kTcKeys + e * kCK + x * 16;
                    int b = bb[x];
                    if (b < 0 || b >= num_blocks) {
                        set_error(err, PA_ERR_OUT_OF_RANGE);
                        b = 0;
                    }
                    // 16 rows of D codes (K), or the D x 16 transposed piece
                    // (V): 16 * D contiguous bytes of the pool either way
                    const int64_t bh = static_cast<int64_t>(b) * n_kv + kvh;
                    const uint8_t* src =
                        k_chunk ? k_codes + (bh * BS + key0 % BS) * D
                                : v_codes + (bh * (BS / 16) + (key0 % BS) / 16) * (16 * D);
                    bulk_load(buf + x * 16 * D, src, 16 * D, bar);
                }
            }
        };
        // on a wait that ran out (error recorded): let the copies of chunks n
        // and n + 1 land (bounded) before the CTA can exit
        auto drain = [&](int n) {
            for (int m = n; m < min(n + kDepth, total); ++m)
                mbar_wait(smem_u32(&cbars[m % kDepth]), (m / kDepth) & 1, err);
        };
        for (int n = 0; n < min(kDepth, total); ++n) request(n);
#pragma unroll 1
        for (int n = 0; n < total; ++n) {
            const int g = pw + kNc * n, j = g / kPerTile, item = g % kPerTile;
            const bool k_chunk = item < kKChunks;
            const int e = k_chunk ? item : item - kKChunks;
            const int st = j % kTcStages;
            if (j >= kTcStages &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&(k_chunk ? k_empty : v_empty)[st]),
                                                   ((j / kTcStages) - 1) & 1, err))) {
                drain(n);
                break;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&cbars[n % kDepth]), (n / kDepth) & 1, err))) {
                drain(n);
                break;
            }
            const uint32_t dst = k_chunk ? sbase + Ly::kOffK + st * Ly::kKBytes
                                         : sbase + Ly::kOffV + st * Ly::kVBytes;
            const int keep_tile = L - j * kTcKeys;        // valid keys of this tile (may exceed 128)
            // kCK x D codes in units of 16: one K row's d-chunk pair p (or one
            // V^T row of a 16-key piece), each widened into two 16-byte ring
            // chunks.  Every 8 lanes touch 8 distinct 16-byte bank groups in
            // the staging reads and in the ring writes.
            constexpr int kPer = kCK * D / 512;
            const uint8_t* src = stage_ptr + (n % kDepth) * Ly::kCodeBytes;
            uint4 c[kPer];
            int row[kPer], chunk0[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                int su;   // staging unit
                if (k_chunk) {
                    int rl, p;   // row in the chunk, d-chunk pair
                    if constexpr (D == 128) {
                        const int gg = lane >> 3, l8 = lane & 7;
                        rl = 4 * i + 2 * (gg >> 1) + ((l8 >> 2) ^ (gg & 1));
                        p = l8;
                    } else {
                        const int u = lane + 32 * i;
                        rl = u / (D / 16);
                        p = u % (D / 16);
                    }
                    su = rl * (D / 16) + p;
                    row[i] = e * kCK + rl;
                    chunk0[i] = 2 * p;
                } else {
                    su = lane + 32 * i;                      // piece su / D, row d
                    row[i] = su % D;
                    chunk0[i] = 2 * (e * kBoxes + su / D);   // key chunk (8 keys)
                }
                c[i] = *reinterpret_cast<const uint4*>(src + su * 16);
            }
            if (keep_tile < kTcKeys) {   // the tail tile: keys at or past L become zeros
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    if (k_chunk) {
                        if (row[i] >= keep_tile) c[i] = make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        c[i] = keep_codes(c[i], keep_tile - 8 * chunk0[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                uint32_t w[8];
                widen4(c[i].x, w[0], w[1]);
                widen4(c[i].y, w[2], w[3]);
                widen4(c[i].z, w[4], w[5]);
                widen4(c[i].w, w[6], w[7]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ch = chunk0[i] + h;
                    const int rw = row[i];
                    // K: [keys][d] in 64-column halves; V: [d][keys] in 64-key halves
                    const uint32_t addr = dst + (ch >> 3) * ((k_chunk ? kTcKeys : D) * 128) +
                                          rw * 128 + (((ch & 7) ^ (rw & 7)) << 4);
                    st_shared_v4(addr, w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
                }
            }
            fence_proxy_async_smem();   // ring writes -> the MMAs' reads
            __syncwarp();               // and every lane has read the staging buffer
            if (lane == 0) mbar_arrive(smem_u32(&(k_chunk ? k_full : v_full)[st]));
            if (n + kDepth < total) {
                const int jn = (pw + kNc * (n + kDepth)) / kPerTile;
                if (jn > id_tile + 1) {   // move the id window one tile on
                    id_tile += 1;
                    ids[0] = ids[1];
                    ids[1] = piece_ids(id_tile + 1);
                }
                request(n + kDepth);
            }
        }
    } else if ((!F8 && (warp == kKWarp || warp == kVWarp)) || (kDirectK && warp == Wp::kKLoader)) {
        // ------------------------------------------------ TMA producers
        // K and V have separate rings: K of key tile j is released once both
        // S_t(j) are done, V of tile j once both P_t(j) V are.  With direct K
        // (FP8 pool) one warp loads the K codes: a tile is 8 boxes of 16 rows x
        // 128 codes, 128-byte swizzled, as the score MMA reads them.
        if (lane == 0) {
            const bool is_k = F8 || warp == kKWarp;
            const CUtensorMap* map = is_k ? &kmap : &vmap;
            uint64_t* full_bar = is_k ? k_full : v_full;
            uint64_t* empty_bar = is_k ? k_empty : v_empty;
            const uint32_t ring_base = sbase + (is_k ? Ly::kOffK : Ly::kOffV);
            const uint32_t tile_bytes = is_k ? Ly::kKBytes : Ly::kVBytes;
            prefetch_tensormap(map);
            // block ids of the 16-key pieces of a tile, read a tile ahead: eight
            // independent loads whose latency the wait for a free stage hides
            // (read next to each copy they would be serial, the copies being
            // ordered after them)
            constexpr int kPieces = kTcKeys / 16;
            const int32_t* table = block_tables + static_cast<int64_t>(r) * max_blocks;
            auto tile_ids = [&](int j, int (&ids)[kPieces]) {
#pragma unroll
                for (int c = 0; c < kPieces; ++c) {
                    const int key0 = j * kTcKeys + c * 16;
                    const int lb = key0 / BS;
                    // past L the tile's rows are masked: reuse the last block
                    ids[c] = (j >= n_tiles || key0 >= L) ? (c > 0 ? ids[c - 1] : 0)
                                                          : (lb < max_blocks ? __ldg(table + lb) : -1);
                }
            };
            int ids[kPieces], ids_next[kPieces];
            tile_ids(0, ids);
            int loaded = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kTcStages;
                tile_ids(j + 1, ids_next);
                if (j >= kTcStages &&
                    !mbar_wait(smem_u32(&empty_bar[st]), ((j / kTcStages) - 1) & 1, err))
                    break;
                const uint32_t full = smem_u32(&full_bar[st]);
                const uint32_t dst = ring_base + st * tile_bytes;
                mbar_arrive_expect_tx(full, tile_bytes);
#pragma unroll
                for (int c = 0; c < kPieces; ++c) {
                    const int key0 = j * kTcKeys + c * 16;
                    int b = ids[c];
                    if (b < 0 || b >= num_blocks) {
                        set_error(err, PA_ERR_OUT_OF_RANGE);
                        b = 0;   // keep the ring moving; the outputs are flagged invalid
                    }
                    const int row = (b * n_kv + kvh) * BS + (key0 % BS);
                    if constexpr (F8) {
                        tma_load_2d(dst + c * 2048, map, 0, row, full);
                    } else {
#pragma unroll
                        for (int hx = 0; hx < Ly::kHalves; ++hx)
                            tma_load_2d(dst + hx * (kTcKeys * 128) + c * 2048, map, hx * 64, row, full);
                    }
                }
                loaded = j + 1;
#pragma unroll
                for (int c = 0; c < kPieces; ++c) ids[c] = ids_next[c];
            }
            // the last two tiles' copies have landed before the warp can leave
            // (already so unless a wait above ran out; bounded)
            for (int m = max(0, loaded - kTcStages); m < loaded; ++m)
                mbar_wait(smem_u32(&full_bar[m % kTcStages]), (m / kTcStages) & 1, err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the issue loop (warp-uniform descriptors; one
        // elected lane issues each MMA and commit).  Descriptors are built once;
        // each MMA only adds a constant to the start-address field (16-byte
        // units; every operand lies below 256 KB).
        {
            const uint64_t dq = sdesc_sw128(sbase + Ly::kOffQ, 16, 1024);
            const uint64_t dk = sdesc_sw128(sbase + Ly::kOffK, 16, 1024);
            // V: MN-major [keys][d] halves (16-bit pools) or K-major [d][keys] halves (FP8)
            const uint64_t dv = F8 ? sdesc_sw128(sbase + Ly::kOffV, 16, 1024)
                                   : sdesc_sw128(sbase + Ly::kOffV, kTcKeys * 128, 1024);
            constexpr uint32_t kQHalf = (kTcRows * 128) >> 4, kKHalf = (kTcKeys * 128) >> 4;
            constexpr uint32_t kKStage = Ly::kKBytes >> 4, kVStage = Ly::kVBytes >> 4;
            constexpr uint32_t kQTile = Ly::kQBytes >> 4, kQLo = Ly::kQLo >> 4;
            // S_t(j) = Q_t K_j^T; the K stage is released after the last tile's
            auto issue_qk = [&](int t, int j) {
                const int st = j % kTcStages;
                const uint64_t dks = dk + st * kKStage;
                const uint32_t d_s = tmem + Ly::kTmemS + t * 128;
                const uint64_t dqt = dq + t * kQTile;
                if constexpr (kDirectK) {
                    // E4M3 x E4M3: 32 codes (32 bytes) per k-step of the one
                    // 128-byte row; q's hi part, then its lo part, into S
                    static_assert(D == 128, "four k-steps of 32 codes");
#pragma unroll
                    for (int kk = 0; kk < D / 32; kk += 2)
                        umma4_ss<true>(d_s, dqt + kk * 2, dks + kk * 2, dqt + kQLo + kk * 2, dks + kk * 2,
                                       dqt + (kk + 1) * 2, dks + (kk + 1) * 2,
                                       dqt + kQLo + (kk + 1) * 2, dks + (kk + 1) * 2, kIdescQK8,
                                       kk > 0 ? 1u : 0u);
                } else {
                    // 32 bytes per k-step; 4 k-steps per 64-element half
                    auto oq = [&](int kk) { return static_cast<uint32_t>((kk >> 2) * kQHalf + (kk & 3) * 2); };
                    auto ok_ = [&](int kk) { return static_cast<uint32_t>((kk >> 2) * kKHalf + (kk & 3) * 2); };
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk += 4)
                        umma4_ss<false>(d_s, dqt + oq(kk), dks + ok_(kk), dqt + oq(kk + 1), dks + ok_(kk + 1),
                                        dqt + oq(kk + 2), dks + ok_(kk + 2), dqt + oq(kk + 3),
                                        dks + ok_(kk + 3), kIdescQK, kk > 0 ? 1u : 0u);
                }
                umma_commit_elect(smem_u32(&s_full[t]));
            };
            // O_t += P_t(j) V_j, P from TMEM (hi, and lo for bf16, of each 16 keys)
            auto issue_pv = [&](int t, int j) {
                const int st = j % kTcStages;
                const uint64_t dvs = dv + st * kVStage;
                const uint32_t d_o = tmem + Ly::kTmemO + t * D;
                const uint32_t a_p = tmem + Ly::kTmemS + t * 128;
                // keys 16 ks .. +15: 32-key chunk ks / 2 holds hi in its first
                // 16 columns and lo in the next 16 (16 keys = 8 columns)
                auto col = [&](int ks) { return static_cast<uint32_t>((ks >> 1) * 32 + (ks & 1) * 8); };
                // V rows of these 16 keys: 16 rows of 128 B (MN-major), or
                // 32 B into a 64-key half of the [d][keys] tile (K-major)
                auto vst = [&](int ks) {
                    return static_cast<uint32_t>(F8 ? (ks >> 2) * ((D * 128) >> 4) + (ks & 3) * 2
                                                    : ks * (2048 >> 4));
                };
                if constexpr (kOneP) {
#pragma unroll
                    for (int ks = 0; ks < kTcKeys / 16; ks += 4)
                        umma4_ts(d_o, a_p + col(ks), dvs + vst(ks), a_p + col(ks + 1), dvs + vst(ks + 1),
                                 a_p + col(ks + 2), dvs + vst(ks + 2), a_p + col(ks + 3), dvs + vst(ks + 3),
                                 kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
                } else {   // bf16 operands: P's hi part, then its lo part, per 16 keys
#pragma unroll
                    for (int ks = 0; ks < kTcKeys / 16; ks += 2)
                        umma4_ts(d_o, a_p + col(ks), dvs + vst(ks), a_p + col(ks) + 16, dvs + vst(ks),
                                 a_p + col(ks + 1), dvs + vst(ks + 1), a_p + col(ks + 1) + 16,
                                 dvs + vst(ks + 1), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
                }
                if (j + 1 == n_t[t]) umma_commit_elect(smem_u32(&pv_done[t]));   // O_t complete
            };
            // every lane polls; the warp goes on only if all saw the phase
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, err));
            };
            bool ok = wait_all(&q_ready, 0) && wait_all(&k_full[0], 0);
            tc_fence_after();
            if (ok) {
                for (int t = 0; t < kTcTiles; ++t)
                    if (n_t[t] > 0) issue_qk(t, 0);
                umma_commit_elect(smem_u32(&k_empty[0]));
            }
            ok = ok && (n_tiles == 0 || wait_all(&v_full[0], 0));
            // Per key tile j: each tile's P_t(j) V, then its S_t(j + 1).  The
            // waits for the next key tile's K and V sit after a P V, while its
            // MMAs are still queued, so the tensor pipe does not run dry while
            // this warp waits; only the P waits lie on the pipeline's path.
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int st = j % kTcStages, st1 = (j + 1) % kTcStages;
                const bool more = j + 1 < n_tiles;
                const int last_t = j < n_t[1] ? 1 : 0;   // the last tile with key tile j
                bool k_next = false;                      // K(j + 1) has landed
#pragma unroll
                for (int t = 0; t < kTcTiles; ++t) {
                    if (j >= n_t[t]) continue;
                    if (!wait_all(&p_full[t], j & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(t, j);
                    if (t == last_t) umma_commit_elect(smem_u32(&v_empty[st]));   // V(j) read
                    const bool qk = j + 1 < n_t[t];
                    if (qk || (t == last_t && more)) {
                        if (!k_next && !wait_all(&k_full[st1], ((j + 1) / kTcStages) & 1)) {
                            ok = false;
                            break;
                        }
                        k_next = true;
                        if (t == last_t && !wait_all(&v_full[st1], ((j + 1) / kTcStages) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (qk) issue_qk(t, j + 1);
                }
                if (!ok) break;
                if (more) umma_commit_elect(smem_u32(&k_empty[st1]));   // K(j + 1) read
            }
        }
    } else {
        // ------------------------------------------------ softmax warps 0-15
        // Warp w serves tile t = (w / 4) % 2, half hf = w / 8 of every key
        // tile's keys and of O's columns, and reads TMEM lanes 32*(w % 4) ..
        // +31.  The two warps of a row pair meet once per key tile at a named
        // barrier; no warp leaves the loop except right after that meeting,
        // when both see the same stop flag, so neither can wait there alone.
        const int t = (warp >> 2) & 1, quarter = warp & 3, hf = warp >> 3;
        const int rr = quarter * 32 + lane;                 // M row in the tile = TMEM lane
        const int grow = row0 + t * kTcRows + rr;
        const bool valid = grow < rows_total;
        const int pos_local = valid ? grow / group : 0;
        const int head = kvh * group + (valid ? grow - (grow / group) * group : 0);
        const int p_abs = valid ? ctx0 + pos_local : L - 1;   // padding rows see every key
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t s_col = Ly::kTmemS + t * 128 + hf * 64;      // this thread's 64 keys
        const uint32_t o_col = Ly::kTmemO + t * D + hf * (D / 2);   // this thread's O columns
        const int bar_id = 1 + t * 4 + quarter;                      // the pair's named barrier
        const int nt = n_t[t];

        // Q row (this thread's half of it) -> shared memory, 128-byte swizzled
        // rows.  A negative scale is applied as -Q and |scale| (an exact sign
        // flip), so the raw-score max is the scaled max.
        const uint32_t qsign = scale_log2 < 0.f ? 0x80008000u : 0u;
        scale_log2 = fabsf(scale_log2);
        {
            const uint4* qp = reinterpret_cast<const uint4*>(
                q + (static_cast<int64_t>(qs + pos_local) * n_q + head) * D);
            const uint32_t qbase = sbase + Ly::kOffQ + t * Ly::kQBytes;
            if constexpr (kDirectK) {
                // bf16 q -> two E4M3 parts: the row is scaled by 2^-e so that its
                // largest magnitude lands in [128, 256), hi = e4m3(x) and lo =
                // e4m3(x - hi) (exact for every element down to 2^-10 of the
                // row's largest); 2^e goes into the row's softmax scale.  The
                // pair meets to take the row's largest magnitude.
                uint4 v[D / 16];
                float amax = 0.f;
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    v[cc] = valid ? __ldg(qp + hf * (D / 16) + cc) : make_uint4(0, 0, 0, 0);
                    const uint32_t w4[4] = {v[cc].x, v[cc].y, v[cc].z, v[cc].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = Cvt<__nv_bfloat16>::unpack(w4[i]);
                        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
                    }
                }
                xmax[1][t][hf][rr] = amax;   // (tile 1's slot: rewritten only after tile 0's meeting)
                named_bar_sync(bar_id, 64);
                const float rmax = fmaxf(amax, xmax[1][t][hf ^ 1][rr]);
                int e = 0;
                if (rmax > 0.f) {
                    frexpf(rmax, &e);
                    e = max(e - 8, -100);    // rmax * 2^-e in [128, 256) unless tiny
                }
                scale_log2 = ldexpf(scale_log2, e);
                const float down = ldexpf(qsign ? -1.f : 1.f, -e);   // +-2^-e: the sign flip too
                // 64 elements of the row: 4 chunks of 16 codes for each part
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {        // output word i: elements 4i .. 4i+3
                        const uint4 src = v[2 * c4 + (i >> 1)];
                        const uint32_t wa = (i & 1) ? src.z : src.x;
                        const uint32_t wb = (i & 1) ? src.w : src.y;
                        const float2 a = Cvt<__nv_bfloat16>::unpack(wa), b = Cvt<__nv_bfloat16>::unpack(wb);
                        const float x0 = a.x * down, x1 = a.y * down, x2 = b.x * down, x3 = b.y * down;
                        const uint32_t h01 = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
                        const uint32_t h23 = __nv_cvt_float2_to_fp8x2(make_float2(x2, x3), __NV_SATFINITE, __NV_E4M3);
                        uint32_t d01, d23;
                        widen4((h01 & 0xFFFFu) | (h23 << 16), d01, d23);   // hi values as fp16 pairs
                        const float2 e01 = __half22float2(*reinterpret_cast<const __half2*>(&d01));
                        const float2 e23 = __half22float2(*reinterpret_cast<const __half2*>(&d23));
                        const uint32_t l01 = __nv_cvt_float2_to_fp8x2(make_float2(x0 - e01.x, x1 - e01.y), __NV_SATFINITE, __NV_E4M3);
                        const uint32_t l23 = __nv_cvt_float2_to_fp8x2(make_float2(x2 - e23.x, x3 - e23.y), __NV_SATFINITE, __NV_E4M3);
                        hw[i] = (h01 & 0xFFFFu) | (h23 << 16);
                        lw[i] = (l01 & 0xFFFFu) | (l23 << 16);
                    }
                    const int c = hf * (D / 32) + c4;    // 16-byte chunk of the 128-byte row
                    const uint32_t addr = qbase + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
                    st_shared_v4(addr, hw[0], hw[1], hw[2], hw[3]);
                    st_shared_v4(addr + Ly::kQLo, lw[0], lw[1], lw[2], lw[3]);
                }
            } else if constexpr (std::is_same<T, QT>::value) {
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    const int c = hf * (D / 16) + cc;
                    uint4 v = valid ? __ldg(qp + c) : make_uint4(0, 0, 0, 0);
                    v.x ^= qsign; v.y ^= qsign; v.z ^= qsign; v.w ^= qsign;
                    const uint32_t addr = qbase + (c >> 3) * (kTcRows * 128) + rr * 128 +
                                          (((c & 7) ^ (rr & 7)) << 4);
                    st_shared_v4(addr, v.x, v.y, v.z, v.w);
                }
            } else {
                // bf16 q -> fp16: the row's largest magnitude (bf16 bits compare
                // as integers), met with the partner thread's half
                uint4 v[D / 16];
                uint32_t amax = 0;
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    v[cc] = valid ? __ldg(qp + hf * (D / 16) + cc) : make_uint4(0, 0, 0, 0);
                    const uint32_t w4[4] = {v[cc].x, v[cc].y, v[cc].z, v[cc].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        amax = max(amax, max(w4[i] & 0x7FFFu, (w4[i] >> 16) & 0x7FFFu));
                }
                // (the slot of key tile 1's maxima: the pair meets at tile 0 before
                // either writes it again)
                xmax[1][t][hf][rr] = __uint_as_float(amax << 16);
                named_bar_sync(bar_id, 64);
                const float rmax = fmaxf(__uint_as_float(amax << 16), xmax[1][t][hf ^ 1][rr]);
                int e = 0;
                if (rmax > 0.f) {
                    frexpf(rmax, &e);
                    e = max(e - 15, -100);   // rmax * 2^-e in [2^14, 2^15) unless tiny
                }
                scale_log2 = ldexpf(scale_log2, e);
                const float down = ldexpf(1.f, -e);   // 2^-e, a normal float
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    const int c = hf * (D / 16) + cc;
                    const uint32_t w4[4] = {v[cc].x, v[cc].y, v[cc].z, v[cc].w};
                    uint32_t h4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float lo = __uint_as_float(w4[i] << 16) * down;
                        const float hi = __uint_as_float(w4[i] & 0xFFFF0000u) * down;
                        h4[i] = Cvt<__half>::pack(lo, hi) ^ qsign;
                    }
                    const uint32_t addr = qbase + (c >> 3) * (kTcRows * 128) + rr * 128 +
                                          (((c & 7) ^ (rr & 7)) << 4);
                    st_shared_v4(addr, h4[0], h4[1], h4[2], h4[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&q_ready));
        }

        // smallest query position of this warp's rows (rows are position-major)
        const int wrow = row0 + t * kTcRows + quarter * 32;
        const int warp_min_pos = wrow < rows_total ? ctx0 + wrow / group : L - 1;
        float m_raw = -INFINITY, l = 0.f;
        bool stop = false;   // a wait of this warp ran out
        bool quit = false;   // the pair left the loop together
        for (int j = 0; j < nt; ++j) {
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[t]), j & 1, err));
            if (ok) tc_fence_after();
            // S_t(j) done implies P_t(j - 1) V done (issued earlier, committed
            // in order): O may be rescaled now, and P may overwrite S.
            const int key0 = j * kTcKeys, hkey0 = key0 + hf * 64;
            const bool full_tile = key0 + kTcKeys - 1 <= warp_min_pos;

            // pass 1: max over this thread's 64 raw scores, swapped with the
            // partner's (scores stay unscaled until the exponent: p =
            // 2^(s*c - m*c) is one FFMA and one EX2)
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (ok) {
                uint32_t sa[32], sb[32];       // both loads in flight, one wait
                tmem_ld32(lane_addr + s_col, sa);
                tmem_ld32(lane_addr + s_col + 32, sb);
                tmem_ld_wait();
                if (full_tile) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        m4[i & 3] = max3f(m4[i & 3], __uint_as_float(sa[i]), __uint_as_float(sb[i]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (hkey0 + i <= p_abs) m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(sa[i]));
                        if (hkey0 + 32 + i <= p_abs) m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(sb[i]));
                    }
                }
            }
            float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            xmax[j & 1][t][hf][rr] = mx;
            xstop[j & 1][t][hf][rr] = (!ok || stop) ? 1 : 0;
            named_bar_sync(bar_id, 64);
            mx = fmaxf(mx, xmax[j & 1][t][hf ^ 1][rr]);
            stop = stop || !ok || xstop[j & 1][t][hf ^ 1][rr] != 0;
            if (__any_sync(0xffffffffu, stop)) {   // the partner warp sees the same flags
                quit = true;
                break;
            }

            // lazy: move the reference max only when the first tile sets it or
            // the max grew by more than 2^8 (written so that scale 0 stays finite)
            const bool first = m_raw == -INFINITY;
            const bool resc = first ? (mx > -INFINITY) : ((mx - m_raw) * scale_log2 > 8.f);
            float fac = 1.f;
            if (resc) {
                fac = first ? 0.f : fast_exp2((m_raw - mx) * scale_log2);
                m_raw = mx;
                l *= fac;
            }
            const float neg_mc = -m_raw * scale_log2;
            if (j >= 1 && __any_sync(0xffffffffu, resc)) {   // TMEM access is warp-wide
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + o_col + c0, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac);
                    tmem_st32(lane_addr + o_col + c0, o);
                }
            }

            // pass 2, per 32 keys: exponent, row sum, P (hi/lo split for bf16),
            // written over those 32 keys' own score columns (hi in the first
            // 16, lo in the next 16), so no score is overwritten before it is read
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // full tiles
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t sr[32];
                tmem_ld32(lane_addr + s_col + h2 * 32, sr);
                tmem_ld_wait();
                uint32_t ph[16], pl[16];
                if (full_tile) {
                    // pairs of keys in paired fp32 instructions: the exponent's
                    // argument, the row sum and P's lo residual
                    const float2 c2 = make_float2(scale_log2, scale_log2), n2 = make_float2(neg_mc, neg_mc);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 x = fma2(make_float2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                                              c2, n2);
                        const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        s2[i & 1] = add2(s2[i & 1], pp);
                        if constexpr (kOneP) {
                            ph[i] = Cvt<__half>::pack(pp.x, pp.y);
                        } else {
                            // hi: the upper 16 bits of each (truncation); lo: the exact
                            // remainder, rounded to bf16
                            const uint32_t u0 = __float_as_uint(pp.x), u1 = __float_as_uint(pp.y);
                            ph[i] = __byte_perm(u0, u1, 0x7632);
                            const float2 r = sub2(pp, make_float2(__uint_as_float(u0 & 0xFFFF0000u),
                                                                  __uint_as_float(u1 & 0xFFFF0000u)));
                            pl[i] = Cvt<T>::pack(r.x, r.y);
                        }
                    }
                } else {   // masked keys give exactly 0 (even with scale 0, where -inf * 0 is NaN)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int k = hkey0 + h2 * 32 + 2 * i;
                        const float p0 = k <= p_abs ? fast_exp2(fmaf(__uint_as_float(sr[2 * i]), scale_log2, neg_mc)) : 0.f;
                        const float p1 = k + 1 <= p_abs ? fast_exp2(fmaf(__uint_as_float(sr[2 * i + 1]), scale_log2, neg_mc)) : 0.f;
                        s4[i & 3] += p0 + p1;
                        if constexpr (kOneP) ph[i] = Cvt<__half>::pack(p0, p1);
                        else split_trunc<T>(p0, p1, ph[i], pl[i]);
                    }
                }
                tmem_st16(lane_addr + s_col + h2 * 32, ph);            // over the scores
                if constexpr (!kOneP) tmem_st16(lane_addr + s_col + h2 * 32 + 16, pl);   // just read

            }
            l += ((s4[0] + s4[1]) + (s4[2] + s4[3])) + ((s2[0].x + s2[0].y) + (s2[1].x + s2[1].y));
            tmem_st_wait();

            if (!F8 && key0 + kTcKeys > L) {   // FP8: the producers wrote zeros there
                // keys at or past L (only in the request's last key tile) may hold
                // anything, even NaN: zero those V rows so P = 0 keeps them out,
                // after the tile's V has landed.  Both tiles' rows may do this for
                // the same key tile; they write the same zeros.  A wait that runs
                // out skips the work; the pair stops at its next meeting.
                if (__all_sync(0xffffffffu, mbar_wait(smem_u32(&v_full[j % kTcStages]), (j / kTcStages) & 1, err))) {
                    const int valid_rows = max(0, L - key0);
                    const int per_half = (kTcKeys - valid_rows) * 8;      // 16-byte pieces
                    const uint32_t vb = sbase + Ly::kOffV + (j % kTcStages) * Ly::kKBytes;
                    for (int i = (hf * 4 + quarter) * 32 + lane; i < per_half * Ly::kHalves; i += 8 * 32) {
                        const int hx = i / per_half;
                        const int rem = i - hx * per_half;
                        st_shared_v4(vb + hx * (kTcKeys * 128) + valid_rows * 128 + rem * 16, 0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                } else {
                    stop = true;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_full[t]));
        }

        // ------------------------------------------------ epilogue: O / l
        // the pair meets once more, to add its partial sums, unless it left
        // the loop together; a late failure of either warp skips the output
        if (!quit && nt > 0) {
            xsum[t][hf][rr] = l;
            xstop_end[t][hf][rr] = stop ? 1 : 0;
            named_bar_sync(bar_id, 64);
            const float lsum = l + xsum[t][hf ^ 1][rr];
            stop = stop || xstop_end[t][hf ^ 1][rr] != 0;
            const bool ok = !__any_sync(0xffffffffu, stop) &&
                            mbar_wait(smem_u32(&pv_done[t]), 0, err);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float inv = (F8 ? v_scale : 1.f) / lsum;
                const int64_t obase = (static_cast<int64_t>(qs + pos_local) * n_q + head) * D;
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + o_col + c0, o);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * inv;
                    if (valid) store_row<T>(out, obase, hf * (D / 2) + c0, v, 32, out_dtype);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, typename QT, int D, int BS, bool F8>
static cudaError_t run_prefill_tc(const PrefillArgs& a, cudaStream_t s, float sl2)
{
    constexpr bool kBq = std::is_same<QT, __nv_bfloat16>::value;
    using Ly = PfLayout<T, D, F8, kBq>;
    auto kern = prefill_tc_kernel<T, QT, D, BS, F8>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(Ly::kDynBytes));
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap kmap{}, vmap{};
    const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * a.cache.n_kv_heads * BS;
    if constexpr (!F8) {
        if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, 64, 16) != PA_OK ||
            encode_pool_map(&vmap, a.v_cache, a.cache.dtype, D, rows, 64, 16) != PA_OK)
            return cudaErrorInvalidValue;
    } else if constexpr (Ly::kDirectK) {
        // K codes read by the score MMA: boxes of 16 rows x 128 codes, 128-byte
        // swizzle (the other FP8 copies are plain bulk copies; vmap stays unused)
        if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, D, 16, 128) != PA_OK)
            return cudaErrorInvalidValue;
    }
    const int group = a.n_q / a.cache.n_kv_heads;
    const int64_t tiles = (static_cast<int64_t>(a.max_q) * group + kTcTiles * kTcRows - 1) /
                          (kTcTiles * kTcRows);
    dim3 grid(static_cast<unsigned>(tiles), a.cache.n_kv_heads, a.num_reqs);
    kern<<<grid, PfWarps<F8, D, kBq>::kThreads, Ly::kDynBytes, s>>>(
        kmap, vmap, static_cast<const uint8_t*>(a.k_cache), static_cast<const uint8_t*>(a.v_cache),
        a.out, a.out_dtype, static_cast<const QT*>(a.q), a.block_tables, a.max_blocks,
        a.q_start, a.context_lens, a.max_q, a.n_q, a.cache.n_kv_heads, group, a.cache.num_blocks,
        F8 ? sl2 * a.cache.k_scale : sl2, F8 ? a.cache.v_scale : 1.f, a.err);
    return cudaGetLastError();
}

template <typename T, typename QT, bool F8>
static cudaError_t run_prefill_tc_dt(const PrefillArgs& a, cudaStream_t s, float sl2)
{
    const int D = a.cache.head_dim, BS = a.cache.block_size;
    if (D == 64 && BS == 16) return run_prefill_tc<T, QT, 64, 16, F8>(a, s, sl2);
    if (D == 64 && BS == 32) return run_prefill_tc<T, QT, 64, 32, F8>(a, s, sl2);
    if (D == 128 && BS == 16) return run_prefill_tc<T, QT, 128, 16, F8>(a, s, sl2);
    if (D == 128 && BS == 32) return run_prefill_tc<T, QT, 128, 32, F8>(a, s, sl2);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s)
{
    const float sl2 = a.scale * 1.4426950408889634f;
    if (a.cache.dtype == PA_BF16) return run_prefill_tc_dt<__nv_bfloat16, __nv_bfloat16, false>(a, s, sl2);
    if (a.cache.dtype == PA_F16) return run_prefill_tc_dt<__half, __half, false>(a, s, sl2);
    if (a.cache.dtype == PA_FP8_E4M3)   // fp16 operands; q in the activation type
        return a.cache.act_dtype == PA_BF16 ? run_prefill_tc_dt<__half, __nv_bfloat16, true>(a, s, sl2)
                                            : run_prefill_tc_dt<__half, __half, true>(a, s, sl2);
    return cudaErrorInvalidValue;
}

}  // namespace pa
