#pragma once
// Tensor-core paged decode kernel, shared by the decode and the multi-query
// (draft verification) entry points.
//
// Paged decode attention: one query row per (sequence, query head) against
// the sequence's K/V read through its block table ("How the attention kernel
// actually reads paged blocks": look the block up once, q.k against its keys,
// softmax-weighted sum of its values).
//
// Work unit = (sequence s, KV head [8-row sub-group], partition j of
// part_tokens tokens).  Long contexts are split into partitions whose (max,
// sum, unnormalised output) are combined by decode_reduce_kernel; a sequence
// that fits in one partition is finished by the partition kernel itself.
//
// Tensor-core path (bf16/fp16, head_dim 64/128, block 16/32), persistent:
//   - a grid of (SMs x resident CTAs) walks a compact list of the live units:
//     each CTA builds the prefix sum of partitions per sequence in shared
//     memory and maps unit numbers to (sequence, partition, head group) by
//     binary search, so skewed lengths cost no empty CTAs;
//   - the g query heads sharing one KV head form the M rows of an m16n8k16
//     MMA, so each K/V slab is read from HBM once for the whole group;
//   - each warp owns a ring of NS stages of 16 K/V rows; lane 0 streams them
//     with 2-D TMA tile loads (128-byte swizzle, so ldmatrix reads are bank
//     conflict free); a 32-token block is two stages, so the ring and the
//     occupancy do not depend on the block size;
//   - online softmax in registers with quad shuffles;
//   - P is split into hi + lo halves of the input type and placed in rows
//     0-7 and 8-15 of the A operand, so P.V costs one MMA yet keeps ~16 bits
//     of P (rows 8-15 would otherwise be padding).  Groups of more than 8 heads
//     are handled as several 8-head sub-groups.
// Multi-query instantiations (MQ) take q_per_seq query rows per sequence: the
// rows of a KV head are (head, query) pairs, head-major, 8 per sub-group (16
// per unit when a KV head has more than 8), and query i of q_per_seq sees the
// keys up to L - q_per_seq + i.
// FP8 pools: a stage's K codes arrive by TMA and its V piece (stored
// transposed, 16 tokens x head_dim) by one 1-D bulk copy; fragments are
// widened to fp16 in registers.  With at most 4 query heads a KV head the
// FP8 decode runs transposed (4-row units, RU 4): the stage's 16 tokens are
// the MMA rows, see kTr below.
#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"

#include <math.h>

#include <mutex>
#include <type_traits>

namespace pa {

constexpr int kDecWarps = 4;
constexpr int kRows = 16;            // K/V rows per pipeline stage
constexpr int kMaxPartBlocks = 128;   // blocks per partition (part_tokens / block_size)
constexpr int kPrefixCap = 1024;      // sequences whose partition prefix sum fits in smem

__device__ __forceinline__ void store_any(void* out, int64_t idx, float v, pa_dtype dt)
{
    if (dt == PA_F32)
        static_cast<float*>(out)[idx] = v;
    else if (dt == PA_BF16)
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// Resident CTAs per SM: FP8 stages cost the same fragment work for half the
// bytes, so that path is bound by per-warp latency and runs more warps; so do
// 16-bit pools with head_dim 64 (half the bytes per row, and the register
// count of those variants fits 3 CTAs of 4 warps).
constexpr int decode_ctas_per_sm(bool fp8, int D = 128, int RU = 8)
{
    return RU == 4 ? 4 : (fp8 || (D == 64 && RU == 8) ? 3 : 2);
}
constexpr int kSmemPerSm = 233472;    // 228 KB of shared memory per SM
// bound on the kernel's static shared memory (ptxas: 5,712-5,936 B, of which the
// prefix table is 4 KB)
constexpr int kStaticSmem = 6144;
constexpr int kPreferSepRed = 1;      // give the combine its own buffer when it fits
constexpr int kStaticUnitsPerCta = 4; // batches up to this many units per CTA: round robin

// Dynamic shared memory a CTA may use at the resident count above.
constexpr int decode_dyn_avail(bool fp8, int D = 128, int RU = 8)
{
    return kSmemPerSm / decode_ctas_per_sm(fp8, D, RU) - 1024 /* reserved */ - kStaticSmem -
           1024 /* align */;
}

// Ring depth per warp: about `budget` bytes of K+V in flight per warp, at least
// 2 stages, and no more than the dynamic shared memory holds.  Depth comes
// before a separate combine buffer: when the two do not fit together, the
// combine aliases the (then idle) rings.
template <typename T, int D, bool FP8, int RU = 8>
constexpr int decode_stages()
{
    constexpr int stage = 2 * kRows * D * (FP8 ? 1 : static_cast<int>(sizeof(T)));
    constexpr int budget = FP8 ? 12288 : 24576;
    constexpr int ns = budget / stage > 2 ? budget / stage : 2;
    constexpr int cap = (decode_dyn_avail(FP8, D, RU) - 1024) / (kDecWarps * stage);
    static_assert(cap >= 2, "a ring of two stages per warp must fit");
    return ns < cap ? ns : cap;
}

// FP8 pools: a stage holds 16 rows of E4M3 K codes (swizzled rows of D bytes)
// and the matching D x 16 piece of the transposed V codes (as in the pool).
// RU: rows of the MMA tile a work unit fills (8 = one sub-group of up to 8
// heads with P's hi/lo halves in rows 0-7 / 8-15; 16 = sixteen (head, query)
// rows, P's halves in two MMAs; 4 = FP8 decode of up to 4 heads a KV head,
// computed transposed: the 16 tokens of a stage are the MMA rows, see below).
template <typename T, int D, int NS, bool FP8 = false, int RU = 8>
struct DecodeCfg {
    static constexpr int kElem = FP8 ? 1 : static_cast<int>(sizeof(T));
    static constexpr int kSlabBytes = kRows * D * kElem;    // 16 rows of K or V as stored
    static constexpr int kStageBytes = 2 * kSlabBytes;
    static constexpr int kWarpBytes = NS * kStageBytes;
    static constexpr int kRingBytes = kDecWarps * kWarpBytes;
    static constexpr int kReduceBytes = kDecWarps * RU * (D + 2) * 4;
    // the combine buffer sits after the rings when both fit, else it aliases them
    static constexpr bool kSepRed =
        kPreferSepRed && kRingBytes + kReduceBytes <= decode_dyn_avail(FP8, D, RU);
    static constexpr int kRedOffset = kSepRed ? kRingBytes : 0;
    static constexpr int kDynBytes =
        (kSepRed ? kRingBytes + kReduceBytes
                 : (kRingBytes > kReduceBytes ? kRingBytes : kReduceBytes)) + 1024;
    static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
    static_assert(kMaxPartBlocks <= kDecWarps * 32, "one block id per thread");
};

// Four E4M3 codes (one fragment word) widened exactly (every E4M3 value is an
// fp16 value) to two f16x2 words: lo = codes 0,1 and hi = codes 2,3.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi) : "r"(w));
}

template <typename QT, typename T>
__device__ __forceinline__ uint32_t q_pair(const QT* p)
{
    return __ldg(reinterpret_cast<const unsigned int*>(p));   // q already in the MMA type
}

template <typename T, typename QT, int D, int BS, int NS, bool FP8, bool MQ, int RU = 8>
__global__ void __launch_bounds__(kDecWarps * 32, decode_ctas_per_sm(FP8, D, RU))
decode_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const uint8_t* __restrict__ v_codes, void* __restrict__ out, pa_dtype out_dtype,
                  const QT* __restrict__ q,
                  const int32_t* __restrict__ block_tables, int max_blocks,
                  const int32_t* __restrict__ context_lens, int num_seqs, int n_q, int nq_arg,
                  int n_kv, int group, int num_blocks, float scale_log2, float v_scale,
                  float* __restrict__ ws_ml, float* __restrict__ ws_acc, int part_tokens,
                  int max_parts, unsigned* __restrict__ ticket, unsigned* err)
{
    using Cfg = DecodeCfg<T, D, NS, FP8, RU>;
    static_assert(!FP8 || std::is_same<T, __half>::value, "FP8 pools compute in fp16");
    constexpr bool R16 = RU == 16;
    static_assert(RU == 8 || (RU == 16 && MQ && !FP8) || (RU == 4 && FP8 && !MQ),
                  "16-row units: multi-query, 16-bit pools; 4-row units: FP8 decode");
    // Transposed FP8 decode (RU 4): S^T = K q^T with the stage's 16 tokens as
    // the M rows and 8 columns: the unit's <= 4 heads, then the same heads
    // again (same q).  Columns 0-3 carry P's hi part and columns 4-7 its lo
    // part, so O^T = V^T P^T (D rows, the V piece as it is stored) keeps ~22
    // bits of P in one MMA per 16 rows of d.  Per stage: 8 + 8 MMAs instead of
    // 16 + 16, and half the O accumulators.
    constexpr bool kTr = RU == 4;
    constexpr int kHalves = D / 64;           // 64-column halves (one 128-byte swizzled row each)
    constexpr int kHalfTile = kRows * 128;
    constexpr int kCPB = BS / kRows;          // stages per block
    static_assert(BS % kRows == 0, "block_size must be a multiple of 16");

    __shared__ int s_prefix[kPrefixCap];
    __shared__ int s_scan[kDecWarps * 32];
    __shared__ int s_blk[2][kMaxPartBlocks];   // this unit's and the next unit's block ids
    __shared__ int s_total;
    __shared__ long long s_next;
    __shared__ long long s_rowoff[RU];   // MQ: output row of each row of the sub-group
    __shared__ __align__(8) uint64_t s_bar[kDecWarps * NS];
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                               ~static_cast<uintptr_t>(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // launched as a programmatic dependent: every input may come from the
    // kernel before this one in the stream
    grid_dependency_wait();
    // a KV head serves group x nq rows (head-major: row = head * nq + query),
    // taken RU at a time; plain decode (MQ false) has nq = 1 at compile time
    const int nq = MQ ? nq_arg : 1;
    const int n_sub = (group * nq + RU - 1) / RU;
    const int n_groups = n_kv * n_sub;
    const bool use_prefix = num_seqs <= kPrefixCap;

    // ---- units: first every full partition, then every sequence's last one.
    // The last partitions are the ragged, cheaper units, so handing them out
    // last evens out the tail of the static round-robin assignment.
    // s_prefix[s] = inclusive prefix sum of (partitions of s) - 1.
    if (use_prefix) {
        const int per = (num_seqs + kDecWarps * 32 - 1) / (kDecWarps * 32);
        const int b0 = tid * per, b1 = min(num_seqs, b0 + per);
        int local = 0;
        for (int i = b0; i < b1; ++i) {
            const int L = __ldg(context_lens + i);
            const int p = L > 0 ? min((L + part_tokens - 1) / part_tokens, max_parts) - 1 : 0;
            s_prefix[i] = p;
            local += p;
        }
        s_scan[tid] = local;
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int i = 0; i < kDecWarps * 32; ++i) {
                const int v = s_scan[i];
                s_scan[i] = acc;
                acc += v;
            }
            s_total = acc;                  // full partitions
        }
        __syncthreads();
        int run = s_scan[tid];
        for (int i = b0; i < b1; ++i) {
            run += s_prefix[i];
            s_prefix[i] = run;
        }
    } else if (tid == 0) {
        s_total = num_seqs * (max_parts - 1);
    }
    if (tid < kDecWarps * NS) mbar_init(smem_u32(&s_bar[tid]), 1);
    fence_mbar_init();
    __syncthreads();

    const int n_full = s_total;
    const int64_t units = (static_cast<int64_t>(n_full) + num_seqs) * n_groups;
    const uint32_t ring = smem_u32(smem) + warp * Cfg::kWarpBytes;
    const uint32_t bar0 = smem_u32(&s_bar[warp * NS]);
    const int g = lane >> 2, t4 = lane & 3;
    uint32_t kt = 0;   // stages this warp has consumed so far: its ring position and phase
    if (lane == 0) {
        prefetch_tensormap(&kmap);
        if constexpr (!FP8) prefetch_tensormap(&vmap);   // (FP8 V: bulk copies)
    }

    // Units are handed out dynamically: unit blockIdx.x first, then tickets
    // from a counter that starts at zero for every launch (or, for batches of
    // at most a few units per CTA, round robin with no counter).  Work for the next
    // unit overlaps the current one: its ticket is drawn one unit ahead, its
    // block ids are loaded (one per thread) while the current unit streams,
    // its q fragments while the current unit's warps combine, and - when the
    // combine buffer does not alias the rings - its first stages are issued
    // before that combine.
    struct Unit {
        int s, part, L, tok0, kvh, h0, r0, nh, nblk, nchunk, blk0, nparts;
        bool live;
    };
    auto describe = [&](int64_t uu) {
        Unit x{};
        x.live = false;
        if (uu >= units) return x;
        const int gp = static_cast<int>(uu / n_groups);
        const int grp = static_cast<int>(uu - static_cast<int64_t>(gp) * n_groups);
        if (gp >= n_full) {                           // a sequence's last partition
            x.s = gp - n_full;
            const int Ls = __ldg(context_lens + x.s);
            x.part = Ls > 0 ? min((Ls + part_tokens - 1) / part_tokens, max_parts) - 1 : 0;
        } else if (use_prefix) {
            int lo = 0, hi = num_seqs - 1;            // first s with prefix[s] > gp
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (s_prefix[mid] > gp) hi = mid; else lo = mid + 1;
            }
            x.s = lo;
            x.part = gp - (lo ? s_prefix[lo - 1] : 0);
        } else {
            x.s = gp / (max_parts - 1);
            x.part = gp - x.s * (max_parts - 1);
        }
        x.L = __ldg(context_lens + x.s);
        x.tok0 = x.part * part_tokens;
        x.live = x.tok0 < x.L && x.L >= nq;           // same decision in every thread
        if (x.L > 0 && x.L < nq) set_error(err, PA_ERR_OUT_OF_RANGE);   // fewer keys than queries
        x.kvh = grp / n_sub;
        const int sub = grp - x.kvh * n_sub;
        x.h0 = x.kvh * group;                         // first query head of the KV head
        x.r0 = sub * RU;                              // first row of the sub-group
        x.nh = min(RU, group * nq - x.r0);            // rows in the sub-group
        const int tok1 = min(x.L, x.tok0 + part_tokens);
        x.nblk = (tok1 - x.tok0 + BS - 1) / BS;
        x.nchunk = (tok1 - x.tok0 + kRows - 1) / kRows;
        x.blk0 = x.tok0 / BS;
        x.nparts = min((x.L + part_tokens - 1) / part_tokens, max_parts);
        // without the prefix sums (very large batches) the full-partition
        // numbering covers every partition index below max_parts - 1: a
        // sequence's own last partition there belongs to the second numbering
        if (!use_prefix && gp < n_full && x.part >= x.nparts - 1) x.live = false;
        return x;
    };
    // block id i of unit x (-1 if the table has no such entry), checked
    // against the pool: a bad id flags the device error and drops the unit
    auto load_id = [&](const Unit& x, int i, int& bad) {
        const int lb = x.blk0 + i;
        int b = -1;
        if (lb < max_blocks) b = __ldg(block_tables + static_cast<int64_t>(x.s) * max_blocks + lb);
        if (b < 0 || b >= num_blocks) {
            bad = 1;
            set_error(err, PA_ERR_OUT_OF_RANGE);
        }
        return b;
    };
    // query fragments of unit x: rows 0-7 = rows g of the sub-group; rows 8-15
    // zero (RU 8) or rows g + 8 (RU 16, in qb)
    uint32_t qa[D / 16][2];
    uint32_t qb[R16 ? D / 16 : 1][2];
    float row_l2 = scale_log2;   // softmax scale (log2 domain) of row g's scores
    // the unit row this thread's q fragments hold: row g, or (kTr) column g,
    // whose head is g mod 4
    const int gq = kTr ? (g & 3) : g;
    auto load_q = [&](const Unit& x) {
        if constexpr (FP8 && std::is_same<QT, __nv_bfloat16>::value) {
            // bf16 q over an FP8 pool: the raw bf16 pairs of row g, made fp16
            // operands by scale_q once the unit starts (so their latency
            // overlaps the combine)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (gq < x.nh) {
                    const int hh = (x.r0 + gq) / nq, qi = x.r0 + gq - hh * nq;
                    const QT* row =
                        q + ((static_cast<int64_t>(x.s) * nq + qi) * n_q + x.h0 + hh) * D + kk * 16;
                    qa[kk][0] = __ldg(reinterpret_cast<const unsigned int*>(row + 4 * t4));
                    qa[kk][1] = __ldg(reinterpret_cast<const unsigned int*>(row + 4 * t4 + 2));
                } else {
                    qa[kk][0] = qa[kk][1] = 0u;
                }
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if constexpr (R16) {
                    if (g + 8 < x.nh) {
                        const int hh = (x.r0 + g + 8) / nq, qi = x.r0 + g + 8 - hh * nq;
                        const QT* row =
                            q + ((static_cast<int64_t>(x.s) * nq + qi) * n_q + x.h0 + hh) * D + kk * 16;
                        qb[kk][0] = q_pair<QT, T>(row + 2 * t4);
                        qb[kk][1] = q_pair<QT, T>(row + 2 * t4 + 8);
                    } else {
                        qb[kk][0] = 0u;
                        qb[kk][1] = 0u;
                    }
                }
                if (gq < x.nh) {
                    const int hh = (x.r0 + gq) / nq, qi = x.r0 + gq - hh * nq;
                    const QT* row =
                        q + ((static_cast<int64_t>(x.s) * nq + qi) * n_q + x.h0 + hh) * D + kk * 16;
                    if constexpr (FP8) {
                        // k order of the FP8 fragments: columns 4*t4 .. 4*t4+3 of the chunk
                        qa[kk][0] = q_pair<QT, T>(row + 4 * t4);
                        qa[kk][1] = q_pair<QT, T>(row + 4 * t4 + 2);
                    } else {
                        qa[kk][0] = q_pair<QT, T>(row + 2 * t4);
                        qa[kk][1] = q_pair<QT, T>(row + 2 * t4 + 8);
                    }
                } else {
                    qa[kk][0] = 0u;
                    qa[kk][1] = 0u;
                }
            }
        }
    };
    // bf16 q over an FP8 pool -> fp16 operands (whole warp).  The quad's
    // threads hold row g's columns 16*kk + 4*t4 .. +3; they meet on its largest
    // magnitude (bf16 bits order as integers), the row is scaled by 2^-e so
    // that this lands in [2^14, 2^15), exact for every element down to 2^-29 of
    // the largest, and 2^e goes into the row's softmax scale: no bf16 query
    // overflows fp16 or sinks into its subnormals.
    auto scale_q = [&]() {
        if constexpr (FP8 && std::is_same<QT, __nv_bfloat16>::value) {
            uint32_t amax = 0;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    amax = max(amax, max(qa[kk][h] & 0x7FFFu, (qa[kk][h] >> 16) & 0x7FFFu));
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            // e from the exponent field (bf16 subnormals take the floor, -100)
            const int e = amax == 0u ? 0 : max(static_cast<int>((amax >> 7) & 0xFFu) - 141, -100);
            row_l2 = scale_log2 * __int_as_float((127 + e) << 23);    // exact: powers of two
            const float down = __int_as_float((127 - e) << 23);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 f = Cvt<__nv_bfloat16>::unpack(qa[kk][h]);
                    qa[kk][h] = Cvt<__half>::pack(f.x * down, f.y * down);
                }
        }
    };
    // stage k of a unit (blk = its block ids, kvh_ its KV head) into this
    // warp's ring slot (base + k) % NS
    auto issue = [&](const int* blk, int kvh_, int k, uint32_t base) {
        const int c = warp + k * kDecWarps;
        const int b = blk[c / kCPB];
        const uint32_t st = (base + k) % NS;
        const uint32_t kdst = ring + st * Cfg::kStageBytes;
        const uint32_t vdst = kdst + Cfg::kSlabBytes;
        const uint32_t bar = bar0 + st * 8;
        const int row = (b * n_kv + kvh_) * BS + (c % kCPB) * kRows;
        mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
        if constexpr (FP8) {
            tma_load_2d(kdst, &kmap, 0, row, bar);                       // 16 rows x D codes
            // the piece's transposed V codes: D x 16, contiguous in the pool
            bulk_load(vdst, v_codes + ((static_cast<int64_t>(b) * n_kv + kvh_) * kCPB + c % kCPB) *
                                          Cfg::kSlabBytes,
                      Cfg::kSlabBytes, bar);
        } else {
#pragma unroll
            for (int hx = 0; hx < kHalves; ++hx) {
                tma_load_2d(kdst + hx * kHalfTile, &kmap, hx * 64, row, bar);
                tma_load_2d(vdst + hx * kHalfTile, &vmap, hx * 64, row, bar);
            }
        }
    };
    auto my_stages = [&](const Unit& x) {
        return x.nchunk > warp ? (x.nchunk - warp + kDecWarps - 1) / kDecWarps : 0;
    };

    float* red_o = reinterpret_cast<float*>(smem + Cfg::kRedOffset);   // [warps][RU][D]
    float* red_m = red_o + kDecWarps * RU * D;                          // [warps][RU]
    float* red_l = red_m + kDecWarps * RU;                              // [warps][RU]

    // FP8: tokens past the sequence may hold anything (even NaN): zero their
    // codes in every row of the stage's transposed V piece (whole warp)
    auto zero_v_tail = [&](uint32_t vbase, int valid) {
        uint8_t* vt = smem + (vbase - smem_u32(smem));
        for (int row = lane; row < D; row += 32) {
            uint4 w = *reinterpret_cast<uint4*>(vt + row * 16);
            uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int keep = min(4, max(0, valid - 4 * e));     // bytes kept
                ww[e] &= keep >= 4 ? 0xFFFFFFFFu : ((1u << (8 * keep)) - 1u);
            }
            *reinterpret_cast<uint4*>(vt + row * 16) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
    };

    // ---- the first unit: ids checked before any load is issued
    int64_t u = blockIdx.x;
    if (u >= units) return;                           // uniform over the CTA
    Unit cu = describe(u);
    {
        int bad = 0;
        if (cu.live && tid < cu.nblk) s_blk[0][tid] = load_id(cu, tid, bad);
        load_q(cu);
        const int any_bad = __syncthreads_or(bad);
        if (tid == 0)
            s_next = ticket ? static_cast<long long>(gridDim.x) + atomicAdd(ticket, 1u)
                            : u + static_cast<long long>(gridDim.x);
        cu.live = cu.live && !any_bad;
        __syncthreads();
    }
    int64_t un = s_next;
    int cb = 0;                                       // s_blk buffer of the current unit
    bool issued = false;                              // its first stages are in flight

    // O accumulators: [D / 8] n-tiles of O (rows = heads), or (kTr) [D / 16]
    // m-tiles of O^T (rows = d, columns = the 8 columns above)
    constexpr int kOT = kTr ? D / 16 : D / 8;
    float o[kOT][4];
    float m_run, l_run;     // row g (kTr: column 2*t4)
    float m_run1, l_run1;   // row g + 8 (RU 16; kTr: column 2*t4 + 1)
    // this warp's partial rows (running max, sum, unnormalised O) -> the
    // combine buffer [warp][row]
    auto write_partials = [&]() {
        if constexpr (kTr) {
            if (t4 < 2) {   // columns 2*t4 and 2*t4 + 1: heads, hi and lo parts merged
                float* dst = red_o + (warp * RU + 2 * t4) * D + g;
#pragma unroll
                for (int mt = 0; mt < kOT; ++mt) {
                    dst[16 * mt] = o[mt][0];
                    dst[16 * mt + 8] = o[mt][2];
                    dst[D + 16 * mt] = o[mt][1];
                    dst[D + 16 * mt + 8] = o[mt][3];
                }
                if (g == 0) {
                    red_m[warp * RU + 2 * t4] = m_run;
                    red_l[warp * RU + 2 * t4] = l_run;
                    red_m[warp * RU + 2 * t4 + 1] = m_run1;
                    red_l[warp * RU + 2 * t4 + 1] = l_run1;
                }
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                float* dst = red_o + (warp * RU + g) * D + nt * 8 + 2 * t4;
                if constexpr (R16) {
                    dst[0] = o[nt][0];
                    dst[1] = o[nt][1];
                    dst[8 * D] = o[nt][2];           // row g + 8
                    dst[8 * D + 1] = o[nt][3];
                } else {
                    dst[0] = o[nt][0] + o[nt][2];
                    dst[1] = o[nt][1] + o[nt][3];
                }
            }
            if (t4 == 0) {
                red_m[warp * RU + g] = m_run;
                red_l[warp * RU + g] = l_run;
                if constexpr (R16) {
                    red_m[warp * RU + g + 8] = m_run1;
                    red_l[warp * RU + g + 8] = l_run1;
                }
            }
        }
    };
    while (u < units) {
        const Unit nx = describe(un);
        // the next unit's block ids: in flight while this unit streams
        int nb_bad = 0, nb_id = -1;
        if (nx.live && tid < nx.nblk) nb_id = load_id(nx, tid, nb_bad);

        const int s = cu.s, part = cu.part, L = cu.L, tok0 = cu.tok0, kvh = cu.kvh;
        const int h0 = cu.h0, r0 = cu.r0, nh = cu.nh, nchunk = cu.nchunk, nparts = cu.nparts;
        // keys this thread's row may see: query qi of nq sits at L - nq + qi
        const int lim = g < nh ? L - nq + (r0 + g) % nq + 1 : L;
        const int lim1 = (R16 && g + 8 < nh) ? L - nq + (r0 + g + 8) % nq + 1 : L;
        int timed_out = 0;
        if (cu.live) {
            // ---- per-warp TMA ring over the partition's 16-row stages --------
            const int my_n = nchunk > warp ? (nchunk - warp + kDecWarps - 1) / kDecWarps : 0;
            if (!issued && lane == 0) {
                fence_proxy_async_smem();
                for (int k = 0; k < min(NS, my_n); ++k) issue(s_blk[cb], kvh, k, kt);
            }

            scale_q();
            // kTr: softmax scale of this thread's two columns (heads 2*t4 and
            // 2*t4 + 1, mod 4), held by the quads g = 2*t4 and 2*t4 + 1
            float cl2_0 = row_l2, cl2_1 = row_l2;
            if constexpr (kTr) {
                cl2_0 = __shfl_sync(0xffffffffu, row_l2, 8 * t4);
                cl2_1 = __shfl_sync(0xffffffffu, row_l2, 8 * t4 + 4);
            }
#pragma unroll
            for (int i = 0; i < kOT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            m_run = -INFINITY;
            m_run1 = -INFINITY;
            l_run1 = 0.f;
            l_run = 0.f;

            for (int k = 0; k < my_n; ++k) {
                const uint32_t st = (kt + k) % NS;
                const bool ok = mbar_wait(bar0 + st * 8, ((kt + k) / NS) & 1u, err);
                if (!__all_sync(0xffffffffu, ok)) {     // leave together: shuffles follow
                    timed_out = 1;
                    break;
                }
                const int pos0 = tok0 + (warp + k * kDecWarps) * kRows;
                const int valid = min(kRows, L - pos0);
                const uint32_t kbase = ring + st * Cfg::kStageBytes;
                const uint32_t vbase = kbase + Cfg::kSlabBytes;
                if constexpr (kTr) {
                    if (valid < kRows) zero_v_tail(vbase, valid);
                    // S^T = K q^T.  Row r of the tile is token 4*((r&7)>>1) + 2*(r>>3)
                    // + (r&1) of the stage: after the transpose below, P^T comes out
                    // in the token order of the V fragments.  Fragment words hold four
                    // consecutive codes (k order permuted as q was loaded).
                    float st[4] = {0.f, 0.f, 0.f, 0.f}, st2[4] = {0.f, 0.f, 0.f, 0.f};
                    {
                        const int mi = lane >> 3, i = lane & 7;
                        const int tok = 4 * (i >> 1) + 2 * (mi & 1) + (i & 1);
#pragma unroll
                        for (int c2 = 0; c2 < D / 32; ++c2) {   // chunks 2*c2 and 2*c2 + 1
                            const int cidx = 2 * c2 + (mi >> 1);
                            const int sw = D == 128 ? (cidx ^ (tok & 7)) : (cidx ^ ((tok >> 1) & 3));
                            uint32_t w[4], a[4];
                            ldsm_x4(kbase + tok * D + (sw << 4), w[0], w[1], w[2], w[3]);
                            e4m3x4_to_h2x2(w[0], a[0], a[2]);
                            e4m3x4_to_h2x2(w[1], a[1], a[3]);
                            MmaOp<T>::run(st, a, qa[2 * c2][0], qa[2 * c2][1]);
                            e4m3x4_to_h2x2(w[2], a[0], a[2]);
                            e4m3x4_to_h2x2(w[3], a[1], a[3]);
                            MmaOp<T>::run(st2, a, qa[2 * c2 + 1][0], qa[2 * c2 + 1][1]);
                        }
                    }
                    // online softmax down the columns (log2 domain): this thread has
                    // tokens tA and tA + 2 of columns 2*t4 and 2*t4 + 1; the column
                    // max meets over the eight lanes of each t4
                    const int tA = pos0 + 4 * (g >> 1) + (g & 1);
                    const float z0 = tA < L ? (st[0] + st2[0]) * cl2_0 : -INFINITY;
                    const float z1 = tA < L ? (st[1] + st2[1]) * cl2_1 : -INFINITY;
                    const float z2 = tA + 2 < L ? (st[2] + st2[2]) * cl2_0 : -INFINITY;
                    const float z3 = tA + 2 < L ? (st[3] + st2[3]) * cl2_1 : -INFINITY;
                    float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
                    for (int w = 4; w < 32; w <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, w));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, w));
                    }
                    // (every stage holds a visible token, so the maxima are finite)
                    const float mn0 = fmaxf(m_run, mx0), mn1 = fmaxf(m_run1, mx1);
                    if (__any_sync(0xffffffffu, mn0 != m_run || mn1 != m_run1)) {
                        const float a0 = fast_exp2(m_run - mn0), a1 = fast_exp2(m_run1 - mn1);
                        l_run *= a0;
                        l_run1 *= a1;
#pragma unroll
                        for (int mt = 0; mt < kOT; ++mt) {
                            o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
                        }
                    }
                    m_run = mn0;
                    m_run1 = mn1;
                    const float p0 = fast_exp2(z0 - mn0), p1 = fast_exp2(z1 - mn1);
                    const float p2 = fast_exp2(z2 - mn0), p3 = fast_exp2(z3 - mn1);
                    l_run += p0 + p2;
                    l_run1 += p1 + p3;
                    // P^T as the B operand: columns 0-3 take P's hi part, columns 4-7
                    // (the same heads) its lo part; each 8 x 8 block of the score
                    // layout is transposed in registers
                    uint32_t hu, lu, hv, lv;
                    split_pair<T>(p0, p1, hu, lu);   // rows g: tokens tA
                    split_pair<T>(p2, p3, hv, lv);   // rows g + 8: tokens tA + 2
                    const uint32_t pb0 = movmatrix_trans(t4 < 2 ? hu : lu);
                    const uint32_t pb1 = movmatrix_trans(t4 < 2 ? hv : lv);
                    // O^T += V^T P^T: m-tile mt is rows 16*mt .. +15 of the V piece
                    // (row d holds the stage's 16 tokens of element d)
#pragma unroll
                    for (int q2 = 0; q2 < D / 32; ++q2) {
                        const int d_row = 32 * q2 + 8 * (lane >> 3) + (lane & 7);
                        uint32_t w[4], a[4];
                        ldsm_x4(vbase + d_row * 16, w[0], w[1], w[2], w[3]);
                        e4m3x4_to_h2x2(w[0], a[0], a[2]);
                        e4m3x4_to_h2x2(w[1], a[1], a[3]);
                        MmaOp<T>::run(o[2 * q2], a, pb0, pb1);
                        e4m3x4_to_h2x2(w[2], a[0], a[2]);
                        e4m3x4_to_h2x2(w[3], a[1], a[3]);
                        MmaOp<T>::run(o[2 * q2 + 1], a, pb0, pb1);
                    }
                } else {
                    float sc[2][4];
                    float sc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};

                    if constexpr (FP8) {
                        if (valid < kRows) zero_v_tail(vbase, valid);
                        // S = Q K^T.  Column j of n-tile nt is token 4*(j/2) + 2*nt + j%2,
                        // which leaves P in the token order the V fragments use below.
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                            const int i = lane & 7;
                            const int r = 4 * (i >> 1) + 2 * nt + (i & 1);
#pragma unroll
                            for (int kq = 0; kq < D / 64; ++kq) {
                                const int cidx = kq * 4 + (lane >> 3);
                                const int sw = D == 128 ? (cidx ^ (r & 7)) : (cidx ^ ((r >> 1) & 3));
                                uint32_t w[4];
                                ldsm_x4(kbase + r * D + (sw << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj) {
                                    const int kk = kq * 4 + jj;
                                    const uint32_t a[4] = {qa[kk][0], 0u, qa[kk][1], 0u};
                                    uint32_t b0, b1;
                                    e4m3x4_to_h2x2(w[jj], b0, b1);
                                    // two accumulator chains (even / odd 16 columns) halve the
                                    // dependent MMA sequence per n-tile
                                    MmaOp<T>::run((jj & 1) ? sc2[nt] : sc[nt], a, b0, b1);
                                }
                            }
                            sc[nt][0] += sc2[nt][0]; sc[nt][1] += sc2[nt][1];
                            sc[nt][2] += sc2[nt][2]; sc[nt][3] += sc2[nt][3];
                        }
                    } else {
                        if (valid < kRows) {
                            // rows past the sequence may hold anything (even NaN): zero them in
                            // V so that 0 * row stays 0 inside the MMA
                            uint8_t* vgen = smem + (vbase - smem_u32(smem));
                            const int nbytes = (kRows - valid) * 128;
                            for (int hx = 0; hx < kHalves; ++hx)
                                for (int off = lane * 16; off < nbytes; off += 32 * 16)
                                    *reinterpret_cast<uint4*>(vgen + hx * kHalfTile + valid * 128 + off) =
                                        make_uint4(0, 0, 0, 0);
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        // S = Q K^T for the 16 rows
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                            for (int kc = 0; kc < D / 16; kc += 2) {
                                const int r = nt * 8 + (lane & 7);
                                const int chunk = kc * 2 + (lane >> 3);
                                const uint32_t addr = kbase + (chunk >> 3) * kHalfTile + r * 128 +
                                                      (((chunk & 7) ^ (r & 7)) << 4);
                                uint32_t b0, b1, b2, b3;
                                ldsm_x4(addr, b0, b1, b2, b3);
                                const uint32_t a0[4] = {qa[kc][0], R16 ? qb[R16 ? kc : 0][0] : 0u, qa[kc][1],
                                                        R16 ? qb[R16 ? kc : 0][1] : 0u};
                                const uint32_t a1[4] = {qa[kc + 1][0], R16 ? qb[R16 ? kc + 1 : 0][0] : 0u,
                                                        qa[kc + 1][1], R16 ? qb[R16 ? kc + 1 : 0][1] : 0u};
                                MmaOp<T>::run(sc[nt], a0, b0, b1);
                                MmaOp<T>::run(sc[nt], a1, b2, b3);
                            }
                        }
                    }

                    // online softmax on row g (log2 domain)
                    float mx = -INFINITY;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int p = pos0 + (FP8 ? 4 * t4 + 2 * nt + e : nt * 8 + 2 * t4 + e);
                            const float z = p < lim ? sc[nt][e] * row_l2 : -INFINITY;
                            sc[nt][e] = z;
                            mx = fmaxf(mx, z);
                        }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float m_new = fmaxf(m_run, mx);
                    // a row with no visible key so far (several queries per sequence)
                    // keeps m = -inf: exponents are then taken against 0, giving 0
                    const float m_use = (MQ && m_new == -INFINITY) ? 0.f : m_new;
                    float m_new1 = -INFINITY, m_use1 = 0.f;
                    if constexpr (R16) {   // the second row of this thread, same steps
                        float mx1 = -INFINITY;
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int e = 2; e < 4; ++e) {
                                const int p = pos0 + nt * 8 + 2 * t4 + e - 2;
                                const float z = p < lim1 ? sc[nt][e] * scale_log2 : -INFINITY;
                                sc[nt][e] = z;
                                mx1 = fmaxf(mx1, z);
                            }
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                        m_new1 = fmaxf(m_run1, mx1);
                        m_use1 = m_new1 == -INFINITY ? 0.f : m_new1;
                    }
                    // rescale only when some row's running max moved (warp-uniform
                    // branch; after the first stages the max rarely moves).  The first
                    // stage has m_run = -inf: alpha = 0 clears the (zero) state.
                    if (__any_sync(0xffffffffu, m_new != m_run || (R16 && m_new1 != m_run1))) {
                        const float alpha = fast_exp2(m_run - m_use);
                        const float alpha1 = R16 ? fast_exp2(m_run1 - m_use1) : alpha;
                        l_run *= alpha;
                        l_run1 *= alpha1;
#pragma unroll
                        for (int i = 0; i < D / 8; ++i) {
                            o[i][0] *= alpha; o[i][1] *= alpha; o[i][2] *= alpha1; o[i][3] *= alpha1;
                        }
                    }
                    m_run = m_new;
                    m_run1 = m_new1;
                    float psum = 0.f, psum1 = 0.f;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < (R16 ? 4 : 2); ++e) {
                            const float p = fast_exp2(sc[nt][e] - (e < 2 ? m_use : m_use1));
                            sc[nt][e] = p;
                            if (e < 2) psum += p; else psum1 += p;
                        }
                    l_run += psum;
                    l_run1 += psum1;

                    // O += P V, P as hi (rows 0-7) + lo (rows 8-15); RU 16: rows g and
                    // g + 8 both real, hi in pa and lo in pb, two MMAs
                    uint32_t pa[4], pb[4];
                    if constexpr (R16) {
                        split_pair<T>(sc[0][0], sc[0][1], pa[0], pb[0]);
                        split_pair<T>(sc[0][2], sc[0][3], pa[1], pb[1]);
                        split_pair<T>(sc[1][0], sc[1][1], pa[2], pb[2]);
                        split_pair<T>(sc[1][2], sc[1][3], pa[3], pb[3]);
                    } else {
                        split_pair<T>(sc[0][0], sc[0][1], pa[0], pa[1]);
                        split_pair<T>(sc[1][0], sc[1][1], pa[2], pa[3]);
                    }
                    if constexpr (FP8) {
                        // transposed V tile: row d holds tokens 0..15; a fragment word is
                        // tokens 4*t4 .. 4*t4+3 of row d, the k order P is in
#pragma unroll
                        for (int nd = 0; nd < D / 8; nd += 4) {
                            const int d_row = (nd + (lane >> 3)) * 8 + (lane & 7);
                            uint32_t w[4];
                            ldsm_x4(vbase + d_row * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                            {
                                uint32_t b0, b1;
                                e4m3x4_to_h2x2(w[jj], b0, b1);
                                MmaOp<T>::run(o[nd + jj], pa, b0, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int nt = 0; nt < D / 8; nt += 2) {
                            const int mi = lane >> 3;
                            const int r = (mi & 1) * 8 + (lane & 7);
                            const int chunk = nt + (mi >> 1);
                            const uint32_t addr = vbase + (chunk >> 3) * kHalfTile + r * 128 +
                                                  (((chunk & 7) ^ (r & 7)) << 4);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(addr, b0, b1, b2, b3);
                            MmaOp<T>::run(o[nt], pa, b0, b1);
                            MmaOp<T>::run(o[nt + 1], pa, b2, b3);
                            if constexpr (R16) {
                                MmaOp<T>::run(o[nt], pb, b0, b1);
                                MmaOp<T>::run(o[nt + 1], pb, b2, b3);
                            }
                        }
                    }

                }
                __syncwarp();
                if (lane == 0 && k + NS < my_n) {
                    fence_proxy_async_smem();
                    issue(s_blk[cb], kvh, k + NS, kt);
                }
            }
            kt += my_n;
            // ---- this warp's share of the combine
            if constexpr (kTr) {
                // column sums over the eight lanes of each t4; a head's hi and lo
                // columns (t4 and t4 + 2) add up
#pragma unroll
                for (int w = 4; w < 32; w <<= 1) {
                    l_run += __shfl_xor_sync(0xffffffffu, l_run, w);
                    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, w);
                }
#pragma unroll
                for (int mt = 0; mt < kOT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], 2);
            } else {
                l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
                l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
                if constexpr (R16) {
                    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, 1);
                    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, 2);
                }
            }
            if constexpr (Cfg::kSepRed) write_partials();
        }
        if (nx.live && tid < nx.nblk) s_blk[cb ^ 1][tid] = nb_id;
        if (MQ && cu.live && tid < nh) {
            const int gr = r0 + tid;
            s_rowoff[tid] = (static_cast<int64_t>(s) * nq + gr % nq) * n_q + h0 + gr / nq;
        }
        // every ring is idle and (separate buffer) the partials are written
        const int flags = __syncthreads_or(timed_out | (nb_bad << 1));
        if (flags & 1) return;
        if (tid == 0)
            s_next = ticket ? static_cast<long long>(gridDim.x) + atomicAdd(ticket, 1u)
                            : un + static_cast<long long>(gridDim.x);
        // this CTA's last unit: the kernel after this one may be scheduled now
        if (un >= units) allow_dependent_launch();
        const bool next_live = nx.live && !(flags & 2);
        if (cu.live) {
            if constexpr (!Cfg::kSepRed) {
                // the combine buffer aliases the rings: written after the barrier
                write_partials();
                fence_proxy_async_smem();   // these generic writes precede later TMA writes here
                __syncthreads();
            }
        }
        issued = false;
        if constexpr (Cfg::kSepRed) {
            if (next_live && lane == 0) {
                fence_proxy_async_smem();
                const int n1 = my_stages(nx);
                for (int k = 0; k < min(NS, n1); ++k) issue(s_blk[cb ^ 1], nx.kvh, k, kt);
            }
            issued = true;
        }
        if (next_live) load_q(nx);                    // its latency overlaps the combine
        if (cu.live) {
            for (int idx = tid; idx < nh * D; idx += kDecWarps * 32) {
                const int hh = idx / D, dd = idx - hh * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red_m[w * RU + hh]);
                // M = -inf: no key of this partition is visible to the row (a
                // later query's keys only); it contributes l = 0, acc = 0
                const float M_use = (MQ && M == -INFINITY) ? 0.f : M;
                float lsum = 0.f, acc = 0.f;
#pragma unroll
                for (int w = 0; w < kDecWarps; ++w) {
                    const float f = exp2f(red_m[w * RU + hh] - M_use);
                    lsum += f * red_l[w * RU + hh];
                    acc += f * red_o[(w * RU + hh) * D + dd];
                }
                acc *= v_scale;                                    // 1 unless the pool is FP8
                const int64_t sh = MQ ? s_rowoff[hh] : static_cast<int64_t>(s) * n_q + h0 + r0 + hh;
                if (nparts == 1) {
                    store_any(out, sh * D + dd, acc / lsum, out_dtype);
                } else {
                    const int64_t w_idx = sh * max_parts + part;
                    ws_acc[w_idx * D + dd] = acc;
                    if (dd == 0) {
                        ws_ml[2 * w_idx] = M;
                        ws_ml[2 * w_idx + 1] = lsum;
                    }
                }
            }
        }
        // the combine's reads are done before any warp writes partials (or, when
        // they alias the rings, TMA data) again; s_next is visible to all
        __syncthreads();
        u = un;
        un = s_next;
        cu = nx;
        cu.live = next_live;
        cb ^= 1;
    }
}

inline int decode_sm_count()
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

template <typename T, typename QT, int D, int BS, bool FP8, bool MQ, int RU = 8>
cudaError_t run_mma(const DecodeArgs& a, cudaStream_t s, float scale_log2)
{
    // FP8 runs 3 CTAs per SM (registers capped at 168 by the launch bounds):
    // Llama-3-8B batch 0.273 -> 0.231 ms against 2 CTAs with 24 KB rings.
    constexpr int NS = decode_stages<T, D, FP8, RU>();
    using Cfg = DecodeCfg<T, D, NS, FP8, RU>;
    auto kern = decode_mma_kernel<T, QT, D, BS, NS, FP8, MQ, RU>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int per_sm = 1;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Cfg::kDynBytes);
        if (attr_err == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecWarps * 32,
                                                          Cfg::kDynBytes) != cudaSuccess)
            per_sm = 1;
        if (per_sm < 1) per_sm = 1;
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap kmap{}, vmap{};
    const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * a.cache.n_kv_heads * BS;
    if constexpr (FP8) {
        // K: rows of D codes, 128- (D 128) or 64-byte (D 64) swizzle; V's
        // 16-token pieces are plain bulk copies (the kernel leaves vmap unused)
        if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, D, kRows, D) != PA_OK)
            return cudaErrorInvalidValue;
    } else {
        if (encode_pool_map(&kmap, a.k_cache, a.cache.dtype, D, rows, 64, kRows) != PA_OK ||
            encode_pool_map(&vmap, a.v_cache, a.cache.dtype, D, rows, 64, kRows) != PA_OK)
            return cudaErrorInvalidValue;
    }
    const int group = a.n_q / a.cache.n_kv_heads;
    const int64_t upper = static_cast<int64_t>(a.num_seqs) * a.max_parts * a.cache.n_kv_heads *
                          ((group * a.q_per_seq + RU - 1) / RU);
    const int64_t resident = static_cast<int64_t>(decode_sm_count()) * per_sm;
    const unsigned grid = static_cast<unsigned>(upper < resident ? upper : resident);
    // small batches (at most kStaticUnitsPerCta units per resident CTA, counted
    // with every sequence at the longest length) are dealt round robin: no
    // counter to clear, so no memset before the launch
    unsigned* ticket = upper <= kStaticUnitsPerCta * resident ? nullptr : a.ticket;
    if (ticket) {
        const cudaError_t e0 = cudaMemsetAsync(ticket, 0, sizeof(unsigned), s);
        if (e0 != cudaSuccess) return e0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecWarps * 32);
    cfg.dynamicSmemBytes = Cfg::kDynBytes;
    cfg.stream = s;
    // with no memset in front, the kernel is a programmatic dependent of the
    // kernel before it (the cache write): it is scheduled while that one
    // drains and waits for it before reading any input
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ticket ? 0 : 1;
    return cudaLaunchKernelEx(
        &cfg, kern, kmap, vmap, static_cast<const uint8_t*>(a.v_cache), a.out, a.out_dtype,
        static_cast<const QT*>(a.q), a.block_tables, a.max_blocks, a.context_lens, a.num_seqs,
        a.n_q, a.q_per_seq, a.cache.n_kv_heads, group, a.cache.num_blocks,
        FP8 ? scale_log2 * a.cache.k_scale : scale_log2, FP8 ? a.cache.v_scale : 1.f, a.ws_ml,
        a.ws_acc, a.part_tokens, a.max_parts, ticket, a.err);
}

// Tensor-core kernels by shape; cudaErrorNotSupported for other shapes.
template <typename T, bool MQ>
cudaError_t run_mma_tc(const DecodeArgs& a, cudaStream_t s, float sl2)
{
    const int D = a.cache.head_dim, BS = a.cache.block_size;
    if constexpr (MQ) {
        // more than 8 (head, query) rows per KV head: 16-row units, so each K/V
        // stage is read and widened once for all of them
        if (a.q_per_seq * (a.n_q / a.cache.n_kv_heads) > 8) {
            if (D == 64 && BS == 16) return run_mma<T, T, 64, 16, false, MQ, 16>(a, s, sl2);
            if (D == 64 && BS == 32) return run_mma<T, T, 64, 32, false, MQ, 16>(a, s, sl2);
            if (D == 128 && BS == 16) return run_mma<T, T, 128, 16, false, MQ, 16>(a, s, sl2);
            if (D == 128 && BS == 32) return run_mma<T, T, 128, 32, false, MQ, 16>(a, s, sl2);
            return cudaErrorNotSupported;
        }
    }
    if (D == 64 && BS == 16) return run_mma<T, T, 64, 16, false, MQ>(a, s, sl2);
    if (D == 64 && BS == 32) return run_mma<T, T, 64, 32, false, MQ>(a, s, sl2);
    if (D == 128 && BS == 16) return run_mma<T, T, 128, 16, false, MQ>(a, s, sl2);
    if (D == 128 && BS == 32) return run_mma<T, T, 128, 32, false, MQ>(a, s, sl2);
    return cudaErrorNotSupported;
}

template <typename QT, bool MQ>
cudaError_t run_fp8_qt(const DecodeArgs& a, cudaStream_t s, float sl2)
{
    const int D = a.cache.head_dim, BS = a.cache.block_size;
    if constexpr (!MQ) {
        // up to 4 query heads a KV head: the transposed kernel (4-row units)
        if (a.n_q / a.cache.n_kv_heads <= 4) {
            if (D == 64 && BS == 16) return run_mma<__half, QT, 64, 16, true, false, 4>(a, s, sl2);
            if (D == 64 && BS == 32) return run_mma<__half, QT, 64, 32, true, false, 4>(a, s, sl2);
            if (D == 128 && BS == 16) return run_mma<__half, QT, 128, 16, true, false, 4>(a, s, sl2);
            if (D == 128 && BS == 32) return run_mma<__half, QT, 128, 32, true, false, 4>(a, s, sl2);
            return cudaErrorNotSupported;
        }
    }
    if (D == 64 && BS == 16) return run_mma<__half, QT, 64, 16, true, MQ>(a, s, sl2);
    if (D == 64 && BS == 32) return run_mma<__half, QT, 64, 32, true, MQ>(a, s, sl2);
    if (D == 128 && BS == 16) return run_mma<__half, QT, 128, 16, true, MQ>(a, s, sl2);
    if (D == 128 && BS == 32) return run_mma<__half, QT, 128, 32, true, MQ>(a, s, sl2);
    return cudaErrorNotSupported;
}

// The attention kernel of a decode call for every cache dtype the tensor
// cores cover (FP32 pools: cudaErrorNotSupported).
template <bool MQ>
cudaError_t run_mma_any(const DecodeArgs& a, cudaStream_t s, float sl2)
{
    switch (a.cache.dtype) {
        case PA_BF16: return run_mma_tc<__nv_bfloat16, MQ>(a, s, sl2);
        case PA_F16: return run_mma_tc<__half, MQ>(a, s, sl2);
        case PA_FP8_E4M3:
            return a.cache.act_dtype == PA_BF16 ? run_fp8_qt<__nv_bfloat16, MQ>(a, s, sl2)
                                                : run_fp8_qt<__half, MQ>(a, s, sl2);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
