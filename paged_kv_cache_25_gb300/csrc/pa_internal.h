// Host-side internals shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Tokens per decode partition for a launch: every partition of a sequence but
// its last covers exactly this many tokens (a multiple of the block size).
int decode_partition_tokens(int64_t seq_groups, int block_size, int max_context_len);

// Records a host-side failure message for pa_last_error_message().
pa_status fail(pa_status st, const char* fmt, ...);
pa_status cuda_fail(cudaError_t e, const char* what);

// Device address of this device's error word (cached per device).
unsigned* device_error_word();

// Encodes a 2-D tiled tensor map over a pool viewed as rows of head_dim
// elements: dims {head_dim, rows}, box {box_x, box_y}, 128-byte swizzle.
// swizzle: 0 none, 64 or 128 (bytes); row_elems = elements per row of the view
pa_status encode_pool_map(CUtensorMap* map, const void* base, pa_dtype dt, int row_elems,
                          uint64_t rows, int box_x, int box_y, int swizzle = 128);

// Profiling events for the main decode kernel (may be null).
void profile_events(cudaEvent_t* start, cudaEvent_t* stop);

inline int elem_bytes(pa_dtype d) { return d == PA_F32 ? 4 : (d == PA_FP8_E4M3 ? 1 : 2); }

// ---- launchers (defined next to their kernels) ----
cudaError_t launch_cache_write(const void* k, const void* v, void* kc, void* vc,
                               const int64_t* slots, int T, const pa_cache_desc& c,
                               unsigned* err, cudaStream_t s);
cudaError_t launch_cache_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* kc,
                                   void* vc, const int64_t* slots, int T, const pa_cache_desc& c,
                                   unsigned* err, cudaStream_t s);

cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, int src_blocks, void* dst_k,
                               void* dst_v, int dst_blocks, const pa_cache_desc& layout,
                               const int32_t* mapping, int pairs, unsigned* err, cudaStream_t s);

struct DecodeArgs {
    void* out; pa_dtype out_dtype; const void* q;
    const void* k_cache; const void* v_cache; pa_cache_desc cache;
    const int32_t* block_tables; int max_blocks;
    const int32_t* context_lens; int num_seqs; int n_q; float scale;
    int q_per_seq;     // query rows per sequence (1 for decode; k+1 to verify k drafts)
    float* ws_ml;      // [B][q_per_seq][n_q][J][2] (m, l) or null
    float* ws_acc;     // [B][q_per_seq][n_q][J][d] or null
    int part_tokens;   // tokens per partition
    int max_parts;     // J: partitions of the longest possible sequence
    unsigned* ticket;  // work counter in the workspace's control area; null: units are
                       // dealt round robin (unit blockIdx.x + k * gridDim.x), no counter
    unsigned* err;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// attention kernel of a call with q_per_seq > 1 (decode_verify.cu)
cudaError_t launch_decode_mq(const DecodeArgs& a, cudaStream_t s, float scale_log2);

struct PrefillArgs {
    void* out; pa_dtype out_dtype; const void* q;
    const void* k_cache; const void* v_cache; pa_cache_desc cache;
    const int32_t* block_tables; int max_blocks;
    const int32_t* q_start; const int32_t* context_lens;
    int num_reqs; int max_q; int n_q; float scale;
    unsigned* err;
};
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

}  // namespace pa
