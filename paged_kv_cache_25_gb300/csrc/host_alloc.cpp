// Host-side block allocator, page tables and slot mapping ("Life of a prompt",
// "Back to the queue, and into vLLM proper": a FIFO free-block queue on the
// CPU, a page table per sequence, one more block every block_size tokens,
// blocks back in the queue as soon as a sequence lets go of them; "vLLM
// Serving ...", "Sharing and copy-on-write": reference counts let several
// tables point at one physical block).
#include <cstdint>
#include <deque>
#include <vector>

#include "../../include/pa.h"

struct pa_alloc {
    std::deque<int32_t> free_q;     // head = next block handed out
    std::vector<int32_t> refs;      // references per physical block
};

namespace {
pa_status host_fail(pa_status st) { return st; }
}

extern "C" {

pa_alloc* pa_alloc_create(int num_blocks, const int32_t* initial_order)
{
    if (num_blocks < 0) return nullptr;
    pa_alloc* a = new pa_alloc;
    a->refs.assign(static_cast<size_t>(num_blocks), 0);
    std::vector<uint8_t> seen(static_cast<size_t>(num_blocks), 0);
    for (int i = 0; i < num_blocks; ++i) {
        const int32_t id = initial_order ? initial_order[i] : i;
        if (id < 0 || id >= num_blocks || seen[id]) {   // not a permutation
            delete a;
            return nullptr;
        }
        seen[id] = 1;
        a->free_q.push_back(id);
    }
    return a;
}

int pa_alloc_blocks(pa_alloc* a, int n, int32_t* out)
{
    if (!a || n < 0 || static_cast<size_t>(n) > a->free_q.size()) return -1;
    for (int i = 0; i < n; ++i) {
        out[i] = a->free_q.front();
        a->free_q.pop_front();
        a->refs[out[i]] = 1;
    }
    return 0;
}

void pa_alloc_share(pa_alloc* a, const int32_t* ids, int n)
{
    if (!a) return;
    for (int i = 0; i < n; ++i)
        if (ids[i] >= 0 && static_cast<size_t>(ids[i]) < a->refs.size() && a->refs[ids[i]] > 0)
            ++a->refs[ids[i]];
}

void pa_alloc_free(pa_alloc* a, const int32_t* ids, int n)
{
    if (!a) return;
    for (int i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (id < 0 || static_cast<size_t>(id) >= a->refs.size() || a->refs[id] == 0) continue;
        if (--a->refs[id] == 0) a->free_q.push_back(id);
    }
}

int pa_alloc_num_free(const pa_alloc* a) { return a ? static_cast<int>(a->free_q.size()) : 0; }

int pa_alloc_refcount(const pa_alloc* a, int block_id)
{
    if (!a || block_id < 0 || static_cast<size_t>(block_id) >= a->refs.size()) return -1;
    return a->refs[block_id];
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

pa_status pa_alloc_build_tables(pa_alloc* a, int num_seqs, const int32_t* lens,
                                const uint8_t* sharer, int prefix_tokens, int block_size,
                                int max_blocks_per_seq, int32_t* tables)
{
    if (!a || num_seqs < 0 || !lens || !tables || block_size <= 0 || max_blocks_per_seq <= 0 ||
        prefix_tokens < 0 || prefix_tokens % block_size != 0)
        return host_fail(PA_ERR_INVALID_ARG);
    // check sizes before taking anything, so a failure leaves the queue as it was
    bool any_sharer = false;
    int64_t want = 0;
    const int n_prefix = prefix_tokens / block_size;
    for (int s = 0; s < num_seqs; ++s) {
        if (lens[s] < 0) return host_fail(PA_ERR_INVALID_ARG);
        const int64_t blocks = (static_cast<int64_t>(lens[s]) + block_size - 1) / block_size;
        if (blocks > max_blocks_per_seq) return host_fail(PA_ERR_INVALID_ARG);
        const bool sh = sharer && sharer[s] && n_prefix > 0;
        if (sh && lens[s] < prefix_tokens) return host_fail(PA_ERR_INVALID_ARG);
        any_sharer = any_sharer || sh;
        want += sh ? blocks - n_prefix : blocks;
    }
    if (any_sharer) want += n_prefix;
    if (want > static_cast<int64_t>(a->free_q.size())) return host_fail(PA_ERR_OUT_OF_RANGE);

    std::vector<int32_t> prefix(static_cast<size_t>(any_sharer ? n_prefix : 0));
    if (any_sharer) pa_alloc_blocks(a, n_prefix, prefix.data());
    bool first = true;
    for (int s = 0; s < num_seqs; ++s) {
        int32_t* row = tables + static_cast<int64_t>(s) * max_blocks_per_seq;
        for (int i = 0; i < max_blocks_per_seq; ++i) row[i] = -1;
        const int blocks = (lens[s] + block_size - 1) / block_size;
        int have = 0;
        if (any_sharer && sharer[s]) {
            for (int i = 0; i < n_prefix; ++i) row[i] = prefix[i];
            if (!first) pa_alloc_share(a, prefix.data(), n_prefix);
            first = false;
            have = n_prefix;
        }
        pa_alloc_blocks(a, blocks - have, row + have);
    }
    return PA_OK;
}

pa_status pa_slot_mapping(const int32_t* tables, int max_blocks_per_seq, int block_size,
                          const int32_t* seq, const int32_t* pos, int num_tokens, int64_t* slots)
{
    if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq <= 0)
        return host_fail(PA_ERR_INVALID_ARG);
    if (num_tokens == 0) return PA_OK;
    if (!tables || !seq || !pos || !slots) return host_fail(PA_ERR_INVALID_ARG);
    for (int t = 0; t < num_tokens; ++t) {
        if (seq[t] < 0 || pos[t] < 0) return host_fail(PA_ERR_INVALID_ARG);
        const int logical = pos[t] / block_size;
        if (logical >= max_blocks_per_seq) return host_fail(PA_ERR_INVALID_ARG);
        const int32_t phys = tables[static_cast<int64_t>(seq[t]) * max_blocks_per_seq + logical];
        if (phys < 0) return host_fail(PA_ERR_INVALID_ARG);
        slots[t] = static_cast<int64_t>(phys) * block_size + pos[t] % block_size;
    }
    return PA_OK;
}

int64_t pa_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int elem_bytes)
{
    // one K and one V vector per KV head, per layer
    return 2ll * n_layers * n_kv_heads * head_dim * elem_bytes;
}

int64_t pa_pool_blocks(int64_t pool_bytes, int block_size, int64_t bytes_per_token)
{
    const int64_t per_block = static_cast<int64_t>(block_size) * bytes_per_token;
    return per_block > 0 ? pool_bytes / per_block : 0;
}

}  // extern "C"
