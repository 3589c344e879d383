// Host prefix cache over the physical block pool: automatic reuse of K/V
// blocks whose tokens, and every token before them, match an earlier request.
//
//   - a full block's fingerprint chains the fingerprint of the block before it
//     with the block's own token ids ("Inference engineering", Trick 3;
//     "The hands-on guide to LLM Inference with vLLM", Automatic Prefix
//     Caching), here FNV-1a 64 over the parent fingerprint (8 bytes, little
//     endian) then each token id (4 bytes, little endian); block 0's parent is 0;
//   - a lookup table maps fingerprints to blocks whose K/V have been computed;
//     an entry also keeps the parent fingerprint and the tokens, so a hit means
//     the contents are equal, never just the 64-bit fingerprint;
//   - a request reuses its leading run of hitting full blocks ("vLLM Serving",
//     "Prefix caching (automatic KV reuse)"); each block counts the requests
//     using it;
//   - a block whose count drops to zero keeps its entry and waits on an LRU
//     list; blocks are taken from the free queue first and, only when it is
//     empty, by evicting the least recently released cached block.
// Host memory only; not thread-safe (one owner thread).
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

constexpr uint64_t kFnvBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

uint64_t fnv1a_bytes(uint64_t h, uint64_t v, int nbytes)
{
    for (int i = 0; i < nbytes; ++i) {
        h ^= (v >> (8 * i)) & 0xFFu;
        h *= kFnvPrime;
    }
    return h;
}

uint64_t block_hash(uint64_t parent, const int32_t* tokens, int bs)
{
    uint64_t h = fnv1a_bytes(kFnvBasis, parent, 8);
    for (int i = 0; i < bs; ++i) h = fnv1a_bytes(h, static_cast<uint32_t>(tokens[i]), 4);
    return h;
}

}  // namespace

struct pa_prefix {
    int n = 0, bs = 0;
    std::vector<int> ref;
    std::deque<int> free_q;                          // never-cached (or evicted) free blocks
    std::vector<int> prev, next;                     // LRU list of cached blocks with count 0
    int lru_head = -1, lru_tail = -1, lru_size = 0;
    std::vector<uint8_t> in_lru, cached;
    std::vector<uint64_t> hash, parent;
    std::vector<int32_t> toks;                       // [n][bs] tokens of cached blocks
    std::unordered_multimap<uint64_t, int> table;

    void lru_push_back(int b)
    {
        prev[b] = lru_tail;
        next[b] = -1;
        if (lru_tail >= 0) next[lru_tail] = b; else lru_head = b;
        lru_tail = b;
        in_lru[b] = 1;
        ++lru_size;
    }
    void lru_remove(int b)
    {
        if (prev[b] >= 0) next[prev[b]] = next[b]; else lru_head = next[b];
        if (next[b] >= 0) prev[next[b]] = prev[b]; else lru_tail = prev[b];
        prev[b] = next[b] = -1;
        in_lru[b] = 0;
        --lru_size;
    }
    // cached block holding exactly (parent, tokens), or -1
    int find(uint64_t h, uint64_t par, const int32_t* t) const
    {
        auto range = table.equal_range(h);
        for (auto it = range.first; it != range.second; ++it) {
            const int b = it->second;
            if (parent[b] == par && std::memcmp(&toks[static_cast<size_t>(b) * bs], t,
                                                sizeof(int32_t) * bs) == 0)
                return b;
        }
        return -1;
    }
    void uncache(int b)
    {
        auto range = table.equal_range(hash[b]);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second == b) {
                table.erase(it);
                break;
            }
        cached[b] = 0;
    }
    int take_one()
    {
        int b;
        if (!free_q.empty()) {
            b = free_q.front();
            free_q.pop_front();
        } else {
            b = lru_head;                            // evict the least recently released
            lru_remove(b);
            uncache(b);
        }
        ref[b] = 1;
        return b;
    }
    // leading full blocks of tokens that hit; ids into out (may be NULL)
    int hits(const int32_t* tokens, int n_tokens, int32_t* out) const
    {
        uint64_t par = 0;
        int k = 0;
        for (; k < n_tokens / bs; ++k) {
            const int32_t* t = tokens + static_cast<size_t>(k) * bs;
            const int b = find(block_hash(par, t, bs), par, t);
            if (b < 0) break;
            if (out) out[k] = b;
            par = hash[b];
        }
        return k;
    }
};

extern "C" {

uint64_t pa_prefix_block_hash(uint64_t parent, const int32_t* tokens, int block_size)
{
    if (!tokens || block_size <= 0) return 0;
    return block_hash(parent, tokens, block_size);
}

pa_prefix* pa_prefix_create(int num_blocks, int block_size, const int32_t* free_order)
{
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_prefix* p = new (std::nothrow) pa_prefix;
    if (!p) return nullptr;
    p->n = num_blocks;
    p->bs = block_size;
    p->ref.assign(num_blocks, 0);
    p->prev.assign(num_blocks, -1);
    p->next.assign(num_blocks, -1);
    p->in_lru.assign(num_blocks, 0);
    p->cached.assign(num_blocks, 0);
    p->hash.assign(num_blocks, 0);
    p->parent.assign(num_blocks, 0);
    p->toks.assign(static_cast<size_t>(num_blocks) * block_size, 0);
    std::vector<uint8_t> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
        const int b = free_order ? free_order[i] : i;
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete p;
            return nullptr;
        }
        seen[b] = 1;
        p->free_q.push_back(b);
    }
    return p;
}

void pa_prefix_destroy(pa_prefix* p) { delete p; }

int pa_prefix_lookup(const pa_prefix* p, const int32_t* tokens, int n_tokens)
{
    if (!p || n_tokens < 0 || (n_tokens > 0 && !tokens)) return -1;
    return p->hits(tokens, n_tokens, nullptr);
}

int pa_prefix_acquire(pa_prefix* p, const int32_t* tokens, int n_tokens, int32_t* table,
                      int table_len)
{
    if (!p || n_tokens <= 0 || !tokens || !table) return -2;
    const int need = (n_tokens + p->bs - 1) / p->bs;
    if (table_len < need) return -2;
    std::vector<int32_t> hit(need);
    const int k = p->hits(tokens, n_tokens, hit.data());
    int hit_in_lru = 0;
    for (int i = 0; i < k; ++i) hit_in_lru += p->in_lru[hit[i]];
    const int64_t avail = static_cast<int64_t>(p->free_q.size()) + p->lru_size - hit_in_lru;
    if (avail < need - k) return -1;                 // nothing taken
    for (int i = 0; i < k; ++i) {
        const int b = hit[i];
        if (p->in_lru[b]) p->lru_remove(b);
        ++p->ref[b];
        table[i] = b;
    }
    for (int i = k; i < need; ++i) table[i] = p->take_one();
    for (int i = need; i < table_len; ++i) table[i] = -1;
    return k;
}

int pa_prefix_alloc(pa_prefix* p, int n, int32_t* out)
{
    if (!p || n < 0 || (n > 0 && !out)) return -2;
    if (static_cast<int64_t>(p->free_q.size()) + p->lru_size < n) return -1;
    for (int i = 0; i < n; ++i) out[i] = p->take_one();
    return 0;
}

int pa_prefix_commit(pa_prefix* p, const int32_t* tokens, int n_tokens, const int32_t* table)
{
    if (!p || n_tokens < 0 || (n_tokens > 0 && (!tokens || !table))) return -2;
    const int full = n_tokens / p->bs;
    for (int i = 0; i < full; ++i)                   // every full block must be held
        if (table[i] < 0 || table[i] >= p->n || p->ref[table[i]] <= 0) return -2;
    // first pass: a block to enter must not hold other contents already
    std::vector<uint64_t> hs(full), ps(full);
    std::vector<int> have(full);
    uint64_t par = 0;
    for (int i = 0; i < full; ++i) {
        const int32_t* t = tokens + static_cast<size_t>(i) * p->bs;
        hs[i] = block_hash(par, t, p->bs);
        ps[i] = par;
        have[i] = p->find(hs[i], par, t);
        if (have[i] < 0 && p->cached[table[i]]) return -2;
        par = hs[i];
    }
    int added = 0;
    for (int i = 0; i < full; ++i) {
        // have == table[i]: cached already; another block: the same contents
        // were cached first by another request, so table[i] stays private
        if (have[i] >= 0) continue;
        const int b = table[i];
        p->cached[b] = 1;
        p->hash[b] = hs[i];
        p->parent[b] = ps[i];
        std::memcpy(&p->toks[static_cast<size_t>(b) * p->bs], tokens + static_cast<size_t>(i) * p->bs,
                    sizeof(int32_t) * p->bs);
        p->table.emplace(hs[i], b);
        ++added;
    }
    return added;
}

int pa_prefix_release(pa_prefix* p, const int32_t* table, int n_blocks)
{
    if (!p || n_blocks < 0 || (n_blocks > 0 && !table)) return -2;
    std::vector<int> drops(0);
    for (int i = 0; i < n_blocks; ++i) {
        const int b = table[i];
        if (b < 0) continue;
        if (b >= p->n) return -2;
        drops.push_back(b);
    }
    // a block listed twice must hold two references
    std::unordered_map<int, int> cnt;
    for (int b : drops) ++cnt[b];
    for (const auto& kv : cnt)
        if (p->ref[kv.first] < kv.second) return -2;
    // deepest block first: among blocks released together the end of a
    // sequence is evicted before its prefix
    for (int i = static_cast<int>(drops.size()) - 1; i >= 0; --i) {
        const int b = drops[i];
        if (--p->ref[b] == 0) {
            if (p->cached[b]) p->lru_push_back(b); else p->free_q.push_back(b);
        }
    }
    return 0;
}

int pa_prefix_num_free(const pa_prefix* p) { return p ? static_cast<int>(p->free_q.size()) : -1; }
int pa_prefix_num_evictable(const pa_prefix* p) { return p ? p->lru_size : -1; }
int pa_prefix_num_cached(const pa_prefix* p) { return p ? static_cast<int>(p->table.size()) : -1; }
int pa_prefix_refcount(const pa_prefix* p, int block)
{
    return (p && block >= 0 && block < p->n) ? p->ref[block] : -1;
}

}  // extern "C"
