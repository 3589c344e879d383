"""Oracle of the host prefix cache (TEST INFRASTRUCTURE ONLY).

Only ``tests/`` may import this module; the product library never does, and
this module imports nothing from the product package.

What it follows:

* "The hands-on guide to LLM Inference with vLLM", Automatic Prefix Caching: a
  block's contents are fixed by its own tokens and every token before them, so
  each block is fingerprinted and a lookup table keeps the blocks already
  computed; a new request reuses every block found there.
* "Inference engineering", Trick 3 (Prefix caching): a page's fingerprint is
  built from its tokens and the fingerprint of the page before it; only full
  pages are cached; pages count the requests using them; when memory is
  needed the least recently used unused pages are thrown out first.
* "vLLM Serving ...", Prefix caching (automatic KV reuse): matching blocks are
  put into the new request's block table; under memory pressure cached blocks
  are evicted LRU.

Readings where the pages leave a step open (listed with the others in the
design notes): the fingerprint is FNV-1a 64 (its published definition: offset
basis 0xcbf29ce484222325, prime 0x100000001b3, xor then multiply per byte) over
the parent fingerprint as 8 little-endian bytes and each token id as 4
little-endian bytes, the first block's parent being 0; a table entry keeps the
parent fingerprint and the tokens, so a hit is an exact content match; a
request reuses its leading run of hits; a block enters the table when the
request that wrote it commits it; new blocks come from the free queue (FIFO,
as in "Life of a prompt") and only when it is empty from the LRU end of the
unused cached blocks; blocks released together count as released from the
end of the sequence backwards.

Written plainly: Python lists and dicts, no shared code with the product.
"""
from __future__ import annotations

FNV_BASIS = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
_MASK = (1 << 64) - 1


def fnv1a64(data: bytes, h: int = FNV_BASIS) -> int:
    """FNV-1a, 64 bits: for each byte, xor it in, then multiply by the prime."""
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & _MASK
    return h


def block_hash(parent: int, tokens) -> int:
    data = int(parent).to_bytes(8, "little")
    for t in tokens:
        data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


class PrefixCache:
    def __init__(self, num_blocks: int, block_size: int, order=None):
        self.n, self.bs = num_blocks, block_size
        self.free = [int(b) for b in (range(num_blocks) if order is None else order)]
        assert sorted(self.free) == list(range(num_blocks))
        self.lru = []            # unused cached blocks, least recently released first
        self.ref = [0] * num_blocks
        self.entry = {}          # block -> (hash, parent, tokens)
        self.where = {}          # (hash, parent, tokens) -> block

    # ---- queries -------------------------------------------------------
    def hit_blocks(self, tokens):
        out, parent = [], 0
        for k in range(len(tokens) // self.bs):
            t = tuple(int(x) for x in tokens[k * self.bs:(k + 1) * self.bs])
            h = block_hash(parent, t)
            b = self.where.get((h, parent, t))
            if b is None:
                break
            out.append(b)
            parent = h
        return out

    def lookup(self, tokens) -> int:
        return len(self.hit_blocks(tokens))

    def num_free(self):
        return len(self.free)

    def num_evictable(self):
        return len(self.lru)

    def num_cached(self):
        return len(self.where)

    # ---- changes -------------------------------------------------------
    def _take(self):
        if self.free:
            b = self.free.pop(0)
        else:
            b = self.lru.pop(0)                      # least recently released
            del self.where[self.entry.pop(b)]
        self.ref[b] = 1
        return b

    def acquire(self, tokens, table_len):
        """(hit count, table) or None when the pool cannot supply the rest."""
        need = -(-len(tokens) // self.bs)
        hits = self.hit_blocks(tokens)
        spare = len(self.free) + len([b for b in self.lru if b not in hits])
        if spare < need - len(hits):
            return None
        for b in hits:
            if b in self.lru:
                self.lru.remove(b)
            self.ref[b] += 1
        table = hits + [self._take() for _ in range(need - len(hits))]
        return len(hits), table + [-1] * (table_len - need)

    def alloc(self, n):
        if len(self.free) + len(self.lru) < n:
            return None
        return [self._take() for _ in range(n)]

    def commit(self, tokens, table) -> int:
        parent, todo = 0, []
        for k in range(len(tokens) // self.bs):
            assert self.ref[table[k]] > 0
            t = tuple(int(x) for x in tokens[k * self.bs:(k + 1) * self.bs])
            h = block_hash(parent, t)
            if (h, parent, t) not in self.where:
                assert table[k] not in self.entry, "block already holds other contents"
                todo.append((table[k], (h, parent, t)))
            parent = h
        for b, key in todo:
            self.entry[b] = key
            self.where[key] = b
        return len(todo)

    def release(self, table):
        ids = [int(b) for b in table if b >= 0]
        for b in set(ids):
            assert self.ref[b] >= ids.count(b)
        for b in reversed(ids):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                (self.lru if b in self.entry else self.free).append(b)
