"""Host prefix cache: the oracle pinned against the FNV-1a definition and a
brute-force model of prefix reuse, then the library checked against the oracle
operation by operation (CPU only)."""
import numpy as np
import pytest

from oracle import prefix_cache as ref
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    return pa.lib()


# ------------------------------------------------------------------ oracle pins

def test_fnv1a64_published_vectors():
    # FNV-1a 64 test values from the algorithm's published definition
    assert ref.fnv1a64(b"") == 0xCBF29CE484222325
    assert ref.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert ref.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_chains_every_earlier_token():
    rng = np.random.default_rng(5)
    toks = rng.integers(0, 50000, size=64)
    bs = 16

    def chain(t):
        out, parent = [], 0
        for k in range(len(t) // bs):
            parent = ref.block_hash(parent, t[k * bs:(k + 1) * bs])
            out.append(parent)
        return out

    base = chain(toks)
    assert len(set(base)) == 4
    for pos in (0, 17, 40, 63):
        t2 = toks.copy()
        t2[pos] += 1
        c2 = chain(t2)
        k = pos // bs
        assert c2[:k] == base[:k]                        # blocks before the change keep theirs
        assert all(a != b for a, b in zip(c2[k:], base[k:]))   # this and every later block change
    # the token bytes are little endian: token 1 differs from token 256
    assert ref.block_hash(0, [1]) != ref.block_hash(0, [256])


def _common_full_blocks(a, b, bs):
    k = 0
    while (k + 1) * bs <= min(len(a), len(b)) and list(a[k * bs:(k + 1) * bs]) == list(b[k * bs:(k + 1) * bs]):
        k += 1
    return k


def test_oracle_hits_equal_brute_force_longest_cached_prefix():
    """Large pool (no eviction): a request hits exactly the longest run of
    leading full blocks that some committed request shares with it, and the
    hit blocks are the blocks that first committed those contents."""
    rng = np.random.default_rng(11)
    for bs in (2, 3, 4):
        pc = ref.PrefixCache(4000, bs)
        committed = []            # token lists of committed requests
        first_block = {}          # full-prefix tuple -> block id that first cached it
        for _ in range(120):
            if committed and rng.random() < 0.6:       # extend or branch off an earlier request
                base = committed[rng.integers(len(committed))]
                cut = int(rng.integers(0, len(base) + 1))
                toks = list(base[:cut]) + list(rng.integers(0, 2, size=int(rng.integers(1, 9))))
            else:
                toks = list(rng.integers(0, 2, size=int(rng.integers(1, 13))))
            expect = max([min(_common_full_blocks(toks, c, bs), len(c) // bs) for c in committed],
                         default=0)
            k, table = pc.acquire(toks, 8)
            assert k == expect
            for i in range(k):
                assert table[i] == first_block[tuple(toks[:(i + 1) * bs])]
            pc.commit(toks, table)
            for i in range(len(toks) // bs):
                first_block.setdefault(tuple(toks[:(i + 1) * bs]), int(table[i]))
            committed.append(toks)
            if rng.random() < 0.5:
                pc.release(table)


def test_oracle_eviction_is_least_recently_released():
    bs = 2
    pc = ref.PrefixCache(6, bs)
    a = [1, 1, 2, 2]          # 2 full blocks
    b = [3, 3, 4, 4]
    ka, ta = pc.acquire(a, 2)
    pc.commit(a, ta)
    kb, tb = pc.acquire(b, 2)
    pc.commit(b, tb)
    pc.release(ta)            # released first: evicted first, deepest block first
    pc.release(tb)
    assert pc.num_free() == 2 and pc.num_evictable() == 4
    got = pc.alloc(3)          # 2 free blocks, then 1 eviction
    assert list(got[:2]) == [4, 5]
    assert got[2] == ta[1]     # a's second block went first
    assert pc.lookup(a) == 1 and pc.lookup(b) == 2
    got2 = pc.alloc(1)
    assert got2[0] == ta[0] and pc.lookup(a) == 0
    # with nothing free, b's blocks are the only source: a request hitting both
    # of them still needs a third block
    assert pc.acquire(b + [9], 3) is None
    pc.release(got2)          # ta[0] lost its entry: back to the free queue
    assert pc.num_free() == 1
    # a hit takes a cached block off the LRU list: it is no longer evictable
    kb2, tb2 = pc.acquire(b + [9], 3)
    assert kb2 == 2 and list(tb2[:2]) == list(tb)
    assert pc.num_evictable() == 0 and pc.alloc(1) is None


def test_oracle_invariants_under_random_streams_with_eviction():
    rng = np.random.default_rng(23)
    bs, nb = 4, 24
    pc = ref.PrefixCache(nb, bs, order=rng.permutation(nb))
    live = {}                  # id -> (tokens, table)
    stems = [list(rng.integers(0, 3, size=12)) for _ in range(3)]
    for step in range(600):
        op = rng.random()
        if op < 0.5 or not live:
            stem = stems[rng.integers(3)]
            toks = stem[:int(rng.integers(0, 13))] + list(rng.integers(0, 3, size=int(rng.integers(1, 7))))
            r = pc.acquire(toks, 6)
            if r is not None:
                k, table = r
                if rng.random() < 0.8:
                    pc.commit(toks, table)
                live[step] = (toks, table)
        else:
            key = list(live)[rng.integers(len(live))]
            pc.release(live.pop(key)[1])
        # counts: every block is free, evictable or held, never two of these
        held = {}
        for toks, table in live.values():
            for b in table:
                if b >= 0:
                    held[b] = held.get(b, 0) + 1
        for b in range(nb):
            assert pc.ref[b] == held.get(b, 0)
        assert len(pc.free) + len(pc.lru) + len(held) == nb
        assert not set(pc.free) & set(pc.lru)
        assert all(b in pc.entry for b in pc.lru) and not any(b in pc.entry for b in pc.free)
        # every cached block's entry is the contents of the requests using it
        for toks, table in live.values():
            parent = 0
            for i in range(len(toks) // bs):
                h = ref.block_hash(parent, toks[i * bs:(i + 1) * bs])
                if table[i] in pc.entry:
                    assert pc.entry[table[i]] == (h, parent, tuple(toks[i * bs:(i + 1) * bs]))
                parent = h


# ------------------------------------------------------------------ library vs oracle

def test_library_block_hash_matches_oracle():
    rng = np.random.default_rng(3)
    for bs in (1, 16, 32):
        for _ in range(20):
            t = rng.integers(-2**31, 2**31, size=bs, dtype=np.int64).astype(np.int32)
            parent = int(rng.integers(0, 2**63))
            assert pa.pa_prefix_block_hash(parent, t) == ref.block_hash(parent, t)


@pytest.mark.parametrize("seed,bs,nb", [(1, 4, 32), (2, 16, 40), (3, 2, 12), (4, 32, 64)])
def test_library_matches_oracle_op_by_op(seed, bs, nb):
    rng = np.random.default_rng(seed)
    order = rng.permutation(nb)
    lib_c, orc = pa.PrefixCache(nb, bs, order), ref.PrefixCache(nb, bs, order)
    stems = [list(rng.integers(0, 4, size=5 * bs)) for _ in range(4)]
    live = []
    for step in range(500):
        op = rng.random()
        if op < 0.45 or not live:
            stem = stems[rng.integers(4)]
            toks = stem[:int(rng.integers(0, 5 * bs + 1))] + list(
                rng.integers(0, 4, size=int(rng.integers(1, 2 * bs))))
            tl = -(-len(toks) // bs) + 1
            assert lib_c.lookup(toks) == orc.lookup(toks)
            a, b = lib_c.acquire(toks, tl), orc.acquire(toks, tl)
            assert (a is None) == (b is None)
            if a is not None:
                assert a[0] == b[0] and list(a[1]) == list(b[1])
                if rng.random() < 0.85:
                    assert lib_c.commit(toks, a[1]) == orc.commit(toks, b[1])
                live.append(list(a[1]))
        elif op < 0.55:
            n = int(rng.integers(0, 4))
            a, b = lib_c.alloc(n), orc.alloc(n)
            assert (a is None) == (b is None)
            if a is not None:
                assert list(a) == list(b)
                live.append(list(a))
        else:
            table = live.pop(int(rng.integers(len(live))))
            lib_c.release(table)
            orc.release(table)
        assert lib_c.num_free() == orc.num_free()
        assert lib_c.num_evictable() == orc.num_evictable()
        assert lib_c.num_cached() == orc.num_cached()
        assert [lib_c.refcount(i) for i in range(nb)] == orc.ref


def test_library_rejects_bad_calls_without_changing_state():
    c = pa.PrefixCache(8, 4)
    k, table = c.acquire(list(range(9)), 3)
    with pytest.raises(pa.PAError):
        c.release([table[0], table[0]])            # one reference only
    with pytest.raises(pa.PAError):
        c.release([99])
    assert [c.refcount(int(b)) for b in table] == [1, 1, 1]
    with pytest.raises(pa.PAError):
        c.commit(list(range(8)), [table[0], 7])    # block 7 is not held
    assert c.num_cached() == 0
    with pytest.raises(pa.PAError):
        c.acquire(list(range(9)), 2)               # table too short
    assert c.commit(list(range(9)), table) == 2
    # a held block that already caches other contents cannot be entered again
    with pytest.raises(pa.PAError):
        c.commit([5, 5, 5, 5], [table[0]])
    assert c.num_cached() == 2
    with pytest.raises(pa.PAError):
        pa.PrefixCache(4, 4, [0, 1, 1, 2])
