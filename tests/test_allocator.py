"""Host block allocator: the reference model pinned to published facts and
worked cases, then the library's allocator checked against the model on
random lifecycles (same ids, tables, refcounts and counters at every step).
"""
import numpy as np
import pytest

from oracle.allocator_model import AllocatorModel, OutOfBlocks, block_hash, fnv1a64


@pytest.fixture(scope="module")
def pkv():
    import block_paged_kv_gb300 as m
    return m


# ---------------------------------------------------------------------------
# pins of the model
# ---------------------------------------------------------------------------
def test_fnv1a64_published_vectors():
    # the test vectors published with the FNV-1a definition
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_identity_carries_its_prefix():
    a = list(range(16))
    h0 = block_hash(0, a)
    assert block_hash(0, a) == h0
    assert block_hash(h0, a) != h0                # same tokens, different parent
    assert block_hash(0, a, extra=7) != h0        # an extra key (image digest) changes it
    assert block_hash(0, a[::-1]) != h0           # token order matters


def _hold(m, n_tokens):
    r = m.begin()
    m.reserve(r, n_tokens)
    return r


@pytest.mark.parametrize("cur,maxb,short,expect", [
    (100, 1000, 30, 200),    # doubling covers the shortfall
    (100, 1000, 150, 250),   # the shortfall is larger: jump straight to it
    (600, 1000, 10, 1000),   # never past the maximum
])
def test_grow_rule_worked_numbers(cur, maxb, short, expect):
    m = AllocatorModel(1, cur, maxb)
    _hold(m, cur)                       # every block in use, nothing cached
    r = m.begin()
    m.reserve(r, short)
    assert m.num_blocks == expect and m.grows == 1
    assert m.table(r) == list(range(cur, cur + short))   # the new ids, lowest first


def test_out_of_blocks_changes_nothing():
    m = AllocatorModel(1, 4, 6)
    _hold(m, 4)
    r = m.begin()
    m.reserve(r, 2)                     # grows to 6 (min(6, max(8, 6)))
    before = (m.num_blocks, list(m.free), list(m.lru), m.table(r))
    with pytest.raises(OutOfBlocks):
        m.reserve(r, 3)
    assert (m.num_blocks, list(m.free), list(m.lru), m.table(r)) == before


def test_shared_prompt_lifecycle_by_hand():
    bs = 4
    m = AllocatorModel(bs, 16, 16)
    system = [7] * 8 + [1, 2, 3]        # 2 full blocks + 3 tokens
    a = m.begin()
    assert m.find_cached_prefix(a, system) == 0
    m.reserve(a, len(system))
    assert m.table(a) == [0, 1, 2]
    m.publish(a, system)                # blocks 0, 1 full -> published; 2 stays private
    b = m.begin()
    assert m.find_cached_prefix(b, system + [9, 9]) == 8   # both full blocks shared
    m.reserve(b, len(system) + 2)       # 13 tokens: 4 blocks, 2 of them new
    assert m.table(b) == [0, 1, 3, 4]
    assert m.refcount[0] == 2 and m.refcount[1] == 2 and m.refcount[2] == 1
    m.release(a)                        # 0, 1 still held by b; 2 freed (never published)
    assert m.refcount[0] == 1 and 2 in m.free and m.lru == []
    m.publish(b, system + [9, 9])       # b's third block (id 3) is full: published
    m.release(b)
    assert m.lru == [0, 1, 3]           # cache-only in release order
    assert 4 in m.free                  # the partial last block was never published
    # a new request reuses the three cached blocks; the LRU empties in turn
    c = m.begin()
    assert m.find_cached_prefix(c, system + [9, 9, 5]) == 12
    assert m.table(c) == [0, 1, 3] and m.lru == []


def test_sliding_expiry_by_hand():
    bs = 4
    m = AllocatorModel(bs, 8, 8)
    toks = list(range(18))                      # 5 blocks, the last partial
    r = m.begin()
    m.reserve(r, len(toks))
    m.publish(r, toks)                          # blocks 0..3 published
    m.expire(r, 9)                              # window starts at token 9: blocks 0, 1 expire
    assert m.table(r) == [-1, -1, 2, 3, 4]
    assert m.lru == [0, 1] and m.refcount[0] == 0
    s = m.begin()                               # the expired blocks still serve as a prefix
    assert m.find_cached_prefix(s, toks[:8]) == 8 and m.table(s) == [0, 1]
    m.release(r)
    assert m.lru == [2, 3] and 4 in m.free


def test_lru_eviction_order():
    bs = 1
    m = AllocatorModel(bs, 3, 3)
    for tok in (10, 20, 30):            # three single-block prompts, released in order
        r = m.begin()
        m.reserve(r, 1)
        m.publish(r, [tok])
        m.release(r)
    assert m.lru == [0, 1, 2] and m.free == []
    r = m.begin()
    m.reserve(r, 2)                     # no room to grow: evict the two oldest
    assert m.table(r) == [0, 1] and m.lru == [2]
    s = m.begin()
    assert m.find_cached_prefix(s, [10]) == 0 and m.find_cached_prefix(m.begin(), [30]) == 1


# ---------------------------------------------------------------------------
# the library's allocator against the model
# ---------------------------------------------------------------------------
def _invariants(m: AllocatorModel):
    held = {}
    for t in m.tables.values():
        for b in t:
            if b >= 0:
                held[b] = held.get(b, 0) + 1
    for b in range(m.num_blocks):
        assert m.refcount[b] == held.get(b, 0)
    states = [set(m.free), set(m.lru), set(held)]
    assert sum(len(x) for x in states) == m.num_blocks
    assert set().union(*states) == set(range(m.num_blocks))
    assert set(m.lru) <= set(m.hash_of_block)


@pytest.mark.parametrize("seed", range(12))
def test_library_matches_model_on_random_lifecycles(pkv, seed):
    bs = [1, 4, 16][seed % 3]
    init, maxb = [(8, 64), (32, 32), (0, 40), (16, 200)][seed % 4]
    rng = np.random.default_rng(seed)
    prompts = [list(rng.integers(0, 5, size=int(rng.integers(1, 6)) * bs)) for _ in range(5)]
    m = AllocatorModel(bs, init, maxb)
    a = pkv.BlockAllocator(bs, init, maxb)
    live = {}   # model request id -> (library request id, tokens so far)
    for step in range(300):
        op = rng.integers(0, 4)
        if op == 0 or not live:
            toks = list(prompts[rng.integers(0, len(prompts))]) + \
                list(rng.integers(0, 5, size=int(rng.integers(0, 2 * bs + 1))))
            keys = None
            if rng.integers(0, 4) == 0:
                keys = [int(x) for x in rng.integers(0, 3, size=len(toks) // bs)]
            r, q = m.begin(), a.begin()
            assert m.find_cached_prefix(r, toks, keys) == a.find_cached_prefix(q, toks, keys)
            err_m = err_a = None
            try:
                m.reserve(r, len(toks))
            except OutOfBlocks:
                err_m = True
            try:
                a.reserve(q, len(toks))
            except pkv.PkvError as e:
                err_a = e.code == pkv.PKV_ERR_OUT_OF_BLOCKS
            assert err_m == err_a
            if err_m:
                m.release(r)
                a.release(q)
            else:
                m.publish(r, toks, keys)
                a.publish(q, toks, keys)
                live[r] = (q, toks)
        elif op == 1:
            # decode a few tokens into a live request, publishing full blocks
            r = list(live)[rng.integers(0, len(live))]
            q, toks = live[r]
            toks = toks + list(rng.integers(0, 5, size=int(rng.integers(1, bs + 2))))
            try:
                m.reserve(r, len(toks))
                ok_m = True
            except OutOfBlocks:
                ok_m = False
            try:
                a.reserve(q, len(toks))
                ok_a = True
            except pkv.PkvError as e:
                assert e.code == pkv.PKV_ERR_OUT_OF_BLOCKS
                ok_a = False
            assert ok_m == ok_a
            if ok_m:
                m.publish(r, toks)
                a.publish(q, toks)
                live[r] = (q, toks)
        elif op == 2 and rng.integers(0, 2) == 0:
            # a sliding window moves: expire the blocks before it
            r = list(live)[rng.integers(0, len(live))]
            q, toks = live[r]
            first = int(rng.integers(0, len(toks) + 1))
            m.expire(r, first)
            a.expire(q, first)
        else:
            r = list(live)[rng.integers(0, len(live))]
            q, _ = live.pop(r)
            m.release(r)
            a.release(q)
        assert a.stats() == m.stats(), step
        for r, (q, _) in live.items():
            assert list(a.table(q)) == m.table(r)
        for b in range(m.num_blocks):
            assert a.refcount(b) == m.refcount[b]
        _invariants(m)


def test_allocator_tables_drive_the_slot_mapping(pkv, orc):
    # tables built by the allocator for rows sharing a prompt give the slots
    # the oracle's slot mapping gives for the same tables
    bs = 16
    a = pkv.BlockAllocator(bs, 64, 256)
    prompt = list(range(40))
    rows = []
    for i in range(4):
        r = a.begin()
        toks = prompt + [100 + i] * (5 + 7 * i)
        a.find_cached_prefix(r, toks)
        a.reserve(r, len(toks) + 1)
        a.publish(r, toks)
        rows.append((r, len(toks)))
    width = max(len(a.table(r)) for r, _ in rows)
    tables = np.full((len(rows), width), -1, dtype=np.int32)
    for i, (r, _) in enumerate(rows):
        t = a.table(r)
        tables[i, :len(t)] = t
    assert all((tables[i, :2] == tables[0, :2]).all() for i in range(4))   # 2 shared full blocks
    new_rows = np.arange(len(rows), dtype=np.int32)
    new_pos = np.array([n for _, n in rows], dtype=np.int32)
    nb = a.stats()[0]
    got = pkv.slot_mapping_host(tables, nb, new_rows, new_pos, bs)
    ref, bad = orc.slot_mapping(tables, nb, new_rows, new_pos, bs)
    assert bad == 0 and np.array_equal(got, ref)
