"""Reference model of the host block allocator (test infrastructure).

Only ``tests/`` imports this module.  It restates, with plain Python lists
and dicts, the block lifecycle the pages describe ("paged-cache.md": the
BlockAllocator row of the component table - per-block refcounts, LRU
eviction, a prefix-hash table for reuse across requests; the
PagedKVCacheAdapter per-request lifecycle find_cached_prefix ->
allocate_suffix_blocks -> record_tokens / register_full_blocks_for_reuse ->
release_request; the pool-sizing passage's grow rule), with the readings the
library's header states where the pages are silent:

- a full block's hash is FNV-1a (64-bit) over the little-endian bytes of the
  parent block's hash (0 for the first block), the block's token ids as int32
  and one 64-bit extra key; equal hashes are equal blocks;
- free blocks are handed out lowest id first;
- cache-only blocks (published, no request holds them) are evicted in the
  order they became cache-only;
- a reservation short of free blocks grows the pool once, before evicting,
  when free + cache-only blocks cannot cover it:
  new size = min(max, max(2 * current, current + shortfall of free blocks)).

Parity status: pinned by tests/test_allocator.py (FNV-1a published test
vectors, the grow rule's worked numbers, hand-traced lifecycles).
"""
from __future__ import annotations

import struct
from typing import Dict, List, Optional, Sequence

FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: for each byte, xor it in, then multiply by the prime
    (mod 2^64), starting from the offset basis."""
    h = FNV_OFFSET
    for b in data:
        h ^= b
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent: int, tokens: Sequence[int], extra: int = 0) -> int:
    data = struct.pack("<Q", parent) + b"".join(struct.pack("<i", int(t)) for t in tokens) \
        + struct.pack("<Q", extra)
    return fnv1a64(data)


class OutOfBlocks(Exception):
    pass


class AllocatorModel:
    def __init__(self, block_size: int, initial_blocks: int, max_blocks: int):
        assert block_size > 0 and 0 <= initial_blocks <= max_blocks
        self.bs = block_size
        self.max_blocks = max_blocks
        self.num_blocks = initial_blocks
        self.refcount: List[int] = [0] * initial_blocks
        self.block_of_hash: Dict[int, int] = {}
        self.hash_of_block: Dict[int, int] = {}
        self.free: List[int] = list(range(initial_blocks))  # kept sorted
        self.lru: List[int] = []  # cache-only blocks, oldest first
        self.grows = 0
        self.next_req = 0
        self.tables: Dict[int, List[int]] = {}
        self.chains: Dict[int, List[int]] = {}
        self.done: Dict[int, int] = {}  # leading blocks already published (or hit)
        self.fresh: Dict[int, bool] = {}

    # -- request lifecycle -------------------------------------------------
    def begin(self) -> int:
        r = self.next_req
        self.next_req += 1
        self.tables[r], self.chains[r], self.done[r], self.fresh[r] = [], [], 0, True
        return r

    def find_cached_prefix(self, r: int, tokens: Sequence[int],
                           extra_keys: Optional[Sequence[int]] = None) -> int:
        assert self.fresh[r]
        self.fresh[r] = False
        parent = 0
        for i in range(len(tokens) // self.bs):
            h = block_hash(parent, tokens[i * self.bs:(i + 1) * self.bs],
                           extra_keys[i] if extra_keys is not None else 0)
            if h not in self.block_of_hash:
                break
            b = self.block_of_hash[h]
            if b in self.lru:
                self.lru.remove(b)
            self.refcount[b] += 1
            self.tables[r].append(b)
            self.chains[r].append(h)
            parent = h
        self.done[r] = len(self.tables[r])
        return len(self.tables[r]) * self.bs

    def reserve(self, r: int, n_tokens: int) -> None:
        self.fresh[r] = False
        k = -(-n_tokens // self.bs) - len(self.tables[r])
        if k <= 0:
            return
        if k > len(self.free):
            if k > len(self.free) + len(self.lru) and self.num_blocks < self.max_blocks:
                want = max(2 * self.num_blocks, self.num_blocks + (k - len(self.free)))
                new = min(want, self.max_blocks)
                self.free = sorted(self.free + list(range(self.num_blocks, new)))
                self.refcount += [0] * (new - self.num_blocks)
                self.num_blocks = new
                self.grows += 1
            if k > len(self.free) + len(self.lru):
                raise OutOfBlocks()
            while len(self.free) < k:
                b = self.lru.pop(0)
                del self.block_of_hash[self.hash_of_block.pop(b)]
                self.free = sorted(self.free + [b])
        for _ in range(k):
            b = self.free.pop(0)
            self.refcount[b] = 1
            self.tables[r].append(b)

    def publish(self, r: int, tokens: Sequence[int],
                extra_keys: Optional[Sequence[int]] = None) -> None:
        nfull = len(tokens) // self.bs
        assert nfull <= len(self.tables[r])
        for i in range(self.done[r], nfull):
            parent = self.chains[r][i - 1] if i > 0 else 0
            h = block_hash(parent, tokens[i * self.bs:(i + 1) * self.bs],
                           extra_keys[i] if extra_keys is not None else 0)
            self.chains[r].append(h)
            b = self.tables[r][i]
            if b >= 0 and h not in self.block_of_hash:
                self.block_of_hash[h] = b
                self.hash_of_block[b] = h
        self.done[r] = max(self.done[r], nfull)

    def _drop(self, b: int) -> None:
        self.refcount[b] -= 1
        if self.refcount[b] > 0:
            return
        if b in self.hash_of_block:
            self.lru.append(b)
        else:
            self.free = sorted(self.free + [b])

    def expire(self, r: int, first_live_token: int) -> None:
        """A sliding window's expired blocks: those wholly before
        first_live_token leave the table (entry -1, the null sentinel)."""
        t = self.tables[r]
        for i in range(min(first_live_token // self.bs, len(t))):
            if t[i] >= 0:
                self._drop(t[i])
                t[i] = -1

    def release(self, r: int) -> None:
        for b in self.tables.pop(r):
            if b >= 0:
                self._drop(b)
        del self.chains[r], self.done[r], self.fresh[r]

    # -- views ---------------------------------------------------------------
    def table(self, r: int) -> List[int]:
        return list(self.tables[r])

    def stats(self):
        return self.num_blocks, len(self.free), len(self.lru), self.grows
