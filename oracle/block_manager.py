"""Plain Python model of the host KV block manager (TEST INFRASTRUCTURE ONLY).

Written from the pages, step by step, with Python lists and dicts; the tests
run the same operation sequences through it and through the C++ manager in
``libpa.so`` and compare every observable result.  It shares no code with the
C++ manager; the hash (64-bit FNV-1a) and the shuffle (splitmix64 driving a
Fisher-Yates pass) are each implemented here from their published definitions.

Sources (page title, section):
  "vLLM 核心工程深度剖析" - "2.2 显存分配器实现": a free list and reference counts;
      allocate takes blocks and sets ref 1; append_slot adds a block when the
      last one is full; free decrements and returns blocks reaching 0.
      "4.1 Beam Search 中的 CoW": fork copies the parent's table, ref += 1 each.
  "PagedAttention 笔记" - "写时复制是正确性的边界": writing into a shared block:
      allocate a new block, copy, remap, ref_count of the old block -1, write.
  "PagedAttention是什麼？" - "vLLM v1的Block Pool", "Eviction與Free Queue": new
      blocks from the head of the free queue, freed blocks to its tail; a freed
      block keeps its hash until the queue hands it out again.
  "PagedAttention 详解：缓存的存储结构" - "使用流程": full prompt blocks get a chained
      hash h_i = hash(tokens_i, h_{i-1}); a hit reuses the cached block, a miss
      allocates a new one.
"""
from __future__ import annotations

import struct

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1

OK, ERR_INVALID, ERR_UNKNOWN, ERR_NO_BLOCKS, ERR_EXISTS = 0, -1, -2, -3, -4


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """FNV-1a, 64-bit: for each byte, h ^= byte; h *= prime (mod 2^64)."""
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def chain_hash(parent: int, tokens) -> int:
    """Hash of one full block given its parent's hash (0 for the first block)."""
    return fnv1a64(struct.pack("<Q", parent) + struct.pack(f"<{len(tokens)}i", *tokens))


class SplitMix64:
    """splitmix64 (Steele, Lea, Flood 2014)."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, shuffle_seed: int = 0):
        self.B = block_size
        self.num_blocks = num_blocks
        order = list(range(num_blocks))
        if shuffle_seed:
            rng = SplitMix64(shuffle_seed)
            for i in range(num_blocks - 1, 0, -1):  # Fisher-Yates from the top
                j = rng.next() % (i + 1)
                order[i], order[j] = order[j], order[i]
        self.free_queue = order              # head = index 0
        self.ref = [0] * num_blocks
        self.cache = {}                      # hash -> block
        self.cached_info = {}                # block -> (hash, parent hash, tokens)
        self.tables = {}                     # seq -> list of blocks
        self.lens = {}                       # seq -> tokens

    # -- free queue
    def _take(self) -> int:
        b = self.free_queue.pop(0)
        if b in self.cached_info:            # handed out again: its cache entry goes
            h = self.cached_info.pop(b)[0]
            if self.cache.get(h) == b:
                del self.cache[h]
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free_queue.append(b)

    def num_free(self) -> int:
        return len(self.free_queue)

    # -- operations
    def allocate(self, seq, num_tokens: int) -> int:
        if num_tokens < 0:
            return ERR_INVALID
        if seq in self.tables:
            return ERR_EXISTS
        need = -(-num_tokens // self.B)
        if need > len(self.free_queue):
            return ERR_NO_BLOCKS
        self.tables[seq] = [self._take() for _ in range(need)]
        self.lens[seq] = num_tokens
        return OK

    def allocate_with_prefix(self, seq, tokens):
        """Returns (status, number of leading blocks served from the cache)."""
        if seq in self.tables:
            return ERR_EXISTS, 0
        n = len(tokens)
        full, need = n // self.B, -(-n // self.B)
        hashes, hits = [], []
        parent, chain = 0, True
        for i in range(full):
            blk_tokens = list(tokens[i * self.B:(i + 1) * self.B])
            h = chain_hash(parent, blk_tokens)
            hashes.append(h)
            if chain:
                b = self.cache.get(h)
                if b is not None and self.cached_info[b][1] == parent and self.cached_info[b][2] == blk_tokens:
                    hits.append(b)
                else:
                    chain = False
            parent = h
        queued_hits = sum(1 for b in hits if b in self.free_queue)
        if need - len(hits) > len(self.free_queue) - queued_hits:
            return ERR_NO_BLOCKS, 0
        table = []
        for b in hits:
            if b in self.free_queue:
                self.free_queue.remove(b)
            self.ref[b] += 1
            table.append(b)
        for i in range(len(hits), need):
            b = self._take()
            table.append(b)
            if i < full and hashes[i] not in self.cache:
                self.cache[hashes[i]] = b
                self.cached_info[b] = (hashes[i], hashes[i - 1] if i else 0, list(tokens[i * self.B:(i + 1) * self.B]))
        self.tables[seq] = table
        self.lens[seq] = n
        return OK, len(hits)

    def append_slot(self, seq):
        """Returns (status, slot, cow_src, cow_dst)."""
        if seq not in self.tables:
            return ERR_UNKNOWN, -1, -1, -1
        table, n = self.tables[seq], self.lens[seq]
        off = n % self.B
        src = dst = -1
        if off == 0:                                  # last block full (or none): a new block
            if not self.free_queue:
                return ERR_NO_BLOCKS, -1, -1, -1
            table.append(self._take())
        elif self.ref[table[-1]] > 1:                 # shared partial block: copy-on-write
            if not self.free_queue:
                return ERR_NO_BLOCKS, -1, -1, -1
            src = table[-1]
            dst = self._take()
            table[-1] = dst
            self._release(src)
        self.lens[seq] = n + 1
        return OK, table[-1] * self.B + off, src, dst

    def fork(self, parent, child) -> int:
        if parent not in self.tables:
            return ERR_UNKNOWN
        if child in self.tables:
            return ERR_EXISTS
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1
        return OK

    def free(self, seq) -> int:
        if seq not in self.tables:
            return ERR_UNKNOWN
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lens[seq]
        return OK
