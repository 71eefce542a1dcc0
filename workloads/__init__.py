"""Seeded synthetic inputs for paged decode attention and its write kernels.

This module only *builds inputs*: random values, block-ID assignment through a
small host allocator (free list, reference counts, fork, copy-on-write remap)
and the slot_mapping / block_tables / seq_lens metadata a serving scheduler
would hand to the kernels.  It holds none of the attention arithmetic and none
of the kernels' address decoding.  Both the CUDA path (through the tests and
the benchmark) and the CPU oracle consume the same arrays it returns; neither
of them is imported here.

Every array is produced by numpy's PCG64 generator from an explicit seed.
Storage conventions: 'f32' -> float32, 'f16' -> float16, 'bf16' -> uint16
holding bfloat16 bit patterns (round-to-nearest-even from float32).
Cache layout: [num_blocks][num_kv_heads][block_size][head_size], dense.

Host-side bookkeeping follows "vLLM 核心工程深度剖析" section "2.2 显存分配器实现"
(free list + reference counts, allocate / append_slot / free) and section
"4.1 Beam Search 中的 CoW" (fork shares the parent's blocks, ref += 1), and
"PagedAttention 笔记" section "写时复制是正确性的边界" (allocate a new block, copy,
remap, ref -= 1, then write).  slot = block_id * block_size + offset follows
"PagedAttention 详解：缓存的存储结构" section "写入新 K/V".
"""
from __future__ import annotations

import dataclasses
import math
from collections import deque

import numpy as np

NP_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
# quiet-NaN fill for unused slots and unreferenced blocks in every workload
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> storage array of ``dtype`` (bf16: RNE on the bit pattern)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    u = x.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def nan_array(shape, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.full(shape, np.nan, dtype=np.float32)
    if dtype == "f16":
        return np.full(shape, NAN_BITS["f16"], dtype=np.uint16).view(np.float16)
    return np.full(shape, NAN_BITS["bf16"], dtype=np.uint16)


def normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return to_storage(rng.standard_normal(shape, dtype=np.float32), dtype)


class OutOfBlocks(RuntimeError):
    pass


class BlockAllocator:
    """Host block pool: FIFO free list over a seeded permutation of block IDs,
    reference counts, per-sequence block tables."""

    def __init__(self, num_blocks: int, block_size: int, rng: np.random.Generator | None = None,
                 shuffle: bool = True):
        self.num_blocks = num_blocks
        self.block_size = block_size
        ids = rng.permutation(num_blocks) if (shuffle and rng is not None) else np.arange(num_blocks)
        self.free_list = deque(int(b) for b in ids)
        self.ref_count = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    def num_free(self) -> int:
        return len(self.free_list)

    def _take(self) -> int:
        if not self.free_list:
            raise OutOfBlocks("KV block pool exhausted")
        b = self.free_list.popleft()
        self.ref_count[b] += 1
        return b

    def allocate(self, seq: int, num_tokens: int, fixed: list[int] | None = None) -> list[int]:
        """New sequence holding ``num_tokens`` tokens.  ``fixed`` pins the block IDs."""
        need = -(-num_tokens // self.block_size)
        if fixed is not None:
            if len(fixed) != need:
                raise ValueError("fixed block list has the wrong length")
            for b in fixed:
                self.free_list.remove(b)
                self.ref_count[b] += 1
            blocks = list(fixed)
        else:
            if need > len(self.free_list):
                raise OutOfBlocks("KV block pool exhausted")
            blocks = [self._take() for _ in range(need)]
        self.tables[seq] = blocks
        self.lens[seq] = num_tokens
        return blocks

    def append_slot(self, seq: int) -> int:
        """Room for one more token; returns its slot (block * B + offset)."""
        pos = self.lens[seq]
        blocks = self.tables[seq]
        if pos // self.block_size >= len(blocks):
            blocks.append(self._take())
        self.lens[seq] = pos + 1
        return blocks[pos // self.block_size] * self.block_size + pos % self.block_size

    def fork(self, parent: int, child: int) -> None:
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref_count[b] += 1

    def cow(self, seq: int, logical: int) -> tuple[int, int]:
        """Give ``seq`` a private copy of its logical block; returns the (src, dst) pair to copy."""
        src = self.tables[seq][logical]
        dst = self._take()
        self.tables[seq][logical] = dst
        self._release(src)
        return src, dst

    def _release(self, b: int) -> None:
        self.ref_count[b] -= 1
        if self.ref_count[b] < 0:
            raise RuntimeError(f"reference count of block {b} went negative")
        if self.ref_count[b] == 0:
            self.free_list.append(b)  # FIFO: a freed block is reused last

    def free(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self._release(b)
        self.lens.pop(seq)

    def table_array(self, seqs: list[int], width: int | None = None) -> np.ndarray:
        width = width if width is not None else max((len(self.tables[s]) for s in seqs), default=0)
        width = max(width, 1)
        out = np.zeros((len(seqs), width), dtype=np.int32)
        for i, s in enumerate(seqs):
            t = self.tables[s]
            out[i, :len(t)] = t
        return out


@dataclasses.dataclass
class Workload:
    """One decode step: optional block copies, then optional appends, then attention."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    scale: float
    q: np.ndarray                      # [N, Hq, D]
    k_cache: np.ndarray | None         # [num_blocks, Hkv, B, D], state before the step's writes
    v_cache: np.ndarray | None         # (None when only the metadata was built)
    block_tables: np.ndarray           # int32 [N, M]
    seq_lens: np.ndarray               # int32 [N]
    copy_pairs: np.ndarray | None = None     # int32 [n, 2] (src, dst)
    slot_mapping: np.ndarray | None = None   # int64 [T]
    new_key: np.ndarray | None = None        # [T, Hkv, D]
    new_value: np.ndarray | None = None
    partition_size: int = 0
    info: dict = dataclasses.field(default_factory=dict)
    query_start: np.ndarray | None = None     # prefill: int32 [N + 1] chunk offsets into q

    @property
    def num_seqs(self) -> int:
        return int(len(self.seq_lens))

    @property
    def num_query_tokens(self) -> int:
        return int(self.q.shape[0])

    def prefill_flops(self) -> int:
        """Algorithmic FLOPs of prefill attention: query j of a chunk of n at the
        end of L cached tokens sees L - n + j + 1 keys, and each key costs 2 D
        (q . k) + 2 D (p v) per query head: 4 D Hq (n L - n (n - 1) / 2) per sequence."""
        n = np.diff(self.query_start.astype(np.int64))
        L = self.seq_lens.astype(np.int64)
        keys = n * L - n * (n - 1) // 2
        return int(4 * self.head_size * self.num_q_heads * keys.sum())

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def cache_elem_bytes(self) -> int:
        """Bytes per cache element: 1 for an FP8 cache, else those of the dtype."""
        return 1 if self.info.get("kv_dtype") == "fp8" else ELEM_BYTES[self.dtype]

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one attention call reads (each token once per KV head)."""
        return int(self.seq_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_size * self.cache_elem_bytes

    def unique_kv_bytes(self) -> int:
        """K+V bytes of distinct (block, slot) pairs read: shared prefix blocks count once."""
        seen = set()
        for s in range(self.num_seqs):
            L = int(self.seq_lens[s])
            nb = -(-L // self.block_size)
            for j in range(nb):
                used = min(self.block_size, L - j * self.block_size)
                b = int(self.block_tables[s, j])
                seen.update((b, o) for o in range(used))
        return len(seen) * 2 * self.num_kv_heads * self.head_size * ELEM_BYTES[self.dtype]

    def step_bytes(self) -> int:
        """Algorithmic HBM bytes of the whole step: copies + appends + attention."""
        eb = ELEM_BYTES[self.dtype]
        total = self.kv_bytes()
        total += 2 * self.num_query_tokens * self.num_q_heads * self.head_size * eb  # q in, out
        total += int(np.sum(-(-self.seq_lens.astype(np.int64) // self.block_size))) * 4  # table reads
        if self.copy_pairs is not None:
            total += len(self.copy_pairs) * 2 * 2 * self.num_kv_heads * self.block_size * self.head_size * eb
        if self.slot_mapping is not None:
            total += int(np.sum(self.slot_mapping >= 0)) * 2 * 2 * self.num_kv_heads * self.head_size * eb
            total += len(self.slot_mapping) * 8
        return total


def _fill_tokens(k_cache, v_cache, rng, alloc: BlockAllocator, seq: int, t0: int, t1: int, dtype: str):
    """Random N(0,1) keys/values for tokens [t0, t1) of ``seq``."""
    if t1 <= t0:
        return
    B = alloc.block_size
    pos = np.arange(t0, t1)
    blocks = np.asarray(alloc.tables[seq], dtype=np.int64)[pos // B]
    offs = pos % B
    Hkv, D = k_cache.shape[1], k_cache.shape[3]
    k_cache[blocks, :, offs, :] = normal(rng, (len(pos), Hkv, D), dtype)
    v_cache[blocks, :, offs, :] = normal(rng, (len(pos), Hkv, D), dtype)


def build_decode(name: str, *, seed: int, dtype: str, seq_lens, num_q_heads: int, num_kv_heads: int,
                 head_size: int, block_size: int, num_blocks: int | None = None, pool_factor: float = 1.2,
                 append_last: bool = False, fixed_tables: dict | None = None, shuffle: bool = True,
                 table_width: int | None = None, partition_size: int = 0, materialize: bool = True) -> Workload:
    """Independent sequences.  With ``append_last`` the last token of every sequence
    is written by the step's reshape_and_cache (its slot starts out as NaN).
    ``materialize=False`` skips the host caches (k_cache = v_cache = None): the
    metadata, q and the new tokens are still built; see ``device_caches``."""
    rng = np.random.default_rng(seed)
    seq_lens = [int(x) for x in seq_lens]
    need = sum(-(-L // block_size) for L in seq_lens)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * need))
    alloc = BlockAllocator(num_blocks, block_size, rng, shuffle=shuffle)
    fixed_tables = fixed_tables or {}
    for s, L in enumerate(seq_lens):
        alloc.allocate(s, L - 1 if (append_last and L > 0) else L, fixed=fixed_tables.get(s))
    shape = (num_blocks, num_kv_heads, block_size, head_size)
    k_cache = v_cache = None
    if materialize:
        k_cache, v_cache = nan_array(shape, dtype), nan_array(shape, dtype)
        for s in range(len(seq_lens)):
            _fill_tokens(k_cache, v_cache, rng, alloc, s, 0, alloc.lens[s], dtype)
    slot_mapping = new_key = new_value = None
    if append_last:
        slots = []
        for s, L in enumerate(seq_lens):
            slots.append(alloc.append_slot(s) if L > 0 else -1)
        slot_mapping = np.asarray(slots, dtype=np.int64)
        new_key = normal(rng, (len(seq_lens), num_kv_heads, head_size), dtype)
        new_value = normal(rng, (len(seq_lens), num_kv_heads, head_size), dtype)
    q = normal(rng, (len(seq_lens), num_q_heads, head_size), dtype)
    width = table_width if table_width is not None else max(1, max(-(-L // block_size) for L in seq_lens))
    tables = alloc.table_array(list(range(len(seq_lens))), width)
    return Workload(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_size=head_size, block_size=block_size, num_blocks=num_blocks,
                    scale=1.0 / math.sqrt(head_size), q=q, k_cache=k_cache, v_cache=v_cache,
                    block_tables=tables, seq_lens=np.asarray(seq_lens, dtype=np.int32),
                    slot_mapping=slot_mapping, new_key=new_key, new_value=new_value,
                    partition_size=partition_size, info={"seed": seed, "append_last": append_last})


# ---------------------------------------------------------------------------
# The five workloads.  Seeds are 1000 + workload index.
# ---------------------------------------------------------------------------

def tiny_f32() -> Workload:
    """4 seqs, lens {1, 15, 16, 35}, 4 q heads = 4 kv heads, head_size 64, B = 16,
    pool of 32 blocks.  The 35-token sequence uses the table [7, 3, 12]; the others
    take block IDs from a seeded permutation of the remaining IDs."""
    lens = [1, 15, 16, 35]
    rng = np.random.default_rng(1000)
    rest = [int(b) for b in rng.permutation(32) if b not in (3, 7, 12)]
    fixed = {0: [rest[0]], 1: [rest[1]], 2: [rest[2]], 3: [7, 3, 12]}
    return build_decode("tiny_f32", seed=1000, dtype="f32", seq_lens=lens, num_q_heads=4, num_kv_heads=4,
                        head_size=64, block_size=16, num_blocks=32, fixed_tables=fixed)


def mha_f16(num_seqs: int = 64, max_len: int = 2048, min_len: int = 128, num_heads: int = 32,
            num_blocks: int = 8192, materialize: bool = True) -> Workload:
    """MHA fp16: lens uniform in [128, 2048], 32 heads, D = 128, B = 16, pool of 8192
    shuffled blocks; the step appends one token per sequence, then attends over it."""
    rng = np.random.default_rng(1001)
    lens = rng.integers(min_len, max_len, size=num_seqs, endpoint=True)
    w = build_decode("mha_f16", seed=1001, dtype="f16", seq_lens=lens, num_q_heads=num_heads,
                     num_kv_heads=num_heads, head_size=128, block_size=16, num_blocks=num_blocks,
                     append_last=True, materialize=materialize)
    return w


def gqa_lens(num_seqs: int, rng: np.random.Generator, median: float = 1200.0, sigma: float = 0.6,
             lo: int = 64, hi: int = 4096) -> np.ndarray:
    return np.clip(np.rint(rng.lognormal(math.log(median), sigma, size=num_seqs)), lo, hi).astype(np.int64)


def gqa_bf16(num_seqs: int = 128, hi: int = 4096, materialize: bool = True) -> Workload:
    """GQA bf16: 128 seqs, 64 q heads / 8 kv heads, D = 128, B = 32, lens
    lognormal(ln 1200, 0.6) clamped to [64, 4096]; pool = 1.2x the blocks needed."""
    rng = np.random.default_rng(1002)
    lens = gqa_lens(num_seqs, rng, hi=hi)
    return build_decode("gqa_bf16", seed=1002, dtype="bf16", seq_lens=lens, num_q_heads=64, num_kv_heads=8,
                        head_size=128, block_size=32, pool_factor=1.2, materialize=materialize)


def shared_prefix_f16(num_prompts: int = 16, branches: int = 8, prefix_len: int = 1024,
                      max_suffix: int = 256, num_heads: int = 32, block_size: int = 16,
                      num_blocks: int = 4096, seed: int = 1003, materialize: bool = True) -> Workload:
    """Parallel sampling: each prompt's prefix blocks are shared by its branches
    (ref_count = branches).  Before appending its suffix, each branch takes a
    private copy of the last shared block (one (src, dst) copy pair per branch),
    remaps its table and drops its reference; then its suffix tokens are written
    through slot_mapping and attention runs over prefix + suffix."""
    rng = np.random.default_rng(seed)
    D = 128
    alloc = BlockAllocator(num_blocks, block_size, rng)
    shape = (num_blocks, num_heads, block_size, D)
    k_cache = v_cache = None
    if materialize:
        k_cache, v_cache = nan_array(shape, "f16"), nan_array(shape, "f16")
    seqs, pairs, slots = [], [], []
    last_logical = (prefix_len - 1) // block_size
    suffix_lens = rng.integers(1, max_suffix, size=num_prompts * branches, endpoint=True)
    for p in range(num_prompts):
        root = 10_000 + p
        alloc.allocate(root, prefix_len)
        if materialize:
            _fill_tokens(k_cache, v_cache, rng, alloc, root, 0, prefix_len, "f16")
        for b in range(branches):
            alloc.fork(root, len(seqs) + 0)
            seqs.append(len(seqs))
        alloc.free(root)  # the prompt itself no longer holds the blocks
    for s in seqs:
        pairs.append(alloc.cow(s, last_logical))
    for s in seqs:
        for _ in range(int(suffix_lens[s])):
            slots.append(alloc.append_slot(s))
    # freed copy sources must not have been handed out again within this step
    srcs = {a for a, _ in pairs}
    for s in seqs:
        assert not srcs.intersection(alloc.tables[s]), "copy source reused in the same step"
    T = len(slots)
    new_key = normal(rng, (T, num_heads, D), "f16")
    new_value = normal(rng, (T, num_heads, D), "f16")
    q = normal(rng, (len(seqs), num_heads, D), "f16")
    lens = np.asarray([alloc.lens[s] for s in seqs], dtype=np.int32)
    tables = alloc.table_array(seqs)
    w = Workload(name="shared_prefix_f16", dtype="f16", num_q_heads=num_heads, num_kv_heads=num_heads,
                 head_size=D, block_size=block_size, num_blocks=num_blocks, scale=1.0 / math.sqrt(D), q=q,
                 k_cache=k_cache, v_cache=v_cache, block_tables=tables, seq_lens=lens,
                 copy_pairs=np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
                 slot_mapping=np.asarray(slots, dtype=np.int64), new_key=new_key, new_value=new_value,
                 info={"seed": seed, "prefix_len": prefix_len, "branches": branches,
                       "ref_counts_after": {int(b): alloc.ref_count[int(b)] for b in set(tables.reshape(-1))}})
    return w


def long_bf16(block_size: int = 16, num_seqs: int = 8, seq_len: int = 32768, partition_size: int = 512,
              materialize: bool = True) -> Workload:
    """Long context: 8 seqs of 32768 tokens, 32 q heads / 8 kv heads, D = 128, block
    size swept over {16, 32, 64}, pool exactly the blocks needed (shuffled), split
    into 512-token partitions merged by log-sum-exp."""
    nb = num_seqs * (-(-seq_len // block_size))
    return build_decode(f"long_bf16_b{block_size}", seed=1004, dtype="bf16", seq_lens=[seq_len] * num_seqs,
                        num_q_heads=32, num_kv_heads=8, head_size=128, block_size=block_size, num_blocks=nb,
                        partition_size=partition_size, materialize=materialize)


def build_prefill(name: str, *, seed: int, dtype: str, prefix_lens, chunk_lens, num_q_heads: int, num_kv_heads: int,
                  head_size: int, block_size: int, pool_factor: float = 1.2, materialize: bool = True) -> Workload:
    """Chunked prefill: sequence s already holds prefix_lens[s] tokens in the cache
    and this step appends chunk_lens[s] new tokens (their K/V written through
    slot_mapping, slots start as NaN), then runs prefill attention for the chunk's
    queries over the whole context.  q is packed [sum chunk_lens, Hq, D]."""
    rng = np.random.default_rng(seed)
    prefix_lens = [int(x) for x in prefix_lens]
    chunk_lens = [int(x) for x in chunk_lens]
    totals = [a + b for a, b in zip(prefix_lens, chunk_lens)]
    need = sum(-(-L // block_size) for L in totals)
    num_blocks = max(1, math.ceil(pool_factor * need))
    alloc = BlockAllocator(num_blocks, block_size, rng)
    for s, P in enumerate(prefix_lens):
        alloc.allocate(s, P)
    shape = (num_blocks, num_kv_heads, block_size, head_size)
    k_cache = v_cache = None
    if materialize:
        k_cache, v_cache = nan_array(shape, dtype), nan_array(shape, dtype)
        for s, P in enumerate(prefix_lens):
            _fill_tokens(k_cache, v_cache, rng, alloc, s, 0, P, dtype)
    slots = []
    for s, n in enumerate(chunk_lens):  # the chunk's slots: block * B + offset, in token order
        start = alloc.lens[s]
        need_blocks = -(-(start + n) // block_size) - len(alloc.tables[s])
        for _ in range(need_blocks):
            alloc.tables[s].append(alloc._take())
        alloc.lens[s] = start + n
        pos = np.arange(start, start + n)
        blocks = np.asarray(alloc.tables[s], dtype=np.int64)[pos // block_size]
        slots.extend((blocks * block_size + pos % block_size).tolist())
    T = len(slots)
    new_key = new_value = q = None
    if materialize:
        new_key = normal(rng, (T, num_kv_heads, head_size), dtype)
        new_value = normal(rng, (T, num_kv_heads, head_size), dtype)
        q = normal(rng, (T, num_q_heads, head_size), dtype)
    else:  # shapes only; the benchmark draws these on the device
        q = np.empty((T, num_q_heads, head_size), NP_STORAGE[dtype])
    tables = alloc.table_array(list(range(len(totals))))
    return Workload(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_size=head_size,
                    block_size=block_size, num_blocks=num_blocks, scale=1.0 / math.sqrt(head_size), q=q,
                    k_cache=k_cache, v_cache=v_cache, block_tables=tables,
                    seq_lens=np.asarray(totals, dtype=np.int32), slot_mapping=np.asarray(slots, dtype=np.int64),
                    new_key=new_key, new_value=new_value, info={"seed": seed, "prefix_lens": prefix_lens},
                    query_start=np.concatenate([[0], np.cumsum(chunk_lens)]).astype(np.int32))


def mha_fp8(num_seqs: int = 64, max_len: int = 2048, min_len: int = 128, num_heads: int = 32,
            num_blocks: int = 8192, materialize: bool = True) -> Workload:
    """The MHA fp16 decode step over an FP8 (E4M3) cache: lens uniform in [128, 2048],
    32 heads, D = 128, B = 16, pool of 8192 shuffled blocks, one appended token per
    sequence.  Host arrays are fp16 (q, new K/V and the pools before quantisation);
    the cache holds E4M3 codes of x / scale with the scales in ``info`` (about
    max|x| / 448 for N(0,1) pools of this size)."""
    rng = np.random.default_rng(1006)
    lens = rng.integers(min_len, max_len, size=num_seqs, endpoint=True)
    w = build_decode("mha_fp8", seed=1006, dtype="f16", seq_lens=lens, num_q_heads=num_heads,
                     num_kv_heads=num_heads, head_size=128, block_size=16, num_blocks=num_blocks,
                     append_last=True, materialize=materialize)
    w.info.update(kv_dtype="fp8", k_scale=0.0123, v_scale=0.0117)
    return w


def gqa_fp8(num_seqs: int = 128, hi: int = 4096, materialize: bool = True) -> Workload:
    """The GQA decode shapes (128 seqs, 64 q / 8 kv heads, D = 128, B = 32, lognormal
    lens) over an FP8 (E4M3) cache with fp16 queries; scales in ``info``."""
    rng = np.random.default_rng(1007)
    lens = gqa_lens(num_seqs, rng, hi=hi)
    w = build_decode("gqa_fp8", seed=1007, dtype="f16", seq_lens=lens, num_q_heads=64, num_kv_heads=8,
                     head_size=128, block_size=32, pool_factor=1.2, materialize=materialize)
    w.info.update(kv_dtype="fp8", k_scale=0.0123, v_scale=0.0117)
    return w


def prefill_bf16(num_seqs: int = 16, materialize: bool = True, max_prefix: int = 2048, min_chunk: int = 256,
                 max_chunk: int = 2048) -> Workload:
    """Chunked prefill, bf16: 16 sequences, cached prefix U[0, 2048] tokens, new
    chunk U[256, 2048] tokens, 32 q / 8 kv heads, D = 128, B = 16."""
    rng = np.random.default_rng(1005)
    prefix = rng.integers(0, max_prefix, size=num_seqs, endpoint=True)
    chunk = rng.integers(min_chunk, max_chunk, size=num_seqs, endpoint=True)
    return build_prefill("prefill_bf16", seed=1005, dtype="bf16", prefix_lens=prefix, chunk_lens=chunk, num_q_heads=32,
                         num_kv_heads=8, head_size=128, block_size=16, materialize=materialize)


def prefill_f16(num_seqs: int = 16, materialize: bool = True) -> Workload:
    """The prefill_bf16 shapes (same prefix and chunk lengths) in fp16, where P enters the value
    MMA as one fp16 term instead of two bf16 terms."""
    rng = np.random.default_rng(1005)
    prefix = rng.integers(0, 2048, size=num_seqs, endpoint=True)
    chunk = rng.integers(256, 2048, size=num_seqs, endpoint=True)
    return build_prefill("prefill_f16", seed=1008, dtype="f16", prefix_lens=prefix, chunk_lens=chunk, num_q_heads=32,
                         num_kv_heads=8, head_size=128, block_size=16, materialize=materialize)


WORKLOADS = {
    "tiny_f32": lambda materialize=True: tiny_f32(),
    "mha_f16": mha_f16,
    "gqa_bf16": gqa_bf16,
    "shared_prefix_f16": shared_prefix_f16,
    "long_bf16_b16": lambda materialize=True: long_bf16(16, materialize=materialize),
    "long_bf16_b32": lambda materialize=True: long_bf16(32, materialize=materialize),
    "long_bf16_b64": lambda materialize=True: long_bf16(64, materialize=materialize),
    "prefill_bf16": prefill_bf16,
    "prefill_f16": prefill_f16,
    "mha_fp8": mha_fp8,
    "gqa_fp8": gqa_fp8,
}


def device_caches(w: Workload, device, seed: int | None = None):
    """K and V pools generated on the device with torch's seeded generator: every
    slot N(0, 1) in the workload dtype (used for timing, where unused slots need no
    poison and host generation of gigabyte pools would dominate the run)."""
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.info.get("seed", 0) if seed is None else seed))
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_size)
    out = []
    for _ in range(2):
        t = torch.empty(shape, dtype=tdt, device=device)
        flat = t.view(-1)
        step = 1 << 26
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(tdt)
        out.append(t)
    return out[0], out[1]


def host_sample(w: Workload, seqs, seed: int = 7) -> Workload:
    """The sub-workload of sequences ``seqs`` with a compact host pool holding only
    their blocks (freshly drawn N(0,1) values; copy pairs and appends restricted to
    those sequences).  Used to time the CPU evaluation on a bounded sample."""
    rng = np.random.default_rng(seed)
    seqs = [int(s) for s in seqs]
    B = w.block_size
    used = []
    for s in seqs:
        used.extend(int(b) for b in w.block_tables[s, :-(-int(w.seq_lens[s]) // B)])
    srcs = []
    if w.copy_pairs is not None:
        used_set = set(used)
        srcs = [int(a) for a, b in w.copy_pairs if int(b) in used_set]
        used.extend(srcs)
    ids = sorted(set(used))
    remap = {b: i for i, b in enumerate(ids)}
    shape = (max(1, len(ids)), w.num_kv_heads, B, w.head_size)
    k = normal(rng, shape, w.dtype)
    v = normal(rng, shape, w.dtype)
    tables = np.zeros((len(seqs), w.max_blocks_per_seq), np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(w.seq_lens[s]) // B)
        tables[i, :n] = [remap[int(b)] for b in w.block_tables[s, :n]]
    pairs = None
    if w.copy_pairs is not None:
        pairs = np.asarray([(remap[int(a)], remap[int(b)]) for a, b in w.copy_pairs if int(b) in remap and
                            int(a) in remap], np.int32).reshape(-1, 2)
    slots = nk = nv = None
    if w.slot_mapping is not None:
        keep = [t for t, sl in enumerate(w.slot_mapping) if sl >= 0 and int(sl) // B in remap]
        slots = np.asarray([remap[int(w.slot_mapping[t]) // B] * B + int(w.slot_mapping[t]) % B for t in keep],
                           np.int64)
        nk, nv = w.new_key[keep], w.new_value[keep]
    return Workload(name=w.name + "_sample", dtype=w.dtype, num_q_heads=w.num_q_heads,
                    num_kv_heads=w.num_kv_heads, head_size=w.head_size, block_size=B, num_blocks=shape[0],
                    scale=w.scale, q=w.q[seqs], k_cache=k, v_cache=v, block_tables=tables,
                    seq_lens=w.seq_lens[seqs].copy(), copy_pairs=pairs, slot_mapping=slots, new_key=nk,
                    new_value=nv, partition_size=w.partition_size, info=dict(w.info))


def apply_writes_host(w: Workload, k_cache: np.ndarray, v_cache: np.ndarray, copy_fn, append_fn) -> None:
    """Run the step's writes on host pools with the given implementations (copy, then append)."""
    if w.copy_pairs is not None and len(w.copy_pairs):
        copy_fn(k_cache, v_cache, w.copy_pairs)
    if w.slot_mapping is not None and len(w.slot_mapping):
        append_fn(k_cache, v_cache, w.new_key, w.new_value, w.slot_mapping)
