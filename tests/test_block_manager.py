"""Host KV block manager (C++ in libpa.so) against the page-derived Python model (no GPU)."""
import json
import os

import numpy as np
import pytest

from oracle import block_manager as M
from paged_kv_cache_32_gb300 import block_manager as BM


@pytest.fixture(scope="module", autouse=True)
def built():
    import paged_kv_cache_32_gb300 as pa
    pa.build()


def test_hash_and_shuffle_generators_match_published_vectors(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "hash_vectors.json")))
    for text, want in g["fnv1a64"].items():
        assert M.fnv1a64(text.encode()) == int(want, 16)
    r = M.SplitMix64(g["splitmix64_seed"])
    assert [r.next() for _ in range(5)] == g["splitmix64_first5"]


def test_free_queue_order_and_shuffle_match_model():
    for seed in (0, 1, 99, 2 ** 63 + 5):
        bm, m = BM.BlockManager(37, 4, seed), M.BlockManagerModel(37, 4, seed)
        bm.allocate(1, 37 * 4)
        assert m.allocate(1, 37 * 4) == M.OK
        assert list(bm.build_tables([1])[0][0]) == m.tables[1]
        assert sorted(m.tables[1]) == list(range(37))


def test_copy_on_write_sequence_from_the_page():
    """P8 shared by two branches (ref 2); branch A appends into it: allocate a new
    block, copy P8 to it, remap A, P8's ref drops to 1, the token lands in the copy."""
    bm = BM.BlockManager(16, 4)
    bm.allocate(0, 6)                      # blocks [0, 1]; block 1 holds 2 of 4 slots
    bm.fork(0, 1)                          # branch B shares both
    assert bm.ref_count(1) == 2
    slot, src, dst = bm.append_slot(0)     # branch A writes its 7th token
    assert (src, dst) == (1, 2)            # new block 2 = copy of shared block 1
    assert slot == 2 * 4 + 2               # token 6 -> offset 2 of the private copy
    assert bm.ref_count(1) == 1 and bm.ref_count(2) == 1
    assert list(bm.build_tables([0, 1])[0][0]) == [0, 2] and list(bm.build_tables([0, 1])[0][1]) == [0, 1]
    slot, src, dst = bm.append_slot(1)     # branch B now owns block 1 alone: no copy
    assert (src, dst) == (-1, -1) and slot == 1 * 4 + 2


def test_full_last_block_appends_a_new_block_without_copy():
    bm = BM.BlockManager(8, 4)
    bm.allocate(0, 8)
    bm.fork(0, 1)
    slot, src, dst = bm.append_slot(0)
    assert (src, dst) == (-1, -1) and slot == 2 * 4 + 0


def test_reference_counts_free_and_exhaustion():
    bm = BM.BlockManager(4, 16)
    bm.allocate(0, 35)                     # 3 blocks, the last 3/16 filled
    assert bm.num_free() == 1 and bm.seq_len(0) == 35 and bm.num_seq_blocks(0) == 3
    with pytest.raises(BM.BlockManagerError):
        bm.allocate(1, 20)                 # needs 2 blocks, 1 free
    bm.fork(0, 1)
    bm.free(0)
    assert bm.num_free() == 1              # still held by the fork
    bm.free(1)
    assert bm.num_free() == 4
    with pytest.raises(BM.BlockManagerError):
        bm.free(1)


def test_reservation_waste_example_with_16_token_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "reservation_waste.json")))
    bm = BM.BlockManager(4096, g["block_size"])
    for r in range(g["requests"]):
        bm.allocate(r, g["used_per_request"])
    held = (4096 - bm.num_free()) * g["block_size"]
    used = g["requests"] * g["used_per_request"]
    assert held - used == g["requests"] * (-g["used_per_request"] % g["block_size"])   # 8 x 4 = 32 slots
    assert (g["expected"]["wasted"], held - used) == (20768, 32)


def test_prefix_cache_hits_full_blocks_only_and_evicts_on_reuse():
    B = 4
    bm = BM.BlockManager(12, B)
    prompt = list(range(100, 111))                     # 11 tokens: 2 full blocks + 3
    assert bm.allocate_with_prefix(0, prompt) == 0
    t0 = bm.build_tables([0])[0][0]
    assert bm.allocate_with_prefix(1, prompt[:8] + [7, 7]) == 2     # same two full blocks
    t1 = bm.build_tables([1])[0][0]
    assert list(t1[:2]) == list(t0[:2]) and t1[2] != t0[2]          # partial block never shared
    assert bm.ref_count(int(t0[0])) == 2
    assert bm.allocate_with_prefix(2, [100, 101, 102, 999] + prompt[4:8]) == 0   # first block differs
    bm.free(0)
    bm.free(1)
    assert bm.allocate_with_prefix(3, prompt[:8]) == 2      # cached blocks survive while queued
    bm.free(3)
    bm.free(2)
    bm.allocate(4, 12 * B)                                  # cycles the whole queue: evicts every entry
    bm.free(4)
    assert bm.allocate_with_prefix(5, prompt[:8]) == 0


def _run_ops(seed, n_ops=400, num_blocks=48, B=4):
    rng = np.random.default_rng(seed)
    bm, m = BM.BlockManager(num_blocks, B, seed + 1), M.BlockManagerModel(num_blocks, B, seed + 1)
    live, next_id = [], 0
    vocab = rng.integers(0, 5, size=200)     # few distinct tokens: prefix hits happen
    for _ in range(n_ops):
        op = rng.choice(["alloc", "prefix", "append", "fork", "free"], p=[0.15, 0.15, 0.4, 0.15, 0.15])
        if op in ("alloc", "prefix") or not live:
            n = int(rng.integers(0, 14))
            if op == "prefix":
                toks = [int(x) for x in vocab[:n]] if rng.random() < 0.7 else [int(x) for x in rng.integers(0, 5, n)]
                want_rc, want_hits = m.allocate_with_prefix(next_id, toks)
                try:
                    got_hits, got_rc = bm.allocate_with_prefix(next_id, toks), 0
                except BM.BlockManagerError as e:
                    got_hits, got_rc = 0, e.status
                assert (got_rc, got_hits if got_rc == 0 else 0) == (want_rc, want_hits if want_rc == 0 else 0)
            else:
                want_rc = m.allocate(next_id, n)
                try:
                    bm.allocate(next_id, n)
                    got_rc = 0
                except BM.BlockManagerError as e:
                    got_rc = e.status
                assert got_rc == want_rc
            if want_rc == 0:
                live.append(next_id)
            next_id += 1
        elif op == "append":
            s = int(rng.choice(live))
            want = m.append_slot(s)
            try:
                got = (0,) + bm.append_slot(s)
            except BM.BlockManagerError as e:
                got = (e.status, -1, -1, -1)
            assert got == want
        elif op == "fork":
            s = int(rng.choice(live))
            assert m.fork(s, next_id) == 0
            bm.fork(s, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = int(rng.choice(live))
            live.remove(s)
            assert m.free(s) == 0
            bm.free(s)
        assert bm.num_free() == m.num_free()
        if live:
            tables, lens = bm.build_tables(live, width=num_blocks)
            for i, s in enumerate(live):
                assert list(tables[i][:len(m.tables[s])]) == m.tables[s] and lens[i] == m.lens[s]
        assert [bm.ref_count(b) for b in range(num_blocks)] == m.ref


@pytest.mark.parametrize("seed", range(6))
def test_random_operation_sequences_match_model(seed):
    _run_ops(seed)


def test_decode_step_batch_api():
    bm = BM.BlockManager(64, 4, 3)
    for s in range(4):
        bm.allocate(s, 5)
    bm.fork(0, 10)
    slots, pairs = bm.append_slots([0, 1, 2, 3, 10])
    assert slots.shape == (5,) and pairs.shape == (1, 2)   # only seq 0 hits its shared partial block
    tables, lens = bm.build_tables([0, 1, 2, 3, 10])
    assert list(lens) == [6] * 5
    for i, s in enumerate([0, 1, 2, 3, 10]):
        assert slots[i] == tables[i, 1] * 4 + 1
