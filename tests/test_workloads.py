"""Host-side input construction: the block allocator used to build workloads (no GPU)."""
import json
import os

import numpy as np
import pytest

import workloads as W


def test_refcount_fork_free():
    a = W.BlockAllocator(8, 4, np.random.default_rng(0))
    blocks = a.allocate(0, 10)                       # 3 blocks
    assert len(blocks) == 3 and all(a.ref_count[b] == 1 for b in blocks)
    a.fork(0, 1)
    assert all(a.ref_count[b] == 2 for b in blocks)
    a.free(0)
    assert all(a.ref_count[b] == 1 for b in blocks) and a.num_free() == 5   # still referenced by seq 1
    a.free(1)
    assert a.num_free() == 8


def test_append_slot_allocates_on_block_boundary():
    a = W.BlockAllocator(4, 4, np.random.default_rng(1))
    a.allocate(0, 3)
    first = a.tables[0][0]
    assert a.append_slot(0) == first * 4 + 3             # fills the last free slot
    s = a.append_slot(0)                                 # needs a new block
    assert len(a.tables[0]) == 2 and s == a.tables[0][1] * 4


def test_cow_gives_private_block_and_drops_reference():
    a = W.BlockAllocator(8, 4, np.random.default_rng(2))
    a.allocate(0, 6)
    a.fork(0, 1)
    shared = a.tables[0][1]
    src, dst = a.cow(1, 1)
    assert src == shared and dst != shared
    assert a.tables[1][1] == dst and a.tables[0][1] == shared
    assert a.ref_count[shared] == 1 and a.ref_count[dst] == 1


def test_pool_exhaustion_raises():
    a = W.BlockAllocator(2, 4)
    a.allocate(0, 8)
    with pytest.raises(W.OutOfBlocks):
        a.allocate(1, 1)


def test_reservation_waste_example(golden_dir):
    """Contiguous reservation wastes 63% in the page's example; 16-token blocks waste
    only the unfilled tail of each request's last block."""
    g = json.load(open(os.path.join(golden_dir, "reservation_waste.json")))
    reserved = g["requests"] * g["reserved_per_request"]
    used = g["requests"] * g["used_per_request"]
    e = g["expected"]
    assert (reserved, used, reserved - used) == (e["reserved"], e["used"], e["wasted"])
    assert round(100 * (reserved - used) / reserved) == e["waste_percent"]
    a = W.BlockAllocator(4096, g["block_size"])
    for r in range(g["requests"]):
        a.allocate(r, g["used_per_request"])
    held = (4096 - a.num_free()) * g["block_size"]
    assert held - used == g["requests"] * (-g["used_per_request"] % g["block_size"])
    assert held - used < g["requests"] * g["block_size"]


def test_tiny_workload_matches_config():
    w = W.tiny_f32()
    assert list(w.seq_lens) == [1, 15, 16, 35]
    assert list(w.block_tables[3]) == [7, 3, 12]
    assert w.num_blocks == 32 and w.k_cache.shape == (32, 4, 16, 64)
    used = set()
    for s, L in enumerate(w.seq_lens):
        used.update(int(b) for b in w.block_tables[s, :-(-int(L) // 16)])
    assert len(used) == 6                      # 1 + 1 + 1 + 3 distinct blocks
    # unused blocks are NaN-poisoned so a wrong gather shows up in the output
    unused = [b for b in range(32) if b not in used]
    assert np.isnan(w.k_cache[unused]).all()


def test_bf16_storage_rounding():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], dtype=np.float32)
    bits = W.to_storage(x, "bf16")
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    import torch
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(back, ref)


def test_shared_prefix_structure_small():
    w = W.shared_prefix_f16(num_prompts=2, branches=4, prefix_len=32, max_suffix=5, num_heads=2,
                            block_size=16, num_blocks=64, seed=5)
    assert w.num_seqs == 8 and len(w.copy_pairs) == 8
    # each branch's last prefix block is a private copy; earlier prefix blocks are shared by 4
    for p in range(2):
        rows = w.block_tables[4 * p:4 * p + 4]
        assert len(set(rows[:, 0])) == 1
        assert len(set(rows[:, 1])) == 4
    assert len(w.slot_mapping) == int(np.sum(w.seq_lens - 32))
