"""CUDA library vs the CPU fp64 oracle, element by element (needs a GB300).

Attention: max abs error <= 1e-5 (fp32) / 3e-3 (fp16, bf16) against fp64.
Slot writes and block copies: bit-exact over the whole pool (untouched bytes
included).  Unused slots and unreferenced blocks hold NaN, so any read past a
sequence's end or through a wrong block ID poisons the output.
"""
import zlib

import numpy as np
import pytest

import oracle as O
import workloads as W
from harness import TOL, GpuStep, max_abs_err, oracle_step, out_f64, rising_keys, to_numpy_storage, within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    return pa


def check_step(w: W.Workload, threads: int = 0, partition_size=None):
    import torch
    g = GpuStep(w)
    g.writes()
    g.decode(partition_size=partition_size)
    torch.cuda.synchronize()
    k_ref, v_ref, ref = oracle_step(w, threads)
    assert int(g.err.item()) == 0
    assert np.array_equal(to_numpy_storage(g.k, w.dtype).view(np.uint8), k_ref.view(np.uint8))
    assert np.array_equal(to_numpy_storage(g.v, w.dtype).view(np.uint8), v_ref.view(np.uint8))
    got = out_f64(g.out)
    assert not np.isnan(got).any()
    ok, err, ratio = within_bound(got, ref, w.dtype)
    assert ok, f"{w.name}: max abs err {err}, worst err/bound {ratio}"
    if ref.size and np.max(np.abs(ref)) < 1.0:
        assert err <= TOL[w.dtype], f"{w.name}: max abs err {err}"   # the stated tolerance, unchanged
    return err, g


# ---------------------------------------------------------------- the five workloads at full size
def test_tiny_f32():
    check_step(W.tiny_f32())


def test_mha_f16_with_append():
    err, _ = check_step(W.mha_f16())
    print("mha_f16 max abs err", err)


def test_mha_f16_full_size_fused_append():
    """The benchmarked form of the MHA fp16 step: one pa_decode_append call at full size.  Both pools
    equal the oracle's after its append bit for bit, every output element meets the oracle, and the
    output equals the two-call path (pa_reshape_and_cache, then pa_decode) bit for bit."""
    import torch
    w = W.mha_f16()
    g = GpuStep(w)
    g.pa.pa_decode_append(g.out, g.q, g.k, g.v, g.nk, g.nv, g.tables, g.lens, w.scale,
                          partition_size=w.partition_size, workspace=g.ws, err_flag=g.err, desc=g.desc)
    torch.cuda.synchronize()
    k_ref, v_ref, ref = oracle_step(w)
    assert int(g.err.item()) == 0
    assert np.array_equal(to_numpy_storage(g.k, w.dtype).view(np.uint8), k_ref.view(np.uint8))
    assert np.array_equal(to_numpy_storage(g.v, w.dtype).view(np.uint8), v_ref.view(np.uint8))
    got = out_f64(g.out)
    ok, err, ratio = within_bound(got, ref, w.dtype)
    assert ok, f"max abs err {err}, worst err/bound {ratio}"
    if np.max(np.abs(ref)) < 1.0:
        assert err <= TOL[w.dtype]
    two = GpuStep(w)
    two.writes()
    two.decode()
    torch.cuda.synchronize()
    assert torch.equal(g.out.view(torch.int16), two.out.view(torch.int16))


def test_gqa_bf16():
    w = W.gqa_bf16()
    err, g = check_step(w)
    # the bf16 tolerance needs |out| well below 1 (half an ulp at [1, 2) is 3.9e-3)
    assert float(np.max(np.abs(out_f64(g.out)))) < 0.75


def test_shared_prefix_f16_cow_and_append():
    check_step(W.shared_prefix_f16())


@pytest.mark.parametrize("block_size", [16, 32, 64])
def test_long_bf16_split(block_size):
    check_step(W.long_bf16(block_size))


# ---------------------------------------------------------------- small cases: tiles, ragged tails, edge cases
SMALL = [
    # dtype, Hq, Hkv, D, B, lens
    ("f16", 8, 8, 128, 16, [1, 15, 16, 17, 31, 32, 33, 100]),
    ("bf16", 16, 2, 128, 32, [1, 31, 32, 33, 64, 65, 300]),
    ("bf16", 32, 8, 128, 64, [63, 64, 65, 127, 129, 700]),
    ("f16", 16, 1, 64, 16, [5, 16, 250, 513]),        # G = 16: two head groups per kv head
    ("bf16", 12, 4, 64, 32, [0, 1, 2, 40, 1000]),     # G = 3, an empty sequence
    ("f16", 4, 4, 64, 48, [47, 48, 49, 200]),          # B = 48: 16-token slabs, 3 per block
    ("f32", 8, 2, 128, 16, [1, 16, 17, 90, 600]),
    ("f32", 4, 4, 64, 8, [1, 7, 8, 9, 64]),           # fp32 takes any block size
    # large blocks (8 and 16 slabs of 16 tokens per block), as the benchmark's block-size sweep
    # times them: G = 1 and G = 8, ragged tails inside a block and across blocks
    ("f16", 4, 4, 128, 128, [1, 127, 128, 129, 300, 1000]),
    ("f16", 16, 2, 128, 128, [2, 127, 128, 129, 500, 1100]),
    ("bf16", 4, 4, 128, 128, [3, 127, 128, 129, 260, 900]),
    ("bf16", 16, 2, 128, 128, [1, 127, 128, 129, 450, 1200]),
    ("f16", 4, 4, 128, 256, [1, 255, 256, 257, 700, 1300]),
    ("f16", 8, 1, 128, 256, [2, 255, 256, 257, 600, 1500]),
    ("bf16", 4, 4, 128, 256, [3, 255, 256, 257, 513, 1400]),
    ("bf16", 16, 2, 128, 256, [1, 255, 256, 257, 800, 1600]),
    # 8-token blocks: a 16-token slab comes from two blocks (two 8-row copies), its second half
    # absent when the sequence ends inside the first
    ("f16", 4, 4, 128, 8, [1, 7, 8, 9, 15, 16, 17, 24, 300]),
    ("bf16", 16, 2, 128, 8, [2, 8, 9, 23, 33, 1000]),
    ("f16", 8, 1, 64, 8, [3, 8, 16, 25, 513]),
    ("bf16", 4, 4, 64, 8, [1, 9, 40, 777]),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}-Hq{c[1]}-Hkv{c[2]}-D{c[3]}-B{c[4]}")
@pytest.mark.parametrize("partition", [0, "one_block", "big"])
def test_small_cases(case, partition):
    dtype, Hq, Hkv, D, B, lens = case
    w = W.build_decode("small", seed=zlib.crc32(repr(case).encode()) % 10000, dtype=dtype, seq_lens=lens, num_q_heads=Hq, num_kv_heads=Hkv,
                       head_size=D, block_size=B, pool_factor=1.3, append_last=True)
    # the 16-bit kernels' partitions are whole 16-token slabs: with 8-token blocks, two blocks
    part = {0: 0, "one_block": B if dtype == "f32" else max(B, 16), "big": 8 * max(B, 32)}[partition]
    check_step(w, partition_size=part)


# ---------------------------------------------------------------- running maxima that move and stay
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("partition", [0, 64])
def test_rising_scores_running_max(dtype, partition):
    """Scores rising along each sequence by about 8 (log2 units) per 16-token slab: a head's running
    max moves on the slabs whose scores exceed it by more than 8 and stays on the others, so both the
    kept weights (up to 2^8) and the rescale of O run, within partitions and across the merge."""
    w = W.build_decode(f"rising_{dtype}", seed=7700, dtype=dtype, seq_lens=[1, 16, 17, 300, 1000, 2100],
                       num_q_heads=16, num_kv_heads=2, head_size=128, block_size=16, append_last=True)
    rising_keys(w, 0.03, seed=7701)
    check_step(w, partition_size=partition)


# ---------------------------------------------------------------- the partition merge
MANY = [  # dtype, Hq, Hkv, B, lens; one block per partition: up to 157 partitions in a sequence
    ("f16", 8, 1, 16, [2500, 1100, 17, 0, 1040]),    # G = 8: one group of eight query heads
    ("bf16", 16, 1, 16, [2500, 1100, 17, 0, 1040]),  # G = 16: two head groups per kv head
    ("f16", 4, 4, 32, [4100, 33, 2080]),             # G = 1
    ("f32", 6, 2, 16, [1300, 20]),                   # G = 3, the CUDA-core kernel
]


@pytest.mark.parametrize("case", MANY, ids=lambda c: f"{c[0]}-Hq{c[1]}-Hkv{c[2]}-B{c[3]}")
def test_merge_many_partitions_garbage_workspace(case):
    """Up to 157 partitions in a sequence (the merge splits a row's partitions over eight
    warps), ragged counts per sequence (157, 69, 2, none, 65) and a workspace full of garbage
    (every partial is written before it is read).  A second call on the same workspace gives
    the bit-identical output."""
    import torch
    dtype, Hq, Hkv, B, lens = case
    w = W.build_decode("many_parts", seed=zlib.crc32(repr(case).encode()) % 10000, dtype=dtype, seq_lens=lens,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_size=128, block_size=B, pool_factor=1.2)
    g = GpuStep(w)
    need = g.pa.pa_decode_workspace_size(w.num_seqs, Hq, w.max_blocks_per_seq, g.desc, B)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")
    g.pa.pa_decode(g.out, g.q, g.k, g.v, g.tables, g.lens, w.scale, partition_size=B, workspace=ws,
                   err_flag=g.err, desc=g.desc)
    first = g.out.clone()
    g.pa.pa_decode(g.out, g.q, g.k, g.v, g.tables, g.lens, w.scale, partition_size=B, workspace=ws,
                   err_flag=g.err, desc=g.desc)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(first, g.out)
    _, _, ref = oracle_step(w)
    got = out_f64(g.out)
    ok, err, ratio = within_bound(got, ref, w.dtype)
    assert ok, f"{case}: max abs err {err}, worst err/bound {ratio}"


# ---------------------------------------------------------------- the default split at the extremes
def _default_split_check(w):
    """Decode at the default partition size on a workspace full of garbage, twice: bit-identical
    calls, within the bound of the fp64 oracle, and no device error."""
    import torch
    g = GpuStep(w)
    need = g.pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, g.desc, 0)
    ws = torch.full((max(need, 1),), 0x7F, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        out = torch.full_like(g.q, float("nan"))
        g.pa.pa_decode(out, g.q, g.k, g.v, g.tables, g.lens, w.scale, partition_size=0, workspace=ws,
                       err_flag=g.err, desc=g.desc)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = O.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=w.dtype,
                            num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
    ok, err, ratio = within_bound(out_f64(outs[1]), ref, w.dtype)
    assert ok, f"{w.name}: max abs err {err}, worst err/bound {ratio}"


def test_many_short_sequences():
    """40 000 sequences of 0 to 40 tokens (1 in 8 empty), 2 q / 1 kv heads, D = 64: a grid of
    40 000 work items of one to three slabs; empty sequences get zero rows."""
    rng = np.random.default_rng(2024)
    lens = rng.integers(1, 41, size=40000)
    lens[::8] = 0
    w = W.build_decode("short_many", seed=2024, dtype="bf16", seq_lens=lens, num_q_heads=2, num_kv_heads=1,
                       head_size=64, block_size=16, pool_factor=1.1)
    _default_split_check(w)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_long_sequences_default_partitions(dtype):
    """Two sequences of 8192 and 6000 tokens, 32 q / 8 kv heads, B = 32: eight and six 1024-token
    partitions per (sequence, kv head), merged."""
    w = W.build_decode(f"long_default_{dtype}", seed=77, dtype=dtype, seq_lens=[8192, 6000], num_q_heads=32,
                       num_kv_heads=8, head_size=128, block_size=32, pool_factor=1.1)
    _default_split_check(w)


@pytest.mark.parametrize("case", [
    ("f16", 8, 8, 128, 16, [1, 15, 16, 17, 700, 0, 2048, 33]),
    ("bf16", 64, 8, 128, 32, [5, 300, 1200, 4000, 64, 0, 999]),
    ("bf16", 24, 2, 64, 64, [1, 130, 4096, 77]),        # G = 12: two head groups, the second of 4 heads
], ids=lambda c: f"{c[0]}-Hq{c[1]}-Hkv{c[2]}-D{c[3]}-B{c[4]}")
def test_default_split_garbage_workspace(case):
    dtype, Hq, Hkv, D, B, lens = case
    w = W.build_decode("default_mix", seed=zlib.crc32(repr(case).encode()) % 10000, dtype=dtype, seq_lens=lens,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, block_size=B, pool_factor=1.3)
    _default_split_check(w)


# ---------------------------------------------------------------- the decode step with its append fused in
APPEND = [  # dtype, Hq, Hkv, D, B, lens (the last token of each sequence is the step's new token)
    ("f16", 32, 32, 128, 16, [1, 2, 15, 16, 17, 700, 2048, 0]),  # L = 1: the new token alone; L = 0: nothing
    ("bf16", 64, 8, 128, 32, [64, 1200, 4096, 33, 1]),            # G = 8
    ("bf16", 24, 2, 64, 64, [1, 130, 1500, 64, 65]),              # G = 12: two head groups, the first writes
    ("f16", 8, 2, 128, 8, [1, 8, 9, 16, 17, 300]),                # 8-token blocks: the token in either half
]


@pytest.mark.parametrize("case", APPEND, ids=lambda c: f"{c[0]}-Hq{c[1]}-Hkv{c[2]}-D{c[3]}-B{c[4]}")
@pytest.mark.parametrize("split", ["default", "smallest"])
def test_decode_append_fused(case, split):
    """pa_decode_append stores each sequence's new token at position L - 1 (its slot starts as NaN)
    and attends over it in one launch: the caches equal the oracle's append bit for bit, the output
    meets the oracle, and both equal pa_reshape_and_cache followed by pa_decode bit for bit.  The
    smallest partition (one block, or one 16-token slab for 8-token blocks) puts the new token in
    the last of many partitions."""
    import torch
    dtype, Hq, Hkv, D, B, lens = case
    partition = 0 if split == "default" else max(B, 16)
    w = W.build_decode("append", seed=zlib.crc32(repr(case).encode()) % 10000, dtype=dtype, seq_lens=lens,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, block_size=B, pool_factor=1.3,
                       append_last=True, partition_size=partition)
    g = GpuStep(w)
    g.pa.pa_decode_append(g.out, g.q, g.k, g.v, g.nk, g.nv, g.tables, g.lens, w.scale, partition_size=partition,
                          workspace=g.ws, err_flag=g.err, desc=g.desc)
    torch.cuda.synchronize()
    k_ref, v_ref, ref = oracle_step(w)
    assert int(g.err.item()) == 0
    assert np.array_equal(to_numpy_storage(g.k, dtype).view(np.uint8), k_ref.view(np.uint8))
    assert np.array_equal(to_numpy_storage(g.v, dtype).view(np.uint8), v_ref.view(np.uint8))
    ok, err, ratio = within_bound(out_f64(g.out), ref, dtype)
    assert ok, f"max abs err {err}, worst err/bound {ratio}"
    two = GpuStep(w)
    two.writes()
    two.decode()
    torch.cuda.synchronize()
    assert torch.equal(g.out.view(torch.int16), two.out.view(torch.int16))


def test_permuted_block_ids_bit_identical():
    """Relabelling physical blocks leaves the GPU output bit-identical."""
    import torch
    w = W.gqa_bf16(num_seqs=16, hi=1500)
    g1 = GpuStep(w)
    g1.decode()
    perm = np.random.default_rng(3).permutation(w.num_blocks)
    k = np.empty_like(w.k_cache); k[perm] = w.k_cache
    v = np.empty_like(w.v_cache); v[perm] = w.v_cache
    w2 = W.Workload(**{**w.__dict__, "k_cache": k, "v_cache": v,
                       "block_tables": perm[w.block_tables].astype(np.int32)})
    g2 = GpuStep(w2)
    g2.decode()
    torch.cuda.synchronize()
    assert torch.equal(g1.out, g2.out)


def test_bad_block_id_sets_flag_and_stays_in_bounds():
    import torch
    w = W.build_decode("bad", seed=9, dtype="f16", seq_lens=[40, 40], num_q_heads=4, num_kv_heads=4,
                       head_size=128, block_size=16, pool_factor=1.5)
    w.block_tables[1, 1] = w.num_blocks + 1000
    g = GpuStep(w)
    g.decode()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 1
    # sequence 0 is untouched by the bad entry
    ref = O.paged_attention(w.q[:1], w.k_cache, w.v_cache, w.block_tables[:1], w.seq_lens[:1], dtype="f16",
                            num_kv_heads=4, block_size=16, scale=w.scale)
    assert max_abs_err(g.out[:1], ref) <= TOL["f16"]


def test_bad_slot_and_pair_set_flags():
    import torch
    import paged_kv_cache_32_gb300 as pa
    w = W.build_decode("badw", seed=10, dtype="bf16", seq_lens=[20], num_q_heads=2, num_kv_heads=2, head_size=64,
                       block_size=16, pool_factor=2.0)
    g = GpuStep(w)
    before_k = g.k.clone()
    same = lambda a, b: torch.equal(a.view(torch.int16), b.view(torch.int16))  # bitwise: the pool holds NaN
    slots = torch.tensor([w.num_blocks * 16 + 3], dtype=torch.int64, device="cuda")
    key = torch.ones(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_reshape_and_cache(g.k, g.v, key, key.clone(), slots, err_flag=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 2 and same(before_k, g.k)
    g.err.zero_()
    pairs = torch.tensor([[0, w.num_blocks]], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(g.k, g.v, pairs, err_flag=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 3 and same(before_k, g.k)


def test_cow_leaves_other_branches_untouched_on_gpu():
    """After the copies and appends of the shared-prefix step, every block that was
    neither a copy destination nor written by an append is byte-identical."""
    import torch
    w = W.shared_prefix_f16(num_prompts=4, branches=8, prefix_len=1020, max_suffix=40, num_blocks=1024, seed=11)
    g = GpuStep(w)
    g.writes()
    torch.cuda.synchronize()
    k = to_numpy_storage(g.k, "f16").view(np.uint16)
    dsts = set(int(x) for x in w.copy_pairs[:, 1])
    written = set(int(s) // 16 for s in w.slot_mapping)
    keep = [b for b in range(w.num_blocks) if b not in dsts | written]
    assert np.array_equal(k[keep], w.k_cache.view(np.uint16)[keep])
    # 1020 = 63 * 16 + 12: the copied block is partial and the first suffix tokens land in the copy
    assert dsts & written


# ---------------------------------------------------------------- ALiBi (pa_decode_ex)
def alibi_slopes(num_heads: int) -> np.ndarray:
    """The usual geometric slopes 2^(-8 i / H), i = 1..H (a choice of inputs; any slopes are valid)."""
    return (2.0 ** (-8.0 * np.arange(1, num_heads + 1) / num_heads)).astype(np.float32)


@pytest.mark.parametrize("case", [
    ("f16", 8, 8, 128, 16, [1, 15, 33, 300]),
    ("bf16", 16, 2, 128, 32, [2, 64, 65, 700]),
    ("f32", 8, 2, 64, 16, [1, 17, 90, 600]),
], ids=lambda c: f"{c[0]}-Hq{c[1]}-Hkv{c[2]}-D{c[3]}-B{c[4]}")
@pytest.mark.parametrize("partition", [0, "one_block"])
def test_alibi_small_cases(case, partition):
    import torch
    dtype, Hq, Hkv, D, B, lens = case
    w = W.build_decode("alibi", seed=zlib.crc32(repr(case).encode()) % 10000, dtype=dtype, seq_lens=lens,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, block_size=B, pool_factor=1.3)
    slopes = alibi_slopes(Hq)
    g = GpuStep(w)
    part = 0 if partition == 0 else B
    need = g.pa.pa_decode_workspace_size(w.num_seqs, Hq, w.max_blocks_per_seq, g.desc, part)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    g.pa.pa_decode(g.out, g.q, g.k, g.v, g.tables, g.lens, w.scale, partition_size=part, workspace=ws,
                   err_flag=g.err, desc=g.desc, alibi_slopes=torch.from_numpy(slopes).cuda())
    torch.cuda.synchronize()
    ref = O.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=dtype, num_kv_heads=Hkv,
                            block_size=B, scale=w.scale, alibi_slopes=slopes.astype(np.float64))
    ok, err, _ = within_bound(out_f64(g.out), ref, dtype)
    assert ok and int(g.err.item()) == 0, f"max abs err {err}"


def test_alibi_gqa_bf16_full():
    import torch
    w = W.gqa_bf16()
    slopes = alibi_slopes(w.num_q_heads)
    g = GpuStep(w)
    g.pa.pa_decode(g.out, g.q, g.k, g.v, g.tables, g.lens, w.scale, workspace=g.ws, err_flag=g.err, desc=g.desc,
                   alibi_slopes=torch.from_numpy(slopes).cuda())
    torch.cuda.synchronize()
    ref = O.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype="bf16",
                            num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale,
                            alibi_slopes=slopes.astype(np.float64))
    ok, err, _ = within_bound(out_f64(g.out), ref, "bf16")
    assert ok and int(g.err.item()) == 0, f"max abs err {err}"
