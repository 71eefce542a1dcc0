"""Chunked prefill attention on the tensor cores vs the CPU fp64 oracle (needs a GB300).

Sequence s holds seq_lens[s] tokens of which the last n_s are the chunk's
queries ("vLLM 核心工程深度剖析", section "6.1": long prompts are prefilled in
chunks; "PagedAttention 详解：缓存的存储结构", section "使用流程": cached prompt
blocks take part in attention directly, new tokens are written through
slot_mapping).  Each step here first writes the chunk's K/V with
pa_reshape_and_cache, then runs pa_prefill over the whole context.

Bar: every output within the per-element bound of ``harness.bound`` (the stated
3e-3 for fp16/bf16, or half an output ulp + 2^-12 where |out| >= 1, which the
first positions of a chunk reach since position 0 returns v itself).  Unused
slots hold NaN, so any read past a sequence or through a wrong block poisons
the result.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from harness import out_f64, rising_keys, to_numpy_storage, to_torch, within_bound

pytestmark = pytest.mark.gpu

SENTINEL = 123.0  # exactly representable in f16 and bf16; rows no chunk owns must keep it


@pytest.fixture(scope="module", autouse=True)
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    return pa


class PrefillStep:
    """Device copies of a prefill workload and the two calls of one step."""

    def __init__(self, w: W.Workload, device="cuda"):
        import torch
        import paged_kv_cache_32_gb300 as pa
        self.w, self.pa = w, pa
        self.k = to_torch(w.k_cache, w.dtype, device)
        self.v = to_torch(w.v_cache, w.dtype, device)
        self.q = to_torch(w.q, w.dtype, device)
        self.nk = to_torch(w.new_key, w.dtype, device)
        self.nv = to_torch(w.new_value, w.dtype, device)
        self.slots = torch.from_numpy(w.slot_mapping).to(device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.qs = torch.from_numpy(w.query_start).to(device)
        self.out = torch.full_like(self.q, SENTINEL)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.desc = pa.cache_desc(self.k)

    def run(self, max_query_len=None):
        import torch
        w = self.w
        if max_query_len is None:
            max_query_len = int(np.max(np.diff(w.query_start))) if len(w.query_start) > 1 else 0
        if len(self.slots):
            self.pa.pa_reshape_and_cache(self.k, self.v, self.nk, self.nv, self.slots, err_flag=self.err,
                                         desc=self.desc)
        self.pa.pa_prefill(self.out, self.q, self.k, self.v, self.tables, self.lens, self.qs, max_query_len, w.scale,
                           err_flag=self.err, desc=self.desc)
        torch.cuda.synchronize()
        return out_f64(self.out)


def host_pools(w: W.Workload):
    k, v = w.k_cache.copy(), w.v_cache.copy()
    O.reshape_and_cache(k, v, w.new_key, w.new_value, w.slot_mapping, dtype=w.dtype, num_kv_heads=w.num_kv_heads,
                        block_size=w.block_size)
    return k, v


def oracle_prefill(w: W.Workload, k, v, seq_lens=None):
    return O.prefill_attention(w.q, k, v, w.block_tables, w.seq_lens if seq_lens is None else seq_lens,
                               w.query_start, dtype=w.dtype, num_kv_heads=w.num_kv_heads, block_size=w.block_size,
                               scale=w.scale)


def small(dtype, block_size, *, hq=8, hkv=2, seed=7, prefix=(0, 0, 3, 17, 200, 0, 129),
          chunk=(1, 5, 130, 128, 77, 259, 300)):
    """Chunks of 1, 5, 128 (one full query tile), 130 and 259/300 (ragged second
    and third tiles), after cached prefixes of 0, 3, 17, 129 and 200 tokens
    (block-aligned and not), so key tiles end both on and off block and tile edges."""
    return W.build_prefill(f"prefill_small_{dtype}_b{block_size}", seed=seed, dtype=dtype, prefix_lens=prefix,
                           chunk_lens=chunk, num_q_heads=hq, num_kv_heads=hkv, head_size=128, block_size=block_size)


def assert_close(got, ref, dtype, what):
    assert not np.isnan(got).any(), f"{what}: NaN in output"
    ok, err, ratio = within_bound(got, ref, dtype)
    assert ok, f"{what}: max abs err {err}, worst err/bound {ratio}"
    return err


# ---------------------------------------------------------------- small cases, every output compared
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128])
def test_prefill_small_gqa(dtype, block_size):
    w = small(dtype, block_size)
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    # the chunk's K/V writes are bit-exact
    assert np.array_equal(to_numpy_storage(g.k, dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(to_numpy_storage(g.v, dtype).view(np.uint8), v.view(np.uint8))
    err = assert_close(got, oracle_prefill(w, k, v), dtype, w.name)
    print(w.name, "max abs err", err)


def test_prefill_small_mha():
    w = small("bf16", 16, hq=4, hkv=4, seed=11)
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    assert_close(got, oracle_prefill(w, k, v), "bf16", w.name)


@pytest.mark.parametrize("dtype,block_size,hq,hkv", [("bf16", 16, 32, 8), ("f16", 64, 16, 4)])
def test_prefill_many_items_per_cta(dtype, block_size, hq, hkv):
    """More work items (sequence, head, query tile) than SMs, so each persistent CTA walks
    several items and its K/V rings, S buffers, barrier phases and Q buffer run on across
    item boundaries (items of 1 to 3 query tiles and 1 to 11 key tiles); every output and
    both pools compared."""
    w = W.build_prefill(f"prefill_multi_{dtype}", seed=41, dtype=dtype,
                        prefix_lens=[0, 300, 17, 129, 500, 64, 0, 200, 31, 1000, 256, 90],
                        chunk_lens=[300, 129, 256, 1, 77, 200, 130, 45, 260, 150, 128, 300], num_q_heads=hq,
                        num_kv_heads=hkv, head_size=128, block_size=block_size)
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    assert np.array_equal(to_numpy_storage(g.k, dtype).view(np.uint8), k.view(np.uint8))
    assert np.array_equal(to_numpy_storage(g.v, dtype).view(np.uint8), v.view(np.uint8))
    err = assert_close(got, oracle_prefill(w, k, v), dtype, w.name)
    print(w.name, "max abs err", err)


def test_prefill_long_context_many_key_tiles():
    """One 200-token chunk after a 3000-token cached prefix: 25 key tiles, the
    online-softmax rescale of O in tensor memory runs many times."""
    w = W.build_prefill("prefill_long", seed=21, dtype="bf16", prefix_lens=[3000, 1000], chunk_lens=[200, 45],
                        num_q_heads=4, num_kv_heads=1, head_size=128, block_size=32)
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    assert_close(got, oracle_prefill(w, k, v), "bf16", w.name)


def test_prefill_large_scores_rescale():
    """Scaled-up queries make the row max jump between key tiles (large alpha
    corrections) and the softmax very peaked."""
    w = small("bf16", 32, seed=5)
    qf = O.to_f64(w.q, "bf16") * 6.0
    w.q = W.to_storage(qf, "bf16")
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    assert_close(got, oracle_prefill(w, k, v), "bf16", w.name)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_rising_scores(dtype):
    """Scores rising along each sequence by about 9 (log2 units) per 128-key tile: fp16 keeps the
    weights it took with the current reference maxima on some tiles and takes the exact path (tile
    maxima, rescale of O, P stored again) on others; bf16 always takes the exact path."""
    w = W.build_prefill(f"prefill_rising_{dtype}", seed=7720, dtype=dtype, prefix_lens=[700, 1500, 0, 64],
                        chunk_lens=[300, 129, 260, 1], num_q_heads=4, num_kv_heads=2, head_size=128,
                        block_size=16)
    rising_keys(w, 0.0045, seed=7721, positions=[700, 1500, 0, 64])
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    assert_close(got, oracle_prefill(w, k, v), dtype, w.name)


# ---------------------------------------------------------------- the full-size workloads, every row
@pytest.mark.parametrize("name", ["prefill_bf16", "prefill_f16"])
def test_prefill_full_size_every_row(name):
    """The benchmark's prefill workloads at full size (16 sequences, cached prefixes
    U[0, 2048], chunks U[256, 2048], 32 q / 8 kv heads, B = 16; bf16, and the same
    shapes in fp16), launched as the benchmark launches them.  Every output row of
    every query token and head is compared with the float64 oracle (its numpy
    form with library matmuls, pinned to the C oracle on small cases)."""
    from oracle import dense
    w = W.WORKLOADS[name]()
    g = PrefillStep(w)
    got = g.run()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    ref = dense.prefill_attention(w.q, k, v, w.block_tables, w.seq_lens, w.query_start, dtype=w.dtype,
                                  num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
    err = assert_close(got, ref, w.dtype, f"{name} every row")
    print(f"{name} max abs err {err} over {got.shape[0]} query tokens x {got.shape[1]} heads")


# ---------------------------------------------------------------- edges and data errors
def test_prefill_empty_chunks_and_grid_slack():
    """Sequences with no queries are skipped; a max_query_len above the real
    longest chunk only adds CTAs that exit; rows nobody owns are untouched."""
    w = W.build_prefill("prefill_empty", seed=3, dtype="f16", prefix_lens=[40, 10, 0, 64], chunk_lens=[0, 70, 0, 1],
                        num_q_heads=4, num_kv_heads=2, head_size=128, block_size=16)
    g = PrefillStep(w)
    got = g.run(max_query_len=500)
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    assert_close(got, oracle_prefill(w, k, v), "f16", w.name)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_inconsistent_chunk_reported_and_skipped(dtype):
    """A chunk longer than its sequence (L < n) is reported as
    PA_DEVERR_QUERY; its rows keep their old contents and the other sequences
    are still computed.  The chunk before it ends in a ragged query tile, whose
    rows past that chunk (the skipped chunk's) must not be written: fp16 writes
    that tile through its shared-memory stage, bf16 from registers."""
    import torch
    w = small(dtype, 16)
    g = PrefillStep(w)
    bad = 2
    lens = w.seq_lens.copy()
    lens[bad] = int(w.query_start[bad + 1] - w.query_start[bad]) - 1
    g.lens.copy_(torch.from_numpy(lens))
    got = g.run()
    assert int(g.err.item()) == 5
    k, v = host_pools(w)
    ref = oracle_prefill(w, k, v)
    rows = np.arange(w.query_start[bad], w.query_start[bad + 1])
    assert np.all(got[rows] == SENTINEL)
    keep = np.setdiff1d(np.arange(len(got)), rows)
    assert_close(got[keep], ref[keep], dtype, "other sequences")


def test_prefill_bad_block_id_reported():
    """A table entry outside [0, num_blocks) is reported as PA_DEVERR_BLOCK_ID
    and never dereferenced; sequences that do not use it stay exact."""
    import torch
    w = small("f16", 32)
    g = PrefillStep(w)
    bad = 4
    tables = w.block_tables.copy()
    tables[bad, 0] = w.num_blocks + 7
    g.tables.copy_(torch.from_numpy(tables))
    got = g.run()
    assert int(g.err.item()) == 1
    k, v = host_pools(w)
    ref = oracle_prefill(w, k, v)
    rows = np.arange(w.query_start[bad], w.query_start[bad + 1])
    keep = np.setdiff1d(np.arange(len(got)), rows)
    assert_close(got[keep], ref[keep], "f16", "other sequences")


def test_prefill_matches_decode_on_last_query():
    """The last query of a chunk sees the whole sequence, so its output is the
    decode output of that sequence: two kernels, one definition."""
    import torch
    w = small("bf16", 16)
    g = PrefillStep(w)
    got = g.run()
    last = w.query_start[1:] - 1
    q_last = g.q[torch.from_numpy(last.astype(np.int64)).cuda()].contiguous()
    out = torch.empty_like(q_last)
    g.pa.pa_decode(out, q_last, g.k, g.v, g.tables, g.lens, w.scale, err_flag=g.err, desc=g.desc)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    k, v = host_pools(w)
    ref = O.paged_attention(w.q[last], k, v, w.block_tables, w.seq_lens, dtype="bf16", num_kv_heads=w.num_kv_heads,
                            block_size=w.block_size, scale=w.scale)
    assert_close(got[last], ref, "bf16", "prefill last query")
    assert_close(out_f64(out), ref, "bf16", "decode")
