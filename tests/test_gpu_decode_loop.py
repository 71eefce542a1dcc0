"""A real decode loop through the library (needs a GB300).

Prompts that share a prefix are admitted through the prefix cache, every
prompt forks into parallel-sampling branches, and for 20 steps each branch
appends one token: the block manager hands out slots and copy-on-write pairs,
the GPU runs pa_copy_blocks -> pa_reshape_and_cache -> pa_decode, and after
every step the output and the whole cache are checked against the oracle run
on a host mirror fed with the metadata of the page-derived block-manager model
(which must equal the C++ manager's).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from harness import TOL, out_f64, to_numpy_storage, to_torch, within_bound
from oracle import block_manager as M

pytestmark = pytest.mark.gpu

B, D, HKV, HQ, NB = 16, 128, 4, 16, 256
DT = "bf16"


def kv_of(tokens, positions, rng_table):
    """Deterministic K/V for (token id, position): identical prefixes give identical K/V."""
    emb_k, emb_v, pos_k, pos_v = rng_table
    k = emb_k[tokens] + pos_k[positions]
    v = emb_v[tokens] + pos_v[positions]
    return W.to_storage(k, DT), W.to_storage(v, DT)


def test_prefix_cached_parallel_sampling_decode_loop():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    from paged_kv_cache_32_gb300.block_manager import BlockManager
    pa.build()
    rng = np.random.default_rng(2024)
    vocab = 50
    table = (rng.standard_normal((vocab, HKV, D), dtype=np.float32) * 0.5,
             rng.standard_normal((vocab, HKV, D), dtype=np.float32),
             rng.standard_normal((512, HKV, D), dtype=np.float32) * 0.5,
             rng.standard_normal((512, HKV, D), dtype=np.float32) * 0.5)
    shared = list(rng.integers(0, vocab, 40))
    prompts = [shared + list(rng.integers(0, vocab, n)) for n in (5, 17, 30)]

    bm, model = BlockManager(NB, B, shuffle_seed=7), M.BlockManagerModel(NB, B, shuffle_seed=7)
    k_host, v_host = W.nan_array((NB, HKV, B, D), DT), W.nan_array((NB, HKV, B, D), DT)
    k_dev, v_dev = to_torch(k_host, DT), to_torch(v_host, DT)
    desc = pa.cache_desc(k_dev)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(dtype=DT, num_kv_heads=HKV, block_size=B)

    def write(slots, toks, pos):
        nk, nv = kv_of(np.asarray(toks), np.asarray(pos), table)
        O.reshape_and_cache(k_host, v_host, nk, nv, slots, **kw)
        pa.pa_reshape_and_cache(k_dev, v_dev, to_torch(nk, DT), to_torch(nv, DT),
                                torch.from_numpy(slots).cuda(), err_flag=err, desc=desc)

    # ---- admission with the prefix cache: 2 full shared blocks hit for prompts 1 and 2
    for p, toks in enumerate(prompts):
        hits = bm.allocate_with_prefix(p, toks)
        rc, hits_model = model.allocate_with_prefix(p, toks)
        assert rc == 0 and hits == hits_model == (0 if p == 0 else 40 // B)
        tbl = model.tables[p]
        first = hits * B                                   # cached tokens need no recomputation
        pos = np.arange(first, len(toks))
        slots = np.asarray([tbl[i // B] * B + i % B for i in pos], np.int64)
        write(slots, [toks[i] for i in pos], pos)
    # ---- parallel sampling: every prompt forks into 2 branches
    seqs, history = [], {}
    for p in range(3):
        for b in range(2):
            child = 100 + 10 * p + b
            bm.fork(p, child)
            assert model.fork(p, child) == 0
            seqs.append(child)
            history[child] = list(prompts[p])
        bm.free(p)
        assert model.free(p) == 0
    q_rng = np.random.default_rng(5)
    for step in range(20):
        new_tok = {s: int(q_rng.integers(0, vocab)) for s in seqs}
        slots, pairs = bm.append_slots(seqs)
        m_slots, m_pairs = [], []
        for s in seqs:
            rc, slot, src, dst = model.append_slot(s)
            assert rc == 0
            m_slots.append(slot)
            if src >= 0:
                m_pairs.append((src, dst))
        assert list(slots) == m_slots and [tuple(x) for x in pairs] == m_pairs
        m_slots = np.asarray(m_slots, np.int64)
        if m_pairs:
            O.copy_blocks(k_host, v_host, np.asarray(m_pairs, np.int32), head_size=D, **kw)
            pa.pa_copy_blocks(k_dev, v_dev, torch.from_numpy(pairs).cuda(), err_flag=err, desc=desc)
        write(m_slots, [new_tok[s] for s in seqs], [len(history[s]) for s in seqs])
        for s in seqs:
            history[s].append(new_tok[s])
        width = max(len(model.tables[s]) for s in seqs)
        tables, lens = bm.build_tables(seqs, width)
        m_tables = np.zeros_like(tables)
        for i, s in enumerate(seqs):
            m_tables[i, :len(model.tables[s])] = model.tables[s]
        assert np.array_equal(tables, m_tables) and list(lens) == [model.lens[s] for s in seqs]
        q = W.normal(q_rng, (len(seqs), HQ, D), DT)
        out = torch.empty((len(seqs), HQ, D), dtype=torch.bfloat16, device="cuda")
        pa.pa_decode(out, to_torch(q, DT), k_dev, v_dev, torch.from_numpy(tables).cuda(),
                     torch.from_numpy(lens).cuda(), 1.0 / np.sqrt(D), partition_size=32, err_flag=err, desc=desc)
        torch.cuda.synchronize()
        ref = O.paged_attention(q, k_host, v_host, m_tables, np.asarray(lens), scale=1.0 / np.sqrt(D), **kw)
        ok, e, _ = within_bound(out_f64(out), ref, DT)
        assert ok, f"step {step}: max abs err {e}"
        assert int(err.item()) == 0
        assert np.array_equal(to_numpy_storage(k_dev, DT), k_host) and np.array_equal(to_numpy_storage(v_dev, DT), v_host)
    for s in seqs:
        bm.free(s)
    assert bm.num_free() == NB - sum(1 for b in range(NB) if bm.ref_count(b) > 0) == NB
