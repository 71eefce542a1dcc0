"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each check raises AssertionError on failure.  They are written as plain
functions so that ``test_oracle_pins.py`` runs them against the oracle and
``test_oracle_mutants.py`` runs them against deliberately broken copies of it
(every planted mistake must trip at least one pin).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle as O
import workloads as W
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _attn(w: W.Workload, k=None, v=None, tables=None, lens=None, **kw):
    return O.paged_attention(w.q, w.k_cache if k is None else k, w.v_cache if v is None else v,
                             w.block_tables if tables is None else tables, w.seq_lens if lens is None else lens,
                             dtype=w.dtype, num_kv_heads=w.num_kv_heads, block_size=w.block_size,
                             scale=w.scale, **kw)


def small_case(seed, dtype="f32", N=4, Hq=4, Hkv=2, D=8, B=4, lens=None, max_len=13):
    rng = np.random.default_rng(seed)
    if lens is None:
        lens = rng.integers(1, max_len, size=N, endpoint=True)
    return W.build_decode(f"small{seed}", seed=seed, dtype=dtype, seq_lens=lens, num_q_heads=Hq,
                          num_kv_heads=Hkv, head_size=D, block_size=B, pool_factor=1.5)


# ---------------------------------------------------------------------------

def pin_f16_decoding():
    """Exact binary16 -> double for all 65536 bit patterns, against numpy's conversion."""
    L = O.lib()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([L.pao_f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_bf16_decoding():
    """Exact bfloat16 -> double for all 65536 bit patterns, against torch's bfloat16."""
    import torch
    L = O.lib()
    bits = np.arange(65536, dtype=np.int64)
    ref = torch.tensor(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([L.pao_bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_35_token_example():
    """The page's 35-token request, B = 16, table [7, 3, 12]."""
    g = _golden("block_table_35_tokens.json")
    row = np.asarray(g["block_table"], dtype=np.int32)
    for rng_ in g["token_ranges"]:
        for slot, i in enumerate(range(rng_["first_token"], rng_["last_token"] + 1)):
            assert O.locate(row, g["block_size"], i) == (rng_["block"], slot), i
    # the tiny workload's 35-token sequence: attention through the table equals
    # brute force over the contiguous 35 x D key/value arrays laid out by hand
    w = W.tiny_f32()
    s = 3
    assert list(w.block_tables[s]) == g["block_table"] and w.seq_lens[s] == g["seq_len"]
    keys, vals = [], []
    for rng_ in g["token_ranges"]:
        keys.append(w.k_cache[rng_["block"], :, :rng_["slots_filled"], :].astype(np.float64))
        vals.append(w.v_cache[rng_["block"], :, :rng_["slots_filled"], :].astype(np.float64))
    K = np.concatenate(keys, axis=1)  # [H, 35, D]
    V = np.concatenate(vals, axis=1)
    out = _attn(w)
    for h in range(w.num_q_heads):
        sc = w.scale * (K[h] @ w.q[s, h].astype(np.float64))
        p = np.exp(sc - sc.max())
        ref = (p / p.sum()) @ V[h]
        assert np.max(np.abs(out[s, h] - ref)) < 1e-13


def pin_worked_offset():
    """Element offset 206880 of the page's worked example (prior-art key layout)."""
    g = _golden("worked_key_offset.json")
    e = g["expected"]
    row = np.asarray(g["block_table"], dtype=np.int32)
    blk, off = O.locate(row, g["block_size"], g["token"])
    assert (blk, off) == (e["physical_block_number"], e["physical_block_offset"])
    assert g["token"] // g["block_size"] == e["block_idx"]
    args = (g["num_kv_heads"], g["block_size"], g["head_size"], g["x"])
    assert O.key_offset_prior(1, 0, 0, 0, *args) == e["kv_block_stride"]
    assert O.key_offset_prior(0, 1, 0, 0, *args) == e["kv_head_stride"]
    assert O.key_offset_prior(blk, g["kv_head"], off, 0, *args) == e["k_ptr_offset"]


def pin_prior_layout_offsets():
    """The prior-art offsets agree with numpy's row-major indexing of the page's shapes."""
    rng = np.random.default_rng(7)
    for (Hkv, B, D, x) in [(32, 16, 128, 8), (3, 8, 32, 4), (2, 32, 64, 8)]:
        nb = 5
        kshape = (nb, Hkv, D // x, B, x)
        vshape = (nb, Hkv, D, B)
        for _ in range(200):
            b, h, o, d = (int(rng.integers(nb)), int(rng.integers(Hkv)), int(rng.integers(B)), int(rng.integers(D)))
            assert O.key_offset_prior(b, h, o, d, Hkv, B, D, x) == np.ravel_multi_index((b, h, d // x, o, d % x), kshape)
            assert O.value_offset_prior(b, h, o, d, Hkv, B, D) == np.ravel_multi_index((b, h, d, o), vshape)
            assert O.offset_ours(b, h, o, d, Hkv, B, D) == np.ravel_multi_index((b, h, o, d), (nb, Hkv, B, D))


def pin_prior_layout_attention():
    """The same logical cache in the prior-art layout and in ours gives identical attention."""
    for dtype, x in (("f16", 8), ("f32", 4)):
        w = small_case(11, dtype=dtype, N=3, Hq=4, Hkv=2, D=16, B=4)
        nb, H, B, D = w.k_cache.shape
        k_prior = np.ascontiguousarray(w.k_cache.reshape(nb, H, B, D // x, x).transpose(0, 1, 3, 2, 4))
        v_prior = np.ascontiguousarray(w.v_cache.transpose(0, 1, 3, 2))
        a = _attn(w)
        b = _attn(w, k=k_prior, v=v_prior, layout="prior")
        assert np.array_equal(a, b)


def pin_slot_round_trip():
    """Tokens appended through slot_mapping (slot = block * B + offset) are read back
    by attention at the positions the block table gives them."""
    rng = np.random.default_rng(5)
    for B in (1, 4, 16):
        w = W.build_decode("rt", seed=21 + B, dtype="f32", seq_lens=[1, B, 2 * B + 1, 3 * B - 1], num_q_heads=2,
                           num_kv_heads=2, head_size=8, block_size=B, pool_factor=2.0, append_last=True)
        k, v = w.k_cache.copy(), w.v_cache.copy()
        O.reshape_and_cache(k, v, w.new_key, w.new_value, w.slot_mapping, dtype="f32", num_kv_heads=2, block_size=B)
        out = _attn(w, k=k, v=v)
        assert not np.isnan(out).any()  # the appended slot started as NaN
        for s, L in enumerate(w.seq_lens):
            blk = int(w.block_tables[s, (L - 1) // B])
            assert np.array_equal(k[blk, :, (L - 1) % B, :], w.new_key[s])
            assert np.array_equal(v[blk, :, (L - 1) % B, :], w.new_value[s])
        # every slot in a pool maps to a distinct (block, offset)
        nb = 3
        kk = np.zeros((nb, 1, B, 1), np.float32)
        vv = np.zeros_like(kk)
        slots = rng.permutation(nb * B).astype(np.int64)
        key = np.arange(nb * B, dtype=np.float32).reshape(-1, 1, 1) + 1
        O.reshape_and_cache(kk, vv, key, key.copy(), slots, dtype="f32", num_kv_heads=1, block_size=B)
        assert sorted(kk.reshape(-1).tolist()) == list(range(1, nb * B + 1))
        for t, sl in enumerate(slots):
            assert kk[sl // B, 0, sl % B, 0] == t + 1


def pin_padding_slots_skipped():
    k = np.zeros((2, 1, 4, 2), np.float32)
    v = np.zeros_like(k)
    key = np.ones((3, 1, 2), np.float32)
    O.reshape_and_cache(k, v, key, key.copy(), np.array([-1, 5, -7], np.int64), dtype="f32", num_kv_heads=1,
                        block_size=4)
    assert k.sum() == 2 and k[1, 0, 1].tolist() == [1.0, 1.0]


def pin_identity_tables_vs_contiguous():
    """With identity tables the result is plain contiguous attention (numpy and torch SDPA in fp64)."""
    import torch
    for dtype in ("f32", "f16", "bf16"):
        N, Hq, Hkv, D, B = 3, 6, 2, 16, 8
        lens = [5, 16, 23]
        M = 3
        fixed = {s: list(range(s * M, s * M + -(-L // B))) for s, L in enumerate(lens)}
        w = W.build_decode("id", seed=31, dtype=dtype, seq_lens=lens, num_q_heads=Hq, num_kv_heads=Hkv,
                           head_size=D, block_size=B, num_blocks=N * M, fixed_tables=fixed, table_width=M)
        tables = np.arange(N * M, dtype=np.int32).reshape(N, M)
        out = _attn(w, tables=tables)
        Kc = O.to_f64(w.k_cache, dtype).reshape(N, M, Hkv, B, D).transpose(0, 2, 1, 3, 4).reshape(N, Hkv, M * B, D)
        Vc = O.to_f64(w.v_cache, dtype).reshape(N, M, Hkv, B, D).transpose(0, 2, 1, 3, 4).reshape(N, Hkv, M * B, D)
        Q = O.to_f64(w.q, dtype)
        G = Hq // Hkv
        for s, L in enumerate(lens):
            for h in range(Hq):
                Kh, Vh = Kc[s, h // G, :L], Vc[s, h // G, :L]
                sc = (Kh @ Q[s, h]) * w.scale
                p = np.exp(sc - sc.max())
                ref = (p / p.sum()) @ Vh
                assert np.max(np.abs(out[s, h] - ref)) < 1e-12
            qt = torch.from_numpy(Q[s][None, :, None, :])                     # [1, Hq, 1, D]
            kt = torch.from_numpy(np.repeat(Kc[s, :, :L], G, axis=0)[None])   # [1, Hq, L, D]
            vt = torch.from_numpy(np.repeat(Vc[s, :, :L], G, axis=0)[None])
            sd = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=w.scale)[0, :, 0].numpy()
            assert np.max(np.abs(out[s] - sd)) < 1e-12


def pin_permutation_invariance():
    """Relabelling physical blocks (moving their contents, rewriting tables) changes nothing."""
    for dtype in ("f32", "bf16"):
        w = small_case(41, dtype=dtype, N=5, Hq=4, Hkv=4, D=8, B=4, max_len=30)
        base = _attn(w)
        rng = np.random.default_rng(42)
        perm = rng.permutation(w.num_blocks)               # block b moves to perm[b]
        k = np.empty_like(w.k_cache); k[perm] = w.k_cache
        v = np.empty_like(w.v_cache); v[perm] = w.v_cache
        tables = perm[w.block_tables].astype(np.int32)
        assert np.array_equal(_attn(w, k=k, v=v, tables=tables), base)


def pin_shared_prefix_equals_private():
    """Branches that share prefix blocks give the same outputs as the same branches
    holding private copies of the prefix."""
    w = W.shared_prefix_f16(num_prompts=2, branches=3, prefix_len=20, max_suffix=9, num_heads=2, block_size=4,
                            num_blocks=64, seed=77)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    O.copy_blocks(k, v, w.copy_pairs, dtype="f16", num_kv_heads=2, block_size=4, head_size=128)
    O.reshape_and_cache(k, v, w.new_key, w.new_value, w.slot_mapping, dtype="f16", num_kv_heads=2, block_size=4)
    shared = _attn(w, k=k, v=v)
    # private layout: every (seq, logical block) gets its own fresh physical block
    N, M = w.block_tables.shape
    kp = W.nan_array((N * M,) + k.shape[1:], "f16")
    vp = W.nan_array((N * M,) + v.shape[1:], "f16")
    tables = np.arange(N * M, dtype=np.int32).reshape(N, M)
    for s in range(N):
        for j in range(-(-int(w.seq_lens[s]) // 4)):
            kp[tables[s, j]] = k[w.block_tables[s, j]]
            vp[tables[s, j]] = v[w.block_tables[s, j]]
    private = O.paged_attention(w.q, kp, vp, tables, w.seq_lens, dtype="f16", num_kv_heads=2, block_size=4,
                                scale=w.scale)
    assert np.array_equal(shared, private)
    # blocks really are shared: some physical block appears in several tables
    ids, counts = np.unique(w.block_tables[:, 0], return_counts=True)
    assert counts.max() == 3


def pin_cow_isolation():
    """After the copy-on-write copies and the suffix appends, every block that is
    neither a copy destination nor a freshly appended block is byte-identical,
    so no branch's writes reach a block another branch reads."""
    w = W.shared_prefix_f16(num_prompts=2, branches=4, prefix_len=18, max_suffix=7, num_heads=2, block_size=4,
                            num_blocks=80, seed=78)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    O.copy_blocks(k, v, w.copy_pairs, dtype="f16", num_kv_heads=2, block_size=4, head_size=128)
    dsts = set(int(d) for d in w.copy_pairs[:, 1])
    for src, dst in w.copy_pairs:
        assert np.array_equal(k[dst].view(np.uint16), w.k_cache[src].view(np.uint16))
        assert np.array_equal(v[dst].view(np.uint16), w.v_cache[src].view(np.uint16))
    before_k, before_v = k.copy(), v.copy()
    O.reshape_and_cache(k, v, w.new_key, w.new_value, w.slot_mapping, dtype="f16", num_kv_heads=2, block_size=4)
    written = set(int(s) // 4 for s in w.slot_mapping)
    shared = set()
    for s in range(w.num_seqs):
        shared.update(int(b) for b in w.block_tables[s, :18 // 4])  # full prefix blocks, still shared
    assert not written & shared
    for b in range(w.num_blocks):
        if b not in written:
            assert np.array_equal(k[b].view(np.uint16), before_k[b].view(np.uint16)), b
            assert np.array_equal(v[b].view(np.uint16), before_v[b].view(np.uint16)), b
    # the partial last prefix block (18 = 4*4 + 2) was copied, and the branch's
    # first suffix tokens land in its private copy, not in the shared original
    last = 18 // 4
    for s in range(w.num_seqs):
        assert int(w.block_tables[s, last]) in dsts
    for src in set(int(a) for a in w.copy_pairs[:, 0]):
        assert np.array_equal(k[src].view(np.uint16), w.k_cache[src].view(np.uint16))


def pin_brute_force():
    """The C oracle equals an independent pure-Python evaluation on tiny inputs."""
    cases = [
        dict(seed=1, dtype="f32", N=3, Hq=2, Hkv=2, D=4, B=4),
        dict(seed=2, dtype="f16", N=4, Hq=4, Hkv=2, D=8, B=2),
        dict(seed=3, dtype="bf16", N=2, Hq=8, Hkv=1, D=4, B=8),
        dict(seed=4, dtype="f32", N=3, Hq=6, Hkv=3, D=8, B=1, max_len=9),
        dict(seed=5, dtype="f16", N=3, Hq=2, Hkv=1, D=8, B=4, lens=[0, 1, 17]),
    ]
    for c in cases:
        w = small_case(**c)
        got = _attn(w)
        ref = np.array(brute.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=w.dtype,
                                             num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale))
        assert np.max(np.abs(got - ref)) < 1e-12, c


def pin_special_cases():
    """L = 1 gives v_0 exactly; identical keys give mean(v); one dominant score gives v_0."""
    w = small_case(61, dtype="f32", N=2, Hq=2, Hkv=2, D=8, B=4, lens=[1, 9])
    out = _attn(w)
    blk = int(w.block_tables[0, 0])
    assert np.array_equal(out[0], w.v_cache[blk, :, 0, :].astype(np.float64))
    # identical keys in every token of seq 1
    k = w.k_cache.copy()
    L = int(w.seq_lens[1])
    k0 = w.k_cache[int(w.block_tables[1, 0]), :, 0, :].copy()
    vals = []
    for i in range(L):
        b, o = int(w.block_tables[1, i // 4]), i % 4
        k[b, :, o, :] = k0
        vals.append(w.v_cache[b, :, o, :].astype(np.float64))
    out = _attn(w, k=k)
    assert np.max(np.abs(out[1] - np.mean(vals, axis=0))) < 1e-14
    # one dominant score: key 0 aligned with q and scaled up
    k2 = w.k_cache.copy()
    b0 = int(w.block_tables[1, 0])
    k2[b0, :, 0, :] = w.q[1] * np.float32(1000.0)
    out = _attn(w, k=k2)
    assert np.max(np.abs(out[1] - w.v_cache[b0, :, 0, :].astype(np.float64))) < 1e-12


def pin_split_identity():
    """Partition-then-merge equals the unsplit softmax."""
    for dtype in ("f32", "bf16"):
        w = small_case(71, dtype=dtype, N=4, Hq=4, Hkv=2, D=8, B=4, lens=[1, 7, 33, 64])
        base = _attn(w)
        for P in (4, 8, 12, 64, 1000):
            assert np.max(np.abs(_attn(w, partition_size=P) - base)) < 1e-12, P


def pin_zero_length():
    w = small_case(81, dtype="f32", N=3, Hq=2, Hkv=2, D=4, B=4, lens=[0, 3, 0])
    out = _attn(w)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and not np.isnan(out).any()


def pin_bad_block_rejected():
    w = small_case(91, dtype="f32", N=2, Hq=2, Hkv=2, D=4, B=4, lens=[5, 3])
    t = w.block_tables.copy()
    t[0, 1] = w.num_blocks + 3
    try:
        _attn(w, tables=t)
    except O.OracleError:
        return
    raise AssertionError("out-of-range block id was accepted")


def pin_alibi():
    """ALiBi (per-head slope, score_i += slope * (i - (L - 1))): zero slopes change
    nothing, the C oracle equals the pure-Python evaluation, a steep slope leaves
    only the newest token, and the partitioned form still equals the unsplit one."""
    w = small_case(101, dtype="f16", N=3, Hq=4, Hkv=2, D=8, B=4, lens=[1, 9, 23])
    base = _attn(w)
    assert np.array_equal(_attn(w, alibi_slopes=np.zeros(4)), base)
    slopes = np.array([0.5, -0.25, 2.0, 0.125])
    got = _attn(w, alibi_slopes=slopes)
    ref = np.array(brute.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=w.dtype,
                                         num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale,
                                         alibi_slopes=slopes))
    assert np.max(np.abs(got - ref)) < 1e-12
    assert np.max(np.abs(got - base)) > 1e-3          # the bias really acts
    steep = _attn(w, alibi_slopes=np.full(4, 1e4))
    for s, L in enumerate(w.seq_lens):
        blk, off = int(w.block_tables[s, (L - 1) // 4]), (L - 1) % 4
        newest = O.to_f64(w.v_cache[blk, :, off, :], "f16")       # [Hkv, D]
        for h in range(4):
            assert np.max(np.abs(steep[s, h] - newest[h // 2])) < 1e-12
    for P in (4, 8):
        assert np.max(np.abs(_attn(w, alibi_slopes=slopes, partition_size=P) - got)) < 1e-12


def _prefill_case(seed, dtype="f32", lens=(9, 20, 13), chunks=(9, 6, 1), Hq=4, Hkv=2, D=8, B=4):
    w = W.build_decode(f"pf{seed}", seed=seed, dtype=dtype, seq_lens=list(lens), num_q_heads=Hq, num_kv_heads=Hkv,
                       head_size=D, block_size=B, pool_factor=1.5)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = W.normal(np.random.default_rng(seed + 1), (int(qs[-1]), Hq, D), dtype)
    return w, q, qs


def _prefill(w, q, qs, **kw):
    return O.prefill_attention(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, qs, dtype=w.dtype,
                               num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale, **kw)


def pin_prefill():
    """Chunked prefill: one query = decode over the whole context (bit-identical),
    a chunk's last query = decode, the query at position 0 returns v_0, and the
    pure-Python evaluation agrees to 1e-12."""
    w, q, qs = _prefill_case(121, "f16", lens=(9, 20, 13), chunks=(9, 6, 1))
    got = _prefill(w, q, qs)
    ref = np.array(brute.prefill_attention(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, qs, dtype=w.dtype,
                                           num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale))
    assert np.max(np.abs(got - ref)) < 1e-12
    # the last query of every chunk is the decode query of that sequence
    last = q[qs[1:] - 1]
    dec = O.paged_attention(last, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=w.dtype,
                            num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
    assert np.array_equal(got[qs[1:] - 1], dec)
    # sequence 0's chunk starts at position 0: its first query sees token 0 only
    blk = int(w.block_tables[0, 0])
    v0 = O.to_f64(w.v_cache[blk, :, 0, :], w.dtype)
    for h in range(w.num_q_heads):
        assert np.array_equal(got[0, h], v0[h // 2])


def pin_prefill_contiguous():
    """With identity tables the chunk equals causal attention over contiguous K/V
    (numpy with an explicit causal mask, and torch SDPA with a boolean mask, fp64)."""
    import torch
    N, M, B, Hq, Hkv, D = 2, 4, 4, 4, 2, 8
    lens, chunks = [13, 16], [5, 16]
    fixed = {s: list(range(s * M, s * M + -(-L // B))) for s, L in enumerate(lens)}
    w = W.build_decode("pfc", seed=131, dtype="f32", seq_lens=lens, num_q_heads=Hq, num_kv_heads=Hkv, head_size=D,
                       block_size=B, num_blocks=N * M, fixed_tables=fixed, table_width=M)
    tables = np.arange(N * M, dtype=np.int32).reshape(N, M)
    qs = np.array([0, 5, 21], np.int32)
    q = W.normal(np.random.default_rng(132), (21, Hq, D), "f32")
    got = O.prefill_attention(q, w.k_cache, w.v_cache, tables, w.seq_lens, qs, dtype="f32", num_kv_heads=Hkv,
                              block_size=B, scale=w.scale)
    Kc = w.k_cache.astype(np.float64).reshape(N, M, Hkv, B, D).transpose(0, 2, 1, 3, 4).reshape(N, Hkv, M * B, D)
    Vc = w.v_cache.astype(np.float64).reshape(N, M, Hkv, B, D).transpose(0, 2, 1, 3, 4).reshape(N, Hkv, M * B, D)
    for s, (L, n) in enumerate(zip(lens, chunks)):
        Q = q[qs[s]:qs[s + 1]].astype(np.float64)               # [n, Hq, D]
        pos = np.arange(L - n, L)
        mask = np.arange(L)[None, :] <= pos[:, None]             # [n, L]
        for h in range(Hq):
            sc = (Q[:, h] @ Kc[s, h // 2, :L].T) * w.scale
            sc = np.where(mask, sc, -np.inf)
            pr = np.exp(sc - sc.max(axis=1, keepdims=True))
            ref = (pr / pr.sum(axis=1, keepdims=True)) @ Vc[s, h // 2, :L]
            assert np.max(np.abs(got[qs[s]:qs[s + 1], h] - ref)) < 1e-12
        qt = torch.from_numpy(Q.transpose(1, 0, 2)[None])                               # [1, Hq, n, D]
        kt = torch.from_numpy(np.repeat(Kc[s, :, :L], 2, axis=0)[None])
        vt = torch.from_numpy(np.repeat(Vc[s, :, :L], 2, axis=0)[None])
        sd = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask),
                                                              scale=w.scale)[0].numpy().transpose(1, 0, 2)
        assert np.max(np.abs(got[qs[s]:qs[s + 1]] - sd)) < 1e-12


# --------------------------------------------------------------------------- FP8 (E4M3) cache

def pin_e4m3_codes():
    """All 256 E4M3 codes against torch.float8_e4m3fn and against the pure-Python
    decoding from the fields; textbook values: 0x38 = 1, 0x7E = 448 (largest),
    0x08 = 2^-6 (smallest normal), 0x01 = 2^-9 (smallest subnormal), 0x7F NaN."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    got = O.to_f64(codes, "fp8")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    py = np.array([brute.e4m3_value(int(c)) for c in codes])
    assert np.array_equal(py[~nan], got[~nan])
    assert (O.e4m3_to_f64(0x38), O.e4m3_to_f64(0x7E), O.e4m3_to_f64(0x08), O.e4m3_to_f64(0x01)) == \
        (1.0, 448.0, 2.0 ** -6, 2.0 ** -9)
    assert math.isnan(O.e4m3_to_f64(0x7F)) and O.e4m3_to_f64(0xB8) == -1.0


def pin_e4m3_rounding():
    """Writing x / scale as a code: torch's round-to-nearest-even conversion for
    |r| < 464 (random values over the whole range, exact ties between codes,
    subnormal ties), saturation to +-448 from there on (torch turns those into
    NaN instead), and every finite code maps back to itself."""
    import torch
    rng = np.random.default_rng(171)
    r = np.concatenate([rng.standard_normal(4000) * 60, rng.standard_normal(2000) * 0.02,
                        np.ldexp(rng.uniform(1, 2, 2000), rng.integers(-12, 9, 2000))]).astype(np.float32)
    finite = np.array([c for c in range(256) if not math.isnan(brute.e4m3_value(c))], dtype=np.uint8)
    vals = np.array([brute.e4m3_value(int(c)) for c in finite])
    mids = np.unique(np.abs(vals))
    ties = ((mids[:-1] + mids[1:]) / 2).astype(np.float32)  # exact midpoints: ties to the even code
    r = np.concatenate([r, ties, -ties, np.float32([447.9, 448.0, 449.0, 463.99, -463.99])])
    r = r[np.abs(r) < 464]
    ref = torch.from_numpy(r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.quantize_e4m3(r), ref)
    assert list(O.quantize_e4m3(np.float32([464.0, 480.0, 1e6, np.inf, -500.0, -np.inf]))) == [0x7E] * 4 + [0xFE] * 2
    assert np.array_equal(O.quantize_e4m3(vals.astype(np.float32)), finite)


def _fp8_case(seed, k_scale, v_scale, lens=None, Hq=4, Hkv=2, D=8, B=16):
    w = small_case(seed, "f16", Hq=Hq, Hkv=Hkv, D=D, B=B, lens=lens)
    kc = O.quantize_cache_fp8(w.k_cache, k_scale, values=False)
    vc = O.quantize_cache_fp8(w.v_cache, v_scale, values=True)
    return w, kc, vc


def pin_fp8_attention():
    """FP8 attention is the definition on the dequantised caches: with power-of-two
    scales it equals, bit for bit, the float32 evaluation of k_scale * e4m3(code)
    (the value pool taken back to [B][D] with numpy); with any scales it
    agrees with the pure-Python brute force to 1e-12, and its split form with the
    unsplit one."""
    ks, vs = 2.0 ** -5, 2.0 ** -3
    w, kc, vc = _fp8_case(181, ks, vs, B=16)
    assert vc.shape[2:] == (1, w.head_size, 16)
    got = O.paged_attention_fp8(w.q, kc, vc, w.block_tables, w.seq_lens, num_kv_heads=w.num_kv_heads,
                                block_size=w.block_size, scale=w.scale, k_scale=ks, v_scale=vs)
    kd = (O.to_f64(kc, "fp8") * ks).astype(np.float32)
    vd = O.values_from_fp8_layout((O.to_f64(vc, "fp8") * vs).astype(np.float32))
    ref = O.paged_attention(w.q.astype(np.float32), kd, vd, w.block_tables, w.seq_lens, dtype="f32",
                            num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
    assert np.array_equal(got, ref)
    ks, vs = 0.0113, 0.0371
    w, kc, vc = _fp8_case(182, ks, vs, lens=[1, 6, 19, 40], B=32)
    kw = dict(num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale, k_scale=ks, v_scale=vs)
    got = O.paged_attention_fp8(w.q, kc, vc, w.block_tables, w.seq_lens, **kw)
    bf = np.array(brute.paged_attention_fp8(w.q, kc, vc, w.block_tables, w.seq_lens, **kw))
    assert np.max(np.abs(got - bf)) < 1e-12
    split = O.paged_attention_fp8(w.q, kc, vc, w.block_tables, w.seq_lens, partition_size=4, **kw)
    assert np.max(np.abs(got - split)) < 1e-12


def pin_fp8_append():
    """The FP8 append writes the code of x / scale (fp32 division; torch's
    conversion for in-range values) of token t's key at [block][head][offset][d]
    and of its value at [block][head][offset / 16][d][offset % 16]; padding slots
    are skipped and every other byte is left as it was."""
    import torch
    rng = np.random.default_rng(191)
    Hkv, D, B, nb = 2, 16, 32, 3
    kc = rng.integers(0, 256, size=(nb, Hkv, B, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(nb, Hkv, B // 16, D, 16), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    key = (rng.standard_normal((5, Hkv, D)) * 2).astype(np.float16)
    val = (rng.standard_normal((5, Hkv, D)) * 2).astype(np.float16)
    slots = np.array([7, -1, 0, 53, 90], dtype=np.int64)
    ks, vs = 0.0231, 2.0 ** -4
    assert np.abs(key.astype(np.float32) / np.float32(ks)).max() < 448  # torch's conversion saturates nowhere here
    O.reshape_and_cache_fp8(kc, vc, key, val, slots, num_kv_heads=Hkv, block_size=B, k_scale=ks, v_scale=vs)
    kq = torch.from_numpy(key.astype(np.float32) / np.float32(ks)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vq = torch.from_numpy(val.astype(np.float32) / np.float32(vs)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        b, off = sl // B, sl % B
        k0[b, :, off, :] = kq[t]
        v0[b, :, off // 16, :, off % 16] = vq[t]
    assert np.array_equal(kc, k0) and np.array_equal(vc, v0)


def pin_prefill_dense():
    """The numpy float64 form of chunked prefill (library matmuls, used for the benchmark-size
    GPU checks) equals the C oracle and the pure-Python brute force on small cases: GQA and
    MHA, f16/bf16/f32, block sizes 4 and 16, chunks of one token, of a whole sequence and
    ragged ones."""
    from oracle import dense

    def both(w, q, qs):
        kw = dict(dtype=w.dtype, num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
        return (dense.prefill_attention(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, qs, **kw),
                _prefill(w, q, qs))

    w, q, qs = _prefill_case(141, "bf16", lens=(9, 20, 13), chunks=(9, 6, 1))
    got, ref = both(w, q, qs)
    assert np.max(np.abs(got - ref)) < 1e-12
    tiny = np.array(brute.prefill_attention(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, qs, dtype=w.dtype,
                                            num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale))
    assert np.max(np.abs(got - tiny)) < 1e-12
    for seed, dtype, Hq, Hkv, B in ((142, "f16", 8, 2, 16), (143, "f32", 3, 3, 4), (144, "bf16", 16, 2, 16)):
        w, q, qs = _prefill_case(seed, dtype, lens=(40, 70, 5, 33), chunks=(40, 17, 0, 1), Hq=Hq, Hkv=Hkv, D=16,
                                 B=B)
        got, ref = both(w, q, qs)
        assert np.max(np.abs(got - ref)) < 1e-12


ALL_PINS = [
    pin_f16_decoding, pin_bf16_decoding, pin_35_token_example, pin_worked_offset, pin_prior_layout_offsets,
    pin_prior_layout_attention, pin_slot_round_trip, pin_padding_slots_skipped, pin_identity_tables_vs_contiguous,
    pin_permutation_invariance, pin_shared_prefix_equals_private, pin_cow_isolation, pin_brute_force,
    pin_special_cases, pin_split_identity, pin_zero_length, pin_bad_block_rejected, pin_alibi, pin_prefill,
    pin_prefill_contiguous, pin_prefill_dense, pin_e4m3_codes, pin_e4m3_rounding, pin_fp8_attention, pin_fp8_append,
]
