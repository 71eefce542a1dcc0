"""FP8 (E4M3) KV cache: the quantising append and decode attention vs the CPU oracle (needs a GB300).

Reading ("PagedAttention 详解：缓存的存储结构", section "软件地址翻译": cache_t may be
FP8): a key code c stands for k_scale * e4m3(c), a value code for v_scale *
e4m3(c); values are stored [blocks][kv_heads][B/16][D][16] (the pages' [D][B]
value layout tiled in 16-token groups); queries and outputs are fp16.  Both sides quantise nothing on their own for the attention tests: the
host pools are turned into codes once by the oracle's quantiser and the same
bytes go to the GPU.

Bars: the append is bit-exact over the whole pools (untouched bytes included);
attention outputs are within the per-element bound of ``harness.bound`` for
fp16 outputs (3e-3, or half an output ulp + 2^-12 where |out| >= 1).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from harness import out_f64, rising_keys, to_numpy_storage, to_torch, within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    return pa


def u8(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def fp8_pools(w: W.Workload, k_scale: float, v_scale: float):
    """Host code pools of a workload's fp16 pools (NaN slots become NaN codes)."""
    return (O.quantize_cache_fp8(w.k_cache, k_scale, values=False),
            O.quantize_cache_fp8(w.v_cache, v_scale, values=True))


class Fp8Step:
    def __init__(self, w: W.Workload, k_scale: float, v_scale: float, device="cuda"):
        import torch
        import paged_kv_cache_32_gb300 as pa
        self.w, self.pa, self.ks, self.vs = w, pa, k_scale, v_scale
        self.kc_host, self.vc_host = fp8_pools(w, k_scale, v_scale)
        self.k, self.v = u8(self.kc_host), u8(self.vc_host)
        self.q = to_torch(w.q, "f16", device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.desc = pa.cache_desc(self.k)
        self.slots = torch.from_numpy(w.slot_mapping).to(device) if w.slot_mapping is not None else None
        self.nk = to_torch(w.new_key, "f16", device) if w.new_key is not None else None
        self.nv = to_torch(w.new_value, "f16", device) if w.new_value is not None else None

    def append(self):
        if self.slots is not None and len(self.slots):
            self.pa.pa_reshape_and_cache_fp8(self.k, self.v, self.nk, self.nv, self.slots, self.ks, self.vs,
                                             err_flag=self.err, desc=self.desc)

    def decode(self, partition_size=None, alibi=None):
        import torch
        part = self.w.partition_size if partition_size is None else partition_size
        self.pa.pa_decode(self.out, self.q, self.k, self.v, self.tables, self.lens, self.w.scale,
                          partition_size=part, err_flag=self.err, desc=self.desc, k_scale=self.ks,
                          v_scale=self.vs, alibi_slopes=alibi)
        torch.cuda.synchronize()
        return out_f64(self.out)

    def host_after_append(self):
        k, v = self.kc_host.copy(), self.vc_host.copy()
        if self.w.slot_mapping is not None and len(self.w.slot_mapping):
            O.reshape_and_cache_fp8(k, v, self.w.new_key, self.w.new_value, self.w.slot_mapping,
                                    num_kv_heads=self.w.num_kv_heads, block_size=self.w.block_size,
                                    k_scale=self.ks, v_scale=self.vs)
        return k, v

    def oracle(self, k, v, partition_size=0, alibi=None):
        w = self.w
        return O.paged_attention_fp8(w.q, k, v, w.block_tables, w.seq_lens, num_kv_heads=w.num_kv_heads,
                                     block_size=w.block_size, scale=w.scale, k_scale=self.ks, v_scale=self.vs,
                                     partition_size=partition_size, alibi_slopes=alibi)


def assert_close(got, ref, what):
    assert not np.isnan(got).any(), f"{what}: NaN in output"
    ok, err, ratio = within_bound(got, ref, "f16")
    assert ok, f"{what}: max abs err {err}, worst err/bound {ratio}"
    return err


# ---------------------------------------------------------------- running maxima that move and stay
@pytest.mark.parametrize("partition", [0, 64])
def test_fp8_rising_scores_running_max(partition):
    """Scores rising along each sequence by about 8 (log2 units) per 32-token slab: the FP8 kernel's
    running maxima move on the slabs whose scores exceed them by more than 8 and stay on the others."""
    w = W.build_decode("fp8_rising", seed=7710, dtype="f16", seq_lens=[1, 32, 33, 300, 1000, 2100],
                       num_q_heads=16, num_kv_heads=2, head_size=128, block_size=32, append_last=True)
    rising_keys(w, 0.015, seed=7711)
    g = Fp8Step(w, 0.5, 0.02)
    g.append()
    k, v = g.host_after_append()
    got = g.decode(partition_size=partition)
    assert int(g.err.item()) == 0
    assert_close(got, g.oracle(k, v), f"fp8 rising, partition {partition}")


# ---------------------------------------------------------------- the append, bit-exact
def test_fp8_append_bit_exact():
    """Random fp16 rows spanning the E4M3 range after scaling, saturating values, ±inf
    and subnormal-range values; padding slots; every byte of both pools compared."""
    import torch
    import paged_kv_cache_32_gb300 as pa
    rng = np.random.default_rng(301)
    nb, hkv, B, D, T = 12, 4, 32, 128, 40
    kc = rng.integers(0, 256, size=(nb, hkv, B, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(nb, hkv, B // 16, D, 16), dtype=np.uint8)
    key = (rng.standard_normal((T, hkv, D)) * np.exp(rng.uniform(-9, 3, (T, hkv, D)))).astype(np.float16)
    val = (rng.standard_normal((T, hkv, D)) * 4).astype(np.float16)
    key[0, 0, :4] = [np.inf, -np.inf, 60000.0, -6.0]          # saturate with k_scale below
    val[1, 1, :3] = [1e-7, -3e-8, 0.0]
    slots = rng.permutation(nb * B)[:T].astype(np.int64)
    slots[[3, 17]] = -1
    ks, vs = 0.0123, 0.0117
    k_dev, v_dev = u8(kc), u8(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache_fp8(k_dev, v_dev, to_torch(key, "f16"), to_torch(val, "f16"), u8(slots), ks, vs,
                                err_flag=err, desc=pa.cache_desc(k_dev))
    torch.cuda.synchronize()
    O.reshape_and_cache_fp8(kc, vc, key, val, slots, num_kv_heads=hkv, block_size=B, k_scale=ks, v_scale=vs)
    assert int(err.item()) == 0
    assert np.array_equal(k_dev.cpu().numpy(), kc)
    assert np.array_equal(v_dev.cpu().numpy(), vc)


def test_fp8_append_bad_slot_reported():
    import torch
    import paged_kv_cache_32_gb300 as pa
    k_dev = torch.zeros((2, 1, 16, 128), dtype=torch.uint8, device="cuda")
    v_dev = torch.zeros((2, 1, 1, 128, 16), dtype=torch.uint8, device="cuda")
    key = torch.ones((2, 1, 128), dtype=torch.float16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([5, 2 * 16 + 3], dtype=torch.int64, device="cuda")
    pa.pa_reshape_and_cache_fp8(k_dev, v_dev, key, key, slots, 1.0, 1.0, err_flag=err, desc=pa.cache_desc(k_dev))
    torch.cuda.synchronize()
    assert int(err.item()) == 2
    assert int(k_dev[0, 0, 5, 0].item()) == 0x38 and int(v_dev[0, 0, 0, 7, 5].item()) == 0x38  # 1.0 written
    assert int(k_dev.sum().item()) == 0x38 * 128 and int(v_dev.sum().item()) == 0x38 * 128


# ---------------------------------------------------------------- decode, small cases
@pytest.mark.parametrize("block_size", [16, 32, 48, 64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2), (32, 2)])
def test_fp8_decode_small(block_size, hq, hkv):
    """Ragged lengths (1, 15, 16, 17, 100, 300, 777) across several slabs and partitions.  B = 48
    puts the two 16-token halves of some slabs in different blocks (two copies each); multiples
    of 32 fetch a slab as one key box and one value run."""
    w = W.build_decode(f"fp8_b{block_size}_{hq}x{hkv}", seed=311 + block_size + hq, dtype="f16",
                       seq_lens=[1, 15, 16, 17, 100, 300, 777], num_q_heads=hq, num_kv_heads=hkv, head_size=128,
                       block_size=block_size, pool_factor=1.3)
    g = Fp8Step(w, 0.0123, 0.0117)
    k, v = g.host_after_append()
    for part in (0, 2 * block_size, 4 * block_size, 16 * block_size):  # explicit sizes are whole blocks
        got = g.decode(partition_size=part)
        assert int(g.err.item()) == 0
        err = assert_close(got, g.oracle(k, v), f"{w.name} partition {part}")
    print(w.name, "max abs err", err)


def test_fp8_merge_many_partitions():
    """One 16-token block per partition: 157, 69, 2 and 65 partitions in one launch."""
    w = W.build_decode("fp8_many_parts", seed=371, dtype="f16", seq_lens=[2500, 1100, 17, 0, 1040], num_q_heads=16,
                       num_kv_heads=2, head_size=128, block_size=16, pool_factor=1.2)
    g = Fp8Step(w, 0.0123, 0.0117)
    k, v = g.host_after_append()
    got = g.decode(partition_size=16)
    assert int(g.err.item()) == 0
    assert_close(got, g.oracle(k, v), "fp8, one block per partition")


def test_fp8_decode_alibi():
    w = W.build_decode("fp8_alibi", seed=331, dtype="f16", seq_lens=[5, 33, 500], num_q_heads=16, num_kv_heads=2,
                       head_size=128, block_size=16, pool_factor=1.3)
    import torch
    slopes = np.array([2.0 ** (-8.0 * (i + 1) / 16) for i in range(16)])
    g = Fp8Step(w, 0.02, 0.015)
    k, v = g.host_after_append()
    got = g.decode(alibi=torch.tensor(slopes, dtype=torch.float32, device="cuda"))
    assert_close(got, g.oracle(k, v, alibi=slopes), "fp8 + alibi")


def test_fp8_bad_block_id_reported():
    import torch
    w = W.build_decode("fp8_badid", seed=341, dtype="f16", seq_lens=[40, 40], num_q_heads=4, num_kv_heads=4,
                       head_size=128, block_size=16, pool_factor=1.5)
    g = Fp8Step(w, 0.0123, 0.0117)
    tables = w.block_tables.copy()
    tables[1, 1] = w.num_blocks + 3
    g.tables.copy_(torch.from_numpy(tables))
    got = g.decode()
    assert int(g.err.item()) == 1
    k, v = g.host_after_append()
    ref = g.oracle(k, v)
    assert_close(got[0], ref[0], "the sequence with valid blocks")


def test_fp8_copy_blocks_bit_exact():
    """Copy-on-write of whole blocks moves the FP8 bytes of both pools (values tiled) unchanged."""
    import torch
    import paged_kv_cache_32_gb300 as pa
    rng = np.random.default_rng(351)
    kc = rng.integers(0, 256, size=(10, 2, 32, 128), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(10, 2, 2, 128, 16), dtype=np.uint8)
    pairs = np.array([[1, 7], [4, 2], [9, 0]], dtype=np.int32)
    k_dev, v_dev = u8(kc), u8(vc)
    pa.pa_copy_blocks(k_dev, v_dev, u8(pairs), desc=pa.cache_desc(k_dev))
    torch.cuda.synchronize()
    for s, d in pairs:
        kc[d] = kc[s]
        vc[d] = vc[s]
    assert np.array_equal(k_dev.cpu().numpy(), kc) and np.array_equal(v_dev.cpu().numpy(), vc)


def test_fp8_long_context_split():
    """Two 8192-token sequences (B = 64) in 512-token partitions merged by the
    log-sum-exp kernel, GQA 4:1, scores scaled up so the running max moves late."""
    w = W.build_decode("fp8_long", seed=361, dtype="f16", seq_lens=[8192, 6001], num_q_heads=8, num_kv_heads=2,
                       head_size=128, block_size=64, pool_factor=1.1, partition_size=512)
    w.q = (w.q.astype(np.float32) * 3).astype(np.float16)
    g = Fp8Step(w, 0.0123, 0.0117)
    k, v = g.host_after_append()
    got = g.decode()
    assert int(g.err.item()) == 0
    assert_close(got, g.oracle(k, v, partition_size=512), "fp8 long context")


# ---------------------------------------------------------------- the full-size workloads
@pytest.mark.parametrize("name", ["mha_fp8", "gqa_fp8"])
def test_fp8_full_workload(name):
    """The whole step as the benchmark runs it: one appended token per sequence
    (mha) through the FP8 append, then decode; every output compared."""
    w = W.WORKLOADS[name]()
    g = Fp8Step(w, w.info["k_scale"], w.info["v_scale"])
    g.append()
    k, v = g.host_after_append()
    assert np.array_equal(g.k.cpu().numpy(), k) and np.array_equal(g.v.cpu().numpy(), v)
    got = g.decode()
    assert int(g.err.item()) == 0
    ref = g.oracle(k, v)
    err = assert_close(got, ref, name)
    if np.max(np.abs(ref)) < 1.0:
        assert err <= 3e-3
    print(name, "max abs err", err)


def test_fp8_decode_append_full_workload():
    """The benchmarked MHA FP8 step at full size: one pa_decode_append call, whose CTAs quantise and
    attend each sequence's new token, with the last sequences of the grid in half-size partitions.  Both
    pools equal the oracle's quantising append bit for bit, every output meets the oracle, and the output
    equals pa_reshape_and_cache_fp8 followed by pa_decode bit for bit."""
    import torch
    w = W.WORKLOADS["mha_fp8"]()
    fused = Fp8Step(w, w.info["k_scale"], w.info["v_scale"])
    fused.pa.pa_decode_append(fused.out, fused.q, fused.k, fused.v, fused.nk, fused.nv, fused.tables, fused.lens,
                              w.scale, partition_size=w.partition_size, err_flag=fused.err, desc=fused.desc,
                              k_scale=fused.ks, v_scale=fused.vs)
    torch.cuda.synchronize()
    assert int(fused.err.item()) == 0
    k, v = fused.host_after_append()
    assert np.array_equal(fused.k.cpu().numpy(), k) and np.array_equal(fused.v.cpu().numpy(), v)
    assert_close(out_f64(fused.out), fused.oracle(k, v), "mha_fp8 fused")
    two = Fp8Step(w, w.info["k_scale"], w.info["v_scale"])
    two.append()
    two.decode()
    assert int(two.err.item()) == 0
    assert torch.equal(fused.out.view(torch.int16), two.out.view(torch.int16))


# ---------------------------------------------------------------- the decode step with its quantising append fused in
APPEND_FP8 = [  # Hq, Hkv, B, lens (the last token of each sequence is the step's new token)
    (32, 32, 16, [1, 2, 15, 16, 17, 31, 32, 33, 700, 2048, 0]),  # B 16: a slab's halves in two blocks
    (64, 8, 32, [1, 33, 64, 65, 1500, 4096]),                     # B 32: whole slabs, G 8
    (24, 2, 48, [1, 47, 48, 49, 300]),                            # B 48, G 12: two head groups, the first writes
]


@pytest.mark.parametrize("case", APPEND_FP8, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-B{c[2]}")
@pytest.mark.parametrize("split", ["default", "smallest"])
def test_fp8_decode_append_fused(case, split):
    """pa_decode_append over an FP8 cache quantises each sequence's new fp16 row into the slot at
    position L - 1 (which starts as NaN codes) and attends over it in one launch: both pools equal the
    oracle's quantising append bit for bit, the output meets the oracle, and it equals
    pa_reshape_and_cache_fp8 followed by pa_decode bit for bit."""
    import torch
    hq, hkv, B, lens = case
    w = W.build_decode(f"fp8_append_{hq}x{hkv}_b{B}", seed=401 + B + hq, dtype="f16", seq_lens=lens, num_q_heads=hq,
                       num_kv_heads=hkv, head_size=128, block_size=B, pool_factor=1.3, append_last=True)
    part = 0 if split == "default" else B
    fused, two = Fp8Step(w, 0.0123, 0.0117), Fp8Step(w, 0.0123, 0.0117)
    fused.pa.pa_decode_append(fused.out, fused.q, fused.k, fused.v, fused.nk, fused.nv, fused.tables, fused.lens,
                              w.scale, partition_size=part, err_flag=fused.err, desc=fused.desc, k_scale=fused.ks,
                              v_scale=fused.vs)
    torch.cuda.synchronize()
    assert int(fused.err.item()) == 0
    k, v = fused.host_after_append()
    assert np.array_equal(fused.k.cpu().numpy(), k) and np.array_equal(fused.v.cpu().numpy(), v)
    assert_close(out_f64(fused.out), fused.oracle(k, v), f"{w.name} fused, partition {part}")
    two.append()
    two.decode(partition_size=part)
    assert torch.equal(fused.out.view(torch.int16), two.out.view(torch.int16))
