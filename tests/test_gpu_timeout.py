"""The decode kernels' bounded waits, made to run out (needs a GB300).

Every wait of the fp16/bf16 and FP8 decode kernels on an asynchronous copy is
bounded.  When one expires, the kernel raises the CTA's abort flag, the other
warps leave their loops, each warp waits for the copies it already started to
land, PA_DEVERR_TIMEOUT goes to err_flag, and the CTA returns: no trap, no
hang, the context stays usable.  The test hook PA_DECODE_TEST_EXPIRE_FIRST_WAIT
makes the first wait of every warp's ring expire without faulting anything:
the first slab is never requested and that wait is bounded at 20000 cycles,
while the ring's other copies are real and in flight.  Each test checks the
error status, and that the next ordinary call gives the output of a call made
before, bit for bit, which also meets the fp64 oracle.

Reading of the pages: silent corruption is the failure they warn of
("PagedAttention 笔记", section "写时复制是正确性的边界"); here a wait that cannot
complete is reported, not hidden.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from harness import GpuStep, out_f64, to_torch, within_bound

pytestmark = pytest.mark.gpu

PA_DEVERR_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    return pa


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("partition", [0, 256])
def test_expired_wait_reports_timeout_and_next_call_is_clean(dtype, partition):
    import torch
    import paged_kv_cache_32_gb300 as pa
    w = W.build_decode(f"timeout_{dtype}", seed=31, dtype=dtype, seq_lens=[1, 40, 300, 1100, 2000],
                       num_q_heads=16, num_kv_heads=2, head_size=128, block_size=32, pool_factor=1.3,
                       partition_size=partition)
    g = GpuStep(w)
    g.decode()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    before = g.out.clone()
    g.out.fill_(0)
    pa.pa_decode(g.out, g.q, g.k, g.v, g.tables, g.lens, w.scale, partition_size=partition, workspace=g.ws,
                 err_flag=g.err, desc=g.desc, test_flags=pa.PA_DECODE_TEST_EXPIRE_FIRST_WAIT)
    torch.cuda.synchronize()
    assert int(g.err.item()) == PA_DEVERR_TIMEOUT
    g.err.zero_()
    g.decode()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(g.out.view(torch.int16), before.view(torch.int16))
    ref = O.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=dtype,
                            num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
    ok, err, ratio = within_bound(out_f64(g.out), ref, dtype)
    assert ok, f"max abs err {err}, worst err/bound {ratio}"


def test_expired_wait_fp8_cache():
    import torch
    import paged_kv_cache_32_gb300 as pa
    ks, vs = 0.0123, 0.0117
    w = W.build_decode("timeout_fp8", seed=32, dtype="f16", seq_lens=[3, 64, 700, 1500], num_q_heads=8,
                       num_kv_heads=2, head_size=128, block_size=32, pool_factor=1.3, partition_size=512)
    kh = O.quantize_cache_fp8(w.k_cache, ks, values=False)
    vh = O.quantize_cache_fp8(w.v_cache, vs, values=True)
    k = torch.from_numpy(kh).cuda()
    v = torch.from_numpy(vh).cuda()
    q = to_torch(w.q, "f16")
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = pa.cache_desc(k)

    def call(out, flags=0):
        pa.pa_decode(out, q, k, v, tables, lens, w.scale, partition_size=512, err_flag=err, desc=desc, k_scale=ks,
                     v_scale=vs, test_flags=flags)
        torch.cuda.synchronize()

    before = torch.empty_like(q)
    call(before)
    assert int(err.item()) == 0
    call(torch.zeros_like(q), pa.PA_DECODE_TEST_EXPIRE_FIRST_WAIT)
    assert int(err.item()) == PA_DEVERR_TIMEOUT
    err.zero_()
    after = torch.empty_like(q)
    call(after)
    assert int(err.item()) == 0
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    ref = O.paged_attention_fp8(w.q, kh, vh, w.block_tables, w.seq_lens, num_kv_heads=2, block_size=32,
                                scale=w.scale, k_scale=ks, v_scale=vs)
    ok, err_v, ratio = within_bound(out_f64(after), ref, "f16")
    assert ok, f"max abs err {err_v}, worst err/bound {ratio}"
