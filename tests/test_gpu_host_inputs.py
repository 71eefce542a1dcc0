"""Per-step inputs and outputs in pinned host memory.

Under unified addressing every pinned host allocation is mapped into the
device's address space at its host address, so the small per-step tensors of a
decode step (q, block tables, lengths, slot mapping, the new tokens' K/V,
copy-on-write pairs) and the output can stay in host memory: the kernels read
and write them in place over the host link, with no copy in between.  The K/V
caches and the workspace stay in device memory.  Every call must give the same
bytes as with device buffers.
"""
import numpy as np
import pytest

import workloads as W
from harness import GpuStep, oracle_step, out_f64, within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    return pa


def _pinned(t):
    import torch
    h = torch.empty(t.shape, dtype=t.dtype).pin_memory()
    h.copy_(t.cpu())
    return h


def _same(a, b):
    import torch
    return torch.equal(a.cpu().contiguous().view(torch.uint8), b.cpu().contiguous().view(torch.uint8))


def test_decode_append_with_host_inputs_and_output():
    import torch
    w = W.build_decode("host_append", seed=5, dtype="f16", seq_lens=[1, 17, 700, 2048, 0], num_q_heads=16,
                       num_kv_heads=4, head_size=128, block_size=16, pool_factor=1.3, append_last=True,
                       partition_size=512)
    dev, hst = GpuStep(w), GpuStep(w)
    dev.pa.pa_decode_append(dev.out, dev.q, dev.k, dev.v, dev.nk, dev.nv, dev.tables, dev.lens, w.scale,
                            partition_size=512, workspace=dev.ws, err_flag=dev.err, desc=dev.desc)
    out = torch.full(hst.out.shape, float("nan"), dtype=hst.out.dtype).pin_memory()
    hst.pa.pa_decode_append(out, _pinned(hst.q), hst.k, hst.v, _pinned(hst.nk), _pinned(hst.nv), _pinned(hst.tables),
                            _pinned(hst.lens), w.scale, partition_size=512, workspace=hst.ws, err_flag=hst.err,
                            desc=hst.desc)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0 and int(hst.err.item()) == 0
    assert _same(dev.out, out)
    assert _same(dev.k, hst.k) and _same(dev.v, hst.v)
    _, _, ref = oracle_step(w)
    ok, err, ratio = within_bound(out_f64(out), ref, w.dtype)
    assert ok, f"max abs err {err}, worst err/bound {ratio}"


def test_step_with_host_pairs_slots_and_split_decode():
    """Copy-on-write copies, the slot-mapping append and a split decode (fp16, 256-token partitions),
    every per-step input and the output in pinned host memory."""
    import torch
    w = W.shared_prefix_f16(num_prompts=2, branches=4, prefix_len=1020, max_suffix=40, num_blocks=512, seed=13)
    dev, hst = GpuStep(w), GpuStep(w)
    dev.writes()
    dev.decode(partition_size=256)
    hst.pa.pa_copy_blocks(hst.k, hst.v, _pinned(hst.pairs), err_flag=hst.err, desc=hst.desc)
    hst.pa.pa_reshape_and_cache(hst.k, hst.v, _pinned(hst.nk), _pinned(hst.nv), _pinned(hst.slots),
                                err_flag=hst.err, desc=hst.desc)
    need = hst.pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, hst.desc, 256)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.full(hst.out.shape, float("nan"), dtype=hst.out.dtype).pin_memory()
    hst.pa.pa_decode(out, _pinned(hst.q), hst.k, hst.v, _pinned(hst.tables), _pinned(hst.lens), w.scale,
                     partition_size=256, workspace=ws, err_flag=hst.err, desc=hst.desc)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0 and int(hst.err.item()) == 0
    assert _same(dev.k, hst.k) and _same(dev.v, hst.v)
    assert _same(dev.out, out)
    _, _, ref = oracle_step(w)
    ok, err, ratio = within_bound(out_f64(out), ref, w.dtype)
    assert ok, f"max abs err {err}, worst err/bound {ratio}"


def test_gqa_bf16_decode_with_host_inputs():
    import torch
    w = W.gqa_bf16(num_seqs=24, hi=3000)
    dev, hst = GpuStep(w), GpuStep(w)
    dev.decode()
    out = torch.full(hst.out.shape, float("nan"), dtype=hst.out.dtype).pin_memory()
    hst.pa.pa_decode(out, _pinned(hst.q), hst.k, hst.v, _pinned(hst.tables), _pinned(hst.lens), w.scale,
                     partition_size=w.partition_size, workspace=hst.ws, err_flag=hst.err, desc=hst.desc)
    torch.cuda.synchronize()
    assert int(hst.err.item()) == 0
    assert _same(dev.out, out)
    assert np.isfinite(out_f64(out)).all()


def test_fp8_append_and_decode_with_host_inputs():
    """The quantising FP8 append (fp16 key/value rows and slots in host memory) and FP8 decode (q,
    tables, lengths and out in host memory)."""
    import torch
    import oracle as O
    from harness import to_torch
    w = W.build_decode("host_fp8", seed=21, dtype="f16", seq_lens=[3, 64, 900, 2000], num_q_heads=16,
                       num_kv_heads=2, head_size=128, block_size=32, pool_factor=1.3, append_last=True,
                       partition_size=512)
    ks, vs = 0.0123, 0.0117
    kc = O.quantize_cache_fp8(w.k_cache, ks, values=False)
    vc = O.quantize_cache_fp8(w.v_cache, vs, values=True)
    import paged_kv_cache_32_gb300 as pa

    def run(host):
        k = torch.from_numpy(np.ascontiguousarray(kc)).cuda()
        v = torch.from_numpy(np.ascontiguousarray(vc)).cuda()
        desc = pa.cache_desc(k)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        q = to_torch(w.q, "f16", "cuda")
        nk, nv = to_torch(w.new_key, "f16", "cuda"), to_torch(w.new_value, "f16", "cuda")
        slots = torch.from_numpy(w.slot_mapping).cuda()
        tables, lens = torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.seq_lens).cuda()
        out = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
        if host:
            q, nk, nv, slots, tables, lens = (_pinned(t) for t in (q, nk, nv, slots, tables, lens))
            out = torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory()
        pa.pa_reshape_and_cache_fp8(k, v, nk, nv, slots, ks, vs, err_flag=err, desc=desc)
        need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, desc, 512)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        pa.pa_decode(out, q, k, v, tables, lens, w.scale, partition_size=512, workspace=ws, err_flag=err, desc=desc,
                     k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        return k, v, out

    kd, vd, od = run(False)
    kh, vh, oh = run(True)
    assert _same(kd, kh) and _same(vd, vh)
    assert _same(od, oh)
    assert np.isfinite(out_f64(oh)).all()
