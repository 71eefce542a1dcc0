"""pa_decode_noalloc: decode without caller-provided or library-allocated workspace.

Some callers cannot allocate device memory while they decode (a serving plugin
whose host engine owns all device memory, a decode loop that must stay out of
the CUDA allocator).  pa_decode_noalloc serves them with a fixed scratch array
inside the library.  These tests call it through the C ABI and check that it
gives bit-for-bit the output of pa_decode with a workspace the caller
allocated, and that both meet the fp64 oracle, on two calls in a row (the
scratch keeps the previous call's contents).  This file is collected last so
that a failing run has executed every other test.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as W
from harness import GpuStep, out_f64, within_bound

PA_ERR_WORKSPACE = 4
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


def max_scratch_bytes() -> int:
    """PA_NOALLOC_MAX_WORKSPACE_BYTES as include/pa.h defines it (a "(size_t)A << B" expression)."""
    with open(HEADER) as f:
        m = re.search(r"#define\s+PA_NOALLOC_MAX_WORKSPACE_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", f.read())
    assert m, "PA_NOALLOC_MAX_WORKSPACE_BYTES not found in include/pa.h"
    return int(m.group(1)) << int(m.group(2))


def _lib():
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    L = pa.lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    L.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.POINTER(pa.pa_cache_desc),
                                    ctypes.c_float, i32, vp, vp]
    L.pa_decode_noalloc.restype = ctypes.c_int
    return pa, L


def _noalloc(L, g, out, part, stream):
    w = g.w
    return L.pa_decode_noalloc(out.data_ptr(), g.q.data_ptr(), g.k.data_ptr(), g.v.data_ptr(), g.tables.data_ptr(),
                               g.lens.data_ptr(), w.num_seqs, w.num_q_heads, w.max_blocks_per_seq,
                               ctypes.byref(g.desc), w.scale, part, g.err.data_ptr(), stream)


def _decode(L, g, out, ws, part, stream):
    w = g.w
    return L.pa_decode(out.data_ptr(), g.q.data_ptr(), g.k.data_ptr(), g.v.data_ptr(), g.tables.data_ptr(),
                       g.lens.data_ptr(), w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, ctypes.byref(g.desc),
                       w.scale, part, ws.data_ptr(), ws.numel(), g.err.data_ptr(), stream)


def _cases():
    return [
        # (workload, partition size): each needs scratch
        (W.long_bf16(16, num_seqs=2, seq_len=8192, partition_size=512), 512),
        (W.build_decode("noalloc_f16", seed=77, dtype="f16", seq_lens=[1, 200, 700, 1500], num_q_heads=16,
                        num_kv_heads=4, head_size=128, block_size=32, pool_factor=1.3, partition_size=256), 256),
        # the GQA bf16 shapes (128 seqs, 64 q / 8 kv heads, up to 4096 tokens) at the 2048-token
        # partition that keeps them inside the scratch (the default 1024 would need 17 MB)
        (W.gqa_bf16(), 2048),
    ]


@pytest.mark.gpu
def test_noalloc_matches_decode_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa, L = _lib()
    limit = max_scratch_bytes()
    stream = torch.cuda.current_stream().cuda_stream
    for w, part in _cases():
        g = GpuStep(w)
        need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, g.desc, part)
        assert 0 < need <= limit
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(g.q)
        assert _decode(L, g, ref, ws, part, stream) == 0
        outs = []
        for _ in range(2):
            out = torch.full_like(g.q, float("nan"))
            assert _noalloc(L, g, out, part, stream) == 0
            outs.append(out)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        for i, out in enumerate(outs):  # the same kernels on the same inputs: bit-identical
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
                f"{w.name}: call {i + 1} of pa_decode_noalloc differs from pa_decode"
        exact = O.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, dtype=w.dtype,
                                  num_kv_heads=w.num_kv_heads, block_size=w.block_size, scale=w.scale)
        ok, err, ratio = within_bound(out_f64(outs[-1]), exact, w.dtype)
        assert ok, f"{w.name}: max abs err {err} against the oracle, worst err/bound {ratio}"


def test_noalloc_limit_covers_the_documented_workloads():
    """The sizes the header documents: the split workloads fit at their partition sizes;
    the GQA bf16 shapes need more than the limit at the default 1024-token partition
    and fit at 2048."""
    pa, _ = _lib()
    limit = max_scratch_bytes()

    def need(w, part):
        desc = pa.pa_cache_desc(w.num_blocks, w.block_size, w.num_kv_heads, w.head_size,
                                {"f32": pa.PA_F32, "f16": pa.PA_F16, "bf16": pa.PA_BF16}[w.dtype])
        return pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, desc, part)

    assert need(W.mha_f16(materialize=False), 0) <= limit
    assert need(W.shared_prefix_f16(materialize=False), 0) <= limit
    for b in (16, 32, 64):
        assert need(W.long_bf16(b, materialize=False), 512) <= limit
    gqa = W.gqa_bf16(materialize=False)
    assert need(gqa, 0) > limit
    assert 0 < need(gqa, 2048) <= limit


def test_noalloc_rejects_sizes_beyond_the_scratch():
    pa, L = _lib()
    desc = pa.pa_cache_desc(1 << 16, 16, 8, 128, pa.PA_BF16)
    need = pa.pa_decode_workspace_size(4096, 64, 4096, desc, 512)
    assert need > max_scratch_bytes()
    fake = 0x10000  # never dereferenced: the size check comes first
    rc = L.pa_decode_noalloc(fake, fake, fake, fake, fake, fake, 4096, 64, 4096, ctypes.byref(desc), 0.1, 512,
                             None, None)
    assert rc == PA_ERR_WORKSPACE
