"""pa_decode_noalloc: decode without caller-provided or library-allocated workspace.

Some callers cannot allocate device memory while they decode (a serving plugin
whose host engine owns all device memory, a decode loop that must stay out of
the CUDA allocator).  pa_decode_noalloc serves them with a fixed scratch array
inside the library.  These tests call it through the C ABI and check that it
gives the same results as pa_decode with a workspace the caller allocated, on
two calls in a row (the scratch keeps the previous call's contents).  This
file is collected last so that a failing run has executed every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from harness import GpuStep, out_f64, within_bound

PA_ERR_WORKSPACE = 4
MAX_SCRATCH = 16 << 20  # PA_NOALLOC_MAX_WORKSPACE_BYTES in include/pa.h


def _lib():
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    L = pa.lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    L.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.POINTER(pa.pa_cache_desc),
                                    ctypes.c_float, i32, vp, vp]
    L.pa_decode_noalloc.restype = ctypes.c_int
    return pa, L


def _noalloc(L, g, out, stream):
    w = g.w
    return L.pa_decode_noalloc(out.data_ptr(), g.q.data_ptr(), g.k.data_ptr(), g.v.data_ptr(), g.tables.data_ptr(),
                               g.lens.data_ptr(), w.num_seqs, w.num_q_heads, w.max_blocks_per_seq,
                               ctypes.byref(g.desc), w.scale, w.partition_size, g.err.data_ptr(), stream)


def _decode(L, g, out, ws, stream):
    w = g.w
    return L.pa_decode(out.data_ptr(), g.q.data_ptr(), g.k.data_ptr(), g.v.data_ptr(), g.tables.data_ptr(),
                       g.lens.data_ptr(), w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, ctypes.byref(g.desc),
                       w.scale, w.partition_size, ws.data_ptr(), ws.numel(), g.err.data_ptr(), stream)


@pytest.mark.gpu
def test_noalloc_matches_decode_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa, L = _lib()
    cases = [
        W.long_bf16(16, num_seqs=2, seq_len=8192, partition_size=512),                       # split: scratch used
        W.build_decode("noalloc_f16", seed=77, dtype="f16", seq_lens=[1, 200, 700, 1500], num_q_heads=16,
                       num_kv_heads=4, head_size=128, block_size=32, pool_factor=1.3, partition_size=256),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    for w in cases:
        g = GpuStep(w)
        need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, g.desc,
                                           w.partition_size)
        assert 0 < need <= MAX_SCRATCH
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(g.q)
        assert _decode(L, g, ref, ws, stream) == 0
        outs = []
        for _ in range(2):
            out = torch.full_like(g.q, float("nan"))
            assert _noalloc(L, g, out, stream) == 0
            outs.append(out)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        r = out_f64(ref)
        for out in outs:
            ok, err, ratio = within_bound(out_f64(out), r, w.dtype)
            assert ok, f"{w.name}: pa_decode_noalloc differs from pa_decode by {err}"


def test_noalloc_rejects_sizes_beyond_the_scratch():
    pa, L = _lib()
    desc = pa.pa_cache_desc(1 << 16, 16, 8, 128, pa.PA_BF16)
    need = pa.pa_decode_workspace_size(4096, 64, 4096, desc, 512)
    assert need > MAX_SCRATCH
    fake = 0x10000  # never dereferenced: the size check comes first
    rc = L.pa_decode_noalloc(fake, fake, fake, fake, fake, fake, 4096, 64, 4096, ctypes.byref(desc), 0.1, 512,
                             None, None)
    assert rc == PA_ERR_WORKSPACE
