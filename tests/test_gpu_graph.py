"""Decode and prefill steps captured in a CUDA graph.

A serving loop replays its decode step as a CUDA graph.  The decode kernels and
the partition merge are launched as programmatic dependents of the kernel before
them (their CTAs may be scheduled behind its last CTAs and wait on
griddepcontrol.wait), which stream capture records as programmatic edges.  These
tests capture the step (copy-on-write copies, the slot-mapping append, decode
with split partitions), replay it, and check the output bit for bit against the
same calls run eagerly, also after the inputs change in place between replays.
"""
import numpy as np
import pytest

import workloads as W
from harness import GpuStep, out_f64, oracle_step, to_torch, within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    return pa


def _workload(dtype):
    # four sequences, two of them split into several 512-token partitions; one new token each
    return W.build_decode(f"graph_{dtype}", seed=91, dtype=dtype, seq_lens=[300, 2500, 1100, 17], num_q_heads=16,
                          num_kv_heads=4, head_size=128, block_size=32, pool_factor=1.3, partition_size=512,
                          append_last=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_step_graph_replay_matches_eager(dtype):
    import torch
    w = _workload(dtype)
    eager = GpuStep(w)
    eager.step()
    torch.cuda.synchronize()
    assert int(eager.err.item()) == 0
    _, _, ref = oracle_step(w)
    ok, err, ratio = within_bound(out_f64(eager.out), ref, dtype)
    assert ok, f"eager step: max abs err {err}, worst err/bound {ratio}"

    g = GpuStep(w)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one eager call before capture (library setup happens outside the graph)
        g.step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.step()
    for _ in range(3):
        g.out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(g.out, eager.out)

    # inputs changed in place between replays: the replayed step reads the new values
    g.q.mul_(-0.5)
    eager.q.mul_(-0.5)
    graph.replay()
    eager.decode()
    torch.cuda.synchronize()
    assert torch.equal(g.out, eager.out)
    assert not torch.equal(g.out, torch.zeros_like(g.out))


def test_fp8_decode_graph_replay_matches_eager():
    import torch
    import paged_kv_cache_32_gb300 as pa
    w = W.build_decode("graph_fp8", seed=93, dtype="f16", seq_lens=[40, 1500, 700], num_q_heads=16, num_kv_heads=2,
                       head_size=128, block_size=16, pool_factor=1.3, partition_size=256)
    ks, vs = 0.0123, 0.0117
    rng = np.random.default_rng(5)
    # random E4M3 codes below 0x7F (the NaN code), with random signs
    codes_k = rng.integers(0, 0x7F, size=(w.num_blocks, w.num_kv_heads, w.block_size, w.head_size), dtype=np.uint8)
    codes_v = rng.integers(0, 0x7F, size=(w.num_blocks, w.num_kv_heads, w.block_size // 16, w.head_size, 16),
                           dtype=np.uint8)
    codes_k |= rng.integers(0, 2, size=codes_k.shape, dtype=np.uint8) << 7
    codes_v |= rng.integers(0, 2, size=codes_v.shape, dtype=np.uint8) << 7
    k = torch.from_numpy(codes_k).cuda()
    v = torch.from_numpy(codes_v).cuda()
    desc = pa.cache_desc(k)  # uint8 storage: an FP8 E4M3 cache
    q = torch.from_numpy(w.q).cuda()
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, desc, w.partition_size)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out_eager = torch.empty_like(q)
    out_graph = torch.empty_like(q)

    def call(out):
        pa.pa_decode(out, q, k, v, tables, lens, w.scale, partition_size=w.partition_size, workspace=ws,
                     err_flag=err, desc=desc, k_scale=ks, v_scale=vs)
    call(out_eager)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(out_graph)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_graph, out_eager)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_step_graph_replay_matches_eager(dtype):
    """A chunked-prefill step (the chunk's append, then pa_prefill) captured and
    replayed.  The fp16 kernel ends each full output tile with asynchronous
    tensor-map stores, which must have landed when the graph's kernel node
    completes.  More work items than SMs, full and ragged query tiles."""
    import torch
    import paged_kv_cache_32_gb300 as pa
    w = W.build_prefill(f"graph_prefill_{dtype}", seed=95, dtype=dtype,
                        prefix_lens=[0, 300, 17, 129, 500, 64, 0, 200], chunk_lens=[300, 129, 256, 1, 77, 200, 130, 384],
                        num_q_heads=32, num_kv_heads=8, head_size=128, block_size=16)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    max_q = int(np.max(np.diff(w.query_start)))

    class Step:
        def __init__(self):
            self.k = to_torch(w.k_cache, dtype, "cuda")
            self.v = to_torch(w.v_cache, dtype, "cuda")
            self.q = to_torch(w.q, dtype, "cuda")
            self.nk = to_torch(w.new_key, dtype, "cuda")
            self.nv = to_torch(w.new_value, dtype, "cuda")
            self.slots = torch.from_numpy(w.slot_mapping).cuda()
            self.tables = torch.from_numpy(w.block_tables).cuda()
            self.lens = torch.from_numpy(w.seq_lens).cuda()
            self.qs = torch.from_numpy(w.query_start).cuda()
            self.out = torch.zeros_like(self.q)
            self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
            self.desc = pa.cache_desc(self.k)

        def run(self):
            pa.pa_reshape_and_cache(self.k, self.v, self.nk, self.nv, self.slots, err_flag=self.err, desc=self.desc)
            pa.pa_prefill(self.out, self.q, self.k, self.v, self.tables, self.lens, self.qs, max_q, w.scale,
                          err_flag=self.err, desc=self.desc)

    eager = Step()
    eager.run()
    torch.cuda.synchronize()
    assert int(eager.err.item()) == 0
    assert eager.out.dtype == tdt
    # the eager call against the oracle (the last chunk ends with a full tile at the end of out)
    from test_gpu_prefill import host_pools, oracle_prefill
    k, v = host_pools(w)
    ok, err, ratio = within_bound(out_f64(eager.out), oracle_prefill(w, k, v), dtype)
    assert ok, f"eager prefill: max abs err {err}, worst err/bound {ratio}"

    g = Step()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one eager call before capture (library setup happens outside the graph)
        g.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.run()
    for _ in range(3):
        g.out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(g.out, eager.out)

    # queries changed in place between replays: the replayed step reads the new values
    g.q.mul_(-0.5)
    eager.q.mul_(-0.5)
    g.out.zero_()
    graph.replay()
    eager.run()
    torch.cuda.synchronize()
    assert torch.equal(g.out, eager.out)
    assert not torch.equal(g.out, torch.zeros_like(g.out))
