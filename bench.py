"""Benchmark of the paged decode step on GB300.

One step = every row of the hot path over one batch: the copy-on-write block
copies (workloads that have them), the slot-mapping append of the step's new
tokens, and paged decode attention (block-table gather, K/V streaming, QK^T,
online softmax, PV and, for long contexts, the partition merge).

Prints ONE JSON line (rank 0).  ``value`` = KV GB/s: algorithmic K+V bytes the
attention reads per step, summed over ranks, divided by the device time of a
step (max over ranks).  Default workload: MHA fp16 decode (64 seqs, lens
U[128, 2048], 32 heads, D = 128, B = 16, pool 8192, one append per seq).
The timed region holds the steps alone between two CUDA events (see
time_device); per-call breakdowns are timed in loops of their own.

--impl reference times the CPU fp64 evaluation (the test oracle) on the host
cores instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (fraction of GB300 HBM peak) and decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
WORKLOAD_DESC = {
    "mha_f16": "MHA fp16 decode: 64 seqs, seq_lens U[128,2048], 32 q = 32 kv heads, D 128, B 16, pool 8192 shuffled, "
               "each seq's new token appended and attended in one pa_decode_append call",
    "gqa_bf16": "GQA bf16 decode: 128 seqs, 64 q / 8 kv heads, D 128, B 32, lognormal(ln 1200, 0.6) lens in "
                "[64, 4096], pool 1.2x needed, shuffled",
    "shared_prefix_f16": "shared-prefix fp16: 16 prompts x 8 branches, 1024-token shared prefix, suffix U[1,256], "
                         "32 heads, D 128, B 16; 128 CoW block copies + suffix appends, then attention",
    "long_bf16_b16": "long bf16 split-KV: 8 seqs x 32768 tokens, 32 q / 8 kv heads, D 128, B 16, 512-token partitions",
    "long_bf16_b32": "long bf16 split-KV: 8 seqs x 32768 tokens, 32 q / 8 kv heads, D 128, B 32, 512-token partitions",
    "long_bf16_b64": "long bf16 split-KV: 8 seqs x 32768 tokens, 32 q / 8 kv heads, D 128, B 64, 512-token partitions",
    "mha_fp8": "MHA decode over an FP8 E4M3 cache (scales 0.0123 / 0.0117, fp16 q/out): 64 seqs, seq_lens "
               "U[128,2048], 32 heads, D 128, B 16, pool 8192 shuffled; each seq's new token quantised, appended and "
               "attended in one pa_decode_append call",
    "gqa_fp8": "GQA decode over an FP8 E4M3 cache (fp16 q/out): 128 seqs, 64 q / 8 kv heads, D 128, B 32, "
               "lognormal(ln 1200, 0.6) lens in [64, 4096], pool 1.2x needed",
    "prefill_bf16": "chunked prefill bf16: 16 seqs, cached prefix U[0,2048] + chunk U[256,2048] tokens, 32 q / 8 kv "
                    "heads, D 128, B 16, pool 1.2x needed, shuffled; chunk K/V appended, then causal attention",
    "prefill_f16": "chunked prefill fp16, the prefill_bf16 shapes: P enters the value MMA as one fp16 term "
                   "(two bf16 terms for bf16)",
}
TORCH_DT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


# sources that define the decode call's kernels and launch configuration
KERNEL_SOURCES = ("pa_api.cu", "pa_decode_tc.cu", "pa_decode_slab.cuh", "pa_decode_epilogue.cuh", "pa_device.cuh",
                  "pa_internal.h", "pa_merge.cu")


# sources that define the prefill call's kernel
PREFILL_SOURCES = ("pa_prefill_api.cu", "pa_prefill_tc.cu", "pa_prefill.h", "pa_device.cuh", "pa_internal.h")
# sources that define the decode call on an FP8 cache
FP8_SOURCES = ("pa_api.cu", "pa_decode_fp8.cu", "pa_decode_epilogue.cuh", "pa_device.cuh", "pa_internal.h",
               "pa_merge.cu")


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_32_gb300", "csrc")
    for fn in sources:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary,
    valid only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    sources = (PREFILL_SOURCES if workload.startswith("prefill") else FP8_SOURCES if "fp8" in workload
               else KERNEL_SOURCES)
    if not entry or entry.get("source_sha") != kernel_source_hash(sources):
        return None
    return entry.get("dram_bytes_per_launch")


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's libnvidia-ml, reads only)
    about every 0.5 ms on a background thread, so that even a few-millisecond timed region gets several
    samples.  Raises OSError at construction when NVML is unavailable."""
    # clock-event reason bits of NVML's public API
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        handle = None
        try:  # match the CUDA device by its PCI address when torch exposes it
            import torch
            pr = torch.cuda.get_device_properties(index)
            bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.dev)) == 0:
                handle = self.dev
        except (AttributeError, RuntimeError, ImportError):
            handle = None
        if handle is None and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0 else None
        self.samples = []
        self.running = False
        self.thread = None

    def _read(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        while self.running:
            ok = self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(mhz)) == 0  # NVML_CLOCK_SM
            okr = self.reasons_fn(self.dev, ct.byref(rs)) == 0
            okp = self.lib.nvmlDeviceGetPowerUsage(self.dev, ct.byref(mw)) == 0
            if ok:
                self.samples.append((time.time(), float(mhz.value), int(rs.value) if okr else 0,
                                     mw.value / 1000.0 if okp else None))
            time.sleep(0.0005)

    def start(self):
        self.running = True
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def stop(self):
        self.running = False
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        if not inside and self.samples:  # nothing inside: the nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda x: abs(x[0] - mid))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0}
        reasons = sorted(n for n, b in self.REASON_BITS.items() if any(x[2] & b for x in inside))
        pw = [x[3] for x in inside if x[3] is not None]
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_min_mhz": min(x[1] for x in inside),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside),
                "power_w_max": max(pw) if pw else None, "source": "nvml"}


def clock_sampler(index: int):
    """NVML sampling when the driver's library loads, else nvidia-smi."""
    try:
        return NvmlClockSampler(index)
    except (OSError, AttributeError):
        return ClockSampler(index)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [p for (t, p) in self.samples if t0 - 0.05 <= t <= t1 + 0.05]
        if not inside:  # the timed region was shorter than the sampling period: nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda tp: abs(tp[0] - mid))[1]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------- GPU arm
class DeviceStep:
    """All device buffers of one workload and the library calls of one step."""

    def __init__(self, w: W.Workload, device, alibi: bool = False):
        import torch
        import paged_kv_cache_32_gb300 as pa
        self.pa, self.w, self.dev = pa, w, device
        # ALiBi: the usual geometric per-head slopes 2^(-8 i / H)
        self.alibi = (torch.tensor([2.0 ** (-8.0 * (i + 1) / w.num_q_heads) for i in range(w.num_q_heads)],
                                   dtype=torch.float32, device=device) if alibi else None)
        tdt = getattr(torch, TORCH_DT[w.dtype])
        self.fp8 = w.info.get("kv_dtype") == "fp8"
        self.k_scale, self.v_scale = w.info.get("k_scale"), w.info.get("v_scale")
        self.k, self.v = W.device_caches(w, device)
        if self.fp8:
            # E4M3 codes of x / scale (torch's conversion: inputs only), saturated at +-448 as the library's
            # append does (torch's conversion turns values past the range into NaN codes, which a draw of
            # a billion N(0, 1) values / 0.0123 reaches); values [blocks][heads][B/16][D][16]
            self.k = (self.k.float() / self.k_scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            self.v = (self.v.float() / self.v_scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            nb, hkv, bs, d = self.v.shape
            self.v = self.v.view(nb, hkv, bs // 16, 16, d).transpose(3, 4).contiguous()
            torch.cuda.empty_cache()
        self.desc = pa.cache_desc(self.k)

        def t(a, dtype=None):
            if a is None:
                return None
            if w.dtype == "bf16" and dtype is None and a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.q = t(w.q)
        self.tables = t(w.block_tables)
        self.lens = t(w.seq_lens)
        self.pairs = t(w.copy_pairs) if w.copy_pairs is not None and len(w.copy_pairs) else None
        self.slots = t(w.slot_mapping) if w.slot_mapping is not None and len(w.slot_mapping) else None
        self.nk = t(w.new_key) if self.slots is not None else None
        self.nv = t(w.new_value) if self.slots is not None else None
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.part = pa.pa_decode_partition_size(w.max_blocks_per_seq, self.desc, w.partition_size)
        need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, self.desc,
                                           w.partition_size)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.ws_bytes = need
        self.pmax = 1 if need == 0 else -(-w.max_blocks_per_seq * w.block_size // self.part)
        # a step whose writes are each sequence's new token at its last position, on a 16-bit cache:
        # the append runs inside the decode call (pa_decode_append)
        self.fused = bool(w.info.get("append_last")) and w.dtype in ("f16", "bf16") and \
            self.pairs is None and self.slots is not None
        assert tdt == self.q.dtype

    def launches_per_step(self) -> int:
        return (self.pairs is not None) + (self.slots is not None and not self.fused) + 1 + (self.pmax > 1)

    @property
    def single_call(self) -> bool:
        """The step is the attention call alone (no copy-on-write copies, the append fused or absent)."""
        return self.pairs is None and (self.slots is None or self.fused)

    def append(self, stream, nk, nv, slots):
        if self.fp8:
            self.pa.pa_reshape_and_cache_fp8(self.k, self.v, nk, nv, slots, self.k_scale, self.v_scale,
                                             err_flag=self.err, stream=stream, desc=self.desc)
        else:
            self.pa.pa_reshape_and_cache(self.k, self.v, nk, nv, slots, err_flag=self.err, stream=stream,
                                         desc=self.desc)

    def writes(self, stream):
        if self.pairs is not None:
            self.pa.pa_copy_blocks(self.k, self.v, self.pairs, err_flag=self.err, stream=stream, desc=self.desc)
        if self.slots is not None and not self.fused:
            self.append(stream, self.nk, self.nv, self.slots)

    def step_decode(self, stream, q=None, tables=None, lens=None, nk=None, nv=None, out=None):
        """The step's attention: with the append fused in when the step allows it."""
        if not self.fused:
            self.decode(stream, q=q, tables=tables, lens=lens, out=out)
            return
        self.pa.pa_decode_append(self.out if out is None else out, self.q if q is None else q, self.k, self.v,
                                 self.nk if nk is None else nk,
                                 self.nv if nv is None else nv, self.tables if tables is None else tables,
                                 self.lens if lens is None else lens, self.w.scale,
                                 partition_size=self.w.partition_size, workspace=self.ws, err_flag=self.err,
                                 stream=stream, desc=self.desc,
                                 alibi_slopes=self.alibi, k_scale=self.k_scale if self.fp8 else None,
                                 v_scale=self.v_scale if self.fp8 else None)

    def decode(self, stream, q=None, tables=None, lens=None, out=None):
        self.pa.pa_decode(self.out if out is None else out, self.q if q is None else q, self.k, self.v,
                          self.tables if tables is None else tables, self.lens if lens is None else lens,
                          self.w.scale, partition_size=self.w.partition_size, workspace=self.ws,
                          err_flag=self.err, stream=stream, desc=self.desc, alibi_slopes=self.alibi,
                          k_scale=self.k_scale if self.fp8 else None, v_scale=self.v_scale if self.fp8 else None)

    def attend(self, stream):
        self.step_decode(stream)

    def decode_bytes(self, with_append: bool | None = None) -> int:
        """Algorithmic HBM bytes of one pa_decode call: K+V of every token, q in,
        out, table entries, and the split-KV partial results (written then read);
        with the append fused in (default: when the step fuses it), also the new
        tokens' K/V read and written."""
        w = self.w
        eb = W.ELEM_BYTES[w.dtype]
        b = w.kv_bytes() + 2 * w.num_seqs * w.num_q_heads * w.head_size * eb
        if self.fused if with_append is None else with_append:  # each new row read (key and value, the workload dtype) and written (the cache's codes)
            b += int(np.sum(w.seq_lens > 0)) * w.num_kv_heads * w.head_size * 2 * (eb + (1 if self.fp8 else eb))
        b += int(np.sum(-(-w.seq_lens.astype(np.int64) // w.block_size))) * 4 + w.num_seqs * 4
        if self.pmax > 1:
            nparts = -(-w.seq_lens.astype(np.int64) // self.part)
            multi = nparts[nparts > 1]
            b += 2 * int(multi.sum()) * w.num_q_heads * (w.head_size + 2) * 4
        return b


class PrefillDeviceStep:
    """Device buffers of a chunked-prefill workload and the calls of one step:
    the chunk's K/V appended through slot_mapping, then prefill attention of the
    chunk's queries over each whole sequence."""

    def __init__(self, w: W.Workload, device):
        import torch
        import paged_kv_cache_32_gb300 as pa
        self.pa, self.w, self.dev = pa, w, device
        tdt = getattr(torch, TORCH_DT[w.dtype])
        self.k, self.v = W.device_caches(w, device)
        self.desc = pa.cache_desc(self.k)
        gen = torch.Generator(device=device)
        gen.manual_seed(int(w.info.get("seed", 0)) + 1)
        T = w.num_query_tokens

        def draw(heads):
            return torch.randn((T, heads, w.head_size), generator=gen, device=device, dtype=torch.float32).to(tdt)
        self.q, self.nk, self.nv = draw(w.num_q_heads), draw(w.num_kv_heads), draw(w.num_kv_heads)
        self.slots = torch.from_numpy(w.slot_mapping).to(device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.qs = torch.from_numpy(w.query_start).to(device)
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.max_q = int(np.diff(w.query_start).max())

    def writes(self, stream):
        self.pa.pa_reshape_and_cache(self.k, self.v, self.nk, self.nv, self.slots, err_flag=self.err, stream=stream,
                                     desc=self.desc)

    def attend(self, stream):
        self.pa.pa_prefill(self.out, self.q, self.k, self.v, self.tables, self.lens, self.qs, self.max_q, self.w.scale,
                           err_flag=self.err, stream=stream, desc=self.desc)


def time_device(ds, steps: int, warmup: int, world: int, call=None):
    """Device times of a step (ds.writes, then ds.attend), in three loops of `steps` each.

    1. The timed region: the steps back to back on one stream between two CUDA events, with a
       barrier and a device synchronisation on both sides and nothing else on the stream.  An
       event recorded between two launches ends the overlap of a launch with the previous one's
       end (programmatic dependent launch), so per-call events would slow the loop they time.
    2. The attention call alone (`call`, default ds.attend), back to back between two events: its
       mean duration.
    3. Per-step event pairs around the writes and the call, for medians; each call there pays
       its launch's own start-up.
    Returns (mean step ms of 1, mean call ms of 2, call ms list of 3, writes ms list of 3,
    wall-clock window of all three)."""
    import torch
    stream = torch.cuda.Stream()
    ev_pair = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            ds.writes(stream)
            ds.attend(stream)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        start, end = ev_pair()
        start.record(stream)
        for _ in range(steps):
            ds.writes(stream)
            ds.attend(stream)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms_step = start.elapsed_time(end) / steps
        call = call or ds.attend
        a, b = ev_pair()
        a.record(stream)
        for _ in range(steps):
            call(stream)
        b.record(stream)
        stream.synchronize()
        call_ms = a.elapsed_time(b) / steps
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(stream)
            ds.writes(stream)
            ev[i][1].record(stream)
            ds.attend(stream)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
    decode_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    write_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
    return ms_step, call_ms, decode_ms, write_ms, (t0, t1)


def time_calls(fn, steps: int, warmup: int) -> float:
    """Mean device time in ms of fn(stream) over `steps` back-to-back calls, CUDA events on the
    launching stream, after `warmup` untimed calls."""
    import torch
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn(stream)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn(stream)
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / steps


def bench_secondary(device, steps: int, warmup: int, peak: float):
    """The secondary measurements: the cost of the block-table indirection (the MHA fp16 decode
    with each sequence's blocks contiguous and in order, i.e. identity tables, against the
    shuffled pool), a block-size sweep on the same sequences, and the two write calls at sizes
    where bandwidth means something, plus their decode-step sizes.  Byte counts are algorithmic
    (reads + writes for the writes, like the copy peak)."""
    import torch
    import paged_kv_cache_32_gb300 as pa
    lens = np.random.default_rng(1001).integers(128, 2048, size=64, endpoint=True)  # the mha_f16 lengths
    res = {}

    def decode(name, block_size, shuffle, num_blocks=None, dtype="f16"):
        w = W.build_decode(name, seed=1001, dtype=dtype, seq_lens=lens, num_q_heads=32, num_kv_heads=32,
                           head_size=128, block_size=block_size, num_blocks=num_blocks, shuffle=shuffle,
                           materialize=False)
        ds = DeviceStep(w, device)
        ms = time_calls(ds.decode, steps, warmup)
        err = int(ds.err.item())
        gbs = ds.decode_bytes() / (ms * 1e-3) / 1e9
        del ds
        torch.cuda.empty_cache()
        if err:
            raise RuntimeError(f"device error flag {err} in {name}")
        return {"decode_ms": round(ms, 5), "decode_gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}

    shuffled = decode("tables_shuffled", 16, True, 8192)
    identity = decode("tables_identity", 16, False, 8192)
    res["block_tables"] = {"workload": "mha_f16 sequences, B 16, pool 8192", "shuffled": shuffled,
                           "identity": identity,
                           "shuffled_over_identity_time": round(shuffled["decode_ms"] / identity["decode_ms"], 4)}
    res["block_size_sweep"] = {"workload": "mha_f16 sequences, shuffled pool 1.2x needed (B 8: two 8-row copies "
                                           "per 16-token slab)",
                               **{f"B{b}": decode(f"sweep_b{b}", b, True) for b in (8, 16, 32, 64, 128, 256)}}
    # the pages' claim that one-token blocks are catastrophic, on the one kernel that takes any block size (the
    # fp32 CUDA-core kernel, a correctness path: one table entry and one dependent row load per token at B 1)
    res["block_size_probe_fp32"] = {"workload": "mha_f16 sequences in fp32, shuffled pool 1.2x needed",
                                    **{f"B{b}": decode(f"probe_f32_b{b}", b, True, dtype="f32") for b in (16, 1)}}

    # the write calls on an MHA fp16 pool (8192 blocks of 16 slots, 32 heads, D 128)
    gen = torch.Generator(device=device)
    gen.manual_seed(1001)
    nb, hkv, B, D = 8192, 32, 16, 128
    k = torch.randn((nb, hkv, B, D), generator=gen, device=device, dtype=torch.float32).to(torch.float16)
    v = torch.randn((nb, hkv, B, D), generator=gen, device=device, dtype=torch.float32).to(torch.float16)
    desc = pa.cache_desc(k)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    perm = torch.randperm(nb * B, generator=gen, device=device)
    writes = {}
    for T in (64, 16384):  # a decode step's appends; a prefill chunk's worth
        key = torch.randn((T, hkv, D), generator=gen, device=device, dtype=torch.float32).to(torch.float16)
        val = torch.randn((T, hkv, D), generator=gen, device=device, dtype=torch.float32).to(torch.float16)
        slots = perm[:T].contiguous()
        ms = time_calls(lambda st: pa.pa_reshape_and_cache(k, v, key, val, slots, err_flag=err, stream=st, desc=desc),
                        steps, warmup)
        nbytes = T * 2 * hkv * D * 2 * 2 + T * 8  # K and V rows read and written, slots read
        writes[f"reshape_and_cache_{T}_tokens"] = {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    bperm = torch.randperm(nb, generator=gen, device=device).to(torch.int32)
    for n in (128, 2048):  # the shared-prefix step's copies; a large copy-on-write burst
        pairs = torch.stack([bperm[:n], bperm[n:2 * n]], dim=1).contiguous()
        ms = time_calls(lambda st: pa.pa_copy_blocks(k, v, pairs, err_flag=err, stream=st, desc=desc), steps, warmup)
        nbytes = n * 2 * hkv * B * D * 2 * 2 + n * 8  # both caches' blocks read and written, pairs read
        writes[f"copy_blocks_{n}_pairs"] = {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"device error flag {int(err.item())} in the write calls")
    res["writes"] = {"pool": "MHA fp16, 8192 blocks x 32 heads x 16 x 128", **writes}
    del k, v
    torch.cuda.empty_cache()
    return res


def _pinned_mapped(t) -> None:
    """The pinned host tensor is mapped into the device's address space at its host address (true
    of every pinned allocation under unified addressing); checked through the driver before a
    kernel is given the pointer."""
    import ctypes
    drv = ctypes.CDLL("libcuda.so.1")
    dptr = ctypes.c_uint64(0)
    CU_POINTER_ATTRIBUTE_DEVICE_POINTER = 3
    rc = drv.cuPointerGetAttribute(ctypes.byref(dptr), ctypes.c_int(CU_POINTER_ATTRIBUTE_DEVICE_POINTER),
                                   ctypes.c_uint64(t.data_ptr()))
    if rc != 0 or dptr.value != t.data_ptr():
        raise RuntimeError(f"pinned host memory is not mapped at its host address (driver status {rc})")


def time_e2e(ds: DeviceStep, steps: int, warmup: int, world: int):
    """The same step through the public API with its per-step inputs (q, tables, lengths, slots,
    new K/V, copy pairs) in pinned host memory and its output going to pinned host memory, inside
    the timed region; the K/V caches and the workspace are resident device state.  Two ways, each
    timed over `steps` steps between two events:
      zero-copy (reported): the library's kernels read the inputs and write the output in place in
        host memory, over the host link (the pointers are host addresses mapped into the device's
        address space);
      copy: one cudaMemcpyAsync of all inputs (one pinned staging buffer, 256-byte aligned each) to
        device memory, the step on device buffers, and the output copied back.
    Returns (zero-copy ms per step, copy ms per step, input bytes, output bytes)."""
    import torch
    tensors = [(k, t) for k, t in (("q", ds.q), ("tables", ds.tables), ("lens", ds.lens), ("slots", ds.slots),
                                   ("nk", ds.nk), ("nv", ds.nv), ("pairs", ds.pairs)) if t is not None]
    offs, total = {}, 0
    for k, t in tensors:
        offs[k] = total
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=ds.dev)
    dev, hst = {}, {}
    for k, t in tensors:
        n = t.numel() * t.element_size()
        host_buf[offs[k]:offs[k] + n].copy_(t.detach().contiguous().view(-1).view(torch.uint8).cpu())
        dev[k] = dev_buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        hst[k] = host_buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    out_host = torch.empty(ds.out.shape, dtype=ds.out.dtype).pin_memory()
    _pinned_mapped(host_buf)
    _pinned_mapped(out_host)
    h2d = total
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.Stream()

    def step(bufs, out):
        if ds.pairs is not None:
            ds.pa.pa_copy_blocks(ds.k, ds.v, bufs["pairs"], err_flag=ds.err, stream=stream, desc=ds.desc)
        if ds.slots is not None and not ds.fused:
            ds.append(stream, bufs["nk"], bufs["nv"], bufs["slots"])
        ds.step_decode(stream, q=bufs["q"], tables=bufs["tables"], lens=bufs["lens"], nk=bufs.get("nk"),
                       nv=bufs.get("nv"), out=out)

    def zero_copy():
        step(hst, out_host)

    def copied():
        dev_buf.copy_(host_buf, non_blocking=True)
        step(dev, ds.out)
        out_host.copy_(ds.out, non_blocking=True)

    res = []
    with torch.cuda.stream(stream):
        for fn in (zero_copy, copied):
            for _ in range(warmup):
                fn()
            stream.synchronize()
            barrier(world)
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            start.record(stream)
            for _ in range(steps):
                fn()
            end.record(stream)
            torch.cuda.synchronize()
            barrier(world)
            res.append(start.elapsed_time(end) / steps)
    return res[0], res[1], h2d, d2h


def block_manager_step_us(w: W.Workload, steps: int = 200, model=None) -> float:
    """Host time of one decode step's metadata with a block manager: one
    append_slots call for every sequence (slots + copy-on-write pairs) and one
    build_tables call, averaged over `steps` steps.  Every sequence gets private
    blocks here (the pool is sized for that, also for workloads whose own pool
    relies on shared prefixes)."""
    pool = int(np.sum(-(-w.seq_lens.astype(np.int64) // w.block_size))) + w.num_seqs * (steps // w.block_size + 2)
    if model is None:
        from paged_kv_cache_32_gb300.block_manager import BlockManager
        bm = BlockManager(pool, w.block_size, shuffle_seed=1)
        seqs = np.arange(w.num_seqs, dtype=np.int64)
        for s in seqs:
            bm.allocate(int(s), int(w.seq_lens[s]))
        t0 = time.perf_counter()
        for _ in range(steps):
            bm.append_slots(seqs)
            bm.build_tables(seqs)
        return 1e6 * (time.perf_counter() - t0) / steps
    m = model(pool, w.block_size, 1)
    for s in range(w.num_seqs):
        m.allocate(s, int(w.seq_lens[s]))
    t0 = time.perf_counter()
    for _ in range(steps):
        for s in range(w.num_seqs):
            m.append_slot(s)
        width = max(len(m.tables[s]) for s in range(w.num_seqs))
        tables = np.zeros((w.num_seqs, width), np.int32)
        for s in range(w.num_seqs):
            tables[s, :len(m.tables[s])] = m.tables[s]
    return 1e6 * (time.perf_counter() - t0) / steps


def cpu_baseline(w_meta: W.Workload, budget_s: float = 12.0):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    workload (whole sequences, in order), repeated until the budget is used."""
    import oracle as O
    threads = O.max_threads()
    n = w_meta.num_seqs
    take = list(range(min(n, 16)))
    sample = W.host_sample(w_meta, take)
    kw = dict(dtype=sample.dtype, num_kv_heads=sample.num_kv_heads, block_size=sample.block_size)
    reps, t_total = 0, 0.0
    while t_total < budget_s and reps < 10000:
        k, v = sample.k_cache.copy(), sample.v_cache.copy()
        t0 = time.perf_counter()
        W.apply_writes_host(sample, k, v,
                            lambda kk, vv, pairs: O.copy_blocks(kk, vv, pairs, head_size=sample.head_size, **kw),
                            lambda kk, vv, nk, nv, sl: O.reshape_and_cache(kk, vv, nk, nv, sl, **kw))
        O.paged_attention(sample.q, k, v, sample.block_tables, sample.seq_lens, scale=sample.scale,
                          threads=threads, **kw)
        t_total += time.perf_counter() - t0
        reps += 1
    gbs = reps * sample.kv_bytes() / t_total / 1e9
    # the same evaluation on one thread, over the first two sequences of the sample
    one = W.host_sample(w_meta, take[:2])
    reps1, t1 = 0, 0.0
    while t1 < budget_s / 4 and reps1 < 10000:
        t0 = time.perf_counter()
        O.paged_attention(one.q, one.k_cache, one.v_cache, one.block_tables, one.seq_lens, scale=one.scale,
                          threads=1, dtype=one.dtype, num_kv_heads=one.num_kv_heads, block_size=one.block_size)
        t1 += time.perf_counter() - t0
        reps1 += 1
    from oracle.block_manager import BlockManagerModel
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "block_manager_model_step_us": round(block_manager_step_us(w_meta, 50, BlockManagerModel), 1),
            "sample": f"{len(take)} of {n} sequences ({int(sample.seq_lens.sum())} tokens) x {reps} repetitions, "
                      f"{t_total:.1f} s wall, OpenMP over (seq, q head)",
            "tokens_per_s": reps * len(take) / t_total,
            "single_thread": {"value": round(reps1 * one.kv_bytes() / t1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"2 sequences ({int(one.seq_lens.sum())} tokens) x {reps1} repetitions, "
                                        f"{t1:.1f} s wall, attention only"}}


def run_ours(args, world, rank, local):
    import torch
    import paged_kv_cache_32_gb300 as pa
    pa.build()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    w = W.WORKLOADS[args.workload](materialize=False)
    if args.partition is not None:
        w.partition_size = args.partition
    ds = DeviceStep(w, device)
    sampler = clock_sampler(local)
    sampler.start()
    ms_step, call_ms, decode_ms, write_ms, (t0, t1) = time_device(ds, args.steps, args.warmup, world)
    ms_step = all_max(ms_step, world)
    # the decode call's duration: the timed region's mean step when the step is that call alone,
    # else the mean of the back-to-back calls
    dec_ms = ms_step if ds.single_call else all_max(call_ms, world)
    e2e_ms, e2e_copy_ms, h2d, d2h = time_e2e(ds, args.steps, args.warmup, world)
    e2e_ms = all_max(e2e_ms, world)
    e2e_copy_ms = all_max(e2e_copy_ms, world)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    err = int(ds.err.item())
    if err:
        raise RuntimeError(f"device error flag {err}")
    if not bool(torch.isfinite(ds.out.float()).all()):
        raise RuntimeError("non-finite decode output")

    kv = w.kv_bytes()
    value = world * kv / (ms_step * 1e-3) / 1e9
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs") if peaks else None
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    dbytes = ds.decode_bytes()
    achieved = dbytes / (dec_ms * 1e-3) / 1e9
    traffic = ncu_traffic(args.workload)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded; K/V pools drawn N(0,1) on device)",
        "config": {"workload": args.workload, "description": WORKLOAD_DESC.get(args.workload, args.workload),
                   "num_seqs": w.num_seqs, "tokens": int(w.seq_lens.sum()), "kv_bytes_per_step": kv,
                   "partition_size": ds.part, "l2": "inputs larger than L2 (K/V working set "
                   f"{kv / 1e9:.2f} GB vs 0.13 GB L2); no flush", "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * w.num_seqs / (ms_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": ("pa_decode_append (decode_tc_kernel with the append fused in + "
                                                 "merge_kernel when split)" if ds.fused else
                                                 "pa_decode (decode_tc_kernel + merge_kernel when split)"),
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": dbytes, "launch_ms": round(dec_ms, 5),
                     "launch_ms_stat": (f"mean over the timed region of {args.steps} steps (the step is this call)"
                                        if ds.single_call else
                                        f"mean of {args.steps} back-to-back calls between two CUDA events"),
                     "launch_ms_events_median": round(statistics.median(decode_ms), 5),
                     "launch_ms_events_mean": round(statistics.mean(decode_ms), 5),
                     "nominal_peak": NOMINAL_HBM_GBS},
        "writes_ms": round(statistics.median(write_ms), 5),
        "e2e": {"value": round(world * kv / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "method": "inputs and output in pinned host memory, read and written in place by the kernels over "
                          "the host link (zero-copy)",
                "copy_path": {"value": round(world * kv / (e2e_copy_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                              "ms_per_step": round(e2e_copy_ms, 5),
                              "method": "one cudaMemcpyAsync of the inputs in, the step on device buffers, the output "
                                        "copied back"}},
        "gpu_launches": ds.launches_per_step() * args.steps,
        "block_manager": {"step_us": round(block_manager_step_us(w), 2), "seqs": w.num_seqs,
                          "ops": "append_slots + build_tables (C++ manager in libpa)"},
        "clocks": clocks,
    }
    if not args.no_extra and world == 1:
        line["other_workloads"] = {}
        sampler_x = clock_sampler(local)
        sampler_x.start()
        for name in args.extra:
            if name == args.workload:
                continue
            base, _, suffix = name.partition("+")
            wx = W.WORKLOADS[base](materialize=False)
            dx = DeviceStep(wx, device, alibi=suffix == "alibi")
            steps_x = max(EXTRA_STEPS, args.steps)
            # the decode call's own fraction: a step that fuses its append is timed as a step, and its
            # attention alone as back-to-back pa_decode calls
            msx, callx, dmx, _, (tx0, tx1) = time_device(dx, steps_x, args.warmup, 1,
                                                         call=dx.decode if dx.fused else None)
            if int(dx.err.item()):
                raise RuntimeError(f"device error flag {int(dx.err.item())} in {name}")
            if not bool(torch.isfinite(dx.out.float()).all()):
                raise RuntimeError(f"non-finite decode output in {name}")
            dm = msx if dx.single_call and not dx.fused else callx
            ab = dx.decode_bytes(with_append=False)
            line["other_workloads"][name] = {
                "kv_gbs_step": round(wx.kv_bytes() / (msx * 1e-3) / 1e9, 1), "ms_per_step": round(msx, 5),
                "steps": steps_x, "decode_ms": round(dm, 5),
                "decode_ms_stat": ("mean step of the timed region" if dx.single_call and not dx.fused else
                                   "mean of back-to-back pa_decode calls"),
                "step": "pa_decode_append (append fused)" if dx.fused else
                        "+".join(x for x, t in (("pa_copy_blocks", dx.pairs), ("pa_reshape_and_cache", dx.slots))
                                 if t is not None) + ("+" if dx.pairs is not None or dx.slots is not None else "") +
                        "pa_decode",
                "decode_ms_events_median": round(statistics.median(dmx), 5),
                "decode_achieved_gbs": round(ab / (dm * 1e-3) / 1e9, 1),
                "decode_frac": round(ab / (dm * 1e-3) / 1e9 / peak, 4), "tokens_per_s": round(wx.num_seqs / (msx * 1e-3), 1),
                "window": (tx0, tx1)}
            if name == "shared_prefix_f16":
                line["other_workloads"][name]["unique_kv_bytes"] = wx.unique_kv_bytes()
            del dx
            torch.cuda.empty_cache()
        sampler_x.stop()
        for name, rec in line["other_workloads"].items():
            rec["clocks"] = sampler_x.summary(*rec.pop("window"))
    if not args.no_extra and world == 1 and args.prefill:
        line["prefill"] = bench_prefill(args.prefill, device, max(5, min(args.steps, 20)), args.warmup, peaks)
        torch.cuda.empty_cache()
        for name in args.prefill_extra:
            line.setdefault("prefill_other", {})[name] = bench_prefill(name, device, max(5, min(args.steps, 20)),
                                                                        args.warmup, peaks)
            torch.cuda.empty_cache()
    if not args.no_extra and world == 1 and not args.no_secondary:
        line["secondary"] = bench_secondary(device, max(5, min(args.steps, 50)), args.warmup, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if "other_workloads" in line:
        line["targets"] = targets_summary(line, peak)  # last key: the records keep the line's tail
    if rank == 0:
        print(json.dumps(line), flush=True)


# decode workloads that carry the >= 0.75-of-peak bandwidth target (GQA and long context), and the FP8 ones
TARGET_WORKLOADS = ("gqa_bf16", "long_bf16_b16", "long_bf16_b32", "long_bf16_b64", "mha_fp8", "gqa_fp8")
EXTRA_STEPS = 200  # timed steps of every non-headline decode workload (each step is 0.1-0.3 ms)


def targets_summary(line, peak):
    """Compact per-workload decode fractions of the HBM peak, with the clocks seen while each was timed."""
    out = {"peak_gbs": peak, "stat": "decode call: mean over the workload's timed steps where the step is that "
                                     "call, else over back-to-back calls"}
    for name in TARGET_WORKLOADS + (line["config"]["workload"],):
        rec = line["other_workloads"].get(name)
        if rec is None and name == line["config"]["workload"]:
            rf = line["roofline"]
            rec = {"decode_frac": rf["frac"], "decode_achieved_gbs": rf["achieved"], "decode_ms": rf["launch_ms"],
                   "clocks": line["clocks"]}
        if rec is None:
            continue
        c = rec.get("clocks") or {}
        out[name] = {"frac": rec["decode_frac"], "gbs": rec["decode_achieved_gbs"], "ms": rec["decode_ms"],
                     "sm_mhz": c.get("sm_mhz"), "reasons": c.get("reasons")}
    return out


def bench_prefill(name: str, device, steps: int, warmup: int, peaks):
    """Chunked prefill on the tensor cores: the chunk's K/V append and the
    attention call, timed per launch with CUDA events on the launching stream.
    Its roofline is the dense bf16 tensor peak: algorithmic FLOPs (4 D Hq per
    visible (query, key) pair) over the attention launch's duration."""
    import torch
    w = W.WORKLOADS[name](materialize=False)
    ps = PrefillDeviceStep(w, device)
    sampler = clock_sampler(torch.cuda.current_device())
    sampler.start()
    ms_step, att, att_ms, write_ms, (t0, t1) = time_device(ps, steps, warmup, 1)
    sampler.stop()
    if int(ps.err.item()):
        raise RuntimeError(f"device error flag {int(ps.err.item())} in prefill")
    if not bool(torch.isfinite(ps.out.float()).all()):
        raise RuntimeError(f"non-finite prefill output in {name}")
    flops = w.prefill_flops()
    tflops = flops / (att * 1e-3) / 1e12
    peak = (peaks or {}).get("bf16_tflops")  # fp16 and bf16 share the dense tensor rate
    peak_src = "measured (burst)" if peak else "fallback"
    peak = peak or 1900.0
    T = w.num_query_tokens
    return {"workload": name, "description": WORKLOAD_DESC.get(name, name), "query_tokens": T,
            "context_tokens": int(w.seq_lens.sum()), "ms_per_step": round(ms_step, 5),
            "attention_ms": round(att, 5), "attention_ms_stat": f"mean of {steps} back-to-back calls",
            "attention_ms_events_median": round(statistics.median(att_ms), 5),
            "append_ms": round(statistics.median(write_ms), 5),
            "query_tokens_per_s": round(T / (ms_step * 1e-3), 1), "gpu_launches": 2 * steps,
            "roofline": {"bound": "tensor", "kernel": "pa_prefill (prefill_tc_kernel)", "achieved": round(tflops, 1),
                         "peak": peak, "peak_source": peak_src, "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": ncu_traffic(name), "algorithmic_flops_per_launch": flops,
                         "sustained_peak": (peaks or {}).get("bf16_tflops_sustained")},
            "l2": "q + out + K/V of the chunk's sequences exceed L2; no flush",
            "clocks": sampler.summary(t0, t1)}


def run_reference(args, world, rank):
    """CPU fp64 evaluation (the oracle) of the same step on bounded samples."""
    if rank != 0:
        return
    import oracle as O
    w = W.WORKLOADS[args.workload](materialize=False)
    threads = O.max_threads()
    n_take = min(w.num_seqs, 4)
    samples = [W.host_sample(w, [(i * n_take + j) % w.num_seqs for j in range(n_take)], seed=i)
               for i in range(max(1, min(args.steps, 8)))]
    kw = lambda s: dict(dtype=s.dtype, num_kv_heads=s.num_kv_heads, block_size=s.block_size)

    def step(s):
        k, v = s.k_cache.copy(), s.v_cache.copy()
        W.apply_writes_host(s, k, v,
                            lambda kk, vv, pairs: O.copy_blocks(kk, vv, pairs, head_size=s.head_size, **kw(s)),
                            lambda kk, vv, nk, nv, sl: O.reshape_and_cache(kk, vv, nk, nv, sl, **kw(s)))
        O.paged_attention(s.q, k, v, s.block_tables, s.seq_lens, scale=s.scale, threads=threads, **kw(s))
    for i in range(args.warmup):
        step(samples[i % len(samples)])
    t0 = time.perf_counter()
    kv = 0
    for i in range(args.steps):
        s = samples[i % len(samples)]
        step(s)
        kv += s.kv_bytes()
    dt = time.perf_counter() - t0
    value = kv / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "description": WORKLOAD_DESC.get(args.workload, args.workload),
                       "sample_seqs_per_step": n_take},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_take} of {w.num_seqs} sequences per step, CPU fp64 oracle"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mha_f16", choices=sorted(k for k in W.WORKLOADS if not k.startswith("prefill")))
    ap.add_argument("--extra", nargs="*", default=["gqa_bf16", "gqa_bf16+alibi", "long_bf16_b16", "long_bf16_b32",
                                                   "long_bf16_b64", "shared_prefix_f16", "mha_fp8", "gqa_fp8"])
    ap.add_argument("--no-extra", action="store_true", help="time only the headline workload")
    ap.add_argument("--prefill", default="prefill_bf16", help="chunked-prefill workload timed beside decode ('' = none)")
    ap.add_argument("--prefill-extra", nargs="*", default=["prefill_f16"],
                    help="further chunked-prefill workloads, reported under prefill_other")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the block-table, block-size and write-call measurements")
    ap.add_argument("--partition", type=int, default=None,
                    help="tokens per split-KV partition (multiple of the block size; 0 = library default)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
