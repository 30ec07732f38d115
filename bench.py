#!/usr/bin/env python
"""Benchmark of the TurboQuant KV-cache hot path on one GB300 (or N replicas).

One step = the whole hot path on one batch: the fused store of each
sequence's newest token (tq_store) followed by split-K decode attention over
the packed paged cache (tq_decode_attention: stage 1 + stage 2).  Default
workload: the largest single-GPU configuration, Qwen3-32B-shaped decode
(B=64, 64 q / 8 kv heads, head_dim 128, contexts uniform in [16K, 32K],
block_size 64, preset turboquant_k3v4_nc, fp16, 2% Student-t(3)
coordinates, random block-table permutation), synthetic seeded data.

Prints ONE JSON line (rank 0).  `value` is packed-KV bytes read per step
divided by the device-timed step (GB/s), summed over ranks; `e2e` is the same
metric with every step's inputs copied from pinned host memory and the
attention output copied back, inside the timed region.  With the default
workload the line also carries a row per configuration (`configs`: the tiny
case, the Llama-3-8B shape, the Qwen3-32B shape, the 256K-token case, and
the 16K-token mixed-batch store followed by decode over its cache, every
preset), the 1M-token store, the dequantisation and a 32K-256K context sweep.

--impl reference times the CPU oracle (the slow plain-C definition of the
method) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import re
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

from quantized_kv_cache_04_gb300 import workloads as wl  # noqa: E402

SLOT = {"turboquant_k8v4": 196, "turboquant_4bit_nc": 134, "turboquant_k3v4_nc": 118,
        "turboquant_3bit_nc": 102, "turboquant_2bit_nc": 70}
L2_BYTES = 129 * 2**20
NOMINAL_HBM_GBS = 8000.0


def _args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="qwen3_32b",
                   choices=["llama3_8b", "qwen3_32b", "long", "store_mixed", "sweep", "tiny", "store_large"],
                   help="store_large: only the 2^20-token store of --preset (default k3v4_nc)")
    p.add_argument("--preset", default=None, choices=sorted(SLOT))
    p.add_argument("--ctx", type=int, default=None)
    p.add_argument("--batch", type=int, default=None)
    p.add_argument("--splits", type=int, default=None, help="0 = library picks")
    p.add_argument("--soa", action="store_true",
                   help="cache blocks in the SoA byte convention (TQ_LAYOUT_SOA)")
    p.add_argument("--v-threshold", type=float, default=0.0,
                   help="sparse V: rows with softmax factor <= this skip the value sum (0 = dense)")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true", help="skip the store-throughput side run")
    return p.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _describe(w) -> str:
    ctx = (f"ctx {int(w.seq_lens[0])}" if len(set(w.seq_lens.tolist())) == 1
           else f"ctx {int(w.seq_lens.min())}-{int(w.seq_lens.max())}")
    return (f"{w.name} decode: B={w.B}, Hq={w.Hq}, Hk={w.Hk}, D={w.D}, {ctx}, "
            f"bs {w.block_size}, {w.preset}, {w.dtype}")


def _kv_bytes(w) -> int:
    return int(w.seq_lens.astype(np.int64).sum()) * w.Hk * SLOT[w.preset]


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons of the GPU, sampled
    every 2 ms by a thread through NVML (read-only queries, libnvidia-ml
    through ctypes), or every 50 ms through nvidia-smi where NVML cannot be
    loaded.  Started before the warm-up; mark() brackets the timed region."""
    NAMES = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
             0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, uuid: str | None = None):
        self.idx, self.uuid = gpu_index, uuid
        self.rows = []                 # (time, sm_mhz, max_mhz, power_w, reasons bitmask)
        self.windows, self.err, self.source = [], None, None
        self.stop = threading.Event()
        self.proc = None

    def _nvml(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = nv.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.idx), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        clk, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))       # 1 = NVML_CLOCK_SM

        def sample():
            nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            reasons_fn(h, ctypes.byref(rs))
            return (time.time(), float(clk.value), float(mx.value), pw.value / 1000.0, int(rs.value))
        sample()
        return sample

    def _loop_nvml(self, sample):
        while not self.stop.is_set():
            self.rows.append(sample())
            time.sleep(0.002)

    def _loop_smi(self):
        for line in self.proc.stdout:
            r = [x.strip() for x in line.split(",")]
            if len(r) < 7:
                continue
            try:
                bits = sum(b for b, v in zip((0x8, 0x40, 0x20, 0x4), r[3:7]) if v.lower().startswith("active"))
                self.rows.append((time.time(), float(r[0]), float(r[1]), float(r[2]), bits))
            except ValueError:
                pass

    def __enter__(self):
        try:
            sample = self._nvml()
            self.source = "nvml, 2 ms"
            self.t = threading.Thread(target=self._loop_nvml, args=(sample,), daemon=True)
        except Exception as e:
            self.err = f"nvml: {e}"
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi, 50 ms"
                self.t = threading.Thread(target=self._loop_smi, daemon=True)
            except Exception as e2:  # pragma: no cover
                self.err += f"; nvidia-smi: {e2}"
                return self
        self.t.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5.0:
            time.sleep(0.005)            # the sampler is live before the first timed step
        return self

    def mark(self, start: bool):
        if start:
            self.windows.append([time.time(), None])
        elif self.windows:
            self.windows[-1][1] = time.time()

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # pragma: no cover
                self.proc.kill()
        if getattr(self, "t", None):
            self.t.join(timeout=2)

    def summary(self):
        rows = list(self.rows)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.err or "no samples"}
        inside = [r for r in rows for a, b in self.windows if b and a <= r[0] <= b]
        use = inside or rows
        pmax = max(r[3] for r in use)
        load = [r for r in use if r[3] >= 0.25 * pmax] or use
        reasons = sorted({n for r in use for bit, n in self.NAMES.items() if r[4] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in load), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside),
                "power_w_max": round(pmax, 1), "source": self.source,
                "window": "samples inside the timed steps (all samples if none fell inside); "
                          "median SM clock over those at >= 25% of their peak power"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the decode kernels' code (both stages, both stage-1 paths):
    the sources with their // comments removed and whitespace runs folded,
    so that an edit of a comment keeps a recorded measurement valid."""
    h = hashlib.sha256()
    for f in ("tq_decode.cu", "tq_decode_mma.cu", "tq_decode_mma.cuh", "tq_decode_mma_sparse.cu",
              "tq_internal.h", "tq_device.cuh"):
        text = open(os.path.join(ROOT, "quantized_kv_cache_04_gb300", "csrc", f), encoding="utf-8").read()
        code = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def _traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    it was taken on is the one being timed (else null)."""
    sha = kernel_source_hash()
    f = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(f):
        return None
    for line in open(f):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == workload \
                and parts[1] == kernel and parts[2] == sha:
            return float(parts[3])
    return None


# ---------------------------------------------------------------- GPU setup
class Problem:
    """Device-resident cache, queries and per-step inputs of one workload."""

    def __init__(self, w, dev, splits, v_threshold: float = 0.0, soa: bool = False):
        import torch
        import quantized_kv_cache_04_gb300 as tq
        self.w, self.dev = w, dev
        self.vthr = float(v_threshold)
        self.c = tq.TQCache(w.preset_id | (tq.TQ_LAYOUT_SOA if soa else 0), w.num_blocks,
                            w.block_size, w.Hk, device=dev)
        self.c.cache[w.guard_block] = 0xFF          # never read if paging is right
        CH = 32768
        for b in range(w.B):
            n = int(w.seq_lens[b])
            for t0 in range(0, n, CH):
                t1 = min(n, t0 + CH)
                K, V = wl.gen_kv(w, b, t0, t1, dev)
                sm = torch.from_numpy(w.slot_mapping(b, np.arange(t0, t1))).to(dev)
                self.c.store(K, V, sm)
        # the step's new token of every sequence: its last position
        nk, nv = [], []
        for b in range(w.B):
            n = int(w.seq_lens[b])
            K, V = wl.gen_kv(w, b, n - 1, n, dev)
            nk.append(K[0])
            nv.append(V[0])
        self.new_k = torch.stack(nk).contiguous()
        self.new_v = torch.stack(nv).contiguous()
        last = np.array([w.slot_mapping(b, [int(w.seq_lens[b]) - 1])[0] for b in range(w.B)],
                        np.int64)
        self.new_sm = torch.from_numpy(last).to(dev)
        self.q = wl.gen_q(w, dev).contiguous()
        self.bt = torch.from_numpy(w.block_table).to(dev)
        self.sl = torch.from_numpy(w.seq_lens).to(dev)
        self.max_len = int(w.seq_lens.max())
        self.S = (splits if splits else w.num_splits) or tq.tq_decode_pick_splits(
            self.c.preset, w.D, w.B, w.Hq, w.Hk, self.max_len)
        self.ws = self.c.workspace(w.B, w.Hq, self.S)
        self.out = torch.empty((w.B, w.Hq, w.D), dtype=self.q.dtype, device=dev)
        self.lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()

    def store(self):
        self.c.store(self.new_k, self.new_v, self.new_sm)

    def decode(self):
        self.c.decode(self.q, self.bt, self.sl, self.max_len, self.out, self.lse, self.ws,
                      num_splits=self.S, v_threshold=self.vthr)


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (the slowest replica's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(kv_bytes_per_rank: int, step_ms: float, world: int) -> float:
    """Whole-job GB/s: every replica reads its own cache each step, and the
    step time is the slowest replica's."""
    return world * kv_bytes_per_rank / (step_ms * 1e-3) / 1e9


def time_device(p: Problem, steps: int, warmup: int, world: int, gpu_index: int, gpu_uuid=None):
    import torch
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index, gpu_uuid) as clk:
        for _ in range(warmup):
            p.store()
            p.decode()
        torch.cuda.synchronize()
        _barrier(world)
        torch.cuda.synchronize()
        clk.mark(True)
        # the steps back to back: no event between the store and the decode,
        # whose stage 1 is launched as a programmatic dependent of the store
        e0.record(st)
        for i in range(steps):
            p.store()
            p.decode()
        e1.record(st)
        torch.cuda.synchronize()
        clk.mark(False)
        # the decode calls alone, back to back: the per-call duration of the
        # dominant kernels (stage 1 + stage 2) for the roofline
        e2.record(st)
        for i in range(steps):
            p.decode()
        e3.record(st)
        torch.cuda.synchronize()
    _barrier(world)
    total_ms = e0.elapsed_time(e1)
    dec_ms = e2.elapsed_time(e3) / steps
    return total_ms, dec_ms, clk.summary()


def time_calls(fn, calls: int, flush_bytes: int = 0) -> float:
    """Mean device time of fn() in ms: back to back between two events, or,
    with flush_bytes > 0 (inputs smaller than L2), the median of single
    calls with a buffer of that size written in between (L2 flushed)."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    if flush_bytes <= 0:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(st)
        for _ in range(calls):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / calls
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device="cuda")
    ts = []
    for _ in range(calls):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    del flush
    return float(np.median(ts))


def decode_row(w, dev, peak_gbs: float, calls: int = 50) -> dict:
    """One configuration's row: the decode call (stage 1 + stage 2) and the
    step (store of every sequence's newest token + decode), the library's
    split count (or the configuration's own).  Inputs larger than L2 run
    back to back; smaller ones are timed one call at a time with L2 flushed
    in between."""
    import torch
    p = Problem(w, dev, None)
    kvb = _kv_bytes(w)
    small = kvb <= L2_BYTES
    flush = 256 * 2**20 if small else 0

    def step():
        p.store()
        p.decode()
    dec_ms = time_calls(p.decode, calls, flush)
    step_ms = time_calls(step, calls, flush)
    row = {"workload": _describe(w), "preset": w.preset, "batch": w.B, "q_heads": w.Hq,
           "kv_heads": w.Hk, "block_size": w.block_size, "num_splits": p.S,
           "kernel": "tensor-core" if _kernel_kind(p) == 1 else "CUDA-core",
           "packed_kv_bytes": kvb, "decode_ms": round(dec_ms, 5), "step_ms": round(step_ms, 5),
           "gbs": round(kvb / dec_ms / 1e6, 1), "frac_of_measured_hbm": round(kvb / dec_ms / 1e6 / peak_gbs, 4),
           "decode_tok_s": round(w.B / (step_ms * 1e-3), 1),
           "l2": "flushed between calls (inputs smaller than L2)" if small else "inputs larger than L2"}
    del p
    torch.cuda.empty_cache()
    return row


def _kernel_kind(p) -> int:
    import quantized_kv_cache_04_gb300 as tq
    return tq.tq_decode_kernel_kind(p.c.preset, p.w.D, p.w.Hq, p.w.Hk)


def other_shape_rows(dev, peak_gbs: float) -> list:
    """Decode at 32K contexts in shapes outside the configurations: groups of
    16 query heads (128 q / 8 kv heads: two CTAs of 8 query heads per kv
    head), 2 or 4 kv heads with Lloyd-Max keys (token rows that are not
    whole 16-byte units), and 1 or 3 kv heads with 3-bit keys (token rows
    not 4-byte aligned: the CUDA-core stage 1)."""
    rows = []
    for preset, hq, hk in (("turboquant_k8v4", 128, 8), ("turboquant_k3v4_nc", 128, 8),
                           ("turboquant_4bit_nc", 8, 2), ("turboquant_k3v4_nc", 8, 2),
                           ("turboquant_3bit_nc", 16, 4), ("turboquant_k3v4_nc", 8, 1),
                           ("turboquant_k3v4_nc", 12, 3)):
        w = wl.make("sweep", preset=preset, ctx=32768, q_heads=hq, kv_heads=hk)
        rows.append(decode_row(w, dev, peak_gbs, 30))
    return rows


def config_rows(dev, peak_gbs: float, headline: dict) -> dict:
    """A row per configuration: 1 tiny, 2 Llama-3-8B shape, 3 Qwen3-32B shape
    (the headline's own numbers), 4 the 256K-token case, 5 the mixed-batch
    store of 16,384 tokens in one call and the decode (32 query heads) over
    the resulting cache, every preset."""
    rows = {"1_tiny": decode_row(wl.make("tiny"), dev, peak_gbs, 50),
            "2_llama3_8b": decode_row(wl.make("llama3_8b"), dev, peak_gbs, 100),
            "3_qwen3_32b": headline,
            "4_long": decode_row(wl.make("long"), dev, peak_gbs, 30)}
    store = time_store_mixed(dev)
    mixed = {}
    for preset in SLOT:
        r = decode_row(wl.make("store_mixed", preset=preset), dev, peak_gbs, 50)
        r["store"] = store[preset]
        mixed[preset] = r
    rows["5_store_mixed"] = mixed
    return rows


def time_e2e(p: Problem, steps: int, warmup: int, world: int):
    """Same step with host inputs: pinned H2D of q, new K/V, slot mapping,
    block table and seq_lens, then D2H of the attention output and LSE.  The
    step's inputs sit packed in one pinned buffer and travel in one copy into
    one device buffer whose views the store and decode take; the output and
    LSE share one device buffer and come back in one copy."""
    import torch
    st = torch.cuda.current_stream()

    def layout(ts):
        offs, o = [], 0
        for t in ts:
            offs.append(o)
            o += (t.numel() * t.element_size() + 15) // 16 * 16
        return offs, o

    def view(buf, off, t):
        n = t.numel() * t.element_size()
        return buf[off:off + n].view(t.dtype).view(t.shape)

    ins = [p.q, p.new_k, p.new_v, p.new_sm, p.bt, p.sl]
    in_offs, in_bytes = layout(ins)
    hin = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(in_bytes, dtype=torch.uint8, device=p.dev)
    for t, o in zip(ins, in_offs):
        view(hin, o, t).copy_(t.cpu())
    p.q, p.new_k, p.new_v, p.new_sm, p.bt, p.sl = [view(din, o, t) for t, o in zip(ins, in_offs)]
    outs = [p.out, p.lse]
    out_offs, out_bytes = layout(outs)
    dout = torch.empty(out_bytes, dtype=torch.uint8, device=p.dev)
    hout = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    p.out, p.lse = [view(dout, o, t) for t, o in zip(outs, out_offs)]
    h2d, d2h = in_bytes, out_bytes

    def step():
        din.copy_(hin, non_blocking=True)
        p.store()
        p.decode()
        hout.copy_(dout, non_blocking=True)

    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    _barrier(world)
    e0.record(st)
    for _ in range(steps):
        step()
    e1.record(st)
    torch.cuda.synchronize()
    _barrier(world)
    return e0.elapsed_time(e1) / steps, h2d, d2h


def time_store_mixed(dev):
    """Store throughput side run: 16384 new tokens of 16 varlen sequences,
    bs 32, 8 kv heads, every preset in turn (fp16 inputs)."""
    import torch
    import quantized_kv_cache_04_gb300 as tq
    res = {}
    for preset in SLOT:
        w = wl.make("store_mixed", preset=preset)
        ks, vs, sms = [], [], []
        for b in range(w.B):
            n = int(w.seq_lens[b])
            K, V = wl.gen_kv(w, b, 0, n, dev)
            ks.append(K)
            vs.append(V)
            sms.append(w.slot_mapping(b, np.arange(n)))
        K, V = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
        sm = torch.from_numpy(np.concatenate(sms)).to(dev)
        c = tq.TQCache(preset, w.num_blocks, w.block_size, w.Hk, device=dev)
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
        for _ in range(5):
            c.store(K, V, sm)
        ts = []
        for _ in range(30):
            flush.zero_()                           # evict L2 between runs
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            c.store(K, V, sm)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = float(np.median(ts))
        N = K.shape[0]
        moved = N * w.Hk * (2 * 2 * w.D + SLOT[preset]) + 8 * N
        res[preset] = {"tokens": N, "ms": round(ms, 4), "mtok_s": round(N / ms / 1e3, 2),
                       "gbs": round(moved / ms / 1e6, 1)}
    return res


def time_store_large(dev, tokens: int = 1 << 20, presets=tuple(SLOT)):
    """Store throughput at scale: 2^20 tokens (16 sequences of 64K, the
    Llama-3-8B shape: 8 kv heads, bs 16, bf16) in one call, every preset;
    median of 10 calls, L2 flushed between them."""
    import torch
    import quantized_kv_cache_04_gb300 as tq
    res = {}
    for preset in presets:
        w = wl.make("sweep", ctx=tokens // 16, preset=preset)
        ks, vs, sms = [], [], []
        for b in range(w.B):
            n = int(w.seq_lens[b])
            K, V = wl.gen_kv(w, b, 0, n, dev)
            ks.append(K)
            vs.append(V)
            sms.append(w.slot_mapping(b, np.arange(n)))
        K, V = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
        del ks, vs
        sm = torch.from_numpy(np.concatenate(sms)).to(dev)
        c = tq.TQCache(preset, w.num_blocks, w.block_size, w.Hk, device=dev)
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
        for _ in range(3):
            c.store(K, V, sm)
        ts = []
        for _ in range(10):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            c.store(K, V, sm)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = float(np.median(ts))
        N = K.shape[0]
        moved = N * w.Hk * (2 * 2 * w.D + SLOT[preset]) + 8 * N
        res[preset] = {"tokens": N, "ms": round(ms, 4), "mtok_s": round(N / ms / 1e3, 2),
                       "gbs": round(moved / ms / 1e6, 1)}
        del K, V, sm, c, flush
        torch.cuda.empty_cache()
    return res


def time_dequant(p: "Problem", peak_gbs: float, calls: int = 20):
    """Dequantisation side run: every cached token of the workload back to
    fp16 K and V (tq_dequant over the whole slot list).  Bytes = slots read +
    slot mapping + K and V written; outputs and cache together exceed L2."""
    import torch
    w = p.w
    sm = torch.from_numpy(np.concatenate([w.slot_mapping(b, np.arange(int(w.seq_lens[b])))
                                          for b in range(w.B)])).to(p.dev)
    N = sm.numel()
    ko = torch.empty((N, w.Hk, w.D), dtype=torch.float16, device=p.dev)
    vo = torch.empty_like(ko)
    for _ in range(3):
        p.c.dequant(sm, ko, vo)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(calls):
        p.c.dequant(sm, ko, vo)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / calls
    nbytes = N * w.Hk * SLOT[w.preset] + 8 * N + 2 * N * w.Hk * w.D * 2
    del ko, vo
    torch.cuda.empty_cache()
    return {"tokens": N, "kv_heads": w.Hk, "out_dtype": "f16", "ms": round(ms, 5),
            "bytes": nbytes, "gbs": round(nbytes / ms / 1e6, 1),
            "frac_of_measured_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}


def time_long_context(dev, peak_gbs: float, ctxs=(32768, 65536, 131072, 262144), presets=tuple(SLOT),
                      calls: int = 50):
    """Decode-only side run at long contexts: the Llama-3-8B shape (bs 16)
    for every preset at each context with batch 2^20 / ctx, the library's
    split count; mean decode-call time over `calls` back-to-back calls
    (inputs > L2)."""
    import torch
    res = []
    for ctx, preset in [(c, pr) for pr in presets for c in ctxs]:
        w = wl.make("sweep", ctx=ctx, preset=preset)
        p = Problem(w, dev, None)
        for _ in range(5):
            p.decode()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(calls):
            p.decode()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / calls
        kvb = _kv_bytes(w)
        res.append({"ctx": ctx, "batch": w.B, "preset": w.preset, "num_splits": p.S,
                    "decode_ms": round(ms, 5), "gbs": round(kvb / ms / 1e6, 1),
                    "frac_of_measured_hbm": round(kvb / ms / 1e6 / peak_gbs, 4)})
        del p
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- oracle timing
def _oracle_sample(w, tokens: int, seq: int = 0):
    """Oracle cache for the first `tokens` positions of sequence `seq` (all kv
    heads), built by the oracle from CPU-drawn inputs of the same workload."""
    import oracle as orc
    n = min(tokens, int(w.seq_lens[seq]))
    K, V = wl.gen_kv(w, seq, 0, n, "cpu")
    lay = orc.layout(w.preset_id)
    s = orc.signs(w.D, 42)
    c32, m32 = ((np.zeros(1, np.float32),) * 2 if lay["key_fp8"]
                else orc.codebook(w.D, lay["key_bits"]))
    bs = w.block_size
    nb = (n + bs - 1) // bs
    cache = np.zeros((nb, bs, w.Hk, lay["slot_size_aligned"]), np.uint8)
    t0 = time.perf_counter()
    orc.store(w.preset_id, K.float().numpy(), V.float().numpy(), np.arange(n, dtype=np.int64),
              cache, bs, s, c32, m32)
    store_s = time.perf_counter() - t0
    bt = np.arange(nb, dtype=np.int32)[None, :]
    q = wl.gen_q(w, "cpu")[seq:seq + 1].float().numpy()
    return dict(n=n, cache=cache, bt=bt, q=q, s=s, c32=c32, store_s=store_s,
                bytes=n * w.Hk * SLOT[w.preset])


def _oracle_decode_once(w, smp):
    import oracle as orc
    t0 = time.perf_counter()
    orc.decode_dense(w.preset_id, smp["q"], smp["cache"], smp["bt"],
                     np.array([smp["n"]], np.int32), w.Hk, w.block_size, smp["s"], smp["c32"])
    return time.perf_counter() - t0


def _cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm
    implementer and part numbers)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    fields = {}
    for line in info:
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    return " ".join(f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields) or "unknown"


def cpu_baseline(w, budget_s: float = 10.0):
    """The oracle's decode on the host, over whole sequences of the workload
    in order until about budget_s seconds of decode work (or all of them):
    one thread, then the same sequences decoded concurrently by one thread
    per host core (the oracle's C calls run without the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    probe = _oracle_sample(w, 256)
    per_tok = _oracle_decode_once(w, probe) / probe["n"]
    nbytes, dec_s, store_s, ntok, nseq = 0, 0.0, 0.0, 0, 0
    samples = []
    for seq in range(w.B):
        # a sequence longer than the remaining budget contributes a prefix
        n = min(int(w.seq_lens[seq]), max(256, int((budget_s - dec_s) / per_tok)))
        smp = _oracle_sample(w, n, seq)
        dec_s += _oracle_decode_once(w, smp)
        store_s += smp["store_s"]
        nbytes += smp["bytes"]
        ntok += smp["n"]
        nseq += 1
        samples.append(smp)
        if dec_s >= budget_s:
            break
    ncpu = os.cpu_count() or 1
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=ncpu) as ex:
        list(ex.map(lambda smp: _oracle_decode_once(w, smp), samples))
    par_s = time.perf_counter() - t0
    return {"value": round(nbytes / dec_s / 1e9, 6), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "cpu_model": _cpu_model(), "nproc": ncpu,
            "multi_core": {"value": round(nbytes / par_s / 1e9, 6), "unit": "GB/s",
                           "cores": min(ncpu, len(samples)),
                           "sample": f"the same {len(samples)} sequences, one per thread "
                                     f"({par_s:.1f} s wall)"},
            "sample": (f"sequences 0..{nseq - 1} of {w.B} in order ({ntok} tokens; a sequence "
                       f"past the budget contributes a prefix), all {w.Hk} kv heads, "
                       f"{w.Hq // w.Hk} q heads each: dense fp64 decode over the oracle's cache "
                       f"({dec_s:.1f} s); the oracle's store of the same tokens took {store_s:.1f} s"),
            "store_tok_s": round(ntok / store_s, 1)}


def run_reference(args, w, rank, world):
    """Reference arm: the CPU oracle timed on the host cores, each step one
    decode of a bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return
    probe = _oracle_sample(w, 256)
    t = _oracle_decode_once(w, probe)
    budget = 120.0 / max(1, args.steps + args.warmup)     # whole run ~2 minutes
    tokens = int(min(int(w.seq_lens[0]), max(16, 256 * budget / max(t, 1e-6))))
    smp = _oracle_sample(w, tokens)
    for _ in range(args.warmup):
        _oracle_decode_once(w, smp)
    ts = [_oracle_decode_once(w, smp) for _ in range(args.steps)]
    step_s = float(np.mean(ts))
    val = smp["bytes"] / step_s / 1e9
    sample = (f"sequence 0, first {smp['n']} tokens x {w.Hk} kv heads x {w.Hq // w.Hk} q heads "
              f"per step: dense fp64 oracle decode over the oracle's cache")
    print(json.dumps({
        "impl": "reference", "metric": "decode-attn HBM GB/s on packed KV", "value": round(val, 6),
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _describe(w), "sample_tokens": smp["n"]},
        "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_store_large(args, rank):
    """Only the 2^20-token store of one preset (for profiling the store)."""
    import torch
    import quantized_kv_cache_04_gb300 as tq
    if args.impl == "reference" or not torch.cuda.is_available():
        print(json.dumps({"impl": args.impl, "unavailable": "the store-only mode times the GPU store"}))
        return
    tq.load(build_if_missing=True)
    dev = torch.device("cuda", 0)
    preset = args.preset or "turboquant_k3v4_nc"
    r = time_store_large(dev, presets=(preset,))[preset]
    if rank == 0:
        print(json.dumps({"metric": "store Mtok/s", "value": r["mtok_s"], "unit": "Mtok/s",
                          "preset": preset, "store": r}), flush=True)


def main():
    args = _args()
    rank, world, local = _dist()
    if args.workload == "store_large":
        run_store_large(args, rank)
        return
    w = wl.make(args.workload, preset=args.preset, ctx=args.ctx, batch=args.batch)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    import torch
    assert torch.cuda.is_available(), "bench.py --impl ours needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import quantized_kv_cache_04_gb300 as tq
    tq.load(build_if_missing=True)
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    if len(vis) > local and vis[local].strip().isdigit():
        gpu_index = int(vis[local])
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # pragma: no cover
        gpu_uuid = None

    p = Problem(w, dev, args.splits, args.v_threshold, args.soa)
    assert args.warmup >= 3
    total_ms, dec_ms, clocks = time_device(p, args.steps, args.warmup, world, gpu_index, gpu_uuid)
    step_ms = _max_over_ranks(total_ms / args.steps, world)
    dec_ms = _max_over_ranks(dec_ms, world)
    kvb = _kv_bytes(w)
    value = _job_value(kvb, step_ms, world)

    e2e_steps = args.e2e_steps or max(10, min(args.steps, 500))
    e2e_ms, h2d, d2h = time_e2e(p, e2e_steps, 3, world)
    e2e_ms = _max_over_ranks(e2e_ms, world)
    out_ok = bool(torch.isfinite(p.out.float()).all().item())

    peak, peak_kind = _peaks()
    achieved = kvb / (dec_ms * 1e-3) / 1e9
    line = {
        "metric": "decode-attn HBM GB/s on packed KV", "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": _describe(w), "preset": w.preset, "batch": w.B,
                   "seq_len": int(w.seq_lens.max()), "block_size": w.block_size,
                   "num_splits": p.S, "sparse_v_threshold": args.v_threshold,
                   "block_layout": "soa" if args.soa else "aos", "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": f"inputs larger than L2 ({kvb / 1e6:.0f} MB packed KV > 129 MiB L2)"
                   if kvb > L2_BYTES else "inputs smaller than L2 (not flushed)"},
        "e2e": {"value": round(world * kvb / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5), "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": _traffic(args.workload, "tq_decode_attention"),
                     "kernel": "tq_decode_attention (stage1 + stage2): CUDA events around the same number of back-to-back calls after the timed steps",
                     "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "algorithmic_bytes": kvb},
        "tokens_per_s": round(world * w.B / (step_ms * 1e-3), 1),
        "kv_tokens_per_s": round(world * int(w.seq_lens.sum()) / (step_ms * 1e-3), 1),
        "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "decode_ms": round(dec_ms, 5),
        "output_finite": out_ok,
    }
    default = (args.workload == "qwen3_32b" and args.preset is None and args.ctx is None
               and args.batch is None and not args.soa and args.v_threshold == 0.0)
    if not args.no_extra and rank == 0:
        line["dequant"] = time_dequant(p, peak)
        head = {"workload": _describe(w), "preset": w.preset, "batch": w.B, "q_heads": w.Hq,
                "kv_heads": w.Hk, "block_size": w.block_size, "num_splits": p.S,
                "kernel": "tensor-core" if _kernel_kind(p) == 1 else "CUDA-core",
                "packed_kv_bytes": kvb, "decode_ms": round(dec_ms, 5), "step_ms": round(step_ms, 5),
                "gbs": round(achieved, 1), "frac_of_measured_hbm": round(achieved / peak, 4),
                "decode_tok_s": round(w.B / (step_ms * 1e-3), 1), "l2": "inputs larger than L2",
                "note": "the headline run above"}
        del p
        torch.cuda.empty_cache()
        if default:
            line["configs"] = config_rows(dev, peak, head)
            line["long_context"] = time_long_context(dev, peak)
            line["other_shapes"] = other_shape_rows(dev, peak)
        line["store_1m"] = time_store_large(dev)
        line["store_mtok_s"] = {k: v["mtok_s"] for k, v in line["store_1m"].items()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
