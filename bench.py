"""Benchmark: decode attention over the Hadamard-rotated 4-bit KV cache.

One step = one new token through 16 attention layers: per layer, store the
token's K/V rows (4 KV heads, head_dim 256) into the 4-bit cache, rotate the
24 query heads, split-T decode over T = context + 1 keys (512-key partitions
plus the tail), log-sum-exp merge and rotate back.  The main line is the
32,768-token context (16 layers, heavy-tailed bf16 data); the 262,144-token
context is measured in the same run and reported under "long_context".

value   = microseconds per layer-token (lower is better), device time with the
          inputs resident in HBM; the 16 layer caches (604 MB at 32K, 4.8 GB at
          262K) exceed the 129 MB L2, so every step reads the cache from HBM.
e2e     = the same step through the C ABI with the step's inputs copied from
          pinned host memory and the outputs copied back inside the timed region.
roofline= the decode kernel: algorithmic bytes (codes + scales of K and V of every
          attended position, 1152 B per position per layer) / average launch time
          measured with CUDA events on the launching stream; peak = measured HBM
          copy bandwidth.
clocks  = SM clock and throttle reasons sampled through NVML every 0.5 ms inside
          the timed region (nvidia-smi every 100 ms where NVML cannot be loaded).
--impl reference times the CPU oracle on the host cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS, HK, HQ, D, PS = 16, 4, 24, 256, 16
KERNELS_PER_LAYER = 3  # store + query rotation (one launch), split-T decode, merge
# DRAM bytes of one decode launch (dram__bytes_read.sum + dram__bytes_write.sum
# from an ncu capture of the current kernel at each context); to be dropped
# whenever the kernel changes.
TRAFFIC_BYTES = {32768: 37867008 + 0, 262144: 302277120 + 10575104}
BYTES_PER_POS_LAYER = HK * 2 * (D // 2 + 2 * (D // 32))   # 1152


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--context", type=int, default=32768)
    ap.add_argument("--long-context", type=int, default=262144)
    ap.add_argument("--no-long", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the other hot-path rows (batched decode, prefill, "
                    "fp8, bf16 cache, store)")
    ap.add_argument("--only", choices=["batched", "prefill", "fp8", "bf16", "q4_0", "window", "tq4", "fp8_prefill", "fused_merge"], default=None,
                    help="run only one of the other hot-path rows and print its measurement (for profiling)")
    ap.add_argument("--layers", type=int, default=16, help="layers per step (16 for the benchmark; fewer "
                    "only to profile a small case)")
    args = ap.parse_args()
    global LAYERS
    LAYERS = args.layers
    return args


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*), mapped to the
# names of nvidia-smi's clocks_event_reasons fields; power-brake slowdown is
# one of the causes nvidia-smi reports as hw_slowdown.
NVML_REASONS = ((0x8, "hw_slowdown"), (0x80, "hw_slowdown"), (0x40, "hw_thermal_slowdown"),
                (0x20, "sw_thermal_slowdown"), (0x4, "sw_power_cap"))


def nvml_reason_names(mask):
    return sorted({name for bit, name in NVML_REASONS if mask & bit})


class _Nvml:
    """SM clock, its maximum and the clock-event reasons, read through the
    driver's management library; one read takes microseconds."""

    def __init__(self, index):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.lib, self.ct = lib, ctypes
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            lib.nvmlShutdown()
            raise OSError("no NVML handle for device %d" % index)
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)

    def read(self):
        ct = self.ct
        mhz, mask = ct.c_uint(0), ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, ct.c_int(1), ct.byref(mhz)) != 0:
            return None
        if self.reasons_fn(self.h, ct.byref(mask)) != 0:
            return None
        return float(mhz.value), int(mask.value)

    def close(self):
        self.lib.nvmlShutdown()


class Clocks:
    """Samples the SM clock and the throttle reasons.  Through NVML a thread
    polls every half millisecond and keeps only the samples taken between
    begin() and end() (the timed region, which at 32K lasts a few
    milliseconds); without NVML, nvidia-smi samples every 100 ms for the whole
    block."""

    def __init__(self, index=0):
        self.samples, self.proc, self.index = [], None, index
        self.nvml, self.active, self.stop = None, False, False
        self.source = None

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.index)
            self.source = "nvml"
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def begin(self):
        self.active = True

    def end(self):
        self.active = False

    def _poll(self):
        while not self.stop:
            if self.active:
                r = self.nvml.read()
                if r is not None:
                    mhz, mask = r
                    self.samples.append((mhz, self.nvml.max_mhz, nvml_reason_names(mask)))
            time.sleep(0.0005)

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                mhz, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.samples.append((mhz, mx, [names[i] for i in range(4) if parts[2 + i].lower() == "active"]))

    def __exit__(self, *a):
        self.stop = True
        if self.nvml:
            self.t.join(timeout=5)
            self.nvml.close()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        return clock_summary(self.samples, self.source)


def clock_summary(samples, source):
    """samples: (sm MHz, max SM MHz, [active reason names]) per read."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0, "source": source}
    return {"sm_mhz": statistics.median(s[0] for s in samples), "sm_max_mhz": max(s[1] for s in samples),
            "reasons": sorted({r for s in samples for r in s[2]}), "samples": len(samples), "source": source}


def reduce_max_over_ranks(x, world, device):
    """Max of a host float over all ranks (replicas time independently; the job
    time is the slowest replica's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def aggregate_us_per_unit(max_elapsed_ms, units_per_rank, world):
    """Whole-job time per unit: the slowest replica's elapsed time divided by the
    units all replicas processed."""
    return max_elapsed_ms * 1e3 / (units_per_rank * world)


# --------------------------------------------------------------------------- workload

class Workload:
    """16 layers of 4-bit caches holding `context` positions, plus the new token's
    K/V rows and queries for each (step, layer)."""

    def __init__(self, K, synth, torch, context, n_inputs, seed, device):
        self.K, self.torch = K, torch
        self.context = context
        self.T = context + 1
        self.n_pages = (self.T + PS - 1) // PS
        self.caches = []
        dev = device
        for layer in range(LAYERS):
            c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, self.n_pages, device=dev)
            chunk = 32768
            for s0 in range(0, context, chunk):
                n = min(chunk, context - s0)
                k = synth.heavy_tailed((n, HK, D), dev, seed, layer, "k", s0, subset=(seed, layer, "k"))
                v = synth.heavy_tailed((n, HK, D), dev, seed, layer, "v", s0, subset=(seed, layer, "v"))
                K.store(c, k, v, torch.arange(s0, s0 + n, dtype=torch.int32, device=dev))
            self.caches.append(c)
        # per (input set, layer): the new token's K/V rows and the queries
        self.new_k = torch.stack([synth.heavy_tailed((n_inputs, 1, HK, D), dev, seed, layer, "newk",
                                                     subset=(seed, layer, "k")) for layer in range(LAYERS)], 1)
        self.new_v = torch.stack([synth.heavy_tailed((n_inputs, 1, HK, D), dev, seed, layer, "newv",
                                                     subset=(seed, layer, "v")) for layer in range(LAYERS)], 1)
        self.q = torch.stack([synth.heavy_tailed((n_inputs, 1, HQ, D), dev, seed, layer, "q")
                              for layer in range(LAYERS)], 1)
        self.slot = torch.tensor([context], dtype=torch.int32, device=dev)
        self.seq = torch.tensor([self.T], dtype=torch.int32, device=dev)
        self.bt = torch.arange(self.n_pages, dtype=torch.int32, device=dev).reshape(1, -1)
        self.qrot = torch.empty((1, HQ, D), dtype=torch.float32, device=dev)
        self.out = torch.empty((LAYERS, 1, HQ, D), dtype=torch.float32, device=dev)
        self.ws = K.alloc_workspace(self.caches[0], 1, HQ, self.T, device=dev)
        self.sm_scale = 1.0 / math.sqrt(D)
        torch.cuda.synchronize()

    def decode_only(self):
        """The 16 layers' decode launches alone (for the per-launch timing)."""
        for layer in range(LAYERS):
            self.K.decode_attn(self.caches[layer], self.qrot, self.seq, self.bt, self.T, self.sm_scale, self.ws)

    def step(self, i, ev=None, new_k=None, new_v=None, q=None, out=None):
        """One token through the 16 layers; ev = list of (start, end) events per decode."""
        K = self.K
        new_k = self.new_k[i] if new_k is None else new_k
        new_v = self.new_v[i] if new_v is None else new_v
        q = self.q[i] if q is None else q
        out = self.out if out is None else out
        for layer in range(LAYERS):
            c = self.caches[layer]
            # store the new token + rotate the query (one launch), decode, merge
            K.store_rotate(c, new_k[layer], new_v[layer], self.slot, q[layer], out=self.qrot)
            if ev is not None:
                ev[layer][0].record()
            K.decode_attn(c, self.qrot, self.seq, self.bt, self.T, self.sm_scale, self.ws)
            if ev is not None:
                ev[layer][1].record()
            K.merge(c, self.ws, 1, HQ, self.seq, self.T, out[layer])
        return KERNELS_PER_LAYER * LAYERS   # kernels launched


def capture(torch, fn):
    """Capture fn() (launches on the current stream) into a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    torch.cuda.synchronize()
    return g


def time_device(W, steps, warmup, torch, clk=None):
    """Device time of `steps` steps (one graph replay each) and the average
    duration of one decode launch (a graph of the 16 layers' decode launches,
    timed with CUDA events on the replay stream).  `clk` samples the clocks
    from the first timed replay until the device has finished them."""
    n_in = W.new_k.shape[0]
    graphs = [capture(torch, lambda i=i: W.step(i)) for i in range(n_in)]
    dec_graph = capture(torch, W.decode_only)
    for i in range(warmup):
        graphs[i % n_in].replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk:
        clk.begin()
    t0.record()
    for s in range(steps):
        graphs[s % n_in].replay()
    t1.record()
    torch.cuda.synchronize()
    if clk:
        clk.end()
    total_ms = t0.elapsed_time(t1)
    for _ in range(2):
        dec_graph.replay()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record()
    for s in range(steps):
        dec_graph.replay()
    d1.record()
    torch.cuda.synchronize()
    dec_avg_ms = d0.elapsed_time(d1) / (steps * LAYERS)
    return total_ms, dec_avg_ms, KERNELS_PER_LAYER * LAYERS * steps, graphs


def time_e2e(W, steps, warmup, torch, graphs):
    """Host buffers in, host buffers out, copies inside the timed region: the
    step's new K/V rows and queries are copied from pinned host memory into the
    device buffers the captured step reads, the step graph runs, and the 16
    layers' outputs are copied back."""
    n_in = W.new_k.shape[0]
    hk = [W.new_k[i].cpu().pin_memory() for i in range(n_in)]
    hv = [W.new_v[i].cpu().pin_memory() for i in range(n_in)]
    hq = [W.q[i].cpu().pin_memory() for i in range(n_in)]
    hout = torch.empty(W.out.shape, dtype=torch.float32).pin_memory()

    def one(i):
        W.new_k[i].copy_(hk[i], non_blocking=True)
        W.new_v[i].copy_(hv[i], non_blocking=True)
        W.q[i].copy_(hq[i], non_blocking=True)
        graphs[i].replay()
        hout.copy_(W.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for i in range(warmup):
        one(i % n_in)
    torch.cuda.synchronize()
    t = time.perf_counter()
    for s in range(steps):
        one(s % n_in)
    el = time.perf_counter() - t
    h2d = sum(x.numel() * x.element_size() for x in (hk[0], hv[0], hq[0]))
    d2h = hout.numel() * hout.element_size()
    return el * 1e3, h2d, d2h


def cpu_baseline_decode(context, n_heads, seed=99):
    """Time the CPU oracle on one layer-token at `context` (store the new token and
    attend with n_heads of the 24 query heads); returns (us per layer-token, desc)."""
    import numpy as np
    import torch

    import oracle as O
    from bit_quantized_kv_store_gb300 import synth
    T = context + 1
    n_pages = (T + PS - 1) // PS
    c = O.Cache(O.Q4, HK, D, PS, n_pages)
    # fill the cache (not timed): the oracle's own store of the same kind of data
    kv_heads = sorted({h // (HQ // HK) for h in range(n_heads)})
    k = synth.heavy_tailed((T, HK, D), "cpu", seed, "k").view(torch.int16).numpy().view(np.uint16)
    v = synth.heavy_tailed((T, HK, D), "cpu", seed, "v").view(torch.int16).numpy().view(np.uint16)
    O.store(c, k[:context], v[:context], np.arange(context, dtype=np.int32))
    q = synth.heavy_tailed((1, HQ, D), "cpu", seed, "q").view(torch.int16).numpy().view(np.uint16)
    bt = np.arange(n_pages, dtype=np.int32).reshape(1, -1)
    t = time.perf_counter()
    O.store(c, k[context:], v[context:], np.array([context], np.int32))
    O.decode(c, q[:, :n_heads], [T], bt, 1 / 16)
    el = time.perf_counter() - t
    us = el * 1e6 * (HQ / n_heads)
    return us, f"one layer-token at context {context}: store of the new token + {n_heads} of {HQ} query heads " \
               f"(KV heads {kv_heads}), scaled to 24 heads; oracle is single-threaded"


METRIC = "decode attn us/layer-token and achieved HBM GB/s vs peak (4-bit KV)"


def workload_config(context, world):
    return {"workload": f"single-sequence decode, context {context} (T={context + 1}), 16 layers, 4 KV / 24 q heads, "
                        f"head_dim 256, bf16 inputs, 5% Student-t(3)x10 channels",
            "l2": "16 layer caches exceed L2 (no flush needed)", "parallelism": f"replicas x{world}"}


def run_reference(args):
    """--impl reference: the CPU oracle on the host cores, same metric and config;
    each of the W warm-up and K timed steps is one bounded sample (one layer-token,
    6 of the 24 query heads, scaled to 24)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for s in range(args.warmup):
        cpu_baseline_decode(args.context, 6, seed=900 + s)
    samples = []
    for s in range(args.steps):
        us, desc = cpu_baseline_decode(args.context, 6, seed=1000 + s)
        samples.append(us)
    us = statistics.mean(samples)
    line = {"impl": "reference", "metric": METRIC, "value": us,
            "unit": "us/layer-token", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us * LAYERS / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.context, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": us, "unit": "us/layer-token", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": us, "unit": "us/layer-token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# --------------------------------------------------------------------------- the other hot-path rows

def _events_time(torch, fn, iters, warmup=3):
    """Average device time (ms) of fn() over iters runs, CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def measure_rows(K, synth, torch, dev, peak, tflops_peak, only=None):
    """Batched ragged paged decode, prefill chunk, fp8 latent decode (dense and
    gathered), the bf16-cache comparison and the store, each timed with CUDA
    events (inputs resident in HBM).  `only` restricts to one row."""
    out = {}
    seed = 1234 + 3
    want = lambda name: only is None or only == name
    # ---- batched ragged paged decode: 32 sequences, lengths ~ U{1024..65536}, 16-token pages, shuffled tables
    if want("batched"):
        out.update(_row_batched(K, synth, torch, dev, peak, seed))
    if want("prefill"):
        out.update(_row_prefill(K, synth, torch, dev, tflops_peak, seed))
    if want("fp8"):
        out.update(_row_fp8(K, synth, torch, dev, seed))
    if want("bf16"):
        out.update(_row_bf16(K, synth, torch, dev, seed))
    if want("q4_0"):
        out.update(_row_q4_0(K, synth, torch, dev, peak, seed))
    if want("window"):
        out.update(_row_window(K, synth, torch, dev, peak, seed))
    if want("tq4"):
        out.update(_row_tq4(K, synth, torch, dev, peak, seed))
    if want("fp8_prefill"):
        out.update(_row_fp8_prefill(K, synth, torch, dev, seed))
    if want("fused_merge"):
        out.update(_row_fused_merge(K, synth, torch, dev, seed))
    return out


def _row_batched(K, synth, torch, dev, peak, seed):
    out = {}
    lens = synth.ragged_lengths(32, 1024, 65536, seed, "lens").tolist()
    T = [L + 1 for L in lens]
    pages = [(t + PS - 1) // PS for t in T]
    n_pages = sum(pages)
    perm = synth.page_permutation(n_pages, seed, "perm")
    bt = torch.zeros((32, max(pages)), dtype=torch.int32)
    off = 0
    for i, npg in enumerate(pages):
        bt[i, :npg] = perm[off:off + npg]
        off += npg
    bt = bt.to(dev)
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, n_pages, device=dev)
    for i, L in enumerate(lens):
        k = synth.heavy_tailed((L, HK, D), dev, seed, i, "k", subset=(seed, "k"))
        v = synth.heavy_tailed((L, HK, D), dev, seed, i, "v", subset=(seed, "v"))
        pos = torch.arange(L, device=dev)
        slots = (bt[i][pos // PS] * PS + pos % PS).to(torch.int32)
        K.store(c, k, v, slots)
    new_k = synth.heavy_tailed((32, HK, D), dev, seed, "nk", subset=(seed, "k"))
    new_v = synth.heavy_tailed((32, HK, D), dev, seed, "nv", subset=(seed, "v"))
    q = synth.heavy_tailed((32, HQ, D), dev, seed, "q")
    new_slots = torch.tensor([int(bt[i][lens[i] // PS]) * PS + lens[i] % PS for i in range(32)], dtype=torch.int32,
                             device=dev)
    seq = torch.tensor(T, dtype=torch.int32, device=dev)
    qrot = torch.empty((32, HQ, D), dtype=torch.float32, device=dev)
    o = torch.empty((32, HQ, D), dtype=torch.float32, device=dev)
    ws = K.alloc_workspace(c, 32, HQ, max(T), device=dev)

    def batched_step():
        K.store_rotate(c, new_k, new_v, new_slots, q, out=qrot)  # 32 x 4 x (K, V) = 256 rows: the fused form
        K.decode_attn(c, qrot, seq, bt, max(T), 1 / 16, ws)
        K.merge(c, ws, 32, HQ, seq, max(T), o)

    ms = _events_time(torch, batched_step, 10)
    dec_ms = _events_time(torch, lambda: K.decode_attn(c, qrot, seq, bt, max(T), 1 / 16, ws), 10)
    byts = sum(T) * BYTES_PER_POS_LAYER
    out["batched_paged_decode"] = {
        "workload": "32 sequences, lengths U{1024..65536} (+1 new token each), 16-token pages, shuffled block "
                    "tables, 1 layer, 4 KV / 24 q heads", "us_per_step": ms * 1e3, "decode_kernel_us": dec_ms * 1e3,
        "cache_bytes": byts, "achieved_GBs": byts / (dec_ms * 1e-3) / 1e9, "frac_of_hbm_peak": byts / (dec_ms * 1e-3) / 1e9 / peak,
        "kernel": "decode_q4_round_kernel"}
    del c, ws
    torch.cuda.empty_cache()
    return out


def _row_prefill(K, synth, torch, dev, tflops_peak, seed):
    """Prefill chunk: 4096 queries at depth 16384, causal over decoded 4-bit slots;
    also the store of the chunk's rows."""
    out = {}
    depth, nq = 16384, 4096
    Tp = depth + nq
    npg = (Tp + PS - 1) // PS
    bt1 = synth.page_permutation(npg, seed, "pf").to(torch.int32).to(dev)
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, npg, device=dev)
    k = synth.heavy_tailed((Tp, HK, D), dev, seed, "pfk", subset=(seed, "k"))
    v = synth.heavy_tailed((Tp, HK, D), dev, seed, "pfv", subset=(seed, "v"))
    pos = torch.arange(Tp, device=dev)
    slots = (bt1[pos // PS] * PS + pos % PS).to(torch.int32)
    K.store(c, k[:depth], v[:depth], slots[:depth])
    qp = synth.heavy_tailed((nq, HQ, D), dev, seed, "pfq")
    op = torch.empty((nq, HQ, D), dtype=torch.float32, device=dev)
    kc, vc, sc = k[depth:].contiguous(), v[depth:].contiguous(), slots[depth:].contiguous()

    def prefill():
        K.store(c, kc, vc, sc)
        K.prefill_attn(c, qp, depth, bt1, 1 / 16, out=op)

    ms = _events_time(torch, prefill, 2, warmup=1)
    st_ms = _events_time(torch, lambda: K.store(c, kc, vc, sc), 10)
    flops = sum(depth + i + 1 for i in range(nq)) * HQ * 4 * D
    out["prefill_chunk"] = {"workload": "4096-token chunk at depth 16384 (store + causal attention over decoded "
                                        "4-bit slots), 4 KV / 24 q heads", "ms": ms, "flop": flops,
                            "TFLOPs": flops / (ms * 1e-3) / 1e12, "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 /
                            tflops_peak, "kernel": "prefill_tc_kernel (tcgen05, TMEM accumulators)"}
    rows = nq * HK * 2
    out["store"] = {"workload": "4096 tokens x 4 KV heads x (K, V) bf16 rows of 256 -> 4-bit rotated rows",
                    "us": st_ms * 1e3, "rows_per_s": rows / (st_ms * 1e-3),
                    "GBs": rows * (512 + 144) / (st_ms * 1e-3) / 1e9}
    del c, k, v
    torch.cuda.empty_cache()
    return out


def _row_fp8(K, synth, torch, dev, seed):
    """fp8 latent rows: dense absorbed decode over 262144 rows, 128 heads, and a 2048-row gather."""
    out = {}
    Tf, Hf, DL, R = 262144, 128, 512, 64
    npg = Tf // PS
    c = K.Cache(K.FMT_FP8_ROW, 1, DL, PS, npg, device=dev, rope_dim=R)
    for s0 in range(0, Tf, 65536):
        rows_ = synth.latent_rows(65536, DL + R, dev, seed, "fp8", s0)
        K.store(c, rows_, None, torch.arange(s0, s0 + 65536, dtype=torch.int32, device=dev))
    qf = synth.normal((1, Hf, DL + R), dev, seed, "fp8q")
    btf = torch.arange(npg, dtype=torch.int32, device=dev).reshape(1, -1)
    seqf = torch.tensor([Tf], dtype=torch.int32, device=dev)
    of = torch.empty((1, Hf, DL), dtype=torch.float32, device=dev)
    wsf = K.alloc_workspace(c, 1, Hf, Tf, device=dev)
    smf = 1 / math.sqrt(DL + R)

    def fp8_dense():
        K.decode_attn(c, qf, seqf, btf, Tf, smf, wsf)
        K.merge(c, wsf, 1, Hf, seqf, Tf, of)

    ms = _events_time(torch, fp8_dense, 3, warmup=1)
    flops = Hf * Tf * 2 * (DL + R + DL)
    byts = Tf * (DL + R + 8)
    sel = synth.distinct_sorted(2048, Tf, seed, "sel").to(torch.int32).to(dev).reshape(1, -1)
    wsg = K.alloc_workspace(c, 1, Hf, Tf, n_sel=2048, device=dev)

    def fp8_gather():
        K.decode_attn(c, qf, seqf, btf, Tf, smf, wsg, sel=sel)
        K.merge(c, wsg, 1, Hf, seqf, Tf, of, n_sel=2048)

    gms = _events_time(torch, fp8_gather, 5)
    out["fp8_latent"] = {"workload": "absorbed decode, 128 heads x (512 latent + 64 rope) e4m3 rows, context 262144, "
                                     "split-T + merge", "us": ms * 1e3, "flop": flops, "TFLOPs": flops / (ms * 1e-3) / 1e12,
                         "GBs": byts / (ms * 1e-3) / 1e9, "gather_2048_us": gms * 1e3,
                         "kernel": "decode_fp8_kernel (mma.sync f16, split query) + merge_kernel"}
    del c, wsf, wsg
    torch.cuda.empty_cache()
    return out


def _row_fp8_prefill(K, synth, torch, dev, seed):
    """fp8 latent prefill past the old caps: a 32-row chunk at positions 1048544 ..
    1048575 (1M keys), 128 heads, causal; one streaming CTA per (row, 32 heads)."""
    out = {}
    n_q, Hf, DL, R = 32, 128, 512, 64
    T = 1 << 20
    npg = T // PS
    c = K.Cache(K.FMT_FP8_ROW, 1, DL, PS, npg, device=dev, rope_dim=R)
    for s0 in range(0, T, 65536):
        rows_ = synth.latent_rows(65536, DL + R, dev, seed, "fp8pf", s0)
        K.store(c, rows_, None, torch.arange(s0, s0 + 65536, dtype=torch.int32, device=dev))
    q = synth.normal((n_q, Hf, DL + R), dev, seed, "fp8pfq")
    bt = torch.arange(npg, dtype=torch.int32, device=dev)
    sm = 1 / math.sqrt(DL + R)
    ws = torch.zeros(K.lib().kvq_prefill_fp8_workspace_size(c.ref, n_q, Hf), dtype=torch.uint8, device=dev)
    o = torch.empty((n_q, Hf, DL), dtype=torch.float32, device=dev)
    depth = T - n_q
    ms = _events_time(torch, lambda: K.prefill_attn_fp8(c, q, depth, bt, sm, workspace=ws, out=o), 3, warmup=1)
    keys = sum(depth + i + 1 for i in range(n_q))
    flops = keys * Hf * 2 * (DL + R + DL)
    out["fp8_prefill_1m"] = {"workload": "fp8 latent prefill chunk of 32 rows at positions 1048544..1048575, 128 heads, "
                                         "causal over (512 + 64) e4m3 rows",
                             "ms": ms, "flop": flops, "TFLOPs": flops / (ms * 1e-3) / 1e12,
                             "kernel": "decode_fp8_kernel (streaming: one CTA per row x 32 heads, the row one "
                                       "partition) + merge_kernel"}
    del c, ws
    torch.cuda.empty_cache()
    return out


def _row_bf16(K, synth, torch, dev, seed):
    """bf16-cache comparison at 32K (same kernel structure, unrotated bf16 rows)."""
    out = {}
    Tb = 32769
    npg = (Tb + PS - 1) // PS
    c = K.Cache(K.FMT_BF16, HK, D, PS, npg, device=dev)
    k = synth.heavy_tailed((Tb, HK, D), dev, seed, "bk", subset=(seed, "k"))
    v = synth.heavy_tailed((Tb, HK, D), dev, seed, "bv", subset=(seed, "v"))
    K.store(c, k, v, torch.arange(Tb, dtype=torch.int32, device=dev))
    qb = synth.heavy_tailed((1, HQ, D), dev, seed, "bq").float()
    btb = torch.arange(npg, dtype=torch.int32, device=dev).reshape(1, -1)
    seqb = torch.tensor([Tb], dtype=torch.int32, device=dev)
    ob = torch.empty((1, HQ, D), dtype=torch.float32, device=dev)
    wsb = K.alloc_workspace(c, 1, HQ, Tb, device=dev)
    dms = _events_time(torch, lambda: K.decode_attn(c, qb, seqb, btb, Tb, 1 / 16, wsb), 10)
    byts = Tb * HK * 2 * D * 2
    out["bf16_cache_32k"] = {"workload": "bf16 (unrotated) cache, context 32768, 1 layer, same split-T + merge",
                             "decode_kernel_us": dms * 1e3, "cache_bytes": byts, "achieved_GBs": byts / (dms * 1e-3) / 1e9,
                             "bytes_vs_4bit": byts / (Tb * BYTES_PER_POS_LAYER),
                             "kernel": "decode_bf16_kernel (mma.sync bf16, split query and P)"}
    del c, wsb
    torch.cuda.empty_cache()
    return out


def _row_q4_0(K, synth, torch, dev, peak, seed):
    """The unrotated 4-bit format at 32K: the store of 4096 tokens (no rotation) and
    the decode kernel (the same kernel as the rotated format)."""
    out = {}
    Tq = 32769
    npg = (Tq + PS - 1) // PS
    c = K.Cache(K.FMT_Q4_0, HK, D, PS, npg, device=dev)
    k = synth.heavy_tailed((Tq, HK, D), dev, seed, "q0k", subset=(seed, "k"))
    v = synth.heavy_tailed((Tq, HK, D), dev, seed, "q0v", subset=(seed, "v"))
    K.store(c, k, v, torch.arange(Tq, dtype=torch.int32, device=dev))
    sk, sv = k[:4096].contiguous(), v[:4096].contiguous()
    slots = torch.arange(4096, dtype=torch.int32, device=dev)
    st_ms = _events_time(torch, lambda: K.store(c, sk, sv, slots), 10)
    q = synth.heavy_tailed((1, HQ, D), dev, seed, "q0q").float()
    bt = torch.arange(npg, dtype=torch.int32, device=dev).reshape(1, -1)
    seq = torch.tensor([Tq], dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, 1, HQ, Tq, device=dev)
    dms = _events_time(torch, lambda: K.decode_attn(c, q, seq, bt, Tq, 1 / 16, ws), 10)
    byts = Tq * BYTES_PER_POS_LAYER
    out["q4_0_cache_32k"] = {"workload": "unrotated 4-bit cache (Q4_0), context 32768, 1 layer, same split-T + merge",
                             "decode_kernel_us": dms * 1e3, "cache_bytes": byts,
                             "achieved_GBs": byts / (dms * 1e-3) / 1e9, "frac_of_hbm_peak": byts / (dms * 1e-3) / 1e9 / peak,
                             "store_4096_tokens_us": st_ms * 1e3, "kernel": "decode_q4_round_kernel"}
    del c, ws
    torch.cuda.empty_cache()
    return out


def _row_tq4(K, synth, torch, dev, peak, seed):
    """TQ4 rows (randomized Hadamard + 16-level Lloyd-Max codebook, one fp16 scale
    per row: 130 bytes per row) at 262K: the split-T decode kernel, the full step
    (query rotation, decode, merge, inverse rotation) and a 4096-token store."""
    out = {}
    Tq = 262145
    npg = (Tq + PS - 1) // PS
    c = K.Cache(K.FMT_TQ4, HK, D, PS, npg, device=dev, signs=synth.sign_mask(D, seed, "tq4"))
    for s0 in range(0, Tq, 65536):
        n = min(65536, Tq - s0)
        k = synth.heavy_tailed((n, HK, D), dev, seed, "tqk", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), dev, seed, "tqv", s0, subset=(seed, "v"))
        K.store(c, k, v, torch.arange(s0, s0 + n, dtype=torch.int32, device=dev))
    sk = synth.heavy_tailed((4096, HK, D), dev, seed, "tqsk")
    sv = synth.heavy_tailed((4096, HK, D), dev, seed, "tqsv")
    slots = torch.arange(4096, dtype=torch.int32, device=dev)
    st_ms = _events_time(torch, lambda: K.store(c, sk, sv, slots), 10)
    q = synth.heavy_tailed((1, HQ, D), dev, seed, "tqq")
    qr = K.tq4_rotate(c, q)
    bt = torch.arange(npg, dtype=torch.int32, device=dev).reshape(1, -1)
    seq = torch.tensor([Tq], dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, 1, HQ, Tq, device=dev)
    o = torch.empty((1, HQ, D), dtype=torch.float32, device=dev)
    dms = _events_time(torch, lambda: K.decode_attn(c, qr, seq, bt, Tq, 1 / 16, ws), 10)
    step_ms = _events_time(torch, lambda: K.decode(c, q, seq, bt, Tq, 1 / 16, ws, out=o), 10)
    byts = Tq * HK * 2 * (D // 2 + 2)
    out["tq4_cache_262k"] = {"workload": "TQ4 rows (rotated int4 + Lloyd-Max codebook, 130 B/row), context 262144, "
                                         "1 layer, 4 KV / 24 q heads",
                             "decode_kernel_us": dms * 1e3, "cache_bytes": byts,
                             "achieved_GBs": byts / (dms * 1e-3) / 1e9,
                             "frac_of_hbm_peak": byts / (dms * 1e-3) / 1e9 / peak,
                             "step_us": step_ms * 1e3, "store_4096_tokens_us": st_ms * 1e3,
                             "kernel": "decode_q4_round_kernel<TQ4> (prmt level tables, movmatrix for V)"}
    del c, ws
    torch.cuda.empty_cache()
    return out


def _row_fused_merge(K, synth, torch, dev, seed):
    """Decode + merge as two launches against one launch whose last CTA per
    (sequence, KV head) merges (kvq_decode_merged), at 32769 and 262145 keys of
    one sequence, one layer."""
    out = {}
    T = 262145
    npg = (T + PS - 1) // PS
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, npg, device=dev)
    for s0 in range(0, T, 65536):
        n = min(65536, T - s0)
        k = synth.heavy_tailed((n, HK, D), dev, seed, "fmk", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), dev, seed, "fmv", s0, subset=(seed, "v"))
        K.store(c, k, v, torch.arange(s0, s0 + n, dtype=torch.int32, device=dev))
    q = K.rotate_query(synth.heavy_tailed((1, HQ, D), dev, seed, "fmq"))
    bt = torch.arange(npg, dtype=torch.int32, device=dev).reshape(1, -1)
    o = torch.empty((1, HQ, D), dtype=torch.float32, device=dev)
    for Tq in (32769, 262145):
        seq = torch.tensor([Tq], dtype=torch.int32, device=dev)
        ws = K.alloc_workspace(c, 1, HQ, Tq, device=dev)

        def two():
            K.decode_attn(c, q, seq, bt, Tq, 1 / 16, ws)
            K.merge(c, ws, 1, HQ, seq, Tq, o)

        two_ms = _events_time(torch, two, 20)
        one_ms = _events_time(torch, lambda: K.decode_merged(c, q, seq, bt, Tq, 1 / 16, ws, out=o), 20)
        out[f"fused_merge_{Tq - 1}"] = {"workload": f"one sequence, {Tq} keys, 1 layer",
                                         "decode_then_merge_us": two_ms * 1e3, "decode_merged_us": one_ms * 1e3,
                                         "kernel": "decode_q4_round_kernel with the last-CTA merge"}
    del c
    torch.cuda.empty_cache()
    return out


def _row_window(K, synth, torch, dev, peak, seed):
    """Decode window (speculative verify): 4 draft rows of one sequence at context
    262144 sharing its block table; the window call against the same rows decoded
    as 4 independent sequences (block table repeated, sequence-major order) and
    against one row."""
    out = {}
    R, T0 = 4, 262144
    T = T0 + R
    npg = (T + PS - 1) // PS
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, npg, device=dev)
    for s0 in range(0, T, 65536):
        n = min(65536, T - s0)
        k = synth.heavy_tailed((n, HK, D), dev, seed, "wk", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), dev, seed, "wv", s0, subset=(seed, "v"))
        K.store(c, k, v, torch.arange(s0, s0 + n, dtype=torch.int32, device=dev))
    q = K.rotate_query(synth.heavy_tailed((R, HQ, D), dev, seed, "wq"))
    bt = torch.arange(npg, dtype=torch.int32, device=dev)
    lens = torch.arange(T0 + 1, T + 1, dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, R, HQ, T, device=dev)
    win_ms = _events_time(torch, lambda: K.decode_window(c, q, lens, bt, T, 1 / 16, ws), 10)
    bt_rep = bt.reshape(1, -1).repeat(R, 1).contiguous()
    rows_ms = _events_time(torch, lambda: K.decode_attn(c, q, lens, bt_rep, T, 1 / 16, ws), 10)
    one_ms = _events_time(torch, lambda: K.decode_attn(c, q[:1], lens[:1], bt_rep[:1], T, 1 / 16, ws), 10)
    byts = T0 * BYTES_PER_POS_LAYER
    out["decode_window_262k"] = {
        "workload": "4 draft rows at positions 262144..262147 of one sequence, shared block table, 1 layer",
        "window_us": win_ms * 1e3, "as_4_sequences_us": rows_ms * 1e3, "one_row_us": one_ms * 1e3,
        "window_us_per_row": win_ms * 1e3 / R, "cache_GBs_once": byts / (win_ms * 1e-3) / 1e9,
        "kernel": "decode_q4_round_kernel, window mode: the 4 rows' 24 (row, head) columns in one CTA"}
    del c, ws
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    from bit_quantized_kv_store_gb300 import _lib as K
    from bit_quantized_kv_store_gb300 import build, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    K.lib()
    peak, peak_kind = load_peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max_over_ranks(x, world, dev)

    if args.only:
        tf_peak = 1922.8
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                tf_peak = json.load(f).get("bf16_tflops", tf_peak)
        except OSError:
            pass
        if rank == 0:
            print(json.dumps(measure_rows(K, synth, torch, dev, peak, tf_peak, only=args.only)))
        return

    n_inputs = 4
    W = Workload(K, synth, torch, args.context, n_inputs, 1234 + 1 + rank, dev)
    barrier()
    with Clocks(local) as clk:
        total_ms, dec_avg_ms, launches, graphs = time_device(W, args.steps, args.warmup, torch, clk)
    barrier()
    total_ms = max_over_ranks(total_ms)
    us_per_lt = aggregate_us_per_unit(total_ms, LAYERS * args.steps, world)
    bytes_per_launch = W.T * BYTES_PER_POS_LAYER
    achieved = bytes_per_launch / (dec_avg_ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = time_e2e(W, max(3, args.steps // 2), 2, torch, graphs)
    del graphs
    e2e_ms = max_over_ranks(e2e_ms)
    e2e_us = e2e_ms * 1e3 / (LAYERS * max(3, args.steps // 2) * world)

    long = None
    if not args.no_long:
        del W
        torch.cuda.empty_cache()
        WL = Workload(K, synth, torch, args.long_context, 2, 1234 + 2 + rank, dev)
        lsteps = max(3, args.steps // 4)
        barrier()
        with Clocks(local) as clk2:
            ltot, lavg, _, lgraphs = time_device(WL, lsteps, max(3, args.warmup // 2), torch, clk2)
        del lgraphs
        ltot = max_over_ranks(ltot)
        lbytes = WL.T * BYTES_PER_POS_LAYER
        lach = lbytes / (lavg * 1e-3) / 1e9
        long = {"context": args.long_context, "value": ltot * 1e3 / (LAYERS * lsteps * world),
                "unit": "us/layer-token", "decode_kernel_us": lavg * 1e3,
                "roofline": {"bound": "hbm", "achieved": lach, "peak": peak, "unit": "GB/s", "frac": lach / peak,
                             "traffic": TRAFFIC_BYTES.get(args.long_context), "bytes_per_launch": lbytes,
                             "kernel": "decode_q4_round_kernel"},
                "clocks": clk2.summary()}
        del WL

    rows = None
    if not args.no_rows and rank == 0:
        tf_peak = 1922.8
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                tf_peak = json.load(f).get("bf16_tflops", tf_peak)
        except OSError:
            pass
        rows = measure_rows(K, synth, torch, dev, peak, tf_peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        us, desc = cpu_baseline_decode(args.context, HQ)
        cpu = {"value": us, "unit": "us/layer-token", "cores": 1, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": us_per_lt, "unit": "us/layer-token", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 codes + fp16 scales; f16 MMA, fp32 accumulate",
            "data": "synthetic",
            "config": workload_config(args.context, world),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": TRAFFIC_BYTES.get(args.context), "bytes_per_launch": bytes_per_launch,
                         "kernel": "decode_q4_round_kernel",
                         "decode_kernel_us": dec_avg_ms * 1e3, "peak_kind": peak_kind},
            "e2e": {"value": e2e_us, "unit": "us/layer-token", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "long_context": long,
            "rows": rows,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
