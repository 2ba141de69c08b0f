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
e2e     = the same step through the public API, call by call (32 C-ABI calls a
          step; 48 with --step separate), with the step's inputs copied from pinned host memory and the
          outputs copied back inside the timed region; graph_replay_value is the
          same with the step replayed as a captured CUDA graph.
roofline= the decode kernel: algorithmic bytes (codes + scales of K and V of every
          attended position, 1152 B per position per layer) / average launch time
          measured with CUDA events on the launching stream; peak = measured HBM
          copy bandwidth.
clocks  = SM clock and throttle reasons sampled through NVML every 0.5 ms inside
          the timed region (nvidia-smi every 100 ms where NVML cannot be loaded).
cpu_baseline = the CPU oracle (single-threaded) on bounded samples of every
          workload, in spawned processes side by side on the host cores.
The other rows (batched decode, prefill, store, fp8, bf16, TQ4, windows, ...)
are printed in full on a line of their own before the headline line; the
headline carries their timings and fractions under roofline.other_kernels and
the 262K figures under roofline.long_context.
--impl reference times the CPU oracle, one layer-token per step.
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
# Launches per layer of a step: the fused form (kvq_decode_step: store, rotation
# and split-T decode in one launch, then the merge) or the separate one
# (kvq_store_rotate, kvq_decode_attn, kvq_merge).
KERNELS_PER_LAYER = {"fused": 2, "separate": 3}
# DRAM bytes of one decode launch (dram__bytes_read.sum + dram__bytes_write.sum
# from an ncu capture at each context), valid only for the kernel sources whose
# SHA-256 (first 16 hex digits, over TRAFFIC_SOURCES in order) is recorded
# beside them: once those sources change, the bench reports no traffic until
# the capture is taken again.
TRAFFIC_SOURCES = ("bit_quantized_kv_store_gb300/csrc/decode_q4.cu", "bit_quantized_kv_store_gb300/csrc/common.cuh")
TRAFFIC_CAPTURE = {"sources_sha16": "0bbdc4eda11d7094",
                   "bytes": {32768: 37857024 + 0, 262144: 302254336 + 10246144}}
BYTES_PER_POS_LAYER = HK * 2 * (D // 2 + 2 * (D // 32))   # 1152


def sources_sha16(paths=TRAFFIC_SOURCES):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_bytes(context):
    """ncu DRAM bytes of one decode launch at `context`, or None when the capture
    predates the current kernel sources."""
    if sources_sha16() != TRAFFIC_CAPTURE["sources_sha16"]:
        return None
    return TRAFFIC_CAPTURE["bytes"].get(context)


def decode_kernel_name(torch, positions, sequences=1):
    """The decode kernel the library runs for `sequences` sequences of `positions`
    keys: the warp-specialised form when the grid (512-key partitions x KV heads x
    sequences) fits one wave of two CTAs per SM, else the round kernel."""
    ctas = -(-positions // 512) * HK * sequences
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return "decode_q4_spec_kernel" if ctas <= 2 * sms else "decode_q4_round_kernel"


def resolve_step(torch, form, positions):
    """The step form for `positions` keys: auto takes the single launch of
    kvq_decode_step while the decode grid fits one wave (there the warp-specialised
    kernel rotates the queries in its prologue at no cost), else the three
    launches, whose decode kernel runs alone (its events time it alone)."""
    if form != "auto":
        return form
    return "fused" if decode_kernel_name(torch, positions) == "decode_q4_spec_kernel" else "separate"


def _r(x, digits=4):
    """Round a float to `digits` significant digits for the compact summaries."""
    if x is None or not isinstance(x, float) or x == 0 or not math.isfinite(x):
        return x
    return round(x, max(0, digits - 1 - int(math.floor(math.log10(abs(x))))))


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
    ap.add_argument("--only", choices=["batched", "prefill", "fp8", "bf16", "q4_0", "window", "tq4", "fp8_prefill", "fused_merge",
                                       "decode_step"], default=None,
                    help="run only one of the other hot-path rows and print its measurement (for profiling)")
    ap.add_argument("--step", choices=["auto", "fused", "separate"], default="auto",
                    help="the step's launches per layer: fused (kvq_decode_step + kvq_merge), separate "
                         "(kvq_store_rotate + kvq_decode_attn + kvq_merge), or auto: fused while the decode grid "
                         "fits one wave of two CTAs per SM, else separate"),
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

    def __init__(self, K, synth, torch, context, n_inputs, seed, device, step_form="auto"):
        self.K, self.torch = K, torch
        self.step_form = resolve_step(torch, step_form, context + 1)
        self.kernels_per_layer = KERNELS_PER_LAYER[self.step_form]
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
        # per (input set, layer): the new token's K/V rows and the queries, one
        # input set in one contiguous buffer (a step's inputs are one copy)
        nk, nq = LAYERS * HK * D, LAYERS * HQ * D
        self.inbuf = torch.empty((n_inputs, 2 * nk + nq), dtype=torch.bfloat16, device=dev)
        self.new_k = self.inbuf[:, :nk].view(n_inputs, LAYERS, 1, HK, D)
        self.new_v = self.inbuf[:, nk:2 * nk].view(n_inputs, LAYERS, 1, HK, D)
        self.q = self.inbuf[:, 2 * nk:].view(n_inputs, LAYERS, 1, HQ, D)
        self.new_k.copy_(torch.stack([synth.heavy_tailed((n_inputs, 1, HK, D), dev, seed, layer, "newk",
                                                         subset=(seed, layer, "k")) for layer in range(LAYERS)], 1))
        self.new_v.copy_(torch.stack([synth.heavy_tailed((n_inputs, 1, HK, D), dev, seed, layer, "newv",
                                                         subset=(seed, layer, "v")) for layer in range(LAYERS)], 1))
        self.q.copy_(torch.stack([synth.heavy_tailed((n_inputs, 1, HQ, D), dev, seed, layer, "q")
                                  for layer in range(LAYERS)], 1))
        self.slot = torch.tensor([context], dtype=torch.int32, device=dev)
        self.seq = torch.tensor([self.T], dtype=torch.int32, device=dev)
        self.bt = torch.arange(self.n_pages, dtype=torch.int32, device=dev).reshape(1, -1)
        self.qrot = torch.empty((1, HQ, D), dtype=torch.float32, device=dev)
        self.out = torch.empty((LAYERS, 1, HQ, D), dtype=torch.float32, device=dev)
        self.ws = K.alloc_workspace(self.caches[0], 1, HQ, self.T, device=dev)
        self.sm_scale = 1.0 / math.sqrt(D)
        # per (input set, layer): the views a step hands to the API, made once (a
        # serving loop keeps its per-layer buffers; slicing them again on every
        # call would add torch's view overhead to each call)
        self.views = [[(self.new_k[i][layer], self.new_v[i][layer], self.q[i][layer]) for layer in range(LAYERS)]
                      for i in range(n_inputs)]
        self.out_views = [self.out[layer] for layer in range(LAYERS)]
        torch.cuda.synchronize()

    def decode_only(self):
        """The 16 layers' decode launches alone (for the per-launch timing): the
        step's decode kernel (the fused launch, or kvq_decode_attn)."""
        for layer in range(LAYERS):
            if self.step_form == "fused":
                new_k, new_v, q = self.views[0][layer]
                self.K.decode_step(self.caches[layer], new_k, new_v, q, self.seq, self.bt, self.T, self.sm_scale,
                                   self.ws)
            else:
                self.K.decode_attn(self.caches[layer], self.qrot, self.seq, self.bt, self.T, self.sm_scale, self.ws)

    def step(self, i, ev=None):
        """One token through the 16 layers (input set i); ev = list of (start, end)
        events per decode."""
        K = self.K
        views, outs = self.views[i], self.out_views
        for layer in range(LAYERS):
            c = self.caches[layer]
            new_k, new_v, q = views[layer]
            if self.step_form == "fused":
                # store the new token, rotate the query and decode (one launch), merge
                if ev is not None:
                    ev[layer][0].record()
                K.decode_step(c, new_k, new_v, q, self.seq, self.bt, self.T, self.sm_scale, self.ws)
            else:
                # store the new token + rotate the query (one launch), decode, merge
                K.store_rotate(c, new_k, new_v, self.slot, q, out=self.qrot)
                if ev is not None:
                    ev[layer][0].record()
                K.decode_attn(c, self.qrot, self.seq, self.bt, self.T, self.sm_scale, self.ws)
            if ev is not None:
                ev[layer][1].record()
            K.merge(c, self.ws, 1, HQ, self.seq, self.T, outs[layer])
        return self.kernels_per_layer * LAYERS   # kernels launched


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
    return total_ms, dec_avg_ms, W.kernels_per_layer * LAYERS * steps, graphs


def time_e2e(W, steps, warmup, torch, graphs=None):
    """Host buffers in, host buffers out, copies inside the timed region: every
    step copies its new K/V rows and queries (one pinned host buffer) into the
    device buffer the step reads, runs the 16 layers, and copies the 16 layers'
    outputs back.  graphs=None: the step is issued call by call through the
    public API (kvq_store_rotate, kvq_decode_attn, kvq_merge per layer: host-side
    validation, tensor-map encoding and launch on every call); otherwise the
    captured step graphs are replayed."""
    n_in = W.inbuf.shape[0]
    hin = [W.inbuf[i].cpu().pin_memory() for i in range(n_in)]  # a step's K/V rows and queries
    hout = torch.empty(W.out.shape, dtype=torch.float32).pin_memory()

    def one(i):
        W.inbuf[i].copy_(hin[i], non_blocking=True)
        if graphs is None:
            W.step(i)
        else:
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
    h2d = hin[0].numel() * hin[0].element_size()
    d2h = hout.numel() * hout.element_size()
    return el * 1e3, h2d, d2h


# --------------------------------------------------------------------------- the CPU oracle legs
#
# The oracle (single-threaded C, fp64 attention) timed on the host cores on
# bounded samples of each workload.  Every leg runs in a process of its own
# (started with `spawn`, after the GPU measurements) with one thread; the legs
# run side by side on separate cores.  Cache fills use the oracle's own store
# and are not timed; the timed part is what the GPU step does: store the new
# tokens and attend.

def _oracle_env():
    import numpy as np
    import torch
    torch.set_num_threads(1)
    import oracle as O
    from bit_quantized_kv_store_gb300 import synth
    return np, torch, O, synth


def _bits(t):
    import numpy as np
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class OracleLayerToken:
    """One 4-bit cache of `context` positions filled by the oracle's store; step()
    stores one new token (4 KV heads, K and V) at position `context` and attends
    all 24 query heads over T = context + 1 keys: one layer-token of the
    benchmark's step."""

    def __init__(self, context, seed):
        np, torch, O, synth = _oracle_env()
        self.np, self.O = np, O
        self.T = context + 1
        n_pages = (self.T + PS - 1) // PS
        self.c = O.Cache(O.Q4, HK, D, PS, n_pages)
        chunk = 32768
        for s0 in range(0, context, chunk):
            n = min(chunk, context - s0)
            k = _bits(synth.heavy_tailed((n, HK, D), "cpu", seed, "k", s0, subset=(seed, "k")))
            v = _bits(synth.heavy_tailed((n, HK, D), "cpu", seed, "v", s0, subset=(seed, "v")))
            O.store(self.c, k, v, np.arange(s0, s0 + n, dtype=np.int32))
        self.new_k = _bits(synth.heavy_tailed((1, HK, D), "cpu", seed, "newk", subset=(seed, "k")))
        self.new_v = _bits(synth.heavy_tailed((1, HK, D), "cpu", seed, "newv", subset=(seed, "v")))
        self.q = _bits(synth.heavy_tailed((1, HQ, D), "cpu", seed, "q"))
        self.slot = np.array([context], np.int32)
        self.bt = np.arange(n_pages, dtype=np.int32).reshape(1, -1)

    def step(self):
        t = time.perf_counter()
        self.O.store(self.c, self.new_k, self.new_v, self.slot)
        self.O.decode(self.c, self.q, [self.T], self.bt, 1 / math.sqrt(D))
        return time.perf_counter() - t


def cpu_leg_c1(context=32768, seed=1234 + 1):
    """32K context: all 16 layers of one step (16 layer-tokens on one filled cache)."""
    w = OracleLayerToken(context, seed)
    el = sum(w.step() for _ in range(LAYERS))
    return {"value": el * 1e6 / LAYERS, "unit": "us/layer-token", "seconds": el,
            "sample": f"all {LAYERS} layers of one step at context {context}, 24 heads (one oracle-filled cache "
                      f"reused per layer)"}


def cpu_leg_c2(context=262144, seed=1234 + 2):
    """262K context: one full layer-token; the 16-layer step is extrapolated."""
    w = OracleLayerToken(context, seed)
    el = w.step()
    return {"value": el * 1e6, "unit": "us/layer-token", "seconds": el,
            "extrapolated_step_s": el * LAYERS,
            "sample": f"one layer-token at context {context} (store + 24 heads); the {LAYERS}-layer step "
                      f"extrapolated x{LAYERS}"}


def cpu_leg_c3_decode(seed=1234 + 3):
    """The ragged paged batch: 32 sequences, one layer, the whole batch."""
    np, torch, O, synth = _oracle_env()
    lens = synth.ragged_lengths(32, 1024, 65536, seed, "lens").tolist()
    T = [L + 1 for L in lens]
    pages = [(t + PS - 1) // PS for t in T]
    perm = synth.page_permutation(sum(pages), seed, "perm").numpy().astype(np.int32)
    bt = np.zeros((32, max(pages)), np.int32)
    off = 0
    for i, npg in enumerate(pages):
        bt[i, :npg] = perm[off:off + npg]
        off += npg
    c = O.Cache(O.Q4, HK, D, PS, sum(pages))
    for i, L in enumerate(lens):
        pos = np.arange(L)
        k = _bits(synth.heavy_tailed((L, HK, D), "cpu", seed, i, "k", subset=(seed, "k")))
        v = _bits(synth.heavy_tailed((L, HK, D), "cpu", seed, i, "v", subset=(seed, "v")))
        O.store(c, k, v, (bt[i][pos // PS] * PS + pos % PS).astype(np.int32))
    nk = _bits(synth.heavy_tailed((32, HK, D), "cpu", seed, "nk", subset=(seed, "k")))
    nv = _bits(synth.heavy_tailed((32, HK, D), "cpu", seed, "nv", subset=(seed, "v")))
    q = _bits(synth.heavy_tailed((32, HQ, D), "cpu", seed, "q"))
    slots = np.array([bt[i][lens[i] // PS] * PS + lens[i] % PS for i in range(32)], np.int32)
    t = time.perf_counter()
    O.store(c, nk, nv, slots)
    O.decode(c, q, T, bt, 1 / math.sqrt(D))
    el = time.perf_counter() - t
    return {"value": el * 1e6, "unit": "us/step", "seconds": el, "keys": sum(T),
            "sample": "the whole batch: 32 sequences (lengths U{1024..65536}), store of the 32 new tokens + "
                      "24 heads each, 1 layer"}


def cpu_leg_c3_prefill(seed=1234 + 3, n_rows=64):
    """The 4096-token chunk at depth 16384: the chunk's store and 64 seeded query
    rows (the first, the last and 62 drawn at random); rows/s and the chunk's
    time extrapolated from them."""
    np, torch, O, synth = _oracle_env()
    depth, nq = 16384, 4096
    Tp = depth + nq
    npg = (Tp + PS - 1) // PS
    bt = synth.page_permutation(npg, seed, "pf").numpy().astype(np.int32)
    c = O.Cache(O.Q4, HK, D, PS, npg)
    pos = np.arange(Tp)
    slots = (bt[pos // PS] * PS + pos % PS).astype(np.int32)
    k = _bits(synth.heavy_tailed((Tp, HK, D), "cpu", seed, "pfk", subset=(seed, "k")))
    v = _bits(synth.heavy_tailed((Tp, HK, D), "cpu", seed, "pfv", subset=(seed, "v")))
    O.store(c, k[:depth], v[:depth], slots[:depth])
    q = _bits(synth.heavy_tailed((nq, HQ, D), "cpu", seed, "pfq"))
    rows = np.unique(np.concatenate([[0, nq - 1], synth.distinct_sorted(n_rows - 2, nq, seed, "pfrows").numpy()]))
    t = time.perf_counter()
    O.store(c, k[depth:], v[depth:], slots[depth:])
    t_store = time.perf_counter() - t
    O.prefill(c, q, depth, bt, 1 / math.sqrt(D), rows=rows.astype(np.int32))
    t_rows = time.perf_counter() - t - t_store
    per_row = t_rows / rows.size
    # rows attend 16385 .. 20480 keys; the sampled rows' mean key count scales the chunk
    keys_sampled = float(np.mean(depth + rows + 1))
    keys_chunk = depth + (nq + 1) / 2
    return {"value": rows.size / t_rows, "unit": "query rows/s", "seconds": t_store + t_rows,
            "rows": int(rows.size), "store_s": t_store,
            "extrapolated_chunk_s": t_store + per_row * nq * keys_chunk / keys_sampled,
            "sample": f"{rows.size} seeded rows of the 4096-token chunk at depth 16384 (first, last, random), "
                      f"24 heads, after the chunk's store; the chunk's time extrapolated by keys"}


def cpu_leg_c4(seed=1234 + 4):
    """fp8 latent rows at 262,144 tokens: the dense absorbed decode (128 heads,
    one full run) and the 2048-row gather."""
    np, torch, O, synth = _oracle_env()
    Tf, Hf, DL, R = 262144, 128, 512, 64
    npg = Tf // PS
    c = O.Cache(O.FP8, 1, DL, PS, npg, rope_dim=R)
    for s0 in range(0, Tf, 65536):
        rows = synth.latent_rows(65536, DL + R, "cpu", seed, "fp8", s0).numpy()
        O.store(c, rows, None, np.arange(s0, s0 + 65536, dtype=np.int32))
    q = synth.normal((1, Hf, DL + R), "cpu", seed, "fp8q").numpy()
    bt = np.arange(npg, dtype=np.int32).reshape(1, -1)
    sel = synth.distinct_sorted(2048, Tf, seed, "sel").numpy().astype(np.int32).reshape(1, -1)
    sm = 1 / math.sqrt(DL + R)
    t = time.perf_counter()
    O.decode(c, q, [Tf], bt, sm)
    dense = time.perf_counter() - t
    t = time.perf_counter()
    O.decode(c, q, [Tf], bt, sm, sel=sel)
    gather = time.perf_counter() - t
    return {"value": dense * 1e6, "unit": "us/decode", "seconds": dense + gather, "gather_2048_us": gather * 1e6,
            "sample": "one full dense absorbed decode, 128 heads x 262144 e4m3 rows (512 + 64), and one gather of "
                      "2048 selected rows"}


CPU_LEGS = {"c1_32k_16_layers": cpu_leg_c1, "c2_262k_one_layer": cpu_leg_c2, "c3_batch_decode": cpu_leg_c3_decode,
            "c3_prefill_64_rows": cpu_leg_c3_prefill, "c4_fp8_dense_and_gather": cpu_leg_c4}


def _run_leg(name):
    os.environ["OMP_NUM_THREADS"] = "1"
    return name, CPU_LEGS[name]()


def cpu_baselines(names=None):
    """Run the oracle legs side by side in spawned single-threaded processes;
    returns {name: result}."""
    import concurrent.futures as cf
    import multiprocessing as mp
    names = list(CPU_LEGS) if names is None else names
    workers = max(1, min(len(names), (os.cpu_count() or 1) - 1))
    out = {}
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        for name, res in ex.map(_run_leg, names):
            res["cores"] = 1
            out[name] = res
    return out, workers


METRIC = "decode attn us/layer-token and achieved HBM GB/s vs peak (4-bit KV)"


def workload_config(context, world, step_form="auto"):
    fused = "store + rotation + decode in one launch (kvq_decode_step), merge"
    separate = "store + rotation (kvq_store_rotate), decode (kvq_decode_attn), merge"
    launches = {"fused": fused, "separate": separate,
                "auto": f"{fused} while the decode grid fits one wave of two CTAs per SM, else {separate}"}[step_form]
    return {"workload": f"single-sequence decode, context {context} (T={context + 1}), 16 layers, 4 KV / 24 q heads, "
                        f"head_dim 256, bf16 inputs, 5% Student-t(3)x10 channels",
            "step": f"per layer: {launches}",
            "l2": "16 layer caches exceed L2 (no flush needed)", "parallelism": f"replicas x{world}"}


def run_reference(args):
    """--impl reference: the CPU oracle on one host core, same metric and config.
    Its step is one layer-token of the 32K workload (store the new token, attend
    the 24 query heads over 32,769 keys): the metric is per layer-token, so the
    line reports what was timed, with no extrapolation."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = OracleLayerToken(args.context, 1234 + 1)
    for _ in range(args.warmup):
        w.step()
    samples = [w.step() for _ in range(args.steps)]
    us = statistics.mean(samples) * 1e6
    desc = (f"one layer-token per step (1 of the {LAYERS} layers) at context {args.context}: store of the new token + "
            f"24 of 24 query heads; single-threaded oracle")
    line = {"impl": "reference", "metric": METRIC, "value": us,
            "unit": "us/layer-token", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1e3, "step": "one layer-token", "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.context, int(os.environ.get("WORLD_SIZE", "1")), args.step),
            "cpu_baseline": {"value": us, "unit": "us/layer-token", "cores": 1, "kind": "oracle", "sample": desc,
                             "host_cores": os.cpu_count()},
            "e2e": {"value": us, "unit": "us/layer-token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# --------------------------------------------------------------------------- the other hot-path rows

L2_BYTES = 129 * 2 ** 20
_flush_bufs = None


def _l2_flush(torch):
    """Write a buffer of twice the L2 size, then read another one of the same
    size: the next launch finds none of its inputs in L2, and L2 holds clean
    lines only (no write-back of the flush's own lines lands in the timed
    region)."""
    global _flush_bufs
    if _flush_bufs is None:
        _flush_bufs = [torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") for _ in range(2)]
    _flush_bufs[0].zero_()
    _flush_bufs[1].sum()


def _events_time(torch, fn, iters, warmup=3, flush=True):
    """Average device time (ms) of fn() over iters runs, CUDA events on the current
    stream around each run; with `flush`, L2 is flushed before every run
    (outside the events), so single-layer rows whose data would fit in L2 read
    it from HBM."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if not flush:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in ev:
        _l2_flush(torch)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / iters


def rows_summary(rows):
    """The rows' timings and roofline fractions only (floats, 4 significant digits)."""
    return {name: {k: _r(v) for k, v in row.items() if isinstance(v, float)} for name, row in rows.items()}


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
        out.update(_row_prefill(K, synth, torch, dev, tflops_peak, seed, peak))
    if want("fp8"):
        out.update(_row_fp8(K, synth, torch, dev, seed, tflops_peak))
    if want("bf16"):
        out.update(_row_bf16(K, synth, torch, dev, seed, peak))
    if want("q4_0"):
        out.update(_row_q4_0(K, synth, torch, dev, peak, seed))
    if want("window"):
        out.update(_row_window(K, synth, torch, dev, peak, seed))
    if want("tq4"):
        out.update(_row_tq4(K, synth, torch, dev, peak, seed))
    if want("fp8_prefill"):
        out.update(_row_fp8_prefill(K, synth, torch, dev, seed, tflops_peak))
    if want("fused_merge"):
        out.update(_row_fused_merge(K, synth, torch, dev, seed))
    if want("decode_step"):
        out.update(_row_decode_step(K, synth, torch, dev, seed, peak))
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


def _row_prefill(K, synth, torch, dev, tflops_peak, seed, peak):
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
    # as a prompt's layers store their chunks: 16 layers' stores (distinct inputs
    # and caches, 343 MB, over L2) captured in one graph and replayed, per launch
    spg = nq // PS
    lk = [synth.heavy_tailed((nq, HK, D), dev, seed, "pfsk", i) for i in range(LAYERS)]
    lv = [synth.heavy_tailed((nq, HK, D), dev, seed, "pfsv", i) for i in range(LAYERS)]
    lc = [K.Cache(K.FMT_Q4_HAD32, HK, D, PS, spg, device=dev) for _ in range(LAYERS)]
    lslots = torch.arange(nq, dtype=torch.int32, device=dev)
    g = capture(torch, lambda: [K.store(lc[i], lk[i], lv[i], lslots) for i in range(LAYERS)])
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    gst_ms = e0.elapsed_time(e1) / (reps * LAYERS)
    out["store"] = {"workload": "4096 tokens x 4 KV heads x (K, V) bf16 rows of 256 -> 4-bit rotated rows; one "
                                "launch with L2 flushed (us), and 16 layers' stores in one graph (graph_us_per_layer)",
                    "us": st_ms * 1e3, "rows_per_s": rows / (st_ms * 1e-3),
                    "GBs": rows * (512 + 144) / (st_ms * 1e-3) / 1e9,
                    "frac_of_hbm_peak": rows * (512 + 144) / (st_ms * 1e-3) / 1e9 / peak,
                    "graph_us_per_layer": gst_ms * 1e3,
                    "graph_frac_of_hbm_peak": rows * (512 + 144) / (gst_ms * 1e-3) / 1e9 / peak}
    del c, k, v, lk, lv, lc, g
    torch.cuda.empty_cache()
    return out


def _row_fp8(K, synth, torch, dev, seed, tflops_peak):
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

    gms = _events_time(torch, fp8_gather, 20)
    out["fp8_latent"] = {"workload": "absorbed decode, 128 heads x (512 latent + 64 rope) e4m3 rows, context 262144, "
                                     "split-T + merge", "us": ms * 1e3, "flop": flops, "TFLOPs": flops / (ms * 1e-3) / 1e12,
                         "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / tflops_peak,
                         "GBs": byts / (ms * 1e-3) / 1e9, "gather_2048_us": gms * 1e3,
                         "kernel": "decode_fp8_kernel (mma.sync f16, split query) + merge_kernel"}
    del c, wsf, wsg
    torch.cuda.empty_cache()
    return out


def _row_fp8_prefill(K, synth, torch, dev, seed, tflops_peak):
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
                             "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / tflops_peak,
                             "kernel": "decode_fp8_kernel (streaming: one CTA per row x 32 heads, the row one "
                                       "partition) + merge_kernel"}
    del c, ws
    torch.cuda.empty_cache()
    return out


def _row_bf16(K, synth, torch, dev, seed, peak):
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
                             "frac_of_hbm_peak": byts / (dms * 1e-3) / 1e9 / peak,
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
    # timed as the headline times its decode: 16 distinct layer caches (604 MB,
    # over L2), the 16 launches captured in one graph and replayed, per launch
    layers = [c]
    for _ in range(LAYERS - 1):
        cl = K.Cache(K.FMT_Q4_0, HK, D, PS, npg, device=dev)
        K.store(cl, k, v, torch.arange(Tq, dtype=torch.int32, device=dev))
        layers.append(cl)
    g = capture(torch, lambda: [K.decode_attn(cl, q, seq, bt, Tq, 1 / 16, ws) for cl in layers])
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    gms = e0.elapsed_time(e1) / (reps * LAYERS)
    byts = Tq * BYTES_PER_POS_LAYER
    out["q4_0_cache_32k"] = {"workload": "unrotated 4-bit cache (Q4_0), context 32768, same split-T + merge; the "
                                         "decode timed over 16 layer caches in one graph (as the headline), and as "
                                         "one launch with L2 flushed",
                             "decode_kernel_us": gms * 1e3, "cache_bytes": byts,
                             "achieved_GBs": byts / (gms * 1e-3) / 1e9, "frac_of_hbm_peak": byts / (gms * 1e-3) / 1e9 / peak,
                             "single_launch_us": dms * 1e3,
                             "store_4096_tokens_us": st_ms * 1e3, "kernel": decode_kernel_name(torch, Tq)}
    del c, ws, layers, g
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


def _row_decode_step(K, synth, torch, dev, seed, peak):
    """The 32K step with the new token stored and the query rotated inside the
    decode launch (kvq_decode_step + kvq_merge: two launches per layer) against
    the three-launch step (kvq_store_rotate + kvq_decode_attn + kvq_merge), both
    as graphs of 16 layers, plus the fused launch alone."""
    W = Workload(K, synth, torch, 32768, 1, seed, dev, "separate")

    def fused():
        for layer in range(LAYERS):
            nk, nv, q = W.views[0][layer]
            K.decode_step(W.caches[layer], nk, nv, q, W.seq, W.bt, W.T, W.sm_scale, W.ws)
            K.merge(W.caches[layer], W.ws, 1, HQ, W.seq, W.T, W.out_views[layer])

    def fused_only():
        for layer in range(LAYERS):
            nk, nv, q = W.views[0][layer]
            K.decode_step(W.caches[layer], nk, nv, q, W.seq, W.bt, W.T, W.sm_scale, W.ws)

    res = {}
    for name, fn in (("fused", fused), ("three", lambda: W.step(0)), ("kernel", fused_only)):
        g = capture(torch, fn)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(20):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        res[name] = a.elapsed_time(b) / (20 * LAYERS) * 1e3
    byts = W.T * BYTES_PER_POS_LAYER
    out = {"decode_step_32k": {
        "workload": "one sequence, 32768 + 1 keys, 16 layers: store + rotation + decode fused in one launch, then the "
                    "merge", "us_per_layer_token": res["fused"], "three_launch_us_per_layer_token": res["three"],
        "fused_kernel_us": res["kernel"], "fused_kernel_GBs": byts / (res["kernel"] * 1e-6) / 1e9,
        "fused_kernel_frac_of_hbm_peak": byts / (res["kernel"] * 1e-6) / 1e9 / peak,
        "kernel": decode_kernel_name(torch, W.T) + " with the new token stored by its partition's CTA and the query "
                                                   "rotated in the kernel"}}
    del W
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
    # the same cache, attended at 2048 selected positions of the first row (a
    # sparse-attention selection; 512-entry partitions, as the dense keys)
    sel = synth.distinct_sorted(2048, T0 + 1, seed, "q4sel").to(torch.int32).to(dev).reshape(1, -1)
    wsg = K.alloc_workspace(c, 1, HQ, T0 + 1, n_sel=2048, device=dev)
    og = torch.empty((1, HQ, D), dtype=torch.float32, device=dev)

    def gather():
        K.decode_attn(c, q[:1], lens[:1], bt_rep[:1], T0 + 1, 1 / 16, wsg, sel=sel)
        K.merge(c, wsg, 1, HQ, lens[:1], T0 + 1, og, n_sel=2048)

    g_ms = _events_time(torch, gather, 10)
    gd_ms = _events_time(torch, lambda: K.decode_attn(c, q[:1], lens[:1], bt_rep[:1], T0 + 1, 1 / 16, wsg, sel=sel), 10)
    out["q4_gather_262k"] = {
        "workload": "2048 selected positions of a 262145-key sequence (4-bit rotated cache), 4 KV / 24 q heads, "
                    "decode + merge", "gather_2048_us": g_ms * 1e3, "decode_us": gd_ms * 1e3,
        "kernel": "decode_q4_spec_kernel in gather mode (rows resolved once per CTA, copied by cp.async; "
                  "the round kernel for grids over one wave)"}
    del c, ws, wsg
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
    W = Workload(K, synth, torch, args.context, n_inputs, 1234 + 1 + rank, dev, args.step)
    barrier()
    with Clocks(local) as clk:
        total_ms, dec_avg_ms, launches, graphs = time_device(W, args.steps, args.warmup, torch, clk)
    barrier()
    total_ms = max_over_ranks(total_ms)
    us_per_lt = aggregate_us_per_unit(total_ms, LAYERS * args.steps, world)
    bytes_per_launch = W.T * BYTES_PER_POS_LAYER
    achieved = bytes_per_launch / (dec_avg_ms * 1e-3) / 1e9
    e2e_steps = max(3, args.steps // 2)
    calls_per_step = W.kernels_per_layer * LAYERS
    step_form = W.step_form
    g_ms, h2d, d2h = time_e2e(W, e2e_steps, 2, torch, graphs)
    del graphs
    c_ms, _, _ = time_e2e(W, e2e_steps, 2, torch, None)
    g_us = max_over_ranks(g_ms) * 1e3 / (LAYERS * e2e_steps * world)
    c_us = max_over_ranks(c_ms) * 1e3 / (LAYERS * e2e_steps * world)

    long = None
    if not args.no_long:
        del W
        torch.cuda.empty_cache()
        WL = Workload(K, synth, torch, args.long_context, 2, 1234 + 2 + rank, dev, args.step)
        lsteps = max(3, args.steps // 4)
        barrier()
        with Clocks(local) as clk2:
            ltot, lavg, _, lgraphs = time_device(WL, lsteps, max(3, args.warmup // 2), torch, clk2)
        del lgraphs
        ltot = max_over_ranks(ltot)
        lbytes = WL.T * BYTES_PER_POS_LAYER
        lach = lbytes / (lavg * 1e-3) / 1e9
        c2 = clk2.summary()
        long = {"context": args.long_context, "value": _r(ltot * 1e3 / (LAYERS * lsteps * world)),
                "unit": "us/layer-token", "steps": lsteps, "decode_kernel_us": _r(lavg * 1e3),
                "achieved": _r(lach), "peak": peak, "frac": _r(lach / peak, 3),
                "traffic": traffic_bytes(args.long_context), "bytes_per_launch": lbytes,
                "kernel": decode_kernel_name(torch, WL.T), "step": WL.step_form,
                "clocks": {"sm_mhz": c2["sm_mhz"], "sm_max_mhz": c2["sm_max_mhz"], "reasons": c2["reasons"],
                           "samples": c2["samples"]}}
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
        legs, workers = cpu_baselines()
        c1 = legs["c1_32k_16_layers"]
        cpu = {"value": c1["value"], "unit": c1["unit"], "cores": 1, "kind": "oracle", "sample": c1["sample"],
               "host_cores": os.cpu_count(), "legs_side_by_side": workers,
               "configs": {k: {kk: (_r(vv) if isinstance(vv, float) else vv) for kk, vv in v.items()
                               if kk != "sample"} for k, v in legs.items()},
               "samples": {k: v["sample"] for k, v in legs.items()}}

    if rank == 0:
        if rows is not None:
            # the other rows in full, on a line of their own ahead of the headline
            print(json.dumps({"rows": rows}))
        line = {
            "metric": METRIC,
            "value": us_per_lt, "unit": "us/layer-token", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 codes + fp16 scales; f16 MMA, fp32 accumulate",
            "data": "synthetic",
            "config": workload_config(args.context, world, args.step),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic_bytes(args.context), "bytes_per_launch": bytes_per_launch,
                         "kernel": decode_kernel_name(torch, args.context + 1), "step": step_form,
                         "decode_kernel_us": dec_avg_ms * 1e3, "peak_kind": peak_kind,
                         "long_context": None if long is None else
                         {k: long[k] for k in ("context", "value", "decode_kernel_us", "achieved", "frac", "traffic",
                                               "kernel", "step")},
                         "other_kernels": None if rows is None else rows_summary(rows)},
            "e2e": {"value": c_us, "unit": "us/layer-token", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": f"per call through the C ABI ({calls_per_step} calls per step)",
                    "graph_replay_value": g_us},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "long_context": long,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
