#!/usr/bin/env python
"""Benchmark of indexer-driven sparse attention on one GB300 (or N independent replicas).

Headline: million-token decode (batch 1, context 1,048,320 = 262,080 pooled blocks,
12 layers, 16 query / 2 KV heads, budget 2048). One step = one decode token through
all 12 layers; each layer-step pools the newest complete block, scores every pooled
block, selects the top 512, and runs the split-K gathered attention with its LSE merge.
The 12 layer-steps are replayed as one CUDA graph, layers in stream order.
Metric: layer-steps/s (plus the algorithmic HBM GB/s it implies). The same JSON line
carries the prefill chunk (4096 queries over a 262,144-token history) in chunk tok/s.

Inputs are synthetic (seeded), already resident in HBM for `value`; `e2e` adds the
per-step host->device copy of the new token's inputs and the device->host read of the
step's result through the same C-ABI path. The working set (12 x 64 MiB pooled keys
+ 12 x 2 GiB K/V) is far larger than L2, so no explicit flush is needed between steps.

`--impl reference` times the fp64 CPU oracle on the host cores on a bounded sample of
the same workload (one layer-step per step).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode layer-steps/s at 1M ctx (+ HBM GB/s; prefill chunk tok/s)"
UNIT = "layer-steps/s"
N_LAYERS = 12
CTX_1M = 1048320


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--path", choices=["fused", "separate"], default="fused",
                    help="fused: qsa_decode_step (one launch per layer-step); separate: the five calls")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kv-host", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-mla", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the tiny / long / batched decode legs")
    ap.add_argument("--prefetch", action="store_true",
                    help="headline graph with each layer-step's L2 prefetch hint of the next layer's keys")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-instrument", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--case", choices=sorted(CASES),
                    help="run one kernel's case a few times and exit (the target of ncu captures)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sust=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


def recorded_traffic(kernel: str):
    """DRAM bytes per launch (read + write) from the committed ncu capture of `kernel`,
    or None when the kernel's sources changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        m = hashlib.sha256()
        for name in rec["sources"]:
            with open(os.path.join(ROOT, "indexer_driven_sparse_gb300", "csrc", name), "rb") as f:
                m.update(f.read())
        return float(rec["dram_bytes_per_launch"]) if m.hexdigest() == rec["sha256"] else None
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qsa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax = float(f[2])
                    power.append(float(f[3]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        finally:
            try:
                os.remove(self.path)
            except OSError:
                pass
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


class DeviceEvents:
    """Timing events recorded as graph nodes (cudaEventRecordExternal) on a capturing
    stream, so per-kernel durations can be read after each graph replay."""

    def __init__(self):
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.events = []

    def new(self):
        ev = ctypes.c_void_p()
        if self.rt.cudaEventCreate(ctypes.byref(ev)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        self.events.append(ev)
        return ev

    def record(self, ev, stream_handle: int):
        if self.rt.cudaEventRecordWithFlags(ev, ctypes.c_void_p(stream_handle), 1) != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed")

    def elapsed_ms(self, a, b) -> float:
        ms = ctypes.c_float()
        if self.rt.cudaEventElapsedTime(ctypes.byref(ms), a, b) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return ms.value


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- decode

class DecodeLayers:
    """12 layers of the million-token decode workload resident in HBM."""

    def __init__(self, n_layers, device, fused=True, prefetch=False):
        import torch
        from indexer_driven_sparse_gb300 import inputs as I
        from indexer_driven_sparse_gb300.pipeline import DecodeBatch
        self.fused = fused
        self.prefetch = prefetch
        self.w = I.million_decode(seed=0, device=device, n_layers=n_layers)
        self.b = DecodeBatch(16, 2, self.w.ctx_len, device=device)
        self.pooled = []
        for L in self.w.layers:
            pk = self.b.new_pooled()
            self.b.pool(L.raw_idx_k, pk)
            self.pooled.append(pk)
        p = self.w.ctx_len[0]
        nblk = (p + 1) // 4
        i32 = dict(dtype=torch.int32, device=device)
        self.inc_begin = torch.tensor([nblk - 1], **i32)   # newest complete block
        self.inc_end = torch.tensor([nblk], **i32)
        torch.cuda.synchronize()
        st = self.b.device_status()
        if st[0] != 0:
            raise RuntimeError(f"device status after pooling: {st}")

    def layer_step(self, l, events=None, stream_handle=None):
        """Pool the newest block, then score -> top-k -> attend for layer l."""
        from indexer_driven_sparse_gb300 import binding as qb
        b, L = self.b, self.w.layers[l]
        rec = (lambda name: events(l, name)) if events else (lambda name: None)
        if self.fused:
            # the next layer's pooled keys (layer 0's after the last layer: the next token's
            # first layer) are prefetched into L2 during this layer-step's exchanges
            nxt = self.pooled[(l + 1) % len(self.pooled)] if self.prefetch else None
            rec("step0")
            b.fused_step(L.raw_idx_k, self.pooled[l], L.q_idx, L.q, L.k_cache, L.v_cache, next_read=nxt)
            rec("step1")
            return
        rec("pool0")
        qb.qsa_pool_keys(b.cfg, L.raw_idx_k, b.tok_off, b.blk_off, self.inc_begin, self.inc_end, 1, self.pooled[l],
                         b.ws)
        rec("pool1")
        b.score(L.q_idx, self.pooled[l])
        rec("score1")
        b.topk()
        rec("topk1")
        b.attend(L.q, L.k_cache, L.v_cache)
        rec("attend1")

    def step(self, events=None):
        for l in range(len(self.w.layers)):
            self.layer_step(l, events)


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_graph(g, stream, steps, warmup, world):
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(steps):
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return t0.elapsed_time(t1) / 1000.0


def time_graph_per_replay(g, stream, steps, warmup, flush=None):
    """Each replay timed alone with CUDA events on the launching stream; with `flush` (a
    tensor larger than L2) the buffer is rewritten between replays, outside the timed
    events, so every replay starts with a cold L2. Returns the per-replay seconds."""
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            if flush is not None:
                flush.add_(1)
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / 1000.0 for a, b in ev]


def decode_config_leg(name, w, pk, steps, warmup, cold=False):
    """A decode workload's layers resident in HBM, one CUDA graph of its fused layer-steps
    (layers in stream order). Warm: replays back to back; cold (optional): L2 flushed by
    writing a 512 MiB buffer between replays. Reports layer-steps/s (mean and median over
    replays), the algorithmic bytes per layer-step and the HBM roofline fraction."""
    import torch
    from indexer_driven_sparse_gb300 import accounting as A
    from indexer_driven_sparse_gb300.pipeline import DecodeBatch
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len, device="cuda")
    pooled = []
    for L in w.layers:
        pk_l = b.new_pooled()
        b.pool(L.raw_idx_k, pk_l)
        pooled.append(pk_l)
    stream = torch.cuda.Stream()

    n_l = len(w.layers)

    def body():
        for l, L in enumerate(w.layers):
            b.fused_step(L.raw_idx_k, pooled[l], L.q_idx, L.q, L.k_cache, L.v_cache)

    with torch.cuda.stream(stream):
        body()
    torch.cuda.synchronize()
    st = b.fused_status()
    if st[0] != 0:
        raise RuntimeError(f"device status in the {name} leg: {st}")
    g = capture(body, stream)
    t_all = time_graph(g, stream, steps, warmup, 1)
    per = time_graph_per_replay(g, stream, steps, 0)
    nbytes = A.decode_layer_step_bytes(w.ctx_len, w.n_q_heads, w.n_kv_heads)
    us_mean = 1e6 * t_all / (steps * n_l)
    us_med = 1e6 * statistics.median(per) / n_l
    gbs = nbytes / (us_mean * 1e-6) / 1e9
    out = {"workload": name, "batch": w.batch, "layers": n_l, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
           "layer_steps_per_s": 1e6 / us_mean, "us_per_layer_step_mean": us_mean,
           "us_per_layer_step_median": us_med, "algorithmic_bytes_per_layer_step": nbytes,
           "hbm_gbs_algorithmic": gbs, "roofline_frac": gbs / pk["hbm"], "peak_gbs": pk["hbm"],
           "gpu_launches_per_layer_step": 1}
    if cold:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        per_c = time_graph_per_replay(g, stream, steps, 0, flush=flush.view(torch.int32))
        us_c = 1e6 * statistics.mean(per_c) / n_l
        out.update({"cold_l2_us_per_layer_step_mean": us_c,
                    "cold_l2_us_per_layer_step_median": 1e6 * statistics.median(per_c) / n_l,
                    "cold_l2_layer_steps_per_s": 1e6 / us_c,
                    "cold_l2_hbm_gbs_algorithmic": nbytes / (us_c * 1e-6) / 1e9,
                    "cold_l2_roofline_frac": nbytes / (us_c * 1e-6) / 1e9 / pk["hbm"]})
        del flush
    del g
    return out


def config_legs(pk, steps, warmup):
    """Throughput of the tiny (1 layer), long (12 layers) and batched (B = 32, 12 layers)
    decode workloads, each through the fused step; the tiny and long ones also cold-L2."""
    import torch
    from indexer_driven_sparse_gb300 import inputs as I
    legs = {}
    for name, make, cold in (("tiny_decode_ctx4096", lambda: I.tiny_decode(device="cuda"), True),
                             ("long_decode_ctx131072", lambda: I.long_decode(device="cuda"), True),
                             ("batched_decode_b32", lambda: I.batched_decode(device="cuda"), False)):
        w = make()
        legs[name] = decode_config_leg(name, w, pk, steps, warmup, cold)
        del w
        torch.cuda.empty_cache()
    return legs


def instrumented_kernel_times(dl, stream, steps):
    """Per-kernel mean durations (us) from event nodes inside a replayed step graph."""
    import torch
    ev = DeviceEvents()
    marks = {}
    h = stream.cuda_stream

    def events(l, name):
        e = ev.new()
        ev.record(e, h)
        marks[(l, name)] = e

    def body():
        ev_first = ev.new()
        ev.record(ev_first, h)
        marks[("start",)] = ev_first
        dl.step(events)

    g = capture(body, stream)
    if dl.fused:
        spans = {"decode_step": ("step0", "step1")}
    else:
        spans = {"pool": ("pool0", "pool1"), "score": ("pool1", "score1"), "topk": ("score1", "topk1"),
                 "attend": ("topk1", "attend1")}
    sums = {k: 0.0 for k in spans}
    n_layers = len(dl.w.layers)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize()
        for l in range(n_layers):
            for k, (a, b) in spans.items():
                sums[k] += ev.elapsed_ms(marks[(l, a)], marks[(l, b)])
    return {k: 1000.0 * v / (steps * n_layers) for k, v in sums.items()}


def e2e_decode(dl, stream, steps, warmup):
    """Same step with the new token's inputs copied host->device from pinned memory
    and the last layer's output read back, every step. The layers' q and q_idx live in
    one staging buffer (one copy for all layers); the new token's K, V and raw indexer-key
    rows are appended to caches stacked with a fixed layer stride (one strided copy each,
    qsa_copy_rows). The copies and the layer-steps are one CUDA graph, replayed and waited
    for on the host once per step."""
    import torch
    from indexer_driven_sparse_gb300 import binding as qb
    b, layers = dl.b, dl.w.layers
    n_l = len(layers)
    p = dl.w.ctx_len[0]
    # per layer: q [16,256] + q_idx [128] + new token k,v [2,256] each + raw idx key [128] (bf16)
    qq = 16 * 256 + 128
    per_layer = qq + 2 * 2 * 256 + 128
    # restack the caches (same values) and re-home q / q_idx into the staging buffer
    stacked = {}
    for name in ("k_cache", "v_cache", "raw_idx_k"):
        t0 = getattr(layers[0], name)
        allt = torch.empty((n_l,) + tuple(t0.shape), dtype=t0.dtype, device=t0.device)
        for l, L in enumerate(layers):
            allt[l].copy_(getattr(L, name))
            setattr(L, name, allt[l])
        stacked[name] = allt
    dev_q = torch.empty(n_l * qq, dtype=torch.bfloat16, device="cuda")
    for l, L in enumerate(layers):
        dev_q[l * qq:l * qq + 4096].copy_(L.q.view(-1))
        dev_q[l * qq + 4096:(l + 1) * qq].copy_(L.q_idx.view(-1))
        L.q = dev_q[l * qq:l * qq + 4096].view(L.q.shape)
        L.q_idx = dev_q[l * qq + 4096:(l + 1) * qq].view(L.q_idx.shape)
    torch.cuda.synchronize()
    host_in = torch.empty(n_l * per_layer, dtype=torch.bfloat16).pin_memory()
    host_in.copy_(torch.randn(host_in.shape, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16) / 16)
    h_q = host_in[:n_l * qq]
    h_k = host_in[n_l * qq:n_l * (qq + 512)]
    h_v = host_in[n_l * (qq + 512):n_l * (qq + 1024)]
    h_r = host_in[n_l * (qq + 1024):]
    rows = []                               # (dst, dst pitch, src, row bytes) of the appended rows
    for name, src, row in (("k_cache", h_k, 1024), ("v_cache", h_v, 1024), ("raw_idx_k", h_r, 256)):
        allt = stacked[name]
        rows.append((allt[0, p].data_ptr(), allt.stride(0) * 2, src.data_ptr(), row))
    host_out = torch.empty(16 * 256 + 32, dtype=torch.bfloat16).pin_memory()
    out_view = b.out.view(-1)
    lse_view = b.lse.view(torch.bfloat16).view(-1)

    def body():
        # the step's copies in, the 12 layer-steps, the result out: one graph per step
        dev_q.copy_(h_q, non_blocking=True)
        for dst, pitch, src, row in rows:
            qb.qsa_copy_rows(dst, pitch, src, row, row, n_l, stream)
        for l in range(n_l):
            dl.layer_step(l)
        host_out[:4096].copy_(out_view, non_blocking=True)
        host_out[4096:].copy_(lse_view, non_blocking=True)

    g = capture(body, stream)

    def one_step():
        g.replay()
        stream.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one_step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            one_step()
        dt = time.perf_counter() - t0
    h2d = host_in.numel() * 2
    d2h = host_out.numel() * 2
    return dt, h2d, d2h


def kv_host_bench(dl, stream, steps, warmup, n_layers=2):
    """The fused step with each layer's K/V cache and raw indexer keys in pinned host memory
    (the pooled keys stay in HBM): the selected rows are gathered over the host link."""
    import torch
    b, layers = dl.b, dl.w.layers[:n_layers]
    host = []
    for L in layers:
        hk, hv, hr = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (L.k_cache, L.v_cache, L.raw_idx_k))
        hk.copy_(L.k_cache)
        hv.copy_(L.v_cache)
        hr.copy_(L.raw_idx_k)
        host.append((hk, hv, hr))
    torch.cuda.synchronize()

    def body():
        for l, L in enumerate(layers):
            hk, hv, hr = host[l]
            b.fused_step(hr, dl.pooled[l], L.q_idx, L.q, hk, hv)

    with torch.cuda.stream(stream):
        body()
    torch.cuda.synchronize()
    st = b.fused_status()
    if st[0] != 0:
        raise RuntimeError(f"device status with host K/V: {st}")
    g = capture(body, stream)
    t = time_graph(g, stream, steps, warmup, 1)
    del g
    n = steps * len(layers)
    p = dl.w.ctx_len[0]
    kv_bytes = (2048 + (p % 4) + 1) * 2 * 2 * 256 * 2      # selected tokens + tail, K and V, both heads
    out = {"layers": len(layers), "layer_steps_per_s": n / t, "us_per_layer_step": 1e6 * t / n,
           "kv_bytes_per_layer_step": kv_bytes, "host_gather_gbs": kv_bytes * n / t / 1e9,
           "note": "K/V and raw indexer keys in pinned host memory; pooled keys in HBM"}
    out["with_row_cache"] = rowcache_bench(b, dl, layers, host, stream, steps)
    out["host_link"] = host_link_bench(host[0][0], stream)
    return out


def rowcache_bench(b, dl, layers, host, stream, steps, n_slots=16384):
    """The same host-memory layers through qsa_decode_step_rowcache, eager (every call takes a
    new epoch, so a captured graph cannot replay it): the first step of each layer misses
    everywhere and fills the cache; the steps after it repeat the same selection and hit
    everywhere (the pages measured 60-85 % overlap between consecutive steps)."""
    import torch
    from indexer_driven_sparse_gb300 import binding as qb
    caches = [qb.rowcache_new(b.cfg, n_slots) for _ in layers]
    epoch = [0]
    # the first call of the row-cache kernel sizes its grid on the host: make it before timing
    L0, h0 = layers[0], host[0]
    b.fused_step_rowcache(h0[2], dl.pooled[0], L0.q_idx, L0.q, h0[0], h0[1], qb.rowcache_new(b.cfg, n_slots),
                          n_slots, 1)
    torch.cuda.synchronize()

    def body():
        epoch[0] += 1
        for l, L in enumerate(layers):
            hk, hv, hr = host[l]
            b.fused_step_rowcache(hr, dl.pooled[l], L.q_idx, L.q, hk, hv, caches[l], n_slots, epoch[0])

    res = {}
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        body()                                        # cold: every row missed and cached
        e1.record(stream)
        torch.cuda.synchronize()
        res["cold_us_per_layer_step"] = e0.elapsed_time(e1) * 1e3 / len(layers)
        for _ in range(3):
            body()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            body()
        e1.record(stream)
    torch.cuda.synchronize()
    st = b.fused_status()
    if st[0] != 0:
        raise RuntimeError(f"device status with the row cache: {st}")
    us = e0.elapsed_time(e1) * 1e3 / (steps * len(layers))
    res.update({"hot_us_per_layer_step": us, "hot_layer_steps_per_s": 1e6 / us, "n_slots": n_slots,
                "timing": "eager launches (one epoch per call), CUDA events on the stream"})
    del caches
    return res


def host_link_bench(hk, stream, nbytes=1 << 29, reps=5):
    """The host link's bandwidth, through this library's calls: bulk copies of 512 MiB between
    pinned host memory and HBM (qsa_copy_rows), and a kernel streaming 512 MiB of bf16 K rows out
    of mapped pinned host memory (qsa_quantize_kv_fp8 reads each row once and writes its FP8
    codes and scales to HBM)."""
    import torch
    from indexer_driven_sparse_gb300 import binding as qb
    src = hk.view(-1)[: nbytes // 2]                          # pinned, bf16
    dev = torch.empty(nbytes // 2, dtype=torch.bfloat16, device="cuda")
    rows = nbytes // 512
    codes = torch.empty(rows, 256, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, 2, dtype=torch.float32, device="cuda")
    res = {}
    for name, fn in (("h2d_copy_gbs", lambda: qb.qsa_copy_rows(dev, nbytes, src, nbytes, nbytes, 1, stream)),
                     ("d2h_copy_gbs", lambda: qb.qsa_copy_rows(src, nbytes, dev, nbytes, nbytes, 1, stream)),
                     ("zero_copy_read_gbs", lambda: qb.qsa_quantize_kv_fp8(src.view(rows, 256), codes, scales, stream))):
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        res[name] = nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    res["bytes"] = nbytes
    res["note"] = "copies: one cudaMemcpy2DAsync of 512 MiB; zero-copy: 16-byte loads of mapped pinned memory"
    del dev, codes, scales
    return res


def fp8_keys_bench(dl, stream, steps, warmup, pk):
    """Decode with FP8 indexer keys (128 E4M3 codes + one fp32 scale per pooled block): per
    layer, re-pool the newest block into codes, then score -> top-k -> attention as separate
    calls; and each scan alone (FP8 and bf16 keys) over the same 12 layers."""
    import torch
    from indexer_driven_sparse_gb300 import accounting as A
    from indexer_driven_sparse_gb300 import binding as qb
    b, layers = dl.b, dl.w.layers
    keys = []
    for L in layers:
        codes, scales = b.new_fp8_keys()
        b.pool_fp8(L.raw_idx_k, codes, scales)
        keys.append((codes, scales))
    torch.cuda.synchronize()

    def step():
        for l, L in enumerate(layers):
            codes, scales = keys[l]
            qb.qsa_pool_keys_fp8(b.cfg, L.raw_idx_k, b.tok_off, b.blk_off, dl.inc_begin, dl.inc_end, 1, codes,
                                 scales, b.ws)
            b.step_fp8(L.q_idx, L.q, L.k_cache, L.v_cache, codes, scales)

    def scan_fp8():
        for l, L in enumerate(layers):
            b.score_fp8(L.q_idx, *keys[l])

    def scan_bf16():
        for l, L in enumerate(layers):
            b.score(L.q_idx, dl.pooled[l])

    def fused():
        for l, L in enumerate(layers):
            codes, scales = keys[l]
            b.fused_step_fp8(L.raw_idx_k, codes, scales, L.q_idx, L.q, L.k_cache, L.v_cache)

    us = {}
    for name, fn in (("fused", fused), ("step", step), ("scan_fp8", scan_fp8), ("scan_bf16", scan_bf16)):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        st = b.fused_status() if name == "fused" else b.device_status()
        if st[0] != 0:
            raise RuntimeError(f"device status in the FP8 leg ({name}): {st}")
        g = capture(fn, stream)
        t = time_graph(g, stream, steps, warmup, 1)
        del g
        us[name] = 1e6 * t / (steps * len(layers))
    ctx = dl.w.ctx_len
    b8, b16 = A.score_scan_bytes_fp8(ctx), A.score_scan_bytes(ctx)
    g8 = b8 / (us["scan_fp8"] * 1e-6) / 1e9
    g16 = b16 / (us["scan_bf16"] * 1e-6) / 1e9
    fb = A.decode_layer_step_bytes_fp8(ctx, 16)
    fg = fb / (us["fused"] * 1e-6) / 1e9
    return {"fused_layer_steps_per_s": 1e6 / us["fused"], "fused_us_per_layer_step": us["fused"],
            "fused_algorithmic_bytes": fb, "fused_hbm_gbs_algorithmic": fg, "fused_frac": fg / pk["hbm"],
            "path": "fused: qsa_decode_step_fp8 (one launch per layer-step); separate: pool_fp8 (newest block), "
                    "score_fp8, topk, attention + merge",
            "layer_steps_per_s": 1e6 / us["step"], "us_per_layer_step": us["step"],
            "scan_fp8_us": us["scan_fp8"], "scan_fp8_bytes": b8, "scan_fp8_gbs": g8,
            "scan_fp8_frac": g8 / pk["hbm"], "scan_bf16_us": us["scan_bf16"], "scan_bf16_bytes": b16,
            "scan_bf16_gbs": g16, "scan_bf16_frac": g16 / pk["hbm"], "peak_src": pk["src"],
            "gpu_launches_per_layer_step": 5}


def fp8_kv_bench(dl, stream, steps, warmup, pk):
    """Decode with FP8 K/V rows (codes + one fp32 scale per 128 dims, qsa_quantize_kv_fp8) on the
    same 12 million-token layers: the fused step (qsa_decode_step_fp8kv) in a 12-layer graph over
    bf16 indexer keys and over FP8 indexer keys, each against its algorithmic bytes."""
    import torch
    from indexer_driven_sparse_gb300 import accounting as A
    from indexer_driven_sparse_gb300 import binding as qb
    b, layers = dl.b, dl.w.layers
    kv8, keys8 = [], []
    for L in layers:
        planes = []
        for x in (L.k_cache, L.v_cache):
            c = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
            sc = torch.empty(x.shape[:-1] + (2,), dtype=torch.float32, device=x.device)
            qb.qsa_quantize_kv_fp8(x, c, sc)
            planes += [c, sc]
        kv8.append(tuple(planes))
        codes, scales = b.new_fp8_keys()
        b.pool_fp8(L.raw_idx_k, codes, scales)
        keys8.append((codes, scales))
    torch.cuda.synchronize()
    out = {"format": "K and V rows as 256 E4M3 codes + 2 fp32 scales per token and KV head (264 B of 512)",
           "kv_bytes_per_layer_step": A.kv_read_bytes_fp8(A.attended(dl.w.ctx_len[0])), "peak_src": pk["src"],
           "gpu_launches_per_layer_step": 1}
    for name, fp8_keys in (("bf16_keys", False), ("fp8_keys", True)):
        def fn():
            for l, L in enumerate(layers):
                keys = keys8[l] if fp8_keys else dl.pooled[l]
                b.fused_step_fp8kv(L.raw_idx_k, keys, L.q_idx, L.q, kv8[l])
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        st = b.fused_status()
        if st[0] != 0:
            raise RuntimeError(f"device status in the FP8 K/V leg ({name}): {st}")
        g = capture(fn, stream)
        t = time_graph(g, stream, steps, warmup, 1)
        del g
        us = 1e6 * t / (steps * len(layers))
        nbytes = A.decode_layer_step_bytes_fp8kv(dl.w.ctx_len, 16, fp8_keys)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"layer_steps_per_s": 1e6 / us, "us_per_layer_step": us, "algorithmic_bytes": nbytes,
                     "hbm_gbs_algorithmic": gbs, "frac": gbs / pk["hbm"]}
    del kv8, keys8
    torch.cuda.empty_cache()
    return out


def mla_bench(steps, warmup, pk, batch=64):
    """Sparse MLA decode (MQA form, tensor cores): `batch` queries of 64 heads, each over its
    own 2048 rows of a million-token FP8 cache (656 B per row)."""
    import torch
    from indexer_driven_sparse_gb300 import accounting as A
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import inputs as I
    H, rows = 64, 2048
    w = I.mla_workload(1 << 20, [rows] * batch, H, seed=0, device="cuda")
    ws = qb.sparse_mla_workspace(H, batch, rows)
    out = torch.empty(batch, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(batch, H, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        qb.qsa_sparse_mla_decode(w.q, w.kv, w.rows, w.n_rows, out, lse, ws)

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    st = qb.qsa_read_device_status(ws)
    if st[0] != 0:
        raise RuntimeError(f"sparse MLA device status {st}")
    g = capture(call, stream)
    n = max(20, steps // 4)
    t = time_graph(g, stream, n, max(3, warmup), 1) / n
    del g
    flops = batch * A.sparse_mla_query_flops(H, rows)
    nbytes = batch * A.sparse_mla_query_bytes(H, rows)
    ach = flops / t / 1e12
    # DRAM bytes of the tile kernel from its capture on 16 queries, scaled by the query count
    # (each query's tiles read and write the same amounts)
    cap = recorded_traffic("mla_tr")
    traffic = cap * batch / 16 if cap is not None else None
    # 191 FLOP/B is below GB300's ridge (measured bf16 / measured HBM, about 283 FLOP/B), so
    # the binding roofline is HBM; the tensor fraction is reported beside it
    gbs = nbytes / t / 1e9
    return {"workload": f"sparse MLA decode: {batch} queries x 64 heads, 2048 FP8 rows each (656 B), "
                        "million-token cache",
            "queries_per_s": batch / t, "us_per_call": t * 1e6,
            "algorithmic_gflop": flops / 1e9, "algorithmic_mb": nbytes / 1e6, "hbm_gbs": gbs,
            "intensity_flop_per_byte": flops / nbytes, "ridge_flop_per_byte": pk["bf16"] * 1e12 / (pk["hbm"] * 1e9),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": gbs / pk["hbm"], "traffic": traffic, "kernel": "mla_tr + mla_merge_tr"},
            "tensor_frac": ach / pk["bf16"], "tensor_tflops": ach,
            "gpu_launches_per_call": 2}


# ----------------------------------------------------------------------------- prefill

def union_stats(c, nc, p0, att_flops):
    """Selection structure of a prefill chunk (reporting only, from the blocks the chunk
    selected): the mean overlap of consecutive queries' top-512 sets, and the union of the
    selected blocks (and own blocks) per 16-query tile, which the tensor-core kernel packs
    into 64-token chunks of 128 (query, head) rows; executed FLOPs are estimated as
    chunks x 64 tokens x 128 rows x 256 dims x 2 (QK and PV) x 2 FLOP for each of 2 KV heads."""
    import torch
    blocks = c.blocks[:nc].long()
    prev, cur = blocks[:-1].contiguous(), blocks[1:].contiguous()
    idx = torch.searchsorted(prev, cur).clamp(max=prev.shape[1] - 1)
    overlap = (torch.gather(prev, 1, idx) == cur).float().mean(dim=1).mean().item()
    own = ((p0 + torch.arange(nc, device=blocks.device)) // 4).unsqueeze(1)
    tiles = torch.cat([blocks, own], dim=1).view(nc // 16, -1)
    srt = torch.sort(tiles, dim=1).values
    union = 1 + (srt[:, 1:] != srt[:, :-1]).sum(dim=1)
    chunks = torch.div(4 * union + 63, 64, rounding_mode="floor")
    executed = float(chunks.sum().item()) * 2 * 64 * 128 * 256 * 2 * 2
    return {"mean_consecutive_overlap": overlap, "union_blocks_per_16_query_tile": float(union.float().mean().item()),
            "chunks_estimate": int(2 * chunks.sum().item()), "executed_gflop_estimate": executed / 1e9,
            "executed_over_algorithmic": executed / att_flops}


def prefill_bench(steps, warmup, pk):
    import torch
    from indexer_driven_sparse_gb300 import accounting as A
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import inputs as I
    from indexer_driven_sparse_gb300.pipeline import PrefillChunk
    w = I.prefill_chunk(device="cuda")
    L = w.layers[0]
    p0, nc = w.ctx_len[0], w.n_chunk
    c = PrefillChunk(16, 2, p0, nc, 8192, device="cuda")
    pooled = c.new_pooled()
    c.pool(L.raw_idx_k, pooled)            # history blocks (setup)
    i32 = dict(dtype=torch.int32, device="cuda")
    chunk_begin = torch.tensor([p0 // 4], **i32)
    chunk_end = torch.tensor([(p0 + nc) // 4], **i32)
    stream = torch.cuda.Stream()

    def chunk():
        qb.qsa_pool_keys(c.cfg, L.raw_idx_k, c.tok_off, c.blk_off, chunk_begin, chunk_end, nc // 4, pooled, c.ws)
        c.run(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)

    def attend_only():
        c.attend(L.q, L.k_cache, L.v_cache)

    def score_only():
        c.score(L.q_idx, pooled)

    def topk_only():
        c.topk()

    def select_only():
        c.select(L.q_idx, pooled)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        chunk()
    torch.cuda.synchronize()
    st = c.device_status()
    if st[0] != 0:
        raise RuntimeError(f"prefill device status {st}")
    n = max(2, steps // 20)
    g_chunk = capture(chunk, stream)
    t_chunk = time_graph(g_chunk, stream, n, max(1, warmup), 1) / n
    g_att = capture(attend_only, stream)
    t_att = time_graph(g_att, stream, n, max(1, warmup), 1) / n
    phases = {"attention": t_att * 1e3}
    for name, fn in (("select", select_only), ("score", score_only), ("topk", topk_only)):
        g1 = capture(fn, stream)
        phases[name] = time_graph(g1, stream, n, max(1, warmup), 1) / n * 1e3
        del g1
    # the same attention with K/V in pinned host memory: gathered over the link, or staged into
    # a device arena first (one bulk copy of the rows per call)
    hk, hv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (L.k_cache, L.v_cache))
    hk.copy_(L.k_cache)
    hv.copy_(L.v_cache)
    stage = torch.empty(2 * hk.numel() * 2, dtype=torch.uint8, device="cuda")
    host = {}
    for name, fn in (("zero_copy_ms", lambda: c.attend(L.q, hk, hv)),
                     ("staged_ms", lambda: c.attend_staged(L.q, hk, hv, stage))):
        g1 = capture(fn, stream)
        host[name] = time_graph(g1, stream, n, max(1, warmup), 1) / n * 1e3
        del g1
    host["staged_bytes"] = stage.numel()
    del hk, hv
    # the same attention over FP8 K/V rows (qsa_sparse_prefill_chunk_fp8kv: the rows dequantised
    # into the bf16 stage by one launch, then the same kernel); the dequantiser alone (two calls,
    # K then V) against the HBM roofline
    kv8 = []
    for t in (L.k_cache, L.v_cache):
        codes = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
        scales = torch.empty(t.shape[:-1] + (2,), dtype=torch.float32, device="cuda")
        qb.qsa_quantize_kv_fp8(t, codes, scales)
        kv8 += [codes, scales]
    half = L.k_cache.numel() * 2
    kx = stage[:half].view(torch.bfloat16).view(L.k_cache.shape)
    vx = stage[half:].view(torch.bfloat16).view(L.v_cache.shape)

    def dequant():
        qb.qsa_dequantize_kv_fp8(kv8[0], kv8[1], kx)
        qb.qsa_dequantize_kv_fp8(kv8[2], kv8[3], vx)

    fp8kv = {}
    for name, fn in (("attention_ms", lambda: c.attend_fp8kv(L.q, kv8, stage)), ("dequant_ms", dequant)):
        g1 = capture(fn, stream)
        fp8kv[name] = time_graph(g1, stream, n, max(1, warmup), 1) / n * 1e3
        del g1
    st = c.device_status()
    if st[0] != 0:
        raise RuntimeError(f"prefill device status after the FP8 K/V leg {st}")
    dq_bytes = A.kv_dequant_bytes_fp8(p0 + nc)
    dq_gbs = dq_bytes / (fp8kv["dequant_ms"] * 1e-3) / 1e9
    # DRAM bytes of one launch over K (its capture), twice for the K and V launches
    dq_cap = recorded_traffic("dequantize_kv_fp8")
    fp8kv.update({"format": "K and V rows as 256 E4M3 codes + 2 fp32 scales per token and KV head",
                  "fp8_kv_bytes": A.kv_read_bytes_fp8(p0 + nc), "bf16_stage_bytes": stage.numel(),
                  "dequant_roofline": {"bound": "hbm", "achieved": dq_gbs, "peak": pk["hbm"], "unit": "GB/s",
                                       "frac": dq_gbs / pk["hbm"], "algorithmic_bytes": dq_bytes,
                                       "traffic": 2 * dq_cap if dq_cap is not None else None,
                                       "kernel": "dequantize_kv_fp8 (two launches: K, V)"},
                  "gpu_launches_per_call": 4})
    del kv8, stage, kx, vx
    att_flops = A.prefill_attention_flops(p0, nc)
    score_flops = A.prefill_score_flops(p0, nc)
    ach = att_flops / t_att / 1e12
    unions = {"correlated_rho_0.985": dict(union_stats(c, nc, p0, att_flops), attention_ms=t_att * 1e3)}
    # the stress datum: independent queries (rho = 0), the worst case for union tiles
    w0 = I.prefill_chunk(device="cuda", rho=0.0)
    L0 = w0.layers[0]
    c0 = PrefillChunk(16, 2, p0, nc, 8192, device="cuda")
    pooled0 = c0.new_pooled()
    c0.pool(L0.raw_idx_k, pooled0)
    with torch.cuda.stream(stream):
        c0.run(L0.q_idx, L0.q, L0.k_cache, L0.v_cache, pooled0)
    torch.cuda.synchronize()
    st = c0.device_status()
    if st[0] != 0:
        raise RuntimeError(f"prefill device status (independent queries) {st}")
    g1 = capture(lambda: c0.attend(L0.q, L0.k_cache, L0.v_cache), stream)
    t_att0 = time_graph(g1, stream, n, max(1, warmup), 1) / n
    del g1
    unions["independent_rho_0"] = dict(union_stats(c0, nc, p0, att_flops), attention_ms=t_att0 * 1e3,
                                       attention_tflops=att_flops / t_att0 / 1e12)
    del w0, L0, c0, pooled0
    torch.cuda.empty_cache()
    return {
        "selection_overlap_and_union_tiles": unions,
        "attention_kv_in_host_memory": host,
        "attention_fp8_kv": fp8kv,
        "workload": f"prefill chunk: {nc} queries at p0={p0}, 16 q / 2 kv heads, intervals 8192",
        "chunk_tok_s": nc / t_chunk, "ms_per_chunk": t_chunk * 1e3,
        "attention_only_tok_s": nc / t_att, "ms_attention": t_att * 1e3,
        "phases_ms": phases,
        "attention_gflop_algorithmic": att_flops / 1e9, "scoring_gflop_algorithmic": score_flops / 1e9,
        "roofline": {"bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": ach / pk["bf16"], "traffic": recorded_traffic("prefill_tc"),
                     "kernel": "prefill_tc (algorithmic FLOPs)"},
    }


# ----------------------------------------------------------------------------- single-kernel cases

def _case_decode_step(reps):
    """One million-token layer (about 2.2 GB on the device): pool, then `reps` fused
    decode steps (qsa_decode_step, one launch each)."""
    import torch
    from indexer_driven_sparse_gb300 import inputs as I
    from indexer_driven_sparse_gb300.pipeline import DecodeBatch
    w = I.million_decode(n_layers=1)
    L = w.layers[0]
    b = DecodeBatch(16, 2, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    for _ in range(reps):
        b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
    torch.cuda.synchronize()
    return b.fused_status()


def _case_decode_trace(reps):
    """Phase trace of the fused decode step on one million-token layer: the workspace's debug
    word asks every CTA's thread 0 to stamp %globaltimer at 16 points of the launch; prints the
    median over the CTAs of each stamp, in us from the earliest first stamp, for `reps` eager
    launches (the last one's table)."""
    import numpy as np
    import torch
    from indexer_driven_sparse_gb300 import inputs as I
    from indexer_driven_sparse_gb300.pipeline import DecodeBatch
    w = I.million_decode(n_layers=1)
    L = w.layers[0]
    b = DecodeBatch(16, 2, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    for _ in range(3):
        b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
    torch.cuda.synchronize()
    n_slots, max_ctas = 16, 256                       # the kernel's trace slots per CTA and CTA bound
    ws = b.step_ws
    tr = ws[ws.numel() - max_ctas * n_slots * 8:].view(torch.int64).view(max_ctas, n_slots)
    table = None
    for _ in range(reps):
        ws.view(torch.int32)[3] = 0x7ACE              # the header's debug word: trace this launch
        tr.zero_()
        b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
        torch.cuda.synchronize()
        ws.view(torch.int32)[3] = 0
        t = tr.cpu().numpy().astype(np.int64)
        t = t[t[:, 0] > 0]
        rel = np.where(t > 0, (t - t[:, 0].min()) / 1000.0, np.nan)
        table = {f"slot{i}": [round(float(np.nanmedian(rel[:, i])), 2), round(float(np.nanmin(rel[:, i])), 2),
                              round(float(np.nanmax(rel[:, i])), 2)] for i in range(n_slots)}
    print(json.dumps({"decode_trace_us_median_min_max": table, "ctas": int(t.shape[0])}))
    return b.fused_status()


def _case_decode_fp8(reps):
    """One million-token layer with FP8 indexer keys: pool into codes + scales, then `reps`
    times the standalone FP8 scan (qsa_index_score_fp8) and the fused FP8 step."""
    import torch
    from indexer_driven_sparse_gb300 import inputs as I
    from indexer_driven_sparse_gb300.pipeline import DecodeBatch
    w = I.million_decode(n_layers=1)
    L = w.layers[0]
    b = DecodeBatch(16, 2, w.ctx_len)
    codes, scales = b.new_fp8_keys()
    b.pool_fp8(L.raw_idx_k, codes, scales)
    for _ in range(reps):
        b.score_fp8(L.q_idx, codes, scales)
        b.fused_step_fp8(L.raw_idx_k, codes, scales, L.q_idx, L.q, L.k_cache, L.v_cache)
    torch.cuda.synchronize()
    st = b.device_status()
    return st if st[0] != 0 else b.fused_status()


def _case_decode_fp8kv(reps):
    """One million-token layer with FP8 K/V rows (bf16 indexer keys): quantise K and V, pool,
    then `reps` fused steps over the FP8 rows (qsa_decode_step_fp8kv)."""
    import torch
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import inputs as I
    from indexer_driven_sparse_gb300.pipeline import DecodeBatch
    w = I.million_decode(n_layers=1)
    L = w.layers[0]
    b = DecodeBatch(16, 2, w.ctx_len)
    planes = []
    for x in (L.k_cache, L.v_cache):
        c = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        sc = torch.empty(x.shape[:-1] + (2,), dtype=torch.float32, device=x.device)
        qb.qsa_quantize_kv_fp8(x, c, sc)
        planes += [c, sc]
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    for _ in range(reps):
        b.fused_step_fp8kv(L.raw_idx_k, pooled, L.q_idx, L.q, planes)
    torch.cuda.synchronize()
    return b.fused_status()


def _case_mla(reps):
    """Sparse MLA decode: 16 queries x 64 heads over 2048 rows each of a million-token FP8
    cache (about 0.7 GB on the device), `reps` calls."""
    import torch
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import inputs as I
    w = I.mla_workload(1 << 20, [2048] * 16, 64, seed=0, device="cuda")
    ws = qb.sparse_mla_workspace(64, 16, 2048)
    out = torch.empty(16, 64, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(16, 64, dtype=torch.float32, device="cuda")
    for _ in range(reps):
        qb.qsa_sparse_mla_decode(w.q, w.kv, w.rows, w.n_rows, out, lse, ws)
    torch.cuda.synchronize()
    return qb.qsa_read_device_status(ws)


def _case_dequant_kv_fp8(reps):
    """The prefill chunk's history and chunk (266,240 tokens x 2 KV heads) as FP8 K/V rows,
    dequantised `reps` times into a bf16 stage (qsa_sparse_prefill_chunk_fp8kv's first launch;
    about 1.1 GB on the device)."""
    import torch
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import inputs as I
    w = I.prefill_chunk(device="cuda")
    L = w.layers[0]
    kv8 = []
    for t in (L.k_cache, L.v_cache):
        codes = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
        scales = torch.empty(t.shape[:-1] + (2,), dtype=torch.float32, device="cuda")
        qb.qsa_quantize_kv_fp8(t, codes, scales)
        kv8 += [codes, scales]
    del w, L
    kx = torch.empty(kv8[0].shape, dtype=torch.bfloat16, device="cuda")
    for _ in range(reps):
        qb.qsa_dequantize_kv_fp8(kv8[0], kv8[1], kx)
    torch.cuda.synchronize()
    return (0, 0)


def _case_prefill(reps, attention_only):
    """The prefill chunk (4096 queries over 262,144 tokens, about 1.1 GB on the device):
    pool + score + top-k once, then `reps` chunk attentions (or whole chunks)."""
    import torch
    from indexer_driven_sparse_gb300 import inputs as I
    from indexer_driven_sparse_gb300.pipeline import PrefillChunk
    w = I.prefill_chunk(device="cuda")
    L = w.layers[0]
    c = PrefillChunk(16, 2, w.ctx_len[0], w.n_chunk, 8192, device="cuda")
    pooled = c.new_pooled()
    c.pool(L.raw_idx_k, pooled)
    c.run(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    for _ in range(reps):
        if attention_only:
            c.attend(L.q, L.k_cache, L.v_cache)
        else:
            c.run(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    torch.cuda.synchronize()
    return c.device_status()


CASES = {
    "decode_step": lambda reps: _case_decode_step(reps),
    "decode_fp8": lambda reps: _case_decode_fp8(reps),
    "decode_fp8kv": lambda reps: _case_decode_fp8kv(reps),
    "decode_trace": lambda reps: _case_decode_trace(reps),
    "mla": lambda reps: _case_mla(reps),
    "dequant_kv_fp8": lambda reps: _case_dequant_kv_fp8(reps),
    "prefill_attention": lambda reps: _case_prefill(reps, True),
    "prefill_chunk": lambda reps: _case_prefill(reps, False),
}


def case_main(args):
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import build as qbuild
    qbuild.build()
    qb.load()
    st = CASES[args.case](max(1, args.steps))
    print(json.dumps({"case": args.case, "reps": max(1, args.steps), "device_status": list(st)}))
    return 0 if st[0] == 0 else 1


# ----------------------------------------------------------------------------- CPU oracle leg

_ORACLE_CASE = {}


def _oracle_layer_steps(seconds: float) -> int:
    """Layer-steps of the fp64 oracle (pool the newest block, then the whole decode query)
    completed in `seconds` on the drawn million-token layer."""
    import oracle as O
    c = _ORACLE_CASE
    p, raw = c["p"], c["raw"]
    n, t0 = 0, time.perf_counter()
    while True:
        O.pool_keys(raw[4 * (p // 4 - 1):4 * (p // 4)])
        O.decode_query(p, c["qi"][0], c["pooled"], c["q"][0], c["k"], c["v"], 2)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            return n


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline_child(seconds: float):
    """Time the fp64 oracle on one layer of the million-token decode workload (CPU draw
    of the same recipe): one process with single-threaded BLAS, then one worker per host
    core (forked after the draw, so they share it; no CUDA in this process). Prints one
    JSON object."""
    import multiprocessing as mp

    import numpy as np
    import torch
    import oracle as O
    from indexer_driven_sparse_gb300 import inputs as I
    torch.set_num_threads(1)
    t_setup = time.perf_counter()
    w = I.million_decode(seed=0, device="cpu", n_layers=1)
    L = w.layers[0]
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    raw = bits(L.raw_idx_k)
    _ORACLE_CASE.update(p=w.ctx_len[0], raw=raw, qi=bits(L.q_idx), q=bits(L.q), k=bits(L.k_cache),
                        v=bits(L.v_cache), pooled=O.pool_keys(raw))   # setup: pooled once
    del w, L
    setup = time.perf_counter() - t_setup
    t0 = time.perf_counter()
    n1 = _oracle_layer_steps(seconds)
    dt1 = time.perf_counter() - t0
    cores = os.cpu_count() or 1
    all_s = max(seconds * 2.0 / 3.0, 1.0)
    with mp.get_context("fork").Pool(cores) as pool:
        t0 = time.perf_counter()
        counts = pool.map(_oracle_layer_steps, [all_s] * cores)
        dt_all = time.perf_counter() - t0
    print(json.dumps({"value": n1 / dt1, "n": n1, "seconds": dt1, "setup_s": setup,
                      "all_value": sum(counts) / dt_all, "all_n": sum(counts), "all_seconds": dt_all,
                      "cores": cores, "model": _cpu_model()}))


def run_cpu_baseline(seconds: float):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
                        "--cpu-seconds", str(seconds)], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "error": r.stderr[-400:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["all_value"], "unit": UNIT, "cores": d["cores"], "kind": "oracle",
            "cpu_model": d["model"], "nproc": d["cores"],
            "sample": f"one million-token layer (CPU draw of the same recipe), fp64 numpy, single-threaded BLAS "
                      f"per worker: {d['all_n']} layer-steps in {d['all_seconds']:.1f} s over {d['cores']} "
                      f"forked workers (one per core)",
            "single_core": {"value": d["value"], "cores": 1, "layer_steps": d["n"], "seconds": d["seconds"]}}


def reference_main(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"                  # before numpy loads its BLAS: one host core
    import numpy as np
    import torch
    import oracle as O
    from indexer_driven_sparse_gb300 import inputs as I
    w = I.million_decode(seed=0, device="cpu", n_layers=1)
    L = w.layers[0]
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    raw, qi, q, k, v = bits(L.raw_idx_k), bits(L.q_idx), bits(L.q), bits(L.k_cache), bits(L.v_cache)
    p = w.ctx_len[0]
    pooled = O.pool_keys(raw)

    def step():
        O.pool_keys(raw[4 * (p // 4 - 1):4 * (p // 4)])
        O.decode_query(p, qi[0], pooled, q[0], k, v, 2)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    val = args.steps / dt
    cores = 1
    line = {"metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "million_decode_ctx1048320 (one layer-step per step)", "batch": 1,
                       "ctx": CTX_1M, "n_q_heads": 16, "n_kv_heads": 2, "head_dim": 256, "budget": 2048},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "one million-token layer (CPU draw of the same recipe), fp64 numpy"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- main

def main(argv=None):
    args = parse_args(argv)
    if args.cpu_baseline_child:
        cpu_baseline_child(args.cpu_seconds)
        return 0
    if args.impl == "reference":
        return reference_main(args)
    if args.case:
        return case_main(args)

    cpu_base = None
    rank, local, world = dist_setup()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = run_cpu_baseline(args.cpu_seconds)   # before any CUDA work in this process

    import torch
    from indexer_driven_sparse_gb300 import accounting as A
    from indexer_driven_sparse_gb300 import binding as qb
    from indexer_driven_sparse_gb300 import build as qbuild
    qbuild.build()
    qb.load()
    torch.cuda.set_device(local)
    pk = peaks()

    dl = DecodeLayers(args.layers, "cuda", fused=args.path == "fused", prefetch=args.prefetch)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dl.step()                               # eager warm-up, checks status below
    torch.cuda.synchronize()
    st = dl.b.fused_status() if dl.fused else dl.b.device_status()
    if st[0] != 0:
        raise RuntimeError(f"device status {st}")
    g = capture(dl.step, stream)

    with ClockSampler(local) as clk:
        t = time_graph(g, stream, args.steps, args.warmup, world)
        per_step = time_graph_per_replay(g, stream, args.steps, 0)
    clocks = clk.summary()
    t = max_over_ranks(t, world)
    n_layers = len(dl.w.layers)
    layer_steps = world * args.steps * n_layers
    value = layer_steps / t
    bytes_ls = A.decode_layer_step_bytes(dl.w.ctx_len, 16)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"million_decode_ctx{CTX_1M}", "path": args.path, "batch": 1, "ctx": CTX_1M,
                   "layers": n_layers,
                   "n_q_heads": 16, "n_kv_heads": 2, "head_dim": 256, "idx_dim": 128, "ratio": 4,
                   "budget": 2048, "parallelism": f"replicas{world}",
                   "l2_prefetch": "each layer-step prefetches the next layer's pooled keys into L2 "
                                  "(qsa_decode_step_prefetch)" if args.prefetch else "none",
                   "l2": "inputs larger than L2 (12 x 64 MiB pooled keys + 12 x 2 GiB K/V), no flush"},
        "hbm_gbs_algorithmic": bytes_ls * value / world / 1e9,
        "us_per_layer_step": 1e6 * t / (args.steps * n_layers),
        "us_per_layer_step_median": 1e6 * statistics.median(per_step) / n_layers,
        "us_per_layer_step_mean": 1e6 * statistics.mean(per_step) / n_layers,
        "clocks": clocks,
        "gpu_launches": None,
    }
    launches_per_layer = 1 if dl.fused else 5    # fused step | pool, score, topk, attention, merge
    line["gpu_launches"] = launches_per_layer * n_layers * args.steps

    if dl.fused:
        # the same graph with the other setting of the L2 prefetch hint (qsa_decode_step_prefetch)
        dl.prefetch = not args.prefetch
        g_alt = capture(dl.step, stream)
        t_alt = time_graph(g_alt, stream, args.steps, args.warmup, world)
        dl.prefetch = args.prefetch
        del g_alt
        us_alt = 1e6 * t_alt / (args.steps * n_layers)
        line["with_l2_prefetch" if not args.prefetch else "without_l2_prefetch"] = {
            "layer_steps_per_s": 1e6 / us_alt, "us_per_layer_step": us_alt,
            "hbm_gbs_algorithmic": bytes_ls / (us_alt * 1e-6) / 1e9,
            "frac": bytes_ls / (us_alt * 1e-6) / 1e9 / pk["hbm"],
            "note": "each layer-step prefetches the next layer's pooled keys into L2 during its exchanges"}
    if dl.fused:
        # The step graph holds only the 12 fused launches, back to back (each a programmatic
        # dependent of the previous one), so a launch's share of the step time is its duration
        # as it runs in the step: step time / layers.
        us_k = 1e6 * t / (args.steps * n_layers)
        ach = bytes_ls / (us_k * 1e-6) / 1e9
        line["roofline"] = {"bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s",
                            "frac": ach / pk["hbm"], "traffic": recorded_traffic("decode_step"),
                            "kernel": "decode_step", "algorithmic_bytes": bytes_ls, "us_per_launch": us_k,
                            "timing": "graph of 12 fused launches; step time / 12 (CUDA events on the stream)",
                            "peak_src": pk["src"]}
    if not args.no_instrument:
        # event nodes between the launches serialise them (no programmatic dependent launch
        # overlap), so these per-launch times are upper bounds, reported for the phase split only
        kt = instrumented_kernel_times(dl, stream, max(5, min(50, args.steps)))
        line["kernel_us_event_nodes"] = kt
        if not dl.fused:
            algo = {"score": A.score_scan_bytes(dl.w.ctx_len)}
            ach = algo["score"] / (kt["score"] * 1e-6) / 1e9
            line["roofline"] = {"bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s",
                                "frac": ach / pk["hbm"], "traffic": None, "kernel": "score",
                                "note": "separate calls: the score scan", "peak_src": pk["src"]}

    if not args.no_e2e:
        dt, h2d, d2h = e2e_decode(dl, stream, max(10, args.steps // 4), max(3, args.warmup))
        n = max(10, args.steps // 4)
        line["e2e"] = {"value": n * n_layers / dt * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h}

    if not args.no_kv_host:
        line["decode_kv_in_host_memory"] = kv_host_bench(dl, stream, max(20, args.steps // 4), max(3, args.warmup))

    if not args.no_fp8:
        line["decode_fp8_indexer_keys"] = fp8_keys_bench(dl, stream, max(20, args.steps // 4), max(3, args.warmup),
                                                         pk)

    if not args.no_fp8:
        line["decode_fp8_kv"] = fp8_kv_bench(dl, stream, max(20, args.steps // 4), max(3, args.warmup), pk)

    if not args.no_mla:
        line["sparse_mla_decode"] = mla_bench(args.steps, args.warmup, pk)

    if not args.no_prefill:
        del g
        line["prefill"] = prefill_bench(args.steps, args.warmup, pk)

    if not args.no_configs:
        del dl
        torch.cuda.empty_cache()
        line["decode_configs"] = config_legs(pk, max(20, args.steps // 4), max(3, args.warmup))

    if cpu_base is not None:
        line["cpu_baseline"] = cpu_base
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
