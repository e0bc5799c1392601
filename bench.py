"""Benchmark: paged mixed-codec decode attention on one GB300.

Default workload (the mixed-tier decode the metric is quoted on): batch 1, 24
layers, 14 query / 2 KV heads, head_dim 64, a 16,384-token context in 1024-token
pages -- newest 4 pages FP16, next 4 FP8 e4m3 (fp32 scale per page and KV
head), next 4 INT8, oldest 4 INT4 group-32 -- K/V ~ N(0,1) with 1% of elements
x8.  One step = one decoded token through all 24 layers: 24 calls of
argus_paged_decode_attn replayed as one CUDA graph; L2 is flushed (a 2 x L2
write) before every timed step, outside the timed region.

Printed value: decode attention microseconds per token per layer (lower is
better), plus the effective KV bandwidth against the HBM roofline.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--no-legs]

The same line also carries "legs": the other four workloads (tiny FP16 decode,
batched BF16/FP8 decode and demotion, sparse selected-page decode, windowed
prefill), each timed with L2 flushed and reported against its roofline.

--impl reference times the CPU oracle (double precision, one process per host
core) on a bounded sample of the same workload.  Under torchrun every rank
runs an independent replica (the path has no exchange step); rank 0 prints.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn µs/token/layer & effective KV GB/s (% of GB300 HBM peak)"
WORKLOAD = ("mixed_tier_decode: batch 1, 24 layers, 14 q / 2 kv heads, head_dim 64, 16384 tokens in "
            "1024-token pages (4 FP16 newest, 4 FP8 e4m3, 4 INT8, 4 INT4 g32 oldest), N(0,1) with 1% x8")
LAYERS, HQ, HKV, D, P, NPAGES = 24, 14, 2, 64, 1024, 16
CTX = NPAGES * P


def kv_bytes_per_layer():
    from mixed_precision_paged_argus_gb300 import accounting as A
    tiers = [A.FP16, A.FP8_E4M3, A.INT8, A.INT4_G32]
    return sum(A.kv_bytes(c, 4 * P, HKV, D, 4) for c in tiers)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "mixed_precision_paged_argus_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key, src_files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel_key]
        if t.get("source_hash") == source_hash(src_files):
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------- clocks

class NvmlClockSampler:
    """Samples the SM clock, its maximum, power and the clock-event reasons
    through NVML (read-only queries) from a background thread about every
    0.5 ms, so that even a timed region of a few milliseconds is covered."""
    REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
               (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))

    def __init__(self, dev_index):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                self.lib = ctypes.CDLL(name)
                break
            except OSError:
                pass
        if self.lib is None or self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("NVML unavailable")
        self.handle = ctypes.c_void_p()
        ok = False
        try:
            import torch
            pr = torch.cuda.get_device_properties(dev_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle)) == 0
        except Exception:
            ok = False
        if not ok:
            idx = dev_index
            cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [x for x in cvd.split(",") if x.strip()]
            if parts and all(x.strip().isdigit() for x in parts) and dev_index < len(parts):
                idx = int(parts[dev_index])
            if self.lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.handle)) != 0:
                raise RuntimeError("NVML: no handle for device %d" % idx)
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.stop_evt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        ct = self.ct
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(sm)) != 0:
            return
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        self.reasons_fn(self.handle, ct.byref(rs))
        self.samples.append((sm.value, mx.value, mw.value / 1000.0, rs.value))

    def _run(self):
        while not self.stop_evt.is_set():
            self._sample()
            time.sleep(0.0005)

    def start(self):
        self._sample()
        self.thread.start()

    def stop(self):
        self.stop_evt.set()
        self.thread.join(timeout=5)
        self._sample()
        rows = self.samples
        if not rows:
            return None
        reasons = sorted({name for r in rows for bit, name in self.REASONS if r[3] & bit})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_median": statistics.median(r[2] for r in rows),
                "source": "nvml, ~0.5 ms sampling during the timed steps"}


class SmiClockSampler:
    """Fallback: nvidia-smi in a loop (200 ms); covers long timed regions only."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi -lms 200"}


def ClockSampler(dev_index):
    try:
        return NvmlClockSampler(dev_index)
    except Exception:
        return SmiClockSampler(dev_index)


# ---------------------------------------------------------------- workload

def max_over_ranks(value, world, dev):
    """The largest of every rank's value (the slowest replica sets the time),
    followed by a barrier; the value itself when there is one rank."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


def aggregate_us_per_token_layer(ms_step, world):
    """Whole-job rate for N independent replicas: every rank decodes one token
    through all layers per step, so the job finishes world * LAYERS
    token-layers per (max-over-ranks) step."""
    return ms_step * 1000.0 / (LAYERS * max(1, world))


def build_mixed_tier(dev):
    """Device pools for all 24 layers (one pool per codec, 4 slots per layer),
    per-layer block tables and queries.  Setup only: quantisation by the
    library's own kernel, not timed."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W
    g = argus.geom(HQ, HKV, D, P)
    tiers = W.mixed_tier_codecs(NPAGES)
    pools = {c: argus.Pool.empty(c, 4 * LAYERS, HKV, P, D, device=dev, zero=True)
             for c in (W.FP16, W.FP8_E4M3, W.INT8, W.INT4_G32)}
    tables, qs = [], []
    for layer in range(LAYERS):
        src = W.normal((NPAGES, 2, HKV, P, D), W.FP16, W.seed_of("mixed_tier", layer, 1), device=dev,
                       outlier_seed=W.seed_of("mixed_tier", layer, 5))
        perm = W.permutation(4, W.seed_of("mixed_tier", layer, 4))
        table = np.zeros(NPAGES, np.int32)
        for codec, pool in pools.items():
            pages = [p for p in range(NPAGES) if tiers[p] == codec]
            slots = [4 * layer + int(perm[i]) for i in range(4)]
            argus.quantize_pages(g, W.FP16, src, NPAGES, torch.tensor(pages, dtype=torch.int32, device=dev),
                                 pool, torch.tensor(slots, dtype=torch.int32, device=dev), len(pages))
            table[pages] = slots
        tables.append(torch.from_numpy(table.reshape(1, NPAGES)).to(dev))
        qs.append(W.normal((1, HQ, D), W.FP16, W.seed_of("mixed_tier", layer, 0), device=dev))
        del src
    torch.cuda.synchronize()
    codec_row = torch.from_numpy(tiers.reshape(1, NPAGES).astype(np.uint8)).to(dev)
    lens = torch.tensor([CTX], dtype=torch.int32, device=dev)
    return g, [pools[c] for c in sorted(pools)], tables, qs, codec_row, lens


def run_gpu(args, rank, world):
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    argus.lib()
    g, pools, tables, qs, codec_row, lens = build_mixed_tier(dev)
    scale = W.softmax_scale(D)
    outs = [torch.empty((1, HQ, D), dtype=torch.float16, device=dev) for _ in range(LAYERS)]
    # layer after layer: no call writes another's inputs, so each decode grid
    # may start during its predecessor's tail (programmatic dependent launch)
    arg_list = [argus.decode_args(g, 1, qs[l], pools, codec_row, tables[l], lens, NPAGES, scale, out=outs[l],
                                  pdl=True) for l in range(LAYERS)]
    ws_bytes = max(argus.decode_workspace_bytes(a) for a in arg_list)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)

    def step_layers():
        for a in arg_list:
            argus.paged_decode_attn(a, ws, ws_bytes, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step_layers()                       # first calls set kernel attributes (outside capture)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step_layers()
    torch.cuda.synchronize()

    def timed(n, fn):
        times = []
        for _ in range(n):
            with torch.cuda.stream(stream):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return times

    timed(args.warmup, graph.replay)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_wall0 = time.perf_counter()
    times = timed(args.steps, graph.replay)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    torch.cuda.synchronize()
    ms_step = max_over_ranks(sum(times) / len(times), world, dev)

    # ---- end to end through the public API with host buffers
    q_host = torch.empty((LAYERS, 1, HQ, D), dtype=torch.float16).pin_memory()
    for l in range(LAYERS):
        q_host[l].copy_(qs[l].cpu())
    out_host = torch.empty((LAYERS, 1, HQ, D), dtype=torch.float16).pin_memory()
    q_dev = torch.empty((LAYERS, 1, HQ, D), dtype=torch.float16, device=dev)
    out_dev = torch.empty((LAYERS, 1, HQ, D), dtype=torch.float16, device=dev)
    e2e_args = [argus.decode_args(g, 1, q_dev[l], pools, codec_row, tables[l], lens, NPAGES, scale,
                                  out=out_dev[l], pdl=True) for l in range(LAYERS)]

    def e2e_step():
        q_dev.copy_(q_host, non_blocking=True)
        for a in e2e_args:
            argus.paged_decode_attn(a, ws, ws_bytes, stream=stream)
        out_host.copy_(out_dev, non_blocking=True)

    timed(args.warmup, e2e_step)
    e2e_times = timed(args.steps, e2e_step)
    ms_e2e = max_over_ranks(sum(e2e_times) / len(e2e_times), world, dev)
    return ms_step, ms_e2e, clocks, t_wall, q_host.numel() * 2, out_host.numel() * 2


# ---------------------------------------------------------------- other workloads
# Each leg builds one of the other four synthetic workloads on the device, times
# it as a CUDA graph with L2 flushed before every timed replay, and reports
# absolute numbers plus the fraction of the roofline.  Legs never change the
# headline value above.

class Timer:
    def __init__(self, dev):
        import torch
        self.torch = torch
        self.stream = torch.cuda.Stream(device=dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)

    def graph(self, fn):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            fn()
            fn()
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        torch.cuda.synchronize()
        return g

    def time(self, replay, n, warm):
        torch = self.torch
        out = []
        for i in range(warm + n):
            with torch.cuda.stream(self.stream):
                self.flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                replay()
                e1.record(self.stream)
            e1.synchronize()
            if i >= warm:
                out.append(e0.elapsed_time(e1))
        return sum(out) / len(out)


def leg_tiny(dev, timer, steps, warm, hbm):
    """Batch 1, 1 layer, 14 q / 2 KV heads, head_dim 64, 4 FP16 pages of 1024."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W, accounting as A
    Hq, Hkv, D_, P_ = 14, 2, 64, 1024
    g = argus.geom(Hq, Hkv, D_, P_)
    pool = argus.Pool(W.FP16, W.normal((4, 2, Hkv, P_, D_), W.FP16, W.seed_of("tiny_fp16", 0, 1), device=dev),
                      None, 4)
    q = W.normal((1, Hq, D_), W.FP16, W.seed_of("tiny_fp16", 0, 0), device=dev)
    out = torch.empty((1, Hq, D_), dtype=torch.float16, device=dev)
    a = argus.decode_args(g, 1, q, [pool], torch.zeros((1, 4), dtype=torch.uint8, device=dev),
                          torch.arange(4, dtype=torch.int32, device=dev).reshape(1, 4),
                          torch.tensor([4096], dtype=torch.int32, device=dev), 4, W.softmax_scale(D_), out=out)
    ws = torch.empty(max(1, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)
    gr = timer.graph(lambda: argus.paged_decode_attn(a, ws, stream=timer.stream))
    ms = timer.time(gr.replay, steps, warm)
    nbytes = A.kv_bytes(A.FP16, 4096, Hkv, D_, 4) + 2 * Hq * D_ * 2
    return {"workload": "tiny_fp16_decode: batch 1, 14 q / 2 kv, head_dim 64, 4 x 1024-token FP16 pages",
            "us_per_step": ms * 1e3, "us_per_token_layer": ms * 1e3, "bytes": nbytes,
            "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "note": "2 MiB per step: launch-latency bound, the HBM fraction is not meaningful"}


def leg_batched(dev, timer, steps, warm, hbm):
    """Batch 32, 32 q / 8 KV heads, head_dim 128, 16-token pages, lengths
    U[8192, 32768], random physical slots; demotion of the BF16 pages to FP8 /
    INT8 / INT4 / INT2 / INT1, and BF16, FP8, INT2 and INT1 decode (each also
    under a 4096-token window with 4 sink tokens)."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W, accounting as A
    B, Hq, Hkv, D_, P_, MAXP = 32, 32, 8, 128, 16, 2048
    lens = W.uniform_ints(B, 8192, 32768, W.seed_of("batched", 0, 3))
    table, n_slots = W.paged_block_table(lens, P_, MAXP, W.seed_of("batched", 0, 4))
    g = argus.geom(Hq, Hkv, D_, P_)
    bf = argus.Pool(W.BF16, W.normal((n_slots, 2, Hkv, P_, D_), W.BF16, W.seed_of("batched", 0, 1), device=dev),
                    None, n_slots)
    q = W.normal((B, Hq, D_), W.BF16, W.seed_of("batched", 0, 0), device=dev)
    d_table = torch.from_numpy(table).to(dev)
    d_lens = torch.from_numpy(lens.astype(np.int32)).to(dev)
    ids = torch.arange(n_slots, dtype=torch.int32, device=dev)
    res = {"workload": "batched_decode: batch 32, 32 q / 8 kv, head_dim 128, 16-token pages, lengths U[8192,32768] "
                       "(sum %d tokens), slots a random permutation" % int(lens.sum())}
    tokens = int(lens.sum())
    pages = int(sum((L + P_ - 1) // P_ for L in lens))
    # demotion of every BF16 page
    for name, codec in (("fp8", W.FP8_E4M3), ("int8", W.INT8), ("int4", W.INT4_G32), ("int2", W.INT2_G32),
                        ("int1", W.INT1_G32)):
        dst = argus.Pool.empty(codec, n_slots, Hkv, P_, D_, device=dev)
        gr = timer.graph(lambda: argus.quantize_pages(g, W.BF16, bf.codes, n_slots, ids, dst, ids, n_slots,
                                                      stream=timer.stream))
        ms = timer.time(gr.replay, max(3, steps // 5), warm)
        nb = A.quantize_bytes(codec, 2, n_slots * 2 * Hkv, P_, D_)
        res["quantize_" + name] = {"us": ms * 1e3, "bytes": nb, "gbs": nb / (ms * 1e-3) / 1e9,
                                   "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm}
        if codec == W.FP8_E4M3:
            fp8 = dst
        elif codec == W.INT2_G32:
            int2 = dst
        elif codec == W.INT1_G32:
            int1 = dst
        else:
            del dst
        torch.cuda.synchronize()
    for name, pool, codec in (("bf16", bf, W.BF16), ("fp8", fp8, W.FP8_E4M3), ("int2", int2, W.INT2_G32),
                              ("int1", int1, W.INT1_G32)):
        out = torch.empty((B, Hq, D_), dtype=torch.bfloat16, device=dev)
        d_codec = torch.full((B, MAXP), codec, dtype=torch.uint8, device=dev)
        a = argus.decode_args(g, B, q, [pool], d_codec, d_table, d_lens, MAXP, W.softmax_scale(D_), out=out)
        ws = torch.empty(max(1, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)
        gr = timer.graph(lambda: argus.paged_decode_attn(a, ws, stream=timer.stream))
        ms = timer.time(gr.replay, steps, warm)
        nb = A.kv_bytes(codec, tokens, Hkv, D_, pages) + 2 * B * Hq * D_ * 2
        res["decode_" + name] = {"us_per_step": ms * 1e3, "us_per_token_layer": ms * 1e3 / B, "bytes": nb,
                                 "gbs": nb / (ms * 1e-3) / 1e9, "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm}
        # the same rows under a sliding window of the newest 4096 tokens plus 4 sink tokens
        WIN, SINK = 4096, 4
        aw = argus.decode_args(g, B, q, [pool], d_codec, d_table, d_lens, MAXP, W.softmax_scale(D_), out=out,
                               window_tokens=WIN, sink_tokens=SINK)
        wsw = torch.empty(max(1, argus.decode_workspace_bytes(aw)), dtype=torch.uint8, device=dev)
        gr = timer.graph(lambda: argus.paged_decode_attn(aw, wsw, stream=timer.stream))
        ms = timer.time(gr.replay, steps, warm)
        vis = [A.window_visible(L, P_, WIN, SINK) for L in lens]
        nb = A.kv_bytes(codec, sum(t for t, _ in vis), Hkv, D_, sum(n for _, n in vis)) + 2 * B * Hq * D_ * 2
        res["decode_%s_window" % name] = {"window": WIN, "sinks": SINK, "us_per_step": ms * 1e3,
                                          "bytes": nb, "gbs": nb / (ms * 1e-3) / 1e9,
                                          "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm}
    del bf, fp8, int2, int1
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def leg_sparse(dev, timer, steps, warm, hbm):
    """Batch 8, 12 layers, 32 q / 4 KV heads, head_dim 128, 262144 tokens in
    64-token FP8 pages with bf16 compressed keys; per layer the indexer picks
    the top 32 pages plus the newest one per KV head, then decode reads only
    those."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W, accounting as A
    B, L_, Hq, Hkv, D_, P_, NP, K_ = 8, 12, 32, 4, 128, 64, 4096, 32
    width = 2 * K_ + 8
    g = argus.geom(Hq, Hkv, D_, P_)
    pools, ckeys, qs = [], [], []
    ids = torch.arange(NP, dtype=torch.int32, device=dev)
    for layer in range(L_):
        pool = argus.Pool.empty(W.FP8_E4M3, B * NP, Hkv, P_, D_, device=dev)
        ck = torch.empty((B, NP, Hkv, D_), dtype=torch.bfloat16, device=dev)
        for b in range(B):
            src = W.normal((NP, 2, Hkv, P_, D_), W.BF16, W.seed_of("sparse", layer, 1) * 16 + b, device=dev)
            argus.quantize_pages(g, W.BF16, src, NP, ids, pool, ids + b * NP, NP, ckey_out=ck[b])
            del src
        pools.append(pool)
        ckeys.append(ck)
        qs.append(W.normal((B, Hq, D_), W.BF16, W.seed_of("sparse", layer, 0), device=dev))
    torch.cuda.synchronize()
    table = (torch.arange(B * NP, dtype=torch.int32, device=dev)).reshape(B, NP)
    codec = torch.full((B, NP), W.FP8_E4M3, dtype=torch.uint8, device=dev)
    lens = torch.full((B,), NP * P_, dtype=torch.int32, device=dev)
    npages = torch.full((B,), NP, dtype=torch.int32, device=dev)
    sel = torch.empty((B, Hkv, width), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    drops = torch.zeros(1, dtype=torch.int32, device=dev)
    sws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=dev)
    outs = [torch.empty((B, Hq, D_), dtype=torch.bfloat16, device=dev) for _ in range(L_)]
    # pdl=2: each decode grid starts during the select's tail and reads the
    # selection after it completes
    args = [argus.decode_args(g, B, qs[l], [pools[l]], codec, table, lens, NP, W.softmax_scale(D_), out=outs[l],
                              sel_pages=sel, sel_count=cnt, sel_width=width, pdl=2) for l in range(L_)]
    dws = torch.empty(max(argus.decode_workspace_bytes(a) for a in args), dtype=torch.uint8, device=dev)

    def step(select=True, decode=True):
        for l in range(L_):
            if select:
                argus.select_pages(g, B, qs[l], ckeys[l], npages, NP, K_, True, sel, cnt, width, drops, sws,
                                   stream=timer.stream)
            if decode:
                argus.paged_decode_attn(args[l], dws, stream=timer.stream)

    ms = timer.time(timer.graph(step).replay, steps, warm)
    ms_sel = timer.time(timer.graph(lambda: step(decode=False)).replay, steps, warm)
    ms_dec = timer.time(timer.graph(lambda: step(select=False)).replay, steps, warm)
    slab = B * NP * Hkv * D_ * 2
    sel_bytes = B * Hkv * (K_ + 1) * (2 * P_ * D_ + 8)
    per_layer = slab + sel_bytes + 2 * B * Hq * D_ * 2
    nb = L_ * per_layer
    res = {"workload": "sparse_decode: batch 8, 12 layers, 32 q / 4 kv, head_dim 128, 262144 tokens in 64-token "
                       "FP8 pages, top-32 + newest page per kv head",
           "us_per_step": ms * 1e3, "us_per_step_layer": ms * 1e3 / L_, "bytes_per_step": nb,
           "gbs": nb / (ms * 1e-3) / 1e9, "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm,
           "select_us_per_step": ms_sel * 1e3, "select_gbs": L_ * slab / (ms_sel * 1e-3) / 1e9,
           "decode_us_per_step": ms_dec * 1e3, "decode_gbs": L_ * sel_bytes / (ms_dec * 1e-3) / 1e9,
           "drops": int(drops.item())}
    del pools, ckeys
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def leg_sparse_host(dev, timer, steps, warm, hbm):
    """One layer of the sparse selected-page decode with its FP8 pool in
    page-locked host memory (the host-RAM tier): batch 8, 32 q / 4 KV heads,
    head_dim 128, 4096 64-token pages per sequence; the indexer scores the
    device-resident compressed keys, decode reads the 33 selected pages per KV
    head in place over the host link."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W
    B, Hq, Hkv, D_, P_, NP, K_ = 8, 32, 4, 128, 64, 4096, 32
    width = 2 * K_ + 8
    g = argus.geom(Hq, Hkv, D_, P_)
    ids = torch.arange(NP, dtype=torch.int32, device=dev)
    pool = argus.Pool.empty(W.FP8_E4M3, B * NP, Hkv, P_, D_, device=dev)
    ck = torch.empty((B, NP, Hkv, D_), dtype=torch.bfloat16, device=dev)
    for b in range(B):
        src = W.normal((NP, 2, Hkv, P_, D_), W.BF16, W.seed_of("sparse", 0, 1) * 16 + b, device=dev)
        argus.quantize_pages(g, W.BF16, src, NP, ids, pool, ids + b * NP, NP, ckey_out=ck[b])
        del src
    q = W.normal((B, Hq, D_), W.BF16, W.seed_of("sparse", 0, 0), device=dev)
    torch.cuda.synchronize()
    host = pool.to_host()
    del pool
    torch.cuda.empty_cache()
    table = torch.arange(B * NP, dtype=torch.int32, device=dev).reshape(B, NP)
    codec = torch.full((B, NP), W.FP8_E4M3, dtype=torch.uint8, device=dev)
    lens = torch.full((B,), NP * P_, dtype=torch.int32, device=dev)
    npages = torch.full((B,), NP, dtype=torch.int32, device=dev)
    sel = torch.empty((B, Hkv, width), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    drops = torch.zeros(1, dtype=torch.int32, device=dev)
    sws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D_), dtype=torch.bfloat16, device=dev)
    a = argus.decode_args(g, B, q, [host], codec, table, lens, NP, W.softmax_scale(D_), out=out, sel_pages=sel,
                          sel_count=cnt, sel_width=width, pdl=2)
    dws = torch.zeros(max(16, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)

    def select():
        argus.select_pages(g, B, q, ck, npages, NP, K_, True, sel, cnt, width, drops, sws, stream=timer.stream)

    def decode():
        argus.paged_decode_attn(a, dws, stream=timer.stream)

    select()
    torch.cuda.synchronize()
    ms_dec = timer.time(timer.graph(decode).replay, steps, warm)
    ms_all = timer.time(timer.graph(lambda: (select(), decode())).replay, steps, warm)
    host_bytes = B * Hkv * (K_ + 1) * (2 * P_ * D_ + 8)
    res = {"workload": "sparse_decode_host_pool: one layer of the sparse workload (batch 8, 32 q / 4 kv, head_dim 128, "
                       "4096 x 64-token FP8 pages per sequence) with the FP8 pool in page-locked host memory",
           "decode_us_per_layer": ms_dec * 1e3, "select_plus_decode_us_per_layer": ms_all * 1e3,
           "host_bytes_per_layer": host_bytes, "host_gbs": host_bytes / (ms_dec * 1e-3) / 1e9,
           "context": "the pages report 166 us per layer for in-place host reads over PCIe 4.0 x16 on an RTX 3090 Ti "
                      "(another machine: context only)"}
    del host, ck
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def leg_prefill(dev, timer, steps, warm, tflops_peak):
    """16 q / 2 KV heads, head_dim 128, 1048576 cached BF16 tokens and a
    1024-token causal chunk; eight 131072-token windows plus the chunk window,
    folded by log2-sum-exp into an fp32 accumulator."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W, accounting as A
    Hq, Hkv, D_, NQ, CTX, WIN = 16, 2, 128, 1024, 1 << 20, 131072
    kv_len = CTX + NQ
    q = W.normal((Hq, NQ, D_), W.BF16, W.seed_of("prefill", 0, 0), device=dev)
    k = W.normal((Hkv, kv_len, D_), W.BF16, W.seed_of("prefill", 0, 1), device=dev)
    v = W.normal((Hkv, kv_len, D_), W.BF16, W.seed_of("prefill", 0, 2), device=dev)
    g = argus.geom(Hq, Hkv, D_, 16)
    acc_o = torch.empty((Hq, NQ, D_), dtype=torch.float32, device=dev)
    acc_l = torch.empty((Hq, NQ), dtype=torch.float32, device=dev)
    wins = [(w, w + WIN) for w in range(0, CTX, WIN)] + [(CTX, CTX + NQ)]
    ws = torch.empty(max(16, max(argus.window_prefill_workspace_bytes(g, NQ, w1 - w0) for w0, w1 in wins)),
                     dtype=torch.uint8, device=dev)

    def run():
        for i, (w0, w1) in enumerate(wins):
            argus.window_prefill_attn(g, NQ, q, k[:, w0:], v[:, w0:], kv_len * D_, w1 - w0, w0, CTX,
                                      W.softmax_scale(D_), acc_o, acc_l, 1 if i else 0, ws=ws,
                                      stream=timer.stream)

    ms = timer.time(timer.graph(run).replay, max(3, steps // 10), warm)
    flops = A.prefill_flops(Hq, D_, NQ, NQ * CTX + NQ * (NQ + 1) // 2)
    res = {"workload": "windowed_prefill: 16 q / 2 kv, head_dim 128, 1048576 cached bf16 tokens + 1024-token "
                       "causal chunk, 131072-token windows folded by log2-sum-exp",
           "ms": ms, "flops": flops, "tflops": flops / (ms * 1e-3) / 1e12,
           "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / tflops_peak,
           "splits": (argus.window_prefill_workspace_bytes(g, NQ, WIN) - Hkv * WIN * D_ * 2 - 16)
                     // (Hq * NQ * (D_ + 1) * 4),
           "note": "useful FLOPs 4*D*Hq*visible pairs; Q.K^T in bf16, P.V in fp16 (P * 2^7, V converted per "
                   "window to fp16 scaled by a power of two); each 128-row query tile's window split into key "
                   "ranges over all SMs, partials folded"}
    del q, k, v
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def leg_prefill_paged(dev, timer, steps, warm, tflops_peak):
    """The windowed prefill over a paged, mixed-codec cache: the same 16 q / 2 KV
    heads, head_dim 128, 1048576 cached tokens, now in 64-token FP8 e4m3 pages
    at random physical slots, with the 1024-token chunk in BF16 pages; each of
    the eight 131072-token windows and the chunk window is staged through the
    block table (dequantised to scaled fp16) and attended with fp16 MMAs, folded
    by log2-sum-exp.  Timed: staging and attention of all nine windows."""
    import torch
    import mixed_precision_paged_argus_gb300.argus as argus
    from mixed_precision_paged_argus_gb300 import workloads as W, accounting as A
    Hq, Hkv, D_, NQ, CTX, WIN, P_ = 16, 2, 128, 1024, 1 << 20, 131072, 64
    n_cache, n_chunk = CTX // P_, NQ // P_
    n_pages = n_cache + n_chunk
    g = argus.geom(Hq, Hkv, D_, P_)
    perm = W.permutation(n_cache, W.seed_of("prefill", 0, 4))
    fp8 = argus.Pool.empty(W.FP8_E4M3, n_cache, Hkv, P_, D_, device=dev)
    bf = argus.Pool.empty(W.BF16, n_chunk, Hkv, P_, D_, device=dev)
    step_pages = 4096                                  # demote the cache in pieces (bounded source buffer)
    for p0 in range(0, n_cache, step_pages):
        n = min(step_pages, n_cache - p0)
        src = W.normal((n, 2, Hkv, P_, D_), W.BF16, W.seed_of("prefill", 0, 1) * 64 + p0 // step_pages, device=dev)
        argus.quantize_pages(g, W.BF16, src, n, torch.arange(n, dtype=torch.int32, device=dev), fp8,
                             torch.from_numpy(perm[p0:p0 + n].astype(np.int32)).to(dev), n)
        del src
    src = W.normal((n_chunk, 2, Hkv, P_, D_), W.BF16, W.seed_of("prefill", 0, 3), device=dev)
    ids = torch.arange(n_chunk, dtype=torch.int32, device=dev)
    argus.quantize_pages(g, W.BF16, src, n_chunk, ids, bf, ids, n_chunk)
    del src
    table = torch.from_numpy(np.concatenate([perm, np.arange(n_chunk)]).astype(np.int32)).to(dev)
    codecs = torch.from_numpy(np.array([W.FP8_E4M3] * n_cache + [W.BF16] * n_chunk, np.uint8)).to(dev)
    q = W.normal((Hq, NQ, D_), W.BF16, W.seed_of("prefill", 0, 0), device=dev)
    acc_o = torch.empty((Hq, NQ, D_), dtype=torch.float32, device=dev)
    acc_l = torch.empty((Hq, NQ), dtype=torch.float32, device=dev)
    wins = [(w, WIN) for w in range(0, CTX, WIN)] + [(CTX, NQ)]
    ws = torch.empty(max(argus.paged_window_prefill_workspace_bytes(g, NQ, wl) for _, wl in wins), dtype=torch.uint8,
                     device=dev)
    # the staging decision: each query row would read every visible page in place
    tok_fp8 = 2 * Hkv * D_                              # bytes per cached token (K + V codes), FP8 pages
    cache_bytes = int(n_cache * (2 * Hkv * P_ * D_ + 2 * Hkv * 4) + n_chunk * 2 * Hkv * P_ * D_ * 2)
    rows = [int(CTX * tok_fp8 + (i + 1) * 2 * Hkv * D_ * 2) for i in range(NQ)]
    stage = argus.staging_moves_less(rows, cache_bytes)

    def run():
        for i, (w0, wl) in enumerate(wins):
            argus.paged_window_prefill_attn(g, NQ, q, [fp8, bf], codecs, table, n_pages, w0, wl, CTX,
                                            W.softmax_scale(D_), acc_o, acc_l, 1 if i else 0, ws, stream=timer.stream)

    ms = timer.time(timer.graph(run).replay, max(3, steps // 10), warm)
    flops = A.prefill_flops(Hq, D_, NQ, NQ * CTX + NQ * (NQ + 1) // 2)
    res = {"workload": "paged_windowed_prefill: 16 q / 2 kv, head_dim 128, 1048576 cached tokens in 64-token FP8 e4m3 "
                       "pages (random slots) + 1024-token chunk in BF16 pages, 131072-token windows staged through "
                       "the block table and folded by log2-sum-exp",
           "ms": ms, "flops": flops, "tflops": flops / (ms * 1e-3) / 1e12,
           "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / tflops_peak,
           "staging_moves_less": stage, "rows_read_in_place_bytes": sum(rows), "cache_bytes": cache_bytes,
           "note": "timed: per window, dequantise + scale to fp16 (two passes over the window's codes), query to "
                   "fp16, then Q.K^T and P.V in fp16 on tcgen05 (same FLOP count as the BF16 leg); fp16 dense peak "
                   "= bf16 dense peak"}
    del fp8, bf, q, ws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_legs(steps, warm):
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    timer = Timer(dev)
    hbm, tf, _ = peaks()
    out = {}
    for name, fn, arg in (("tiny_fp16", leg_tiny, hbm), ("batched", leg_batched, hbm),
                          ("sparse", leg_sparse, hbm), ("sparse_host", leg_sparse_host, hbm),
                          ("prefill", leg_prefill, tf),
                          ("prefill_paged_fp8", leg_prefill_paged, tf)):
        t0 = time.perf_counter()
        try:
            out[name] = fn(dev, timer, steps, warm, arg)
        except Exception as e:  # a leg failure is reported, never hidden
            out[name] = {"error": "%s: %s" % (type(e).__name__, e)}
        out[name]["wall_s"] = time.perf_counter() - t0
    return out


# ---------------------------------------------------------------- oracle leg

def _oracle_layer(job):
    """One layer of the mixed-tier workload in the oracle: generate, demote
    (oracle), then decode it `reps` times.  Returns (seconds of decode, reps)."""
    layer, reps = job
    import oracle
    from oracle import codecs as C
    from mixed_precision_paged_argus_gb300 import workloads as W
    tiers = W.mixed_tier_codecs(NPAGES)
    src = W.to_bits(W.normal((NPAGES, 2, HKV, P, D), W.FP16, W.seed_of("mixed_tier", layer, 1),
                             outlier_seed=W.seed_of("mixed_tier", layer, 5)))
    q64 = C.f16_bits_to_f64(W.to_bits(W.normal((1, HQ, D), W.FP16, W.seed_of("mixed_tier", layer, 0))))
    pools, table = {}, np.zeros((1, NPAGES), np.int32)
    for codec in (0, 2, 3, 4):
        pages = [p for p in range(NPAGES) if tiers[p] == codec]
        codes, meta = C.alloc_pool(codec, 4, HKV, P, D)
        C.quantize_pages(src, C.CODEC_FP16, pages, codec, codes, meta, [0, 1, 2, 3])
        pools[codec] = (codes, meta)
        table[0, pages] = [0, 1, 2, 3]
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_decode(q64, HKV, P, pools, tiers.reshape(1, -1).astype(np.uint8), table,
                            np.array([CTX]), float(np.float32(1 / math.sqrt(D))))
    return time.perf_counter() - t0, reps


def oracle_leg(budget_s=15.0):
    """Oracle throughput on the host cores: one process per core (spawn), each
    demoting one layer and then decoding it repeatedly for about budget_s / 2
    seconds; the rate is the decodes of all processes over the summed time."""
    import multiprocessing as mp
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    cores = os.cpu_count() or 1
    t_one, _ = _oracle_layer((0, 1))               # calibrate (also warms imports)
    reps = max(1, int(budget_s / 2 / max(t_one, 1e-3)))
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_layer, [(l % LAYERS, reps) for l in range(cores)])
    wall = time.perf_counter() - t0
    n = sum(r for _, r in res)
    per_layer = sum(t for t, _ in res) / n          # decode seconds per layer-decode on one core
    us_per_token_layer = per_layer / cores * 1e6
    return {"value": us_per_token_layer, "unit": "us/token/layer", "cores": cores, "kind": "oracle",
            "sample": "%d layer-decodes of the mixed-tier workload (one token, 16384-token context each; %d "
                      "layers x %d repeats) on %d processes; decode time only, %.1f s wall incl. oracle "
                      "demotion" % (n, cores, reps, cores, wall),
            "single_core_us_per_token_layer": per_layer * 1e6}


# ---------------------------------------------------------------- oracle per leg
# The oracle (float64, plain numpy) timed on the host cores for each of the
# other workloads, as a reported baseline beside the GPU legs.  Every job builds
# its own seeded inputs of the workload's shape on the CPU; only the steps the
# GPU leg times are timed (demotion of the pools is set-up, not part of a
# decode step).  Jobs are top-level functions for a spawned process pool.

def _cpu_tiny(reps):
    """Single-threaded: the tiny FP16 decode, `reps` times."""
    import oracle
    from oracle import codecs as C
    from mixed_precision_paged_argus_gb300 import workloads as W
    Hq, Hkv, D_, P_ = 14, 2, 64, 1024
    src = W.to_bits(W.normal((4, 2, Hkv, P_, D_), W.FP16, W.seed_of("tiny_fp16", 0, 1)))
    q64 = C.f16_bits_to_f64(W.to_bits(W.normal((1, Hq, D_), W.FP16, W.seed_of("tiny_fp16", 0, 0))))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_decode(q64, Hkv, P_, {0: (src, None)}, np.zeros((1, 4), np.uint8),
                            np.arange(4, dtype=np.int32)[None], np.array([4096]), W.softmax_scale(D_))
    return (time.perf_counter() - t0) / reps


def _cpu_batched_row(job):
    """One sequence of the batched workload (BF16 pages, or demoted to FP8
    first, untimed): seconds of the oracle's decode of that row."""
    b, codec = job
    import oracle
    from oracle import codecs as C
    from mixed_precision_paged_argus_gb300 import workloads as W
    Hq, Hkv, D_, P_ = 32, 8, 128, 16
    L = int(W.uniform_ints(32, 8192, 32768, W.seed_of("batched", 0, 3))[b])
    n = (L + P_ - 1) // P_
    src = W.to_bits(W.normal((n, 2, Hkv, P_, D_), W.BF16, W.seed_of("batched", b, 1) * 64 + 7))
    q64 = C.bf16_bits_to_f64(W.to_bits(W.normal((1, Hq, D_), W.BF16, W.seed_of("batched", b, 0) * 64 + 7)))
    if codec == C.CODEC_BF16:
        pools = {codec: (src, None)}
    else:
        codes, meta = C.alloc_pool(codec, n, Hkv, P_, D_)
        C.quantize_pages(src, C.CODEC_BF16, list(range(n)), codec, codes, meta, list(range(n)))
        pools = {codec: (codes, meta)}
    t0 = time.perf_counter()
    oracle.paged_decode(q64, Hkv, P_, pools, np.full((1, n), codec, np.uint8), np.arange(n, dtype=np.int32)[None],
                        np.array([L]), W.softmax_scale(D_))
    return time.perf_counter() - t0


def _cpu_sparse_task(job):
    """One (layer, sequence) of the sparse workload: indexer scores over the
    4096 compressed keys, top-32 + newest selection, decode over the selected
    FP8 pages.  Timed: scores, selection and decode (the selected pages'
    codes are demoted beforehand, untimed)."""
    layer, b = job
    import oracle
    from oracle import codecs as C
    from mixed_precision_paged_argus_gb300 import workloads as W
    Hq, Hkv, D_, P_, NP, K_ = 32, 4, 128, 64, 4096, 32
    width = 2 * K_ + 8
    ck = W.to_bits(W.normal((1, NP, Hkv, D_), W.BF16, W.seed_of("sparse", layer, 6) * 16 + b))
    q64 = C.bf16_bits_to_f64(W.to_bits(W.normal((1, Hq, D_), W.BF16, W.seed_of("sparse", layer, 0) * 16 + b)))
    # the pool: only the pages a selection can name are materialised (demoted)
    t0 = time.perf_counter()
    sel, cnt, _ = oracle.select_pages(q64, ck, [NP], Hkv, K_, True, width)
    t_sel = time.perf_counter() - t0
    pages = sorted(set(int(x) for x in sel[0].ravel() if x >= 0))
    slot_of = {p: i for i, p in enumerate(pages)}
    src = W.to_bits(W.normal((len(pages), 2, Hkv, P_, D_), W.BF16, W.seed_of("sparse", layer, 1) * 16 + b))
    codes, meta = C.alloc_pool(C.CODEC_FP8_E4M3, len(pages), Hkv, P_, D_)
    C.quantize_pages(src, C.CODEC_BF16, list(range(len(pages))), C.CODEC_FP8_E4M3, codes, meta,
                     list(range(len(pages))))
    table = np.zeros((1, NP), np.int32)
    for p_, i in slot_of.items():
        table[0, p_] = i
    t1 = time.perf_counter()
    oracle.paged_decode(q64, Hkv, P_, {C.CODEC_FP8_E4M3: (codes, meta)}, np.full((1, NP), C.CODEC_FP8_E4M3, np.uint8),
                        table, np.array([NP * P_]), W.softmax_scale(D_), sel_pages=sel, sel_count=cnt,
                        sel_width=width)
    return t_sel + (time.perf_counter() - t1)


def _cpu_prefill_row(job):
    """One query row of the windowed prefill: its attention against each of the
    eight 131072-token windows of the cache and the chunk window, folded by
    log2-sum-exp (the oracle's window_attention and fold_lse).  Seconds."""
    hq, i = job
    import oracle
    from oracle import codecs as C
    from mixed_precision_paged_argus_gb300 import workloads as W
    NQ, CTX, WIN, D_ = 1024, 1 << 20, 131072, 128
    q = np.zeros((1, NQ, D_))
    q[0, i] = C.bf16_bits_to_f64(W.to_bits(W.normal((D_,), W.BF16, W.seed_of("prefill", hq, 0) * 1024 + i)))
    acc_o, acc_l = None, None
    spent = 0.0
    for w0, wl in [(w, WIN) for w in range(0, CTX, WIN)] + [(CTX, NQ)]:
        k = C.bf16_bits_to_f64(W.to_bits(W.normal((1, wl, D_), W.BF16, W.seed_of("prefill", hq, 1) * 64 + w0 // WIN)))
        v = C.bf16_bits_to_f64(W.to_bits(W.normal((1, wl, D_), W.BF16, W.seed_of("prefill", hq, 2) * 64 + w0 // WIN)))
        t0 = time.perf_counter()
        o, l = oracle.window_attention(q, k, v, w0, CTX, W.softmax_scale(D_), rows=[i])
        acc_o, acc_l = (o, l) if acc_o is None else oracle.fold_lse(acc_o, acc_l, o, l)
        spent += time.perf_counter() - t0
    return spent


def cpu_legs():
    """The oracle's time for the tiny (one core), batched, sparse and prefill
    workloads; returns {leg: cpu_baseline dict}."""
    import multiprocessing as mp
    from oracle import codecs as C
    cores = os.cpu_count() or 1
    out = {}
    per = _cpu_tiny(1)
    reps = max(1, int(2.0 / max(per, 1e-4)))
    per = _cpu_tiny(reps)
    out["tiny_fp16"] = {"value": per * 1e6, "unit": "us/step", "cores": 1, "kind": "oracle",
                        "sample": "%d full steps (the whole workload), single-threaded" % reps}
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        for name, codec in (("decode_bf16", C.CODEC_BF16), ("decode_fp8", C.CODEC_FP8_E4M3)):
            t0 = time.perf_counter()
            secs = pool.map(_cpu_batched_row, [(b, codec) for b in range(32)])
            wall = time.perf_counter() - t0
            out["batched_" + name] = {
                "value": sum(secs) / cores * 1e6, "unit": "us/step", "cores": cores, "kind": "oracle",
                "sample": "one full step (all 32 sequences) in %d processes; value = summed decode seconds / cores "
                          "(%.1f s wall incl. input generation%s)" % (cores, wall,
                                                                      ", FP8 demotion untimed" if codec else "")}
        t0 = time.perf_counter()
        secs = pool.map(_cpu_sparse_task, [(l, b) for l in range(12) for b in range(8)])
        wall = time.perf_counter() - t0
        out["sparse"] = {"value": sum(secs) / cores * 1e6, "unit": "us/step", "cores": cores, "kind": "oracle",
                         "sample": "one full step (12 layers x 8 sequences: scores, top-k, decode over the selected "
                                   "FP8 pages; their demotion untimed) in %d processes (%.1f s wall)" % (cores, wall)}
        rows = [(hq, i) for hq in (0, 9) for i in (0, 1, 511, 1023)]
        t0 = time.perf_counter()
        secs = pool.map(_cpu_prefill_row, rows)
        wall = time.perf_counter() - t0
        per_row = sum(secs) / len(rows)
        out["prefill"] = {"value": per_row * 16 * 1024 / cores * 1e3, "unit": "ms/step (extrapolated)", "cores": cores,
                          "kind": "oracle",
                          "sample": "EXTRAPOLATED: %d sampled query rows (heads 0 and 9; rows 0, 1, 511, 1023), each "
                                    "against all nine windows and folded; mean %.3f s per row x 16384 rows / %d "
                                    "cores (%.1f s wall)" % (len(rows), per_row, cores, wall)}
    return out


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="argus", choices=["argus", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="skip the other four workloads")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    n_gpus = max(args.gpus, world)

    if args.impl == "reference":
        if rank != 0:
            return
        cb = oracle_leg()
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "us/token/layer",
                "n_gpus": n_gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step":
                cb["value"] * LAYERS / 1000.0, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOAD, "batch": 1, "layers": LAYERS},
                "cpu_baseline": {"value": cb["value"], "unit": cb["unit"], "cores": cb["cores"],
                                 "kind": "oracle", "sample": cb["sample"]},
                "e2e": {"value": cb["value"], "unit": "us/token/layer", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    cpu = None
    cpu_leg = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_leg()                         # before the first GPU call (spawned pool)
        if not args.no_legs:
            cpu_leg = cpu_legs()
    ms_step, ms_e2e, clocks, t_wall, h2d, d2h = run_gpu(args, rank, world)
    legs = None
    if rank == 0 and not args.no_legs:
        legs = run_legs(max(5, args.steps // 2), args.warmup)
    if rank != 0:
        return
    hbm, _, peak_kind = peaks()
    bytes_layer = kv_bytes_per_layer()
    launch_ms = ms_step / LAYERS
    achieved = bytes_layer / (launch_ms * 1e-3) / 1e9
    us_tl = aggregate_us_per_token_layer(ms_step, world)
    traffic = profiled_traffic("decode_mixed_tier", ["decode.cu", "common.cuh"])
    line = {
        "metric": METRIC, "value": us_tl, "unit": "us/token/layer", "n_gpus": n_gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 mma / f32 accumulate (fp16, fp8, int8, int4 pages)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "layers": LAYERS, "context": CTX, "page_tokens": P,
                   "l2": "flushed (2x L2 write) before every timed step, outside the timed region",
                   "replay": "24 x (decode + split-combine) launches as one CUDA graph, chained by "
                             "programmatic dependent launch",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "kv_bytes_per_layer": bytes_layer,
        "kv_gbs": achieved,
        "kv_frac_of_8tbs": achieved / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "peak_kind": peak_kind + " (hbm_gbs)",
                     "kernel": "argus decode_kernel<64,f16 query,f16 family>",
                     "per_launch_bytes": bytes_layer},
        "e2e": {"value": ms_e2e * 1000.0 / LAYERS, "unit": "us/token/layer", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "per step: pinned q for 24 layers copied H2D, 24 argus_paged_decode_attn calls through "
                       "the ctypes binding, outputs copied D2H; CUDA events on the stream"},
        "gpu_launches": 2 * LAYERS * args.steps,
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if legs is not None:
        if cpu_leg:
            # each leg's oracle time beside it
            for key, cb in cpu_leg.items():
                if key.startswith("batched_"):
                    target = legs.get("batched", {}).get(key[len("batched_"):])
                else:
                    target = legs.get(key)
                if isinstance(target, dict):
                    target["cpu_baseline"] = cb
        line["legs"] = legs
    print(json.dumps(line))


if __name__ == "__main__":
    main()
