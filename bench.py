"""Benchmark of the paged-KV attention step on GB300.

Headline (``value``): HBM throughput of one decode step of the Llama-3.1-8B-
shaped batch (64 sequences, context U[512, 4096], 32 query / 8 KV heads,
head_dim 128, bf16 KV, 20,000-block permuted pool) -- algorithmic bytes (every
valid key's K and V once, plus q and out) over the device time of the step.
Beside it, in the same run: the mixed unified step (120 decodes + a 1022-token
chunk after a shared 2,000-token prefix, one copy-on-write) as tokens/s, the
roofline of the dominant kernel, an end-to-end number through the public API
with host buffers, and the CPU oracle on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same step on its own GPU (independent
replicas: the step has no exchange), timing is max over ranks, and ``value``
is the sum of all ranks' bytes over that time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn decode HBM TB/s (fraction of peak); mixed-step tokens/s"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _tensor_peak():
    """Dense bf16 tensor peak (burst figure: the prefill kernel is timed in
    isolation), as measured on these GPUs (MEASURED_PEAKS.json), else the
    fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def _max_over_ranks(values, device):
    """Replicas: every rank runs the same step on its own GPU; a job's time
    is the slowest rank's.  Returns the element-wise max over ranks (the
    values themselves on one process)."""
    import torch
    import torch.distributed as dist
    vals = [float(v) for v in values]
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor(vals, dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        vals = [float(x) for x in t.tolist()]
    return vals


def _job_rate(units_per_rank, ms, world_size, scale=1e12):
    """Whole-job rate: the units all ranks processed / the job's time (ms),
    in units of `scale` per second."""
    return units_per_rank * world_size / (ms * 1e-3) / scale


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                                    delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # the timed region starts once the sampler is producing lines
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 3.0:
            self.file.flush()
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def _device_inputs(wl, dev, casc=None):
    import torch
    from paged_kv_cache_82_gb300.metadata import build_step_metadata
    md = build_step_metadata(wl.requests)
    d = {
        "kc": wl.k_cache.to(dev), "vc": wl.v_cache.to(dev),
        "q": wl.q.to(dev),
        "bt": torch.from_numpy(md["block_tables"]).to(dev),
        "sl": torch.from_numpy(md["seq_lens"]).to(dev),
        "qsl": torch.from_numpy(md["query_start_loc"]).to(dev),
        "slots": torch.from_numpy(md["slot_mapping"]).to(dev),
        "md": md,
    }
    if wl.write_new:
        d["key"] = wl.key.to(dev)
        d["value"] = wl.value.to(dev)
    if wl.copy_pairs:
        d["pairs"] = torch.tensor(wl.copy_pairs, dtype=torch.int64, device=dev)
    d["out"] = torch.empty_like(d["q"])
    import paged_kv_cache_82_gb300 as pa
    from paged_kv_cache_82_gb300.metadata import cascade_prefix_blocks
    # a step whose requests share leading blocks runs as a cascade where
    # that measured faster (the engine knows the shared prefix from its
    # block manager); casc forces a prefix length (0: the plain step)
    if casc is None:
        casc = cascade_prefix_blocks(wl.requests,
                                     wl.num_q_heads // wl.num_kv_heads,
                                     wl.cache_dtype)
    d["casc"] = casc
    sizes = (wl.q.shape[0], wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
             len(wl.requests), md["max_query_len"], md["max_seq_len"])
    if wl.sliding_window > 0:
        nbytes = pa.pa_attention_window_workspace_size(*sizes, wl.sliding_window)
    elif d["casc"] > 0:
        nbytes = pa.pa_attention_cascade_workspace_size(*sizes)
    else:
        nbytes = pa.pa_attention_workspace_size(*sizes)
    d["ws"] = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    return d


def _step(pa, wl, d):
    """One pass of the hot path over the step: copy-on-write copies, K/V
    writes, attention.  Returns the number of our kernel launches (the
    library's own count)."""
    n0 = pa.pa_launch_count()
    cdt = wl.cache_dtype
    if wl.copy_pairs:
        pa.pa_copy_blocks(d["kc"], d["vc"], d["pairs"], cache_dtype=cdt)
    if wl.write_new:
        pa.pa_reshape_and_cache(d["key"], d["value"], d["kc"], d["vc"],
                                d["slots"], k_scale=wl.k_scale,
                                v_scale=wl.v_scale, cache_dtype=cdt)
    md = d["md"]
    if wl.sliding_window > 0:
        pa.pa_attention_window(d["q"], d["kc"], d["vc"], d["bt"], d["sl"],
                               d["qsl"], md["max_query_len"], md["max_seq_len"],
                               wl.scale, wl.sliding_window, wl.k_scale,
                               wl.v_scale, out=d["out"], workspace=d["ws"],
                               cache_dtype=cdt)
    elif d.get("casc", 0) > 0:
        pa.pa_attention_cascade(d["q"], d["kc"], d["vc"], d["bt"], d["sl"],
                                d["qsl"], md["max_query_len"], md["max_seq_len"],
                                wl.scale, d["casc"], wl.k_scale, wl.v_scale,
                                out=d["out"], workspace=d["ws"], cache_dtype=cdt)
    else:
        pa.pa_attention(d["q"], d["kc"], d["vc"], d["bt"], d["sl"], d["qsl"],
                        md["max_query_len"], md["max_seq_len"], wl.scale,
                        wl.k_scale, wl.v_scale, out=d["out"], workspace=d["ws"],
                        cache_dtype=cdt)
    return pa.pa_launch_count() - n0


def _cascade_vs_plain(pa, wl, dev, steps, warmup, flush):
    """Step time of a shared-prefix step run as a cascade (the prefix forced)
    and as the plain step, and the prefix length the host policy picks."""
    import torch
    from paged_kv_cache_82_gb300.metadata import (cascade_prefix_blocks,
                                                  common_prefix_blocks)
    res = {}
    for mode, n in (("cascade", common_prefix_blocks(wl.requests)),
                    ("plain", 0)):
        d = _device_inputs(wl, dev, casc=n)
        st, _, _ = _time_steps(pa, wl, d, steps, warmup, flush)
        flags = pa.pa_get_device_error()
        if flags:
            raise RuntimeError(f"device error flags 0x{flags:x} ({mode})")
        res[mode + "_ms"] = statistics.median(st)
        del d
        torch.cuda.empty_cache()
    res["speedup"] = res["plain_ms"] / res["cascade_ms"]
    res["policy_blocks"] = cascade_prefix_blocks(
        wl.requests, wl.num_q_heads // wl.num_kv_heads, wl.cache_dtype)
    return res


def _window_decode(pa, dev, flush, steps, warmup, peak_gbs):
    """A sliding-window layer's decode step: every query sees its last
    `window` keys (pa_attention_window: the window's view, then the head-group
    decode kernel over the view's pages), against pa_attention over the whole
    contexts of the same batch."""
    import torch
    import workloads
    wl = workloads.sliding_window_decode()
    byts = wl.kv_bytes() + wl.qo_bytes()
    res = {"workload": "Llama-3.1-8B shape: " + wl.description,
           "window_kv_bytes": wl.kv_bytes()}
    for mode in ("window", "whole_context"):
        if mode == "whole_context":
            W, wl.sliding_window = wl.sliding_window, 0
        d = _device_inputs(wl, dev)
        st, kt, _ = _time_steps(pa, wl, d, steps, warmup, flush)
        flags = pa.pa_get_device_error()
        if flags:
            raise RuntimeError(f"device error flags 0x{flags:x} ({mode})")
        res[mode + "_step_ms"] = statistics.mean(st)
        if mode == "window":
            res["kernel_ms"] = statistics.mean(kt)
        del d
        torch.cuda.empty_cache()
    wl.sliding_window = W
    res["step_tbs"] = byts / (res["window_step_ms"] * 1e-3) / 1e12
    res["kernel_tbs"] = byts / (res["kernel_ms"] * 1e-3) / 1e12
    res["frac_of_measured_hbm"] = res["kernel_tbs"] * 1e3 / peak_gbs
    res["speedup_vs_whole_context"] = (res["whole_context_step_ms"] /
                                       res["window_step_ms"])
    return res


def _block_manager_host(n_requests=160, prompt=2000, shared=1024,
                        out_tokens=64):
    """Host cost of the block manager and step planner: a first-come
    first-served serving loop over requests that share a 1024-token prompt
    prefix (prefix-cache hits), 2048-token budget, up to 128 running
    requests; per step schedule() + the step's metadata + update().  Pure
    host work (no GPU): microseconds per planned step."""
    import random
    from paged_kv_cache_82_gb300.block_manager import KVCacheManager, Scheduler
    from paged_kv_cache_82_gb300.metadata import build_step_metadata
    rnd = random.Random(82009)
    head = [rnd.randrange(32000) for _ in range(shared)]
    sched = Scheduler(KVCacheManager(40000), token_budget=2048,
                      max_num_seqs=128, long_prefill_threshold=512)
    for i in range(n_requests):
        tail = [rnd.randrange(32000) for _ in range(prompt - shared)]
        sched.add_request(f"r{i}", head + tail, out_tokens)
    t0 = time.perf_counter()
    steps = tokens = 0
    while (sched.waiting or sched.running) and steps < 5000:
        plan = sched.schedule()
        if plan.requests:
            build_step_metadata(plan.requests, block_tables=plan.block_tables)
        tokens += sum(plan.scheduled.values())
        sched.update(plan, {rid: 1 for rid in plan.scheduled})
        steps += 1
    dt = time.perf_counter() - t0
    return {"workload": (f"{n_requests} requests, {prompt}-token prompts sharing "
                         f"a {shared}-token prefix, {out_tokens} output tokens "
                         "each; budget 2048 tokens, <= 128 running, prompt "
                         "chunks <= 512"),
            "steps": steps, "tokens": tokens,
            "us_per_step": dt / max(steps, 1) * 1e6,
            "finished": len(sched.finished)}


def _time_steps(pa, wl, d, steps, warmup, flush):
    """Device time of the step and of its main attention kernel.

    The step (all its launches) is captured once in a CUDA graph and replayed
    -- the way a serving engine runs its decode steps -- with the L2 flushed
    (a 512 MiB read) before every timed replay; CUDA events on the stream
    bracket each replay.  The main kernel is timed separately on eager calls
    through the library's event hook, which brackets just that launch.
    Returns (step ms list, kernel ms list, launches in the timed replays)."""
    import torch
    for _ in range(warmup):
        _step(pa, wl, d)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        launches_per_step = _step(pa, wl, d)      # one more warm call
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            _step(pa, wl, d)
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ms = []
    for _ in range(steps):
        flush.sum()          # read 512 MiB: evicts the previous step's lines
        s0, s1 = ev(), ev()
        s0.record()
        graph.replay()
        s1.record()
        s1.synchronize()
        step_ms.append(s0.elapsed_time(s1))
    kern_ms = []
    k0, k1 = ev(), ev()
    pa.pa_set_profile_events(k0, k1)
    try:
        for _ in range(steps):
            flush.sum()
            _step(pa, wl, d)
            k1.synchronize()
            kern_ms.append(k0.elapsed_time(k1))
    finally:
        pa.pa_set_profile_events(None, None)
    del graph
    return step_ms, kern_ms, launches_per_step * steps


def _e2e(pa, wl, d, steps, warmup):
    """Same step through the public API from pinned host buffers: per step the
    host->device copy of the step's inputs (q, the metadata, and the new K/V
    and slots when the step writes them) packed in one pinned buffer, the
    step, and the device->host copy of its output, all inside the timed
    region.  As a serving loop runs them, the copies go on a second stream
    and overlap the neighbouring steps: the inputs of step k + 1 upload while
    step k runs and the output of step k downloads while step k + 1 runs
    (inputs and outputs double-buffered on the device and the host)."""
    import torch
    md = d["md"]
    parts = {
        "q": wl.q,
        "bt": torch.from_numpy(md["block_tables"]),
        "sl": torch.from_numpy(md["seq_lens"]),
        "qsl": torch.from_numpy(md["query_start_loc"]),
    }
    if wl.write_new:
        parts["slots"] = torch.from_numpy(md["slot_mapping"])
        parts["key"] = wl.key
        parts["value"] = wl.value
    # per buffer: one pinned staging buffer and one device buffer,
    # 256-byte aligned views
    offs, total = {}, 0
    for k, t in parts.items():
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_in, dev_in, views, out_h, out_d = [], [], [], [], []
    for _ in range(2):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        db = torch.empty(total, dtype=torch.uint8, device=d["q"].device)
        dd = dict(d)
        for k, t in parts.items():
            n = t.numel() * t.element_size()
            hb[offs[k]:offs[k] + n].copy_(t.contiguous().view(-1).view(torch.uint8))
            dd[k] = db[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        dd["out"] = torch.empty_like(d["out"])
        host_in.append(hb)
        dev_in.append(db)
        views.append(dd)
        out_h.append(torch.empty(d["out"].shape, dtype=d["out"].dtype).pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in parts.values())
    d2h = out_h[0].numel() * out_h[0].element_size()
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        with torch.cuda.stream(copy):
            dev_in[0].copy_(host_in[0], non_blocking=True)
            in_ready[0].record(copy)
        for k in range(n):
            i = k & 1
            comp.wait_event(in_ready[i])
            _step(pa, wl, views[i])
            done[i].record(comp)
            with torch.cuda.stream(copy):
                if k + 1 < n:
                    # buffer 1 - i was last read by step k - 1
                    if k >= 1:
                        copy.wait_event(done[1 - i])
                    dev_in[1 - i].copy_(host_in[1 - i], non_blocking=True)
                    in_ready[1 - i].record(copy)
                copy.wait_event(done[i])
                out_h[i].copy_(views[i]["out"], non_blocking=True)

    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
        enable_timing=True)
    e0.record(comp)
    run(steps)
    e1.record(copy)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


def _cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else the Arm
    implementer / part codes), with the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        name = fields["model name"]
    elif fields.get("CPU implementer"):
        part = fields.get("CPU part", "?")
        arm = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1",
               "0xd49": "Arm Neoverse N2", "0xd0c": "Arm Neoverse N1"}
        known = arm.get(part) if fields["CPU implementer"] == "0x41" else None
        name = (f"{known + ' (' if known else ''}implementer "
                f"{fields['CPU implementer']}, part {part}{')' if known else ''}")
    else:
        name = platform.processor() or "unknown"
    return f"{platform.machine()}: {name}"


def _cpu_baseline(wl, bytes_per_step, budget_s=12.0, max_reps=20):
    """The oracle, as it stands, on the host cores: whole decode steps of the
    same workload until about `budget_s` of CPU work."""
    import oracle
    md = oracle.step_metadata(wl.requests)
    cores = os.cpu_count() or 1
    times = []
    t_start = time.perf_counter()
    while len(times) < max_reps and (time.perf_counter() - t_start) < budget_s:
        t0 = time.perf_counter()
        oracle.paged_attention(wl.q, wl.k_cache, wl.v_cache,
                               md["block_tables"], md["seq_lens"],
                               md["query_start_loc"], scale=wl.scale,
                               cache_dtype=wl.cache_dtype, num_threads=cores)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    return {"value": bytes_per_step / t / 1e12, "unit": "TB/s", "cores": cores,
            "cpu": _cpu_model(),
            "kind": "oracle",
            "sample": (f"{len(times)} whole decode steps of the same batch "
                       f"(64 seqs), fp64, {cores} threads, "
                       f"{t * 1e3:.0f} ms per step")}


def _traffic_record(kernel_src_hash):
    """DRAM bytes per launch of the main kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "attn_fast_cfg2_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != kernel_src_hash:
        return None
    return rec.get("dram_bytes_per_launch")


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("attn_fast.cu", "pa_common.cuh", "pa_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_82_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _cache_ops(pa, dev, flush, steps, warmup, peak_gbs):
    """HBM rate of pa_reshape_and_cache and pa_copy_blocks on their own:
    algorithmic bytes (every element read once and written once) over the
    device time of one call, the L2 flushed before each."""
    import torch
    T, Hkv, D, NB = 32768, 8, 128, 2 * 32768 // 16 + 8192
    gen = torch.Generator(device="cpu").manual_seed(82007)
    key = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16).to(dev)
    value = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16).to(dev)
    slots = torch.randperm(NB * 16, generator=gen)[:T].to(dev)
    res = {}

    def timed(fn):
        for _ in range(warmup):
            fn()
        ts = []
        for _ in range(steps):
            flush.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    for name, cdt, eb in (("reshape_and_cache_bf16", "bf16", 2),
                          ("reshape_and_cache_bf16_to_fp8", "e4m3", 1)):
        tdt = torch.bfloat16 if cdt == "bf16" else torch.uint8
        kc = torch.zeros(NB, Hkv, 16, D, dtype=tdt, device=dev)
        vc = torch.zeros_like(kc)
        ms = timed(lambda: pa.pa_reshape_and_cache(
            key, value, kc, vc, slots, k_scale=0.0125, v_scale=0.015,
            cache_dtype=cdt))
        byts = 2 * T * Hkv * D * (2 + eb)
        res[name] = {"tokens": T, "bytes": byts, "ms": ms,
                     "tbs": byts / (ms * 1e-3) / 1e12,
                     "frac_of_measured_hbm": byts / (ms * 1e-3) / 1e9 / peak_gbs}
        del kc, vc
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = torch.randperm(NB, generator=gen)
    pairs = torch.stack([perm[:4096], perm[4096:8192]], 1).to(dev)
    ms = timed(lambda: pa.pa_copy_blocks(kc, vc, pairs))
    byts = 2 * 2 * 4096 * Hkv * 16 * D * 2
    res["copy_blocks_bf16"] = {"pairs": 4096, "bytes": byts, "ms": ms,
                               "tbs": byts / (ms * 1e-3) / 1e12,
                               "frac_of_measured_hbm":
                                   byts / (ms * 1e-3) / 1e9 / peak_gbs}
    if pa.pa_get_device_error():
        raise RuntimeError("device error flags (cache ops)")
    return res


def _headline_config(wl, ws):
    """The `config` object of the headline line, identical in both arms: the
    workload and its sizes (the reference arm attends a bounded sample of it,
    described in its cpu_baseline)."""
    return {
        "workload": ("Llama-3.1-8B-shaped decode: 64 seqs, context "
                     "U[512,4096], 32q/8kv heads, head_dim 128, bf16 KV, "
                     "block 16, 20,000-block permuted pool"),
        "kv_bytes": wl.kv_bytes(), "q_out_bytes": wl.qo_bytes(),
        "l2": "flushed between timed steps (512 MiB read); KV 595 MB > L2",
        "parallelism": f"replicas x{ws}",
    }


def run_ours(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import paged_kv_cache_82_gb300 as pa
    import workloads
    pa.load_library()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    if args.only == "cascade-sweep":
        # the cascade's crossover: decode steps behind a shared prefix,
        # cascade against plain, over prefix lengths and request counts
        cdt = args.cache_dtype
        for priv in ((256, 2048), (1024, 8192)):
            for pb in (32, 64, 128, 256, 512, 1024, 4096):
                for n in (2, 8, 32, 64, 128):
                    if priv[0] == 1024 and (pb not in (128, 256) or n not in (8, 32)):
                        continue
                    wls = workloads.shared_prefix_decode(n, pb, *priv,
                                                         cache_dtype=cdt)
                    r = _cascade_vs_plain(pa, wls, dev, args.steps, args.warmup,
                                          flush)
                    print(json.dumps({"prefix_blocks": pb, "decodes": n,
                                      "private": list(priv), "cache": cdt, **{
                                          k: round(v, 4) if isinstance(v, float)
                                          else v for k, v in r.items()}}),
                          flush=True)
        return

    if args.only != "all":
        make = {"decode": workloads.config2, "mixed": workloads.config4,
                "prefill": workloads.prefill_chunk, "mha": workloads.config3,
                "fp8long": workloads.config5,
                "prefillfp8": lambda **k: workloads.prefill_chunk(
                    cache_dtype="e4m3", **k),
                "int4": lambda **k: workloads.config2(cache_dtype="int4", **k),
                "nvfp4": lambda **k: workloads.config2(cache_dtype="nvfp4",
                                                       **k)}[args.only]
        # a smaller batch of the same shape (profiler captures); the mixed
        # step keeps its shared prefix and chunk, with fewer decodes and a
        # pool sized to them
        if args.batch and args.only == "mixed":
            wl = make(num_decodes=args.batch,
                      num_blocks=200 + args.batch * 520 + 64)
        else:
            wl = make(batch=args.batch) if args.batch else make()
        d = _device_inputs(wl, dev)
        step_ms, kern_ms, _ = _time_steps(pa, wl, d, args.steps, args.warmup,
                                          flush)
        flags = pa.pa_get_device_error()
        byts = wl.kv_bytes() + wl.qo_bytes()
        km = statistics.mean(kern_ms)
        print(f"{args.only}: step {statistics.mean(step_ms):.4f} ms, "
              f"attention kernels {km:.4f} ms, "
              f"{byts / km / 1e9:.3f} TB/s, "
              f"{workloads.attention_flops(wl) / km / 1e9:.1f} TFLOP/s, "
              f"flags 0x{flags:x}")
        if flags:
            raise SystemExit(2)
        return

    # ---- decode step (headline)
    wl = workloads.config2()
    d = _device_inputs(wl, dev)
    kv_bytes = wl.kv_bytes()
    alg_bytes = kv_bytes + wl.qo_bytes()
    sampler = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall0 = time.perf_counter()
    step_ms, kern_ms, launches = _time_steps(pa, wl, d, args.steps,
                                             args.warmup, flush)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    flags = pa.pa_get_device_error()
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x}")
    ms, kern = _max_over_ranks([statistics.mean(step_ms),
                                statistics.mean(kern_ms)], dev)
    value = _job_rate(alg_bytes, ms, ws)
    peak_gbs, peak_kind = _peaks()
    achieved_gbs = alg_bytes / (kern * 1e-3) / 1e9
    traffic = _traffic_record(_kernel_hash())

    # ---- end to end through the public API with host buffers
    e2e_ms, h2d, d2h = _e2e(pa, wl, d, max(3, args.steps // 2), 2)
    e2e_ms = _max_over_ranks([e2e_ms], dev)[0]
    e2e_value = _job_rate(alg_bytes, e2e_ms, ws)
    del d

    # ---- mixed unified step (tokens/s)
    wl4 = workloads.config4()
    d4 = _device_inputs(wl4, dev)
    m_step, m_kern, m_launch = _time_steps(pa, wl4, d4, args.steps,
                                           args.warmup, flush)
    flags = pa.pa_get_device_error()
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x} (mixed step)")
    m_ms = _max_over_ranks([statistics.mean(m_step)], dev)[0]
    m_bytes = wl4.kv_bytes() + wl4.qo_bytes()
    mixed = {
        "workload": ("Llama-3.1-8B shape, bf16: 120 decodes (private context "
                     "U[1024,8192] after a shared 2000-token prefix) + one "
                     "1022-token chunked prefill after the prefix; 1 "
                     "copy_blocks, 1142-token reshape_and_cache, attention"),
        "tokens_per_s": wl4.num_tokens * ws / (m_ms * 1e-3),
        "ms_per_step": m_ms,
        "unique_kv_bytes": wl4.kv_bytes(), "logical_kv_bytes":
            wl4.kv_bytes(unique=False),
        "hbm_tbs": m_bytes / (m_ms * 1e-3) / 1e12,
        "frac_of_measured_hbm": m_bytes / (m_ms * 1e-3) / 1e9 / peak_gbs,
        "attention_kernels_ms": statistics.mean(m_kern),
    }
    del d4

    # ---- decodes behind a long shared prefix: the cascade against the
    # plain step (the prefix read once per KV head, in key ranges)
    wls = workloads.shared_prefix_decode()
    sp = _cascade_vs_plain(pa, wls, dev, max(3, args.steps // 10), args.warmup,
                           flush)
    shared_prefix = {
        "workload": ("Llama-3.1-8B shape, bf16: " + wls.description +
                     "; 32 K/V writes, attention"),
        "unique_kv_bytes": wls.kv_bytes(),
        "logical_kv_bytes": wls.kv_bytes(unique=False),
        "tbs_unique_cascade": (wls.kv_bytes() + wls.qo_bytes()) /
                              (sp["cascade_ms"] * 1e-3) / 1e12,
        **sp,
    }
    del wls

    # ---- a sliding-window layer's decode step (the window's keys only),
    # against the same batch without the window
    window = _window_decode(pa, dev, flush, max(3, args.steps // 10),
                            args.warmup, peak_gbs)

    # ---- the other decode workloads of the scope (kernel and step TB/s)
    others = {}
    for name, make in (("mha_fp16_32x8192", workloads.config3),
                       ("fp8_long_context_70b", workloads.config5),
                       ("int4_decode_llama31_8b",
                        lambda: workloads.config2(cache_dtype="int4")),
                       ("nvfp4_decode_llama31_8b",
                        lambda: workloads.config2(cache_dtype="nvfp4")),
                       ("bf16_head_dim_64_decode",
                        lambda: workloads.config2(head_dim=64))):
        wlo = make()
        do = _device_inputs(wlo, dev)
        o_step, o_kern, _ = _time_steps(pa, wlo, do, max(3, args.steps // 10),
                                        args.warmup, flush)
        flags = pa.pa_get_device_error()
        if flags:
            raise RuntimeError(f"device error flags 0x{flags:x} ({name})")
        ob = wlo.kv_bytes() + wlo.qo_bytes()
        others[name] = {
            "workload": wlo.description,
            "bytes": ob,
            "keys_per_s": sum(r.seq_len for r in wlo.requests) /
                          (statistics.mean(o_step) * 1e-3),
            "kernel_tbs": ob / (statistics.mean(o_kern) * 1e-3) / 1e12,
            "step_tbs": ob / (statistics.mean(o_step) * 1e-3) / 1e12,
            "frac_of_measured_hbm": ob / (statistics.mean(o_kern) * 1e-3) / 1e9 / peak_gbs,
        }
        del do, wlo

    # ---- the cache kernels alone at a size that fills the GPU: the K/V
    # writes of a 32,768-token prefill (bf16 -> bf16, and bf16 -> FP8) and
    # copy-on-write copies of 4,096 blocks (Llama-3.1-8B shape)
    cache_ops = _cache_ops(pa, dev, flush, max(3, args.steps // 10),
                           args.warmup, peak_gbs)

    # ---- prefill tiles alone: one long chunked prefill (tensor cores)
    wlp = workloads.prefill_chunk()
    dp = _device_inputs(wlp, dev)
    p_sampler = ClockSampler(local)
    torch.cuda.synchronize()
    p_sampler.start()
    p_step, p_kern, _ = _time_steps(pa, wlp, dp, args.steps, args.warmup,
                                    flush)
    torch.cuda.synchronize()
    p_clocks = p_sampler.stop()
    flags = pa.pa_get_device_error()
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x} (prefill step)")
    p_km = statistics.mean(p_kern)
    p_tflops = workloads.attention_flops(wlp) / (p_km * 1e-3) / 1e12
    bf16_peak, bf16_kind = _tensor_peak()
    prefill = {
        "workload": ("Llama-3.1-8B shape, bf16: one request, 4096-token "
                     "chunk after 4096 cached tokens (causal)"),
        "kernel": "prefill_tc_kernel (bf16, tcgen05): one grid, the step has no decode work",
        "bound": "tensor", "achieved": p_tflops, "peak": bf16_peak,
        "unit": "TFLOP/s", "frac": p_tflops / bf16_peak,
        "peak_kind": bf16_kind, "kernels_ms": p_km,
        "ms_per_step": statistics.mean(p_step),
        "flops": workloads.attention_flops(wlp),
        "clocks": p_clocks,
    }
    del dp

    # ---- the same chunk over an FP8 cache (tiles widened to f16 on chip)
    wlp8 = workloads.prefill_chunk(cache_dtype="e4m3")
    dp8 = _device_inputs(wlp8, dev)
    p8_step, p8_kern, _ = _time_steps(pa, wlp8, dp8, max(3, args.steps // 4),
                                      args.warmup, flush)
    flags = pa.pa_get_device_error()
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x} (fp8 prefill)")
    p8_km = statistics.mean(p8_kern)
    p8_tflops = workloads.attention_flops(wlp8) / (p8_km * 1e-3) / 1e12
    prefill_fp8 = {
        "workload": ("Llama-3.1-8B shape, bf16 q, FP8 E4M3 KV: one request, "
                     "4096-token chunk after 4096 cached tokens (causal)"),
        "kernel": ("prefill_tc_kernel (FP8 pages widened to f16 in shared "
                   "memory, f16 tcgen05): one grid, the step has no decode work"),
        "bound": "tensor", "achieved": p8_tflops, "peak": bf16_peak,
        "unit": "TFLOP/s", "frac": p8_tflops / bf16_peak,
        "peak_kind": bf16_kind + " (f16 rate = bf16 rate)",
        "kernels_ms": p8_km, "flops": workloads.attention_flops(wlp8),
    }
    del dp8

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(wl, alg_bytes)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": _headline_config(wl, ws),
        "wall_s": wall,
        "roofline": {
            "bound": "hbm", "kernel": "attn_decode_hg_kernel (bf16, KV-head groups of 4)",
            "achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
            "frac": achieved_gbs / peak_gbs, "peak_kind": peak_kind,
            "traffic": traffic, "kernel_ms": kern,
            "frac_of_8TBs_spec": achieved_gbs / 8000.0,
        },
        "e2e": {"value": e2e_value, "unit": "TB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "copies": ("pinned, on a second stream: step k+1's inputs "
                           "upload and step k's output downloads while "
                           "step k / k+1 runs")},
        "gpu_launches": launches,
        "clocks": clocks,
        "mixed_step": mixed,
        "shared_prefix_decode": shared_prefix,
        "sliding_window_decode": window,
        "block_manager_host": _block_manager_host(),
        "prefill_step": prefill,
        "prefill_step_fp8": prefill_fp8,
        "other_decodes": others,
        "cache_ops": cache_ops,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    """The oracle as it stands, on the host cores: each step attends a
    bounded sample of the decode batch (its first n requests, n chosen so
    that warm-up + K steps take about a minute), reported in the same unit
    as the GPU arm (algorithmic bytes of the sample / time)."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import workloads
    wl = workloads.config2()
    import oracle
    cores = os.cpu_count() or 1

    def runner(n):
        reqs = wl.requests[:n]
        md = oracle.step_metadata(reqs)
        q = wl.q[:n]  # one query token per request
        def one():
            oracle.paged_attention(q, wl.k_cache, wl.v_cache,
                                   md["block_tables"], md["seq_lens"],
                                   md["query_start_loc"], scale=wl.scale,
                                   cache_dtype=wl.cache_dtype,
                                   num_threads=cores)
        keys = sum(r.num_computed + r.num_new for r in reqs)
        nbytes = (keys * wl.num_kv_heads * wl.head_dim * 2 * 2 +
                  2 * n * wl.num_q_heads * wl.head_dim * 2)
        return one, nbytes

    # size the sample from a timed call on all requests
    full, _ = runner(len(wl.requests))
    t0 = time.perf_counter()
    full()
    t_full = time.perf_counter() - t0
    budget_s = 60.0 / (args.steps + args.warmup)
    n = max(1, min(len(wl.requests),
                   int(len(wl.requests) * budget_s / max(t_full, 1e-6))))
    one, nbytes = runner(n)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    value = nbytes / (ms * 1e-3) / 1e12
    sample = (f"first {n} of the {len(wl.requests)} decode requests per step "
              f"({nbytes} KV + q/out bytes), fp64, {cores} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _headline_config(wl, ws),
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores,
                         "cpu": _cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "decode", "mixed", "prefill",
                                       "mha", "fp8long", "int4", "nvfp4",
                                       "prefillfp8", "cascade-sweep"],
                    default="all",
                    help="profiling runs: time just one step kind, no JSON "
                         "line (cascade-sweep: one JSON line per shared-"
                         "prefix decode step, cascade against plain)")
    ap.add_argument("--cache-dtype", choices=["bf16", "e4m3"], default="bf16",
                    help="with --only cascade-sweep: the cache type")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --only decode/mha/fp8long/mixed: that many "
                         "(decode) requests instead of the workload's own")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
