#!/usr/bin/env python
"""Benchmark of the streamed-expert MoE decode path on B300.

Default workload: a 30-layer MoE-only stack (H=2816, E=128 experts of
I=704, top-8, int4 group-64 experts with fp16 scale/bias, bf16 shared expert
2816->2112->2816), all experts resident in HBM, batch 1, decode steps with
the stack output fed back as the next input. One step = one token through all
30 layers. Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|streaming|batched]

--workload prefill times the 4096-token grouped layer (tcgen05 GEMMs);
--workload streaming runs the decode stack with the experts in pinned host
memory behind the 16-slot-per-layer LFU cache (metadata on the device; the
host-metadata mode on 1-4 copy streams beside it) and reports the hit rate, the
bytes fetched per token, the copy stall and the host-link bandwidth;
--workload batched runs the stack with 64 tokens per step through the grouped
tcgen05 path (routed and shared experts).

--impl reference times the CPU oracle (the plain single-threaded C reference
of the same layer) on the host cores, on a bounded sample of the same
workload. Multi-GPU runs are independent replicas (one sequence per GPU).
"""
from __future__ import annotations

import argparse
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

METRIC = "MoE decode tok/s (1 B300) and expert-weight HBM GB/s as % of peak"
H, I, E, K_ACT, S, L = 2816, 704, 128, 8, 2112, 30
SEED = 1
WORKLOAD_FMT = ("%d-layer MoE-only decode stack: H=2816, 128 experts of I=704 (int4 codes, fp16 scale+bias per 64), "
            "top-8 softmax routing, GELU-gated FFNs, bf16 shared expert 2816->2112->2816, RMSNorm; batch 1, "
            "output fed back each step; all experts resident in HBM; seed 1")

# algorithmic bytes per launch (weights read + activations), per kernel kind
ROUTED_GU = K_ACT * 2 * (I * H // 2 + I * (H // 64) * 4)       # 17,842,176
SHARED_GU = 2 * S * H * 2                                       # 23,789,568
ROUTED_D = K_ACT * (H * I // 2 + H * (I // 64) * 4)            # 8,921,088
SHARED_D = H * S * 2                                            # 11,894,784
ROUTER = E * H * 2                                              # 720,896
ACT_X = H * 2
ACT_H = (K_ACT * I + S) * 4
BYTES = {
    "router": ROUTER + ACT_X + E * 4 + K_ACT * 8,
    "gateup": ROUTED_GU + SHARED_GU + ACT_X + ACT_H,
    "down": ROUTED_D + SHARED_D + ACT_H + 2 * ACT_X,
}


def set_layers(n_layers: int) -> None:
    """Per-token byte counts for a stack of n_layers (30 in the benchmark workload)."""
    global L, ROUTED_PER_TOKEN, WEIGHTS_PER_TOKEN, WORKLOAD
    L = n_layers
    WORKLOAD = WORKLOAD_FMT % L
    BYTES["layer"] = L * (ROUTER + ROUTED_GU + SHARED_GU + ROUTED_D + SHARED_D + 2 * ACT_X)   # one launch = L layers
    ROUTED_PER_TOKEN = L * (ROUTED_GU + ROUTED_D)                  # expert-weight bytes per token
    WEIGHTS_PER_TOKEN = L * (ROUTER + ROUTED_GU + SHARED_GU + ROUTED_D + SHARED_D)


set_layers(L)


# DRAM traffic of the fused kernel taken from an ncu capture (not measured in this run): read + write bytes of a
# 4-layer stack of the same kernel, scaled by 30/4 to the 30-layer launch. Reported only while the kernel's code
# (its source and the headers it includes, without // comments and blank lines, plus the nvcc flags) is the one
# that was captured; null otherwise.
FUSED_TRAFFIC = {"code_sha256": "9aa74b6ac320a31c4079b3591632e0cd597bc4a0daf54be30b81cedc4260bfa6",
                 "bytes_per_layer": (252876544 + 2872320) / 4,
                 "capture": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch of a 4-layer stack "
                            "(profiles/k_fused_stack_decode30.md)"}
FUSED_SOURCES = ("tf_fused.cu", "tf_device.cuh", "tf_internal.h")


def code_hash(paths, extra=""):
    import hashlib
    lines = []
    for path in paths:
        for ln in open(path).read().splitlines():
            i = ln.find("//")
            ln = (ln[:i] if i >= 0 else ln).rstrip()
            if ln:
                lines.append(ln)
    lines.append(extra)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def fused_code_hash():
    from bit_expert_streaming_layer_b300 import build as kb
    csrc = os.path.join(ROOT, "bit_expert_streaming_layer_b300", "csrc")
    paths = [os.path.join(csrc, f) for f in FUSED_SOURCES] + [os.path.join(ROOT, "include", "tf.h")]
    return code_hash(paths, " ".join(kb.ARCH + kb.COMMON[:4]))


def fused_traffic(n_layers):
    if FUSED_TRAFFIC["code_sha256"] is None:
        return None
    try:
        h = fused_code_hash()
    except OSError:
        return None
    return int(FUSED_TRAFFIC["bytes_per_layer"] * n_layers) if h == FUSED_TRAFFIC["code_sha256"] else None


def spread(ms_list):
    """Median, p10 and p90 of per-step times (ms)."""
    a = np.asarray(ms_list, np.float64)
    return {"median_ms": round(float(np.median(a)), 5), "p10_ms": round(float(np.percentile(a, 10)), 5),
            "p90_ms": round(float(np.percentile(a, 90)), 5), "n": int(a.size)}


def host_info():
    """CPU model and core count of this host, GPU name."""
    model = ""
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    info = {"nproc": os.cpu_count(), "cpu_model": model}
    try:
        import torch
        if torch.cuda.is_available():
            info["gpu"] = torch.cuda.get_device_name(0)
    except Exception:
        pass
    return info


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle baseline

def _oracle_layer(O, W, x, l, mt, shared=None):
    """One layer of the decode stack on the oracle: (output bits, seconds of oracle time). Weight generation is
    not timed."""
    Wr = W.router_weights(SEED, l, E, H)
    shared = shared if shared is not None else W.shared_weights(SEED, l, H, S)
    t0 = time.perf_counter()
    r, z, idx, w = O.route(x, Wr, mt=mt)
    el = time.perf_counter() - t0
    experts = W.experts_parallel(SEED, l, idx, H, I)
    t0 = time.perf_counter()
    out, _ = O.layer_combine(x, r, experts, w, shared, mt=mt)
    return out, el + time.perf_counter() - t0


def oracle_baseline(n_layers: int = 6):
    """Time the CPU oracle on a bounded sample: the first n_layers of step 0 of the stack
    (routing + 8 experts + shared expert + combine), single thread. Returns tok/s for 30 layers."""
    import oracle as O
    import workload as W
    O.build()
    x = W.hidden(SEED, 0, 1, H)[0]
    elapsed, outs = 0.0, []
    for l in range(n_layers):
        x, dt = _oracle_layer(O, W, x, l, False)
        outs.append(x)
        elapsed += dt
    per_layer = elapsed / n_layers
    return {"value": 1.0 / (per_layer * L), "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": "%d of the 30 layers of one decode step (step 0, seed %d), single-threaded fp32 C oracle; "
                      "tok/s = 1 / (30 x mean layer time); weight generation not timed" % (n_layers, SEED),
            "seconds": elapsed, "outputs": outs}


def oracle_baseline_all_cores(ref_outputs):
    """The same oracle with OpenMP over its independent output rows, on all host cores, for one whole decode
    step (all layers of step 0); the layers the single-threaded sample covered must come out bit-identical."""
    import oracle as O
    import workload as W
    from concurrent.futures import ThreadPoolExecutor
    O.build()
    with ThreadPoolExecutor(min(32, os.cpu_count() or 1)) as ex:    # generation, not timed
        shared = list(ex.map(lambda l: W.shared_weights(SEED, l, H, S), range(L)))
    x = W.hidden(SEED, 0, 1, H)[0]
    elapsed = 0.0
    for l in range(L):
        x, dt = _oracle_layer(O, W, x, l, True, shared[l])
        elapsed += dt
        if l < len(ref_outputs):
            assert np.array_equal(x, ref_outputs[l]), "the all-cores oracle differs from the single-threaded one"
    return {"value": 1.0 / elapsed, "unit": "tok/s", "cores": O.threads(True), "kind": "oracle",
            "sample": "one whole decode step (all %d layers of step 0, seed %d), the fp32 C oracle with OpenMP "
                      "over its output rows (per-row sums unchanged; outputs bit-identical to the single-threaded "
                      "oracle on the layers both ran); weight generation not timed" % (L, SEED),
            "bit_identical_layers": len(ref_outputs), "seconds": round(elapsed, 3)}


def cpu_baselines(n_layers):
    one = oracle_baseline(n_layers)
    allc = oracle_baseline_all_cores(one["outputs"])
    return ({k: one[k] for k in ("value", "unit", "cores", "kind", "sample")},
            {k: allc[k] for k in ("value", "unit", "cores", "kind", "sample", "bit_identical_layers")})


# ------------------------------------------------------------------ GPU arm

def run_ours(args, rank, world):
    import torch
    import bit_expert_streaming_layer_b300 as B
    from workload.model import SyntheticStack, hidden_tensor

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stack = SyntheticStack(SEED, L, H=H, I=I, E=E, k=K_ACT, S=S, resident=True, device=dev)
    fused = None
    if args.path == "fused":
        fws = torch.zeros(B.tf_stack_workspace_bytes(L, E), dtype=torch.uint8, device=dev)
        fused = B.Stack(stack.layers, fws)
        fused.set_prefetch(args.prefetch)
    x0 = hidden_tensor(SEED, 0, 1, H, device=dev)[0]
    a = torch.empty(H, dtype=torch.bfloat16, device=dev)
    b = torch.empty(H, dtype=torch.bfloat16, device=dev)
    scratch = torch.empty(H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    a.copy_(x0)

    def step(src, dst):
        if fused is not None:
            B.tf_stack_step(fused, src, dst, stream)
        else:
            B.tf_stack_decode(stack.layers, src, dst, scratch, None, stream)

    cur, nxt = a, b
    for _ in range(args.warmup):
        step(cur, nxt)
        cur, nxt = nxt, cur
    torch.cuda.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    prof_steps = min(args.steps, args.profile_steps)
    B.tf_profile_begin(prof_steps * (1 if args.path == "fused" else L))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(args.steps):
        step(cur, nxt)
        cur, nxt = nxt, cur
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    prof = B.tf_profile_end()
    clocks = sampler.stop()
    if fused is not None:
        B.tf_stack_check(fused, stream)
    ms = evs[0].elapsed_time(evs[-1])
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    assert not torch.isnan(cur.float()).any(), "NaN in the stack output"

    # end to end through the public API with host buffers: H2D input, D2H output, every step
    hx = torch.empty(H, dtype=torch.bfloat16, pin_memory=True)
    hy = torch.empty(H, dtype=torch.bfloat16, pin_memory=True)
    hx.copy_(x0.cpu())
    e2e_steps = args.steps
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        a.copy_(hx, non_blocking=True)
        step(a, b)
        hy.copy_(b, non_blocking=True)
        stream.synchronize()
        hx.copy_(hy)
    e2e_s = time.perf_counter() - t0

    gpu_launches = sum(n for _, n in prof.values())
    if fused is not None:
        B.tf_stack_check(fused, stream)
        fused.close()
    stack.close()
    return ms, prof, clocks, gpu_launches, e2e_s, e2e_steps, step_ms


# ------------------------------------------------------------------ streamed experts (LFU cache, host store)

STREAM_SEED, STREAM_ZIPF, STREAM_SLOTS = 2, 1.1, 16
PREFILL_CHUNK, PREFILL_PROMPT = 128, 512     # chunked prefill through the cache: tokens per chunk, per prompt
STREAM_ALPHA = 0.1     # Zipf bias scale
STREAM_NOISE = 1.5     # sigma of the per-(step, layer) router-logit noise (the token-dependent part of the logits)
STREAM_METRIC = "MoE decode tok/s with experts streamed from pinned host memory through a 16-slot LFU cache (1 B300)"
STREAM_WORKLOAD = ("30-layer MoE-only decode stack, batch 1, a fresh x ~ N(0,1) per step (the next token's input); "
                   "experts (12.9 GB, 3,840 x 3.36 MB) in "
                   "pinned host memory, a 16-slot-per-layer LFU cache in HBM (1.61 GB) with its metadata on the "
                   "device, misses copied by a kernel reading the mapped host store on a high-priority stream, "
                   "overlapped with the shared expert (the host-metadata mode, cudaMemcpyAsync on 1-4 copy "
                   "streams, reported beside it); router logit bias = Zipf(1.1) "
                   "popularity (alpha %.2f) over a seeded per-layer rank->expert map + N(0, %.2f) noise per (step, layer) "
                   "(the synthetic weights route every token alike beyond layer 0) + 30 on the previous step's 8 ids "
                   "with probability 0.5 per (step, layer); seed 2")


def h2d_probe(dev, copy_stream, n_slots=32, reps=5):
    """Pinned host -> device copy bandwidth in GB/s: n_slots expert blobs, one copy each."""
    import torch
    import bit_expert_streaming_layer_b300 as B
    slot = B.tf_expert_slot_bytes(H, I)
    src = torch.empty(n_slots * slot, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n_slots * slot, dtype=torch.uint8, device=dev)
    best = 0.0
    with torch.cuda.stream(copy_stream):
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(copy_stream)
            for i in range(n_slots):
                dst[i * slot:(i + 1) * slot].copy_(src[i * slot:(i + 1) * slot], non_blocking=True)
            e1.record(copy_stream)
            copy_stream.synchronize()
            best = max(best, n_slots * slot / (e0.elapsed_time(e1) / 1000.0) / 1e9)
    return best


def run_streaming(args):
    """The decode stack with every expert in pinned host memory behind a 16-slot-per-layer LFU cache in HBM, in two
    modes on the same host store: the LFU metadata on the device (no host wait inside a token; the misses copied by
    a kernel reading the mapped host store) and on the host (one host wait per layer; the misses copied by the
    copy engine, cudaMemcpyAsync, on 1..4 copy streams). The line's value is the device-metadata mode."""
    import torch
    import bit_expert_streaming_layer_b300 as B
    import workload as W
    from workload.model import SyntheticStack, hidden_tensor

    seed, alpha, sigma = STREAM_SEED, args.alpha, args.noise
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stack = SyntheticStack(seed, L, H=H, I=I, E=E, k=K_ACT, S=S, resident=False, n_slots=STREAM_SLOTS,
                           T_max=PREFILL_CHUNK, device=dev)
    zipf_h = np.stack([W.zipf_bias(seed, l, E, STREAM_ZIPF, alpha)[0] for l in range(L)])
    bias_h = torch.empty(L, E, dtype=torch.float32, pin_memory=True)
    bias_hn = bias_h.numpy()
    bias_d = torch.empty(L, E, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    copy_streams = [torch.cuda.Stream(dev) for _ in range(4)]
    fetch = torch.cuda.Stream(dev, priority=-1)
    probe = h2d_probe(dev, copy_streams[0])
    sweep = [int(v) for v in args.slot_sweep.split(",") if v.strip()] if args.slot_sweep else []
    n_copy_points = 4
    n_inputs = args.warmup + args.steps + min(args.steps, 32) + min(args.steps, 64)
    xs = torch.stack([hidden_tensor(seed, t, 1, H, device=dev)[0] for t in range(n_inputs)])
    noise = np.stack([np.stack([W.route_noise(seed, l, t, E, sigma) for l in range(L)]) for t in range(n_inputs)])
    bufs = [torch.empty(H, dtype=torch.bfloat16, device=dev) for _ in range(5)]   # 0-1 outputs, 2-3 scratch, 4 input
    idx_views = [stack.layers[l].routing_tensors()[0][0] for l in range(L)]

    def new_device_cache(n_slots):
        pool = torch.zeros(L * n_slots * stack.slot, dtype=torch.uint8, device=dev)
        state = torch.zeros(B.tf_device_cache_state_bytes(L, n_slots, E, 0), dtype=torch.uint8, device=dev)
        c = B.DeviceCache(L, n_slots, E, stack.slot, pool, stack.store, state, 0)
        c.set_fetch_ctas(args.fetch_ctas)
        return c

    class Run:
        """One cache (host or device metadata) fed a sequence of tokens; counts what its steps did."""

        def __init__(self, mode, cache):
            self.mode, self.cache, self.prev = mode, cache, [None] * L
            self.zero()

        def zero(self):
            self.t = {"hits": 0, "misses": 0, "bytes": 0, "stall_ms": 0.0, "copy_ms": 0.0, "shared_ms": 0.0,
                      "tokens": 0}

        def token(self, step, src, dst, measure=0):
            for l in range(L):
                bias_hn[l] = zipf_h[l] + noise[step, l]
                if self.prev[l] is not None and W.coin(seed, l, step):
                    bias_hn[l, self.prev[l]] += 30.0
            bias_d.copy_(bias_h, non_blocking=True)
            x = src
            for l in range(L):
                y = dst if l == L - 1 else bufs[2 + l % 2]
                if self.mode == "device":
                    st = B.tf_layer_step_device_cache(stack.layers[l], self.cache, l, x, y, bias_d[l], 0, stream,
                                                      fetch, measure)
                else:
                    st = B.tf_layer_step(stack.layers[l], self.cache, l, step, stack.store, x, y, 1, bias_d[l], 0,
                                         stream, copy_streams[0], measure)
                    self.prev[l] = np.array(st.ids[:K_ACT], dtype=np.int64)
                if self.mode == "host" or measure:
                    for k_, f in (("hits", "hits"), ("misses", "misses"), ("bytes", "bytes_fetched"),
                                  ("stall_ms", "stall_ms"), ("copy_ms", "copy_ms"), ("shared_ms", "shared_ms")):
                        self.t[k_] += getattr(st, f)
                x = y
            if self.mode == "device":
                # the next token's router bias repeats this token's experts: one read of the 30 layers' ids
                ids = torch.stack(idx_views).cpu().numpy()
                for l in range(L):
                    self.prev[l] = ids[l].astype(np.int64)
            self.t["tokens"] += 1

    step = 0

    def timed(run, n_steps, warmup):
        """Every run replays the same tokens from a cold cache (steps 0 ..), so that all modes and sweep points
        see the same routing, hits and misses; only the mechanism differs."""
        nonlocal step
        step = 0
        for _ in range(warmup):
            run.token(step, xs[step], bufs[0])
            step += 1
        torch.cuda.synchronize()
        if run.mode == "device":
            c0 = run.cache.counters()
        run.zero()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_steps):
            run.token(step, xs[step], bufs[step % 2])
            step += 1
        e1.record(stream)
        torch.cuda.synchronize()
        t = dict(run.t)
        if run.mode == "device":
            c1 = run.cache.counters()
            t["hits"], t["misses"] = c1[0] - c0[0], c1[1] - c0[1]
            t["bytes"] = t["misses"] * stack.payload
        return e0.elapsed_time(e1), t

    def measured(run, n_steps):
        nonlocal step
        run.zero()
        for _ in range(n_steps):
            run.token(step, xs[step], bufs[0], measure=1)
            step += 1
        return dict(run.t)

    # ---- device-metadata mode (the line's value)
    dcache = new_device_cache(STREAM_SLOTS)
    drun = Run("device", dcache)
    sampler = ClockSampler(0)
    sampler.start()
    B.tf_profile_begin(min(args.steps, 8) * 6 * L)
    ms, timed_d = timed(drun, args.steps, args.warmup)
    prof = B.tf_profile_end()
    clocks = sampler.stop()
    assert not torch.isnan(bufs[(step - 1) % 2].float()).any(), "NaN in the stack output"
    meas_steps = min(args.steps, 32)
    meas_d = measured(drun, meas_steps)
    # end to end: the input from pinned host memory and the output back, every step
    hy = torch.empty(H, dtype=torch.bfloat16, pin_memory=True)
    hxs = xs.cpu().pin_memory()
    e2e_steps = min(args.steps, 64)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        bufs[4].copy_(hxs[step], non_blocking=True)
        drun.token(step, bufs[4], bufs[0])
        hy.copy_(bufs[0], non_blocking=True)
        stream.synchronize()
        step += 1
    e2e_s = time.perf_counter() - t0
    dcache.close()

    # ---- host-metadata mode: the copy engine on 1, 2, 3 and 4 copy streams (fresh cache per point, same tokens)
    host_points = []
    for n_cs in range(1, n_copy_points + 1):
        hcache = B.ExpertCache(L, STREAM_SLOTS, E, stack.slot, stack.pool)
        if n_cs > 1:
            hcache.set_copy_streams(copy_streams[:n_cs])
        hrun = Run("host", hcache)
        n_steps = args.steps
        hms, th = timed(hrun, n_steps, args.warmup)
        pt = {"copy_streams": n_cs, "steps": n_steps, "tok_s": round(n_steps / (hms / 1000.0), 2),
              "hit_rate": round(th["hits"] / max(1, th["hits"] + th["misses"]), 4),
              "bytes_fetched_per_token": int(th["bytes"] / n_steps),
              "fill_gbs": round(th["bytes"] / (hms / 1000.0) / 1e9, 2)}
        if n_cs == 1:
            mh = measured(hrun, meas_steps)
            pt["stall_us_per_token"] = round(mh["stall_ms"] * 1000.0 / max(1, mh["tokens"]), 1)
            pt["copy_gbs_during_fills"] = round(mh["bytes"] / max(1e-9, mh["copy_ms"] / 1000.0) / 1e9, 2)
        host_points.append(pt)
        hcache.close()

    # ---- slot-count sweep (device-metadata mode), one pool per point, the same tokens from a cold start
    sweep_out = []
    for n_slots in sweep:
        c = new_device_cache(n_slots)
        sms, ts = timed(Run("device", c), args.steps, args.warmup)
        sweep_out.append({"slots_per_layer": n_slots, "steps": args.steps,
                          "tok_s": round(args.steps / (sms / 1000.0), 2),
                          "hit_rate": round(ts["hits"] / max(1, ts["hits"] + ts["misses"]), 4),
                          "bytes_fetched_per_token": int(ts["bytes"] / args.steps),
                          "slot_pool_gb": round(L * n_slots * stack.slot / 1e9, 2)})
        c.close()
    # chunked prefill through the cache (host metadata, a fresh cache): a prompt of PREFILL_PROMPT fresh tokens in
    # chunks of PREFILL_CHUNK, each chunk through the 30 layers, the chunk's experts in waves of the 16 slots;
    # router bias: the layers' Zipf popularity term
    chunked = None
    if not args.no_chunked_prefill:
        pc = B.ExpertCache(L, STREAM_SLOTS, E, stack.slot, stack.pool)
        bias_d.copy_(torch.from_numpy(zipf_h.astype(np.float32)))
        prompt = hidden_tensor(seed, 1 << 20, PREFILL_PROMPT + PREFILL_CHUNK, H, device=dev)
        cb = [torch.empty(PREFILL_CHUNK, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        lstep = [0] * L
        tot_c = {"waves": 0, "hits": 0, "misses": 0, "bytes": 0}

        def chunk(xc):
            cur = xc
            for l in range(L):
                dst = cb[l % 2]
                stc = B.tf_layer_prefill_cached(stack.layers[l], pc, l, lstep[l], stack.store, cur, dst, PREFILL_CHUNK,
                                                bias_d[l], 0, stream, copy_streams[0])
                lstep[l] += stc.waves
                for k_, f in (("waves", "waves"), ("hits", "hits"), ("misses", "misses"), ("bytes", "bytes_fetched")):
                    tot_c[k_] += getattr(stc, f)
                cur = dst
        chunk(prompt[PREFILL_PROMPT:])          # warm-up chunk (also fills the cache from cold)
        torch.cuda.synchronize()
        for k_ in tot_c:
            tot_c[k_] = 0
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for ci in range(PREFILL_PROMPT // PREFILL_CHUNK):
            chunk(prompt[ci * PREFILL_CHUNK:(ci + 1) * PREFILL_CHUNK])
        c1.record(stream)
        torch.cuda.synchronize()
        cms = c0.elapsed_time(c1)
        lookups_c = tot_c["hits"] + tot_c["misses"]
        chunked = {"tokens": PREFILL_PROMPT, "chunk": PREFILL_CHUNK, "tok_s": round(PREFILL_PROMPT / (cms / 1000.0), 1),
                   "ms_per_chunk": round(cms / (PREFILL_PROMPT // PREFILL_CHUNK), 3),
                   "hit_rate": round(tot_c["hits"] / max(1, lookups_c), 4),
                   "bytes_fetched_per_token": int(tot_c["bytes"] / PREFILL_PROMPT),
                   "waves_per_chunk_layer": round(tot_c["waves"] / (L * (PREFILL_PROMPT // PREFILL_CHUNK)), 2),
                   "fill_gbs": round(tot_c["bytes"] / (cms / 1000.0) / 1e9, 2)}
        pc.close()

    # fetch-kernel width (device-metadata mode, 16 slots)
    fetch_sweep = []
    for ctas in [int(v) for v in args.fetch_sweep.split(",") if v.strip()]:
        c = new_device_cache(STREAM_SLOTS)
        c.set_fetch_ctas(ctas)
        fms, tf_ = timed(Run("device", c), args.steps, args.warmup)
        fetch_sweep.append({"fetch_ctas": ctas, "tok_s": round(args.steps / (fms / 1000.0), 2),
                            "fill_gbs": round(tf_["bytes"] / (fms / 1000.0) / 1e9, 2)})
        c.close()
    stack.close()

    n = args.steps
    lookups = timed_d["hits"] + timed_d["misses"]
    fetch_gbs = timed_d["bytes"] / (ms / 1000.0) / 1e9
    launches = sum(v[1] for v in prof.values())
    line = {
        "metric": STREAM_METRIC, "value": round(n / (ms / 1000.0), 2), "unit": "tok/s", "n_gpus": 1, "steps": n,
        "warmup": args.warmup, "ms_per_step": round(ms / n, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": STREAM_WORKLOAD % (alpha, sigma), "layers": L, "slots_per_layer": STREAM_SLOTS,
                   "zipf_s": STREAM_ZIPF, "zipf_alpha": alpha, "logit_noise_sigma": sigma, "repeat_p": 0.5,
                   "repeat_bonus": 30.0, "cache_metadata": "device", "fetch_ctas": args.fetch_ctas,
                   "l2": "no flush: every step streams 1.1 GB of resident shared/router weights plus the cached "
                         "experts, far above the 126 MB L2"},
        "hit_rate": round(timed_d["hits"] / max(1, lookups), 4),
        "bytes_fetched_per_token": int(timed_d["bytes"] / n),
        "roofline": {"bound": "host_link", "achieved": round(fetch_gbs, 2), "peak": round(probe, 2), "unit": "GB/s",
                     "frac": round(fetch_gbs / probe, 4),
                     "peak_source": "pinned host->device copy probe in the same run (32 x 3.36 MB)", "traffic": None},
        "stall_us_per_token": round(meas_d["stall_ms"] * 1000.0 / max(1, meas_d["tokens"]), 1),
        "copy_gbs_during_fills": round(meas_d["bytes"] / max(1e-9, meas_d["copy_ms"] / 1000.0) / 1e9, 2),
        "shared_branch_us_per_token": round(meas_d["shared_ms"] * 1000.0 / max(1, meas_d["tokens"]), 1),
        "measured_steps_for_stall": meas_steps,
        "host_metadata": host_points,
        "kernels": {k: {"event_ms_total": round(v[0], 4), "launches": int(v[1])} for k, v in prof.items() if v[1]},
        "gpu_launches": int(n * L * 6),    # router, shared gate/up and down, LFU, fetch, routed gate/up, routed down
        "clocks": clocks,
        "e2e": {"value": round(e2e_steps / e2e_s, 2), "unit": "tok/s", "h2d_bytes_per_step": H * 2,
                "d2h_bytes_per_step": H * 2},
    }
    if sweep_out:
        line["slot_sweep"] = sweep_out
    if fetch_sweep:
        line["fetch_sweep"] = fetch_sweep
    if chunked:
        line["chunked_prefill"] = chunked
    line["host"] = host_info()
    if not args.no_cpu_baseline:
        base = oracle_baseline(args.oracle_layers)
        line["cpu_baseline"] = {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")}
    return line


# ------------------------------------------------------------------ batched decode (64 tokens per step)

BATCH_T, BATCH_SEED = 64, 3
BATCH_METRIC = "batched MoE decode tok/s, 64 tokens per step (1 B300)"
BATCH_WORKLOAD = ("30-layer MoE-only stack, 64 tokens per step (x ~ N(0,1) [64, 2816] at step 0, the outputs fed back), "
                  "uniform routing (no bias), H=2816, 128 experts of I=704 (int4 g64, fp16 scale+bias), top-8; routed "
                  "experts by grouped dequant-to-16-bit tcgen05 GEMMs (fp16 gate/up, bf16 down), the bf16 shared "
                  "expert 2816->2112->2816 by the "
                  "same GEMM kernel; all experts resident in HBM; seed 3")
PAYLOAD = 3 * (I * H // 2 + I * (H // 64) * 4)       # 3,345,408 B per expert
# kernels behind one profiling bracket of a batched layer step: rms, histogram, positions, inverse init, two
# gathers and the shared plan; four GEMMs and the two split-K sums of the shared expert (64 tokens fit one tile)
BATCH_KERNELS_PER_BRACKET = {"router": 1, "permute": 7, "gemm": 6, "combine": 1}


def batched_cpu_baseline(seed, x_bits, n_tokens=2):
    """The oracle (tensor-core reading, with the shared expert) on n_tokens tokens of layer 0: routing, 8 experts
    and the shared expert; tok/s over 30 layers."""
    import oracle as O
    import workload as W
    O.build()
    shared = W.shared_weights(seed, 0, H, S)
    Wr = W.router_weights(seed, 0, E, H)
    elapsed = 0.0
    for t in range(n_tokens):
        idx = O.route(x_bits[t], Wr, None, K_ACT)[2]
        experts = W.experts_parallel(seed, 0, idx, H, I)   # generation is not timed
        t0 = time.perf_counter()
        r, _, idx, w = O.route(x_bits[t], Wr, None, K_ACT)
        O.layer_combine(x_bits[t], r, experts, w, shared, tc=True)
        elapsed += time.perf_counter() - t0
    return {"value": n_tokens / (elapsed * L), "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": "%d tokens of layer 0 at step 0 (router, 8 experts and the shared expert each), single-threaded "
                      "fp32 C oracle in its tensor-core reading; tok/s = tokens / (30 x their layer time)" % n_tokens}


def run_batched(args):
    import torch
    import bit_expert_streaming_layer_b300 as B
    from workload.model import SyntheticStack, bf16_bits, hidden_tensor

    seed, T = BATCH_SEED, BATCH_T
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stack = SyntheticStack(seed, L, H=H, I=I, E=E, k=K_ACT, S=S, resident=True, T_max=T, device=dev)
    stream = torch.cuda.current_stream(dev)
    x0 = hidden_tensor(seed, 0, T, H, device=dev)
    bufs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    bufs[0].copy_(x0)

    def step(src, dst, st):
        x = src
        for l in range(L):
            y = dst if l == L - 1 else bufs[2 + l % 2]
            B.tf_layer_step(stack.layers[l], None, l, 0, None, x, y, T, None, 0, st)
            x = y

    cur, nxt = 0, 1
    for _ in range(args.warmup):
        step(bufs[cur], bufs[nxt], stream)
        cur, nxt = nxt, cur
    torch.cuda.synchronize()
    # per-kernel times: a few plain steps with every launch bracketed by events
    prof_steps = min(args.steps, 8)
    prof_cap = prof_steps * L           # timed brackets per kind: one per layer of each profiled step
    B.tf_profile_begin(prof_cap)
    for _ in range(prof_steps):
        step(bufs[cur], bufs[nxt], stream)
        cur, nxt = nxt, cur
    torch.cuda.synchronize()
    prof = B.tf_profile_end()
    # the step as two CUDA graphs (one per direction of the ping-pong buffers): a batched layer step
    # enqueues no host synchronisation, so the whole 30-layer step is captured once and replayed
    graphs = None
    if not args.no_graph:
        try:
            cap = torch.cuda.Stream(dev)
            graphs = [torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()]
            for i in range(2):
                with torch.cuda.graph(graphs[i], stream=cap):
                    step(bufs[i], bufs[1 - i], torch.cuda.current_stream(dev))
            torch.cuda.synchronize()
            bufs[0].copy_(x0)
            for i in range(2):       # first replays upload the graphs: keep them out of the timed region
                graphs[i].replay()
            torch.cuda.synchronize()
        except RuntimeError as e:
            print("CUDA graph capture failed (%s); timing plain launches" % e, file=sys.stderr)
            graphs = None
    cur, nxt = 0, 1
    sampler = ClockSampler(0)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        if graphs is not None:
            graphs[cur].replay()
        else:
            step(bufs[cur], bufs[nxt], stream)
        cur, nxt = nxt, cur
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    assert not torch.isnan(bufs[cur].float()).any(), "NaN in the stack output"

    # census (untimed): distinct experts per layer on one more step -> algorithmic bytes
    distinct = []
    x = bufs[cur]
    for l in range(L):
        y = bufs[2 + l % 2]
        B.tf_layer_step(stack.layers[l], None, l, 0, None, x, y, T, None, 0, stream)
        idx = stack.layers[l].routing_tensors(T)[0]
        distinct.append(int(torch.unique(idx).numel()))
        x = y
    torch.cuda.synchronize()
    layer_bytes = [d * PAYLOAD + SHARED_GU + SHARED_D for d in distinct]
    step_bytes = sum(layer_bytes) + L * ROUTER

    # end to end: the 64 inputs from pinned host memory and the 64 outputs back, every step
    hx = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    hy = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    hx.copy_(x0.cpu())
    e2e_steps = min(args.steps, 32)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        bufs[0].copy_(hx, non_blocking=True)
        if graphs is not None:
            graphs[0].replay()
        else:
            step(bufs[0], bufs[1], stream)
        hy.copy_(bufs[1], non_blocking=True)
        stream.synchronize()
        hx.copy_(hy)
    e2e_s = time.perf_counter() - t0
    x_bits = bf16_bits(x0)
    stack.close()

    peak, peak_kind = peaks()
    gemm_ms, gemm_n = prof["gemm"]
    gemm_brackets = min(gemm_n, prof_cap)    # one bracket = the four GEMM launches of one layer
    gemm_avg_s = gemm_ms / max(1, gemm_brackets) / 1000.0
    mean_layer_bytes = sum(layer_bytes) / L
    gemm_gbs = mean_layer_bytes / gemm_avg_s / 1e9
    n = args.steps
    line = {
        "metric": BATCH_METRIC, "value": round(T * n / (ms / 1000.0), 1), "unit": "tok/s", "n_gpus": 1, "steps": n,
        "warmup": args.warmup, "ms_per_step": round(ms / n, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": BATCH_WORKLOAD, "layers": L, "tokens_per_step": T, "cuda_graph": graphs is not None,
                   "l2": "no flush: each step streams about %.1f GB of weights, far above the 126 MB L2"
                         % (step_bytes / 1e9)},
        "distinct_experts_per_layer": round(sum(distinct) / L, 1),
        "weight_bytes_per_step": step_bytes,
        "weight_gbs": round(step_bytes / (ms / n / 1000.0) / 1e9, 1),
        "roofline": {"bound": "hbm", "kernel": "gemm", "achieved": round(gemm_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gemm_gbs / peak, 4), "peak_source": peak_kind + " (hbm_gbs)",
                     "bytes_per_launch": int(mean_layer_bytes),
                     "launch": "the four GEMM launches of one layer (routed gate/up, down; shared gate/up, down)",
                     "traffic": None},
        "kernels": {k: {"event_ms_total": round(v[0], 4), "brackets": int(v[1]), "timed_brackets": min(int(v[1]), prof_cap),
                        "avg_us": round(v[0] / max(1, min(v[1], prof_cap)) * 1000.0, 2)}
                    for k, v in prof.items() if v[1]},
        "gpu_launches": int(n * L * sum(BATCH_KERNELS_PER_BRACKET.values())),   # kernels of the timed steps
        "clocks": clocks,
        "e2e": {"value": round(T * e2e_steps / e2e_s, 1), "unit": "tok/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = batched_cpu_baseline(seed, x_bits)
    return line


# ------------------------------------------------------------------ prefill-shaped layer (grouped path)

PREFILL_T = 4096
PREFILL_FLOP = 2 * PREFILL_T * K_ACT * (2 * I * H + H * I)   # 389.8 GFLOP: gate/up + down GEMMs
PREFILL_WORKLOAD = ("prefill-shaped MoE layer: 4096 tokens x H=2816, 128 experts of I=704 (int4 g64, fp16 scale+bias), "
                    "top-8 of router logits + Zipf(1.2) popularity bias, grouped dequant-to-16-bit tcgen05 GEMMs "
                    "(fp16 gate/up, bf16 down) with "
                    "fp32 accumulation, weighted combine; seed 4")


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured (bf16_tflops, burst)"
    return 1800.0, "fallback"


def prefill_cpu_baseline(seed, x_bits, idx, w, n_tokens=2):
    """The oracle (tensor-core reading) on n_tokens tokens of the layer; tok/s."""
    import oracle as O
    import workload as W
    O.build()
    elapsed = 0.0
    for t in range(n_tokens):
        experts = W.experts_parallel(seed, 0, idx[t], H, I)   # generation is not timed
        t0 = time.perf_counter()
        r = O.rms_scale(x_bits[t])
        O.layer_combine(x_bits[t], r, experts, w[t], None, tc=True)
        elapsed += time.perf_counter() - t0
    return {"value": n_tokens / elapsed, "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": "%d of the 4096 tokens (all 8 experts each), single-threaded fp32 C oracle in its "
                      "tensor-core reading; expert generation not timed" % n_tokens}


def run_prefill(args):
    import torch
    import bit_expert_streaming_layer_b300 as B
    import workload as W
    from workload.model import _u16_to_bf16_tensor, bf16_bits, hidden_tensor, pack_layer_experts

    seed, T = 4, PREFILL_T
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    slot = B.tf_expert_slot_bytes(H, I)
    host = torch.empty(E * slot, dtype=torch.uint8, pin_memory=True)
    pack_layer_experts(seed, 0, E, H, I, host)
    experts = host.to(dev)
    table = B.expert_table(experts, slot)
    Wr = _u16_to_bf16_tensor(W.router_weights(seed, 0, E, H)).to(dev)
    bias = torch.from_numpy(W.zipf_bias(seed, 0, E, 1.2)[0]).to(dev)
    x = hidden_tensor(seed, 0, T, H, device=dev)
    out = torch.empty_like(x)
    idx = torch.empty(T, K_ACT, dtype=torch.int32, device=dev)
    w = torch.empty(T, K_ACT, dtype=torch.float32, device=dev)
    rws = torch.zeros(B.tf_router_workspace_bytes(T, E), dtype=torch.uint8, device=dev)
    gws = torch.zeros(B.tf_moe_grouped_workspace_bytes(T, H, I, E, K_ACT), dtype=torch.uint8, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        B.tf_router_topk(x, T, H, Wr, E, bias, 0, K_ACT, idx, w, None, None, rws, rws.numel(), stream)
        B.tf_moe_ffn_grouped(x, out, T, table, E, idx, w, K_ACT, H, I, None, None, counts, gws, gws.numel(), stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    B.tf_profile_begin(args.steps)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    prof = B.tf_profile_end()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    gemm_ms = prof["gemm"][0] / max(1, min(prof["gemm"][1], args.steps))
    peak, peak_kind = tensor_peak()
    achieved = PREFILL_FLOP / (gemm_ms / 1e3) / 1e12
    cnt = counts.cpu().numpy()
    # end to end: host tokens in, host outputs back, every step
    hx = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    hy = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    hx.copy_(x.cpu())
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x.copy_(hx, non_blocking=True)
        step()
        hy.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    line = {
        "metric": "prefill-shaped MoE layer tok/s (1 B300)", "value": round(T / (ms / 1e3), 1), "unit": "tok/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": PREFILL_WORKLOAD, "tokens": T, "l2": "inputs 0.4 GB of experts + 0.6 GB workspace, "
                   "far above the 126 MB L2"},
        "roofline": {"bound": "tensor", "kernel": "gemm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "flop_per_launch_pair": PREFILL_FLOP, "traffic": None},
        "kernels": {k: {"event_ms_total": round(v[0], 4), "launches": int(v[1])} for k, v in prof.items() if v[1]},
        "expert_load": {"max_tokens": int(cnt.max()), "experts_used": int((cnt > 0).sum())},
        "gpu_launches": int(sum(v[1] for v in prof.values())),
        "clocks": clocks,
        "e2e": {"value": round(T / e2e_s, 1), "unit": "tok/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(seed, bf16_bits(x), idx.cpu().numpy(), w.cpu().numpy())
    return line


ATTN_SHAPE = dict(H=2816, nq=16, nkv=8, d=128)
ATTN_CTX = 4096          # cached positions before the decoded token
ATTN_LAYERS = 4          # distinct layers cycled through, so that weights and caches exceed the L2


def run_attention(args):
    """The attention half of a decoder layer (tf_attn_decode): one decode token at position ATTN_CTX over a
    filled FP16 KV cache, 16 q heads and 8 kv heads of 128 (synthetic Gemma-like shape; the pages give none).
    Steps cycle through ATTN_LAYERS layers with their own weights and caches (about 270 MB in all). The
    roofline counts the step's algorithmic bytes: the four weight matrices once (bf16) plus the K and V rows
    0..pos of the layer's kv heads (fp16)."""
    import torch
    import bit_expert_streaming_layer_b300 as B
    import workload as W

    sh = ATTN_SHAPE
    Hh, nq, nkv, d = sh["H"], sh["nq"], sh["nkv"], sh["d"]
    pos, max_seq = ATTN_CTX, ATTN_CTX + 1
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def dev16(a):
        return torch.from_numpy(a.reshape(-1).view("int16")).to(dev)

    layers = []
    for l in range(ATTN_LAYERS):
        ws = [dev16(m) for m in W.attention_weights(7, l, Hh, nq, nkv, d)]
        desc = B.attn_desc(Hh, nq, nkv, d, max_seq, *ws)
        k, v = W.cache_rows(7, l, pos, nkv, d)
        kc = torch.zeros(B.tf_attn_cache_bytes(desc) // 2, dtype=torch.int16, device=dev)
        vc = torch.zeros_like(kc)
        kc[:k.size] = dev16(k)
        vc[:v.size] = dev16(v)
        layers.append((desc, ws, kc, vc))
    wsb = B.tf_attn_workspace_bytes(layers[0][0])
    wsp = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    x = dev16(W.hidden(7, 0, 1, Hh)[0])
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        desc, _, kc, vc = layers[i % ATTN_LAYERS]
        B.tf_attn_decode(desc, x, out, pos, kc, vc, wsp, wsb, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    weight_bytes = (nq * d * Hh + 2 * nkv * d * Hh + Hh * nq * d) * 2
    cache_bytes = 2 * (pos + 1) * nkv * d * 2
    step_bytes = weight_bytes + cache_bytes
    peak, peak_kind = peaks()
    achieved = step_bytes / (ms / 1e3) / 1e9
    # end to end: the token's x in from pinned host memory and out back, every step
    hx = torch.empty(Hh, dtype=torch.int16, pin_memory=True)
    hy = torch.empty(Hh, dtype=torch.int16, pin_memory=True)
    hx.copy_(x.cpu())
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        x.copy_(hx, non_blocking=True)
        step(i)
        hy.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    return {
        "metric": "attention half of a decoder layer, decode tok/s (1 B300)", "value": round(1e3 / ms, 1),
        "unit": "tok/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "attention decode, H=2816, 16 q / 8 kv heads of 128, position 4096 over a filled "
                   "FP16 KV cache", "l2": "4 layers cycled, %.0f MB of weights and caches" %
                   (ATTN_LAYERS * (weight_bytes + 2 * max_seq * nkv * d * 2) / 1e6)},
        "roofline": {"bound": "hbm", "kernel": "attention step (4 launches)", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": peak_kind + " (hbm_gbs)", "bytes_per_step": step_bytes, "traffic": None},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "e2e": {"value": round(1.0 / e2e_s, 1), "unit": "tok/s", "h2d_bytes_per_step": Hh * 2,
                "d2h_bytes_per_step": Hh * 2},
    }


def run_reference(args):
    """The CPU oracle, as it stands (single-threaded fp32 C), on the decode workload. One step of this arm is one
    layer of the stack: step s runs layer s mod 30 on the previous step's output (the token's layers in order, the
    last layer's output feeding the next token's first layer), so that W + K steps are a bounded sample that ends
    in well under a minute. tok/s = 1 / (30 x the mean measured layer time)."""
    import oracle as O
    import workload as W
    O.build()
    x = W.hidden(SEED, 0, 1, H)[0]
    times = []
    for s in range(args.warmup + args.steps):
        x, dt = _oracle_layer(O, W, x, s % L, False)
        if s >= args.warmup:
            times.append(dt)
    layer_s = float(np.mean(times))
    value = 1.0 / (L * layer_s)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(layer_s * 1000.0, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": L,
                       "step": "one layer of the 30-layer stack (1/30 of a token), outputs fed forward; "
                               "tok/s = 1 / (30 x mean layer time); weight generation not timed"},
            "step_time": spread([t * 1000.0 for t in times]),
            "host": host_info(),
            "cpu_baseline": {"value": round(value, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": "%d layer steps after %d warm-up layer steps of the decode stack, seed %d, "
                                       "single-threaded fp32 C oracle" % (args.steps, args.warmup, SEED)},
            "e2e": {"value": round(value, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["fused", "layers"], default="fused",
                    help="fused: one persistent kernel per step; layers: three kernels per layer")
    ap.add_argument("--profile-steps", type=int, default=64,
                    help="timed steps whose kernels are bracketed by CUDA events (the first ones)")
    ap.add_argument("--oracle-layers", type=int, default=6)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefetch", action="store_true",
                    help="fused path: prefetch the next layer's shared weights into L2 (measured slower)")
    ap.add_argument("--workload", choices=["decode", "prefill", "streaming", "batched", "attention"], default="decode",
                    help="decode: the 30-layer decode stack (the headline line); prefill: the 4096-token grouped "
                         "layer; streaming: the decode stack through the 16-slot LFU cache with a host store; "
                         "batched: the stack with 64 tokens per step; attention: the attention half of a "
                         "decoder layer (RoPE, FP16 KV cache) at position 4096")
    ap.add_argument("--alpha", type=float, default=STREAM_ALPHA,
                    help="streaming: scale of the Zipf(1.1) router bias")
    ap.add_argument("--no-graph", action="store_true",
                    help="batched: time plain launches instead of replaying the step as a CUDA graph")
    ap.add_argument("--slot-sweep", default="",
                    help="streaming: also measure these slot counts per layer, e.g. 8,32,64")
    ap.add_argument("--fetch-ctas", type=int, default=32,
                    help="streaming: CTAs of the kernel that copies missing experts from the host store")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="default (decode) run: skip the short batched / prefill / streaming runs reported beside it")
    ap.add_argument("--no-chunked-prefill", action="store_true",
                    help="streaming: skip the chunked prefill through the cache")
    ap.add_argument("--fetch-sweep", default="",
                    help="streaming: also measure these fetch-kernel widths, e.g. 8,16,64")
    ap.add_argument("--noise", type=float, default=STREAM_NOISE,
                    help="streaming: sigma of the per-(step, layer) router-logit noise")
    ap.add_argument("--layers", type=int, default=L,
                    help="stack depth; the benchmark workload is 30, fewer only for small profiling captures")
    args = ap.parse_args()
    set_layers(args.layers)
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args)
        return

    if args.workload == "prefill":
        if rank == 0:
            print(json.dumps(run_prefill(args)))
        return
    if args.workload == "streaming":
        if rank == 0:
            print(json.dumps(run_streaming(args)))
        return
    if args.workload == "batched":
        if rank == 0:
            print(json.dumps(run_batched(args)))
        return
    if args.workload == "attention":
        if rank == 0:
            print(json.dumps(run_attention(args)))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")

    ms, prof, clocks, launches, e2e_s, e2e_steps, step_ms = run_ours(args, rank, world)
    if rank != 0:
        return
    tok_s = world * args.steps / (ms / 1000.0)
    ms_step = ms / args.steps
    peak, peak_kind = peaks()
    # dominant kernel: largest summed event time among the timed launches
    timed = {k: v for k, v in prof.items() if v[1] > 0}
    cap = min(args.steps, args.profile_steps) * (1 if args.path == "fused" else L)
    dom = max(timed, key=lambda k: timed[k][0])
    dom_ms, dom_n = timed[dom]
    n_timed = min(dom_n, cap)
    avg_s = dom_ms / n_timed / 1000.0
    achieved = BYTES[dom] / avg_s / 1e9
    per_kernel = {k: {"event_ms_total": round(v[0], 4), "launches": int(v[1]),
                      "timed_launches": int(min(v[1], cap)),
                      "avg_us": round(v[0] / max(1, min(v[1], cap)) * 1000, 3),
                      "bytes_per_launch": BYTES.get(k)} for k, v in timed.items()}
    expert_gbs = ROUTED_PER_TOKEN * args.steps / (ms / 1000.0) / 1e9
    line = {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": L, "batch": 1, "steps_fed_back": args.steps, "path": args.path,
                   "l2_prefetch": args.path == "fused" and args.prefetch,
                   "l2": "no flush: each step streams 1.895 GB of weights, 15x the 126 MB L2",
                   "parallelism": "replicas" if world > 1 else "single"},
        "expert_weight_gbs": round(expert_gbs, 1),
        "expert_weight_frac_of_peak": round(expert_gbs / peak, 4),
        "weight_gbs": round(WEIGHTS_PER_TOKEN * args.steps / (ms / 1000.0) / 1e9, 1),
        "weight_frac_of_peak": round(WEIGHTS_PER_TOKEN * args.steps / (ms / 1000.0) / 1e9 / peak, 4),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind + " (hbm_gbs)",
                     "bytes_per_launch": BYTES[dom],
                     "traffic": fused_traffic(L) if (dom == "layer" and args.path == "fused") else None,
                     "traffic_source": "not measured in this run: ncu DRAM read + write bytes of one launch of this "
                                       "kernel's code on a 4-layer stack, scaled by L / 4 (null once the code "
                                       "changes)"},
        "kernels": per_kernel,
        "step_time": spread(step_ms),
        "gpu_launches": int(launches),
        "clocks": clocks,
        "host": host_info(),
        "e2e": {"value": round(world * e2e_steps / e2e_s, 2), "unit": "tok/s", "h2d_bytes_per_step": H * 2,
                "d2h_bytes_per_step": H * 2},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["cpu_baseline_all_cores"] = cpu_baselines(args.oracle_layers)
    if world == 1 and not args.no_other_workloads:
        line["other_workloads"] = other_workloads(args)
    print(json.dumps(line))


def other_workloads(args):
    """Short runs of the batched, prefill and streaming workloads in the same process (fewer steps than their own
    --workload lines), summarised beside the decode line so that every workload has a number from this run."""
    import copy
    out = {}
    plans = (("batched", run_batched, 16, 3), ("prefill", run_prefill, 5, 3), ("streaming", run_streaming, 6, 3),
             ("attention", run_attention, 64, 8))
    for name, fn, steps, warmup in plans:
        a = copy.copy(args)
        a.steps, a.warmup, a.no_cpu_baseline, a.workload = steps, warmup, True, name
        a.slot_sweep, a.fetch_sweep = "", ""
        t0 = time.perf_counter()
        try:
            ln = fn(a)
        except Exception as e:   # one workload failing must not hide the decode line
            out[name] = {"error": "%s: %s" % (type(e).__name__, e)}
            continue
        keep = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "e2e", "hit_rate",
                "bytes_fetched_per_token", "distinct_experts_per_layer", "chunked_prefill", "host_metadata")
        summary = {k: ln[k] for k in keep if k in ln}
        rf = ln.get("roofline", {})
        summary["roofline"] = {k: rf[k] for k in ("bound", "kernel", "achieved", "peak", "unit", "frac") if k in rf}
        summary["clocks"] = ln.get("clocks")
        summary["wall_s"] = round(time.perf_counter() - t0, 1)
        out[name] = summary
    return out


if __name__ == "__main__":
    main()
