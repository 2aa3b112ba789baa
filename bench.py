"""Decode benchmark of the per-head windowed KV path on GB300.

One step = one decode step of the whole hot path over every global layer: append the new
token's K/V into each head's ring, then split-K windowed attention for every query head
(by default through hwkv_append_decode_attn, one launch per layer; ``--path split`` calls
hwkv_append and hwkv_decode_attn separately).  Inputs are synthetic (seeded N(0,1), shapes of the chosen workload)
and already resident in HBM when the timed region starts; the prefill is materialised
into the pool before timing (its bandwidth is reported separately).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload full] [--impl hwkv|reference]

Prints one JSON line on rank 0.  Under torchrun (N > 1) every rank runs an independent
replica of the workload on its own GPU (the path has no exchange step); value is the
tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and resident-KV HBM GB/s (fraction of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per decode launch from one ncu capture of the
# stream-K decode kernel, with the sha256 of its sources (hwkv_decode_tc.cu, then
# hwkv_decode_tile.cuh) it was taken on.  When the kernel source changes the figure no longer
# applies and is reported as null.
DECODE_TRAFFIC = {"source_sha256": "1c00563c90368234af1ad9540ba43971664c11ae329c77154a06aa51d334f0e1",
                  "bytes_per_launch": (621.369856 + 2.454272 + 489.221632 + 0.178432) / 2 * 1e6,
                  "launch": "layers 0 and 1 of the full workload (2-layer run, same per-launch shape)"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------------------------
# distributed helpers (replicas only)
# --------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(local_ms: float, local_units: float, world_size: int):
    """(max time over ranks in ms, total units over ranks); needs an initialised process
    group when world_size > 1."""
    if world_size == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world_size: int):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.5)
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        picked = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.15 <= t <= self.t1 + 0.15]
        if not picked:
            picked = [l for (_, l) in self.lines]
        for line in picked:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": float(np.median(power)) if power else None}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def decode_source_sha() -> str:
    h = hashlib.sha256()
    for name in ("hwkv_decode_tc.cu", "hwkv_decode_tile.cuh"):
        with open(os.path.join(ROOT, "head_budgeted_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# --------------------------------------------------------------------------------------
# algorithmic bytes
# --------------------------------------------------------------------------------------
def attention_bytes(cfg, layer: int, lens) -> int:
    """Resident K and V bytes one decode launch of ``layer`` must read (each once), plus
    q read and out written: sum_s sum_h min(w, len_s) * 2 * D * eb + 2 * B * Hq * D * eb."""
    w = np.asarray(cfg.windows[layer], dtype=np.int64)
    lens = np.asarray(lens, dtype=np.int64)
    kv = int(np.minimum(w[None, :], lens[:, None]).sum()) * 2 * cfg.head_dim * cfg.elem_bytes
    return kv + 2 * cfg.batch * cfg.q_heads * cfg.head_dim * cfg.elem_bytes


def append_bytes(cfg) -> int:
    """Read k_new, v_new and write them into the pool: 2 * (B * H * 2 * D * eb)."""
    return 2 * cfg.batch * cfg.kv_heads * 2 * cfg.head_dim * cfg.elem_bytes


def mean_step_bytes(cfg, first_step: int, steps: int) -> float:
    """Algorithmic bytes of one decode step (all layers), averaged over the given steps."""
    total = 0
    for k in range(steps):
        lens = [cfg.prefill[s] + first_step + k + 1 for s in range(cfg.batch)]
        total += sum(attention_bytes(cfg, l, lens) for l in range(cfg.layers))
    return total / steps + cfg.layers * append_bytes(cfg)


def materialize_bytes(cfg, layer: int) -> int:
    w = np.asarray(cfg.windows[layer], dtype=np.int64)
    L = np.asarray(cfg.prefill, dtype=np.int64)
    return 2 * int(np.minimum(w[None, :], L[:, None]).sum()) * 2 * cfg.head_dim * cfg.elem_bytes


def bench_config(cfg, args, world_size: int, step_bytes=None) -> dict:
    """The ``config`` object of the JSON line; identical for both arms."""
    c = {"workload": workload_desc(cfg), "global_batch": cfg.batch * world_size, "seq_len": max(cfg.prefill),
         "parallelism": "replicas" if world_size > 1 else "single",
         "path": args.path + (" (CUDA graph per step)" if args.graph else ""),
         "kernel": ["auto", "tensor", "simt"][args.kernel],
         "workers": args.workers or "auto", "split_tokens": args.split or "auto",
         "early_reads": args.path == "fused" and not args.no_early_reads}
    if step_bytes is None:
        step_bytes = mean_step_bytes(cfg, args.warmup, args.steps)
    c["l2"] = f"inputs larger than L2: {step_bytes / 1e9:.2f} GB of resident KV read per step"
    return c


def workload_desc(cfg) -> str:
    lens = sorted(set(cfg.prefill))
    ctx = f"ctx {lens[0]}" if len(lens) == 1 else f"ctx {min(lens)}..{max(lens)}"
    return (f"{cfg.name}: {cfg.layers} global layers x {cfg.kv_heads} KV heads, {cfg.q_heads} q heads, "
            f"D{cfg.head_dim}, {cfg.dtype}, block {cfg.block_size}, batch {cfg.batch}, {ctx}, per-head windows "
            f"{sorted(set(int(x) for r in cfg.windows for x in r))}")


# --------------------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of one decode step
# --------------------------------------------------------------------------------------
def oracle_sample(cfg, wl, budget_s: float, device, layers_order=None, step: int = 0, max_layers=None):
    """Times the oracle on whole layers of decode step ``step`` until ``budget_s`` seconds
    of oracle time are spent.  When one pass over the layers would take less than the budget,
    each layer's computation is timed ``reps`` times (from the first layer's time) on the same
    host copy of its windows, so the sample still spends about the budget without drawing the
    windows again.  Returns (seconds, layer evaluations, threads, layers done, reps)."""
    import math
    import oracle
    import workloads
    threads = oracle.default_threads()
    reps = 1
    st_in = wl.step_inputs(step, "cpu") if step == 0 else None
    steps = [(None, st_in[1], st_in[2])] if st_in is not None else None
    spent, done = 0.0, 0
    order = layers_order or list(range(cfg.layers))
    for l in order:
        if max_layers is not None and done >= max_layers:
            break
        hist = {}
        for s in range(cfg.batch):
            k, v = wl.prefill_seq(l, s, device)
            L = cfg.prefill[s]
            for h in range(cfg.kv_heads):
                lo, hi = oracle.window_span(L + step + 1, int(cfg.windows[l][h]))
                hk, hv = wl.history(l, s, h, lo, hi, prefill=(k, v), steps=steps)
                hist[(s, h)] = (lo, hk, hv)
            del k, v
        q = workloads.to_raw(st_in[0][l])
        lens = [cfg.prefill[s] + step + 1 for s in range(cfg.batch)]
        for r in range(reps if done > 0 else 1):
            t0 = time.perf_counter()
            oracle.attention_jobs(q, hist, lens, cfg.windows[l], cfg.scale, threads=threads)
            spent += time.perf_counter() - t0
        if done == 0:  # repetitions per layer for about the budget over one pass
            reps = min(8, max(1, math.ceil(budget_s / max(spent * len(order), 1e-9))))
            for r in range(reps - 1):
                t0 = time.perf_counter()
                oracle.attention_jobs(q, hist, lens, cfg.windows[l], cfg.scale, threads=threads)
                spent += time.perf_counter() - t0
        done += 1
        if spent >= budget_s:
            break
    return spent, done * reps, threads, done, reps


# --------------------------------------------------------------------------------------
# reference arm: the oracle timed on the host cores
# --------------------------------------------------------------------------------------
def oracle_whole_step(cfg, wl, step: int, steps_in, device, threads: int) -> float:
    """Seconds of fp64 oracle time for every layer (all sequences and query heads) of decode
    step ``step``; ``steps_in`` holds the host inputs of steps 0 .. step (the appended tokens
    are part of the windows).  The host copies of each layer's windows are drawn untimed."""
    import oracle
    import workloads
    lens = [cfg.prefill[s] + step + 1 for s in range(cfg.batch)]
    spent = 0.0
    for l in range(cfg.layers):
        hist = {}
        for s in range(cfg.batch):
            k, v = wl.prefill_seq(l, s, device)
            for h in range(cfg.kv_heads):
                lo, hi = oracle.window_span(lens[s], int(cfg.windows[l][h]))
                hk, hv = wl.history(l, s, h, lo, hi, prefill=(k, v), steps=steps_in)
                hist[(s, h)] = (lo, hk, hv)
            del k, v
        q = workloads.to_raw(steps_in[step][0][l])
        t0 = time.perf_counter()
        oracle.attention_jobs(q, hist, lens, cfg.windows[l], cfg.scale, threads=threads)
        spent += time.perf_counter() - t0
    return spent


def run_reference(args, cfg):
    """The reference arm: the fp64 oracle on the host cores, K whole decode steps (every layer,
    sequence and query head of steps W .. W+K-1), each timed; the W warm-up steps run layer 0
    of steps 0 .. W-1 untimed."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import torch
    import oracle
    import workloads
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = workloads.Workload(cfg, device="cpu" if cfg.single_cpu_stream or device.type == "cpu" else device)
    threads = oracle.default_threads()
    total = args.warmup + args.steps
    steps_in = [tuple(t.cpu() for t in wl.step_inputs(i, device)) for i in range(total)]
    one_layer = cfg.with_layers(1)
    for i in range(args.warmup):
        oracle_whole_step(one_layer, wl, i, steps_in, device, threads)
    times = [oracle_whole_step(cfg, wl, args.warmup + k, steps_in, device, threads) for k in range(args.steps)]
    step_s = float(np.mean(times))
    value = cfg.batch / step_s
    sample = (f"{args.steps} whole decode steps (all {cfg.layers} layers x {cfg.batch} seqs x {cfg.q_heads} q heads, "
              f"full resident windows), each timed; {sum(times):.1f} s of fp64 oracle time on {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(cfg, args, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------------------
def run_hwkv(args, cfg):
    import torch
    import workloads
    import head_budgeted_kv_gb300 as hw

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    hw.binding.load()
    stream = torch.cuda.current_stream(dev)

    total = args.warmup + args.steps
    wl = workloads.Workload(cfg, device="cpu" if cfg.single_cpu_stream else dev)
    pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                   cfg.torch_dtype, q_heads=cfg.q_heads, device=dev)
    if args.split or args.kernel or args.workers:
        pool.set_decode_config(args.split, args.kernel, args.workers)
    fused = args.path == "fused"

    # ---- materialise every layer from a contiguous full prefill (timed per launch) ----
    prefill = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    mat_ms, mat_bytes = 0.0, 0
    for l in range(cfg.layers):
        K, V = wl.prefill_layer(l, dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pool.materialize(l, K, V, prefill)
        e1.record(stream)
        e1.synchronize()
        mat_ms += e0.elapsed_time(e1)
        mat_bytes += materialize_bytes(cfg, l)
        del K, V
    torch.cuda.synchronize()

    # ---- per-step inputs, drawn up front (resident before timing) ----
    # steps: warm-up, timed pass, kernel-timing pass, e2e pass (positions keep advancing)
    n_steps = total + 2 * args.steps
    qs, kns, vns = [], [], []
    for i in range(n_steps):
        q, kn, vn = wl.step_inputs(i, dev)
        qs.append(q)
        kns.append(kn)
        vns.append(vn)
    outs = torch.empty((cfg.layers, cfg.batch, cfg.q_heads, cfg.head_dim), dtype=cfg.torch_dtype, device=dev)
    pos_all = [(prefill + i).contiguous() for i in range(n_steps)]
    lens_all = [(prefill + i + 1).contiguous() for i in range(n_steps)]
    torch.cuda.synchronize()

    graph = None
    launches_per_step = None
    if args.graph:
        from head_budgeted_kv_gb300.graph import DecodeStepGraph
        before = hw.binding.hwkv_kernel_launches()
        graph = DecodeStepGraph(pool, cfg.scale, cfg.q_heads, pos_all[0], fused=fused)
        launches_per_step = hw.binding.hwkv_kernel_launches() - before  # kernels recorded per step

    early = fused and not args.no_early_reads
    # Warm-up and timed steps of the fused path go through prepared launches (arguments checked
    # and marshalled before timing): the loop then issues one ctypes call per layer, ~8 us of host
    # time against 20-100 us of kernel, so the host never lets the GPU run dry.  The e2e pass
    # below uses the plain per-call API.
    launchers = None
    if fused and graph is None:
        launchers = [[pool.decode_launch(l, qs[i][l], cfg.scale, pos_all[i], outs[l], kns[i][l], vns[i][l],
                                         early_reads=early) for l in range(cfg.layers)]
                     for i in range(args.warmup + args.steps)]

    def run_step(i, ev=None):
        if graph is not None and ev is None:
            # the step's inputs land in the graph's static buffers; positions advance in-graph
            graph.q.copy_(qs[i], non_blocking=True)
            graph.k_new.copy_(kns[i], non_blocking=True)
            graph.v_new.copy_(vns[i], non_blocking=True)
            graph.replay()
            return
        if launchers is not None and ev is None and i < len(launchers):
            for launch in launchers[i]:
                launch()
            return
        for l in range(cfg.layers):
            if fused:
                if ev is not None:
                    ev[l][0].record(stream)
                # positions are prepared before the timed region and this layer's pool was last
                # written a step ago: the schedule may start before the previous launch ends
                pool.append_decode(l, qs[i][l], cfg.scale, kns[i][l], vns[i][l], pos_all[i], out=outs[l],
                                   early_reads=early)
            else:
                pool.append(l, kns[i][l], vns[i][l], pos_all[i])
                if ev is not None:
                    ev[l][0].record(stream)
                pool.decode(l, qs[i][l], cfg.scale, lens_all[i], out=outs[l])
            if ev is not None:
                ev[l][1].record(stream)

    # the measured loops issue short launches back to back: a collector pause on the host thread
    # would let the GPU run dry, so the collector stays off until the e2e pass is done
    gc.collect()
    gc.disable()
    for i in range(args.warmup):
        run_step(i)
    torch.cuda.synchronize()
    bits = pool.check_device_errors()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} during warm-up")

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = hw.binding.hwkv_kernel_launches()
    barrier(ws)
    torch.cuda.synchronize()
    clocks.mark_start()
    t_start.record(stream)
    for k in range(args.steps):
        run_step(args.warmup + k)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(ws)
    launches = hw.binding.hwkv_kernel_launches() - launches0
    if graph is not None:
        launches = launches_per_step * args.steps
    clock_info = clocks.stop() if rank == 0 else None
    local_ms = t_start.elapsed_time(t_end)
    bits = pool.check_device_errors()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in the timed region")

    # algorithmic bytes of the timed steps (resident K/V + q + out, plus the appends)
    step_bytes = mean_step_bytes(cfg, args.warmup, args.steps)

    # ---- dominant kernel, per launch: the same steps again with events around each launch
    # of the decode kernel (fused: the whole per-layer step; split: decode only) ----
    step_events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(cfg.layers)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        run_step(total + k, step_events[k])
    torch.cuda.synchronize()
    dec_ms, dec_bytes = 0.0, 0
    for k in range(args.steps):
        i = total + k
        lens = [cfg.prefill[s] + i + 1 for s in range(cfg.batch)]
        for l in range(cfg.layers):
            dec_ms += step_events[k][l][0].elapsed_time(step_events[k][l][1])
            dec_bytes += attention_bytes(cfg, l, lens) + (append_bytes(cfg) if fused else 0)
    n_dec = args.steps * cfg.layers
    # the decode kernel's bytes over the timed steps themselves
    timed_dec_bytes = 0
    for k in range(args.steps):
        lens = [cfg.prefill[s] + args.warmup + k + 1 for s in range(cfg.batch)]
        timed_dec_bytes += sum(attention_bytes(cfg, l, lens) + (append_bytes(cfg) if fused else 0)
                               for l in range(cfg.layers))

    # ---- e2e: host (pinned) inputs in, host outputs back, every step ----
    e2e_total = args.steps
    e2e0 = total + args.steps
    h_q = [qs[e2e0 + k].cpu().pin_memory() for k in range(e2e_total)]
    h_k = [kns[e2e0 + k].cpu().pin_memory() for k in range(e2e_total)]
    h_v = [vns[e2e0 + k].cpu().pin_memory() for k in range(e2e_total)]
    h_pos = [pos_all[e2e0 + k].cpu().pin_memory() for k in range(e2e_total)]
    h_out = torch.empty(outs.shape, dtype=outs.dtype).pin_memory()
    # two device sets of inputs and outputs: step k + 1's inputs arrive and step k's outputs
    # leave on a copy stream while the other set is computed on
    d_in = [(torch.empty_like(qs[0]), torch.empty_like(kns[0]), torch.empty_like(vns[0]), torch.empty_like(prefill))
            for _ in range(2)]
    d_outs = [outs, torch.empty_like(outs)]
    d_lens = torch.empty_like(prefill)
    cs = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step on set b computed (inputs read, outputs written)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of set b on the host
    h2d = (h_q[0].numel() * h_q[0].element_size() + h_k[0].numel() * h_k[0].element_size() * 2
           + h_pos[0].numel() * 4)
    d2h = h_out.numel() * h_out.element_size()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def send_inputs(k):
        # step k's inputs into set k % 2, once the step that last read that set has run
        b = k % 2
        with torch.cuda.stream(cs):
            if k >= 2:
                cs.wait_event(ev_done[b])
            for dst, src in zip(d_in[b], (h_q[k], h_k[k], h_v[k], h_pos[k])):
                dst.copy_(src, non_blocking=True)
            ev_in[b].record(cs)

    e0.record(stream)
    if graph is None:
        cs.wait_event(e0)  # every copy lies inside the timed region
        send_inputs(0)
    for k in range(e2e_total):
        if graph is not None:
            graph.q.copy_(h_q[k], non_blocking=True)
            graph.k_new.copy_(h_k[k], non_blocking=True)
            graph.v_new.copy_(h_v[k], non_blocking=True)
            graph.pos.copy_(h_pos[k], non_blocking=True)
            graph.replay()
            h_out.copy_(graph.out, non_blocking=True)
            continue
        b = k % 2
        if k + 1 < e2e_total:
            send_inputs(k + 1)
        d_q, d_k, d_v, d_pos = d_in[b]
        d_out = d_outs[b]
        stream.wait_event(ev_in[b])  # a full dependency: the kernels below start after the copy
        if k >= 2:
            stream.wait_event(ev_out[b])  # set b's previous outputs are on the host
        if fused:
            for l in range(cfg.layers):
                pool.append_decode(l, d_q[l], cfg.scale, d_k[l], d_v[l], d_pos, out=d_out[l], early_reads=early)
        else:
            pool.advance_positions(d_pos, out=d_lens)
            for l in range(cfg.layers):
                pool.append(l, d_k[l], d_v[l], d_pos)
                pool.decode(l, d_q[l], cfg.scale, d_lens, out=d_out[l])
        ev_done[b].record(stream)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[b])
            h_out.copy_(d_out, non_blocking=True)
            ev_out[b].record(cs)
    if graph is None:
        stream.wait_event(ev_out[(e2e_total - 1) % 2])  # the last step's outputs are on the host
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = e0.elapsed_time(e1)
    gc.enable()
    bits = pool.check_device_errors()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in the e2e pass")

    max_ms, units = aggregate(local_ms, cfg.batch * args.steps, ws)
    e2e_max_ms, e2e_units = aggregate(e2e_ms, cfg.batch * e2e_total, ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        spent, evals, threads, done, reps = oracle_sample(cfg, wl, budget_s=args.cpu_budget, device=dev)
        step_s = spent / evals * cfg.layers
        cpu = {"value": cfg.batch / step_s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} of {cfg.layers} layers (all seqs and q heads) of decode step 0, each timed "
                         f"{reps}x, {spent:.1f} s of fp64 oracle time; per-step time = time per layer "
                         f"evaluation x {cfg.layers}"}

    pool_nbytes = pool.nbytes
    use_graph = graph is not None
    pool.close()
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    secondary = None
    if args.secondary and ws == 1:
        # the headline workload's buffers go first: the ragged pool alone is 91 GB
        del pool, graph, qs, kns, vns, outs, launchers, d_in, d_outs, h_q, h_k, h_v, h_out
        gc.collect()
        torch.cuda.empty_cache()
        secondary = secondary_block(args, dev, stream, peak)
    isolated = dec_bytes / (dec_ms / 1e3) / 1e9  # launches separated by events: no overlap
    if fused and not use_graph:
        # every launch of the timed region is the decode kernel: its average duration there is
        # the timed region over the launches (consecutive launches overlap by design)
        achieved = timed_dec_bytes / (local_ms / 1e3) / 1e9
        how = "average over the launches of the timed region (CUDA events around it)"
    else:
        achieved = isolated
        how = "events around each launch in a separate pass of the same steps"
    sha = decode_source_sha()
    # the DRAM counters were taken on the full workload's fused launches: they describe no other
    # workload's launches
    traffic = (DECODE_TRAFFIC["bytes_per_launch"]
               if DECODE_TRAFFIC["source_sha256"] == sha and cfg.name.split("_")[0] == "full" and fused else None)
    value = units / (max_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": bench_config(cfg, args, ws, step_bytes),
        "resident_kv_gbs": step_bytes / (max_ms / args.steps / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": ("fused append + split-K decode attention" if fused else "split-K decode attention")
                               + " (one launch per layer)",
                     "duration": how,
                     "bytes_per_launch": timed_dec_bytes / n_dec,
                     "ms_per_launch": timed_dec_bytes / n_dec / achieved / 1e6,
                     "isolated_launch": {"achieved": isolated, "frac": isolated / peak, "ms": dec_ms / n_dec}},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_units / (e2e_max_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clock_info,
        "materialize": {"gbs": mat_bytes / (mat_ms / 1e3) / 1e9, "ms": mat_ms, "bytes": mat_bytes,
                        "frac": mat_bytes / (mat_ms / 1e3) / 1e9 / peak},
        "pool_bytes": pool_nbytes,
        "secondary": secondary,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------
# secondary workloads of the default line: short timed regions in the same run
# --------------------------------------------------------------------------------------
SECONDARY = ("ragged", "long", "long_full")


def measure_secondary(name: str, args, dev, stream, peak: float) -> dict:
    """Materialises workload ``name`` into its own pool and times ``steps`` fused decode steps
    (every layer, prepared launches with early reads, as the headline line) after ``warmup``
    untimed ones.  The pool and inputs are freed before returning."""
    import torch
    import workloads
    import head_budgeted_kv_gb300 as hw
    cfg = workloads.config(name)
    warmup = args.warmup
    steps = max(1, min(args.steps, cfg.steps - warmup))
    wl = workloads.Workload(cfg, device=dev)
    pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                   cfg.torch_dtype, q_heads=cfg.q_heads, device=dev)
    prefill = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    for l in range(cfg.layers):
        K, V = wl.prefill_layer(l, dev)
        pool.materialize(l, K, V, prefill)
        del K, V
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    total = warmup + steps
    inputs = [wl.step_inputs(i, dev) for i in range(total)]
    pos_all = [(prefill + i).contiguous() for i in range(total)]
    outs = torch.empty((cfg.layers, cfg.batch, cfg.q_heads, cfg.head_dim), dtype=cfg.torch_dtype, device=dev)
    launchers = [[pool.decode_launch(l, inputs[i][0][l], cfg.scale, pos_all[i], outs[l], inputs[i][1][l],
                                     inputs[i][2][l], early_reads=True) for l in range(cfg.layers)]
                 for i in range(total)]
    torch.cuda.synchronize()
    for i in range(warmup):
        for launch in launchers[i]:
            launch()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = hw.binding.hwkv_kernel_launches()
    clocks.mark_start()
    e0.record(stream)
    for i in range(warmup, total):
        for launch in launchers[i]:
            launch()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    launches = hw.binding.hwkv_kernel_launches() - launches0
    clock_info = clocks.stop()
    ms = e0.elapsed_time(e1)
    bits = pool.check_device_errors()
    pool.close()
    del pool, inputs, pos_all, outs, launchers
    torch.cuda.empty_cache()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in the {name} workload")
    step_bytes = mean_step_bytes(cfg, warmup, steps)
    gbs = step_bytes / (ms / steps / 1e3) / 1e9
    return {"workload": workload_desc(cfg), "steps": steps, "warmup": warmup, "ms_per_step": ms / steps,
            "tokens_per_s": cfg.batch * steps / (ms / 1e3), "bytes_per_step": step_bytes, "resident_kv_gbs": gbs,
            "frac": gbs / peak, "peak": peak, "gpu_launches": launches, "clocks": clock_info}


def secondary_block(args, dev, stream, peak: float) -> dict:
    out = {}
    for name in args.secondary:
        out[name] = measure_secondary(name, args, dev, stream, peak)
    if "long" in out and "long_full" in out:
        w, f = out["long"], out["long_full"]
        out["long_full"]["vs_long"] = {"bytes_ratio": f["bytes_per_step"] / w["bytes_per_step"],
                                       "tokens_per_s_ratio": w["tokens_per_s"] / f["tokens_per_s"]}
    return out


# --------------------------------------------------------------------------------------
# decode by shape: the full geometry's first 8 layers at other head dims, groups and dtypes
# --------------------------------------------------------------------------------------
SHAPES = (("bf16 D128 GQA4", {}), ("bf16 D128 GQA8", {"q_heads": 64}), ("bf16 D128 GQA16", {"q_heads": 128}),
          ("bf16 D64 GQA4", {"head_dim": 64}), ("bf16 D64 GQA8", {"head_dim": 64, "q_heads": 64}),
          ("bf16 D64 GQA16", {"head_dim": 64, "q_heads": 128}), ("fp32 D128 GQA4", {"dtype": "f32"}),
          ("fp32 D64 GQA4", {"dtype": "f32", "head_dim": 64}))


def run_shapes(args):
    """Fused append + decode, prepared launches with early reads, on the full workload's first 8
    layers (batch 4, 112K) for each shape of SHAPES: resident-KV GB/s over W warm-up and K timed
    steps.  Prints one JSON line."""
    import dataclasses
    import torch
    import workloads
    import head_budgeted_kv_gb300 as hw
    dev = torch.device("cuda", 0)
    hw.binding.load()
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peak()
    rows = []
    for label, kw in SHAPES:
        if args.shape and args.shape != label:
            continue
        cfg = dataclasses.replace(workloads.config("full").with_layers(8), name="full_8l", **kw)
        wl = workloads.Workload(cfg, device=dev)
        pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                       cfg.torch_dtype, q_heads=cfg.q_heads, device=dev)
        prefill = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
        for l in range(cfg.layers):
            K, V = wl.prefill_layer(l, dev)
            pool.materialize(l, K, V, prefill)
            del K, V
        total = args.warmup + args.steps
        inputs = [wl.step_inputs(i, dev) for i in range(total)]
        pos = [(prefill + i).contiguous() for i in range(total)]
        outs = torch.empty((cfg.layers, cfg.batch, cfg.q_heads, cfg.head_dim), dtype=cfg.torch_dtype, device=dev)
        launches = [[pool.decode_launch(l, inputs[i][0][l], cfg.scale, pos[i], outs[l], inputs[i][1][l],
                                        inputs[i][2][l], early_reads=True) for l in range(cfg.layers)]
                    for i in range(total)]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(total):
            if i == args.warmup:
                e0.record(stream)
            for launch in launches[i]:
                launch()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        bits = pool.check_device_errors()
        pool.close()
        del pool, wl, inputs, pos, outs, launches
        torch.cuda.empty_cache()
        if bits:
            raise RuntimeError(f"device error bits {bits:#x} for {label}")
        nbytes = mean_step_bytes(cfg, args.warmup, args.steps)
        gbs = nbytes / (ms / 1e3) / 1e9
        rows.append({"shape": label, "ms_per_step": ms, "resident_kv_gbs": gbs, "frac": gbs / peak})
    print(json.dumps({"metric": "fused decode resident-KV GB/s by shape (full geometry, first 8 layers)",
                      "unit": "GB/s", "peak": peak, "peak_kind": peak_kind, "steps": args.steps,
                      "warmup": args.warmup, "shapes": rows}), flush=True)


# --------------------------------------------------------------------------------------
# chunked prefill (hwkv_prefill_attn): not the default line
# --------------------------------------------------------------------------------------
def prefill_flops(cfg, layer: int, pos0, n: int) -> int:
    """Algorithmic FLOPs of one prefill launch: every query head of every chunk token does
    2*D (QK) + 2*D (PV) per key of its window [max(0, p+1-w), p]."""
    total = 0
    G, D = cfg.group, cfg.head_dim
    for s in range(cfg.batch):
        for h in range(cfg.kv_heads):
            w = int(cfg.windows[layer][h])
            p = np.arange(int(pos0[s]), int(pos0[s]) + n, dtype=np.int64)
            total += int(np.minimum(w, p + 1).sum()) * G * 4 * D
    return total


def prefill_oracle_sample(cfg, wl, n_chunk: int, budget_s: float):
    """Times the fp64 oracle's chunked prefill on the first tokens of sequence 0's chunk in
    layer 0 (each token attends to its full window: the prior context and the chunk rows before
    it) until ``budget_s`` seconds are spent.  Returns (seconds, tokens, threads)."""
    import numpy as np
    import oracle
    import workloads
    threads = oracle.default_threads()
    l, s = 0, 0
    p0 = cfg.prefill[s]
    k, v = wl.prefill_seq(l, s, "cpu")
    q, kc, vc = wl.chunk_inputs(l, 0, n_chunk, "cpu")
    spent, done, batch = 0.0, 0, 8
    while spent < budget_s and done < n_chunk:
        m = min(batch, n_chunk - done)
        hist = {}
        for h in range(cfg.kv_heads):
            lo = max(0, p0 + done + 1 - int(cfg.windows[l][h]))
            hk = np.concatenate([workloads.to_raw(k[h, min(lo, p0):p0]), workloads.to_raw(kc[s, :done + m, h])])
            hv = np.concatenate([workloads.to_raw(v[h, min(lo, p0):p0]), workloads.to_raw(vc[s, :done + m, h])])
            hist[h] = (min(lo, p0), hk, hv)
        qs = workloads.to_raw(q[s, done:done + m])
        t0 = time.perf_counter()
        oracle.prefill_attention(qs, hist, p0 + done, cfg.windows[l], cfg.scale, threads=threads)
        spent += time.perf_counter() - t0
        done += m
    return spent, done, threads


def run_prefill(args, cfg):
    import torch
    import workloads
    import head_budgeted_kv_gb300 as hw
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hw.binding.load()
    stream = torch.cuda.current_stream(dev)
    wl = workloads.Workload(cfg, device=dev)
    pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                   cfg.torch_dtype, q_heads=cfg.q_heads, device=dev)
    pool.set_prefill_config(args.prefill_max_stages)
    prefill = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    for l in range(cfg.layers):
        K, V = wl.prefill_layer(l, dev)
        pool.materialize(l, K, V, prefill)
        del K, V
    n = args.chunk
    nt = torch.full((cfg.batch,), n, dtype=torch.int32, device=dev)
    chunks = [wl.chunk_inputs(l, 0, n, dev) for l in range(cfg.layers)]
    outs = [torch.empty_like(c[0]) for c in chunks]
    # a pass over every layer per step: warm-up, timed, then end-to-end steps (positions keep
    # advancing by one chunk per step)
    total = args.warmup + args.steps
    pos = [(prefill + i * n).contiguous() for i in range(total + args.steps)]
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    ms, flops, launches = 0.0, 0, 0
    gc.collect()
    gc.disable()  # no collector pause between the measured launches
    for i in range(total):
        k = i - args.warmup
        if k == 0:
            torch.cuda.synchronize()
            clocks.mark_start()
            launches0 = hw.binding.hwkv_kernel_launches()
        if k >= 0:
            ev[k][0].record(stream)
        for l in range(cfg.layers):
            q, kk, vv = chunks[l]
            pool.prefill(l, q, cfg.scale, kk, vv, pos[i], nt, out=outs[l])
        if k >= 0:
            ev[k][1].record(stream)
            flops += sum(prefill_flops(cfg, l, [cfg.prefill[s] + i * n for s in range(cfg.batch)], n)
                         for l in range(cfg.layers))
    torch.cuda.synchronize()
    clocks.mark_end()
    launches = hw.binding.hwkv_kernel_launches() - launches0
    clock_info = clocks.stop() if rank == 0 else None
    for a, b in ev:
        ms += a.elapsed_time(b)
    bits = pool.check_device_errors()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x}")

    # ---- e2e: every step's chunk inputs from pinned host memory, its outputs back; two device
    # sets, so step k + 1's inputs arrive and step k's outputs leave while the other computes ----
    h_in = [[t.cpu().pin_memory() for t in chunks[l]] for l in range(cfg.layers)]
    h_pos = [pos[total + k].cpu().pin_memory() for k in range(args.steps)]
    h_out = [torch.empty(outs[l].shape, dtype=outs[l].dtype).pin_memory() for l in range(cfg.layers)]
    d_in = [[[torch.empty_like(t) for t in chunks[l]] for l in range(cfg.layers)] for _ in range(2)]
    d_pos = [torch.empty_like(prefill) for _ in range(2)]
    d_out = [outs, [torch.empty_like(o) for o in outs]]
    cs = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for row in h_in for t in row) + cfg.batch * 4
    d2h = sum(o.numel() * o.element_size() for o in h_out)

    def send_inputs(k):
        b = k % 2
        with torch.cuda.stream(cs):
            if k >= 2:
                cs.wait_event(ev_done[b])
            for l in range(cfg.layers):
                for dst, src in zip(d_in[b][l], h_in[l]):
                    dst.copy_(src, non_blocking=True)
            d_pos[b].copy_(h_pos[k], non_blocking=True)
            ev_in[b].record(cs)

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs.wait_event(e0)  # every copy lies inside the timed region
    send_inputs(0)
    for k in range(args.steps):
        b = k % 2
        if k + 1 < args.steps:
            send_inputs(k + 1)
        stream.wait_event(ev_in[b])
        if k >= 2:
            stream.wait_event(ev_out[b])
        for l in range(cfg.layers):
            q, kk, vv = d_in[b][l]
            pool.prefill(l, q, cfg.scale, kk, vv, d_pos[b], nt, out=d_out[b][l])
        ev_done[b].record(stream)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[b])
            for l in range(cfg.layers):
                h_out[l].copy_(d_out[b][l], non_blocking=True)
            ev_out[b].record(cs)
    stream.wait_event(ev_out[(args.steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    gc.enable()
    e2e_ms = e0.elapsed_time(e1)
    bits = pool.check_device_errors()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in the e2e pass")
    pool.close()
    if rank != 0:
        return
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (burst, cuBLAS bf16)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    tflops = flops / (ms / 1e3) / 1e12
    tokens = cfg.batch * n * args.steps
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        spent, done, threads = prefill_oracle_sample(cfg, wl, n, budget_s=args.cpu_budget)
        cpu = {"value": done / (spent * cfg.layers), "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"the first {done} chunk tokens of sequence 0 in layer 0 (every query head, full windows), "
                         f"{spent:.1f} s of fp64 oracle time; per-token time scaled by {cfg.layers} layers"}
    line = {"metric": "chunked prefill tokens/s (windowed attention + ring append, all layers)",
            "value": tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": workload_desc(cfg) + f", chunk {n} tokens per sequence on top of the context",
                       "global_batch": cfg.batch, "seq_len": max(cfg.prefill),
                       "l2": "each step streams every layer's prior windows (GBs) from HBM"},
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "traffic": None, "peak_kind": kind,
                         "kernel": "prefill_kernel (tcgen05 bf16, accumulators in tensor memory) + chunk append, one pair per layer"},
            "cpu_baseline": cpu,
            "e2e": {"value": cfg.batch * n * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clock_info}
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=125)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["hwkv", "reference"], default="hwkv")
    p.add_argument("--workload", default="full")
    p.add_argument("--layers", type=int, default=0, help="keep only the first N layers (profiling)")
    p.add_argument("--split", type=int, default=0, help="CUDA-core kernel: tokens per split-K chunk")
    p.add_argument("--workers", type=int, default=0, help="tensor-core kernel: CTAs of the persistent grid")
    p.add_argument("--path", choices=["fused", "split"], default="fused")
    p.add_argument("--graph", action="store_true", help="replay each decode step as one captured CUDA graph")
    p.add_argument("--mode", choices=["decode", "prefill", "shapes"], default="decode")
    p.add_argument("--chunk", type=int, default=2048, help="prefill mode: tokens per sequence per chunk")
    p.add_argument("--shape", default="", help="shapes mode: measure only this shape (e.g. 'fp32 D128 GQA4')")
    p.add_argument("--prefill-max-stages", type=int, default=0,
                   help="prefill mode: split key streams longer than this many 64-key stages (0 = automatic)")
    p.add_argument("--kernel", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-early-reads", action="store_true",
                   help="decode without HWKV_DECODE_EARLY_READS (schedule waits for the previous launch)")
    p.add_argument("--cpu-budget", type=float, default=12.0)
    p.add_argument("--secondary", default="auto",
                   help="comma-separated workloads timed after the headline one in the same run ('none' to skip; "
                        "'auto': ragged,long,long_full for the default full-workload decode line)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    import workloads
    cfg = workloads.config(args.workload)
    if args.layers:
        cfg = cfg.with_layers(args.layers)
    if args.secondary == "auto":
        default_line = (args.workload == "full" and not args.layers and args.path == "fused" and not args.graph
                        and not args.kernel and not args.workers and not args.split and not args.no_early_reads)
        args.secondary = list(SECONDARY) if default_line else []
    elif args.secondary == "none":
        args.secondary = []
    else:
        args.secondary = [n for n in args.secondary.split(",") if n]
        for n in args.secondary:
            workloads.config(n)  # unknown names fail here
    if args.impl == "reference":
        run_reference(args, cfg)
    elif args.mode == "shapes":
        run_shapes(args)
    elif args.mode == "prefill":
        run_prefill(args, cfg)
    else:
        run_hwkv(args, cfg)


if __name__ == "__main__":
    main()
