"""Benchmark of batched paged MLA decode on GB300.

Default (N=1): the DeepSeek-V3-shaped decode (B=64, H=128, q_len=1,
576/512 dims, page_size 64, seq_lens ~ U[1024, 8192], pool 1.25x shuffled,
bf16) -- the configuration the metric is quoted on.  One "step" is one
``mla_decode_run`` (partitioner + decode + combine kernels) over that batch
with every input resident in HBM.  The other four workloads are reported
beside it in ``per_config`` (same method, fewer replays).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank decodes its own replica of the batch (the
path has no exchange step), the timed region is bracketed by a barrier and
synchronisation on both sides, and rank 0 prints one JSON line with the max
time over ranks.  ``--impl reference`` times the fp64 CPU oracle instead, on
bounded samples of the same workload, on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

METRIC = "paged MLA decode µs/call, TFLOP/s, KV GB/s and % of roofline at B=64,H=128"
HEADLINE = "deepseek_v3"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)


# ----------------------------------------------------------------- work model

def work_model(w) -> dict:
    """Algorithmic FLOPs and bytes of one decode call on workload ``w``.

    FLOPs: 2 * H * (576 + 512) per visible (query row, KV row) pair; visible
    pairs n_vis = sum_b sum_{i<q} (L - q + i + 1) (causal) or q * L (dense),
    or, under sparse top-k, the usable list entries of every token.
    Bytes: KV rows read once + Q + O (+ LSE) + page-table/length metadata;
    under sparse top-k the distinct listed rows of each request, the lists
    and the page-table entries of the pages they touch.
    """
    q = w.q_lens.astype(np.int64)
    L = w.seq_lens.astype(np.int64)
    H = w.num_heads
    tokens = int(q.sum())
    e = 1 if w.kv_dtype == "e4m3" else 2
    if w.sparse_idx is not None:
        qs = w.q_start()
        n_vis = rows = pages = 0
        for b in range(w.batch):
            lists = w.sparse_idx[int(qs[b]):int(qs[b + 1])]
            usable = lists[(lists >= 0) & (lists < L[b])]
            n_vis += int(usable.size)
            uniq = np.unique(usable)
            rows += int(uniq.size)
            pages += int(np.unique(uniq // w.page_size).size)
        kv_bytes = rows * 576 * e
        meta = pages * 4 + int(w.sparse_idx.size) * 4
    else:
        if w.causal:
            n_vis = int(np.sum(q * (L - q) + q * (q + 1) // 2))
        else:
            n_vis = int(np.sum(q * L))
        kv_bytes = int(L.sum()) * 576 * e
        meta = int(((L + w.page_size - 1) // w.page_size).sum()) * 4
    total = (kv_bytes + tokens * H * 576 * 2 + tokens * H * 512 * 2
             + (tokens * H * 4 if w.return_lse else 0)
             + meta + 4 * w.batch + (4 * (w.batch + 1) if w.packed else 0))
    return {"flops": 2 * H * (576 + 512) * n_vis, "bytes": total, "kv_bytes": kv_bytes,
            "n_vis": n_vis, "tokens": tokens}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def roofline(w, wm, seconds, peaks):
    tensor_peak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if w.kv_dtype == "e4m3" else 1.0)
    t_mem = wm["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_ten = wm["flops"] / (tensor_peak * 1e12)
    bound = "hbm" if t_mem >= t_ten else "tensor"
    if bound == "hbm":
        achieved = wm["bytes"] / seconds / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    achieved = wm["flops"] / seconds / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": achieved / tensor_peak}


def make_workload(name):
    return mi.WORKLOADS[name]()


def wmx_flops(w) -> int:
    return work_model(w)["flops"]


# ----------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks / throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            mx = smax
            sms.append(sm)
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s in sms if s >= 0.5 * (mx or max(sms))] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ----------------------------------------------------------------- CPU oracle

def time_oracle(w, target_s: float, seed: int = 0, max_pairs: int = 1 << 20):
    """Time the fp64 oracle on a seeded sample of (token, head) pairs sized to
    about ``target_s`` seconds.  Returns (TFLOP/s, seconds, pairs, cores, flops)."""
    import oracle
    rng = np.random.default_rng(seed)
    qs = w.q_start()
    tokens = int(qs[-1])
    H = w.num_heads
    order = rng.permutation(tokens * H)[:max_pairs]
    owner = np.searchsorted(qs[1:], np.arange(tokens), side="right")

    def pair_flops(idx):
        t = idx // H
        b = owner[t]
        i = t - qs[b]
        L = w.seq_lens[b].astype(np.int64)
        q = w.q_lens[b].astype(np.int64)
        if w.sparse_idx is not None:
            lists = w.sparse_idx[t]
            n = np.sum((lists >= 0) & (lists < L[:, None]), axis=1)
        else:
            n = (L - q + i + 1) if w.causal else L
        return int(np.sum(2 * (576 + 512) * n))

    cores = oracle.default_threads()
    n = min(len(order), 4 * cores)
    sel = np.stack([order[:n] // H, order[:n] % H], axis=1)
    t0 = time.perf_counter()
    oracle.run(w, sel=sel, n_threads=cores)
    dt = time.perf_counter() - t0
    n2 = int(min(len(order), max(n, n * target_s / max(dt, 1e-6))))
    sel = np.stack([order[:n2] // H, order[:n2] % H], axis=1)
    t0 = time.perf_counter()
    oracle.run(w, sel=sel, n_threads=cores)
    dt = time.perf_counter() - t0
    fl = pair_flops(order[:n2])
    return fl / dt / 1e12, dt, n2, cores, fl


# ----------------------------------------------------------------- GPU arm

def to_device(w, dev):
    import torch
    q = torch.from_numpy(w.query.view(np.int16)).to(dev).view(torch.bfloat16)
    if w.kv_dtype == "bf16":
        kv = torch.from_numpy(w.kv_cache.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        kv = torch.from_numpy(w.kv_cache).to(dev).view(torch.float8_e4m3fn)
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    qo = torch.from_numpy(w.qo_indptr).to(dev) if w.packed else None
    return q, kv, bt, sl, qo


def sparse_lists(w, dev):
    import torch
    return torch.from_numpy(w.sparse_idx).to(dev) if w.sparse_idx is not None else None


def gpu_case(w, dev, steps, warmup, with_e2e):
    """Time ``steps`` decode calls; returns a dict of measurements."""
    import torch
    import paged_mla_decode_03_gb300 as mla

    q, kv, bt, sl, qo = to_device(w, dev)
    tokens = w.total_q
    plan = mla.Plan(batch=w.batch, num_heads=w.num_heads, max_seq_len_q=w.max_seq_len_q,
                    max_seq_len=w.max_seq_len, page_size=w.page_size,
                    max_pages_per_req=w.block_tables.shape[1], num_pages=w.num_pages,
                    packed=w.packed, max_total_q=tokens, kv_dtype=w.kv_dtype, causal=w.causal,
                    return_lse=w.return_lse, device=dev.index or 0, sparse_top_k=w.sparse_k)
    sp = sparse_lists(w, dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((tokens, w.num_heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((tokens, w.num_heads), dtype=torch.float32, device=dev) if w.return_lse else None
    stream = torch.cuda.Stream(device=dev)
    total_q = tokens if w.packed else 0

    def step(prof=None):
        mla.mla_decode_run_profiled(plan.handle, q, kv, bt, sl, qo, total_q, w.bmm1_scale,
                                    w.bmm2_scale, out, lse, ws, None, stream, prof,
                                    sparse_indices=sp)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    # The timed steps run as CUDA graphs of `steps` calls (how a serving loop
    # issues decode).  Two graphs: plain calls (their replay gives the time per
    # call) and calls with an event pair around each decode kernel (their replay
    # gives the kernel's duration for the roofline; event-record nodes between
    # the kernels cost ~10 us of their own, so they stay out of the per-call
    # figure).  Each graph is replayed once untimed, then once timed.
    # The profiled graph holds at least 200 calls (its untimed replay is the
    # warm-up), so the kernel figure is a median over >= 200 calls whatever
    # `steps` is.
    n_prof = max(steps, 200)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_prof)]
    g_plain, g_prof, g_one = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=stream):
        for k in range(steps):
            step()
    with torch.cuda.graph(g_prof, stream=stream):
        for k in range(n_prof):
            step(ev[k])
    with torch.cuda.graph(g_one, stream=stream):
        step()

    def timed(graph):
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        with torch.cuda.stream(stream):
            graph.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return start.elapsed_time(end)

    total_ms = timed(g_plain)
    prof_total_ms = timed(g_prof)
    kernel_ms = [a.elapsed_time(b) for a, b in ev]
    # Per-call median: a one-call graph replayed 20 times untimed, then
    # n_prof times back to back with an event between consecutive replays.
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_prof + 1)]
    with torch.cuda.stream(stream):
        for _ in range(20):
            g_one.replay()
        for k in range(n_prof):
            marks[k].record(stream)
            g_one.replay()
        marks[n_prof].record(stream)
    stream.synchronize()
    call_ms = [marks[k].elapsed_time(marks[k + 1]) for k in range(n_prof)]
    del g_plain, g_prof, g_one
    res = {"ms_per_step": total_ms / steps, "kernel_ms": statistics.mean(kernel_ms),
           "kernel_ms_median": statistics.median(kernel_ms),
           "call_ms_median": statistics.median(call_ms), "n_median": n_prof,
           "ms_per_step_with_events": prof_total_ms / steps,
           "launches_per_step": mla.mla_decode_kernels_per_run(plan.handle)}

    if with_e2e:
        # end to end through the public API with host buffers: per-step inputs
        # (query + metadata) copied host->device from pinned memory by the
        # library, results copied back.
        hq = q.cpu().pin_memory()
        hbt = bt.cpu().pin_memory()
        hsl = sl.cpu().pin_memory()
        hqo = qo.cpu().pin_memory() if qo is not None else None
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory() if lse is not None else None
        h2d = sum(t.numel() * t.element_size() for t in (hq, hbt, hsl, hqo) if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in (hout, hlse) if t is not None)

        staging = torch.empty(plan.staging_bytes(total_q), dtype=torch.uint8, device=dev)

        def e2e_step():
            # the C ABI's host-buffer entry: it copies the step's inputs in,
            # decodes, and copies the results out, all on `stream`
            plan.run_host(hq, kv, hbt, hsl, hout, staging=staging, workspace=ws, h_qo_indptr=hqo,
                          total_q=total_q, h_lse=hlse, bmm1_scale=w.bmm1_scale,
                          bmm2_scale=w.bmm2_scale, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(warmup):
                e2e_step()
            stream.synchronize()
            s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize(dev)
            s2.record(stream)
            for _ in range(steps):
                e2e_step()
            e2.record(stream)
            torch.cuda.synchronize(dev)
            barrier()
        res["e2e_ms"] = s2.elapsed_time(e2) / steps
        res["h2d_bytes"] = h2d
        res["d2h_bytes"] = d2h
    plan.close()
    del q, kv, bt, sl, qo, ws, out, lse, sp
    torch.cuda.empty_cache()
    return res


def load_traffic():
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary,
    or {} when the kernel source changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    src = os.path.join(ROOT, "paged_mla_decode_03_gb300", "csrc", "mla_decode_sm103.cu")
    try:
        with open(path) as f:
            d = json.load(f)
        with open(src, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
        return d if d.get("kernel_source_sha256_16") == h else {}
    except Exception:
        return {}


def run_gpu(args):
    import torch
    ws_, rank = dist_init("nccl")
    _, _, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    import paged_mla_decode_03_gb300 as mla
    mla.load_library()

    w = make_workload(args.workload)
    wm = work_model(w)
    # the host-buffer entry point has no sparse top-k form
    with_e2e = w.sparse_idx is None
    with ClockSampler(local) as clk:
        r = gpu_case(w, dev, args.steps, args.warmup, with_e2e=with_e2e)
    step_s = reduce_max(r["ms_per_step"] / 1e3, dev)
    kern_s = reduce_max(r["kernel_ms_median"] / 1e3, dev)
    kern_mean_s = reduce_max(r["kernel_ms"] / 1e3, dev)
    call_med_s = reduce_max(r["call_ms_median"] / 1e3, dev)
    e2e_s = reduce_max(r["e2e_ms"] / 1e3, dev) if with_e2e else None
    ev_s = reduce_max(r["ms_per_step_with_events"] / 1e3, dev)
    n = ws_
    value = n * wm["flops"] / step_s / 1e12
    rf = roofline(w, wm, kern_s, peaks)
    tr = load_traffic().get(w.name)
    rf["traffic"] = tr.get("bytes_per_launch") if tr else None
    rf["peak_source"] = peaks["source"]
    step_rf = roofline(w, wm, step_s, peaks)

    def oracle_line(wx, seconds):
        tf, dt, pairs, cores, fl = time_oracle(wx, target_s=seconds)
        return {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "us_per_call": wmx_flops(wx) / (tf * 1e12) * 1e6 if tf > 0 else None,
                "sample": f"{pairs} (token, head) pairs of {wx.name} drawn with seed 0, "
                          f"{fl / 1e9:.2f} GFLOP in {dt:.1f} s (fp64 C oracle, all pairs' "
                          f"visible KV rows)"}

    per_config = []
    if not args.no_extra:
        for name in [n for n in mi.WORKLOADS if n != args.workload]:
            wx = make_workload(name)
            wmx = work_model(wx)
            rx = gpu_case(wx, dev, max(5, args.steps // 4), max(3, args.warmup), with_e2e=False)
            tx = reduce_max(rx["call_ms_median"] / 1e3, dev)
            kx = reduce_max(rx["kernel_ms_median"] / 1e3, dev)
            rfx = roofline(wx, wmx, tx, peaks)
            rkx = roofline(wx, wmx, kx, peaks)
            entry = {
                "workload": wx.name, "us_per_call": tx * 1e6, "decode_kernel_us": kx * 1e6,
                "median_of_calls": rx["n_median"],
                "tflops": wmx["flops"] / tx / 1e12, "kv_gbs": wmx["kv_bytes"] / tx / 1e9,
                "bound": rfx["bound"], "roofline_frac": rfx["frac"],
                "kernel_roofline_frac": rkx["frac"], "dtype": wx.kv_dtype}
            if rank == 0 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = oracle_line(wx, args.cpu_seconds_extra)
            per_config.append(entry)
            del wx

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_line(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "num_heads": w.num_heads,
                       "q_len": int(w.q_lens[0]), "page_size": w.page_size,
                       "seed": w.seed, "kv_dtype": w.kv_dtype,
                       "parallelism": f"replicas x{n}",
                       "l2": "inputs larger than L2 (KV pool > 129 MB), no flush",
                       "timing": "CUDA graph of `steps` plain calls, replayed warm then timed "
                                 "(value, ms_per_step); a graph of max(steps, 200) calls with an "
                                 "event pair around each decode kernel, replayed warm then timed "
                                 "(roofline: median kernel time); a one-call graph replayed 20 "
                                 "times untimed then max(steps, 200) times with an event between "
                                 "calls (us_per_call_median)"},
            "us_per_call": step_s * 1e6,
            "us_per_call_median": call_med_s * 1e6,
            "decode_kernel_us": kern_s * 1e6,
            "decode_kernel_us_mean": kern_mean_s * 1e6,
            "median_of_calls": r["n_median"],
            "us_per_call_with_kernel_events": ev_s * 1e6,
            "kv_gbs": wm["kv_bytes"] / step_s / 1e9,
            "roofline_frac_per_call": step_rf["frac"],
            "roofline": rf,
            "e2e": {"value": n * wm["flops"] / e2e_s / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d_bytes"], "d2h_bytes_per_step": r["d2h_bytes"],
                    "us_per_call": e2e_s * 1e6} if with_e2e else None,
            "gpu_launches": r["launches_per_step"] * args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "per_config": per_config,
            "work": {"flops": wm["flops"], "bytes": wm["bytes"], "kv_bytes": wm["kv_bytes"]},
        }
        print(json.dumps(line), flush=True)


def run_profile_target(args):
    """Plain eager calls of one workload and nothing else: the command the
    ncu captures under profiles/ run (no graphs, no timing, no oracle)."""
    import torch
    import paged_mla_decode_03_gb300 as mla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mla.load_library()
    w = make_workload(args.workload)
    q, kv, bt, sl, qo = to_device(w, dev)
    tokens = w.total_q
    plan = mla.Plan(batch=w.batch, num_heads=w.num_heads, max_seq_len_q=w.max_seq_len_q,
                    max_seq_len=w.max_seq_len, page_size=w.page_size,
                    max_pages_per_req=w.block_tables.shape[1], num_pages=w.num_pages,
                    packed=w.packed, max_total_q=tokens, kv_dtype=w.kv_dtype, causal=w.causal,
                    return_lse=w.return_lse, device=0, sparse_top_k=w.sparse_k)
    sp = sparse_lists(w, dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((tokens, w.num_heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((tokens, w.num_heads), dtype=torch.float32, device=dev) if w.return_lse else None
    for _ in range(args.warmup + args.steps):
        plan.run(q, kv, bt, sl, out, qo_indptr=qo, total_q=tokens if w.packed else 0, lse=lse,
                 workspace=ws, bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale,
                 sparse_indices=sp)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item())
    print(json.dumps({"profile_target": w.name, "calls": args.warmup + args.steps,
                      "launches_per_call": mla.mla_decode_kernels_per_run(plan.handle),
                      "status_word": status}), flush=True)
    if status != 0:
        raise SystemExit(f"device status word {status}")


def run_reference(args):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    w = make_workload(args.workload)
    per_step = []
    tf_last = None
    for k in range(args.warmup + args.steps):
        tf, dt, pairs, cores, fl = time_oracle(w, target_s=args.ref_step_seconds, seed=k)
        if k >= args.warmup:
            per_step.append((tf, dt, pairs, fl))
        tf_last = (pairs, cores)
    tf = sum(p[3] for p in per_step) / sum(p[1] for p in per_step) / 1e12
    step_ms = 1e3 * statistics.mean(p[1] for p in per_step)
    sample = (f"per step ~{tf_last[0]} (token, head) pairs of {w.name} (seeded), "
              f"fp64 C oracle over each pair's visible KV rows")
    line = {
        "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": w.name, "batch": w.batch, "num_heads": w.num_heads,
                   "q_len": int(w.q_lens[0]), "page_size": w.page_size, "kv_dtype": w.kv_dtype},
        "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": tf_last[1], "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--profile-target", action="store_true",
                    help="only run warmup + steps eager calls of --workload (for ncu)")
    ap.add_argument("--workload", default=HEADLINE, choices=list(mi.WORKLOADS),
                    help="workload timed for the JSON line (default: the B=64, H=128 decode)")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-config lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-seconds-extra", type=float, default=3.0,
                    help="oracle seconds per extra workload in per_config")
    ap.add_argument("--ref-step-seconds", type=float, default=5.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    if args.profile_target:
        run_profile_target(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
