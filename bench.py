"""Benchmark: fused multi-head graph-attention layer on the 1e6-node power-law
graph (Zipf(2.1) in-degrees clipped to [1,4096], mean 16; H=8, Dh=64, bf16).

One step = one gat_fused_layer call (SDDMM -> segmented softmax -> weighted
SpMM, fused; one kernel launch) over the whole graph, with the graph's
degree-bucket plan built beforehand (a plan is per graph and shared by every
layer and call on it; its build time is reported as plan_ms).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload fused|edge_softmax|aggregate|sddmm|dense|spmm_heads|
                               edge_softmax_h8|fused_backward|fused_fp8]

Prints one JSON line (rank 0). value = edge-heads/s over all ranks (each rank
runs its own full, independent problem: weak scaling, no collective on the
data path). e2e = the same metric with inputs copied from pinned host memory
and the output copied back inside the timed region. --impl reference times the
fp64 CPU oracle on bounded samples of the same workload.
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

METRIC = "edge-heads/s and achieved HBM GB/s (% of peak), fused CSR attention"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------
# distributed helpers (host logic; exercised by a gloo test on CPU)
# ----------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def relaunch_ranks(n: int) -> int:
    """Run this same command as n ranks, one per GPU of this node, under
    torch.distributed.run (rendezvous on 127.0.0.1); returns its exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def dist_barrier(dist):
    if dist is not None:
        dist.barrier()


def dist_max(dist, x: float, device=None) -> float:
    """Maximum of a float over all ranks (timing reduction only)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# peaks, clocks, profile summaries
# ----------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_ordinal: int):
        # nvidia-smi numbers GPUs physically; map the CUDA ordinal through
        # CUDA_VISIBLE_DEVICES (an index or a UUID) when it is set
        vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        self.gpu = vis[local_ordinal] if local_ordinal < len(vis) else str(local_ordinal)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash() -> str:
    """Hash of the CUDA sources of the fused kernel (to date ncu counters)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_graph_attention_head_gb300", "csrc")
    for f in ("row_engine.cuh", "fused_layer.cu", "common.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch recorded by an ncu capture of the current kernel
    source (profiles/ncu_traffic.json), scaled to the full workload; None when
    no capture matches the current source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
        e = j[kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch_full"])
    except Exception:
        return None


# ----------------------------------------------------------------------------
# L2 persistence (A/B switch; the library itself sets no access policy)
# ----------------------------------------------------------------------------
def l2_persist(torch, stream, tensors, target):
    """--l2-persist: `off` leaves the device as it is; otherwise the context's
    persisting-L2 carve-out is set to the device maximum (a per-context limit,
    gone with the process) and, unless target is `none`, an access-policy
    window (persisting hits, streaming misses, hit ratio = carve-out / window)
    is put on `stream` over tensors[target]. Returns a description."""
    if target == "off":
        return None
    import ctypes
    import glob
    libs = sorted(glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart.so*")) +
                  glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    rt = ctypes.CDLL(libs[0])

    class Window(ctypes.Structure):  # cudaStreamAttrValue.accessPolicyWindow, padded
        _fields_ = [("base_ptr", ctypes.c_void_p), ("num_bytes", ctypes.c_size_t),
                    ("hitRatio", ctypes.c_float), ("hitProp", ctypes.c_int),
                    ("missProp", ctypes.c_int), ("pad", ctypes.c_char * 40)]
    dev = torch.cuda.current_device()
    maxp, maxw = ctypes.c_int(), ctypes.c_int()
    rt.cudaDeviceGetAttribute(ctypes.byref(maxp), 108, dev)  # max persisting L2 bytes
    rt.cudaDeviceGetAttribute(ctypes.byref(maxw), 109, dev)  # max access-policy window bytes
    if rt.cudaDeviceSetLimit(6, ctypes.c_size_t(maxp.value)) != 0:  # persisting L2 limit
        raise RuntimeError("cudaDeviceSetLimit(persisting L2) failed")
    desc = {"carve_out_bytes": maxp.value, "window": target}
    if target != "none":
        if target not in tensors:
            raise ValueError(f"--l2-persist {target}: this workload has {sorted(tensors)}")
        t = tensors[target]
        w = Window()
        w.base_ptr = t.data_ptr()
        w.num_bytes = min(t.numel() * t.element_size(), maxw.value)
        w.hitRatio = min(1.0, maxp.value / w.num_bytes)
        w.hitProp, w.missProp = 2, 1  # persisting, streaming
        if rt.cudaStreamSetAttribute(ctypes.c_void_p(stream.cuda_stream), 1, ctypes.byref(w)) != 0:
            raise RuntimeError("cudaStreamSetAttribute(access policy window) failed")
        desc.update(window_bytes=w.num_bytes, hit_ratio=w.hitRatio)
    return desc


# ----------------------------------------------------------------------------
# fused workload
# ----------------------------------------------------------------------------
def fused_bytes(n_rows, n_edges, H, Dh, esize=2):
    """Algorithmic bytes of one layer under the gather model: per row, its
    row_ptr entry, q row and out row; per edge, its col_idx entry and the k
    and v rows of its source."""
    row = H * Dh * esize
    return (4 + 2 * row) * n_rows + (4 + 2 * row) * n_edges


def fused_unique_bytes(n_rows, n_src, n_edges, H, Dh, esize=2):
    row = H * Dh * esize
    return 4 * (n_rows + 1) + 4 * n_edges + 2 * row * n_rows + 2 * row * n_src


def to_dev(torch, a, dev):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16)
    t = t.to(dev)
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


def host_cpu():
    """The host's CPU model name and logical core count (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu model")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"cpu_model": model or "unknown", "nproc": os.cpu_count() or 1}


def oracle_rows_timed(d, budget_s, block, threads, start_row=0):
    """The oracle (unchanged) on consecutive row blocks until budget_s elapses,
    driven from `threads` host threads at once; each call takes its own block
    and ctypes releases the GIL for the call, so the threads run in parallel.
    Returns (edges, rows, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    rp = d["row_ptr"]
    n = rp.size - 1
    lock = threading.Lock()
    state = {"next": start_row, "edges": 0, "rows": 0}
    t0 = time.perf_counter()

    def worker():
        while time.perf_counter() - t0 < budget_s:
            with lock:
                if state["rows"] >= n:
                    return
                r = state["next"]
                state["next"] = (r + block) % n
                state["rows"] += min(n, r + block) - r
            sel = np.arange(r, min(n, r + block))
            oracle.fused_layer(rp, d["col_idx"], d["q"], d["k"], d["v"], d["H"], d["Dh"],
                               d["scale"], rows=sel)
            with lock:
                state["edges"] += int(rp[sel[-1] + 1] - rp[sel[0]])

    with ThreadPoolExecutor(threads) as ex:
        for f in [ex.submit(worker) for _ in range(threads)]:
            f.result()
    return state["edges"], state["rows"], time.perf_counter() - t0


def cpu_baseline_fused(d, budget_s=10.0, block=20000):
    """The oracle timed on the host's cores: once on one thread, once on every
    core (threads over row blocks); `value` is the all-core rate."""
    host = host_cpu()
    cores = host["nproc"]
    e1, r1, t1 = oracle_rows_timed(d, budget_s / 2, block, 1)
    ea, ra, ta = oracle_rows_timed(d, budget_s / 2, max(1000, block // 4), cores,
                                   start_row=r1 % (d["row_ptr"].size - 1))
    v1, va = e1 * d["H"] / t1, ea * d["H"] / ta
    return {"value": va, "unit": "edge-heads/s", "cores": cores, "kind": "oracle",
            "value_all_cores": va, "cores_all": cores, "value_single_thread": v1,
            "cpu_model": host["cpu_model"], "nproc": host["nproc"],
            "sample": f"all cores: {ra} rows ({ea} edges) in consecutive blocks over {cores} "
                      f"threads, {ta:.1f} s; one thread: {r1} consecutive rows ({e1} edges), "
                      f"{t1:.1f} s; fp64 C loops of the same graph"}


def spread(ms):
    """Median and 10th / 90th percentiles of per-call times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"median_ms": float(np.median(a)), "p10_ms": float(np.percentile(a, 10)),
            "p90_ms": float(np.percentile(a, 90)), "reps": int(a.size)}


def bench_fused(args, rank, world, local, dist):
    import torch
    import sparse_graph_attention_head_gb300 as gat

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t_gen = time.perf_counter()
    d = W.make_fused(seed=3, n=args.n_rows)
    t_gen = time.perf_counter() - t_gen
    n, E, H, Dh = d["n_rows"], d["n_edges"], d["H"], d["Dh"]
    rp_h, ci_h = d["row_ptr"], d["col_idx"]
    rp, ci = to_dev(torch, rp_h, dev), to_dev(torch, ci_h, dev)
    q, k, v = (to_dev(torch, d[x], dev) for x in ("q", "k", "v"))
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    # plan (per graph; timed separately)
    gat.Plan(rp)  # warm the plan kernels once
    torch.cuda.synchronize()
    tp = time.perf_counter()
    plan = gat.Plan(rp)
    plan_ms = (time.perf_counter() - tp) * 1e3
    info = plan.info()
    ws = torch.empty(max(1, gat.gat_fused_layer_workspace_size(plan, H, Dh)), dtype=torch.uint8,
                     device=dev)

    l2 = l2_persist(torch, stream, {"q": q, "k": k, "v": v}, args.l2_persist)

    def step():
        gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], out=out, plan=plan, workspace=ws,
                            stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist_barrier(dist)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for ev_a, ev_b in ev:
            ev_a.record(stream)
            step()
            ev_b.record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    dist_barrier(dist)
    torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    per_launch = [x.elapsed_time(y) for x, y in ev]
    ms_step = dist_max(dist, total_ms / args.steps, None)
    kern_ms = statistics.mean(per_launch)
    sp = spread(per_launch)

    # end to end: every step copies its inputs from pinned host memory, runs the
    # layer and copies the output back. Steps are software-pipelined over two
    # device buffer sets and three streams (host->device copies, the layer,
    # device->host copies), so step i's copies overlap steps i-1 and i+1.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(  # noqa: E731
        np.int16 if a.dtype == np.uint16 else a.dtype)).pin_memory()
    h_in = [pin(rp_h), pin(ci_h), pin(d["q"]), pin(d["k"]), pin(d["v"])]
    h_out = [torch.empty(out.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
    sets = [[rp, ci, q, k, v, out]]
    sets.append([torch.empty_like(x) for x in sets[0]])
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(n_steps):
        for i in range(n_steps):
            b = i % 2
            bufs = sets[b]
            if i >= 2:
                s_h2d.wait_event(comp_done[b])   # set b's previous layer has read its inputs
            with torch.cuda.stream(s_h2d):
                for hsrc, ddst in zip(h_in, bufs[:5]):
                    ddst.view(hsrc.dtype).copy_(hsrc, non_blocking=True)
                h2d_done[b].record(s_h2d)
            stream.wait_event(h2d_done[b])
            if i >= 2:
                stream.wait_event(d2h_done[b])   # set b's previous output has been read back
            gat.gat_fused_layer(bufs[0], bufs[1], bufs[2], bufs[3], bufs[4], d["scale"],
                                out=bufs[5], plan=plan, workspace=ws, stream=stream)
            comp_done[b].record(stream)
            s_d2h.wait_event(comp_done[b])
            with torch.cuda.stream(s_d2h):
                h_out[b].copy_(bufs[5].view(torch.int16), non_blocking=True)
                d2h_done[b].record(s_d2h)

    e2e_run(max(2, args.warmup // 2))
    torch.cuda.synchronize()
    dist_barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(4, args.steps // 4)
    e0.record(s_h2d)
    e2e_run(e2e_steps)
    s_d2h.wait_stream(stream)
    s_d2h.wait_stream(s_h2d)
    e1.record(s_d2h)
    torch.cuda.synchronize()
    dist_barrier(dist)
    e2e_ms = dist_max(dist, e0.elapsed_time(e1) / e2e_steps, None)
    e2e_ok = bool(torch.equal(h_out[(e2e_steps - 1) % 2], out.view(torch.int16).cpu()))

    hbm_peak, _, peak_kind = measured_peaks()
    alg = fused_bytes(n, E, H, Dh)
    achieved = alg / (kern_ms * 1e-3) / 1e9
    traffic = profiled_traffic("fused_engine_kernel")
    res = {
        "metric": METRIC,
        "value": world * E * H / (ms_step * 1e-3),
        "unit": "edge-heads/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step,
        "median_ms": sp["median_ms"], "p10_ms": sp["p10_ms"], "p90_ms": sp["p90_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "fused GAT layer: 1e6 rows, Zipf(2.1) in-degrees clipped to "
                               "[1,4096] rescaled to mean 16, col_idx uniform sorted in-row, "
                               "H=8, Dh=64, q/k/v bf16 N(0,1), seed 3",
                   "n_rows": n, "n_edges": E, "H": H, "Dh": Dh,
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (q/k/v 3.07 GB vs 126 MB L2), no flush",
                   "plan": info, "plan_ms": round(plan_ms, 3), "l2_persist": l2,
                   "generate_s": round(t_gen, 1)},
        "hbm_gbs": achieved,
        "hbm_frac_of_peak": achieved / hbm_peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "kernel": "fused_engine_kernel<bf16,V=2,LE=32,U=3,MINB=5>",
                     "algorithmic_bytes_per_launch": alg,
                     "kernel_ms": kern_ms, "peak_kind": f"{peak_kind} (burst copy)",
                     "unique_byte_frac": fused_unique_bytes(n, n, E, H, Dh) /
                                         (kern_ms * 1e-3) / 1e9 / hbm_peak},
        "e2e": {"value": world * E * H / (e2e_ms * 1e-3), "unit": "edge-heads/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "2 buffer sets, H2D / layer / D2H streams",
                "output_matches_device_run": e2e_ok},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    return res, d


def shard_bounds(row_begin, row_ptr, rank):
    """Rows [r0, r1) and edges [e0, e1) of a rank's row range."""
    r0, r1 = int(row_begin[rank]), int(row_begin[rank + 1])
    return r0, r1, int(row_ptr[r0]), int(row_ptr[r1])


def node_shard(n, world, rank):
    """Node rows [a, b) whose k / v a rank owns before the all-gather: equal
    contiguous blocks of ceil(n / world) rows (the last may be short)."""
    per = (n + world - 1) // world
    return min(n, rank * per), min(n, (rank + 1) * per), per


def bench_rowshard(args, rank, world, local, dist):
    """--mode rowshard: the graph's rows cut into `world` contiguous ranges of
    about equal traffic (gat_partition_rows); each rank owns the k / v rows of
    an equal node block, and one step is an all-gather of k and of v into full
    local tables, then the fused layer over the rank's own rows (the shard as
    a graph of its own: gat_rebase_row_ptr, its own plan). The whole job is one
    graph (strong scaling); value = all edge-heads / the slowest rank's step."""
    import torch
    import sparse_graph_attention_head_gb300 as gat

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = W.make_fused(seed=3, n=args.n_rows)
    n, E, H, Dh = d["n_rows"], d["n_edges"], d["H"], d["Dh"]
    rb = gat.gat_partition_rows(d["row_ptr"], world)
    r0, r1, e0, e1 = shard_bounds(rb, d["row_ptr"], rank)
    a, b, per = node_shard(n, world, rank)
    rp_all = to_dev(torch, d["row_ptr"], dev)
    rp = gat.gat_rebase_row_ptr(rp_all, r0, r1)
    ci = to_dev(torch, d["col_idx"][e0:e1], dev)
    q = to_dev(torch, d["q"][r0:r1], dev)
    kv_shard = [to_dev(torch, d[x][a:b], dev) for x in ("k", "v")]
    kv_full = [torch.empty((per * world, H, Dh), dtype=torch.bfloat16, device=dev)
               for _ in range(2 if dist is not None else 0)]
    kv_pad = [torch.zeros((per, H, Dh), dtype=torch.bfloat16, device=dev)
              for _ in range(2 if dist is not None else 0)]
    out = torch.empty_like(q)
    plan = gat.Plan(rp)
    ws = torch.empty(max(1, gat.gat_fused_layer_workspace_size(plan, H, Dh)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if dist is not None:
            for sh, pad, full in zip(kv_shard, kv_pad, kv_full):
                pad[: sh.shape[0]].copy_(sh)
                dist.all_gather_into_tensor(full, pad)
        # (one rank owns every node: its shards are the full tables)
        k, v = (kv_full[0][:n], kv_full[1][:n]) if dist is not None else kv_shard
        gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], out=out, plan=plan, workspace=ws,
                            stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist_barrier(dist)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    dist_barrier(dist)
    ms = dist_max(dist, t0.elapsed_time(t1) / args.steps, dev)
    return {
        "metric": METRIC, "value": E * H / (ms * 1e-3), "unit": "edge-heads/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "fused GAT layer, row-sharded: 1e6 rows, Zipf(2.1) in-degrees, "
                               "H=8, Dh=64, bf16, seed 3; per step an all-gather of the "
                               "node-sharded k and v, then the fused layer on each rank's rows",
                   "n_rows": n, "n_edges": E, "parallelism": f"{world} row shards",
                   "rank0_rows": [r0, r1], "rank0_edges": e1 - e0},
        "gpu_launches": args.steps, "clocks": clk.summary(),
    }


def bench_reference(args, rank, world):
    """--impl reference: the fp64 oracle, timed per step on a bounded sample."""
    from concurrent.futures import ThreadPoolExecutor
    d = W.make_fused(seed=3)
    import oracle
    oracle.build()
    rp = d["row_ptr"]
    host = host_cpu()
    cores = host["nproc"]
    block = args.ref_rows  # rows per step, split over every core
    sub = max(1, (block + cores - 1) // cores)
    n = rp.size - 1
    pool = ThreadPoolExecutor(cores)

    def part(r0, r1):
        sel = np.arange(r0, r1)
        oracle.fused_layer(rp, d["col_idx"], d["q"], d["k"], d["v"], d["H"], d["Dh"],
                           d["scale"], rows=sel)
        return int(rp[r1] - rp[r0])

    def step(i):
        # one step: `block` consecutive rows, cut into one sub-block per core
        # (ctypes releases the GIL, so the oracle calls run in parallel)
        r0 = (i * block) % n
        r1 = min(n, r0 + block)
        futs = [pool.submit(part, a, min(r1, a + sub)) for a in range(r0, r1, sub)]
        return sum(f.result() for f in futs)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    edges = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    pool.shutdown()
    value = edges * d["H"] / dt
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "edge-heads/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "fused GAT layer: 1e6 rows, Zipf(2.1) in-degrees clipped to "
                               "[1,4096] rescaled to mean 16, col_idx uniform sorted in-row, "
                               "H=8, Dh=64, q/k/v bf16 N(0,1), seed 3",
                   "sample_rows_per_step": block},
        "cpu_baseline": {"value": value, "unit": "edge-heads/s", "cores": cores,
                         "kind": "oracle", "cpu_model": host["cpu_model"],
                         "sample": f"{args.steps} steps of {block} consecutive rows each "
                                   f"({edges} edges), fp64 C loops, {cores} threads "
                                   f"(one sub-block of the step's rows each)"},
        "e2e": {"value": value, "unit": "edge-heads/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------
# the smaller workloads (parity-test cases; timed here for the record)
# ----------------------------------------------------------------------------
def bench_small(name, args):
    import torch
    import sparse_graph_attention_head_gb300 as gat
    dev = torch.device("cuda", 0)
    g = W.WORKLOADS[name][0]() if name in ("edge_softmax", "aggregate", "sddmm", "dense") else None
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    flops, tensor_flops = 0.0, 0.0
    extra = {}
    if name == "spmm_heads":
        # head_dim 32, 8 heads, fp32 weights and features, 1e6-row power-law graph
        g = W.make_spmm_heads(n=args.n_rows)
        rp, ci, w, feat = t(g["row_ptr"]), t(g["col_idx"]), t(g["w"]), t(g["feat"])
        out = torch.empty_like(feat)
        plan = gat.Plan(rp)
        ws = torch.empty(max(1, gat.gat_spmm_weighted_workspace_size(plan, g["H"], g["Dh"])),
                         dtype=torch.uint8, device=dev)
        fn = lambda: gat.gat_spmm_weighted(rp, ci, w, feat, g["H"], g["Dh"], out=out,  # noqa: E731
                                           plan=plan, workspace=ws)
        units, launches = g["n_edges"] * g["H"], 1
        row = 4 * g["H"] * g["Dh"]
        # per row: row_ptr entry and output row; per edge: col_idx entry, H
        # weights and the gathered feature row
        alg_bytes = (4 + row) * g["n_rows"] + (4 + 4 * g["H"] + row) * g["n_edges"]
        flops = 2.0 * g["n_edges"] * g["H"] * g["Dh"]
    elif name == "fused_backward":
        # gradients of the fused layer on the 1e6-row power-law graph (bf16, H=8, Dh=64)
        g = W.make_fused_backward(n=args.n_rows)
        bt = lambda a: t(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
        rp, ci = t(g["row_ptr"]), t(g["col_idx"])
        q, k, v, go = (bt(g[x]) for x in ("q", "k", "v", "dout"))
        plan = gat.Plan(rp)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        tr = gat.Transpose(rp, ci, g["n_src"])
        torch.cuda.synchronize()
        transpose_ms = (time.perf_counter() - t0) * 1e3
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(gat.gat_fused_layer_backward_workspace_size(
            plan, g["n_rows"], g["n_edges"], g["H"], g["Dh"]), dtype=torch.uint8, device=dev)
        extra_l2 = l2_persist(torch, torch.cuda.current_stream(), {"q": q, "k": k, "v": v,
                                                                 "dout": go}, args.l2_persist)
        fn = lambda: gat.gat_fused_layer_backward(rp, ci, q, k, v, go, g["scale"], tr,  # noqa: E731
                                                  plan=plan, dq=dq, dk=dk, dv=dv, workspace=ws)
        units, launches = g["n_edges"] * g["H"], 4
        rb = 2 * g["H"] * g["Dh"]
        # per edge: col_idx, k and v rows (pass A), score and da written then
        # read (8H each way), perm and dst, q and dout rows (pass B); per row:
        # row_ptr, q, dout in, dq out, lse and Delta written (8H; their reads
        # in pass B are gathers of this table); per source: src_ptr, dk, dv out
        alg_bytes = (g["n_edges"] * (4 + 2 * rb + 16 * g["H"] + 8 + 2 * rb)
                     + g["n_rows"] * (4 + 3 * rb + 8 * g["H"]) + g["n_src"] * (4 + 2 * rb))
        flops = 2.0 * g["n_edges"] * g["H"] * g["Dh"] * 6
        extra = {"transpose_build_ms": transpose_ms, "transpose": tr.info(), "l2_persist": extra_l2}
    elif name == "fused_fp8":
        # the fused workload (1e6 rows, Zipf, H=8, Dh=64) with k/v quantised to
        # E4M3 + per (node, head) scales on the device; q/out bf16
        g = W.make_fused(seed=3, n=args.n_rows)
        bt = lambda a: t(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
        rp, ci = t(g["row_ptr"]), t(g["col_idx"])
        q, k, v = (bt(g[x]) for x in ("q", "k", "v"))
        plan = gat.Plan(rp)
        k8, ks = torch.empty(k.shape, dtype=torch.uint8, device=dev), \
            torch.empty(k.shape[:2], dtype=torch.float32, device=dev)
        v8, vs = torch.empty_like(k8), torch.empty_like(ks)
        qa, qb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(2):  # warm, then timed: both tables
            qa.record()
            gat.gat_quantize_fp8(k, k8, ks)
            gat.gat_quantize_fp8(v, v8, vs)
            qb.record()
        torch.cuda.synchronize()
        out = torch.empty_like(q)
        ws = torch.empty(max(1, gat.gat_fused_layer_workspace_size(plan, g["H"], g["Dh"])),
                         dtype=torch.uint8, device=dev)
        fn = lambda: gat.gat_fused_layer_fp8(rp, ci, q, k8, ks, v8, vs, g["scale"],  # noqa: E731
                                             out=out, plan=plan, workspace=ws)
        units, launches = g["n_edges"] * g["H"], 1
        hd = g["H"] * g["Dh"]
        # per row: row_ptr, q and out rows (bf16); per edge: col_idx, the k8 and
        # v8 rows (1 B per element) and their 2H scales
        alg_bytes = g["n_rows"] * (4 + 4 * hd) + g["n_edges"] * (4 + 2 * hd + 8 * g["H"])
        # quantisation error of the layer: the fp8 output against the bf16
        # layer's on the same inputs (both computed here, on the device)
        fn()
        ref = gat.gat_fused_layer(rp, ci, q, k, v, g["scale"], plan=plan,
                                  workspace=torch.empty(max(1, gat.gat_fused_layer_workspace_size(
                                      plan, g["H"], g["Dh"])), dtype=torch.uint8, device=dev))
        diff = (out.float() - ref.float())
        err = {"rel_rms": float(diff.pow(2).mean().sqrt() / ref.float().pow(2).mean().sqrt()),
               "max_abs": float(diff.abs().max()), "ref_rms": float(ref.float().pow(2).mean().sqrt())}
        del ref, diff
        extra = {"quantize_ms_both_tables": qa.elapsed_time(qb),
                 "bytes_vs_bf16_layer": alg_bytes / fused_bytes(g["n_rows"], g["n_edges"],
                                                                 g["H"], g["Dh"]),
                 "error_vs_bf16_layer": err}
    elif name == "sddmm_csr":
        # per-edge scores of the fused workload's graph: out[e,h] = q[row]·k[col]/8,
        # 1e6 rows, Zipf(2.1) degrees, H=8, Dh=64, bf16 q/k, fp32 [E,8] out
        g = W.make_fused(seed=3, n=args.n_rows)
        bt = lambda a: t(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
        rp, ci = t(g["row_ptr"]), t(g["col_idx"])
        q, k = bt(g["q"]), bt(g["k"])
        out = torch.empty((g["n_edges"], g["H"]), dtype=torch.float32, device=dev)
        fn = lambda: gat.gat_sddmm(ci, k, q, g["H"], g["Dh"], scale=g["scale"],  # noqa: E731
                                   row_ptr=rp, out=out)
        units, launches = g["n_edges"] * g["H"], 1
        rb = 2 * g["H"] * g["Dh"]
        # per row: row_ptr entry and q row; per edge: col_idx entry, k row of the
        # source, H fp32 scores out
        alg_bytes = g["n_rows"] * (4 + rb) + g["n_edges"] * (4 + rb + 4 * g["H"])
        flops = 2.0 * g["n_edges"] * g["H"] * g["Dh"]
    elif name == "edge_softmax_h8":
        # 8 heads on the 1e6-row power-law graph (--n-rows: smaller, for captures)
        deg = W.zipf_degrees(np.random.default_rng(3), args.n_rows)
        g = W.make_edge_softmax(seed=6, deg=deg, H=8)
        rp, s = t(g["row_ptr"]), t(g["scores"])
        out = torch.empty_like(s)
        plan = gat.Plan(rp)
        extra = {"l2_persist": l2_persist(torch, torch.cuda.current_stream(), {"scores": s},
                                          args.l2_persist)}
        fn = lambda: gat.gat_edge_softmax(rp, s, g["H"], out=out, plan=plan)  # noqa: E731
        units, launches = g["n_edges"] * g["H"], 1
        alg_bytes = 4 * (g["n_rows"] + 1) + 8 * g["n_edges"] * g["H"]
    elif name == "edge_softmax":
        rp, s = t(g["row_ptr"]), t(g["scores"])
        out = torch.empty_like(s)
        fn = lambda: gat.gat_edge_softmax(rp, s, g["H"], out=out)  # noqa: E731
        units, launches = g["n_edges"] * g["H"], 1
        alg_bytes = 4 * (g["n_rows"] + 1) + 8 * g["n_edges"] * g["H"]
    elif name == "aggregate":
        rp, ci, s = t(g["row_ptr"]), t(g["col_idx"]), t(g["scores"]).reshape(-1, 1)
        vals = t(g["values"]).reshape(g["n_src"], 1, g["F"])
        w = torch.empty_like(s)
        out = torch.empty((g["n_rows"], 1, g["F"]), device=dev)
        # one pass: the softmax of the given scores and the weighted sum together
        fn = lambda: gat.gat_softmax_aggregate(rp, ci, s, vals, 1, g["F"], out=out)  # noqa: E731
        units, launches = g["n_edges"], 1
        # row_ptr; per edge its col_idx, its score and one gathered value row;
        # one output row per row
        alg_bytes = 4 * (g["n_rows"] + 1) + g["n_edges"] * (4 + 4 + 4 * g["F"]) + \
            4 * g["F"] * g["n_rows"]

        def two():
            gat.gat_edge_softmax(rp, s, 1, out=w)
            gat.gat_spmm_weighted(rp, ci, w, vals, 1, g["F"], out=out)
        for _ in range(max(3, args.warmup)):
            two()
        torch.cuda.synchronize()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(50)]
        for ev_a, ev_b in ev2:
            ev_a.record()
            two()
            ev_b.record()
        torch.cuda.synchronize()
        extra["two_launch_median_ms"] = spread([x.elapsed_time(y) for x, y in ev2])["median_ms"]
        extra["two_launch"] = "gat_edge_softmax then gat_spmm_weighted, weights through memory"
    elif name == "sddmm":
        si, di, a, b = t(g["src_idx"]), t(g["dst_idx"]), t(g["src_feat"]), t(g["dst_feat"])
        out = torch.empty((g["n_edges"], 1), device=dev)
        fn = lambda: gat.gat_sddmm(si, a, b, 1, g["F"], dst_idx=di, out=out)  # noqa: E731
        units, launches = g["n_edges"], 1
        alg_bytes = g["n_edges"] * (4 + 4 + 2 * 4 * g["F"] + 4)
        flops = 2.0 * g["n_edges"] * g["F"]
    elif name == "dense":
        keys = ("nodes", "pair_feats", "edge_mask", "ln_w", "ln_b", "Wq", "Wk", "Wv", "W1",
                "b1", "W2", "b2", "Wout")
        tt = {k: t(g[k]) for k in keys}
        out = torch.empty_like(tt["nodes"])
        wk = [tt[k] for k in keys[5:]]
        fn = lambda: gat.gat_dense_masked_attention(  # noqa: E731
            tt["nodes"], tt["pair_feats"], tt["edge_mask"], tt["ln_w"], tt["ln_b"],
            g["ln_eps"], *wk, H=g["H"], out=out)
        units, launches = g["B"] * g["H"] * g["N"] * g["N"], 1
        B_, N_, D_, H_, P_ = g["B"], g["N"], g["D"], g["H"], g["P"]
        # per graph: nodes + pair features + mask in, output out (fp32)
        alg_bytes = B_ * 4 * (2 * N_ * D_ + N_ * N_ * P_ + N_ * N_) + 4 * (4 * D_ * D_)
        proj = 2.0 * N_ * D_ * D_ * 4                        # Q, K, V, out projections
        attn = 2.0 * 2 * H_ * N_ * N_ * (D_ // H_)           # Q K^T and A V
        mlp = 2.0 * N_ * N_ * (P_ * P_ + H_ * P_)            # relation MLP
        flops = B_ * (proj + attn + mlp)
        # the kernel reads the pair features of unmasked pairs only (a masked
        # pair's logit is -inf whatever its relation-MLP bias): the bytes it
        # has to move on this mask, beside the nominal count above
        unmasked = int((g["edge_mask"] >= 0.5).sum())
        # on the tensor cores: the projections, Q K^T and A V, and the relation
        # MLP's first layer over the unmasked pairs
        tensor_flops = B_ * (proj + attn) + 2.0 * P_ * P_ * unmasked
        need = B_ * 4 * (2 * N_ * D_ + N_ * N_) + 4 * P_ * unmasked + 4 * (4 * D_ * D_)
        extra["required_bytes"] = need
        extra["unmasked_pair_frac"] = unmasked / float(B_ * N_ * N_)
        extra["bytes_note"] = ("algorithmic_bytes / hbm_frac: every pair's features (the "
                               "workload's definition); required_bytes / hbm_frac_required: "
                               "the unmasked pairs' features only, as the kernel reads them")
    else:
        raise ValueError(name)
    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    # 50 calls, each bracketed by its own events; rates use the median call
    reps = 50
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    # (the workload closures above may capture names such as a and b: the
    # events get names of their own)
    cold = getattr(args, "cold_l2", False)
    if cold:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    for ev_a, ev_b in evs:
        if cold:
            flush.fill_(1)  # outside the events: evicts the workload's lines from L2
        ev_a.record()
        fn()
        ev_b.record()
    torch.cuda.synchronize()
    sp = spread([x.elapsed_time(y) for x, y in evs])
    ms = sp["median_ms"]
    hbm_peak, bf16_peak, kind = measured_peaks()
    res = {"ms_per_step": ms, "p10_ms": sp["p10_ms"], "p90_ms": sp["p90_ms"], "reps": reps,
           "units_per_s": units / (ms * 1e-3), "launches_per_step": launches,
           "warm": not cold, "algorithmic_bytes": alg_bytes,
           "achieved_gbs": alg_bytes / (ms * 1e-3) / 1e9,
           "hbm_frac": alg_bytes / (ms * 1e-3) / 1e9 / hbm_peak}
    if flops:
        res["achieved_tflops"] = flops / (ms * 1e-3) / 1e12
    if tensor_flops:
        # f16 operands split in two terms: three tensor products per useful one
        # (padding of the small attention tiles not counted); the f16 dense
        # peak is the measured bf16 one
        res["tensor_tflops_useful"] = tensor_flops / (ms * 1e-3) / 1e12
        res["tensor_issue_frac_of_f16_peak"] = 3 * tensor_flops / (ms * 1e-3) / 1e12 / bf16_peak
        res["f16_peak_tflops"] = bf16_peak
        res["peak_kind"] = kind
    if name in ("edge_softmax", "aggregate", "sddmm"):
        # launch-bound at this size: the per-call events above include the
        # host's time to issue the call. The same calls captured in a CUDA
        # graph and replayed give the device time per call.
        per_graph = 20
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            for _ in range(3):
                fn()
        torch.cuda.current_stream().wait_stream(cs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                fn()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_replay = 20
        ga.record()
        for _ in range(n_replay):
            graph.replay()
        gb.record()
        torch.cuda.synchronize()
        g_ms = ga.elapsed_time(gb) / (n_replay * per_graph)
        extra["graph_ms_per_call"] = g_ms
        extra["graph_units_per_s"] = units / (g_ms * 1e-3)
        extra["graph_note"] = f"{per_graph} calls captured in one CUDA graph, {n_replay} replays"
    res.update(extra)
    if "required_bytes" in extra:
        res["hbm_frac_required"] = extra["required_bytes"] / (ms * 1e-3) / 1e9 / hbm_peak
    res["l2"] = ("flushed before each call (twice the L2 size written)" if cold else
                 "warm (inputs may stay in L2 between calls)")
    if name in ("edge_softmax", "aggregate", "sddmm"):
        res["note"] = "L2-resident and launch-latency bound at this size; fractions are not a roofline claim"
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200,
                    help="timed layer calls (200 x ~5 ms: about a second, several clock samples)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gat", choices=["gat", "reference"])
    ap.add_argument("--workload", default="fused",
                    choices=["fused", "edge_softmax", "aggregate", "sddmm", "dense", "spmm_heads",
                             "edge_softmax_h8", "fused_backward", "fused_fp8", "sddmm_csr"])
    ap.add_argument("--config", type=int, choices=[1, 2, 3, 4, 5],
                    help="the workload by its configuration number: 1 edge softmax (384 rows), "
                         "2 softmax + aggregation, 3 COO SDDMM, 4 the fused layer on the "
                         "1e6-row graph (the default), 5 the dense-masked block")
    ap.add_argument("--cold-l2", action="store_true",
                    help="smaller workloads: write a buffer of twice the L2 size before each "
                         "timed call (cold-cache times; by default they are timed warm)")
    ap.add_argument("--ref-rows", type=int, default=40000,
                    help="--impl reference: consecutive rows per step, split over the host's "
                         "cores (~0.2 s of oracle work on 16 cores)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for cpu_baseline (0: skip)")
    ap.add_argument("--n-rows", type=int, default=1_000_000,
                    help="rows of the 1e6-row workloads (fused, fused_backward, fused_fp8, "
                         "sddmm_csr, edge_softmax_h8, spmm_heads; smaller only for profiling "
                         "captures)")
    ap.add_argument("--no-extras", action="store_true", help="skip the smaller workloads")
    ap.add_argument("--l2-persist", default="off",
                    choices=["off", "none", "q", "k", "v", "dout", "scores"],
                    help="A/B of L2 persistence: off (default, device untouched), or the "
                         "device's persisting-L2 carve-out with a window on this table "
                         "(none: carve-out, no window); fused, fused_backward, "
                         "edge_softmax_h8 workloads")
    ap.add_argument("--mode", default="replicas", choices=["replicas", "rowshard"],
                    help="N > 1: independent full problems per rank (replicas, weak scaling) "
                         "or one graph cut into row shards (rowshard, strong scaling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.config is not None:
        args.workload = {1: "edge_softmax", 2: "aggregate", 3: "sddmm", 4: "fused",
                         5: "dense"}[args.config]
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: relaunch this command under the torch launcher
        sys.exit(relaunch_ranks(args.gpus))
    rank, world, local = dist_env()
    if world != args.gpus:
        print(json.dumps({"error": f"--gpus {args.gpus} but the launcher started {world} ranks "
                                   "(WORLD_SIZE); they must agree"}), flush=True)
        sys.exit(2)

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(bench_reference(args, rank, world)), flush=True)
        return

    dist = dist_init(world, "nccl")
    if args.mode == "rowshard":
        res = bench_rowshard(args, rank, world, local, dist)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    if args.workload != "fused":
        if rank == 0:
            print(json.dumps({"workload": args.workload, **bench_small(args.workload, args)}))
        return
    res, d = bench_fused(args, rank, world, local, dist)
    if rank == 0:
        # the side workloads and the CPU baseline are single-GPU measurements:
        # taken at N = 1 only (at N > 1 every rank ends with the headline)
        if not args.no_extras and world == 1:
            res["other_workloads"] = {}
            for nm in ("edge_softmax", "aggregate", "sddmm", "dense", "spmm_heads",
                       "edge_softmax_h8", "fused_backward", "fused_fp8", "sddmm_csr"):
                try:
                    res["other_workloads"][nm] = bench_small(nm, args)
                except Exception as exc:  # keep the headline line if a side workload fails
                    res["other_workloads"][nm] = {"error": repr(exc)}
        if args.cpu_budget > 0 and world == 1:
            res["cpu_baseline"] = cpu_baseline_fused(d, budget_s=args.cpu_budget)
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
