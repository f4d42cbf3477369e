"""Benchmark of the TokenButler decode-time hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one decode step of one Llama-3-8B-shaped attention layer at
N = 32768 cached tokens with a 10% budget (k = 3277 per KV head): append the
new token (K/V rows and its projected key), score all N tokens with the
importance query, keep the top k per KV head, and attend over the gathered
rows. Inputs are seeded synthetic tensors already resident in HBM. The step
rotates over R copies of the layer's caches so that consecutive steps never
find their data in the 126 MB L2 (R x the step's bytes >= 4 x L2).

Prints one JSON line (rank 0). With --gpus N > 1 (torchrun) every rank runs
its own replica of the workload (the (batch, KV head) rows are independent;
there is no collective on the path) and value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "decode steps/sec & tokens/s at N=32K, budget 10%; achieved HBM GB/s vs ~8 TB/s"
UNIT = "decode steps/s"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=synth.WORKLOADS[1].name)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-warm-l2", action="store_true", help="skip the labelled warm-L2 leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--rotate", type=int, default=0, help="cache copies to rotate over (0: enough to defeat L2)")
    ap.add_argument("--agg", default="mean", choices=["mean", "max"],
                    help="how the G query heads' scores combine (mean: the default reading)")
    ap.add_argument("--ragged", default="",
                    help="n1,n2,...: a batch of sequences of these lengths (the workload's heads, k); own line")
    ap.add_argument("--predict", default="",
                    help="B,E,F: the importance-query predictor (O = Hq dp of the workload); prints its own line")
    ap.add_argument("--buffers", default="",
                    help="S,W: sink and local-window buffers with batched key projection; prints its own line")
    ap.add_argument("--offload", action="store_true",
                    help="K/V in pinned host memory (the offloaded cache); prints its own line")
    ap.add_argument("--layers", type=int, default=0,
                    help="L: one decode step of L consumer layers of the workload's shape (the selection of later "
                         "layers overlapping the attention of earlier ones); prints its own line, per-layer figures")
    ap.add_argument("--stack-layers", type=int, default=0,
                    help="run the stack workload with this many layers instead of all of them")
    ap.add_argument("--budget", type=float, default=0.0,
                    help="budget as a fraction of N (k = ceil(frac N)) instead of the workload's k")
    ap.add_argument("--pipeline", action="store_true",
                    help="run the single-layer step as the three-kernel form instead of the cooperative kernel")
    ap.add_argument("--prefill", action="store_true",
                    help="the key projection of a whole prefill (tcgen05), on the B=2, N=65536 prefill "
                         "workload unless --workload names another; prints its own line")
    return ap.parse_args()


def _workload(name):
    for w in synth.WORKLOADS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}")


def _traffic(workload: str):
    """DRAM bytes per launch of the step kernel from the committed ncu capture,
    or None when the capture was taken on another workload or on different
    code (the record carries the code hash of the kernel's translation units
    and every header, comments removed, plus the compiler flags)."""
    from predicted_token_importance_tb_b300 import build
    try:
        with open(os.path.join(ROOT, "profiles", "fused_fast_traffic.json")) as f:
            rec = json.load(f)
        code = build.code_hash(rec["code_units"])
    except (OSError, ValueError, KeyError, TypeError):
        return None
    if rec.get("workload") != workload or rec.get("code_hash") != code:
        return None
    return int(rec["dram_bytes_per_launch"])


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"tb_clocks_gpu{index}_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        mhz = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist_init(n):
    """One process per GPU under torchrun (NCCL); gloo on a host without CUDA (the replicas' host logic)."""
    if n <= 1:
        return 0, 1, None
    import torch.distributed as dist
    cuda = torch.cuda.is_available()
    dist.init_process_group("nccl" if cuda else "gloo")
    rank = dist.get_rank()
    if cuda:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
    return rank, dist.get_world_size(), dist


def _dev():
    return "cuda" if torch.cuda.is_available() else "cpu"


def _barrier(dist):
    if dist is not None:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def _max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_dev())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_dev())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle arm

def _oracle_setup(w):
    import oracle
    n0 = w.N - 1
    L = synth.make_layer(w, cap=w.N, n=n0)
    oK = oracle.as_u16(L["K"]).copy()
    oV = oracle.as_u16(L["V"]).copy()
    oKp = np.zeros((w.B, w.Hkv, w.N, w.dp), dtype=np.uint16)
    oKp[:, :, :n0], _ = oracle.project(np.ascontiguousarray(oK[:, :, :n0]), L["Wk"])
    d = synth.make_step(w, 0, 0, L["outlier_ch"])
    return L, oK, oV, oKp, n0, d


def _oracle_step(w, L, d, oK, oV, oKp, n0):
    """One whole decode step in the oracle (append, score, top-k, attention; OpenMP over rows)."""
    import oracle
    st = oracle.DecodeState()
    oracle.decode_step(st, 0, n0, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=L["Wk"],
                       K=oK, V=oV, Kp=oKp, k=w.k, T=1, r=0, agg=oracle.AGG_MEAN, scale=w.scale)


def _oracle_cores(w) -> int:
    import oracle
    return min(oracle.num_threads(), w.B * w.Hq)


def cpu_baseline(w, seconds: float, threads: int = 0):
    """The oracle as it stands, timed on this host's cores (or on `threads` of them) on a bounded sample of
    whole decode steps."""
    import oracle
    L, oK, oV, oKp, n0, d = _oracle_setup(w)
    before = oracle.num_threads()
    if threads:
        oracle.set_num_threads(threads)
    try:
        cores = _oracle_cores(w)
        done = 0
        t0 = time.perf_counter()
        while True:
            _oracle_step(w, L, d, oK, oV, oKp, n0)
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    finally:
        if threads:
            oracle.set_num_threads(before)
    return {"value": done / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} whole decode steps at N={w.N}, k={w.k} in {el:.1f} s (fp64 C, OpenMP over "
                      f"(batch, head) rows, {cores} thread(s))"}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    L, oK, oV, oKp, n0, d = _oracle_setup(w)
    t1 = time.perf_counter()
    _oracle_step(w, L, d, oK, oV, oKp, n0)
    per_step = time.perf_counter() - t1
    warm = max(0, min(args.warmup, 3))
    for _ in range(warm):
        _oracle_step(w, L, d, oK, oV, oKp, n0)
    # the number of steps timed is capped so the run ends within a few minutes
    timed = max(1, min(args.steps, int(120.0 / max(per_step, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(timed):
        _oracle_step(w, L, d, oK, oV, oKp, n0)
    el = time.perf_counter() - t0
    val = timed / el
    sample = f"{timed} whole decode steps at N={w.N}, k={w.k} (of {args.steps} requested), fp64 C, OpenMP"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": timed, "steps_requested": args.steps, "warmup": warm, "ms_per_step": 1e3 / val,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "N": w.N, "k": w.k, "B": w.B},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": _oracle_cores(w), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_ours(args, w):
    import predicted_token_importance_tb_b300 as tb

    rank, world, dist = _dist_init(args.gpus)
    if dist is None:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    n0 = w.N - 1                     # tokens before the step's append: the step scores N
    cap = w.N
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=n0)
    Wk = L["Wk"].cuda()
    K0, V0 = L["K"].cuda(), L["V"].cuda()
    Kp0 = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K0, cap, Wk, Kp0, 0, n0)
    torch.cuda.synchronize()

    # bytes one step moves (algorithmic): Kp stream, the gathered K/V rows,
    # q / q_imp / out, and the append (new K/V rows in and out, Wk, new Kp row)
    rows = w.B * w.Hkv
    kp_bytes = rows * w.N * w.dp * 2
    gather_bytes = rows * w.k * 2 * w.D * 2
    qio_bytes = (w.B * w.Hq * w.D * 2) * 2 + w.B * w.Hq * w.dp * 2
    append_bytes = rows * w.D * 2 * 2 * 2 + w.Hkv * w.D * w.dp * 2 + rows * w.dp * 2
    step_bytes = kp_bytes + gather_bytes + qio_bytes + append_bytes

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = args.rotate if args.rotate > 0 else max(4, math.ceil(4 * l2 / step_bytes))
    Ks = [K0] + [K0.clone() for _ in range(R - 1)]
    Vs = [V0] + [V0.clone() for _ in range(R - 1)]
    Kps = [Kp0] + [Kp0.clone() for _ in range(R - 1)]
    steps_in = [synth.make_step(w, 0, i, L["outlier_ch"]) for i in range(R)]
    dins = [{k: v.cuda() for k, v in d.items()} for d in steps_in]
    agg = tb.TB_AGG_MAX if args.agg == "max" else tb.TB_AGG_MEAN
    dec = tb.DecodeLayer(shape, w.k, T=1, r=0, agg=agg, scale=w.scale, n_max=n0, pipeline=args.pipeline)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")

    def step(i):
        j = i % R
        d = dins[j]
        dec.step(0, n0, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=Wk, K=Ks[j], V=Vs[j],
                 Kp=Kps[j], out=out)

    # eager sanity pass, then capture M steps as one CUDA graph
    for i in range(R):
        step(i)
    torch.cuda.synchronize()
    tb.check_dev_status(dec.status, "bench warm-up")
    M = min(max(R, (1000 // R) * R), max(args.steps, 1))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graphs = {}

    def graph_of(m):
        if m not in graphs:
            g = torch.cuda.CUDAGraph(keep_graph=True)
            with torch.cuda.graph(g, stream=s):
                for i in range(m):
                    step(i)
            g.instantiate()
            graphs[m] = g
        return graphs[m]

    gM = graph_of(M)
    kernel_nodes = _count_kernel_nodes(gM)
    kernels_per_step = kernel_nodes / M if kernel_nodes is not None else None
    rem = args.steps % M
    g_rem = graph_of(rem) if rem else None
    torch.cuda.synchronize()
    # warm-up: at least W steps, and every graph the timed region replays is replayed (uploaded, its
    # first launch paid) here first, so no freshly instantiated graph runs inside the timed region
    warm_steps = 0
    for _ in range(max(2, -(-args.warmup // M))):
        gM.replay()
        warm_steps += M
    if g_rem is not None:
        g_rem.replay()
        warm_steps += rem
    torch.cuda.synchronize()

    def timed_region():
        """Barrier + synchronize, one untimed replay that keeps the GPU busy while the timed replays are
        submitted (so host submission never shows as idle GPU time), then exactly args.steps steps
        between two events on the launching stream, barrier + synchronize."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        _barrier(dist)
        with torch.cuda.stream(s):
            gM.replay()
            e0.record(s)
            for _ in range(args.steps // M):
                gM.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(s)
        _barrier(dist)
        return e0.elapsed_time(e1)

    clocks = ClockSampler(dev) if rank == 0 else None
    if clocks:
        clocks.start()
    ms = timed_region()
    clk = clocks.stop() if clocks else None
    # four more identical regions, for the median the line also reports
    repeats = [ms] + [timed_region() for _ in range(4)]
    tb.check_dev_status(dec.status, "bench timed region")
    ms = _max_over_ranks(dist, ms)
    ms_median = _max_over_ranks(dist, statistics.median(repeats))
    sec = ms / 1e3
    steps_per_s_rank = args.steps / sec
    total_steps_per_s = steps_per_s_rank * world

    # realised gathered rows (from counts) for the byte accounting
    real_gather = int(dec.counts.sum().item()) * 2 * w.D * 2
    step_bytes_real = kp_bytes + real_gather + qio_bytes + append_bytes
    hbm_peak, peak_kind = _peaks()
    per_step_s = sec / args.steps
    achieved = step_bytes_real / per_step_s / 1e9

    # a labelled warm-L2 figure: the same step on one cache set, so its bytes stay in L2
    warm = None
    if not args.no_warm_l2:
        mw = 200
        gw = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gw, stream=s):
            for _ in range(mw):
                step(0)
        for _ in range(2):
            gw.replay()
        torch.cuda.synchronize()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            gw.replay()
            w0.record(s)
            for _ in range(5):
                gw.replay()
            w1.record(s)
        torch.cuda.synchronize()
        tb.check_dev_status(dec.status, "bench warm-L2 leg")
        wus = w0.elapsed_time(w1) * 1e3 / (5 * mw)
        warm = {"us_per_step": wus, "steps_per_s": 1e6 / wus, "steps": 5 * mw,
                "note": "rotation off: one cache set, L2-resident after the first step (not the headline)"}
        del gw

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(tb, w, shape, dec, Wk, Ks[0], Vs[0], Kps[0], n0, steps_in, dist, world)

    cpu = None
    cpu1 = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
        cpu1 = cpu_baseline(w, args.cpu_seconds / 3, threads=1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": total_steps_per_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": warm_steps, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "dp": w.dp, "N": w.N,
                       "k": w.k, "T": 1, "r": 0, "agg": args.agg, "rotation_sets": R,
                       "l2_defeat": f"inputs rotate over {R} cache copies ({R * step_bytes / 1e6:.0f} MB touched per "
                                    f"rotation, L2 {l2 / 1e6:.0f} MB)",
                       "parallelism": f"replicas x{world}"},
            "tokens_per_s": total_steps_per_s * w.B,
            "hbm_gbs": achieved * world,
            "bytes_per_step": step_bytes_real,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": _traffic(w.name),
                         "kernel": "tb decode step, %s kernel(s) per step" % kernels_per_step,
                         "peak_source": peak_kind},
            "cpu_baseline": cpu,
            "cpu_baseline_1thread": cpu1,
            "e2e": e2e,
            "gpu_launches": int(round(args.steps * kernels_per_step)) if kernels_per_step else None,
            "kernels_per_step": kernels_per_step,
            "kernel_us": ms * 1e3 / args.steps,
            "median_of_5": {"us_per_step": ms_median * 1e3 / args.steps,
                            "note": "median over five identical timed regions of the same length"},
            "warm_l2": warm,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _count_kernel_nodes(g) -> int | None:
    """Kernel nodes in a captured CUDA graph (the launches one replay makes)."""
    try:
        from cuda.bindings import runtime as rt
        graph = g.raw_cuda_graph()
        err, _, n = rt.cudaGraphGetNodes(graph, 0)
        err, nodes, n = rt.cudaGraphGetNodes(graph, n)
        kinds = [rt.cudaGraphNodeGetType(x)[1] for x in nodes[:n]]
        return sum(1 for k in kinds if k == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel)
    except Exception:
        return None


def _e2e(tb, w, shape, dec, Wk, K, V, Kp, n0, steps_in, dist, world, n_steps=300):
    """Same step through the Python API: each step's inputs (q, q_imp, K_new, V_new, packed in one pinned
    host buffer) copied in with one copy, the output copied out, the stream synchronised, every step."""
    names = ["q", "q_imp", "K_new", "V_new"]
    sizes = [steps_in[0][k].numel() for k in names]
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    total = sum(sizes)
    host = []
    for d in steps_in:
        buf = torch.empty(total, dtype=torch.bfloat16).pin_memory()
        for k, o, z in zip(names, offs, sizes):
            buf[o:o + z].copy_(d[k].reshape(-1))
        host.append(buf)
    dbuf = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    dv = {k: dbuf[o:o + z].view(steps_in[0][k].shape) for k, o, z in zip(names, offs, sizes)}
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total * 2
    d2h = out.numel() * out.element_size()
    stream = torch.cuda.current_stream()

    def one(i):
        dbuf.copy_(host[i % len(host)], non_blocking=True)
        dec.step(0, n0, q=dv["q"], q_imp=dv["q_imp"], K_new=dv["K_new"], V_new=dv["V_new"], Wk=Wk, K=K, V=V, Kp=Kp,
                 out=out)
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for i in range(20):
        one(i)
    _barrier(dist)
    t0 = time.perf_counter()
    for i in range(n_steps):
        one(i)
    el = time.perf_counter() - t0
    el = _max_over_ranks(dist, el)
    return {"value": n_steps * world / el, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n_steps, "note": "per step: one H2D copy of q, q_imp, K_new, V_new (packed, pinned), "
                                      "tb_decode_step, D2H of out, stream synchronize"}


def run_offload(args, w):
    """The decode step with K/V in pinned host memory and Kp in HBM: only the selected rows (and the
    appended row) cross the host link. L2 is flushed between steps (outside the timed windows), each
    step is bracketed by its own events; the work is enqueued ahead so the windows hold GPU time only."""
    import predicted_token_importance_tb_b300 as tb

    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    n0 = w.N - 1
    cap = w.N
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=n0)
    Wk = L["Wk"].cuda()
    Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, L["K"].cuda(), cap, Wk, Kp, 0, n0)
    K, V = L["K"].pin_memory(), L["V"].pin_memory()
    R = 18
    dins = [{k: v.cuda() for k, v in synth.make_step(w, 0, i, L["outlier_ch"]).items()} for i in range(R)]
    dec = tb.DecodeLayer(shape, w.k, T=1, r=0, scale=w.scale, n_max=n0)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")

    def step(i):
        d = dins[i % R]
        dec.step(0, n0, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=Wk, K=K, V=V, Kp=Kp,
                 out=out)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    tb.check_dev_status(dec.status, "offload warm-up")
    n_steps = max(1, min(args.steps, 2000))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
    clocks = ClockSampler(dev)
    clocks.start()
    for i in range(n_steps):
        flush.zero_()
        ev[i][0].record()
        step(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    tb.check_dev_status(dec.status, "offload timed steps")
    ms = sum(a.elapsed_time(b) for a, b in ev)
    rows = w.B * w.Hkv
    link = int(dec.counts.sum().item()) * 2 * w.D * 2 + rows * 2 * w.D * 2   # selected rows in, new row out
    hbm = rows * w.N * w.dp * 2 + (w.B * w.Hq * w.D * 2) * 2 + w.B * w.Hq * w.dp * 2 + w.Hkv * w.D * w.dp * 2
    sec = ms / 1e3
    # the link's copy-engine rate for context: 256 MB pinned host -> device
    src = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    dst = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(4):
        dst.copy_(src, non_blocking=True)
    c1.record()
    torch.cuda.synchronize()
    copy_gbs = 4 * (256 << 20) / (c0.elapsed_time(c1) / 1e3) / 1e9
    line = {
        "metric": "decode steps/s with K/V in pinned host memory (offloaded cache), N=32K, budget 10%",
        "value": n_steps / sec, "unit": UNIT, "n_gpus": 1, "steps": n_steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms / n_steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "kv": "pinned host memory, read through unified addressing",
                   "kp": "device memory", "l2_defeat": f"{2 * l2 / 1e6:.0f} MB written between steps, untimed"},
        "link_bytes_per_step": link, "link_gbs": link / (sec / n_steps) / 1e9,
        "link_copy_engine_gbs": copy_gbs, "hbm_bytes_per_step": hbm,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_ragged(args, w):
    """The step for a ragged batch (T = 1, r = 0, the workload's heads and budget) at fixed positions, R
    rotated cache sets, M steps captured in one CUDA graph."""
    import predicted_token_importance_tb_b300 as tb

    ns = [int(v) for v in args.ragged.split(",")]
    B = len(ns)
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    cap = max(ns) + 1
    wb = synth.Workload(f"ragged-B{B}", B=B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, dp=w.dp, N=max(ns), k=w.k, seed=9)
    k = min(w.k, min(ns) + 1)
    shape = tb.Shape(B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(wb, cap=cap, n=max(ns))
    Wk = L["Wk"].cuda()
    K0, V0 = L["K"].cuda(), L["V"].cuda()
    Kp0 = torch.zeros((B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K0, cap, Wk, Kp0, 0, max(ns))
    rows = B * w.Hkv
    step_bytes = (sum((n + 1) * w.Hkv * w.dp * 2 for n in ns) + rows * k * 2 * w.D * 2 + (B * w.Hq * w.D * 2) * 2
                  + B * w.Hq * w.dp * 2 + rows * w.D * 2 * 2 * 2 + w.Hkv * w.D * w.dp * 2 + rows * w.dp * 2)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / step_bytes))
    sets = [(K0, V0, Kp0)] + [(K0.clone(), V0.clone(), Kp0.clone()) for _ in range(R - 1)]
    dins = [{kk: v.cuda() for kk, v in synth.make_step(wb, 0, i, L["outlier_ch"]).items()} for i in range(R)]
    dec = tb.RaggedDecodeLayer(shape, k, T=1, r=0, scale=w.scale, n_max=cap - 1)
    out = torch.empty((B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")

    def step(i):
        K, V, Kp = sets[i % R]
        d = dins[i % R]
        dec.step(0, ns, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=Wk, K=K, V=V, Kp=Kp,
                 out=out)

    for i in range(R):
        step(i)
    torch.cuda.synchronize()
    tb.check_dev_status(dec.status, "ragged warm-up")
    M = R * max(1, 400 // R)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for i in range(M):
            step(i)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // M)
    clocks = ClockSampler(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    tb.check_dev_status(dec.status, "ragged timed steps")
    ms = e0.elapsed_time(e1)
    n = reps * M
    per = ms / 1e3 / n
    hbm_peak, peak_kind = _peaks()
    line = {
        "metric": "decode steps/s for a ragged batch (sequences of different lengths), budget k per sequence",
        "value": n / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": n, "warmup": 3 * M, "ms_per_step": ms / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"lengths": ns, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "dp": w.dp, "k": k, "T": 1, "r": 0,
                   "rotation_sets": R},
        "tokens_per_s": n / (ms / 1e3) * B, "bytes_per_step": step_bytes,
        "roofline": {"bound": "hbm", "achieved": step_bytes / per / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": step_bytes / per / 1e9 / hbm_peak, "peak_source": peak_kind},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_predict(args, w):
    """The predictor MLP for B tokens (hidden E -> F -> Hq dp), weights rotated over enough copies to
    defeat L2, M calls captured in one CUDA graph."""
    import predicted_token_importance_tb_b300 as tb

    B, E, F = (int(v) for v in args.predict.split(","))
    O = w.Hq * w.dp
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    g = torch.Generator().manual_seed(7)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    wbytes = (F * E + O * F) * 2
    R = max(4, math.ceil(4 * l2 / wbytes))
    W1s = [(torch.randn(F, E, generator=g) * E ** -0.5).to(torch.bfloat16).cuda() for _ in range(R)]
    W2s = [(torch.randn(O, F, generator=g) * F ** -0.5).to(torch.bfloat16).cuda() for _ in range(R)]
    xs = [torch.randn(B, E, generator=g).to(torch.bfloat16).cuda() for _ in range(R)]
    q = torch.empty(B, O, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B * F * 4, dtype=torch.uint8, device="cuda")
    M = R * max(1, 2000 // R)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for i in range(M):
            j = i % R
            tb.tb_predict_queries(xs[j], W1s[j], W2s[j], q, ws=ws)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // M)
    clocks = ClockSampler(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    n = reps * M
    per = ms / 1e3 / n
    nbytes = wbytes + B * E * 2 + B * O * 2 + 2 * B * F * 4
    hbm_peak, peak_kind = _peaks()
    line = {
        "metric": "importance-query predictions/s (MLP forward)", "value": n / (ms / 1e3), "unit": "predictions/s",
        "n_gpus": 1, "steps": n, "warmup": 3 * M, "ms_per_step": ms / n, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random weights)",
        "config": {"tokens": B, "hidden": E, "mlp_width": F, "outputs": O, "weight_sets": R},
        "bytes_per_step": nbytes, "kernels_per_step": 2,
        "roofline": {"bound": "hbm", "achieved": nbytes / per / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": nbytes / per / 1e9 / hbm_peak, "peak_source": peak_kind},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_prefill(args, w):
    """Kp = RNE_bf16(K Wk) for all N rows of every (batch, KV head): one tb_project_append per step (the
    tcgen05 kernel), M steps captured in one CUDA graph. K (B Hkv N D bf16) is larger than L2 at the
    prefill workload, so each step streams it from HBM."""
    import predicted_token_importance_tb_b300 as tb

    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    n = w.N
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, n)
    g = torch.Generator(device="cuda").manual_seed(4)
    K = torch.randn((w.B, w.Hkv, n, w.D), device="cuda", generator=g).to(torch.bfloat16)
    Wk = (torch.randn((w.Hkv, w.D, w.dp), device="cuda", generator=g) * w.D ** -0.5).to(torch.bfloat16)
    Kp = torch.empty((w.B, w.Hkv, n, w.dp), dtype=torch.bfloat16, device="cuda")
    kbytes = K.numel() * 2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    status = tb.dev_status()
    tb.tb_project_append(shape, K, n, Wk, Kp, 0, n, dev_status=status)   # once eagerly: attributes, entry points
    torch.cuda.synchronize()
    M = 20
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for _ in range(M):
            tb.tb_project_append(shape, K, n, Wk, Kp, 0, n, dev_status=status)
    for _ in range(max(3, args.warmup // M)):
        graph.replay()
    torch.cuda.synchronize()
    tb.check_dev_status(status)
    reps = max(1, min(args.steps, 4000) // M)
    clocks = ClockSampler(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    tb.check_dev_status(status)
    ms = e0.elapsed_time(e1)
    steps = reps * M
    per = ms / 1e3 / steps
    rows = w.B * w.Hkv * n
    nbytes = rows * (2 * w.D + 2 * w.dp) + w.Hkv * w.D * w.dp * 2
    hbm_peak, peak_kind = _peaks()
    line = {
        "metric": "prefill key projection: cached tokens projected/s (B x N per step, all KV heads)",
        "value": w.B * n / per, "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": max(3, args.warmup // M) * M, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hkv": w.Hkv, "D": w.D, "dp": w.dp, "N": n,
                   "l2_defeat": f"K is {kbytes / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB"},
        "bytes_per_step": nbytes, "flops_per_step": 2 * rows * w.D * w.dp, "kernels_per_step": 1,
        "gpu_launches": steps,
        "roofline": {"bound": "hbm", "achieved": nbytes / per / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": nbytes / per / 1e9 / hbm_peak, "kernel": "tb::project_tc_kernel",
                     "peak_source": peak_kind},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_buffered(args, w):
    """The buffered step (sink S, window W, Kp projected in batches of W) at the bench workload with a
    prediction at every step. R cache sets rotate (L2 defeat); set j advances its own token position, so
    the captured sequence holds the batch projections at their natural rate (one batch per W steps of a
    set). The M captured steps are replayed as one CUDA graph."""
    import predicted_token_importance_tb_b300 as tb

    S, W = (int(x) for x in args.buffers.split(","))
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    R = 16
    m = max(W, 8)                      # steps per set in the captured sequence
    n0 = w.N - 1 - m
    cap = w.N
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=n0)
    Wk = L["Wk"].cuda()
    K0, V0 = L["K"].cuda(), L["V"].cuda()
    P0 = ((n0 + 1 - 2 * W) // W) * W   # prefill projected up to a batch boundary, a window's worth behind
    Kp0 = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K0, cap, Wk, Kp0, 0, P0)
    sets = []
    for j in range(R):
        K, V, Kp = (K0, V0, Kp0) if j == 0 else (K0.clone(), V0.clone(), Kp0.clone())
        layer = tb.BufferedDecodeLayer(shape, w.k, sink=S, window=W, proj_end=P0, T=1, r=0, scale=w.scale,
                                       n_max=cap - 1)
        sets.append((K, V, Kp, layer))
    dins = [{k: v.cuda() for k, v in synth.make_step(w, 0, i, L["outlier_ch"]).items()} for i in range(R)]
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    M = R * m

    def seq():
        for i in range(M):
            j, t = i % R, i // R
            K, V, Kp, layer = sets[j]
            d = dins[j]
            layer.step(t, n0 + t, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=Wk, K=K, V=V,
                       Kp=Kp, out=out)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        seq()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for _, _, _, layer in sets:
        tb.check_dev_status(layer.status, "buffered warm-up")
    reps = max(1, args.steps // M)
    clocks = ClockSampler(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    for _, _, _, layer in sets:
        tb.check_dev_status(layer.status, "buffered timed steps")
    ms = e0.elapsed_time(e1)
    n_steps = reps * M
    layer = sets[0][3]
    rows = w.B * w.Hkv
    sel_rows = int(layer.counts.sum().item())
    P = layer.proj_end.value
    # Kp stream of the candidates, the selected K/V rows, q / q_imp / out, the append (K_new, V_new in, the
    # K/V rows out) and the batch projection per step (a K row in and a Kp row out per row, Wk once a batch)
    step_bytes = (rows * (P - S) * w.dp * 2 + sel_rows * 2 * w.D * 2 + (w.B * w.Hq * w.D * 2) * 2
                  + w.B * w.Hq * w.dp * 2 + rows * 2 * w.D * 2 * 2
                  + rows * (w.D * 2 + w.dp * 2) + w.Hkv * w.D * w.dp * 2 // W)
    hbm_peak, peak_kind = _peaks()
    per_step = ms / 1e3 / n_steps
    line = {
        "metric": "decode steps/s with sink + local-window buffers and batched key projection, N=32K, budget 10%",
        "value": n_steps / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": n_steps, "warmup": 3 * M,
        "ms_per_step": ms / n_steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "sink": S, "window": W, "T": 1, "r": 0, "rotation_sets": R,
                   "steps_per_set_in_graph": m},
        "bytes_per_step": step_bytes, "selected_rows_per_step": sel_rows,
        "roofline": {"bound": "hbm", "achieved": step_bytes / per_step / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": step_bytes / per_step / 1e9 / hbm_peak, "peak_source": peak_kind},
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_layers(args, w):
    """One decode step of L consumer layers of the workload's shape through tb_decode_layers: every layer's
    selection (its n cached tokens scored against the producer's importance query, the top k kept) runs on a
    second stream while earlier layers attend; each layer's attention waits for the previous layer's. R sets
    of L layers rotate (L2 defeat); M steps are captured in one CUDA graph."""
    import predicted_token_importance_tb_b300 as tb

    Lc = args.layers
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    n0 = w.N - 1
    cap = w.N
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    rows = w.B * w.Hkv
    kp_bytes = rows * n0 * w.dp * 2                      # the selection streams the n cached tokens' Kp
    qio_bytes = (w.B * w.Hq * w.D * 2) * 2 + w.B * w.Hq * w.dp * 2
    append_bytes = rows * w.D * 2 * 2 * 2 + w.Hkv * w.D * w.dp * 2 + rows * w.dp * 2
    layer_bytes_est = kp_bytes + rows * w.k * 2 * w.D * 2 + qio_bytes + append_bytes
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / (Lc * layer_bytes_est)))
    base = synth.make_layer(w, cap=cap, n=n0)
    Wk = base["Wk"].cuda()
    K0, V0 = base["K"].cuda(), base["V"].cuda()
    Kp0 = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K0, cap, Wk, Kp0, 0, n0)
    sets = []
    for j in range(R):
        lay = []
        for l in range(Lc):
            first = j == 0 and l == 0
            lay.append((K0 if first else K0.clone(), V0 if first else V0.clone(), Kp0 if first else Kp0.clone()))
        sets.append(lay)
    dins = [[{k: v.cuda() for k, v in synth.make_step(w, l, j, base["outlier_ch"]).items()} for l in range(Lc)]
            for j in range(R)]
    outs = [torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for _ in range(Lc)]
    stack = tb.DecodeStack(shape, Lc, w.k, scale=w.scale, n_max=n0)

    def step(i):
        j = i % R
        lay, d = sets[j], dins[j]
        stack.step(n0, q=[x["q"] for x in d], q_imp=[x["q_imp"] for x in d], K_new=[x["K_new"] for x in d],
                   V_new=[x["V_new"] for x in d], Wk=[Wk] * Lc, K=[x[0] for x in lay], V=[x[1] for x in lay],
                   Kp=[x[2] for x in lay], out=outs)

    for i in range(R):
        step(i)
    torch.cuda.synchronize()
    tb.check_dev_status(stack.status, "layers warm-up")
    M = R * max(1, 100 // R)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g, stream=s):
        for i in range(M):
            step(i)
    g.instantiate()
    kernel_nodes = _count_kernel_nodes(g)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    tb.check_dev_status(stack.status, "layers graph warm-up")
    reps = max(1, args.steps // (M * Lc))
    clocks = ClockSampler(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        g.replay()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    tb.check_dev_status(stack.status, "layers timed steps")
    ms = e0.elapsed_time(e1)
    steps = reps * M
    per_step = ms / 1e3 / steps
    per_layer = per_step / Lc
    gather = sum(int(c.sum().item()) for c in stack.counts) / Lc * 2 * w.D * 2
    layer_bytes = kp_bytes + gather + qio_bytes + append_bytes
    hbm_peak, peak_kind = _peaks()
    achieved = layer_bytes / per_layer / 1e9
    line = {
        "metric": "decode steps/s of an L-layer stack (per-layer time and HBM roofline), N=32K, budget 10%",
        "value": 1.0 / per_step, "unit": "decode steps/s", "n_gpus": 1, "steps": steps, "warmup": 3 * M,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}-x{Lc}layers", "layers": Lc, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "dp": w.dp, "N": w.N, "k": w.k, "T": 1, "r": 0, "rotation_sets": R,
                   "l2_defeat": f"{R} sets of {Lc} layers rotate ({R * Lc * layer_bytes / 1e6:.0f} MB, "
                                f"L2 {l2 / 1e6:.0f} MB)"},
        "us_per_layer": per_layer * 1e6, "bytes_per_layer": layer_bytes,
        "tokens_per_s": w.B / per_step,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_kind,
                     "kernel": "per layer: selection kernel (second stream) + attention kernel, overlapped"},
        "kernels_per_step": kernel_nodes / M if kernel_nodes is not None else None,
        "gpu_launches": int(round(kernel_nodes / M * steps)) if kernel_nodes is not None else None,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_stack(args, w):
    """The 32-layer stack workload: every decode step runs tb_decode_step on each of the L layers in turn (B
    sequences, the prediction every T steps, +-r neighbours, the tail between predictions), for the workload's
    step count. The layers' caches are generated on the device (seeded; the distributions of the synthetic
    recipe: K, V ~ N(0, 1) with the outlier key channels scaled, Wk ~ N(0, 1/D), fresh q, q_imp, K_new, V_new
    ~ N(0, 1) per layer and step). The whole sequence of steps is one CUDA graph; prediction steps and reuse
    steps are also timed on their own. Bytes come from the realised selection sizes."""
    import predicted_token_importance_tb_b300 as tb

    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tb.load_library()
    Lc, steps, n0 = w.layers, w.steps, w.N
    cap = n0 + steps
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    oc = torch.randperm(w.D, generator=torch.Generator().manual_seed(w.seed))[: w.outliers].cuda()
    layers = []
    for l in range(Lc):
        K = torch.zeros((w.B, w.Hkv, cap, w.D), dtype=torch.bfloat16, device="cuda")
        V = torch.zeros_like(K)
        Kf = torch.randn((w.B, w.Hkv, n0, w.D), device="cuda", generator=g)
        Kf[..., oc] *= w.outlier_scale
        K[:, :, :n0] = Kf.to(torch.bfloat16)
        del Kf
        V[:, :, :n0] = torch.randn((w.B, w.Hkv, n0, w.D), device="cuda", generator=g).to(torch.bfloat16)
        Wk = (torch.randn((w.Hkv, w.D, w.dp), device="cuda", generator=g) * w.D ** -0.5).to(torch.bfloat16)
        Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
        tb.tb_project_append(shape, K, cap, Wk, Kp, 0, n0)
        dec = tb.DecodeLayer(shape, w.k, T=w.T, r=w.r, scale=w.scale, n_max=cap - 1)
        layers.append(dict(K=K, V=V, Wk=Wk, Kp=Kp, dec=dec))
    ins = []
    for t in range(steps):
        row = []
        for l in range(Lc):
            kn = torch.randn((w.B, w.Hkv, w.D), device="cuda", generator=g)
            kn[..., oc] *= w.outlier_scale
            row.append(dict(q=torch.randn((w.B, w.Hq, w.D), device="cuda", generator=g).to(torch.bfloat16),
                            q_imp=torch.randn((w.B, w.Hq, w.dp), device="cuda", generator=g).to(torch.bfloat16),
                            K_new=kn.to(torch.bfloat16),
                            V_new=torch.randn((w.B, w.Hkv, w.D), device="cuda", generator=g).to(torch.bfloat16)))
        ins.append(row)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()

    def one(t, l):
        y, d = layers[l], ins[t][l]
        y["dec"].step(t, n0 + t, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=y["Wk"], K=y["K"],
                      V=y["V"], Kp=y["Kp"], out=out)

    # one eager pass: realised selection sizes per step (bytes), status
    rows = w.B * w.Hkv
    sel_rows = []
    for t in range(steps):
        tot = 0
        for l in range(Lc):
            one(t, l)
            tot += int(layers[l]["dec"].counts.sum().item())
        sel_rows.append(tot)
    for y in layers:
        tb.check_dev_status(y["dec"].status, "stack warm-up")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def capture(ts):
        gr = torch.cuda.CUDAGraph(keep_graph=True)
        with torch.cuda.graph(gr, stream=s):
            for t in ts:
                for l in range(Lc):
                    one(t, l)
        return gr

    g_all = capture(range(steps))
    g_pred = capture([0])            # a prediction step of every layer
    g_reuse = capture([w.T - 1])     # the last step of an interval: the longest tail
    for gr in (g_all, g_pred, g_reuse):
        gr.instantiate()
    kernel_nodes = _count_kernel_nodes(g_all)

    def timed(gr, reps):
        for _ in range(2):
            gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            gr.replay()
            e0.record(s)
            for _ in range(reps):
                gr.replay()
            e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    clocks = ClockSampler(dev)
    clocks.start()
    reps = max(1, min(20, args.steps // steps))
    ms_all = timed(g_all, reps)
    clk = clocks.stop()
    ms_pred = timed(g_pred, 20)
    ms_reuse = timed(g_reuse, 20)
    for y in layers:
        tb.check_dev_status(y["dec"].status, "stack timed steps")
    per_step = ms_all / 1e3 / steps
    kp_pred = rows * w.dp * 2       # per cached token per layer, at a prediction step
    qio = (w.B * w.Hq * w.D * 2) * 2 + w.B * w.Hq * w.dp * 2
    append = rows * w.D * 2 * 2 * 2 + w.Hkv * w.D * w.dp * 2 + rows * w.dp * 2
    total = 0
    for t in range(steps):
        total += sel_rows[t] * 2 * w.D * 2 + Lc * (qio + append)
        if t % w.T == 0:
            total += Lc * kp_pred * (n0 + t + 1)
    bytes_per_step = total / steps
    hbm_peak, peak_kind = _peaks()
    achieved = bytes_per_step / per_step / 1e9
    pred_bytes = sel_rows[0] * 2 * w.D * 2 + Lc * (qio + append + kp_pred * (n0 + 1))
    reuse_bytes = sel_rows[w.T - 1] * 2 * w.D * 2 + Lc * (qio + append)
    cpu = None
    if not args.no_cpu_baseline:
        cpu = _stack_cpu_baseline(w)
    line = {
        "metric": f"decode steps/s of the {Lc}-layer stack (B=8, N=16K, k=1024, prediction every T=16 steps, r=1)",
        "value": 1.0 / per_step, "unit": "decode steps/s", "n_gpus": 1, "steps": steps * reps,
        "warmup": 2 * steps, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (device-generated, seeded)",
        "config": {"workload": w.name, "layers": Lc, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "dp": w.dp,
                   "N0": n0, "k": w.k, "T": w.T, "r": w.r, "steps": steps,
                   "l2_defeat": f"{Lc} layers of {(2 * w.D + w.dp) * 2 * rows * cap / 1e9:.2f} GB each per step"},
        "tokens_per_s": w.B / per_step, "us_per_layer_step": per_step * 1e6 / Lc,
        "bytes_per_step": bytes_per_step, "selected_rows_per_step": sum(sel_rows) / steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_kind,
                     "kernel": "tb_decode_step per layer (prediction: append, score, top-k, expand, attention; "
                               "reuse: append with the tail entry, attention)"},
        "prediction_step": {"us": ms_pred * 1e3, "bytes": pred_bytes,
                            "gbs": pred_bytes / (ms_pred / 1e3) / 1e9,
                            "frac": pred_bytes / (ms_pred / 1e3) / 1e9 / hbm_peak},
        "reuse_step": {"us": ms_reuse * 1e3, "bytes": reuse_bytes,
                       "gbs": reuse_bytes / (ms_reuse / 1e3) / 1e9,
                       "frac": reuse_bytes / (ms_reuse / 1e3) / 1e9 / hbm_peak},
        "kernels_per_step": kernel_nodes / steps if kernel_nodes is not None else None,
        "gpu_launches": int(kernel_nodes * reps) if kernel_nodes is not None else None,
        "cpu_baseline": cpu,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def _stack_cpu_baseline(w, layers_sampled: int = 1):
    """The oracle on a bounded sample of the stack: one layer through one prediction interval (T steps),
    scaled to whole 32-layer steps."""
    import oracle
    cap = w.N + w.T
    L = synth.make_layer(w, layer=0, cap=cap, n=w.N)
    oK, oV = oracle.as_u16(L["K"]).copy(), oracle.as_u16(L["V"]).copy()
    oKp = np.zeros((w.B, w.Hkv, cap, w.dp), dtype=np.uint16)
    oKp[:, :, :w.N], _ = oracle.project(np.ascontiguousarray(oK[:, :, :w.N]), L["Wk"])
    st = oracle.DecodeState()
    ds = [synth.make_step(w, 0, t, L["outlier_ch"]) for t in range(w.T)]
    t0 = time.perf_counter()
    for t in range(w.T):
        d = ds[t]
        oracle.decode_step(st, t, w.N + t, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"],
                           Wk=L["Wk"], K=oK, V=oV, Kp=oKp, k=w.k, T=w.T, r=w.r, agg=oracle.AGG_MEAN, scale=w.scale)
    el = time.perf_counter() - t0
    per_layer_step = el / w.T
    return {"value": 1.0 / (per_layer_step * w.layers), "unit": "decode steps/s",
            "cores": min(oracle.num_threads(), w.B * w.Hq), "kind": "oracle",
            "sample": f"layer 0 through one prediction interval ({w.T} steps, {el:.1f} s), scaled to "
                      f"{w.layers}-layer steps"}


def main():
    args = _args()
    w = _workload(args.workload)
    if args.budget > 0:
        import dataclasses
        w = dataclasses.replace(w, k=int(math.ceil(args.budget * w.N - 1e-9)))
    if args.stack_layers > 0:
        import dataclasses
        w = dataclasses.replace(w, layers=args.stack_layers)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.layers:
        run_layers(args, w)
    elif w.layers > 1:
        run_stack(args, w)
    elif args.offload:
        run_offload(args, w)
    elif args.buffers:
        run_buffered(args, w)
    elif args.predict:
        run_predict(args, w)
    elif args.ragged:
        run_ragged(args, w)
    elif args.prefill:
        run_prefill(args, w if args.workload != synth.WORKLOADS[1].name else _workload("prefill-B2-N65536-sweep"))
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
