"""Benchmark of the NVFP4 MoE expert layer on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward of the whole layer (routing, up GEMV/GEMM with relu^2,
down GEMV/GEMM, WeightedRowSum) over one batch of the seeded synthetic
workload, inputs already resident in HBM.  The default workload is decode-1
(1 token, H 2688, I 1856, 128 experts, top-6); other workloads are available
with --workload.  Between timed steps a 256 MB write flushes the 129 MB L2 and
the routing rotates over 8 seeded variants, so weights stream from HBM.  Each
step is bracketed by CUDA events on the launching stream; the forward is
replayed from a CUDA graph or launched directly, whichever was faster over
untimed probe steps (config.graph says which; --no-graph forces direct).

Multi-GPU (torchrun): the layer does not shard across GPUs here, so every
rank runs an independent replica on its own GPU (weak scaling, no data-path
collective); rank 0 reports max-over-ranks time and the summed throughput.

The metric covers decode and prefill, so the same run also measures the
workloads named by --workloads (default decode-32, prefill-4314 and
prefill-16384; prefill with fewer steps) and reports each under "workloads"
with its own tokens/s, roofline (HBM for the streaming kernel, bf16 tensor
peak for the grouped GEMMs, plus the layer's expert flops over its step time
for prefill), end-to-end host-buffer number, clocks and oracle sample.

--impl reference times the fp64 CPU oracle (the only other implementation of
the layer) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nvfp4_quantized_moe_topk_gb300 import workload as W  # noqa: E402

METRIC = "MoE layer tokens/s (decode & prefill) on 1 GB300; % of HBM / bf16 roofline"
N_ROUTINGS = 8


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="decode-1", choices=sorted(W.CONFIGS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--gemv-max-rows", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--gated", action="store_true",
                   help="gated experts (silu(gate) * up) on the same workload shapes, gate weights drawn last")
    p.add_argument("--workloads", default="decode-32,prefill-4314,prefill-16384",
                   help="other workloads measured in the same run and reported under 'workloads' "
                        "(comma-separated; 'none' for the headline workload only)")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- work model
def algorithmic_work(wl, ids_list, T):
    """Per-kernel algorithmic bytes / flops of one forward, averaged over the routings.

    GEMV kernels: bytes = NVFP4 weights of the experts they serve (codes + block
    scales, each read once) + activations read + outputs written.  GEMM kernels:
    flops = 2 * rows * N * K over the rows they serve.  Combine: dst read+write,
    k fp32 rows per token read, ids/weights read.
    """
    H, I, E, k, n = wl.H, wl.I, wl.E, wl.k, wl.n
    up_mats = 2 if wl.gated else 1  # a gated expert's up step reads the gate and the up matrix
    per = {"gemv_up": [0.0, 0.0], "gemv_down": [0.0, 0.0], "gemm_up": [0.0, 0.0], "gemm_down": [0.0, 0.0],
           "combine": [0.0, 0.0], "routing": [0.0, 0.0], "gather": [0.0, 0.0]}
    mat_bytes = H * I // 2 + H * I // 16
    single = decode_single_launch(n, k, T)
    gemm_path = not single and n > T
    for ids in ids_list:
        c = np.bincount(ids.ravel(), minlength=E)
        for e in range(E):
            if c[e] == 0:
                continue
            if gemm_path and c[e] > T:
                per["gemm_up"][1] += 2.0 * c[e] * I * H * up_mats
                per["gemm_down"][1] += 2.0 * c[e] * H * I
                per["gemm_up"][0] += up_mats * mat_bytes + c[e] * (H + I) * 2
                per["gemm_down"][0] += mat_bytes + c[e] * (I * 2 + H * 4)
            else:
                per["gemv_up"][0] += up_mats * mat_bytes + c[e] * (H * 2 + I * 2)
                per["gemv_down"][0] += mat_bytes + c[e] * (I * 2 + H * 4)
                per["gemv_up"][1] += 2.0 * c[e] * I * H * up_mats
                per["gemv_down"][1] += 2.0 * c[e] * H * I
        per["combine"][0] += n * H * 2 * 2 + n * k * H * 4 + n * k * 8
        per["routing"][0] += n * k * 4 * 4
        if gemm_path:
            per["gather"][0] += n * H * 2 + n * k * H * 2  # x read once per token, one row written per pair
    m = len(ids_list)
    out = {kname: (b / m, f / m) for kname, (b, f) in per.items()}
    if gemm_path:
        # experts at or below the threshold run in one streaming launch (both projections)
        out["small_experts"] = (out["gemv_up"][0] + out["gemv_down"][0], out["gemv_up"][1] + out["gemv_down"][1])
        del out["gemv_up"], out["gemv_down"]
    if single:
        # the whole layer is one kernel: the layer's algorithmic bytes -- the
        # NVFP4 weights of every touched expert read once, x read, dst read and
        # written, ids and weights read (8 B per pair); the intermediates stay
        # on chip or in L2 and are not counted
        w_bytes = 0.0
        for ids in ids_list:
            c = np.bincount(ids.ravel(), minlength=E)
            w_bytes += float(np.count_nonzero(c)) * (up_mats + 1) * mat_bytes
        b = w_bytes / m + 3.0 * n * H * 2 + 8.0 * n * k
        flops = sum(out[p][1] for p in ("gemv_up", "gemv_down"))
        out = {"decode": (b, flops)}
    return out


def decode_single_launch(n, k, T):
    """Whether the library runs this batch as its one-launch small-batch kernel."""
    return n <= 64 and n * k <= 1024


def profiled_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu captures, or None
    when there is none or the kernel's sources changed since it was taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    data = json.load(open(path))
    rec = data.get(f"{workload}:{kernel}") or data.get(workload)
    if not rec or rec.get("kernel") != kernel:
        return None
    csrc = os.path.join(ROOT, "nvfp4_quantized_moe_topk_gb300", "csrc")
    h = hashlib.sha256()
    for f in (rec["source"], "common.cuh", "kernels.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return float(rec["bytes_per_launch"]) if h.hexdigest()[:16] == rec["source_sha"] else None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples: $MOE_CLOCKS_DIR if set, else the system temp directory
        out_dir = os.environ.get("MOE_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"moe_clocks_rank{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()
        return False

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        loaded = [s for s in sm if smax is None or s > 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- CPU baseline
def cpu_baseline(wl, seconds: float):
    """The fp64 oracle as it stands, on this host's cores, on a bounded sample.

    The oracle runs the independent values of each step (one intermediate
    feature of one pair, one output column of one pair, one output element)
    in parallel on all of its threads, so a one-token batch uses every core
    too.  Batches of at most 64 tokens run whole, repeated for about
    `seconds`; larger ones on a contiguous token range grown to about that."""
    import oracle

    n_threads = oracle.num_threads()
    if wl.n <= 64:
        t0 = time.perf_counter()
        runs = 0
        while True:
            oracle.moe_forward(wl)
            runs += 1
            if time.perf_counter() - t0 >= seconds or runs >= 1000:
                break
        dt = time.perf_counter() - t0
        toks = runs * wl.n
        sample = f"whole workload ({wl.n} tokens) x {runs} runs"
    else:
        t1 = max(1, min(wl.n, 8))
        while True:
            t0 = time.perf_counter()
            oracle.moe_forward(wl, tok_range=(0, t1))
            dt = time.perf_counter() - t0
            if dt >= seconds * 0.5 or t1 >= wl.n:
                break
            t1 = min(wl.n, max(t1 * 2, int(t1 * seconds / max(dt, 1e-3) * 0.7)))
        toks = t1
        sample = f"tokens [0, {t1}) of {wl.n}"
    return {"value": toks / dt, "unit": "tokens/s", "cores": n_threads, "kind": "oracle", "sample": sample,
            "seconds": dt}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = W.generate(args.workload, gated=args.gated)
    import oracle

    oracle.build()
    per_step = max(1.0, 10.0 / max(1, args.steps))
    for _ in range(args.warmup):
        cpu_baseline(wl, 0.0)
    vals = []
    samples = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        b = cpu_baseline(wl, per_step)
        vals.append(b["value"])
        samples.append(b)
    wall = time.perf_counter() - t_all
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * wall / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "n": wl.n, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                       "activation": "swiglu" if args.gated else "relu2"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": samples[-1]["cores"], "kind": "oracle",
                             "sample": samples[-1]["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- ours
def replica_throughput(ms_local: float, tokens_per_rank: int, dist=None, device=None) -> tuple[float, float]:
    """Each rank runs an independent replica of the layer (no data-path
    collective): the job's step time is the slowest rank's, and its throughput
    is every rank's tokens over that time.  Returns (max ms, tokens/s)."""
    world, ms = 1, float(ms_local)
    if dist is not None:
        import torch

        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_rank / (ms / 1000.0)


def _launches_per_step(n, k, T):
    """Kernels one forward enqueues: the single launch; or routing (one kernel,
    or two above 4096 pairs), gather, small experts, 2 GEMMs, combine; or
    routing, 2 GEMVs, combine."""
    if decode_single_launch(n, k, T):
        return 1
    routing_launches = 1 if n * k <= 4096 else 2
    return routing_launches + (5 if n > T else 3)


def bench_workload(api, torch, name, args, dev, *, steps, warmup, cpu_seconds, dist=None, local=0):
    """Measure one workload: the timed forward steps, the per-kernel roofline,
    the router, the end-to-end host-buffer call and (optionally) the oracle
    on the host cores.  Returns the fields of one result record."""
    world = dist.get_world_size() if dist is not None else 1
    cfg = W.CONFIGS[name]
    wl = W.generate(name, gated=args.gated)
    T = args.gemv_max_rows if args.gemv_max_rows > 0 else 8
    routings = [(wl.topk_ids, wl.topk_weights)] + [
        W.make_routing(wl.n, wl.E, wl.k, cfg["bias_sigma"], seed=5000 + 97 * i) for i in range(1, N_ROUTINGS)]

    def d(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    gate = {}
    if wl.gated:
        gate = dict(gate_codes=d(wl.gate_codes), gate_scales=d(wl.gate_scales), gate_global=d(wl.gate_global))
    layer = api.MoeLayer(wl.H, wl.I, wl.E, wl.k, wl.n, d(wl.up_codes), d(wl.up_scales), d(wl.down_codes),
                         d(wl.down_scales), d(wl.up_global), d(wl.down_global), gemv_max_rows=args.gemv_max_rows,
                         **gate)
    x = d(wl.x)
    dst = d(wl.dst)
    ids_d = [d(r[0]) for r in routings]
    w_d = [d(r[1]) for r in routings]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(W.l2_flush_bytes() // 4, dtype=torch.float32, device=dev)

    def fwd(i):
        layer.forward(x, ids_d[i % N_ROUTINGS], w_d[i % N_ROUTINGS], dst, stream=stream)

    graphs = None
    with torch.cuda.stream(stream):
        for i in range(2 * N_ROUTINGS):
            fwd(i)
        torch.cuda.synchronize()
        if not args.no_graph:
            try:
                graphs = []
                for i in range(N_ROUTINGS):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        fwd(i)
                    graphs.append(g)
                torch.cuda.synchronize()
            except RuntimeError as exc:  # capture refused: launch directly
                print(f"bench: graph capture failed ({exc}); timing direct launches", file=sys.stderr)
                graphs = None
                torch.cuda.synchronize()

    def step(i):
        if graphs is not None:
            graphs[i % N_ROUTINGS].replay()
        else:
            fwd(i)

    if graphs is not None:
        # A replayed one-kernel graph can cost more than the plain launch it
        # holds: time both ways on untimed steps and keep the faster.
        def probe():
            evs = []
            with torch.cuda.stream(stream):
                for i in range(2 * N_ROUTINGS):
                    flush.fill_(float(i))
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    step(i)
                    e1.record(stream)
                    evs.append((e0, e1))
                torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in evs)

        t_graph = probe()
        kept, graphs = graphs, None
        t_direct = probe()
        if t_graph < t_direct:
            graphs = kept

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(warmup):
            flush.fill_(float(i))
            step(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            t_wall = time.perf_counter()
            for i in range(steps):
                flush.fill_(float(i))
                ev[i][0].record(stream)
                step(i)
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            t_wall = time.perf_counter() - t_wall
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms, value = replica_throughput(sum(step_ms) / len(step_ms), wl.n, dist, dev)

    # per-kernel event timing (separate pass, same inputs, no graph) -> roofline of the dominant kernel
    layer.set_timing(True)
    layer.kernel_times()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(float(i))
            fwd(i)
        torch.cuda.synchronize()
    kt = layer.kernel_times()
    layer.set_timing(False)
    per_launch_ms = {kname: tot / cnt for kname, (tot, cnt) in kt.items() if cnt}
    work = algorithmic_work(wl, [r[0] for r in routings], T)
    peaks = load_peaks()

    def roofline_of(kname):
        b_alg, f_alg = work.get(kname, (0.0, 0.0))
        t = per_launch_ms[kname] / 1000.0
        if kname.startswith("gemm"):
            ach = f_alg / t / 1e12
            r = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                 "frac": ach / peaks["bf16_tflops"]}
        else:
            ach = b_alg / t / 1e9
            r = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": ach / peaks["hbm_gbs"]}
        r["traffic"] = profiled_traffic(name + ("+gated" if args.gated else ""), kname)
        r["kernel"] = kname
        r["kernel_ms"] = per_launch_ms[kname]
        r["peak_source"] = peaks["source"]
        return r

    dom = max(per_launch_ms, key=lambda kname: per_launch_ms[kname])
    roof = roofline_of(dom)
    layer_bytes = sum(b for kname, (b, f) in work.items())
    layer_flops = sum(f for kname, (b, f) in work.items() if kname.startswith("gemm"))
    layer_rec = {"alg_bytes": layer_bytes, "alg_gemm_flops": layer_flops,
                 "hbm_frac_whole_layer": layer_bytes / (ms / 1000.0) / 1e9 / peaks["hbm_gbs"],
                 "per_kernel_ms": per_launch_ms}
    if any(kname.startswith("gemm") for kname in per_launch_ms):
        # the prefill figure of merit: all the layer's expert flops (4 R H I, routed rows only,
        # gated 6 R H I) over the whole layer's step time, against the bf16 peak
        f_layer = (6.0 if wl.gated else 4.0) * wl.n * wl.k * wl.H * wl.I
        layer_rec["layer_tflops"] = f_layer / (ms / 1000.0) / 1e12
        layer_rec["layer_tensor_frac"] = layer_rec["layer_tflops"] / peaks["bf16_tflops"]
        layer_rec["gemm_rooflines"] = {kname: roofline_of(kname) for kname in per_launch_ms
                                       if kname.startswith("gemm")}

    # the router that produces the layer's routing (timed on its own, same shapes)
    router = None
    try:
        rng = np.random.Generator(np.random.PCG64(77))
        logits = torch.from_numpy(rng.standard_normal((wl.n, wl.E), dtype=np.float32)).to(dev)
        rbias = (torch.from_numpy(rng.standard_normal(wl.E, dtype=np.float32)).to(dev) * cfg["bias_sigma"]
                 if cfg["bias_sigma"] > 0 else None)
        r_ids = torch.empty((wl.n, wl.k), dtype=torch.int32, device=dev)
        r_w = torch.empty((wl.n, wl.k), dtype=torch.float32, device=dev)
        r_counts = torch.empty(wl.E, dtype=torch.int32, device=dev)
        r_ms = []
        with torch.cuda.stream(stream):
            for i in range(3 + max(steps, 10)):
                flush.fill_(float(i))
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                api.router_topk(logits, rbias, r_ids, r_w, r_counts, stream=stream)
                e1.record(stream)
                r_ms.append((e0, e1))
            torch.cuda.synchronize()
        r_t = statistics.median(a.elapsed_time(b) for a, b in r_ms[3:])
        r_bytes = wl.n * wl.E * 4 + wl.n * wl.k * 8 + wl.E * 4 * (2 if rbias is not None else 1)
        router = {"ms": r_t, "bytes": r_bytes, "gbs": r_bytes / (r_t / 1000.0) / 1e9,
                  "frac_hbm": r_bytes / (r_t / 1000.0) / 1e9 / peaks["hbm_gbs"]}
    except Exception as exc:  # reported, not fatal: the layer line stands on its own
        router = {"error": str(exc)[:200]}

    # end to end through the public host-buffer entry point
    xh = torch.from_numpy(wl.x.view(np.int16)).pin_memory()
    dh = torch.from_numpy(wl.dst.view(np.int16).copy()).pin_memory()
    ih = [torch.from_numpy(r[0]).pin_memory() for r in routings]
    wh = [torch.from_numpy(r[1]).pin_memory() for r in routings]
    for i in range(3):
        layer.forward_host(xh, ih[i % N_ROUTINGS], wh[i % N_ROUTINGS], dh, stream=stream)
    e2e_steps = max(steps, 10)
    # wall time of the synchronous host-buffer call only (the L2 flush runs outside it)
    tot = 0.0
    for i in range(e2e_steps):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        layer.forward_host(xh, ih[i % N_ROUTINGS], wh[i % N_ROUTINGS], dh, stream=stream)
        tot += time.perf_counter() - t1
    e2e_ms, e2e_value = replica_throughput(1000.0 * tot / e2e_steps, wl.n, dist, dev)
    h2d = wl.n * wl.H * 2 * 2 + wl.n * wl.k * 8
    d2h = wl.n * wl.H * 2
    layer.close()
    used_graph = graphs is not None
    del layer, x, dst, ids_d, w_d, flush, graphs
    torch.cuda.empty_cache()

    rec = {
        "value": value, "unit": "tokens/s", "ms_per_step": ms, "steps": steps, "warmup": warmup,
        "config": {"workload": name, "activation": "swiglu" if args.gated else "relu2",
                   "n": wl.n, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "gemv_max_rows": T, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every step (256 MB write)", "routings": N_ROUTINGS,
                   "graph": used_graph},
        "roofline": roof,
        "layer": layer_rec,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "router": router,
        "gpu_launches": _launches_per_step(wl.n, wl.k, T) * steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    rank = dist.get_rank() if dist is not None else 0
    if rank == 0 and cpu_seconds > 0:
        rec["cpu_baseline"] = cpu_baseline(wl, cpu_seconds)
    return rec


def run_ours(args):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    api.load(build_if_missing=True)
    head = bench_workload(api, torch, args.workload, args, dev, steps=args.steps, warmup=args.warmup,
                          cpu_seconds=0.0 if args.no_cpu_baseline else args.cpu_seconds, dist=dist, local=local)
    # The metric covers decode and prefill: the other workloads are measured in
    # the same run, each with its own steps, roofline, end-to-end call and
    # oracle sample (prefill takes fewer steps: milliseconds each).
    extras = {}
    names = [] if args.workloads.strip() in ("", "none") else [w.strip() for w in args.workloads.split(",")]
    for nm in names:
        if nm == args.workload or nm not in W.CONFIGS:
            continue
        steps = args.steps if W.CONFIGS[nm]["n"] <= 64 else max(5, min(args.steps, 20))
        extras[nm] = bench_workload(api, torch, nm, args, dev, steps=steps, warmup=max(3, args.warmup),
                                    cpu_seconds=0.0 if args.no_cpu_baseline else 3.0, dist=dist, local=local)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random NVFP4 weights)",
        "config": head["config"], "roofline": head["roofline"], "layer": head["layer"], "e2e": head["e2e"],
        "router": head["router"], "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if extras:
        line["workloads"] = extras
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
