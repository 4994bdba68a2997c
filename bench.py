#!/usr/bin/env python
"""Benchmark of one learned-optimizer step (small_fc_lopt kind) on GB300.

A step = one lopt_step() over the whole synthetic parameter list (row/column
moments, feature statistics, normalise + MLP + apply).  The metric is
parameters updated per second.  Default workload: the ViT-B/16-shaped list
(150 fp32 tensors, 86,415,592 parameters), MLP 39 -> 32 -> 32 -> 2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mlp tc|fp32]
                    [--workload vit_b16|gpt2_small|decoder_1p3b|...]
                    [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload on its own GPU
(the step has no cross-tensor exchange; weak scaling).  Rank 0 prints one
JSON line.  ``--impl reference`` times the CPU oracle on a bounded sample.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "parameters updated/sec per learned-optimizer step"
UNIT = "params/s"
# Page's fused-CUDA step time on the ViT-B/16 list ("PyLO: Towards Accessible
# Learned Optimizers in PyTorch", section "ステップ時間の削減": 99.59 ms,
# hardware not stated): 86,415,592 params / 0.09959 s.
PAGE_VIT_PARAMS_PER_S = 86415592 / 0.09959
FP32_LANES_PER_SM = 128


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="vit_b16")
    ap.add_argument("--mlp", default="auto", choices=["auto", "tc", "fp32"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-groups", type=int, default=0,
                    help="most groups of tensors per host-buffer step (0: the library's default)")
    ap.add_argument("--profile-one-step", action="store_true",
                    help="after the warm-up, one extra step between cudaProfilerStart and cudaProfilerStop "
                         "(for ncu --profile-from-start off)")
    ap.add_argument("--sweep-mb", type=float, default=0.0,
                    help="single sweep through L2: groups of tensors with at most this many MB of state "
                         "run the three kernels one group after the other (0: one launch per kernel)")
    ap.add_argument("--cpu-sample-elems", type=int, default=100_000_000)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline; never the product path)
# ---------------------------------------------------------------------------
def _single_thread_env():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    os.environ["CUDA_VISIBLE_DEVICES"] = ""


def _pool_init(root):
    _single_thread_env()
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch
    torch.set_num_threads(1)


def _pool_step(job):
    """One worker task: draw tensor ``ti`` of the workload (the same
    generators as the whole list) and time ``steps`` oracle steps on it."""
    workload, ti, steps = job
    import oracle as O
    import synth
    wl = synth.workloads()[workload]
    s = synth.make_list(wl, "cpu", seed=0, indices={ti})[0]
    w = synth.make_weight_sets(1, wl.hidden, seed=1234 + (ti if wl.per_tensor_weights else 0))
    st = O.new_state((s["rows"], s["cols"]), s["param"].numpy(), s["grad"].numpy(),
                     mom=[m.numpy() for m in s["mom"]], rms=s["rms"].numpy(),
                     row=[r.numpy() for r in s["row"]], col=[c.numpy() for c in s["col"]])
    wu = O.unpack_weights(w[0], wl.hidden)
    t0 = time.perf_counter()
    for k in range(steps):
        O.step_tensor(st, wl.first_step + k, 1.0, wu)
    return s["rows"] * s["cols"], time.perf_counter() - t0


def _cpu_model():
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform_machine()


def platform_machine():
    import platform
    return platform.machine()


def oracle_pool(workload: str, tensor_ids, steps: int, cores: int) -> dict:
    """The fp64 oracle over the given tensors of the workload on ``cores``
    host cores: a process pool (spawn start, one single-threaded worker per
    core) that steps whole tensors, largest first.  Returns the wall time of
    the whole set of tensors (after the workers have started)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    import synth
    wl = synth.workloads()[workload]
    size = lambda ti: synth.numel(wl.shapes[ti][1])
    order = sorted(tensor_ids, key=size, reverse=True)
    with ctx.Pool(cores, initializer=_pool_init, initargs=(ROOT,)) as pool:
        pool.map(_pool_step, [(workload, order[-1], 1)] * cores)   # start every worker
        t0 = time.perf_counter()
        res = pool.map(_pool_step, [(workload, ti, steps) for ti in order], chunksize=1)
        wall = time.perf_counter() - t0
    n = sum(r[0] for r in res)
    return {"elements": n, "tensors": len(order), "wall_s": wall, "steps": steps,
            "cpu_s": sum(r[1] for r in res)}


def cpu_baseline(workload: str, max_elems: int) -> dict:
    """The oracle as it stands on every host core, one step over whole
    tensors of the workload: every tensor when the list has at most
    ``max_elems`` parameters, else the largest tensors first up to that many."""
    import synth
    wl = synth.workloads()[workload]
    sizes = [(synth.numel(s), ti) for ti, (_, s) in enumerate(wl.shapes)]
    ids, n = [], 0
    for k, ti in sorted(sizes, key=lambda x: x[1]):
        if n + k > max_elems and ids:
            continue
        ids.append(ti)
        n += k
    cores = min(os.cpu_count() or 1, len(ids))
    res = oracle_pool(workload, ids, 1, cores)
    total = sum(k for k, _ in sizes)
    return {"value": res["elements"] / res["wall_s"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d of %d tensors (%d of %d params, %.0f%%) of %s, one step, fp64 numpy oracle, "
                      "process pool of %d single-threaded workers (%s)"
                      % (res["tensors"], len(wl.shapes), res["elements"], total,
                         100.0 * res["elements"] / total, workload, cores, _cpu_model()),
            "seconds": res["wall_s"]}


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, sampled every few
    milliseconds by a thread of this process through NVML's read-only
    queries (libnvidia-ml through ctypes); ``leg(name)`` labels the samples
    taken from then on.  Falls back to no samples when NVML is missing."""
    NVML_CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id=None, index=0, period_s=0.005):
        import ctypes
        self.samples = []          # (leg, sm_mhz, power_w, reasons bitmask)
        self.period = period_s
        self.cur = "idle"
        self.max_mhz = None
        self.h = None
        self.error = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            rc = -1
            if pci_bus_id:
                rc = self.nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h))
            if rc != 0:
                rc = self.nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
            if rc != 0:
                raise RuntimeError("no NVML handle")
            self.h = h
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
        except Exception as e:   # no NVML: the line reports no samples
            self.error = str(e)
            self.h = None

    def _one(self):
        import ctypes
        mhz, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) != 0:
            return
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw))
        if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) != 0:
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons(self.h, ctypes.byref(rs))
        self.samples.append((self.cur, float(mhz.value), mw.value / 1e3, int(rs.value)))

    def _run(self):
        while not self.stop_flag:
            self._one()
            time.sleep(self.period)

    def __enter__(self):
        self.stop_flag = False
        if self.h is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def leg(self, name):
        self.cur = name

    def __exit__(self, *a):
        self.stop_flag = True
        if self.h is not None:
            self.thread.join(timeout=2)

    def summary(self, legs=("timed", "e2e")):
        """Median SM clock over the samples of the given legs, the reasons
        seen there, and the sample count per leg."""
        per_leg = {}
        for lg, *_ in self.samples:
            per_leg[lg] = per_leg.get(lg, 0) + 1
        sel = [s for s in self.samples if s[0] in legs]
        reasons = set()
        for _, _, _, rs in sel:
            for bit, nm in self.REASONS.items():
                if rs & bit:
                    reasons.add(nm)
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "samples_per_leg": per_leg, "source": "nvml" if self.h is not None else
                    "none (%s)" % self.error}
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sel), "samples_per_leg": per_leg,
                "power_w_max": max(s[2] for s in sel), "period_ms": self.period * 1e3,
                "source": "nvml, in-process thread"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def flat_states(wl, device, seed=0):
    """Per-tensor views into flat buffers (one allocation per state kind,
    tensors packed one after the other on 16-byte boundaries, as in a flat
    parameter buffer)."""
    import torch
    import synth
    shapes = wl.shapes
    offs, n = [], 0
    for _, shape in shapes:
        k = synth.numel(shape)
        offs.append(n)
        n += (k + 3) // 4 * 4
    rows_cols = [synth.rows_cols(s) for _, s in shapes]
    roff, coff, nr, nc = [], [], 0, 0
    for R, C in rows_cols:
        roff.append(nr); coff.append(nc)
        nr += (R + 63) // 64 * 64
        nc += (C + 63) // 64 * 64
    f = lambda m: torch.zeros(m, device=device, dtype=torch.float32)
    flat = {"param": f(n), "grad": f(n), "rms": f(n), "mom": [f(n) for _ in range(3)],
            "row": [f(nr) for _ in range(3)], "col": [f(nc) for _ in range(3)]}
    states = []
    src = synth.make_list(wl, device, seed=seed)
    for ti, ((name, shape), o) in enumerate(zip(shapes, offs)):
        k = synth.numel(shape)
        R, C = rows_cols[ti]
        st = {"name": name, "shape": shape, "rows": R, "cols": C,
              "weight_set": src[ti]["weight_set"],
              "param": flat["param"][o:o + k], "grad": flat["grad"][o:o + k],
              "rms": flat["rms"][o:o + k],
              "mom": [m[o:o + k] for m in flat["mom"]],
              "row": [r[roff[ti]:roff[ti] + R] for r in flat["row"]],
              "col": [c[coff[ti]:coff[ti] + C] for c in flat["col"]]}
        for key in ("param", "grad", "rms"):
            st[key].copy_(src[ti][key])
        for key in ("mom", "row", "col"):
            for dst, s in zip(st[key], src[ti][key]):
                dst.copy_(s)
        states.append(st)
    del src
    return states, flat, n


def _code_only(text: str) -> str:
    """Source text without comments and blank space, so that a change of
    comments alone keeps a traffic record valid."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(path: str) -> str:
    """Hash of the code (comments left out) of a kernel's source and the
    headers it includes."""
    h = hashlib.sha256()
    for name in (path, "lopt_internal.cuh", "tc_layout.cuh"):
        with open(os.path.join(ROOT, "learned_optimizer_step_gb300", "csrc", name), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(kernel_file: str, elements: int):
    """DRAM bytes per launch from the committed ncu summary, scaled to this
    workload, or None when the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(kernel_file)
    except Exception:
        return None
    if not rec or rec.get("source_sha") != kernel_source_sha(kernel_file):
        return None
    return rec["bytes_per_element"] * elements


def algorithmic_bytes(states):
    """Bytes one launch of each kernel must move: K0 reads g; K1 reads p, g,
    m0..2, v; K2 reads them again and writes p, m0..2, v.  A rank-1 tensor
    ([1 x n]) holds its column accumulators c0..2 per element: K0 reads and
    writes them, K1 and K2 read them.  The row and column accumulators of a
    2-D tensor (R + C words each, about 0.1 % of the bytes of the ViT-B/16
    list) are left out."""
    k0 = k1 = k2 = 0
    for s in states:
        n = s["rows"] * s["cols"]
        cols_per_elem = s["rows"] == 1
        k0 += 4 * n + (24 * n if cols_per_elem else 0)
        k1 += 24 * n + (12 * n if cols_per_elem else 0)
        k2 += 44 * n + (12 * n if cols_per_elem else 0)
    return k0, k1, k2


def step_floor_bytes(states):
    """The step's dependency-forced bytes: 72 per element of a 2-D tensor
    (g read once for the row/column moments; p, g, m0..2, v read twice, once
    for the statistics and once for the apply pass; p, m0..2, v written
    once) and 104 per element of a [1 x n] view, whose per-element column
    accumulators are read twice and written once as well (no separate
    row/column pass is forced there).  The kernels here move 120 for such a
    view: the row/column pass reads g and the column accumulators and writes
    them."""
    return sum((104 if s["rows"] == 1 else 72) * s["rows"] * s["cols"] for s in states)


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank's timed region ends with a barrier,
    so the job's time is the maximum."""
    if world <= 1:
        return ms
    import torch
    x = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(x, op=torch.distributed.ReduceOp.MAX)
    return float(x.item())


def job_throughput(numel_per_rank: int, world: int, steps: int, ms_total: float) -> float:
    """Whole-job parameters per second: each replica updates its own list of
    numel_per_rank parameters per step (weak scaling)."""
    return numel_per_rank * world * steps / (ms_total / 1e3)


def mlp_flops_per_element(hidden):
    return 2 * (39 * hidden + hidden * hidden + 2 * hidden)


def run_ours(args, rank, world, local_rank):
    import torch
    import synth
    from learned_optimizer_step_gb300 import LearnedOptimizer, build, MLP_TC
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()
    wl = synth.workloads()[args.workload]
    states, flat, nflat = flat_states(wl, dev)
    n_sets = len(states) if wl.per_tensor_weights else 1
    w = synth.make_weight_sets(n_sets, wl.hidden)
    # auto: the tensor-core path wherever the hidden width allows it (measured
    # faster than the FP32 MLP down to hidden 4)
    path = args.mlp
    eng = LearnedOptimizer(w, wl.hidden, "fp32")
    if path in ("auto", "tc"):
        try:
            eng.set_mlp_path("tc")
            path = "tc"
        except Exception:
            if args.mlp == "tc":
                raise
            path = "fp32"
    if args.sweep_mb > 0:
        eng.set_sweep_bytes(int(args.sweep_mb * 2 ** 20))
    if args.host_groups > 0:
        eng.set_host_groups(args.host_groups)
    prepared = eng.prepare(states)
    numel = prepared.numel
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)

    pci = None
    try:
        pci = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except AttributeError:
        pass
    clk = ClockSampler(pci, local_rank)
    clk.__enter__()
    clk.leg("warmup")
    t = wl.first_step
    for _ in range(args.warmup):
        eng.step(prepared, t, 1.0, stream)
        t += 1
    eng.check()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    if args.profile_one_step:
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        eng.step(prepared, t, 1.0, stream)
        t += 1
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()

    # ---- device-timed region (inputs resident in HBM) ----
    eng.set_kernel_timing(True)
    eng.kernel_times()
    barrier()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk.leg("timed")
    start.record(stream)
    for _ in range(args.steps):
        eng.step(prepared, t, 1.0, stream)
        t += 1
    stop.record(stream)
    barrier()
    clk.leg("idle")
    eng.check()
    ms_total = max_over_ranks(start.elapsed_time(stop), world, dev)
    kms, klaunch = eng.kernel_times()
    eng.set_kernel_timing(False)
    ms_step = ms_total / args.steps
    value = job_throughput(numel, world, args.steps, ms_total)

    # ---- end to end through the public API with host buffers ----
    # every step copies each tensor's gradient in from pinned host memory and
    # its new parameters out (lopt_step_host: groups of tensors pipelined
    # with their copies on two more streams, also across steps)
    h_g = torch.empty(nflat, dtype=torch.float32, pin_memory=True)
    h_g.copy_(flat["grad"])
    h_p = torch.empty(nflat, dtype=torch.float32, pin_memory=True)
    views = [(st["grad"].storage_offset(), st["rows"] * st["cols"]) for st in states]
    g_host = [h_g[o:o + k] for o, k in views]
    p_host = [h_p[o:o + k] for o, k in views]
    eng.step_host(prepared, g_host, p_host, t, 1.0, stream)   # first call builds the groups' schedules
    t += 1
    e2e_steps = max(3, args.steps // 2)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk.leg("e2e")
    e0.record(stream)
    for _ in range(e2e_steps):
        eng.step_host(prepared, g_host, p_host, t, 1.0, stream)
        t += 1
    eng.host_sync(stream)   # the last parameters are in host memory
    e1.record(stream)
    barrier()
    clk.leg("idle")
    clk.__exit__()
    eng.check()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = job_throughput(numel, world, e2e_steps, e2e_ms)

    if rank != 0:
        return None

    # ---- roofline of the dominant kernel ----
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    k_bytes = algorithmic_bytes(states)
    names = ["k_rowcol", "k_stats", "k_apply_tc" if path == "tc" else "k_apply_fp32"]
    files = ["k_rowcol.cu", "k_stats.cu", "k_apply_tc.cu" if path == "tc" else "k_apply.cu"]
    # each kernel's device time per step (one launch per step, or one per
    # group of the single sweep through L2)
    avg_ms = [kms[k] / args.steps for k in range(3)]
    dom = max(range(3), key=lambda k: avg_ms[k])
    sm_max = peaks.get("sm_max_mhz", 2070.0)
    fp32_peak_tflops = props.multi_processor_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    if dom == 2 and path == "fp32":
        flops = mlp_flops_per_element(32 if wl.hidden > 16 else wl.hidden) * numel
        achieved = flops / (avg_ms[2] / 1e3) / 1e12
        roof = {"kernel": names[2], "bound": "alu", "achieved": achieved,
                "peak": fp32_peak_tflops, "unit": "TFLOP/s", "frac": achieved / fp32_peak_tflops,
                "peak_source": "FP32 FMA: %d SMs x 128 lanes x 2 x %.0f MHz" %
                               (props.multi_processor_count, sm_max)}
    else:
        achieved = k_bytes[dom] / (avg_ms[dom] / 1e3) / 1e9
        roof = {"kernel": names[dom], "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": peak_src}
    # the traffic record was captured with one launch per kernel
    tr = traffic_per_launch(files[dom], numel) if args.sweep_mb <= 0 else None
    roof["traffic"] = tr
    step_bytes = step_floor_bytes(states)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / world / PAGE_VIT_PARAMS_PER_S) if args.workload == "vit_b16" else None,
        "dtype": "f32 state, f16 mma operands, f32 accumulate" if path == "tc" else "f32",
        "data": "synthetic",
        "config": {"workload": "%s (%d fp32 tensors, %d params per GPU)" % (args.workload, len(states), numel),
                   "mlp": "39->%d->%d->2, %s path" % (wl.hidden, wl.hidden, path),
                   "per_tensor_weight_sets": wl.per_tensor_weights,
                   "l2": "no flush: each step streams %.2f GB of state (> 129 MB L2)" % (step_bytes / 1e9),
                   "parallelism": "replica per GPU" if world > 1 else "single GPU",
                   **({"sweep": "L2 groups of at most %g MB of state, three launches each" % args.sweep_mb}
                      if args.sweep_mb > 0 else {})},
        "roofline": roof,
        "kernels_ms_avg": {names[k]: avg_ms[k] for k in range(3)},
        "step_roofline": {"algorithmic_bytes": step_bytes,
                          "hbm_floor_ms": step_bytes / (hbm_peak * 1e9) * 1e3,
                          "frac": (step_bytes / (hbm_peak * 1e9) * 1e3) / ms_step},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 4 * numel,
                "d2h_bytes_per_step": 4 * numel},
        "gpu_launches": sum(klaunch),
        "clocks": clk.summary(),
        "gpu": props.name,
    }
    return out


def run_reference(args, rank):
    """The CPU oracle, as it stands, timed on this host's cores: each step is
    one oracle step over a bounded sample of whole tensors of the workload
    (the same sample every step), spread over a process pool."""
    if rank != 0:
        return None
    import synth
    wl = synth.workloads()[args.workload]
    cores = os.cpu_count() or 1
    # about 0.5 M params per core per step: the whole run stays within minutes
    budget = 500_000 * cores
    ids, n = [], 0
    for ti, (_, s) in enumerate(wl.shapes):
        k = synth.numel(s)
        if n + k > budget and ids:
            continue
        ids.append(ti)
        n += k
    cores = min(cores, len(ids))
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    times = []
    with ctx.Pool(cores, initializer=_pool_init, initargs=(ROOT,)) as pool:
        pool.map(_pool_step, [(args.workload, ids[0], 1)] * cores)   # start every worker
        order = sorted(ids, key=lambda ti: synth.numel(wl.shapes[ti][1]), reverse=True)
        for _ in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            pool.map(_pool_step, [(args.workload, ti, 1) for ti in order], chunksize=1)
            times.append(time.perf_counter() - t0)
    times = times[args.warmup:]
    tot = sum(times)
    value = n * len(times) / tot
    sample = ("%d of %d tensors (%d params) of %s per step, fp64 numpy oracle, process pool of %d "
              "single-threaded workers (%s); wall time per step includes each tensor's input draw"
              % (len(ids), len(wl.shapes), n, args.workload, cores, _cpu_model()))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s (%d tensors in the full list)" % (args.workload, len(wl.shapes)),
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        out = run_ours(args, rank, world, local_rank)
        if out is not None and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_sample_elems)
        if out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
