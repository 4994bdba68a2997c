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
# rough single-thread speed of the fp64 oracle on a server core, used only to
# size the reference arm's per-step sample
ORACLE_PARAMS_PER_S = 1.2e6
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
    ap.add_argument("--cpu-sample-elems", type=int, default=6_000_000)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline; never the product path)
# ---------------------------------------------------------------------------
def _oracle_sample_shapes(wl, max_elems):
    """Leading tensors of the workload, up to about max_elems parameters.  A
    leading matrix larger than the whole budget is cut to its first rows."""
    out, n = [], 0
    for name, shape in wl.shapes:
        k = 1
        for s in shape:
            k *= s
        if not out and k > max_elems and len(shape) >= 2:
            shape = (max(1, max_elems // shape[-1]),) + tuple(shape[1:])
            name, k = name + "[leading rows]", shape[0] * shape[-1]
        if out and n + k > max_elems:
            continue
        out.append((name, shape))
        n += k
        if n >= max_elems:
            break
    return out, n


def oracle_worker(workload: str, max_elems: int, steps: int) -> dict:
    """Runs in a fresh single-threaded process: times oracle steps over a
    bounded sample of the workload (inputs drawn by the same generators)."""
    import numpy as np
    import oracle as O
    import synth
    wl = synth.workloads()[workload]
    shapes, n = _oracle_sample_shapes(wl, max_elems)
    states = synth.make_list(wl, "cpu", seed=0, shapes=shapes)
    w = synth.make_weight_sets(len(shapes) if wl.per_tensor_weights else 1, wl.hidden)
    ws = [O.unpack_weights(x, wl.hidden) for x in w]
    ost = [O.new_state((s["rows"], s["cols"]), s["param"].numpy(), s["grad"].numpy(),
                       mom=[m.numpy() for m in s["mom"]], rms=s["rms"].numpy(),
                       row=[r.numpy() for r in s["row"]], col=[c.numpy() for c in s["col"]],
                       weight_set=s["weight_set"]) for s in states]
    times = []
    for k in range(steps):
        t0 = time.perf_counter()
        for st in ost:
            O.step_tensor(st, wl.first_step + k, 1.0, ws[st["weight_set"]])
        times.append(time.perf_counter() - t0)
    return {"elements": n, "tensors": len(shapes), "step_s": times}


def run_oracle_subprocess(workload: str, max_elems: int, steps: int) -> dict:
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.oracle_worker(%r, %d, %d)))" % (ROOT, workload, max_elems, steps))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle subprocess failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(workload: str, max_elems: int) -> dict:
    res = run_oracle_subprocess(workload, max_elems, 1)
    s = res["step_s"][0]
    return {"value": res["elements"] / s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%d leading tensors (%d params) of %s, one step, fp64 numpy, 1 thread"
                      % (res["tensors"], res["elements"], workload),
            "seconds": s}


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.02)
            self.lines.clear()
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

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


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
    m0..2, v; K2 reads them again and writes p, m0..2, v.  Rank-1 tensors
    ([1 x n]) also read their per-element column accumulators (3 words) in
    K1 and K2."""
    k0 = k1 = k2 = 0
    for s in states:
        n = s["rows"] * s["cols"]
        extra = 12 * n if s["rows"] == 1 else 0
        k0 += 4 * n
        k1 += 24 * n + extra
        k2 += 44 * n + extra
    return k0, k1, k2


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
    # auto: tensor cores from hidden 16 up; below that the FP32 MLP is cheaper
    path = args.mlp if not (args.mlp == "auto" and wl.hidden < 16) else "fp32"
    eng = LearnedOptimizer(w, wl.hidden, "fp32")
    if path in ("auto", "tc"):
        try:
            eng.set_mlp_path("tc")
            path = "tc"
        except Exception:
            if args.mlp == "tc":
                raise
            path = "fp32"
    prepared = eng.prepare(states)
    numel = prepared.numel
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)

    t = wl.first_step
    for _ in range(args.warmup):
        eng.step(prepared, t, 1.0, stream)
        t += 1
    eng.check()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- device-timed region (inputs resident in HBM) ----
    eng.set_kernel_timing(True)
    eng.kernel_times()
    barrier()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        start.record(stream)
        for _ in range(args.steps):
            eng.step(prepared, t, 1.0, stream)
            t += 1
        stop.record(stream)
        barrier()
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
    e0.record(stream)
    for _ in range(e2e_steps):
        eng.step_host(prepared, g_host, p_host, t, 1.0, stream)
        t += 1
    eng.host_sync(stream)   # the last parameters are in host memory
    e1.record(stream)
    barrier()
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
    avg_ms = [kms[k] / max(klaunch[k], 1) for k in range(3)]
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
    tr = traffic_per_launch(files[dom], numel)
    roof["traffic"] = tr
    step_bytes = sum(k_bytes)
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
                   "parallelism": "replica per GPU" if world > 1 else "single GPU"},
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
    """The CPU oracle timed on this host on a bounded sample per step."""
    if rank != 0:
        return None
    import synth
    wl = synth.workloads()[args.workload]
    # a bounded sample per step: the whole run stays near two minutes
    per_step = int(min(1_000_000, max(65_536, 120 * ORACLE_PARAMS_PER_S / (args.warmup + args.steps))))
    res = run_oracle_subprocess(args.workload, per_step, args.warmup + args.steps)
    times = res["step_s"][args.warmup:]
    tot = sum(times)
    value = res["elements"] * len(times) / tot
    sample = ("%d leading tensors (%d params) of %s per step, fp64 numpy oracle, 1 thread"
              % (res["tensors"], res["elements"], args.workload))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s (%d tensors in the full list)" % (args.workload, len(wl.shapes)),
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
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
