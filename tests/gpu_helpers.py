"""Shared helpers of the GPU parity tests: build states with the seeded
generators, mirror them into the oracle, and compare."""

from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth

# Tolerances (relative error against max(|oracle|, tensor RMS of oracle)).
TOL_FP32 = 1e-5      # FP32-FMA MLP path, on updated parameters
TOL_TC = 2e-3        # tensor-core MLP path (TF32 / FP16 operands)
TOL_ACC = 2e-6       # accumulators m, v, r, c (fp32 EMA vs fp64)
TOL_STATS = 2e-5     # per-feature sums of squares


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from learned_optimizer_step_gb300 import build
    build.build()
    return torch


def rel_err(got, ref, floor=None) -> float:
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if ref.size == 0:
        return 0.0
    if floor is None:
        floor = float(np.sqrt(np.mean(ref * ref)))
    denom = np.maximum(np.abs(ref), max(floor, 1e-30))
    return float(np.max(np.abs(got - ref) / denom))


def cpu(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def to_oracle(st: dict) -> dict:
    """Oracle state with exactly the GPU state's current values."""
    return O.new_state((st["rows"], st["cols"]), cpu(st["param"]), cpu(st["grad"]),
                       mom=[cpu(m) for m in st["mom"]], rms=cpu(st["rms"]),
                       row=[cpu(r) for r in st["row"]], col=[cpu(c) for c in st["col"]],
                       weight_set=st["weight_set"])


def make_states(shapes, recipe="single", seed=0, device="cuda", per_tensor_weights=False):
    wl = synth.Workload("t", tuple(shapes), 1, 1, recipe, per_tensor_weights)
    return synth.make_list(wl, device, seed=seed)


def compare_step(eng, states, weights, hidden, t, lr, tol, check_acc=True, sample=None):
    """One GPU step and one oracle step from identical inputs; returns the
    worst relative errors (params, accumulators, stats)."""
    torch = need_gpu()
    ref = [to_oracle(s) for s in states]
    eng.step(states, t, lr)
    eng.check()
    torch.cuda.synchronize()
    ws = [O.unpack_weights(weights[i], hidden) for i in range(weights.shape[0])]
    worst = {"param": 0.0, "acc": 0.0, "stats": 0.0}
    for idx, (st, r) in enumerate(zip(states, ref)):
        sidx = None if sample is None else sample(st)
        out = O.step_tensor(r, t, lr, ws[st["weight_set"]], sample_idx=sidx)
        S = eng.feature_stats(idx)
        e_s = rel_err(S, out["S"], floor=1e-300)
        worst["stats"] = max(worst["stats"], e_s)
        if sidx is None:
            e_p = rel_err(cpu(st["param"]), r["param"])
        else:
            gp = cpu(st["param"])[sidx]
            e_p = rel_err(gp, out["sample_param"])
        worst["param"] = max(worst["param"], e_p)
        if check_acc:
            accs = [(st["rms"], r["rms"])] + list(zip(st["mom"], r["mom"])) + \
                   list(zip(st["row"], r["row"])) + list(zip(st["col"], r["col"]))
            for g, o in accs:
                worst["acc"] = max(worst["acc"], rel_err(cpu(g), o))
        assert e_p <= tol, "tensor %d %s: param rel err %.3g > %.3g" % (idx, st.get("name"), e_p, tol)
        assert e_s <= TOL_STATS, "tensor %d: stats rel err %.3g" % (idx, e_s)
    if check_acc:
        assert worst["acc"] <= TOL_ACC, "accumulator rel err %.3g" % worst["acc"]
    return worst
