"""Shared helpers of the GPU parity tests: build states with the seeded
generators, mirror them into the oracle, and compare."""

from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth

# Tolerances on updated parameters.  Primary: max-norm relative error over
# the whole updated parameter list, max|got - ref| / max|ref| (1e-5 for the
# FP32 MLP path, 2e-3 for the tensor-core path: about one unit roundoff of
# its FP16 operands, 10-bit mantissa).  Secondary, per tensor and
# element-wise:
# |got - ref| / max(|ref|, RMS of ref over the tensor), which is much
# stricter for tensors whose parameters are all update (zero-initialised
# biases at step 1): 1e-5 FP32, 1e-2 tensor cores.
TOL_FP32 = 1e-5      # FP32-FMA MLP path
TOL_TC = 2e-3        # tensor-core MLP path (FP16 operands)
TOL_ACC = 2e-6       # accumulators m, v, r, c (fp32 EMA vs fp64), element-wise
TOL_STATS = 2e-5     # per-feature sums of squares, element-wise


def elem_tol(tol: float) -> float:
    """Element-wise bound that goes with a primary (max-norm) tolerance."""
    return tol if tol <= TOL_FP32 else 1e-2


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


def norm_err(got, ref) -> float:
    """Max-norm relative error max|got - ref| / max|ref|."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def param_errors(got, ref):
    """(max-norm, element-wise) relative errors of updated parameters."""
    return norm_err(got, ref), rel_err(got, ref)


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
    num = den = 0.0
    for idx, (st, r) in enumerate(zip(states, ref)):
        sidx = None if sample is None else sample(st)
        out = O.step_tensor(r, t, lr, ws[st["weight_set"]], sample_idx=sidx)
        S = eng.feature_stats(idx)
        e_s = rel_err(S, out["S"], floor=1e-300)
        worst["stats"] = max(worst["stats"], e_s)
        if sidx is None:
            got, want = cpu(st["param"]), r["param"]
        else:
            got, want = cpu(st["param"])[sidx], out["sample_param"]
        num = max(num, float(np.max(np.abs(got - want))))
        den = max(den, float(np.max(np.abs(want))))
        e_pe = rel_err(got, want)
        worst["param_elem"] = max(worst.get("param_elem", 0.0), e_pe)
        if check_acc:
            accs = [(st["rms"], r["rms"])] + list(zip(st["mom"], r["mom"])) + \
                   list(zip(st["row"], r["row"])) + list(zip(st["col"], r["col"]))
            for g, o in accs:
                worst["acc"] = max(worst["acc"], rel_err(cpu(g), o))
        assert e_pe <= elem_tol(tol), "tensor %d %s: param element-wise rel err %.3g" % (idx, st.get("name"), e_pe)
        assert e_s <= TOL_STATS, "tensor %d: stats rel err %.3g" % (idx, e_s)
    worst["param"] = num / max(den, 1e-30)
    assert worst["param"] <= tol, "param max-norm rel err %.3g > %.3g" % (worst["param"], tol)
    if check_acc:
        assert worst["acc"] <= TOL_ACC, "accumulator rel err %.3g" % worst["acc"]
    return worst
