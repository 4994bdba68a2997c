"""Shared helpers of the GPU parity tests: build states with the seeded
generators, mirror them into the oracle, and compare."""

from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth

# Tolerances (reading R10, per tensor, element by element).
#  * Updated parameters p_new: |got - ref| / max(|ref|, RMS of ref over the
#    tensor) <= TOL_P[path]: 1e-5 on the FP32 path (FP32 arithmetic), 2e-3
#    on the tensor-core path (TF32/BF16-class operands).  On the tensor-core path the bound applies
#    to every tensor that is not made of update, i.e. whose pre-step RMS is at
#    least ten times the RMS of its update; a zero-initialised bias after a
#    few steps is all update and is held by the update gate alone.
#  * The update itself, dp = p_old - p_new, against the oracle's
#    lr * (u + wd * p_old): |dp_got - dp_ref| <= TOL_DP[path] * max(|dp_ref|,
#    RMS of dp_ref over the tensor) + one fp32 ulp of p_new (the result is
#    stored in fp32).  FP32 path 1e-5.  Tensor-core path: twice the largest
#    error of an exact FP16-operand MLP (tests/tc_emulation.py) over the
#    workloads of tests/golden/tc_emulation_bound.json, which
#    tests/golden/make_tc_emulation_bound.py writes from the oracle alone.
#  * Tensor-core path only: the update against the emulation of its own
#    roundings, same metric, TOL_TC_EMU; and both update errors as the RMS
#    over the tensor's elements of the error over RMS dp_ref, TOL_TC_DP_RMS
#    and TOL_TC_EMU_RMS (the element-wise maxima sit on a few outliers where
#    one FP16 rounding step is about 1e-2 of the update's RMS; the RMS
#    errors show a systematic mistake far below that), on tensors or samples
#    of at least RMS_MIN_ELEMENTS elements.
TOL_FP32 = 1e-5      # FP32-FMA MLP path: p_new and dp
TOL_TC = 2e-3        # tensor-core MLP path: p_new of tensors not made of update
TOL_ACC = 2e-6       # accumulators m, v, r, c (fp32 EMA vs fp64), element-wise
TOL_STATS = 2e-5     # per-feature sums of squares, element-wise


def _tc_bounds():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "tc_emulation_bound.json")) as f:
        b = json.load(f)
    return (float(b["gate_dp"]), float(b["gate_emulation"]), float(b["gate_dp_rms"]),
            float(b["gate_emulation_rms"]))


# tensor-core path: the update against the oracle and against the FP16
# emulation, per element and as the RMS over the tensor
TOL_TC_DP, TOL_TC_EMU, TOL_TC_DP_RMS, TOL_TC_EMU_RMS = _tc_bounds()
MADE_OF_UPDATE = 10.0   # RMS(p_old) / RMS(dp) below which a tensor is all update
# The RMS gates hold tensors (or samples) of at least this many elements: an
# RMS over fewer is dominated by single elements, which the per-element gates
# hold (the RMS bounds are measured on whole tensors of 768 elements and more
# and on samples of 256 elements plus the two ends, as the full-size tests
# draw them).
RMS_MIN_ELEMENTS = 256


def tol_dp(tol_p: float) -> float:
    """Update gate of the path whose p_new gate is tol_p."""
    return TOL_FP32 if tol_p <= TOL_FP32 else TOL_TC_DP


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


def dp_err(p_old, got_new, ref_new) -> float:
    """Update error of one tensor: max |dp_got - dp_ref| - ulp32(p_new),
    over max(|dp_ref|, RMS of dp_ref); dp = p_old - p_new."""
    p_old = np.asarray(p_old, dtype=np.float64).ravel()
    got_new = np.asarray(got_new, dtype=np.float64).ravel()
    ref_new = np.asarray(ref_new, dtype=np.float64).ravel()
    if ref_new.size == 0:
        return 0.0
    dref = p_old - ref_new
    dgot = p_old - got_new
    rms = float(np.sqrt(np.mean(dref * dref)))
    ulp = np.spacing(np.abs(ref_new).astype(np.float32)).astype(np.float64)
    excess = np.maximum(np.abs(dgot - dref) - ulp, 0.0)
    return float(np.max(excess / np.maximum(np.abs(dref), max(rms, 1e-300))))


def dp_rms_err(p_old, got_new, ref_new) -> float:
    """RMS over the elements of (dp_got - dp_ref), over RMS dp_ref."""
    p_old = np.asarray(p_old, dtype=np.float64).ravel()
    dref = p_old - np.asarray(ref_new, dtype=np.float64).ravel()
    if dref.size == 0:
        return 0.0
    e = (p_old - np.asarray(got_new, dtype=np.float64).ravel()) - dref
    return float(np.sqrt(np.mean(e * e))) / max(float(np.sqrt(np.mean(dref * dref))), 1e-300)


def report(test: str, path: str, worst: dict) -> None:
    """Appends the worst errors a test measured to the JSON-lines file named
    by LOPT_PARITY_REPORT, when that is set (for the design notes)."""
    import json
    import os
    out = os.environ.get("LOPT_PARITY_REPORT")
    if out:
        with open(out, "a") as fh:
            fh.write(json.dumps({"test": test, "path": path, "worst": worst}) + "\n")


def made_of_update(p_old, ref_new) -> bool:
    p_old = np.asarray(p_old, dtype=np.float64).ravel()
    d = p_old - np.asarray(ref_new, dtype=np.float64).ravel()
    return float(np.sqrt(np.mean(p_old * p_old))) < MADE_OF_UPDATE * float(np.sqrt(np.mean(d * d)))


def check_param(name, tol, p_old, got_new, ref_new, emu_new=None, worst=None):
    """The p_new and dp gates of one tensor (and the emulation gate on the
    tensor-core path); records the errors in ``worst``."""
    worst = {} if worst is None else worst
    e_p = rel_err(got_new, ref_new)
    e_dp = dp_err(p_old, got_new, ref_new)
    upd = made_of_update(p_old, ref_new)
    worst["param_elem"] = max(worst.get("param_elem", 0.0), 0.0 if (upd and tol > TOL_FP32) else e_p)
    worst["dp"] = max(worst.get("dp", 0.0), e_dp)
    if not (upd and tol > TOL_FP32):
        assert e_p <= tol, "%s: p_new element-wise rel err %.3g > %.3g" % (name, e_p, tol)
    assert e_dp <= tol_dp(tol), "%s: update rel err %.3g > %.3g" % (name, e_dp, tol_dp(tol))
    big = np.asarray(ref_new).size >= RMS_MIN_ELEMENTS
    if tol > TOL_FP32 and big:
        e_r = dp_rms_err(p_old, got_new, ref_new)
        worst["dp_rms"] = max(worst.get("dp_rms", 0.0), e_r)
        assert e_r <= TOL_TC_DP_RMS, "%s: update RMS rel err %.3g > %.3g" % (name, e_r, TOL_TC_DP_RMS)
    if emu_new is not None:
        e_emu = dp_err(p_old, got_new, emu_new)
        e_er = dp_rms_err(p_old, got_new, emu_new)
        worst["dp_emu"] = max(worst.get("dp_emu", 0.0), e_emu)
        worst["dp_emu_rms"] = max(worst.get("dp_emu_rms", 0.0), e_er)
        assert e_emu <= TOL_TC_EMU, "%s: update vs FP16 emulation rel err %.3g > %.3g" % (name, e_emu, TOL_TC_EMU)
        assert not big or e_er <= TOL_TC_EMU_RMS, "%s: update vs FP16 emulation RMS rel err %.3g > %.3g" % (
            name, e_er, TOL_TC_EMU_RMS)
    return worst


def snapshot(states, tol):
    """Pre-step copies of the given GPU states for the oracle and, on the
    tensor-core path, for the FP16 emulation."""
    return [(to_oracle(s), to_oracle(s) if tol > TOL_FP32 else None) for s in states]


def check_tensor(eng, idx, st, pre, t, lr, w, tol, sidx=None, wd=0.0, worst=None, check_acc=True):
    """Steps the oracle (and the emulation) from ``pre`` = snapshot entry of
    GPU tensor ``idx`` and applies every gate to the GPU's result; ``sidx``
    restricts the parameter comparison to sampled elements."""
    from tests import tc_emulation as E
    worst = {} if worst is None else worst
    for key in ("param", "acc", "stats"):
        worst.setdefault(key, 0.0)
    r, e = pre
    p_old = r["param"].copy()
    out = O.step_tensor(r, t, lr, w, sample_idx=sidx, weight_decay=wd)
    emu_new = None
    if e is not None:
        eo = E.step_tensor(e, t, lr, w, sample_idx=sidx, weight_decay=wd, S=out["S"])
        emu_new = e["param"] if sidx is None else eo["sample_param"]
    S = eng.feature_stats(idx)
    e_s = rel_err(S, out["S"], floor=1e-300)
    worst["stats"] = max(worst["stats"], e_s)
    if sidx is None:
        got, want = cpu(st["param"]), r["param"]
    else:
        got, want, p_old = cpu(st["param"])[sidx], out["sample_param"], p_old[sidx]
    worst["param"] = max(worst["param"], norm_err(got, want))
    check_param("tensor %d %s" % (idx, st.get("name")), tol, p_old, got, want, emu_new, worst)
    if check_acc:
        accs = [(st["rms"], r["rms"])] + list(zip(st["mom"], r["mom"])) + \
               list(zip(st["row"], r["row"])) + list(zip(st["col"], r["col"]))
        for g, o in accs:
            worst["acc"] = max(worst["acc"], rel_err(cpu(g), o))
        assert worst["acc"] <= TOL_ACC, "tensor %d: accumulator rel err %.3g" % (idx, worst["acc"])
    assert e_s <= TOL_STATS, "tensor %d: stats rel err %.3g" % (idx, e_s)
    return worst


def compare_step(eng, states, weights, hidden, t, lr, tol, check_acc=True, sample=None, wd=0.0):
    """One GPU step and one oracle step from identical inputs; returns the
    worst relative errors (params, update, accumulators, stats)."""
    torch = need_gpu()
    pre = snapshot(states, tol)
    eng.step(states, t, lr)
    eng.check()
    torch.cuda.synchronize()
    ws = [O.unpack_weights(weights[i], hidden) for i in range(weights.shape[0])]
    worst = {"param": 0.0, "acc": 0.0, "stats": 0.0}
    for idx, (st, pr) in enumerate(zip(states, pre)):
        sidx = None if sample is None else sample(st)
        check_tensor(eng, idx, st, pr, t, lr, ws[st["weight_set"]], tol, sidx, wd, worst, check_acc)
    return worst
