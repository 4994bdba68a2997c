"""GPU parity on the two largest workloads: the 1.3B-parameter decoder list
(the 50,304 x 2,048 embedding is the longest grid-wide reduction) and the
VeLO-style list (ViT-B/16 plus a 50,000 x 1,000 tensor, one MLP weight set
per tensor, hidden width 4 and 32).

The whole list runs through one lopt_step; the oracle runs once per
workload on a subset of tensors (the largest tensor, one tensor of every
other shape) and both MLP paths are compared with that one oracle result:
per-feature sums of squares and column accumulators in full, updated
parameters at sampled elements."""

import numpy as np
import pytest

import oracle as O
import synth
from tests import tc_emulation as E
from tests.gpu_helpers import TOL_FP32, TOL_TC, check_param, cpu, need_gpu, rel_err, report, to_oracle

pytestmark = pytest.mark.gpu

PATHS = [("fp32", TOL_FP32), ("tc", TOL_TC)]


def _subset(states):
    """Index of the largest tensor and of the first tensor of every other
    (rows, cols, kind) combination."""
    big = max(range(len(states)), key=lambda i: states[i]["rows"] * states[i]["cols"])
    seen, out = set(), [big]
    for i, s in enumerate(states):
        key = (s["rows"], s["cols"], s["name"].split(".")[-1])
        if key not in seen:
            seen.add(key)
            if i != big:
                out.append(i)
    return out


def _samples(st, n_per=256, seed=0):
    n = st["rows"] * st["cols"]
    if n <= 4 * n_per:
        return np.arange(n)
    rng = np.random.default_rng(seed + n)
    return np.unique(np.concatenate([rng.choice(n, size=n_per, replace=False), [0, n - 1]]))


_ORACLE = {}


def _oracle(workload, states):
    """Oracle outputs for the subset of a workload's first step, computed
    once per workload from copies of the inputs taken before the GPU step
    (the GPU-side generators give the same inputs to every test)."""
    if workload not in _ORACLE:
        wl = synth.workloads()[workload]
        n_sets = len(wl.shapes) if wl.per_tensor_weights else 1
        w = synth.make_weight_sets(n_sets, wl.hidden)
        ws = [O.unpack_weights(w[i], wl.hidden) for i in range(n_sets)]
        out = {}
        for i in _subset(states):
            st = states[i]
            r = to_oracle(st)
            e = to_oracle(st)
            sidx = _samples(st)
            p_old = r["param"][sidx].copy()
            res = O.step_tensor(r, wl.first_step, 1.0, ws[st["weight_set"]], sample_idx=sidx)
            emu = E.step_tensor(e, wl.first_step, 1.0, ws[st["weight_set"]], sample_idx=sidx, S=res["S"])
            out[i] = {"sidx": sidx, "param": res["sample_param"], "S": res["S"], "p_old": p_old,
                      "emu": emu["sample_param"],
                      "col0": r["col"][0].copy(), "mom1_sample": r["mom"][1][sidx].copy()}
        _ORACLE[workload] = out
    return _ORACLE[workload]


def _run(workload, path, tol):
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer
    wl = synth.workloads()[workload]
    n_sets = len(wl.shapes) if wl.per_tensor_weights else 1
    w = synth.make_weight_sets(n_sets, wl.hidden)
    eng = LearnedOptimizer(w, wl.hidden, path)
    states = synth.make_list(wl, "cuda", seed=0)
    ref = _oracle(workload, states)   # before the step: inputs as drawn
    eng.step(states, wl.first_step, 1.0)
    eng.check()
    torch.cuda.synchronize()
    worst = {}
    for i, r in ref.items():
        st = states[i]
        got = cpu(st["param"])[r["sidx"]]
        check_param(st["name"], tol, r["p_old"], got, r["param"], r["emu"] if tol > TOL_FP32 else None, worst=worst)
        assert rel_err(eng.feature_stats(i), r["S"], floor=1e-300) <= 2e-5, st["name"]
        assert rel_err(cpu(st["col"][0]), r["col0"]) <= 2e-6, st["name"]
        assert rel_err(cpu(st["mom"][1])[r["sidx"]], r["mom1_sample"]) <= 2e-6, st["name"]
    report(workload, path, worst)
    eng.close()
    del states
    torch.cuda.empty_cache()


@pytest.mark.timeout(1200)
@pytest.mark.parametrize("path,tol", PATHS)
def test_decoder_1p3b_sampled(path, tol):
    """1,311,625,216 parameters in 291 tensors, one launch per kernel."""
    _run("decoder_1p3b", path, tol)


@pytest.mark.timeout(1200)
@pytest.mark.parametrize("workload", ["velo_h4", "velo_h32"])
@pytest.mark.parametrize("path,tol", PATHS)
def test_velo_per_tensor_weight_sets_sampled(workload, path, tol):
    """151 tensors with 151 weight sets, up to a 50M-element tensor."""
    _run(workload, path, tol)
