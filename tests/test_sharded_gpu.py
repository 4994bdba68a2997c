"""Row-sharded step through the C ABI, two ranks simulated on one GPU.

Each simulated rank has its own handle and its own copies of its rows (and
of the replicated column accumulators); the two sums over ranks between the
three calls are done on the host side with torch additions, the way an
all-reduce would.  The ranks' kernels never wait on each other.  Results are
compared with the oracle's unsharded step and with lopt_step on the whole
tensors."""

import numpy as np
import pytest

import oracle as O
from tests.gpu_helpers import (TOL_FP32, TOL_TC, check_param, cpu, make_states, need_gpu, rel_err,
                               to_oracle)

pytestmark = pytest.mark.gpu

SHAPES = [("a", (96, 130)), ("b", (257,)), ("c", (40, 64)), ("d", (7, 5)), ("e", (300, 33))]
PATHS = [("fp32", TOL_FP32), ("tc", TOL_TC)]


def _split(st, r0, r1, torch):
    """Rows [r0, r1) of a state as a new rank-local state (own copies)."""
    C = st["cols"]
    sl = slice(r0 * C, r1 * C)
    return {"name": st["name"], "rows": r1 - r0, "cols": C, "weight_set": st["weight_set"],
            "param": st["param"][sl].clone(), "grad": st["grad"][sl].clone(),
            "mom": [m[sl].clone() for m in st["mom"]], "rms": st["rms"][sl].clone(),
            "row": [r[r0:r1].clone() for r in st["row"]], "col": [c.clone() for c in st["col"]]}


def _engines(path, n, seed=1234):
    need_gpu()
    import synth
    from learned_optimizer_step_gb300 import LearnedOptimizer
    w = synth.make_weight_sets(1, 32, seed=seed)
    return [LearnedOptimizer(w, 32, path) for _ in range(n)], w


@pytest.mark.parametrize("path,tol", PATHS)
def test_two_simulated_ranks_match_oracle(path, tol):
    torch = need_gpu()
    states = make_states(SHAPES, recipe="vit", seed=8)
    ref = [to_oracle(s) for s in states]
    (e0, e1), w = _engines(path, 2)
    # rank 0 owns the first half of every tensor's rows (a rank-1 tensor: all of it)
    cut = [max(1, s["rows"] // 2) if s["rows"] > 1 else 1 for s in states]
    ranks = [[_split(s, 0, c, torch) for s, c in zip(states, cut)],
             [_split(s, c, s["rows"], torch) for s, c in zip(states, cut)]]
    grows = [s["rows"] for s in states]
    bufs = [e0.shard_buffers(ranks[0]), e1.shard_buffers(ranks[1])]
    for e, rk, (x1, x2) in zip((e0, e1), ranks, bufs):
        e.shard_begin(rk, grows, 2, 0.9, x1, x2)
    x1 = bufs[0][0] + bufs[1][0]
    for b in bufs:
        b[0].copy_(x1)
    for e in (e0, e1):
        e.shard_middle()
    x2 = bufs[0][1] + bufs[1][1]
    for b in bufs:
        b[1].copy_(x2)
    for e in (e0, e1):
        e.shard_end()
    e0.check()
    e1.check()
    torch.cuda.synchronize()
    ws = O.unpack_weights(w[0], 32)
    for ti, r in enumerate(ref):
        p_old = r["param"].copy()
        out = O.step_tensor(r, 2, 0.9, ws)
        got = np.concatenate([cpu(ranks[0][ti]["param"]), cpu(ranks[1][ti]["param"])])
        check_param(str(SHAPES[ti]), tol, p_old, got, r["param"])
        for k in range(3):
            for rk in ranks:
                assert rel_err(cpu(rk[ti]["col"][k]), r["col"][k]) <= 2e-6
            got_r = np.concatenate([cpu(ranks[0][ti]["row"][k]), cpu(ranks[1][ti]["row"][k])])
            assert rel_err(got_r, r["row"][k]) <= 2e-6
        S = cpu(x2)[ti * 28:(ti + 1) * 28]
        assert rel_err(S, out["S"], floor=1e-300) <= 2e-5, SHAPES[ti]
        got_m = np.concatenate([cpu(ranks[0][ti]["mom"][2]), cpu(ranks[1][ti]["mom"][2])])
        assert rel_err(got_m, r["mom"][2]) <= 2e-6


@pytest.mark.parametrize("path", ["fp32", "tc"])
def test_one_rank_owning_everything_matches_lopt_step(path):
    """With all rows on one rank (the exchange is then the identity) the
    sharded calls agree with lopt_step up to the rounding of the sums."""
    torch = need_gpu()
    a_states = make_states(SHAPES, recipe="vit", seed=9)
    b_states = make_states(SHAPES, recipe="vit", seed=9)
    (ea, eb), _ = _engines(path, 2)
    ea.step(a_states, 5, 1.0)
    x1, x2 = eb.shard_buffers(b_states)
    eb.sharded_step(b_states, [s["rows"] for s in b_states], 5, 1.0, x1, x2, lambda x: None)
    ea.check()
    eb.check()
    torch.cuda.synchronize()
    for sa, sb in zip(a_states, b_states):
        assert rel_err(cpu(sb["param"]), cpu(sa["param"])) <= 1e-5
        for k in range(3):
            assert rel_err(cpu(sb["col"][k]), cpu(sa["col"][k])) <= 1e-6


def test_phase_order_is_enforced():
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LoptError
    (e,), _ = _engines("fp32", 1)
    states = make_states(SHAPES[:2], recipe="vit", seed=10)
    with pytest.raises(LoptError):
        e.shard_middle()
    with pytest.raises(LoptError):
        e.shard_end()
    x1, x2 = e.shard_buffers(states)
    e.shard_begin(states, [s["rows"] for s in states], 1, 1.0, x1, x2)
    with pytest.raises(LoptError):          # no plain step in the middle of a sharded one
        e.step(states, 1, 1.0)
    with pytest.raises(LoptError):
        e.shard_end()
    e.shard_middle()
    e.shard_end()
    e.check()
    with pytest.raises(LoptError):           # global rows smaller than the local rows
        e.shard_begin(states, [1 for _ in states], 1, 1.0, x1, x2)
    torch.cuda.synchronize()
