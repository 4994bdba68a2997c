"""GPU parity of lopt_step (through the C ABI) against the CPU oracle.

Every test feeds identical seeded inputs to both sides and compares element
by element (small cases) or at sampled elements plus the whole-tensor
statistics and accumulators (full-size lists).  Gates, per tensor and
element by element (tests/gpu_helpers.py): updated parameters relative to
max(|oracle value|, RMS of the tensor's oracle values) within 1e-5 on the
FP32 MLP path and 2e-3 on the tensor-core path (there for every tensor not
made of update); the update p_old - p_new against the oracle's within 1e-5
on the FP32 path and, on the tensor-core path, within the bounds that an
exact FP16-operand emulation sets, per element and as RMS; 2e-6 on
accumulators; 2e-5 on the per-feature sums of squares."""

import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_helpers import (TOL_FP32, TOL_TC, check_param, check_tensor, compare_step, cpu, report,
                               make_states, need_gpu, rel_err, snapshot, to_oracle)

pytestmark = pytest.mark.gpu

EDGE_SHAPES = [("one", (1,)), ("scalar", ()), ("row5", (5,)), ("col7", (7, 1)),
               ("odd", (3, 5)), ("ragged", (33, 129)), ("long", (3072,)),
               ("head", (5, 1000)), ("tall", (1100, 3)), ("cube", (2, 3, 4)),
               ("w", (64, 96))]


def engine(hidden=32, n_sets=1, path="fp32", seed=1234):
    need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer
    w = synth.make_weight_sets(n_sets, hidden, seed=seed)
    return LearnedOptimizer(w, hidden, path), w


PATHS = [("fp32", TOL_FP32), ("tc", TOL_TC)]


@pytest.mark.parametrize("path,tol", PATHS)
def test_single_256x256_three_steps(path, tol):
    torch = need_gpu()
    eng, w = engine(path=path)
    wl = synth.workloads()["single_256x256"]
    states = synth.make_list(wl, "cuda", seed=0)
    for step in range(wl.steps):
        if step > 0:
            synth.refresh_grads(states, wl, step)
        compare_step(eng, states, w, 32, wl.first_step + step, 1.0, tol)


@pytest.mark.parametrize("path,tol", PATHS)
@pytest.mark.parametrize("hidden", [4, 32, 64])
def test_edge_shapes_per_tensor_weights(hidden, path, tol):
    need_gpu()
    if path == "tc" and hidden > 32:
        pytest.skip("the tensor-core path covers hidden widths up to 32")
    eng, w = engine(hidden=hidden, n_sets=len(EDGE_SHAPES), path=path)
    states = make_states(EDGE_SHAPES, recipe="vit", seed=3, per_tensor_weights=True)
    for t in (1, 2):
        compare_step(eng, states, w, hidden, t, 0.5, tol)


@pytest.mark.parametrize("path,tol", PATHS)
def test_odd_hidden_width_is_padded_exactly(path, tol):
    need_gpu()
    eng, w = engine(hidden=5, n_sets=1, path=path)
    states = make_states([("a", (17, 31)), ("b", (40,))], recipe="vit", seed=4)
    compare_step(eng, states, w, 5, 1, 1.0, tol)


@pytest.mark.parametrize("path", ["fp32", "tc"])
def test_ragged_launch_equals_solo_launches_bitwise(path):
    torch = need_gpu()
    eng, w = engine(n_sets=1, path=path)
    a = make_states(EDGE_SHAPES, recipe="vit", seed=5)
    b = make_states(EDGE_SHAPES, recipe="vit", seed=5)
    eng.step(a, 3, 1.0)
    for s in b:
        eng.step([s], 3, 1.0)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        for k in ("param", "rms"):
            assert torch.equal(x[k], y[k]), x["name"]
        for k in ("mom", "row", "col"):
            for u, v in zip(x[k], y[k]):
                assert torch.equal(u, v), x["name"]


@pytest.mark.parametrize("path", ["fp32", "tc"])
@pytest.mark.parametrize("group_bytes", [1, 24 * 40_000, 24 * 400_000])
def test_l2_groups_equal_one_launch_bitwise(path, group_bytes):
    """Single sweep through L2 (lopt_set_sweep_bytes): the list run group by
    group, from one tensor per group to a few groups, gives the same bits as
    one launch of each kernel over the whole list."""
    torch = need_gpu()
    eng, w = engine(n_sets=1, path=path)
    shapes = EDGE_SHAPES + [("big", (600, 700)), ("mid", (300, 200)), ("vec", (5000,))]
    a = make_states(shapes, recipe="vit", seed=8)
    b = make_states(shapes, recipe="vit", seed=8)
    for t in (1, 2):
        eng.set_sweep_bytes(0)
        eng.step(a, t, 1.0)
        eng.set_sweep_bytes(group_bytes)
        eng.step(b, t, 1.0)
    eng.set_sweep_bytes(0)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        for k in ("param", "rms"):
            assert torch.equal(x[k], y[k]), x["name"]
        for k in ("mom", "row", "col"):
            for u, v in zip(x[k], y[k]):
                assert torch.equal(u, v), x["name"]


@pytest.mark.parametrize("path", ["fp32", "tc"])
def test_two_runs_are_bitwise_identical(path):
    torch = need_gpu()
    eng, w = engine(path=path)
    shapes = [("a", (300, 700)), ("b", (700,)), ("c", (2048, 96))]
    a = make_states(shapes, recipe="vit", seed=6)
    b = make_states(shapes, recipe="vit", seed=6)
    for t in (1, 2):
        eng.step(a, t, 1.0)
        eng.step(b, t, 1.0)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x["param"], y["param"])
        assert torch.equal(x["mom"][2], y["mom"][2])


@pytest.mark.parametrize("path,tol", PATHS)
def test_misaligned_views_take_the_scalar_path(path, tol):
    torch = need_gpu()
    eng, w = engine(path=path)
    base = make_states([("w", (40, 64))], recipe="vit", seed=7)[0]
    st = {}
    n = base["rows"] * base["cols"]
    for k in ("param", "grad", "rms"):
        buf = torch.zeros(n + 1, device="cuda")
        buf[1:].copy_(base[k])
        st[k] = buf[1:]                      # 4-byte aligned, not 16-byte
    st["mom"] = []
    for m in base["mom"]:
        buf = torch.zeros(n + 1, device="cuda")
        buf[1:].copy_(m)
        st["mom"].append(buf[1:])
    st.update(row=base["row"], col=base["col"], rows=40, cols=64, weight_set=0, name="mis")
    compare_step(eng, [st], w, 32, 1, 1.0, tol)


@pytest.mark.parametrize("path,tol", PATHS)
def test_zero_gradients(path, tol):
    """Tensors whose gradient is zero everywhere (every row and column
    accumulator stays 0: rho_k = 0 and vhat = 0, reading R2; every feature
    but p is 0 and its normalisation scale is 1/sqrt(eps)), a tensor with an
    all-zero row and column, next to ordinary tensors; two steps."""
    need_gpu()
    eng, w = engine(path=path)
    states = make_states([("z", (64, 96)), ("w", (64, 96)), ("zb", (300,)), ("part", (40, 64))],
                         recipe="vit", seed=13)
    for t in (1, 2):
        states[0]["grad"].zero_()
        states[2]["grad"].zero_()
        g = states[3]["grad"].view(40, 64)
        g[:, 5] = 0.0
        g[7, :] = 0.0
        compare_step(eng, states, w, 32, t, 1.0, tol)
        if t == 1:
            synth.refresh_grads(states, synth.Workload("z", (), 1, 1, "vit"), 1)


def test_validation_leaves_state_untouched():
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LoptError
    eng, w = engine()
    st = make_states([("w", (16, 16))], recipe="vit", seed=8)[0]
    before = st["param"].clone()
    bad = dict(st)
    bad["mom"] = [st["mom"][0], st["mom"][0], st["mom"][2]]   # aliasing
    with pytest.raises(LoptError) as ei:
        eng.step([bad], 1, 1.0)
    assert ei.value.code == -8
    bad = dict(st)
    bad["weight_set"] = 3
    with pytest.raises(LoptError) as ei:
        eng.step([bad], 1, 1.0)
    assert ei.value.code == -1
    torch.cuda.synchronize()
    assert torch.equal(before, st["param"])


def test_resume_from_saved_state_is_bitwise_identical():
    torch = need_gpu()
    eng, w = engine()
    shapes = [("a", (64, 80)), ("b", (80,))]
    wl = synth.Workload("r", tuple(shapes), 4, 1, "vit")
    a = synth.make_list(wl, "cuda", seed=9)
    for t in (1, 2):
        synth.refresh_grads(a, wl, t)
        eng.step(a, t, 1.0)
    saved = [{k: (v.clone() if hasattr(v, "clone") else [x.clone() for x in v] if isinstance(v, list) else v)
              for k, v in s.items()} for s in a]
    eng2, _ = engine()
    for t in (3, 4):
        synth.refresh_grads(a, wl, t)
        synth.refresh_grads(saved, wl, t)
        eng.step(a, t, 1.0)
        eng2.step(saved, t, 1.0)
    torch.cuda.synchronize()
    for x, y in zip(a, saved):
        assert torch.equal(x["param"], y["param"])


@pytest.mark.parametrize("path,tol", PATHS)
def test_identity_mlp_is_normalised_sgd_on_gpu(path, tol):
    """Closed form on the GPU: routing weights make the step normalised SGD."""
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer
    H = 32
    W1 = np.zeros((39, H)); W1[1, 0] = 1.0; W1[1, 1] = -1.0
    W2 = np.zeros((H, H)); W2[0, 0] = 1.0; W2[1, 1] = 1.0
    W3 = np.zeros((H, 2)); W3[0, 0] = 1.0; W3[1, 0] = -1.0
    wf = np.concatenate([W1.ravel(), np.zeros(H), W2.ravel(), np.zeros(H), W3.ravel(),
                         [0.0, 300.0]]).astype(np.float32)
    eng = LearnedOptimizer(wf, H, path)
    st = make_states([("w", (128, 256))], recipe="vit", seed=10)[0]
    p0 = cpu(st["param"]); g = cpu(st["grad"])
    eng.step([st], 1, 0.25)
    torch.cuda.synchronize()
    expect = p0 - 0.25 * 1e-3 * np.exp(0.3) * g / np.sqrt(np.mean(g * g) + 1e-30)
    check_param("routing", tol, p0, cpu(st["param"]), expect)


def _sample(n_per=512, seed=0):
    rng = np.random.default_rng(seed)

    def pick(st):
        n = st["rows"] * st["cols"]
        if n <= 4 * n_per:
            return np.arange(n)
        idx = rng.choice(n, size=n_per, replace=False)
        return np.unique(np.concatenate([idx, [0, n - 1]]))
    return pick


def _unique_shape_subset(states):
    seen, out = set(), []
    for s in states:
        key = (s["rows"], s["cols"], s["name"].split(".")[-1])
        if key not in seen:
            seen.add(key)
            out.append(s)
    return out


@pytest.mark.parametrize("path,tol", PATHS)
def test_vit_b16_full_size_sampled(path, tol):
    """Full ViT-B/16 list in one launch per kernel; for one tensor of each
    distinct shape the stats and accumulators are compared in full, the
    parameters and the update at sampled elements."""
    torch = need_gpu()
    eng, w = engine(path=path)
    wl = synth.workloads()["vit_b16"]
    states = synth.make_list(wl, "cuda", seed=0)
    ref_states = _unique_shape_subset(states)
    pre = dict(zip(map(id, ref_states), snapshot(ref_states, tol)))
    eng.step(states, 1, 1.0)
    eng.check()
    torch.cuda.synchronize()
    ws = O.unpack_weights(w[0], 32)
    pick = _sample()
    worst = {}
    for idx, st in enumerate(states):
        if id(st) in pre:
            check_tensor(eng, idx, st, pre[id(st)], 1, 1.0, ws, tol, pick(st), worst=worst)
    report("vit_b16", path, worst)


@pytest.mark.parametrize("path,tol", PATHS)
def test_gpt2_heavy_tails_late_step_sampled(path, tol):
    """GPT-2-small list, Student-t gradients, t = 9991 with warmed-up
    accumulators; checks the token embedding and one tensor per shape."""
    torch = need_gpu()
    eng, w = engine(path=path)
    wl = synth.workloads()["gpt2_small"]
    states = synth.make_list(wl, "cuda", seed=0)
    ref_states = _unique_shape_subset(states)
    pre = dict(zip(map(id, ref_states), snapshot(ref_states, tol)))
    eng.step(states, wl.first_step, 1.0)
    eng.check()
    torch.cuda.synchronize()
    ws = O.unpack_weights(w[0], 32)
    pick = _sample(seed=1)
    worst = {}
    for idx, st in enumerate(states):
        if id(st) in pre:
            check_tensor(eng, idx, st, pre[id(st)], wl.first_step, 1.0, ws, tol, pick(st),
                         check_acc=False, worst=worst)
    report("gpt2_small", path, worst)


@pytest.mark.parametrize("path,tol", PATHS)
def test_decoupled_weight_decay(path, tol):
    """p - lr * (update + wd * p) against the oracle with the same decay; the
    tensor list mixes staged and misaligned tensors."""
    torch = need_gpu()
    eng, w = engine(path=path)
    eng.set_weight_decay(0.05)
    states = make_states([("a", (96, 130)), ("b", (257,)), ("c", (40, 64))], recipe="vit", seed=3)
    pre = snapshot(states, tol)
    eng.step(states, 4, 0.7)
    eng.check()
    torch.cuda.synchronize()
    ws = O.unpack_weights(w[0], 32)
    for idx, (st, pr) in enumerate(zip(states, pre)):
        check_tensor(eng, idx, st, pr, 4, 0.7, ws, tol, wd=0.05)


@pytest.mark.parametrize("path", ["fp32", "tc"])
def test_zero_weight_decay_is_bitwise_the_plain_step(path):
    torch = need_gpu()
    a, _ = engine(path=path)
    b, _ = engine(path=path)
    b.set_weight_decay(0.0)
    sa = make_states([("a", (64, 200))], recipe="vit", seed=4)
    sb = make_states([("a", (64, 200))], recipe="vit", seed=4)
    a.step(sa, 1, 1.0)
    b.step(sb, 1, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(sa[0]["param"], sb[0]["param"])


def test_weight_decay_rejects_bad_values():
    need_gpu()
    from learned_optimizer_step_gb300 import LoptError
    eng, _ = engine()
    for bad in (-0.1, float("nan"), float("inf")):
        with pytest.raises(LoptError):
            eng.set_weight_decay(bad)


@pytest.mark.parametrize("path,tol", PATHS)
def test_misaligned_column_accumulators(path, tol):
    """Column accumulators 4 bytes off a 16-byte boundary: the kernels take
    their scalar routes for these tensors (the tensor-core apply kernel its
    per-element one instead of four elements per lane); parity with the
    oracle as for aligned buffers."""
    torch = need_gpu()
    eng, w = engine(path=path)
    states = make_states([("w", (64, 96)), ("b", (1000,)), ("h", (5, 1000))], recipe="vit", seed=12)
    for st in states:
        cols = []
        for c in st["col"]:
            buf = torch.zeros(c.numel() + 1, device=c.device, dtype=c.dtype)
            view = buf[1:]
            view.copy_(c)
            cols.append(view)
        st["col"] = cols
    assert all(c.data_ptr() % 16 == 4 for st in states for c in st["col"])
    for t in (1, 2):
        compare_step(eng, states, w, 32, t, 1.0, tol)


def _with_biases(w, hidden, seed, scale=0.3):
    """The weight sets w with seeded non-zero biases b1, b2, b3 (the sets
    the other tests use have zero biases)."""
    w = w.copy()
    rng = np.random.default_rng(seed)
    b1 = 39 * hidden
    b2 = b1 + hidden + hidden * hidden
    b3 = b2 + hidden + 2 * hidden
    for s in range(w.shape[0]):
        w[s, b1:b1 + hidden] = rng.normal(0.0, scale, hidden)
        w[s, b2:b2 + hidden] = rng.normal(0.0, scale, hidden)
        w[s, b3:b3 + 2] = rng.normal(0.0, scale, 2)
    return w


@pytest.mark.parametrize("path,tol", PATHS)
@pytest.mark.parametrize("hidden", [4, 32])
def test_nonzero_biases(hidden, path, tol):
    """Every bias of the MLP non-zero: b1 (the tensor-core path takes it
    through a constant column of layer 1's A operand), b2 and b3."""
    need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer
    w = _with_biases(synth.make_weight_sets(2, hidden, seed=77), hidden, seed=78)
    eng = LearnedOptimizer(w, hidden, path)
    shapes = [("w", (64, 96)), ("b", (1000,)), ("odd", (37, 101)), ("tall", (1100, 3))]
    states = make_states(shapes, recipe="vit", seed=21)
    for i, st in enumerate(states):
        st["weight_set"] = i % 2
    for t in (1, 2):
        compare_step(eng, states, w, hidden, t, 1.0, tol)
