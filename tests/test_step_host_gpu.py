"""Steps with host-memory gradients and parameters (lopt_step_host).

The host-buffer entry point cuts the list into groups of tensors, each
stepped by its own launches while the copies of other groups (also of the
previous and the next call) run on two more streams, with the gradients in
two alternating staging buffers.  Every statistic of the step belongs to one
tensor, so the results must equal lopt_step() on the same inputs bit for
bit; a small list is also checked against the oracle through the host
buffers."""

import numpy as np
import pytest

import oracle as O
from tests.gpu_helpers import TOL_FP32, TOL_TC, check_param, cpu, make_states, need_gpu, rel_err, to_oracle

pytestmark = pytest.mark.gpu

# about 21 Mi elements: up to five groups of at least 4 Mi elements, with
# ragged and small tensors between the large ones
BIG = [("w%d" % i, (1024, 2048)) for i in range(9)] + [("b", (2048,)), ("odd", (37, 1001)),
                                                      ("w9", (1536, 1366)), ("v", (7,))]
SMALL = [("a", (96, 130)), ("b", (257,)), ("c", (40, 64)), ("d", (7, 5))]
PATHS = [("fp32", TOL_FP32), ("tc", TOL_TC)]


def _engine(path, seed=1234):
    import synth
    from learned_optimizer_step_gb300 import LearnedOptimizer
    w = synth.make_weight_sets(1, 32, seed=seed)
    return LearnedOptimizer(w, 32, path), w


def _host(states, torch, pinned=True):
    g = [s["grad"].cpu() for s in states]
    p = [torch.empty(s["rows"] * s["cols"], dtype=torch.float32) for s in states]
    if pinned:
        g = [x.pin_memory() for x in g]
        p = [x.pin_memory() for x in p]
    return g, p


@pytest.mark.parametrize("path", ["fp32", "tc"])
def test_host_step_equals_device_step_bitwise(path):
    torch = need_gpu()
    a = make_states(BIG, recipe="vit", seed=21)
    b = make_states(BIG, recipe="vit", seed=21)
    ea, _ = _engine(path)
    eb, _ = _engine(path)
    for t in (1, 2, 3):
        gen = torch.Generator(device="cuda").manual_seed(100 + t)
        for sa, sb in zip(a, b):   # a new gradient each step, the same on both sides
            sa["grad"].copy_(torch.randn(sa["grad"].shape, device="cuda", generator=gen) * 1e-3)
        g_host, p_host = _host(a, torch)
        for sb in b:
            sb["grad"].zero_()   # not used: the host step brings its own gradient
        ea.step(a, t, 0.5)
        eb.step_host(b, g_host, p_host, t, 0.5)
        ea.check()
        eb.check()               # also waits for the parameter copies
        torch.cuda.synchronize()
        for i, (sa, sb) in enumerate(zip(a, b)):
            assert torch.equal(sa["param"], sb["param"]), (BIG[i], t)
            assert not sb["grad"].any(), (BIG[i], t)
            assert np.array_equal(p_host[i].numpy(), cpu(sa["param"])), (BIG[i], t)
            for k in range(3):
                assert torch.equal(sa["mom"][k], sb["mom"][k])
                assert torch.equal(sa["row"][k], sb["row"][k])
                assert torch.equal(sa["col"][k], sb["col"][k])
            assert torch.equal(sa["rms"], sb["rms"])


@pytest.mark.parametrize("path,groups", [("fp32", 2), ("tc", 2), ("tc", 1), ("tc", 16)])
def test_back_to_back_host_steps_equal_device_steps(path, groups):
    """Four host steps enqueued without a sync in between (the copies of one
    call overlap the kernels of the next, the staging buffers alternate),
    each with its own host buffers, against four lopt_step calls; with one
    group, the default, and more groups than the list allows."""
    torch = need_gpu()
    a = make_states(BIG, recipe="vit", seed=26)
    b = make_states(BIG, recipe="vit", seed=26)
    ea, _ = _engine(path)
    eb, _ = _engine(path)
    eb.set_host_groups(groups)
    steps = []
    for t in (1, 2, 3, 4):
        gen = torch.Generator(device="cuda").manual_seed(200 + t)
        grads = [torch.randn(s["grad"].shape, device="cuda", generator=gen) * 1e-3 for s in a]
        g_host = [x.cpu().pin_memory() for x in grads]
        p_host = [torch.empty(s["rows"] * s["cols"], dtype=torch.float32).pin_memory() for s in a]
        steps.append((grads, g_host, p_host))
    expect = []
    for t, (grads, _, _) in enumerate(steps, 1):
        for sa, gr in zip(a, grads):
            sa["grad"].copy_(gr)
        ea.step(a, t, 0.5)
        expect.append([sa["param"].cpu() for sa in a])
    ea.check()
    for t, (_, g_host, p_host) in enumerate(steps, 1):
        eb.step_host(b, g_host, p_host, t, 0.5)
    eb.host_sync()
    torch.cuda.synchronize()
    eb.check()
    for t, ((_, _, p_host), want) in enumerate(zip(steps, expect), 1):
        for i, (got, w) in enumerate(zip(p_host, want)):
            assert torch.equal(got, w), (BIG[i], t)
    for sa, sb in zip(a, b):
        assert torch.equal(sa["param"], sb["param"])
        for k in range(3):
            assert torch.equal(sa["mom"][k], sb["mom"][k])


@pytest.mark.parametrize("path,tol", PATHS)
def test_host_step_matches_oracle(path, tol):
    torch = need_gpu()
    states = make_states(SMALL, recipe="vit", seed=22)
    ref = [to_oracle(s) for s in states]
    eng, w = _engine(path)
    g_host, p_host = _host(states, torch, pinned=False)   # pageable memory works too
    for s in states:
        s["grad"].fill_(float("nan"))   # not used: the gradient comes from host memory
    eng.step_host(states, g_host, p_host, 4, 0.7)
    eng.check()
    torch.cuda.synchronize()
    ws = O.unpack_weights(w[0], 32)
    for i, r in enumerate(ref):
        p_old = r["param"].copy()
        O.step_tensor(r, 4, 0.7, ws)
        got = p_host[i].numpy().astype(np.float64)
        check_param(str(SMALL[i]), tol, p_old, got, r["param"])


def test_host_step_weight_decay_and_path_follow_the_handle():
    torch = need_gpu()
    a = make_states(SMALL, recipe="vit", seed=23)
    b = make_states(SMALL, recipe="vit", seed=23)
    ea, _ = _engine("fp32")
    eb, _ = _engine("tc")
    g_host, p_host = _host(a, torch)
    eb.step_host(b, g_host, p_host, 1, 1.0)   # builds the parts on the tensor-core path
    eb.set_mlp_path("fp32")
    for e in (ea, eb):
        e.set_weight_decay(0.01)
    a2 = make_states(SMALL, recipe="vit", seed=24)
    b2 = make_states(SMALL, recipe="vit", seed=24)
    g2, p2 = _host(a2, torch)
    ea.step(a2, 2, 1.0)
    eb.step_host(b2, g2, p2, 2, 1.0)
    ea.check()
    eb.check()
    torch.cuda.synchronize()
    for sa, sb in zip(a2, b2):
        assert torch.equal(sa["param"], sb["param"])


def test_host_groups_rejects_bad_values():
    need_gpu()
    from learned_optimizer_step_gb300 import LoptError
    eng, _ = _engine("fp32")
    for bad in (0, -1, 17):
        with pytest.raises(LoptError):
            eng.set_host_groups(bad)
    eng.set_host_groups(16)


def test_host_step_rejects_bad_buffers():
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LoptError
    states = make_states(SMALL, recipe="vit", seed=25)
    eng, _ = _engine("fp32")
    g_host, p_host = _host(states, torch)
    with pytest.raises(ValueError):
        eng.step_host(states, g_host[:-1], p_host, 1, 1.0)
    with pytest.raises(TypeError):                 # device memory is not a host buffer
        eng.step_host(states, [s["grad"] for s in states], p_host, 1, 1.0)
    x1, x2 = eng.shard_buffers(states)
    eng.shard_begin(states, [s["rows"] for s in states], 1, 1.0, x1, x2)
    with pytest.raises(LoptError):                 # not in the middle of a sharded step
        eng.step_host(states, g_host, p_host, 1, 1.0)
    eng.shard_middle()
    eng.shard_end()
    eng.check()
    torch.cuda.synchronize()
