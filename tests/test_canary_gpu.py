"""Out-of-bounds writes on the GPU: every array of a ragged list (p, g,
m0..2, v, r0..2, c0..2 of each tensor) is carved from one device buffer,
with guard zones of known bits before and after it.  After two steps on
each MLP path every guard must still hold its bits: a kernel that writes
past an array, or a tail it does not mask, shows up there.  The arrays are
16-byte aligned (vector routes) or all shifted by one float (scalar
routes); aligned, the results equal those of separately allocated tensors
bit for bit."""

import numpy as np
import pytest

import synth
from tests.gpu_helpers import need_gpu

GUARD = 64                      # floats before and after every array
PATTERN = -12345.6789           # guard value (any value the step never writes)
SHAPES = [("w", (96, 128)), ("b", (128,)), ("odd", (7, 13)), ("one", (1,)), ("tall", (300, 17)),
          ("wide", (3, 5000)), ("r5", (5,)), ("big", (257, 1029)), ("ln", (768,))]


def layout(states, shift):
    """(tensor index, key, k, offset, length) of every array, in floats,
    each GUARD floats after the previous one, at a multiple of 4 plus
    ``shift``; and the buffer length."""
    out, end = [], 0
    for i, s in enumerate(states):
        n, r, c = s["rows"] * s["cols"], len(s["row"][0]), len(s["col"][0])
        for key, k, ln in ([("param", None, n), ("grad", None, n), ("rms", None, n)]
                           + [("mom", k, n) for k in range(3)]
                           + [("row", k, r) for k in range(3)] + [("col", k, c) for k in range(3)]):
            off = (end + GUARD + 3) // 4 * 4 + shift
            out.append((i, key, k, off, ln))
            end = off + ln
    return out, end + GUARD


def carve(torch, states, shift):
    arrays, total = layout(states, shift)
    buf = torch.full((total,), PATTERN, dtype=torch.float32, device="cuda")
    views = [dict(name=s["name"], rows=s["rows"], cols=s["cols"], weight_set=0, mom=[None] * 3,
                  row=[None] * 3, col=[None] * 3) for s in states]
    covered = np.zeros(total, dtype=bool)
    for i, key, k, off, ln in arrays:
        v = buf[off:off + ln]
        src = states[i][key] if k is None else states[i][key][k]
        v.copy_(src)
        if k is None:
            views[i][key] = v
        else:
            views[i][key][k] = v
        covered[off:off + ln] = True
    return buf, views, covered


def test_layout_leaves_guards_and_keeps_alignment():
    """The carving itself (host arithmetic): no overlap, guards of at least
    GUARD floats everywhere, offsets aligned as asked."""
    states = [dict(rows=r, cols=c, row=[np.zeros(r)] * 3, col=[np.zeros(c)] * 3)
              for r, c in (synth.rows_cols(s) for _, s in SHAPES)]
    for shift in (0, 1):
        arrays, total = layout(states, shift)
        prev_end = 0
        for _, _, _, off, ln in arrays:
            assert off - prev_end >= GUARD and off % 4 == shift
            prev_end = off + ln
        assert total - prev_end == GUARD


@pytest.mark.gpu
@pytest.mark.parametrize("path", ["fp32", "tc"])
@pytest.mark.parametrize("shift", [0, 1])
def test_guards_around_every_array_survive_two_steps(path, shift):
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer
    w = synth.make_weight_sets(1, 32)
    wl = synth.Workload("canary", tuple(SHAPES), 1, 1, "vit")
    states = synth.make_list(wl, "cuda", seed=21)
    buf, views, covered = carve(torch, states, shift)
    eng = LearnedOptimizer(w, 32, path)
    ref = LearnedOptimizer(w, 32, path) if shift == 0 else None
    for t in (1, 2):
        eng.step(views, t, 0.5)
        if ref is not None:
            ref.step(states, t, 0.5)
    eng.check()
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    bad = np.flatnonzero(~covered & (host.view(np.uint32) != np.float32(PATTERN).view(np.uint32)))
    assert bad.size == 0, "guard words overwritten at %s" % bad[:8].tolist()
    assert np.all(np.isfinite(host[covered]))
    if ref is not None:
        ref.check()
        for v, s in zip(views, states):
            assert torch.equal(v["param"], s["param"]), v["name"]
            for k in range(3):
                assert torch.equal(v["mom"][k], s["mom"][k]), v["name"]
                assert torch.equal(v["row"][k], s["row"][k]), v["name"]
                assert torch.equal(v["col"][k], s["col"][k]), v["name"]
            assert torch.equal(v["rms"], s["rms"]), v["name"]
        ref.close()
    eng.close()
