"""Pins for the CPU oracle, against facts that do not come from the oracle.

Each test fixes one part of the step with something the mathematics decides:
closed forms of the accumulators and features for constant / rank-1
gradients, the unit mean-square invariant of the normalisation, MLP weights
that reduce the whole step to normalised SGD, invariances, and an independent
scalar brute-force implementation on tiny tensors.

Method: "PyLO: Towards Accessible Learned Optimizers in PyTorch", sections
"融合カーネル戦略" (features, per-feature mean square, normalisation, MLP) and
"PyLO のライブラリ設計" (per-parameter accumulators).
"""

import math

import numpy as np
import pytest

import oracle as O

BM = (0.1, 0.5, 0.9)      # momentum decays, typed in independently here
BF = (0.1, 0.5, 0.9)      # factored decays
B2 = 0.999
XS = (1, 3, 10, 30, 100, 300, 1e3, 3e3, 1e4, 3e4, 1e5)


def zero_weights(hidden=4):
    return np.zeros(O.weight_set_size(hidden))


def pack(W1, b1, W2, b2, W3, b3):
    return np.concatenate([W1.ravel(), b1, W2.ravel(), b2, W3.ravel(), b3])


def run_constant(shape, g, k, p=None, t0=1, hidden=4):
    """k steps with the same gradient, from zero accumulators."""
    R, C = shape
    p = np.zeros(R * C) if p is None else p
    st = O.new_state(shape, p, g)
    w = O.unpack_weights(zero_weights(hidden), hidden)
    for s in range(k):
        O.step_tensor(st, t0 + s, 1.0, w)
    return st


# --------------------------------------------------------------------------
# P1: closed-form EMA accumulators
# --------------------------------------------------------------------------
@pytest.mark.parametrize("k", [1, 2, 5])
def test_p1_ema_closed_form(k):
    rng = np.random.default_rng(1)
    g = rng.normal(size=12) * 0.01
    st = run_constant((3, 4), g, k)
    for a, b in enumerate(BM):
        np.testing.assert_allclose(st["mom"][a], (1 - b ** k) * g, rtol=1e-13, atol=0)
    np.testing.assert_allclose(st["rms"], (1 - B2 ** k) * g * g, rtol=1e-12, atol=0)


# --------------------------------------------------------------------------
# P2: Adafactor rank-1 closed form (non-square, so r/c swaps fail)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("k", [1, 3])
def test_p2_factored_rank1(k):
    a = np.array([0.5, -1.0, 2.0, 0.25, 1.5])
    b = np.array([1.0, -0.3, 0.7, 2.0, -1.1, 0.4, 0.9])
    g = np.outer(a, b).ravel()
    st = run_constant((5, 7), g, k)
    ma2, mb2 = np.mean(a * a), np.mean(b * b)
    for q, beta in enumerate(BF):
        f = 1 - beta ** k
        np.testing.assert_allclose(st["row"][q], f * a * a * mb2, rtol=1e-13)
        np.testing.assert_allclose(st["col"][q], f * b * b * ma2, rtol=1e-13)
        np.testing.assert_allclose(st["rho"][q], f * ma2 * mb2, rtol=1e-13)
        i = np.arange(35) // 7
        j = np.arange(35) % 7
        vhat = O.factored_vhat(st["row"][q], st["col"][q], st["rho"][q], i, j)
        np.testing.assert_allclose(vhat, f * (a[i] ** 2) * (b[j] ** 2), rtol=1e-13)


# --------------------------------------------------------------------------
# Feature closed forms after k constant rank-1 steps
# --------------------------------------------------------------------------
@pytest.mark.parametrize("k", [1, 4])
def test_features_closed_form(k):
    a = np.array([0.5, -1.0, 2.0])
    b = np.array([1.0, -0.3, 0.7, 2.0])
    g = np.outer(a, b).ravel()
    p = np.linspace(-1, 1, 12)
    st = run_constant((3, 4), g, k, p=p)
    F = O.materialised_features(st, k)
    s = np.sign(g)
    i = np.arange(12) // 4
    j = np.arange(12) % 4
    ma2, mb2 = np.mean(a * a), np.mean(b * b)
    exp = np.zeros((12, 39))
    exp[:, 0] = p
    exp[:, 1] = g
    for q in range(3):
        exp[:, 2 + q] = (1 - BM[q] ** k) * g
    exp[:, 5] = math.sqrt(1 - B2 ** k) * np.abs(g)
    for q in range(3):
        exp[:, 6 + q] = (1 - BM[q] ** k) / math.sqrt(1 - B2 ** k) * s
    exp[:, 9] = s / math.sqrt(1 - B2 ** k)
    for q in range(3):
        exp[:, 10 + q] = s / math.sqrt(1 - BF[q] ** k)
        exp[:, 13 + q] = np.sqrt((1 - BF[q] ** k) * mb2) * np.abs(a[i])
        exp[:, 16 + q] = np.sqrt((1 - BF[q] ** k) * ma2) * np.abs(b[j])
    for x in range(3):
        for y in range(3):
            exp[:, 19 + 3 * x + y] = (1 - BM[x] ** k) / math.sqrt(1 - BF[y] ** k) * s
    for q, xs in enumerate(XS):
        exp[:, 28 + q] = math.tanh(k / xs)
    np.testing.assert_allclose(F, exp, rtol=1e-12, atol=1e-300)


# --------------------------------------------------------------------------
# P3: normalisation gives unit mean square; zero features stay zero
# --------------------------------------------------------------------------
def test_p3_unit_mean_square():
    rng = np.random.default_rng(3)
    R, C = 6, 9
    st = O.new_state((R, C), rng.normal(size=R * C) * 0.02, rng.normal(size=R * C) * 1e-3)
    O.refresh_accumulators(st)
    F = O.materialised_features(st, 2)
    S = (F[:, :28] ** 2).sum(axis=0)
    Fn = O.normalise(F, O.normalisation_scales(S, R * C))
    ms = (Fn[:, :28] ** 2).mean(axis=0)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-12)
    # time features are appended un-normalised
    np.testing.assert_array_equal(Fn[:, 28:], F[:, 28:])


def test_p3_zero_column_and_zero_gradient_are_finite():
    R, C = 4, 4
    st = O.new_state((R, C), np.zeros(R * C), np.zeros(R * C))
    rng = np.random.default_rng(4)
    W = rng.normal(size=O.weight_set_size(8))
    probe = O.new_state((R, C), np.zeros(R * C), np.zeros(R * C))
    O.refresh_accumulators(probe)
    F = O.materialised_features(probe, 1)
    assert np.all(F[:, :28] == 0.0)
    out = O.step_tensor(st, 1, 1.0, O.unpack_weights(W, 8))
    assert np.all(out["S"] == 0.0)
    assert np.all(np.isfinite(st["param"]))


# --------------------------------------------------------------------------
# P4: MLP weights that reduce the step to normalised SGD (closed form)
# --------------------------------------------------------------------------
def routing_weights(H, src, c_mag):
    """h1 = (ReLU(f[src]), ReLU(-f[src])), h2 = h1, o0 = h2_0 - h2_1, o1 = c."""
    W1 = np.zeros((39, H)); W1[src, 0] = 1.0; W1[src, 1] = -1.0
    W2 = np.zeros((H, H)); W2[0, 0] = 1.0; W2[1, 1] = 1.0
    W3 = np.zeros((H, 2)); W3[0, 0] = 1.0; W3[1, 0] = -1.0
    b3 = np.array([0.0, c_mag])
    return pack(W1, np.zeros(H), W2, np.zeros(H), W3, b3)


@pytest.mark.parametrize("lr,c_mag,H", [(1.0, 0.0, 32), (0.5, 250.0, 4)])
def test_p4_normalised_sgd(lr, c_mag, H):
    rng = np.random.default_rng(5)
    R, C = 5, 6
    p = rng.normal(size=R * C) * 0.02
    g = rng.normal(size=R * C) * 3e-4
    st = O.new_state((R, C), p, g)
    O.step_tensor(st, 1, lr, O.unpack_weights(routing_weights(H, 1, c_mag), H))
    ghat = g / np.sqrt(np.mean(g * g) + 1e-30)
    expect = p - lr * 1e-3 * math.exp(1e-3 * c_mag) * ghat
    np.testing.assert_allclose(st["param"], expect, rtol=1e-13, atol=1e-18)


def test_p4_golden_normalised_sgd():
    """Hand-computed worked example stored in tests/golden/."""
    import json, pathlib
    fx = json.loads((pathlib.Path(__file__).parent / "golden" /
                     "normalised_sgd_1x4.json").read_text())
    st = O.new_state((1, 4), fx["param"], fx["grad"])
    O.step_tensor(st, 1, fx["lr"], O.unpack_weights(
        routing_weights(fx["hidden"], 1, fx["magnitude_bias"]), fx["hidden"]))
    np.testing.assert_allclose(st["param"], fx["expected_param"], rtol=1e-15)


def test_p4_last_element_feature():
    """Route feature 27 = m_2 * rsqrt(vhat_2): constant magnitude after a
    constant rank-1 gradient, so its normalised value is sign(g)."""
    a = np.array([1.0, -2.0, 0.5]); b = np.array([0.3, -0.7])
    g = np.outer(a, b).ravel()
    p = np.zeros(6)
    st = O.new_state((3, 2), p, g)
    O.step_tensor(st, 1, 1.0, O.unpack_weights(routing_weights(4, 27, 0.0), 4))
    np.testing.assert_allclose(st["param"], -1e-3 * np.sign(g), rtol=1e-12)


def test_p4_time_feature_not_normalised():
    H = 4
    W1 = np.zeros((39, H)); W1[28, 0] = 1.0          # tau_0 = tanh(t / 1)
    W2 = np.eye(H); W3 = np.zeros((H, 2)); W3[0, 0] = 1.0
    w = pack(W1, np.zeros(H), W2, np.zeros(H), W3, np.zeros(2))
    st = O.new_state((2, 2), np.zeros(4), np.full(4, 1e-3))
    O.step_tensor(st, 1, 1.0, O.unpack_weights(w, H))
    np.testing.assert_allclose(st["param"], -1e-3 * math.tanh(1.0), rtol=1e-14)


def test_p4_second_relu_and_biases():
    H = 4
    # h1_0 = ReLU(g_hat); h2_0 = ReLU(-h1_0) = 0, h2_1 = ReLU(h1_0); o0 = h2_0 + h2_1
    W1 = np.zeros((39, H)); W1[1, 0] = 1.0
    W2 = np.zeros((H, H)); W2[0, 0] = -1.0; W2[0, 1] = 1.0
    W3 = np.zeros((H, 2)); W3[0, 0] = 1.0; W3[1, 0] = 1.0
    rng = np.random.default_rng(6)
    g = rng.normal(size=8)
    st = O.new_state((2, 4), np.zeros(8), g)
    O.step_tensor(st, 1, 1.0, O.unpack_weights(pack(W1, np.zeros(H), W2, np.zeros(H), W3, np.zeros(2)), H))
    ghat = g / np.sqrt(np.mean(g * g))
    np.testing.assert_allclose(st["param"], -1e-3 * np.maximum(ghat, 0), rtol=1e-13, atol=1e-300)
    # biases only: h1_0 = .5, h2_0 = 2*.5 - .25, o = (4*.75 + 1, 100)
    W1 = np.zeros((39, H)); b1 = np.array([0.5, 0, 0, 0])
    W2 = np.zeros((H, H)); W2[0, 0] = 2.0; b2 = np.array([-0.25, 0, 0, 0])
    W3 = np.zeros((H, 2)); W3[0, 0] = 4.0; b3 = np.array([1.0, 100.0])
    st = O.new_state((2, 4), np.ones(8), g)
    O.step_tensor(st, 1, 1.0, O.unpack_weights(pack(W1, b1, W2, b2, W3, b3), H))
    np.testing.assert_allclose(st["param"], 1.0 - 4.0 * math.exp(0.1) * 1e-3, rtol=1e-15)


# --------------------------------------------------------------------------
# P5: independent scalar brute force on tiny tensors
# --------------------------------------------------------------------------
def brute_force_step(R, C, p, g, state, t, lr, wflat, H):
    """Scalar loops with the math module only; ``state`` holds python lists."""
    n = R * C
    m = state["m"]; v = state["v"]; r = state["r"]; c = state["c"]
    for k in range(3):
        for e in range(n):
            m[k][e] = BM[k] * m[k][e] + (1 - BM[k]) * g[e]
    for e in range(n):
        v[e] = B2 * v[e] + (1 - B2) * g[e] ** 2
    rho = []
    for k in range(3):
        for i in range(R):
            s = 0.0
            for j in range(C):
                s += g[i * C + j] ** 2
            r[k][i] = BF[k] * r[k][i] + (1 - BF[k]) * s / C
        for j in range(C):
            s = 0.0
            for i in range(R):
                s += g[i * C + j] ** 2
            c[k][j] = BF[k] * c[k][j] + (1 - BF[k]) * s / R
        rho.append(sum(r[k]) / R)
    feats = []
    for e in range(n):
        i, j = divmod(e, C)
        rv = 1 / math.sqrt(v[e] + 1e-30)
        vh = [r[k][i] * c[k][j] / rho[k] if rho[k] > 0 else 0.0 for k in range(3)]
        rvh = [1 / math.sqrt(x + 1e-30) for x in vh]
        f = [p[e], g[e], m[0][e], m[1][e], m[2][e], math.sqrt(v[e]),
             m[0][e] * rv, m[1][e] * rv, m[2][e] * rv, g[e] * rv,
             g[e] * rvh[0], g[e] * rvh[1], g[e] * rvh[2],
             math.sqrt(r[0][i]), math.sqrt(r[1][i]), math.sqrt(r[2][i]),
             math.sqrt(c[0][j]), math.sqrt(c[1][j]), math.sqrt(c[2][j])]
        for a in range(3):
            for b in range(3):
                f.append(m[a][e] * rvh[b])
        feats.append(f)
    scale = []
    for d in range(28):
        s = sum(feats[e][d] ** 2 for e in range(n))
        scale.append(1 / math.sqrt(s / n + 1e-30))
    tau = [math.tanh(t / x) for x in XS]
    # weights
    o = 0
    W1 = [[wflat[o + d * H + h] for h in range(H)] for d in range(39)]; o += 39 * H
    b1 = list(wflat[o:o + H]); o += H
    W2 = [[wflat[o + a * H + h] for h in range(H)] for a in range(H)]; o += H * H
    b2 = list(wflat[o:o + H]); o += H
    W3 = [[wflat[o + a * 2 + h] for h in range(2)] for a in range(H)]; o += 2 * H
    b3 = list(wflat[o:o + 2])
    newp = []
    for e in range(n):
        x = [feats[e][d] * scale[d] for d in range(28)] + tau
        h1 = [max(0.0, b1[h] + sum(x[d] * W1[d][h] for d in range(39))) for h in range(H)]
        h2 = [max(0.0, b2[h] + sum(h1[a] * W2[a][h] for a in range(H))) for h in range(H)]
        out = [b3[q] + sum(h2[a] * W3[a][q] for a in range(H)) for q in range(2)]
        newp.append(p[e] - lr * out[0] * math.exp(out[1] * 1e-3) * 1e-3)
    return newp


@pytest.mark.parametrize("R,C,H", [(2, 3, 4), (1, 4, 8), (3, 1, 4), (1, 1, 4)])
def test_p5_brute_force(R, C, H):
    rng = np.random.default_rng(10 * R + C)
    n = R * C
    W = rng.normal(size=O.weight_set_size(H)) * 0.7
    p = list(rng.normal(size=n) * 0.02)
    bf = {"m": [[0.0] * n for _ in range(3)], "v": [0.0] * n,
          "r": [[0.0] * R for _ in range(3)], "c": [[0.0] * C for _ in range(3)]}
    st = O.new_state((R, C), np.array(p), np.zeros(n))
    w = O.unpack_weights(W, H)
    for t in (1, 2, 3):
        g = list(rng.normal(size=n) * 1e-3)
        st["grad"] = np.array(g)
        O.step_tensor(st, t, 0.7, w)
        p = brute_force_step(R, C, p, g, bf, t, 0.7, list(W), H)
        np.testing.assert_allclose(st["param"], p, rtol=1e-12, atol=1e-300)
        for k in range(3):
            np.testing.assert_allclose(st["mom"][k], bf["m"][k], rtol=1e-14)
            np.testing.assert_allclose(st["row"][k], bf["r"][k], rtol=1e-13)
            np.testing.assert_allclose(st["col"][k], bf["c"][k], rtol=1e-13)
        np.testing.assert_allclose(st["rms"], bf["v"], rtol=1e-14)


# --------------------------------------------------------------------------
# P6: invariances
# --------------------------------------------------------------------------
def test_p6_gradient_scale_invariance():
    """From zero accumulators every per-element feature is homogeneous in g
    (degree 0 or 1), so the normalised features and the update do not change
    when g is scaled."""
    rng = np.random.default_rng(7)
    R, C, H = 4, 5, 8
    p = rng.normal(size=R * C) * 0.02
    g = rng.normal(size=R * C) * 1e-4
    W = O.unpack_weights(rng.normal(size=O.weight_set_size(H)), H)
    s1 = O.new_state((R, C), p, g)
    s2 = O.new_state((R, C), p, 1000.0 * g)
    O.step_tensor(s1, 1, 1.0, W)
    O.step_tensor(s2, 1, 1.0, W)
    np.testing.assert_allclose(s1["param"], s2["param"], rtol=1e-11)


def test_p6_row_and_column_permutation():
    rng = np.random.default_rng(8)
    R, C, H = 4, 6, 8
    p = rng.normal(size=(R, C)) * 0.02
    g = rng.normal(size=(R, C)) * 1e-3
    W = O.unpack_weights(rng.normal(size=O.weight_set_size(H)), H)
    pr = rng.permutation(R); pc = rng.permutation(C)
    a = O.new_state((R, C), p.ravel(), g.ravel())
    b = O.new_state((R, C), p[pr][:, pc].ravel(), g[pr][:, pc].ravel())
    O.step_tensor(a, 2, 1.0, W)
    O.step_tensor(b, 2, 1.0, W)
    np.testing.assert_allclose(a["param"].reshape(R, C)[pr][:, pc],
                               b["param"].reshape(R, C), rtol=1e-12)
    np.testing.assert_allclose(a["row"][1][pr], b["row"][1], rtol=1e-14)
    np.testing.assert_allclose(a["col"][2][pc], b["col"][2], rtol=1e-14)


# --------------------------------------------------------------------------
# P7: indexing with tagged values
# --------------------------------------------------------------------------
def test_p7_indexing_tags():
    R, C = 3, 5
    g = (1.0 + np.arange(R * C)) * 1e-3
    st = O.new_state((R, C), np.zeros(R * C), g)
    O.refresh_accumulators(st)
    G = g.reshape(R, C) ** 2
    for k in range(3):
        np.testing.assert_allclose(st["row"][k], (1 - BF[k]) * G.mean(axis=1), rtol=1e-15)
        np.testing.assert_allclose(st["col"][k], (1 - BF[k]) * G.mean(axis=0), rtol=1e-15)
    F = O.materialised_features(st, 1)
    e = np.arange(R * C)
    np.testing.assert_allclose(F[:, 13], np.sqrt(st["row"][0][e // C]), rtol=1e-15)
    np.testing.assert_allclose(F[:, 18], np.sqrt(st["col"][2][e % C]), rtol=1e-15)
    np.testing.assert_array_equal(F[:, 1], g)


def test_view_rules():
    assert O.view_rows_cols(()) == (1, 1)
    assert O.view_rows_cols((7,)) == (1, 7)
    assert O.view_rows_cols((2, 3, 4)) == (6, 4)
    assert O.weight_set_size(32) == 39 * 32 + 32 + 32 * 32 + 32 + 64 + 2


# ---------------------------------------------------------------------------
# P8: decoupled weight decay (reading R11)
# ---------------------------------------------------------------------------
def _zero_output_weights(H):
    """Any W1, W2; zero output layer, so the learned update is exactly 0."""
    rng = np.random.default_rng(11)
    n = O.weight_set_size(H)
    w = rng.normal(size=n) * 0.3
    w[n - 2 * H - 2:] = 0.0      # W3[H][2] and b3[2] are the last 2H + 2 floats
    return w


@pytest.mark.parametrize("lr,wd", [(1.0, 0.1), (0.3, 1e-2), (2.0, 0.0)])
def test_p8_weight_decay_alone_is_geometric(lr, wd):
    """With the learned update identically zero, one step multiplies every
    parameter by exactly (1 - lr * wd)."""
    rng = np.random.default_rng(12)
    R, C = 4, 7
    p = rng.normal(size=R * C)
    st = O.new_state((R, C), p, rng.normal(size=R * C) * 1e-3)
    O.step_tensor(st, 3, lr, O.unpack_weights(_zero_output_weights(8), 8), weight_decay=wd)
    np.testing.assert_allclose(st["param"], p * (1.0 - lr * wd), rtol=1e-15, atol=0)


def test_p8_weight_decay_on_normalised_sgd():
    """Identity routing plus decay: p - lr * (1e-3 e^(1e-3 c) g_hat + wd p),
    decay taken on the parameter before the step."""
    rng = np.random.default_rng(13)
    R, C, lr, wd, c_mag = 3, 5, 0.7, 0.05, 40.0
    p = rng.normal(size=R * C) * 0.02
    g = rng.normal(size=R * C) * 2e-4
    st = O.new_state((R, C), p, g)
    O.step_tensor(st, 1, lr, O.unpack_weights(routing_weights(4, 1, c_mag), 4), weight_decay=wd)
    ghat = g / np.sqrt(np.mean(g * g) + 1e-30)
    expect = p - lr * (1e-3 * math.exp(1e-3 * c_mag) * ghat + wd * p)
    np.testing.assert_allclose(st["param"], expect, rtol=1e-13, atol=1e-18)


def test_p8_zero_decay_is_the_plain_step():
    rng = np.random.default_rng(14)
    w = O.unpack_weights(rng.normal(size=O.weight_set_size(8)) * 0.2, 8)
    p = rng.normal(size=12)
    g = rng.normal(size=12) * 1e-3
    a, b = O.new_state((3, 4), p, g), O.new_state((3, 4), p, g)
    O.step_tensor(a, 2, 0.5, w)
    O.step_tensor(b, 2, 0.5, w, weight_decay=0.0)
    assert np.array_equal(a["param"], b["param"])


# ---------------------------------------------------------------------------
# P9: the chunked sweeps (feature sums and the update loop run over element
# chunks only to bound host memory) against the scalar brute force
# ---------------------------------------------------------------------------
def test_p9_chunked_sweeps_match_brute_force():
    """Chunks of 5 elements over a 7 x 9 tensor: 13 chunks, the last one
    ragged (3 elements), and chunk edges that cut rows.  A dropped or
    shifted chunk changes the square sums of every feature and leaves
    elements without their update, so the brute force disagrees."""
    import oracle.lopt_oracle as L
    saved = L.CHUNK_ELEMENTS
    L.CHUNK_ELEMENTS = 5
    try:
        _p9_body()
    finally:
        L.CHUNK_ELEMENTS = saved


def _p9_body():
    rng = np.random.default_rng(21)
    R, C, H = 7, 9, 4
    n = R * C
    W = rng.normal(size=O.weight_set_size(H)) * 0.6
    p = list(rng.normal(size=n) * 0.02)
    bf = {"m": [[0.0] * n for _ in range(3)], "v": [0.0] * n,
          "r": [[0.0] * R for _ in range(3)], "c": [[0.0] * C for _ in range(3)]}
    st = O.new_state((R, C), np.array(p), np.zeros(n))
    w = O.unpack_weights(W, H)
    for t in (1, 2):
        g = list(rng.normal(size=n) * 1e-3)
        st["grad"] = np.array(g)
        p_old = st["param"].copy()
        out = O.step_tensor(st, t, 0.9, w)
        p = brute_force_step(R, C, p, g, bf, t, 0.9, list(W), H)
        np.testing.assert_allclose(st["param"], p, rtol=1e-12, atol=1e-300)
        # the square sums over all chunks equal one sum over the whole tensor
        # (features of the refreshed accumulators and the pre-step parameters)
        F = O.features(p_old, st["grad"], st["mom"], st["rms"], st["row"], st["col"],
                       st["rho"], C, t)
        np.testing.assert_allclose(out["S"], (F[:, :28] ** 2).sum(axis=0), rtol=1e-13)


# ---------------------------------------------------------------------------
# P10: the sampled path (updates at chosen elements only, used for the
# full-size checks) equals the full step at the same elements
# ---------------------------------------------------------------------------
def test_p10_sampled_path_equals_full_path():
    rng = np.random.default_rng(22)
    R, C, H = 6, 11, 8
    n = R * C
    W = O.unpack_weights(rng.normal(size=O.weight_set_size(H)) * 0.5, H)
    p = rng.normal(size=n) * 0.02
    m = [rng.normal(size=n) * 1e-3 for _ in range(3)]
    v = rng.random(n) * 1e-6
    row = [rng.random(R) * 1e-6 for _ in range(3)]
    col = [rng.random(C) * 1e-6 for _ in range(3)]
    g = rng.normal(size=n) * 1e-3
    idx = np.array([0, 5, 11, 12, 37, 40, n - 1])
    full = O.new_state((R, C), p, g, m, v, row, col)
    samp = O.new_state((R, C), p, g, m, v, row, col)
    O.step_tensor(full, 4, 0.8, W, weight_decay=0.01)
    out = O.step_tensor(samp, 4, 0.8, W, sample_idx=idx, weight_decay=0.01)
    np.testing.assert_allclose(out["sample_param"], full["param"][idx], rtol=1e-15, atol=1e-300)
    # the update itself: p_old - p_new = lr * (u + wd * p_old)
    np.testing.assert_allclose(0.8 * (out["sample_update"] + 0.01 * p[idx]),
                               p[idx] - full["param"][idx], rtol=1e-12, atol=1e-300)
    # the sampled call leaves the parameters alone but refreshes the accumulators
    np.testing.assert_array_equal(samp["param"], p)
    for k in range(3):
        np.testing.assert_array_equal(samp["mom"][k], full["mom"][k])
        np.testing.assert_array_equal(samp["col"][k], full["col"][k])
