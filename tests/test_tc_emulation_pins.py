"""Pins for the FP16 emulation of the tensor-core MLP path (the second
reference of the tensor-core parity tests, whose distance to the oracle sets
their update gates), against facts that do not come from the emulation:

  * operands that FP16 holds exactly, with sums that stay exact: every
    rounding is then the identity and the emulation must give the oracle's
    MLP output bit for bit (a misplaced bias, scale or time feature, a
    transposed weight or a dropped ReLU breaks it);
  * random operands: the emulation's distance to the oracle stays within
    the first-order error bound of rounding the listed operands to FP16
    (unit roundoff 2^-11), and its RMS matches, within a factor of two, the
    noise that independent FP16 roundings of those operands give (an
    emulation that rounds to a wider or narrower type, or not at all, would
    pass the exact case);
  * saturation at the largest finite FP16 value;
  * the sampled route equals the whole-tensor route at the same elements.

Method: "PyLO: Towards Accessible Learned Optimizers in PyTorch", section
"融合カーネル戦略" (normalised features, per-element MLP, update).
"""

import numpy as np

import oracle as O
from tests import tc_emulation as E

U16 = 2.0 ** -11          # FP16 unit roundoff (11 significant bits)


def weights(rng, hidden, grid=None):
    """One weight set; with ``grid`` every value is a multiple of it in
    [-1, 1] (FP16-exact), else Xavier-like normals with nonzero biases."""
    shapes = [(O.D_FEAT, hidden), (hidden,), (hidden, hidden), (hidden,), (hidden, 2), (2,)]
    if grid is None:
        parts = [rng.normal(0.0, 0.5, s) for s in shapes]
    else:
        n = int(round(1.0 / grid))
        parts = [rng.integers(-n, n + 1, s) * grid for s in shapes]
    return O.unpack_weights(np.concatenate([p.ravel() for p in parts]), hidden)


def oracle_out(F, scales, t, w):
    X = np.concatenate([F[:, :O.N_ELEM_FEATURES],
                        np.broadcast_to(O.time_features(t), (F.shape[0], O.N_TIME_FEATURES))], axis=1)
    return O.mlp(O.normalise(X, scales), w)


def test_exact_operands_give_the_oracle_bitwise():
    rng = np.random.default_rng(5)
    hidden, n = 8, 300
    w = weights(rng, hidden, grid=1.0 / 8)
    w.W1[O.N_ELEM_FEATURES:] = 0.0        # tau . W1_time = 0: the first bias stays exact
    # features in {-1, -1/2, 0, 1/2, 1} / scale, scales powers of two: the
    # normalised features are FP16-exact, layer-1 products multiples of 1/16
    # with |sum| <= 29, so h1 is FP16-exact too.  Scales of 2^24 and 2^-20
    # leave raw features that FP16 cannot hold (below its smallest
    # subnormal, above its largest value): the rounding has to come after
    # the scale.
    scales = 2.0 ** rng.choice([-20, -2, -1, 0, 1, 2, 24], O.N_ELEM_FEATURES).astype(np.float64)
    F = np.zeros((n, O.D_FEAT))
    F[:, :O.N_ELEM_FEATURES] = rng.integers(-2, 3, (n, O.N_ELEM_FEATURES)) * 0.5 / scales
    for t in (1, 77):
        got = E.tc_mlp(F, scales, t, w)
        ref = oracle_out(F, scales, t, w)
        assert np.array_equal(got, ref)
        assert np.count_nonzero(ref) > n       # not a trivially zero network


def first_order_bound(F, scales, t, w):
    """|out_emu - out_exact| bound from rounding, to nearest FP16: the
    normalised features, W1 rows 0..27, the first bias with its time term,
    ReLU(h1) and W2 (each a relative change of at most U16; ReLU is
    1-Lipschitz; second-order terms get a 2 % margin)."""
    a = np.abs
    X = a(F[:, :O.N_ELEM_FEATURES] * scales[None, :])
    W1 = a(w.W1[:O.N_ELEM_FEATURES])
    b1p = a(w.b1 + O.time_features(t) @ w.W1[O.N_ELEM_FEATURES:])
    h1 = np.maximum(F[:, :O.N_ELEM_FEATURES] * scales[None, :] @ w.W1[:O.N_ELEM_FEATURES] + (
        w.b1 + O.time_features(t) @ w.W1[O.N_ELEM_FEATURES:]), 0.0)
    e1 = 2.0 * U16 * (X @ W1) + U16 * b1p             # layer-1 operands
    e1 = e1 + U16 * (h1 + e1)                         # ReLU(h1) rounded
    e2 = e1 @ a(w.W2) + U16 * ((h1 + e1) @ a(w.W2))   # W2 rounded
    return 1.02 * (e2 @ a(w.W3))


def rounding_noise_ms(F, scales, t, w):
    """Mean square of the output error that independent round-to-nearest
    FP16 errors on the same operands give, to first order.  With mantissas
    spread log-uniformly, a rounding's squared relative error averages
    (2^-10)^2 / 12 * E[1/m^2] = 0.18 U16^2, E[1/m^2] = (1/2 - 1/8) / ln 2."""
    q = (2.0 ** -10) ** 2 / 12.0 * (0.5 - 0.125) / np.log(2.0)
    X = F[:, :O.N_ELEM_FEATURES] * scales[None, :]
    W1 = w.W1[:O.N_ELEM_FEATURES]
    b1p = w.b1 + O.time_features(t) @ w.W1[O.N_ELEM_FEATURES:]
    a1 = X @ W1 + b1p
    h1 = np.maximum(a1, 0.0)
    v1 = q * (2.0 * (X ** 2) @ (W1 ** 2) + b1p ** 2)      # X and W1, b1'
    vh1 = (a1 > 0) * v1 + q * h1 ** 2                      # ReLU(h1) rounded
    a2 = h1 @ w.W2 + w.b2
    v2 = vh1 @ (w.W2 ** 2) + q * (h1 ** 2) @ (w.W2 ** 2)   # W2 rounded
    return float(np.mean(((a2 > 0) * v2) @ (w.W3 ** 2)))


def test_random_operands_carry_fp16_rounding_and_no_more():
    rng = np.random.default_rng(11)
    for hidden in (4, 32):
        w = weights(rng, hidden)
        n = 4000
        F = np.zeros((n, O.D_FEAT))
        F[:, :O.N_ELEM_FEATURES] = rng.standard_t(4, (n, O.N_ELEM_FEATURES)) * 3e-2
        scales = np.exp(rng.normal(0.0, 1.0, O.N_ELEM_FEATURES)) * 30.0
        for t in (1, 9991):
            err = E.tc_mlp(F, scales, t, w) - oracle_out(F, scales, t, w)
            bound = first_order_bound(F, scales, t, w)
            assert np.all(np.abs(err) <= bound), float(np.max(np.abs(err) / bound))
            # the RMS error against the rounding-noise model: within a factor
            # of 2 (0.63-1.49 over 20 seeds at hidden 4, 0.83-1.25 at 32);
            # BF16 roundings would sit near 8, FP32 ones near 1e-4
            ratio = float(np.sqrt(np.mean(err ** 2) / rounding_noise_ms(F, scales, t, w)))
            assert 0.5 < ratio < 2.0, (hidden, t, ratio)


def test_fp16_rounding_saturates_at_the_largest_finite_value():
    x = np.array([1e6, -1e6, 65504.0, 65519.0, 1.0 + 2.0 ** -12, 1.0 + 3 * 2.0 ** -12])
    assert E.f16(x).tolist() == [65504.0, -65504.0, 65504.0, 65504.0, 1.0, 1.0 + 2.0 ** -10]


def test_sampled_route_equals_the_whole_tensor_at_the_same_elements():
    rng = np.random.default_rng(3)
    R, C, hidden = 37, 29, 8
    w = weights(rng, hidden)
    p = rng.normal(0.0, 0.02, R * C)
    g = rng.normal(0.0, 1e-3, R * C)
    whole = O.new_state((R, C), p.copy(), g.copy())
    part = O.new_state((R, C), p.copy(), g.copy())
    E.step_tensor(whole, 3, 0.5, w)
    idx = np.array([0, 5, 28, 29, 400, R * C - 1])
    out = E.step_tensor(part, 3, 0.5, w, sample_idx=idx)
    assert np.array_equal(out["sample_param"], whole["param"][idx])
    assert np.array_equal(part["param"], p)     # the sampled route leaves p alone
