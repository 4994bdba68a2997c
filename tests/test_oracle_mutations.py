"""Plants plausible mistakes in the CPU oracle (constants, decays, indices,
feature order, the MLP's biases, transposes and ReLUs, the update and the
weight decay) and checks that a pin catches each one.  Every mutation is applied by monkeypatching the oracle module for
the duration of one test; nothing here touches a GPU."""

import numpy as np
import pytest

import oracle
import oracle.lopt_oracle as L
from tests import test_oracle_pins as pins

PIN_TESTS = [
    lambda: pins.test_p1_ema_closed_form(2),
    lambda: pins.test_p2_factored_rank1(3),
    lambda: pins.test_features_closed_form(4),
    pins.test_p3_unit_mean_square,
    lambda: pins.test_p4_normalised_sgd(0.5, 250.0, 4),
    pins.test_p4_golden_normalised_sgd,
    pins.test_p4_last_element_feature,
    pins.test_p4_time_feature_not_normalised,
    pins.test_p4_second_relu_and_biases,
    pins.test_p6_gradient_scale_invariance,
    pins.test_p7_indexing_tags,
    lambda: pins.test_p8_weight_decay_alone_is_geometric(0.3, 1e-2),
    pins.test_p8_weight_decay_on_normalised_sgd,
    pins.test_p9_chunked_sweeps_match_brute_force,
    pins.test_p10_sampled_path_equals_full_path,
]


def _some_pin_fails():
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            return True
    return False


def _features_with(mutate):
    orig = L.features

    def f(*a, **k):
        return mutate(orig(*a, **k))
    return f


def _mlp_no_relu(layer):
    def mlp(X, w):
        z1 = X @ w.W1 + w.b1
        h1 = z1 if layer == 1 else np.maximum(z1, 0.0)
        z2 = h1 @ w.W2 + w.b2
        h2 = z2 if layer == 2 else np.maximum(z2, 0.0)
        return h2 @ w.W3 + w.b3
    return mlp


def _unpack_transposed(flat, hidden):
    w = _orig_unpack(flat, hidden)
    n = L.D_FEAT * hidden
    w.W1 = np.asarray(flat, dtype=np.float64)[:n].reshape(hidden, L.D_FEAT).T
    return w


_orig_unpack = L.unpack_weights


def _swap_index_19(F):
    F = F.copy()
    blk = F[:, 19:28].reshape(-1, 3, 3).transpose(0, 2, 1).reshape(-1, 9)
    F[:, 19:28] = blk
    return F


def _factored_sums(g2d, row, col):
    sq = g2d * g2d
    G, H = sq.sum(axis=1), sq.sum(axis=0)
    nr = [b * row[k] + (1 - b) * G for k, b in enumerate(L.FACTORED_DECAYS)]
    nc = [b * col[k] + (1 - b) * H for k, b in enumerate(L.FACTORED_DECAYS)]
    return nr, nc, [float(r.mean()) for r in nr]


def _vhat_swapped(r, c, rho, i, j):
    R, C = r.size, c.size
    e = i * C + j
    i2, j2 = e % R, (e // R) % C
    return r[i2] * c[j2] / rho if rho > 0 else np.zeros(i.shape)


def _normalise_all(F, scales):
    Fn = F.copy()
    Fn[:, :L.N_ELEM_FEATURES] *= scales[None, :]
    rms = np.sqrt((F[:, L.N_ELEM_FEATURES:] ** 2).mean(axis=0) + L.EPS)
    Fn[:, L.N_ELEM_FEATURES:] /= rms[None, :]
    return Fn


def _scales_std(S, n):
    return 1.0 / np.sqrt(S / float(n) * 2.0 + L.EPS)


def _sqrt_v_dropped(F):
    F = F.copy()
    F[:, 5] = F[:, 5] ** 2
    return F


def _swap_features(a, b):
    def f(F):
        F = F.copy()
        F[:, [a, b]] = F[:, [b, a]]
        return F
    return f


def _row_col_blocks_swapped(F):
    F = F.copy()
    F[:, 13:16], F[:, 16:19] = F[:, 16:19].copy(), F[:, 13:16].copy()
    return F


def _vhat_without_rho(r, c, rho, i, j):
    return r[i] * c[j]


def _v_of_abs_g(g, mom, rms):
    new_mom = [b * mom[k] + (1.0 - b) * g for k, b in enumerate(L.MOMENTUM_DECAYS)]
    return new_mom, L.RMS_DECAY * rms + (1.0 - L.RMS_DECAY) * np.abs(g)


def _momentum_weights_swapped(g, mom, rms):
    new_mom = [(1.0 - b) * mom[k] + b * g for k, b in enumerate(L.MOMENTUM_DECAYS)]
    return new_mom, L.RMS_DECAY * rms + (1.0 - L.RMS_DECAY) * g * g


def _mlp_variant(drop_b1=False, drop_b2=False, drop_b3=False, w2_t=False, outputs_swapped=False):
    def mlp(X, w):
        h1 = np.maximum(X @ w.W1 + (0.0 if drop_b1 else w.b1), 0.0)
        h2 = np.maximum(h1 @ (w.W2.T if w2_t else w.W2) + (0.0 if drop_b2 else w.b2), 0.0)
        W3, b3 = (w.W3[:, ::-1], w.b3[::-1]) if outputs_swapped else (w.W3, w.b3)
        return h2 @ W3 + (0.0 if drop_b3 else b3)
    return mlp


def _square_sums_last_chunk_dropped(state, cols, t):
    n = state["param"].size
    S = np.zeros(L.N_ELEM_FEATURES)
    starts = list(range(0, n, L.CHUNK_ELEMENTS))
    for e0 in starts[:-1] if len(starts) > 1 else starts:
        idx = np.arange(e0, min(n, e0 + L.CHUNK_ELEMENTS))
        S += (L._features_of(state, cols, t, idx)[:, :L.N_ELEM_FEATURES] ** 2).sum(axis=0)
    return S


def _square_sums_chunk_overlap(state, cols, t):
    n = state["param"].size
    S = np.zeros(L.N_ELEM_FEATURES)
    for e0 in range(0, n, L.CHUNK_ELEMENTS):
        idx = np.arange(e0, min(n, e0 + L.CHUNK_ELEMENTS + 1))   # one element counted twice
        S += (L._features_of(state, cols, t, idx)[:, :L.N_ELEM_FEATURES] ** 2).sum(axis=0)
    return S


_orig_step_tensor = L.step_tensor


def _step_tensor_variant(drop_last_update_chunk=False, sampled_unnormalised=False):
    def step_tensor(state, t, lr, w, sample_idx=None, weight_decay=0.0):
        R, C = state["shape"]
        n = R * C
        if sample_idx is not None and sampled_unnormalised:
            L.refresh_accumulators(state)
            S = L.feature_square_sums(state, C, t)
            F = L._features_of(state, C, t, np.asarray(sample_idx))
            u = L.update_from_output(L.mlp(F, w))
            return {"S": S, "sample_param": L.apply_update(state["param"][sample_idx], u, lr, weight_decay),
                    "sample_update": u}
        if sample_idx is not None or not drop_last_update_chunk:
            return _orig_step_tensor(state, t, lr, w, sample_idx=sample_idx, weight_decay=weight_decay)
        L.refresh_accumulators(state)
        S = L.feature_square_sums(state, C, t)
        scales = L.normalisation_scales(S, n)
        new_p = state["param"].copy()
        starts = list(range(0, n, L.CHUNK_ELEMENTS))
        for e0 in starts[:-1] if len(starts) > 1 else starts:
            idx = np.arange(e0, min(n, e0 + L.CHUNK_ELEMENTS))
            o = L.mlp(L.normalise(L._features_of(state, C, t, idx), scales), w)
            new_p[idx] = L.apply_update(state["param"][idx], L.update_from_output(o), lr, weight_decay)
        state["param"] = new_p
        return {"S": S, "scales": scales, "rho": list(state["rho"])}
    return step_tensor


MUTATIONS = {
    "square sums: last chunk dropped": ("feature_square_sums", _square_sums_last_chunk_dropped),
    "square sums: chunks overlap by one element": ("feature_square_sums", _square_sums_chunk_overlap),
    "update loop: last chunk dropped": ("step_tensor", _step_tensor_variant(drop_last_update_chunk=True)),
    "sampled path: features left unnormalised": ("step_tensor", _step_tensor_variant(sampled_unnormalised=True)),
    "epsilon 1e-8": ("EPS", 1e-8),
    "time scales reversed": ("TIME_SCALES", tuple(reversed(L.TIME_SCALES))),
    "v an EMA of |g|": ("accumulator_update", _v_of_abs_g),
    "momentum weights beta and 1 - beta swapped": ("accumulator_update", _momentum_weights_swapped),
    "vhat without 1 / rho": ("factored_vhat", _vhat_without_rho),
    "sqrt(r) and sqrt(c) blocks swapped": ("features", _features_with(_row_col_blocks_swapped)),
    "features p and g swapped": ("features", _features_with(_swap_features(0, 1))),
    "features m_0 and m_2 swapped": ("features", _features_with(_swap_features(2, 4))),
    "features m_0 rsqrt(v) and g rsqrt(vhat_0) swapped": ("features", _features_with(_swap_features(6, 10))),
    "features g rsqrt(v) and g rsqrt(vhat_0) swapped": ("features", _features_with(_swap_features(9, 10))),
    "features sqrt(r_0) and sqrt(r_2) swapped": ("features", _features_with(_swap_features(13, 15))),
    "b1 dropped": ("mlp", _mlp_variant(drop_b1=True)),
    "b2 dropped": ("mlp", _mlp_variant(drop_b2=True)),
    "b3 dropped": ("mlp", _mlp_variant(drop_b3=True)),
    "W2 read transposed": ("mlp", _mlp_variant(w2_t=True)),
    "direction and magnitude swapped": ("mlp", _mlp_variant(outputs_swapped=True)),
    "output scale 1e-2": ("OUTPUT_SCALE", 1e-2),
    "momentum decays reversed": ("MOMENTUM_DECAYS", (0.9, 0.5, 0.1)),
    "rms decay 0.99": ("RMS_DECAY", 0.99),
    "factored decays reversed": ("FACTORED_DECAYS", (0.9, 0.5, 0.1)),
    "factored sums not means": ("factored_update", _factored_sums),
    "vhat indices transposed": ("factored_vhat", _vhat_swapped),
    "feature 5 is v not sqrt(v)": ("features", _features_with(_sqrt_v_dropped)),
    "m_a*rsqrt(vhat_b) index swapped": ("features", _features_with(_swap_index_19)),
    "time features normalised": ("normalise", _normalise_all),
    "normalised by a wrong mean square": ("normalisation_scales", _scales_std),
    "no ReLU after layer 1": ("mlp", _mlp_no_relu(1)),
    "no ReLU after layer 2": ("mlp", _mlp_no_relu(2)),
    "W1 read transposed": ("unpack_weights", _unpack_transposed),
    "update sign flipped": ("update_from_output",
                            lambda o: -o[:, 0] * np.exp(o[:, 1] * 1e-3) * 1e-3),
    "magnitude not scaled": ("update_from_output",
                             lambda o: o[:, 0] * np.exp(o[:, 1]) * 1e-3),
    "time features off by one step": ("time_features",
                                      lambda t: np.tanh((float(t) + 1) / np.asarray(L.TIME_SCALES))),
    "weight decay sign flipped": ("apply_update", lambda p, u, lr, wd=0.0: p - lr * (u - wd * p)),
    "weight decay after the update": ("apply_update",
                                      lambda p, u, lr, wd=0.0: (p - lr * u) * (1.0 - lr * wd)),
    "weight decay not scaled by lr": ("apply_update", lambda p, u, lr, wd=0.0: p - lr * u - wd * p),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, value = MUTATIONS[name]
    monkeypatch.setattr(L, attr, value)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, value)
    assert _some_pin_fails(), "no pin caught: " + name


def test_unmutated_oracle_passes_all_pins():
    assert not _some_pin_fails()
