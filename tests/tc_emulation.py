"""Emulation, on the CPU, of the roundings of the tensor-core MLP path.

Test infrastructure: it reuses the oracle's features, sums and update rule
(double precision) and inserts exactly the FP16 roundings that the
tensor-core apply kernel makes, with every sum kept in double.  Its distance
to the oracle is what a perfect kernel with those operand types would show,
so the tensor-core parity bound is derived from it and not from the kernel's
own results.

Roundings (RN to FP16, as ``numpy.float16``):
  * layer-1 operand: the 28 features, each normalised (multiplied by its
    scale) and then rounded; a constant 1 against the first bias;
  * W1 rows 0..27 rounded; the first bias b1' = b1 + sum_s tau_s W1[28 + s]
    rounded once;
  * ReLU(h1) and W2 rounded; b2 added unrounded (the accumulator starts
    from it);
  * ReLU(h2), W3 and b3 unrounded (the output layer runs in FP32);
  * every FP16 rounding saturates at +-65504.

Method: "PyLO: Towards Accessible Learned Optimizers in PyTorch", section
"融合カーネル戦略" (normalised features, per-element MLP, update).
"""

from __future__ import annotations

import numpy as np

import oracle as O


def f16(x):
    """Round to nearest FP16, saturating at +-65504 as the kernel's
    conversions do."""
    x = np.clip(np.asarray(x, dtype=np.float64), -65504.0, 65504.0)
    return x.astype(np.float16).astype(np.float64)


def tc_mlp(F: np.ndarray, scales: np.ndarray, t: float, w: O.MLPWeights, perturb=None) -> np.ndarray:
    """The [n x 2] MLP output for the unnormalised feature rows F[:, :28],
    with the tensor-core path's roundings.  ``perturb`` = (rng, d_scale,
    d_feat) multiplies every normalisation scale by 1 + U(-d_scale, d_scale)
    and every feature by 1 + U(-d_feat, d_feat) before the roundings: the
    operand differences a kernel computing in fp32 may legitimately have."""
    if perturb is not None:
        rng, ds, df = perturb
        scales = scales * (1.0 + rng.uniform(-ds, ds, size=scales.shape))
        F = F * (1.0 + rng.uniform(-df, df, size=F.shape))
    X = np.zeros((F.shape[0], 29))
    X[:, :28] = f16(F[:, :28] * scales[None, :28])
    X[:, 28] = 1.0
    H = w.W1.shape[1]
    W1 = np.zeros((29, H))
    W1[:28] = f16(w.W1[:28])
    W1[28] = f16(w.b1 + O.time_features(t) @ w.W1[O.N_ELEM_FEATURES:])
    h1 = f16(np.maximum(X @ W1, 0.0))
    h2 = np.maximum(h1 @ f16(w.W2) + w.b2, 0.0)
    return h2 @ w.W3 + w.b3


def step_tensor(state: dict, t: float, lr: float, w: O.MLPWeights,
                sample_idx: np.ndarray | None = None, weight_decay: float = 0.0, perturb=None,
                S: np.ndarray | None = None) -> dict:
    """Same contract as the oracle's step_tensor (in place; with
    ``sample_idx`` only the sampled updates are returned).  ``S``: the
    oracle's square sums of the same step, if already computed."""
    R, C = state["shape"]
    n = R * C
    O.refresh_accumulators(state)
    if S is None:
        S = O.feature_square_sums(state, C, t)
    scales = O.normalisation_scales(S, n)
    idx_all = np.arange(n) if sample_idx is None else np.asarray(sample_idx, dtype=np.int64)
    new_p = np.empty(idx_all.size)
    chunk = 1 << 20
    for e0 in range(0, idx_all.size, chunk):
        idx = idx_all[e0:e0 + chunk]
        F = O.features(state["param"], state["grad"], state["mom"], state["rms"],
                       state["row"], state["col"], state["rho"], C, t, idx)
        u = O.update_from_output(tc_mlp(F, scales, t, w, perturb))
        new_p[e0:e0 + idx.size] = O.apply_update(state["param"][idx], u, lr, weight_decay)
    out = {"S": S, "scales": scales}
    if sample_idx is not None:
        out["sample_param"] = new_p
        return out
    state["param"] = new_p
    return out
