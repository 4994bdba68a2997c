"""Double-precision CPU oracle for one ``small_fc_lopt`` learned-optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` use it.  It shares no code, tables or constants
with the CUDA library; every constant below is typed in here on its own.

Source: "PyLO: Towards Accessible Learned Optimizers in PyTorch" (MLSys 2026
talk notes).  That page describes *what* one step computes in prose only:

* per-parameter accumulators are kept and updated from the gradient
  (section "PyLO のライブラリ設計", optimiser module);
* a d_feat-wide feature vector is built per element (``construct_features``),
  each feature is divided by its root-mean-square over the whole tensor
  (``compute_squared_average`` + ``feature_normalization``), and a small MLP
  is evaluated per element (``apply_lo``) (section "融合カーネル戦略");
* the naive implementation materialises an [mn x d_feat] feature tensor in
  memory (section "ナイーブ実装のボトルネック") -- this oracle does exactly
  that, on purpose, so that every intermediate can be inspected;
* d_feat ~= 39 and d_hidden ~= 32 for ``small_fc_lopt`` (section
  "メモリ階層の活用").

The page does not list the features, the decay constants, the epsilon or the
output head.  This library adopts the usual small_fc_lopt defaults for them:
feature families p, g, three momenta (decays 0.1/0.5/0.9), one RMS (0.999),
m*rsqrt(v), Adafactor-factored RMS with three decays (0.1/0.5/0.9) and time
features; an MLP d_feat -> 32 -> 32 -> 2 with ReLU; and the output rule
``update = direction * exp(magnitude * 1e-3) * 1e-3``.  The exact list, its
order and the remaining constants are readings, named R1..R10:

R1  EMA form m <- b*m + (1-b)*g, v <- b2*v + (1-b2)*g^2, no bias correction,
    accumulators updated *before* the features are built.
R2  Adafactor factoring with row/column MEANS of g^2; vhat = r_i * c_j / rho,
    rho = mean_i r_i; vhat = 0 when rho == 0.
R3  Feature order (28 per-element + 11 time features = 39), see ``features``.
R4  eps = 1e-30 everywhere (inside every rsqrt and in the normalisation).
R5  The 11 time features are appended after normalisation, un-normalised.
R6  ReLU after both hidden layers, linear output, o0 = direction,
    o1 = magnitude.  Weights per set: W1[39][H], b1[H], W2[H][H], b2[H],
    W3[H][2], b3[2], row-major, concatenated in that order.
R7  p <- p - lr * update.
R11 Decoupled weight decay (section "学習率スケジュールと重み減衰の効果"
    reports that schedules and weight decay change what a learned
    optimiser reaches; it gives no formula): p <- p - lr * (update + wd * p)
    with the parameter before the step, wd = 0 by default (then exactly R7).
R8  t is the caller's 1-based step count.
R10 See the tests for the error metric.

Precision: float64 throughout (inputs arrive as float32 and are widened
exactly).  Big tensors are processed in element chunks only to bound host
memory; the sums over chunks are plain sums.

Pins (``tests/test_oracle_pins.py``): the page prints no worked example, and
the composition of the MLP with random (untrained) weights has no published
value.  Every stage is pinned by closed forms and invariants, and the whole
step, random weights with nonzero biases included, by an independent scalar
brute force on tiny tensors over three steps.
"""

from __future__ import annotations


from dataclasses import dataclass
from typing import List, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# Constants (readings R1-R5; decay values are the small_fc_lopt defaults).
# ---------------------------------------------------------------------------
MOMENTUM_DECAYS = (0.1, 0.5, 0.9)      # three momenta m_k
RMS_DECAY = 0.999                      # one second-moment accumulator v
FACTORED_DECAYS = (0.1, 0.5, 0.9)      # Adafactor row/column accumulators
EPS = 1e-30                            # R4
TIME_SCALES = (1.0, 3.0, 10.0, 30.0, 100.0, 300.0,
               1e3, 3e3, 1e4, 3e4, 1e5)  # R3: tau_s = tanh(t / x_s)
N_ELEM_FEATURES = 28                   # per-element features (normalised)
N_TIME_FEATURES = len(TIME_SCALES)     # 11 (not normalised, R5)
D_FEAT = N_ELEM_FEATURES + N_TIME_FEATURES  # 39
OUTPUT_SCALE = 1e-3                    # update = o0 * exp(o1 * 1e-3) * 1e-3

CHUNK_ELEMENTS = 1 << 20               # host-memory bound only


# ---------------------------------------------------------------------------
# Shapes and weights
# ---------------------------------------------------------------------------
def view_rows_cols(shape: Sequence[int]) -> tuple[int, int]:
    """[R x C] view of a parameter tensor: rank 0 -> [1x1], rank 1 -> [1xn],
    rank >= 2 -> [prod(leading) x last]."""
    shape = tuple(int(s) for s in shape)
    if len(shape) == 0:
        return 1, 1
    if len(shape) == 1:
        return 1, shape[0]
    return int(np.prod(shape[:-1])), shape[-1]


def weight_set_size(hidden: int, d_feat: int = D_FEAT) -> int:
    """Floats in one MLP weight set (R6 layout)."""
    return d_feat * hidden + hidden + hidden * hidden + hidden + hidden * 2 + 2


@dataclass
class MLPWeights:
    W1: np.ndarray  # [39, H]
    b1: np.ndarray  # [H]
    W2: np.ndarray  # [H, H]
    b2: np.ndarray  # [H]
    W3: np.ndarray  # [H, 2]
    b3: np.ndarray  # [2]


def unpack_weights(flat: np.ndarray, hidden: int) -> MLPWeights:
    """Split one flat weight set (R6 layout) into its matrices, in float64."""
    flat = np.asarray(flat, dtype=np.float64).ravel()
    if flat.size != weight_set_size(hidden):
        raise ValueError("weight set has %d floats, expected %d"
                         % (flat.size, weight_set_size(hidden)))
    o = 0

    def take(n, shape):
        nonlocal o
        a = flat[o:o + n].reshape(shape)
        o += n
        return a

    W1 = take(D_FEAT * hidden, (D_FEAT, hidden))
    b1 = take(hidden, (hidden,))
    W2 = take(hidden * hidden, (hidden, hidden))
    b2 = take(hidden, (hidden,))
    W3 = take(hidden * 2, (hidden, 2))
    b3 = take(2, (2,))
    return MLPWeights(W1, b1, W2, b2, W3, b3)


# ---------------------------------------------------------------------------
# S1: factored (Adafactor) second moment -- row/column accumulators (R2)
# ---------------------------------------------------------------------------
def factored_update(g2d: np.ndarray, row: List[np.ndarray], col: List[np.ndarray]):
    """Row/column mean of g^2, their EMAs with the three factored decays, and
    rho_k = mean_i row_k[i].  Returns (new_row, new_col, rho)."""
    sq = g2d * g2d
    row_mean = sq.mean(axis=1)          # G_i, one per row
    col_mean = sq.mean(axis=0)          # H_j, one per column
    new_row, new_col, rho = [], [], []
    for k, b in enumerate(FACTORED_DECAYS):
        r = b * row[k] + (1.0 - b) * row_mean
        c = b * col[k] + (1.0 - b) * col_mean
        new_row.append(r)
        new_col.append(c)
        rho.append(float(r.mean()))
    return new_row, new_col, rho


def factored_vhat(r: np.ndarray, c: np.ndarray, rho: float,
                  rows_idx: np.ndarray, cols_idx: np.ndarray) -> np.ndarray:
    """Rank-1 reconstruction vhat_ij = r_i c_j / rho at the given (i, j)."""
    if rho > 0.0:
        return r[rows_idx] * c[cols_idx] / rho
    return np.zeros(rows_idx.shape, dtype=np.float64)


# ---------------------------------------------------------------------------
# S2: element-wise accumulators (R1)
# ---------------------------------------------------------------------------
def accumulator_update(g: np.ndarray, mom: List[np.ndarray], rms: np.ndarray):
    """Three momenta and one RMS accumulator, each an EMA of g resp. g^2."""
    new_mom = [b * mom[k] + (1.0 - b) * g for k, b in enumerate(MOMENTUM_DECAYS)]
    new_rms = RMS_DECAY * rms + (1.0 - RMS_DECAY) * g * g
    return new_mom, new_rms


# ---------------------------------------------------------------------------
# S3: feature construction (R3) -- materialised, one row per element
# ---------------------------------------------------------------------------
def time_features(t: float) -> np.ndarray:
    """tau_s = tanh(t / x_s), the 11 step-count features."""
    return np.tanh(float(t) / np.asarray(TIME_SCALES, dtype=np.float64))


def features(p, g, mom, rms, row, col, rho, cols: int, t: float,
             elem_idx: np.ndarray | None = None) -> np.ndarray:
    """The [n x 39] feature matrix for the elements ``elem_idx`` (flat,
    row-major over the [R x C] view; all elements if None).  Every array
    argument is the *updated* state (accumulators refreshed first, R1).

    Column order (R3):
      0 p | 1 g | 2-4 m_k | 5 sqrt(v) | 6-8 m_k*rsqrt(v) | 9 g*rsqrt(v)
      10-12 g*rsqrt(vhat_k) | 13-15 sqrt(r_k[i]) | 16-18 sqrt(c_k[j])
      19+3a+b  m_a*rsqrt(vhat_b)  (a, b in 0..2)
      28-38 tanh(t / x_s)
    """
    if elem_idx is None:
        elem_idx = np.arange(p.size)
    i = elem_idx // cols
    j = elem_idx % cols
    P = p[elem_idx]
    G = g[elem_idx]
    M = [m[elem_idx] for m in mom]
    V = rms[elem_idx]
    inv_sqrt_v = 1.0 / np.sqrt(V + EPS)
    vhat = [factored_vhat(row[k], col[k], rho[k], i, j) for k in range(3)]
    inv_sqrt_vhat = [1.0 / np.sqrt(vh + EPS) for vh in vhat]

    F = np.empty((elem_idx.size, D_FEAT), dtype=np.float64)
    F[:, 0] = P
    F[:, 1] = G
    for k in range(3):
        F[:, 2 + k] = M[k]
    F[:, 5] = np.sqrt(V)
    for k in range(3):
        F[:, 6 + k] = M[k] * inv_sqrt_v
    F[:, 9] = G * inv_sqrt_v
    for k in range(3):
        F[:, 10 + k] = G * inv_sqrt_vhat[k]
    for k in range(3):
        F[:, 13 + k] = np.sqrt(row[k][i])
    for k in range(3):
        F[:, 16 + k] = np.sqrt(col[k][j])
    for a in range(3):
        for b in range(3):
            F[:, 19 + 3 * a + b] = M[a] * inv_sqrt_vhat[b]
    F[:, N_ELEM_FEATURES:] = time_features(t)[None, :]
    return F


# ---------------------------------------------------------------------------
# S4 + S5: per-feature mean square over the tensor and normalisation (R5)
# ---------------------------------------------------------------------------
def feature_square_sums(state, cols: int, t: float) -> np.ndarray:
    """S_d = sum over all elements of F[:, d]^2 for the 28 per-element
    features (the kernel-1 statistics of the fused design)."""
    n = state["param"].size
    S = np.zeros(N_ELEM_FEATURES, dtype=np.float64)
    for e0 in range(0, n, CHUNK_ELEMENTS):
        idx = np.arange(e0, min(n, e0 + CHUNK_ELEMENTS))
        F = _features_of(state, cols, t, idx)
        S += (F[:, :N_ELEM_FEATURES] ** 2).sum(axis=0)
    return S


def normalisation_scales(S: np.ndarray, n: int) -> np.ndarray:
    """1 / sqrt(mean square + eps) per per-element feature."""
    return 1.0 / np.sqrt(S / float(n) + EPS)


def normalise(F: np.ndarray, scales: np.ndarray) -> np.ndarray:
    Fn = F.copy()
    Fn[:, :N_ELEM_FEATURES] *= scales[None, :]
    return Fn


# ---------------------------------------------------------------------------
# S6 + S7: per-element MLP and parameter update (R6, R7)
# ---------------------------------------------------------------------------
def mlp(X: np.ndarray, w: MLPWeights) -> np.ndarray:
    """d_feat -> H -> H -> 2, ReLU on both hidden layers."""
    h1 = np.maximum(X @ w.W1 + w.b1, 0.0)
    h2 = np.maximum(h1 @ w.W2 + w.b2, 0.0)
    return h2 @ w.W3 + w.b3


def update_from_output(o: np.ndarray) -> np.ndarray:
    """update = direction * exp(magnitude * 1e-3) * 1e-3."""
    return o[:, 0] * np.exp(o[:, 1] * OUTPUT_SCALE) * OUTPUT_SCALE


def apply_update(p: np.ndarray, u: np.ndarray, lr: float, weight_decay: float = 0.0) -> np.ndarray:
    """R7 / R11: p - lr * (u + weight_decay * p)."""
    return p - lr * (u + weight_decay * p)


# ---------------------------------------------------------------------------
# One tensor, one step
# ---------------------------------------------------------------------------
def new_state(shape, param, grad, mom=None, rms=None, row=None, col=None,
              weight_set: int = 0) -> dict:
    """Oracle-side state of one tensor, widened to float64 (flat arrays)."""
    R, C = view_rows_cols(shape)
    n = R * C
    f64 = lambda a, m: (np.zeros(m) if a is None
                        else np.asarray(a, dtype=np.float64).ravel().copy())
    st = {
        "shape": (R, C),
        "param": f64(param, n),
        "grad": f64(grad, n),
        "mom": [f64(None if mom is None else mom[k], n) for k in range(3)],
        "rms": f64(rms, n),
        "row": [f64(None if row is None else row[k], R) for k in range(3)],
        "col": [f64(None if col is None else col[k], C) for k in range(3)],
        "weight_set": int(weight_set),
    }
    for a in [st["param"], st["grad"], st["rms"]] + st["mom"]:
        if a.size != n:
            raise ValueError("element count does not match the shape")
    return st


def _features_of(state, cols, t, idx):
    return features(state["param"], state["grad"], state["mom"], state["rms"],
                    state["row"], state["col"], state["rho"], cols, t, idx)


def refresh_accumulators(state: dict) -> None:
    """S1 + S2 in place: factored row/column EMAs, rho, momenta and RMS."""
    R, C = state["shape"]
    g = state["grad"]
    state["row"], state["col"], state["rho"] = factored_update(
        g.reshape(R, C), state["row"], state["col"])
    state["mom"], state["rms"] = accumulator_update(g, state["mom"], state["rms"])


def step_tensor(state: dict, t: float, lr: float, w: MLPWeights,
                sample_idx: np.ndarray | None = None, weight_decay: float = 0.0) -> dict:
    """One learned-optimizer step on one tensor, in place.

    Returns a dict of diagnostics: S (the 28 square sums), scales, and -- when
    ``sample_idx`` is given -- the update computed only at those elements
    (the parameter array is then left unchanged, for sampled checks of large
    tensors)."""
    R, C = state["shape"]
    n = R * C
    refresh_accumulators(state)
    S = feature_square_sums(state, C, t)
    scales = normalisation_scales(S, n)
    out = {"S": S, "scales": scales, "rho": list(state["rho"])}
    if sample_idx is not None:
        sample_idx = np.asarray(sample_idx, dtype=np.int64)
        F = _features_of(state, C, t, sample_idx)
        o = mlp(normalise(F, scales), w)
        u = update_from_output(o)
        out["sample_idx"] = sample_idx
        out["sample_param"] = apply_update(state["param"][sample_idx], u, lr, weight_decay)
        out["sample_update"] = u
        return out
    new_p = np.empty_like(state["param"])
    for e0 in range(0, n, CHUNK_ELEMENTS):
        idx = np.arange(e0, min(n, e0 + CHUNK_ELEMENTS))
        F = _features_of(state, C, t, idx)
        o = mlp(normalise(F, scales), w)
        new_p[idx] = apply_update(state["param"][idx], update_from_output(o), lr, weight_decay)
    state["param"] = new_p
    return out


def step(states: List[dict], t: float, lr: float, weight_sets: Sequence[np.ndarray],
         hidden: int, weight_decay: float = 0.0) -> List[dict]:
    """One step over a parameter list; each tensor uses its own weight set."""
    ws = [unpack_weights(wf, hidden) for wf in weight_sets]
    return [step_tensor(st, t, lr, ws[st["weight_set"]], weight_decay=weight_decay) for st in states]


def materialised_features(state: dict, t: float) -> np.ndarray:
    """Full [N x 39] feature matrix of the current (already refreshed) state;
    for inspection in tests."""
    R, C = state["shape"]
    return _features_of(state, C, t, np.arange(R * C))


__all__ = [
    "MOMENTUM_DECAYS", "RMS_DECAY", "FACTORED_DECAYS", "EPS", "TIME_SCALES",
    "N_ELEM_FEATURES", "N_TIME_FEATURES", "D_FEAT", "OUTPUT_SCALE",
    "view_rows_cols", "weight_set_size", "MLPWeights", "unpack_weights",
    "factored_update", "factored_vhat", "accumulator_update", "time_features",
    "features", "feature_square_sums", "normalisation_scales", "normalise",
    "mlp", "update_from_output", "apply_update", "new_state", "refresh_accumulators",
    "step_tensor", "step", "materialised_features",
]
