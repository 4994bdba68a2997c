"""Seeded synthetic inputs: parameter-list shapes, value recipes, MLP weights.

This module holds no arithmetic of the optimizer step.  It only draws random
numbers and lists shapes; both the CUDA path (via the tests and the bench) and
the CPU oracle receive exactly the arrays produced here.

Shapes follow the workloads of "PyLO: Towards Accessible Learned Optimizers in
PyTorch" (section "ステップ時間の削減": ViT-B/16 and GPT-2 step times;
section "JAX リファレンス実装との比較": scaling to ~1B parameters; the VeLO
variant with one weight set per tensor).  No dataset or trained weight is
used: parameters, gradients and MLP weights are drawn from seeded
distributions with the recipes below.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Sequence, Tuple

import numpy as np
import torch

Shape = Tuple[int, ...]

# --------------------------------------------------------------------------
# Shape lists
# --------------------------------------------------------------------------


def _block(d: int, ffn: int, qkv: int) -> List[Tuple[str, Shape]]:
    """One pre-LN transformer block: 4 matrices, 4 biases, 2 LayerNorm pairs."""
    return [
        ("qkv.w", (d, qkv)), ("qkv.b", (qkv,)),
        ("proj.w", (d, d)), ("proj.b", (d,)),
        ("fc1.w", (d, ffn)), ("fc1.b", (ffn,)),
        ("fc2.w", (ffn, d)), ("fc2.b", (d,)),
        ("ln1.w", (d,)), ("ln1.b", (d,)),
        ("ln2.w", (d,)), ("ln2.b", (d,)),
    ]


def vit_b16_shapes() -> List[Tuple[str, Shape]]:
    """ViT-B/16: patch embedding (16*16*3 = 768 inputs), 12 blocks d=768
    ffn=3072, final LayerNorm, 1000-way head.  150 tensors, 86,415,592
    elements."""
    out = [("patch.w", (768, 768)), ("patch.b", (768,))]
    for L in range(12):
        out += [("blk%d.%s" % (L, n), s) for n, s in _block(768, 3072, 2304)]
    out += [("ln_f.w", (768,)), ("ln_f.b", (768,)),
            ("head.w", (768, 1000)), ("head.b", (1000,))]
    return out


def gpt2_small_shapes() -> List[Tuple[str, Shape]]:
    """GPT-2 small: token embedding 50257x768, position embedding 1024x768,
    12 blocks d=768 ffn=3072, final LayerNorm.  148 tensors, 124,439,808
    elements."""
    out = [("wte", (50257, 768)), ("wpe", (1024, 768))]
    for L in range(12):
        out += [("h%d.%s" % (L, n), s) for n, s in _block(768, 3072, 2304)]
    out += [("ln_f.w", (768,)), ("ln_f.b", (768,))]
    return out


def decoder_1p3b_shapes() -> List[Tuple[str, Shape]]:
    """1.3B decoder: vocab 50304 x 2048 embedding, 24 blocks d=2048 ffn=8192,
    final LayerNorm.  291 tensors."""
    out = [("embed", (50304, 2048))]
    for L in range(24):
        out += [("l%d.%s" % (L, n), s) for n, s in _block(2048, 8192, 6144)]
    out += [("ln_f.w", (2048,)), ("ln_f.b", (2048,))]
    return out


def vit_block_shapes() -> List[Tuple[str, Shape]]:
    """Patch embedding plus the first ViT-B/16 block (14 tensors, 7.68M
    elements): a small case for profiler captures (state > L2)."""
    return vit_b16_shapes()[:14]


def velo_style_shapes() -> List[Tuple[str, Shape]]:
    """The ViT-B/16 list plus one 50,000 x 1,000 (50M-element) tensor."""
    return vit_b16_shapes() + [("big", (50000, 1000))]


def numel(shape: Shape) -> int:
    return int(np.prod(shape)) if len(shape) else 1


# --------------------------------------------------------------------------
# Value recipes
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: Tuple[Tuple[str, Shape], ...]
    steps: int
    first_step: int          # t of the first step (1-based)
    recipe: str              # "single", "vit", "gpt2"
    per_tensor_weights: bool = False
    hidden: int = 32


def workloads() -> Dict[str, Workload]:
    return {
        "single_256x256": Workload("single_256x256", (("w", (256, 256)),), 3, 1, "single"),
        "vit_b16": Workload("vit_b16", tuple(vit_b16_shapes()), 10, 1, "vit"),
        "vit_block": Workload("vit_block", tuple(vit_block_shapes()), 10, 1, "vit"),
        "gpt2_small": Workload("gpt2_small", tuple(gpt2_small_shapes()), 10, 9991, "gpt2"),
        "decoder_1p3b": Workload("decoder_1p3b", tuple(decoder_1p3b_shapes()), 5, 1, "vit"),
        "velo_h32": Workload("velo_h32", tuple(velo_style_shapes()), 10, 1, "vit", True, 32),
        "velo_h4": Workload("velo_h4", tuple(velo_style_shapes()), 10, 1, "vit", True, 4),
    }


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


# Decays used only to give the warm-start accumulators of the GPT-2 recipe
# the stationary spread of an EMA of white noise (input synthesis only).
_WARM_DECAYS = (0.1, 0.5, 0.9)
_WARM_SIGMA2 = 3e-6


def make_param(name: str, shape: Shape, recipe: str, seed: int, device) -> torch.Tensor:
    """Initial parameter values: matrices ~ N(0, 0.02^2); LayerNorm weights 1;
    biases 0 (for the ViT/GPT recipes).  The single-tensor recipe draws
    N(0, 0.02^2)."""
    gen = _gen(seed, device)
    if recipe == "single" or len(shape) >= 2:
        return _normal(shape, 0.02, gen, device)
    if name.endswith("ln1.w") or name.endswith("ln2.w") or name.endswith("ln_f.w"):
        return torch.ones(shape, device=device, dtype=torch.float32)
    return torch.zeros(shape, device=device, dtype=torch.float32)


def make_grad(shape: Shape, recipe: str, seed: int, device) -> torch.Tensor:
    """Gradient draw.  single: N(0, 0.01^2).  vit: s * N(0,1) with one scale s
    per tensor, log-uniform in [1e-5, 1e-2].  gpt2: 1e-3 * Student-t(nu=3)."""
    gen = _gen(seed, device)
    if recipe == "single":
        return _normal(shape, 0.01, gen, device)
    if recipe == "vit":
        u = torch.rand((), generator=gen, device=device, dtype=torch.float64).item()
        s = 10.0 ** (-5.0 + 3.0 * u)
        return _normal(shape, s, gen, device)
    if recipe == "gpt2":
        z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        # chi-square with 3 degrees of freedom from three squared normals
        chi = sum(torch.randn(shape, generator=gen, device=device, dtype=torch.float32) ** 2
                  for _ in range(3))
        return 1e-3 * z / torch.sqrt(chi / 3.0)
    raise ValueError(recipe)


def make_accumulators(shape: Shape, rows: int, cols: int, recipe: str, seed: int,
                      device) -> dict:
    """Zero accumulators, except the GPT-2 recipe (step ~10,000) which starts
    from warmed-up values: m_k ~ N(0, s2 (1-b)/(1+b)), v = r = c = s2."""
    n = numel(shape)
    z = lambda m: torch.zeros(m, device=device, dtype=torch.float32)
    if recipe != "gpt2":
        return {"mom": [z(n) for _ in range(3)], "rms": z(n),
                "row": [z(rows) for _ in range(3)], "col": [z(cols) for _ in range(3)]}
    gen = _gen(seed, device)
    mom = [_normal((n,), math.sqrt(_WARM_SIGMA2 * (1 - b) / (1 + b)), gen, device)
           for b in _WARM_DECAYS]
    full = lambda m: torch.full((m,), _WARM_SIGMA2, device=device, dtype=torch.float32)
    return {"mom": mom, "rms": full(n), "row": [full(rows) for _ in range(3)],
            "col": [full(cols) for _ in range(3)]}


def rows_cols(shape: Shape) -> Tuple[int, int]:
    """[R x C] view used by the step: rank 0 -> 1x1, rank 1 -> 1xn,
    rank >= 2 -> prod(leading) x last."""
    if len(shape) == 0:
        return 1, 1
    if len(shape) == 1:
        return 1, int(shape[0])
    return int(np.prod(shape[:-1])), int(shape[-1])


def weight_set_floats(hidden: int, d_feat: int = 39) -> int:
    return d_feat * hidden + hidden + hidden * hidden + hidden + 2 * hidden + 2


def make_weight_sets(n_sets: int, hidden: int, seed: int = 1234,
                     d_feat: int = 39) -> np.ndarray:
    """Xavier-normal MLP weights (std = sqrt(2/(fan_in+fan_out))), zero biases,
    one independent draw per set (seed + set index).  Layout per set:
    W1[d_feat][H], b1[H], W2[H][H], b2[H], W3[H][2], b3[2]."""
    out = np.zeros((n_sets, weight_set_floats(hidden, d_feat)), dtype=np.float32)
    for s in range(n_sets):
        gen = _gen(seed + s, "cpu")
        parts = []
        for fi, fo in ((d_feat, hidden), (hidden, hidden), (hidden, 2)):
            std = math.sqrt(2.0 / (fi + fo))
            parts.append((torch.randn((fi, fo), generator=gen) * std).numpy().ravel())
            parts.append(np.zeros(fo, dtype=np.float32))
        out[s] = np.concatenate(parts).astype(np.float32)
    return out


def make_list(wl: Workload, device, seed: int = 0, shapes=None, indices=None) -> List[dict]:
    """Initial state for every tensor of a workload (torch tensors on
    ``device``): param, grad (step ``wl.first_step``), accumulators.
    ``indices``: only these tensors of the list, drawn exactly as in the
    whole list."""
    shapes = wl.shapes if shapes is None else shapes
    out = []
    for ti, (name, shape) in enumerate(shapes):
        if indices is not None and ti not in indices:
            continue
        R, C = rows_cols(shape)
        s = seed + 7919 * ti
        st = {"name": name, "shape": tuple(shape), "rows": R, "cols": C,
              "param": make_param(name, shape, wl.recipe, s, device).reshape(-1),
              "grad": make_grad(shape, wl.recipe, s + 1, device).reshape(-1),
              "weight_set": ti if wl.per_tensor_weights else 0}
        st.update(make_accumulators(shape, R, C, wl.recipe, s + 2, device))
        out.append(st)
    return out


def refresh_grads(states: List[dict], wl: Workload, step_index: int, seed: int = 0) -> None:
    """Draw a new gradient for every tensor (step_index >= 1), in place."""
    for ti, st in enumerate(states):
        s = seed + 7919 * ti + 104729 * step_index + 1
        g = make_grad(st["shape"], wl.recipe, s, st["grad"].device).reshape(-1)
        st["grad"].copy_(g)


def total_elements(shapes: Sequence[Tuple[str, Shape]]) -> int:
    return sum(numel(s) for _, s in shapes)
