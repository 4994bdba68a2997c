"""Writes tc_emulation_bound.json: the parity bounds of the tensor-core MLP
path, derived from the oracle and its FP16 emulation alone (no GPU result).

For each case (seeded inputs with the shapes and value recipes of the
ViT-B/16, GPT-2-small and VeLO-style workloads, whole tensors):
  * emulated: the update error of an exact FP16-operand MLP against the
    oracle, per tensor, max |dp_emu - dp_ref| / max(|dp_ref|, RMS dp_ref);
  * perturbed: the same metric between two emulations whose operands differ
    by what an fp32 kernel may legitimately differ by (normalisation scales
    within half the 2e-5 bound on the feature square sums, features within
    a few fp32 units): how far a correct kernel may land from the emulation;
  * the same two, as the root mean square over the tensor's elements of the
    error over RMS dp_ref (the largest errors sit on a few outlier elements,
    where one FP16 rounding step is already about 1e-2 of the RMS update;
    the RMS error shows a systematic mistake far below that).
gate_dp / gate_emulation = 2 x the largest emulated / perturbed error, and
gate_dp_rms / gate_emulation_rms likewise, each rounded up to one
significant digit.  Run: python tests/golden/make_tc_emulation_bound.py
(about twenty minutes on one core)."""

import json
import math
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "..", ".."))
import oracle as O          # noqa: E402
import synth                # noqa: E402
from tests import tc_emulation as E   # noqa: E402

D_SCALE = 1e-5              # half the square-sum bound: scale = S^-1/2
D_FEAT = 2.0 ** -21         # a few fp32 units (rsqrt.approx, products)


def dp_err(p_old, ref_new, got_new):
    dref = p_old - ref_new
    rms = float(np.sqrt(np.mean(dref * dref)))
    return float(np.max(np.abs((p_old - got_new) - dref) / np.maximum(np.abs(dref), max(rms, 1e-300))))


def dp_rms_err(p_old, ref_new, got_new):
    dref = p_old - ref_new
    rms = max(float(np.sqrt(np.mean(dref * dref))), 1e-300)
    e = (p_old - got_new) - dref
    return float(np.sqrt(np.mean(e * e))) / rms


def run_case(name, shapes, recipe, t, seed, wseed, hidden=32):
    wl = synth.Workload(name, tuple(shapes), 1, t, recipe)
    sts = synth.make_list(wl, "cpu", seed=seed)
    w = O.unpack_weights(synth.make_weight_sets(1, hidden, seed=wseed)[0], hidden)
    emu_max = pert_max = emu_rms = pert_rms = 0.0
    worst = ""
    for st in sts:
        cp = lambda a: a.numpy().astype(np.float64)
        mk = lambda: O.new_state((st["rows"], st["cols"]), cp(st["param"]), cp(st["grad"]),
                                 mom=[cp(m) for m in st["mom"]], rms=cp(st["rms"]),
                                 row=[cp(r) for r in st["row"]], col=[cp(c) for c in st["col"]])
        a, b, c = mk(), mk(), mk()
        p_old = a["param"].copy()
        O.step_tensor(a, t, 1.0, w)
        E.step_tensor(b, t, 1.0, w)
        E.step_tensor(c, t, 1.0, w, perturb=(np.random.default_rng(seed + 17), D_SCALE, D_FEAT))
        e = dp_err(p_old, a["param"], b["param"])
        if e > emu_max:
            emu_max, worst = e, st["name"]
        pert_max = max(pert_max, dp_err(p_old, b["param"], c["param"]))
        emu_rms = max(emu_rms, dp_rms_err(p_old, a["param"], b["param"]))
        pert_rms = max(pert_rms, dp_rms_err(p_old, b["param"], c["param"]))
    return {"case": name, "t": t, "seed": seed, "weight_seed": wseed, "hidden": hidden,
            "emulated": emu_max, "worst_tensor": worst, "perturbed": pert_max,
            "emulated_rms": emu_rms, "perturbed_rms": pert_rms}


def main():
    vit = synth.vit_b16_shapes()
    vit_sample = vit[:14] + vit[-4:]          # patch, block 0, final LayerNorm, head
    g2 = synth.gpt2_small_shapes()
    cases = []
    for s in range(4):
        cases.append(run_case("vit_b16 sample", vit_sample, "vit", 1, s, 1234 + s))
    cases.append(run_case("vit_b16 sample", vit_sample, "vit", 10, 0, 1234))
    cases.append(run_case("gpt2_small sample", [g2[1]] + g2[2:14], "gpt2", 9991, 0, 1234))
    cases.append(run_case("velo_h4 sample", vit_sample, "vit", 1, 0, 1234, hidden=4))
    mx = lambda key: max(c[key] for c in cases)

    def up(x):   # 2 x, rounded up to one significant digit
        y = 2.0 * x
        e = math.floor(math.log10(y))
        return math.ceil(y / 10.0 ** e) * 10.0 ** e

    out = {"cases": cases, "max_emulated": mx("emulated"), "max_perturbed": mx("perturbed"),
           "max_emulated_rms": mx("emulated_rms"), "max_perturbed_rms": mx("perturbed_rms"),
           "gate_dp": up(mx("emulated")), "gate_emulation": up(mx("perturbed")),
           "gate_dp_rms": up(mx("emulated_rms")), "gate_emulation_rms": up(mx("perturbed_rms")),
           "d_scale": D_SCALE, "d_feat": D_FEAT}
    with open(os.path.join(os.path.dirname(__file__), "tc_emulation_bound.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({k: v for k, v in out.items() if k != "cases"}))


if __name__ == "__main__":
    main()
