"""Writes tc_emulation_bound.json: the parity bounds of the tensor-core MLP
path, derived from the oracle and its FP16 emulation alone (no GPU result).

For each case (seeded inputs with the shapes and value recipes of the
ViT-B/16, GPT-2-small and VeLO-style workloads):
  * emulated: the update error of an exact FP16-operand MLP against the
    oracle, per tensor, max |dp_emu - dp_ref| / max(|dp_ref|, RMS dp_ref);
  * perturbed: the same metric between two emulations whose operands differ
    by what an fp32 kernel may legitimately differ by (normalisation scales
    within half the 2e-5 bound on the feature square sums, features within
    a few fp32 units): how far a correct kernel may land from the emulation;
  * the same two, as the root mean square of the error over RMS dp_ref:
    over the whole tensor, and over each of SAMPLE_DRAWS random samples of
    SAMPLE_SIZE elements plus the two ends, the samples the full-size GPU
    tests compare (the largest errors sit on a few outlier elements, where
    one FP16 rounding step is already about 1e-2 of the RMS update; the RMS
    error shows a systematic mistake far below that, and over a sample of a
    few hundred elements it varies more than over a whole tensor).
The ViT-B/16 and GPT-2 cases take whole tensors of a slice of the list; the
VeLO-style cases (hidden widths 4 and 32, one weight set per tensor) take
the largest tensor, at sampled elements only, and one tensor of every other
shape, whole.
gate_dp / gate_emulation = 2 x the largest emulated / perturbed error, and
gate_dp_rms / gate_emulation_rms likewise over the whole-tensor and sampled
RMS errors, each rounded up to one significant digit.
Run: python tests/golden/make_tc_emulation_bound.py (the cases run in
parallel, one process each; about half an hour on eight cores)."""

import json
import math
import multiprocessing as mp
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


SAMPLE_SIZE = 256           # elements per sample, as the full-size GPU tests draw
SAMPLE_DRAWS = 8            # samples per tensor
WHOLE_MAX = 4_000_000       # larger tensors: sampled elements only


def sample_draws(n, seed):
    """SAMPLE_DRAWS random samples of a tensor of n elements (each with the
    first and last element); one sample of everything for small tensors."""
    if n <= 4 * SAMPLE_SIZE:
        return [np.arange(n)]
    rng = np.random.default_rng(seed + n)
    return [np.unique(np.concatenate([rng.choice(n, size=SAMPLE_SIZE, replace=False), [0, n - 1]]))
            for _ in range(SAMPLE_DRAWS)]


def subset(shapes):
    """The largest tensor and the first tensor of every other (rows, cols,
    kind) combination, as the sampled GPU tests of the large lists pick."""
    rc = [synth.rows_cols(s) for _, s in shapes]
    big = max(range(len(shapes)), key=lambda i: rc[i][0] * rc[i][1])
    seen, out = set(), [big]
    for i, (name, _) in enumerate(shapes):
        key = (rc[i][0], rc[i][1], name.split(".")[-1])
        if key not in seen:
            seen.add(key)
            if i != big:
                out.append(i)
    return sorted(out)


def run_case(args):
    name, shapes, recipe, t, seed, wseed, hidden, per_tensor, indices = args
    wl = synth.Workload(name, tuple(shapes), 1, t, recipe, per_tensor, hidden)
    sts = synth.make_list(wl, "cpu", seed=seed, indices=indices)
    wsets = synth.make_weight_sets(len(shapes) if per_tensor else 1, hidden, seed=wseed)
    emu_max = pert_max = emu_rms = pert_rms = emu_rms_s = pert_rms_s = 0.0
    worst = ""
    for st in sts:
        w = O.unpack_weights(wsets[st["weight_set"]], hidden)
        n = st["rows"] * st["cols"]
        cp = lambda a: a.numpy().astype(np.float64)
        mk = lambda: O.new_state((st["rows"], st["cols"]), cp(st["param"]), cp(st["grad"]),
                                 mom=[cp(m) for m in st["mom"]], rms=cp(st["rms"]),
                                 row=[cp(r) for r in st["row"]], col=[cp(c) for c in st["col"]])
        a, b, c = mk(), mk(), mk()
        draws = sample_draws(n, seed)
        if n > WHOLE_MAX:      # evaluate the union of the samples only
            sidx = np.unique(np.concatenate(draws))
            draws = [np.searchsorted(sidx, d) for d in draws]
        else:
            sidx = None
        p_old = a["param"].copy() if sidx is None else a["param"][sidx].copy()
        ra = O.step_tensor(a, t, 1.0, w, sample_idx=sidx)
        rb = E.step_tensor(b, t, 1.0, w, sample_idx=sidx, S=ra["S"])
        rc = E.step_tensor(c, t, 1.0, w, sample_idx=sidx, S=ra["S"],
                           perturb=(np.random.default_rng(seed + 17), D_SCALE, D_FEAT))
        ref = a["param"] if sidx is None else ra["sample_param"]
        emu = b["param"] if sidx is None else rb["sample_param"]
        per = c["param"] if sidx is None else rc["sample_param"]
        e = dp_err(p_old, ref, emu)
        if e > emu_max:
            emu_max, worst = e, st["name"]
        pert_max = max(pert_max, dp_err(p_old, emu, per))
        if sidx is None:
            emu_rms = max(emu_rms, dp_rms_err(p_old, ref, emu))
            pert_rms = max(pert_rms, dp_rms_err(p_old, emu, per))
        for d in draws:
            emu_rms_s = max(emu_rms_s, dp_rms_err(p_old[d], ref[d], emu[d]))
            pert_rms_s = max(pert_rms_s, dp_rms_err(p_old[d], emu[d], per[d]))
    return {"case": name, "t": t, "seed": seed, "weight_seed": wseed, "hidden": hidden,
            "tensors": len(sts), "emulated": emu_max, "worst_tensor": worst, "perturbed": pert_max,
            "emulated_rms": emu_rms, "perturbed_rms": pert_rms,
            "emulated_rms_sampled": emu_rms_s, "perturbed_rms_sampled": pert_rms_s}


def main():
    vit = synth.vit_b16_shapes()
    vit_sample = vit[:14] + vit[-4:]          # patch, block 0, final LayerNorm, head
    g2 = synth.gpt2_small_shapes()
    velo = synth.velo_style_shapes()
    jobs = [("vit_b16 sample", vit_sample, "vit", 1, s, 1234 + s, 32, False, None) for s in range(4)]
    jobs.append(("vit_b16 sample", vit_sample, "vit", 10, 0, 1234, 32, False, None))
    jobs.append(("gpt2_small sample", [g2[1]] + g2[2:14], "gpt2", 9991, 0, 1234, 32, False, None))
    jobs.append(("velo_h4 sample", vit_sample, "vit", 1, 0, 1234, 4, False, None))
    for h in (4, 32):
        jobs.append(("velo_style h%d subset" % h, velo, "vit", 1, 0, 1234, h, True, subset(velo)))
    with mp.get_context("spawn").Pool(min(len(jobs), os.cpu_count() or 1)) as pool:
        cases = pool.map(run_case, jobs, chunksize=1)
    mx = lambda *keys: max(c[k] for c in cases for k in keys)

    def up(x):   # 2 x, rounded up to one significant digit
        y = 2.0 * x
        e = math.floor(math.log10(y))
        return math.ceil(y / 10.0 ** e) * 10.0 ** e

    out = {"cases": cases, "max_emulated": mx("emulated"), "max_perturbed": mx("perturbed"),
           "max_emulated_rms": mx("emulated_rms", "emulated_rms_sampled"),
           "max_perturbed_rms": mx("perturbed_rms", "perturbed_rms_sampled"),
           "sample_size": SAMPLE_SIZE, "sample_draws": SAMPLE_DRAWS,
           "d_scale": D_SCALE, "d_feat": D_FEAT}
    out.update({"gate_dp": up(out["max_emulated"]), "gate_emulation": up(out["max_perturbed"]),
                "gate_dp_rms": up(out["max_emulated_rms"]), "gate_emulation_rms": up(out["max_perturbed_rms"])})
    with open(os.path.join(os.path.dirname(__file__), "tc_emulation_bound.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({k: v for k, v in out.items() if k != "cases"}))


if __name__ == "__main__":
    main()
