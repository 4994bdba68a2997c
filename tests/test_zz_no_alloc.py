"""GPU test of lopt_rowcol_static(), the entry point that allocates no device
memory.

Some callers may not call cudaMalloc: code running inside a runtime that owns
every device allocation, code held to a fixed device-memory budget, or a path
that cannot afford cudaMalloc's device-wide synchronisation.  For them the
library offers the row/column second-moment update with its scratch taken
from a fixed array inside the library.  This test calls it through the C ABI
and checks that two calls in a row give bit for bit the accumulators of the
regular lopt_step() path (same kernel, same strips, and for these 16-byte
aligned torch tensors the same 128-bit route), and 1/rho within the
accumulator tolerance of its definition.  The file is named so that pytest
collects it last.
"""

import numpy as np
import pytest

import synth
from tests.gpu_helpers import TOL_ACC, cpu, make_states, need_gpu, rel_err

pytestmark = pytest.mark.gpu


def test_static_scratch_rowcol_matches_step_on_two_calls():
    torch = need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer, lopt
    shapes = [("w", (300, 700)), ("b", (1000,)), ("tall", (5000, 12))]
    wl = synth.Workload("noalloc", tuple(shapes), 2, 1, "vit")
    states = synth.make_list(wl, "cuda", seed=21)
    eng = LearnedOptimizer(synth.make_weight_sets(1, 32), 32, "fp32")
    # accumulators driven only by the no-allocation entry point
    mirror = [{"row": [r.clone() for r in s["row"]], "col": [c.clone() for c in s["col"]]}
              for s in states]
    inv_rho = [torch.zeros(3, device="cuda") for _ in states]
    for t in (1, 2):
        if t > 1:
            synth.refresh_grads(states, wl, t)
        eng.step(states, t, 1.0)
        for s, m, ir in zip(states, mirror, inv_rho):
            lopt.rowcol_static(s["grad"], m["row"], m["col"], s["rows"], s["cols"], ir)
        torch.cuda.synchronize()
        for s, m, ir in zip(states, mirror, inv_rho):
            for k in range(3):
                assert torch.equal(m["row"][k], s["row"][k]), (t, s["name"], "row", k)
                assert torch.equal(m["col"][k], s["col"][k]), (t, s["name"], "col", k)
            expect = 1.0 / np.array([cpu(r).mean() for r in s["row"]])
            assert rel_err(cpu(ir), expect) <= TOL_ACC, (t, s["name"])


def test_static_scratch_rejects_oversized_tensor_untouched():
    torch = need_gpu()
    from learned_optimizer_step_gb300 import lopt
    C = 1 << 20                      # 4 MiB of column partials > the fixed scratch
    g = torch.randn(C, device="cuda")
    row = [torch.zeros(1, device="cuda") for _ in range(3)]
    col = [torch.zeros(C, device="cuda") for _ in range(3)]
    ir = torch.zeros(3, device="cuda")
    with pytest.raises(lopt.LoptError) as ei:
        lopt.rowcol_static(g, row, col, 1, C, ir)
    assert ei.value.code == -9
    torch.cuda.synchronize()
    assert all(float(c.abs().max()) == 0.0 for c in col)
