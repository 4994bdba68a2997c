"""Failure detection on the GPU without a fault: the bounded wait every
kernel uses is made to run out on a barrier that never completes, and the
host reads the timeout status; the context stays usable afterwards."""

import time

import pytest

import synth
from tests.gpu_helpers import TOL_FP32, compare_step, make_states, need_gpu

pytestmark = pytest.mark.gpu

LOPT_E_TIMEOUT = -7


def test_bounded_wait_runs_out_and_reports_timeout():
    torch = need_gpu()
    from learned_optimizer_step_gb300 import lopt as L
    lib = L.load_library()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.lopt_selftest_wait(5_000_000)   # 5 ms
    dt = time.perf_counter() - t0
    assert rc == LOPT_E_TIMEOUT, lib.lopt_strerror(rc)
    assert 0.005 <= dt < 5.0


def test_context_usable_after_a_timeout():
    need_gpu()
    from learned_optimizer_step_gb300 import LearnedOptimizer, lopt as L
    assert L.load_library().lopt_selftest_wait(1_000_000) == LOPT_E_TIMEOUT
    w = synth.make_weight_sets(1, 32, seed=1234)
    eng = LearnedOptimizer(w, 32, "fp32")
    states = make_states([("w", (64, 96)), ("b", (96,))], recipe="vit", seed=11)
    compare_step(eng, states, w, 32, 1, 1.0, TOL_FP32)
    eng.check()
