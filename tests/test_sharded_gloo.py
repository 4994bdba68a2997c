"""The row-sharded step's exchange, with two gloo ranks on CPU.

Each rank owns whole rows of every tensor; between the local computations
the ranks add up exactly the quantities the sharded C-ABI entry points put
in their exchange buffers: the column sums of g^2 and the sums of the new
row accumulators (buffer 1), then the 28 feature square sums (buffer 2).
The local parts use the oracle's primitives; the test checks that the
ranks' rows together equal the oracle's unsharded step."""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

SHAPES = [(12, 7), (1, 10), (5, 3), (9, 16)]
SPLITS = [6, 1, 2, 4]          # rows owned by rank 0; rank 1 owns the rest (maybe none)
T_STEP, LR, HIDDEN = 3, 0.8, 8


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(seed):
    rng = np.random.default_rng(seed)
    out = []
    for R, C in SHAPES:
        n = R * C
        out.append({
            "p": rng.normal(size=n) * 0.05, "g": rng.normal(size=n) * 1e-3,
            "m": [rng.normal(size=n) * 1e-4 for _ in range(3)], "v": rng.random(n) * 1e-6,
            "r": [rng.random(R) * 1e-6 for _ in range(3)], "c": [rng.random(C) * 1e-6 for _ in range(3)],
        })
    w = rng.normal(size=39 * HIDDEN + 4 * HIDDEN + HIDDEN * HIDDEN + 2) * 0.3
    return out, w


def _sum(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    dist.all_reduce(t)
    return t.numpy()


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        tensors, wflat = _inputs(7)
        w = O.unpack_weights(wflat, HIDDEN)
        results = []
        for (R, C), split, st in zip(SHAPES, SPLITS, tensors):
            r0, r1 = (0, split) if rank == 0 else (split, R)
            rows = r1 - r0
            sl = slice(r0 * C, r1 * C)
            p, g = st["p"][sl], st["g"][sl]
            # local row moments; this rank's column sums and row-accumulator sums
            sq = (g * g).reshape(rows, C)
            row_mean = sq.mean(axis=1) if rows else np.zeros(0)
            new_row = [b * st["r"][k][r0:r1] + (1 - b) * row_mean for k, b in enumerate(O.FACTORED_DECAYS)]
            x1 = np.concatenate([sq.sum(axis=0), [float(r.sum()) for r in new_row]])
            x1 = _sum(x1)                                              # exchange 1
            col_mean = x1[:C] / R
            new_col = [b * st["c"][k] + (1 - b) * col_mean for k, b in enumerate(O.FACTORED_DECAYS)]
            rho = [float(x1[C + k]) / R for k in range(3)]
            mom, rms = O.accumulator_update(g, [m[sl] for m in st["m"]], st["v"][sl])
            F = O.features(p, g, mom, rms, new_row, new_col, rho, C, T_STEP)
            S = _sum((F[:, :O.N_ELEM_FEATURES] ** 2).sum(axis=0))    # exchange 2
            o = O.mlp(O.normalise(F, O.normalisation_scales(S, R * C)), w)
            results.append((p - LR * O.update_from_output(o), new_col, S))
        out.put((rank, results))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_sharded_step_equals_unsharded_oracle():
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    tensors, wflat = _inputs(7)
    w = O.unpack_weights(wflat, HIDDEN)
    for ti, ((R, C), st) in enumerate(zip(SHAPES, tensors)):
        ref = O.new_state((R, C), st["p"], st["g"], mom=st["m"], rms=st["v"], row=st["r"], col=st["c"])
        out = O.step_tensor(ref, T_STEP, LR, w)
        got = np.concatenate([res[0][ti][0], res[1][ti][0]])
        np.testing.assert_allclose(got, ref["param"], rtol=1e-12, atol=1e-18)
        for rank in (0, 1):   # replicated column accumulators and sums agree on every rank
            for k in range(3):
                np.testing.assert_allclose(res[rank][ti][1][k], ref["col"][k], rtol=1e-13)
            np.testing.assert_allclose(res[rank][ti][2], out["S"], rtol=1e-12)
