"""CPU checks of the ragged schedule that lopt_step launches (host logic,
through lopt_schedule_info; no device call).

The step covers every element of every tensor: K0 by row strips of each
tensor, K1 by chunks of 16,384 elements, K2 by chunks of 4,096 elements
(sizes as the header documents them, typed in here).  Each unit must appear
exactly once; K0 and K1 take the largest work first, K2 runs in tensor
order; the single-sweep groups cut the list into consecutive tensors within
the byte budget and permute units only inside a group.

Method: "PyLO: Towards Accessible Learned Optimizers in PyTorch", section
"融合カーネル戦略" (per-tensor statistics before the apply pass) and
"メモリ階層の活用" (tensor state kept close between the passes).
"""

import numpy as np
import pytest

import synth
from learned_optimizer_step_gb300 import build as B
from learned_optimizer_step_gb300 import lopt as L

K1_CHUNK, K2_CHUNK, MAX_STRIP_ROWS = 16384, 4096, 2048


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    L.load_library()


def cdiv(a, b):
    return -(-a // b)


def random_shapes(rng, n):
    out = []
    for _ in range(n):
        kind = rng.integers(0, 6)
        if kind == 0:
            out.append((1, int(rng.integers(1, 200_000))))
        elif kind == 1:
            out.append((int(rng.integers(1, 60_000)), int(rng.integers(1, 1_200))))
        elif kind == 2:
            out.append((int(rng.integers(1, 8)), int(rng.integers(1, 70_000))))
        else:
            out.append((int(rng.integers(1, 4_096)), int(rng.integers(1, 4_096))))
    return out


def expected_units(shapes, strip_rows):
    k0 = {(i, s) for i, (r, _) in enumerate(shapes) for s in range(cdiv(r, int(strip_rows[i])))}
    k1 = {(i, s) for i, (r, c) in enumerate(shapes) for s in range(cdiv(r * c, K1_CHUNK))}
    k2 = {(i, s) for i, (r, c) in enumerate(shapes) for s in range(cdiv(r * c, K2_CHUNK))}
    return k0, k1, k2


def check_cover(units, expect):
    got = [tuple(u) for u in units.tolist()]
    assert len(got) == len(set(got)), "a unit appears twice"
    assert set(got) == expect


def strip_elems(shapes, strip_rows, units):
    return [int(strip_rows[t]) * shapes[t][1] for t, _ in units.tolist()]


def sizes(shapes, units):
    return [shapes[t][0] * shapes[t][1] for t, _ in units.tolist()]


def non_increasing(xs):
    return all(a >= b for a, b in zip(xs, xs[1:]))


def stable_within_ties(units, keys):
    """Among units of equal key, tensor order and unit order are kept."""
    seen = {}
    for (t, s), k in zip(units.tolist(), keys):
        if k in seen and seen[k] > (t, s):
            return False
        seen[k] = (t, s)
    return True


@pytest.mark.parametrize("seed", range(6))
def test_every_unit_once_largest_work_first(seed):
    rng = np.random.default_rng(seed)
    shapes = random_shapes(rng, int(rng.integers(1, 120)))
    r = L.schedule_info(shapes)
    assert len(r["groups"]) == 0
    strips = r["strip_rows"]
    assert np.all((strips >= 1) & (strips <= MAX_STRIP_ROWS))
    for (rows, _), sr in zip(shapes, strips):
        assert sr <= rows
    e0, e1, e2 = expected_units(shapes, strips)
    check_cover(r["k0"], e0)
    check_cover(r["k1"], e1)
    check_cover(r["k2"], e2)
    k0_keys = strip_elems(shapes, strips, r["k0"])
    assert non_increasing(k0_keys) and stable_within_ties(r["k0"], k0_keys)
    k1_keys = sizes(shapes, r["k1"])
    assert non_increasing(k1_keys) and stable_within_ties(r["k1"], k1_keys)
    assert r["k2"].tolist() == sorted(r["k2"].tolist())        # tensor order


def test_vit_b16_strips_about_32k_elements_within_the_partial_cap():
    """The largest tensors are 2.36M elements: no strip list exceeds 65,536
    column partials."""
    shapes = [synth.rows_cols(s) for _, s in synth.vit_b16_shapes()]
    r = L.schedule_info(shapes)
    for (rows, cols), sr in zip(shapes, r["strip_rows"]):
        n_strips = cdiv(rows, int(sr))
        assert n_strips * cols <= 65536                         # column partials one block sums
        if rows == 1:
            assert n_strips == 1
        else:
            assert int(sr) * cols >= 16384 or n_strips == 1
            # about 32K elements a strip; larger only where one row less per
            # strip would exceed the cap on column partials
            assert int(sr) * cols <= 2 * 32768 or cdiv(rows, int(sr) - 1) * cols > 65536
    assert len(r["k1"]) == sum(cdiv(a * b, K1_CHUNK) for a, b in shapes)


def test_very_large_tensor_gets_many_strips():
    """A 50M-element tensor is not left to a few huge strips: its strips
    are capped by 262,144 column partials (here 262 strips of 191 rows)."""
    r = L.schedule_info([(768, 768), (50000, 1000)])
    sr = int(r["strip_rows"][1])
    n_strips = cdiv(50000, sr)
    assert n_strips * 1000 <= 4 * 65536
    assert n_strips >= 200
    assert r["k0"][0].tolist()[0] == 1                           # its strips go first


def test_tall_thin_and_rank1_views():
    r = L.schedule_info([(100_000, 3), (1, 123_457), (1, 1)])
    assert int(r["strip_rows"][0]) <= MAX_STRIP_ROWS
    assert cdiv(100_000, int(r["strip_rows"][0])) * 3 <= 65536
    assert int(r["strip_rows"][1]) == 1 and int(r["strip_rows"][2]) == 1
    k0 = [tuple(u) for u in r["k0"].tolist()]
    assert (1, 0) in k0 and (2, 0) in k0 and (1, 1) not in k0  # one strip per [1 x n] view


@pytest.mark.parametrize("budget_mb", [1, 64, 96])
@pytest.mark.parametrize("seed", range(3))
def test_sweep_groups_partition_the_list(budget_mb, seed):
    rng = np.random.default_rng(100 + seed)
    shapes = random_shapes(rng, 80)
    budget = budget_mb << 20
    flat = L.schedule_info(shapes)
    r = L.schedule_info(shapes, sweep_bytes=budget)
    g = r["groups"]
    assert len(g) >= 1
    strips = r["strip_rows"]
    assert np.array_equal(strips, flat["strip_rows"])
    per = {0: "k0", 1: "k1", 2: "k2"}
    next_tensor = 0
    for gi, row in enumerate(g.tolist()):
        tensors = None
        for k in range(3):
            first, count = row[2 * k], row[2 * k + 1]
            assert first == (0 if gi == 0 else g[gi - 1][2 * k] + g[gi - 1][2 * k + 1])
            part = r[per[k]][first:first + count]
            ts = sorted({t for t, _ in part.tolist()})
            tensors = ts if tensors is None else tensors
            assert ts == tensors or count == 0
        # consecutive tensors, within the budget unless a single tensor
        assert tensors == list(range(next_tensor, next_tensor + len(tensors)))
        next_tensor += len(tensors)
        state = sum(24 * shapes[t][0] * shapes[t][1] for t in tensors)
        assert state <= budget or len(tensors) == 1
        # the next tensor would not have fitted
        if next_tensor < len(shapes):
            assert state + 24 * shapes[next_tensor][0] * shapes[next_tensor][1] > budget
        k0 = r["k0"][row[0]:row[0] + row[1]]
        assert non_increasing(strip_elems(shapes, strips, k0))
        k1 = r["k1"][row[2]:row[2] + row[3]]
        assert non_increasing(sizes(shapes, k1))
    assert next_tensor == len(shapes)
    for k in ("k0", "k1", "k2"):                                  # same units as one launch
        assert sorted(map(tuple, r[k].tolist())) == sorted(map(tuple, flat[k].tolist()))
    assert r["k2"].tolist() == flat["k2"].tolist()


def test_one_group_over_everything_is_the_plain_schedule():
    shapes = random_shapes(np.random.default_rng(9), 50)
    flat = L.schedule_info(shapes)
    r = L.schedule_info(shapes, sweep_bytes=1 << 50)
    assert len(r["groups"]) == 1
    for k in ("k0", "k1", "k2"):
        assert np.array_equal(r[k], flat[k])


def test_empty_list_and_errors():
    r = L.schedule_info([])
    assert all(len(r[k]) == 0 for k in ("k0", "k1", "k2")) and len(r["groups"]) == 0
    with pytest.raises(L.LoptError) as e:
        L.schedule_info([(0, 5)])
    assert e.value.code == -2
    with pytest.raises(L.LoptError) as e:
        L.schedule_info([(1 << 16, 1 << 15)])                       # 2^31 elements
    assert e.value.code == -2
    with pytest.raises(L.LoptError) as e:
        L.schedule_info([(4, 4)], sweep_bytes=-1)
    assert e.value.code == -1
