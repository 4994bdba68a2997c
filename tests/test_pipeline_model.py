"""A discrete model of the tensor-core apply kernel's hand-offs, run on the
CPU over many random interleavings (some with one role starved).

Roles, in the kernel's order of work: two feature groups (alternate stages;
each hands over tile k once the slot's previous tile, k - S, has released
it), the layer-1 and layer-2 MMA threads (tiles in order), and two epilogue
groups (alternate stages; layer 1 of each pair, the rest of a pair two
pairs later, the last pairs after the stage's layer 1).  A stage is loaded
into the ring once the stage kRingStages before it is done.

Waits on barriers are by phase parity, as mbarrier.try_wait.parity is: a
wait for the n-th completion of a barrier passes as soon as the number of
completions has the parity of n + 1.  The model checks that no wait for a
slot release passes before that release (a pass on an older phase would
let a tile overwrite a slot still in use) and that the pipeline never
stalls.  With one release barrier per slot it does pass early; with one
per tile in a rotation of 64, as the kernel has, it does not.
"""

import random

import pytest

STAGE_TILES, RING, LAG, DONE = 8, 6, 2, 64


def run(slots, rotation, n_stages, seed, starve):
    """Returns (stalled, early_passes) for one random interleaving."""
    K = STAGE_TILES * n_stages
    emitted = [False] * K
    done1 = [False] * K
    layer1 = [False] * K
    done2 = [False] * K
    released = [False] * K
    f_done = [False] * n_stages
    e_done = [False] * n_stages
    B = rotation or slots                 # release barriers
    completions = [0] * B
    early = []

    def loaded(n):
        return n < RING or (f_done[n - RING] and e_done[n - RING])

    def feature(g):
        for n in range(g, n_stages, 2):
            yield loaded, n
            for k in range(n * STAGE_TILES, (n + 1) * STAGE_TILES, 2):
                def can(k=k):
                    for x in (k, k + 1):
                        j = x - slots           # the tile whose release is awaited
                        if j < 0:
                            continue
                        b, phase = (j % B, j // B) if rotation else (x % slots, x // slots - 1)
                        if (completions[b] & 1) == (phase & 1):   # parity says: not yet
                            return False
                    return True

                def act(k=k):
                    for x in (k, k + 1):
                        if x - slots >= 0 and not released[x - slots]:
                            early.append(x)
                        emitted[x] = True
                yield can, act
            yield (lambda: True), (lambda n=n: f_done.__setitem__(n, True))

    def issuer(ready, out):
        for k in range(0, K, 2):
            yield (lambda k=k: ready[k] and ready[k + 1]), (lambda k=k: (out.__setitem__(k, True), out.__setitem__(k + 1, True)))

    def epilogue(g):
        for n in range(g, n_stages, 2):
            yield loaded, n
            k0 = n * STAGE_TILES

            def l1(j):
                k = k0 + j
                return (lambda k=k: done1[k]), (lambda k=k: (layer1.__setitem__(k, True), layer1.__setitem__(k + 1, True)))

            def fin(j):
                k = k0 + j

                def act(k=k):
                    for x in (k, k + 1):
                        released[x] = True
                        completions[(x % B) if rotation else (x % slots)] += 1
                return (lambda k=k: done2[k]), act
            for j in range(0, STAGE_TILES, 2):
                yield l1(j)
                if j >= 2 * LAG:
                    yield fin(j - 2 * LAG)
            for j in range(STAGE_TILES - 2 * LAG, STAGE_TILES, 2):
                yield fin(j)
            yield (lambda: True), (lambda n=n: e_done.__setitem__(n, True))

    actors = [feature(0), feature(1), issuer(emitted, done1), issuer(layer1, done2), epilogue(0), epilogue(1)]
    cur = []
    for a in actors:
        step = next(a, None)
        cur.append(step)
    rng = random.Random(seed)
    slow = rng.randrange(len(actors))

    def ready(i):
        c = cur[i]
        if c is None:
            return False
        cond, arg = c
        return cond(arg) if not callable(arg) else cond()

    while True:
        live = [i for i in range(len(actors)) if ready(i)]
        if not live:
            break
        i = rng.choices(live, weights=[0.02 if starve and i == slow else 1.0 for i in live])[0]
        cond, arg = cur[i]
        if callable(arg):
            arg()
        cur[i] = next(actors[i], None)
    stalled = any(c is not None for c in cur)
    return stalled, early


@pytest.mark.parametrize("slots", [10, 16])
@pytest.mark.parametrize("starve", [False, True])
def test_release_per_tile_rotation_never_passes_early(slots, starve):
    for seed in range(150):
        stalled, early = run(slots, DONE, 14, seed, starve)
        assert not stalled, "stall, seed %d" % seed
        assert not early, "a slot wait passed before the release, tiles %s, seed %d" % (early[:4], seed)


def test_release_per_slot_can_pass_early():
    """The model detects the failure the rotation removes: with one barrier
    per slot, some interleavings let a tile through on an older phase."""
    bad = sum(bool(run(10, 0, 14, seed, True)[1]) for seed in range(150))
    assert bad > 0
