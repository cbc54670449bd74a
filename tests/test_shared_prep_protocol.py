"""The hand-off protocol of the shared-preparation kernel (csrc/kda_fwd_shared.cuh), run as a
model on the CPU under random interleavings of its roles.

Per CTA r of a cluster of VS: a feeder imports chunk n into stage n % NST once the stage is free
and ready[n % NG] says the entry holds chunk n, and, on reusing a stage, releases the entry of the
chunk NST earlier on its owner's gfree; two prep lanes prepare the CTA's own chunks n = r + VS j
(lane j % 2), wait on their own gfree[n % NG] for the entry's previous chunk to have been imported
everywhere, write the entry and arrive on ready[n % NG] of every CTA; the scan consumes stages in
order. mbarriers follow the hardware's parity rule: a wait for the phase with parity p passes as
soon as the barrier's current phase has the other parity. The checks: the run never deadlocks, no
wait passes on a phase other than the one it means (parity aliasing), every import reads the chunk
it expects, and no entry is overwritten before every CTA has imported it. A 16-entry ring passes at
every split; an 8-entry ring at split 8 (each owner's two lanes then share one entry) is caught."""
import random

import pytest

NST, NL = 7, 2


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0  # phase = completed phases

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


class Aliasing(AssertionError):
    pass


def _wait(bar, k):
    """A wait for phase k (parity k & 1): passes when the current phase's parity differs."""
    while (bar.phase & 1) == (k & 1):
        yield False
    if bar.phase != k + 1:
        raise Aliasing(f"wait for phase {k} passed with {bar.phase} phases completed")
    yield True


def run(VS, nch, NG, seed):
    rng = random.Random(seed)
    ready = [[Bar(1) for _ in range(NG)] for _ in range(VS)]
    gfree = [[Bar(VS) for _ in range(NG)] for _ in range(VS)]
    full = [[Bar(1) for _ in range(NST)] for _ in range(VS)]
    empty = [[Bar(1) for _ in range(NST)] for _ in range(VS)]
    entry = [None] * NG                   # the chunk each workspace entry holds
    imported = [set() for _ in range(NG)]  # CTAs that imported the entry's current chunk
    stage = [[None] * NST for _ in range(VS)]

    def feeder(r):
        for n in range(nch):
            s, e = n % NST, n % NG
            if n >= NST:
                yield from _wait(empty[r][s], n // NST - 1)
                m = n - NST
                gfree[m % VS][m % NG].arrive()
            yield from _wait(ready[r][e], n // NG)
            assert entry[e] == n, f"CTA {r} imports entry {e} holding {entry[e]}, expected chunk {n}"
            stage[r][s] = n
            imported[e].add(r)
            full[r][s].arrive()
            yield True

    def prep(r, ln):
        for j in range(ln, nch, NL):
            n = r + VS * j
            if n >= nch:
                return
            e = n % NG
            if n >= NG:
                yield from _wait(gfree[r][e], n // NG - 1)
                assert imported[e] == set(range(VS)), f"entry {e} overwritten before every CTA imported it"
            entry[e] = n
            imported[e] = set()
            yield True
            for q in range(VS):
                ready[q][e].arrive()
            yield True

    def scan(r):
        for n in range(nch):
            s = n % NST
            yield from _wait(full[r][s], n // NST)
            assert stage[r][s] == n
            yield True
            empty[r][s].arrive()

    actors = [feeder(r) for r in range(VS)] + [prep(r, ln) for r in range(VS) for ln in range(NL)] + \
             [scan(r) for r in range(VS)]
    live = list(range(len(actors)))
    stalled = 0
    while live:
        i = rng.choice(live)
        try:
            progressed = next(actors[i])
        except StopIteration:
            live.remove(i)
            stalled = 0
            continue
        stalled = 0 if progressed else stalled + 1
        if stalled > 50 * len(actors) + 1000:
            raise AssertionError(f"deadlock with {len(live)} roles waiting")
    return True


@pytest.mark.parametrize("VS", [2, 4, 8])
@pytest.mark.parametrize("nch", [1, 3, 8, 17, 40, 97])
def test_protocol_holds_with_a_16_entry_ring(VS, nch):
    for seed in range(4):
        assert run(VS, nch, NG=16, seed=seed)


def test_an_8_entry_ring_aliases_at_split_8_only():
    """With VS = NG = 8 an owner's two prep lanes wait on the same gfree barrier, one of them a
    phase ahead: the model must catch the aliasing (the reason the kernel's ring has 16 entries).
    At splits 2 and 4 an 8-entry ring still gives each lane entries of its own and holds -- as the
    kernel did on the GPU with 8 entries, where only split 8 ran into a wait timeout."""
    for seed in range(8):
        with pytest.raises(Aliasing):
            run(8, 64, NG=8, seed=seed)
        for VS in (2, 4):
            assert run(VS, 64, NG=8, seed=seed)
