"""Model check (CPU) of the tensor-core kernel's barrier protocol.

The roles of the kernel in `convolution_epilogue_gb300/csrc/fc_tc.cu` are
written here as generators that follow the kernel's control flow step by
step: producer warps (fill a stage after its "empty" barrier, arrive on
"full"), the MMA warp (one accumulator wait per unit on the unit's last
tile, non-blocking look-ahead tests of the next stage and the next
accumulator, MMAs issued into an in-order tensor pipe whose commits arrive
on barriers when the MMAs before them complete) and epilogue warps (wait a
tile's "accumulator full", read it, arrive on "accumulator empty"); the
parity-class split schedule (two accumulator halves, a unit's stages held
until its second half) is modelled too.  mbarriers have the hardware phase
semantics: a wait on parity P succeeds once the phase of that parity has
completed.

A random scheduler interleaves the roles and the tensor pipe's completions
for many seeds and plan shapes, and checks: no stage is overwritten while an
issued MMA may still read it, no MMA reads a stage before every producer
wrote it, no accumulator tile is overwritten before the epilogue has read it
or read before its MMAs completed, no wait ever sees a barrier more than one
phase ahead of the phase it means, and every run ends (no deadlock).
"""
import random

import pytest


class Barrier:
    def __init__(self, count, name=""):
        self.count, self.pending, self.phases, self.name = count, count, 0, name

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phases += 1
            self.pending = self.count

    def done(self, parity):  # try_wait / test_wait .parity semantics
        return (self.phases & 1) != parity


class Violation(AssertionError):
    pass


def run_model(S, NACC, U, NCH, units, PW, EW, split, seed, max_ticks=200000):
    rng = random.Random(seed)
    a_full = [Barrier(PW) for _ in range(S)]
    a_empty = [Barrier(1, "a_empty") for _ in range(S)]
    nacc_bars = NACC * U if not split else 2
    acc_full = [Barrier(1) for _ in range(nacc_bars)]
    acc_empty = [Barrier(EW) for _ in range(nacc_bars)]
    stage_owner = [None] * S        # chunk index g whose data the stage holds
    stage_writes = [0] * S          # producer warps that wrote the current chunk
    stage_readers = [0] * S         # issued, not yet completed MMAs reading it
    tile_state = {}                 # accumulator bar index -> (unit, "mma" | "ready" | "read")
    pipe = []                       # in-order tensor pipe: ("mma", stage, tile) | ("commit", bar)

    def expect_phase(bar, parity, intended):
        # the wait means phase `intended` (0-based); the barrier must not be
        # more than one completed phase past it (the parity would alias)
        if bar.phases > intended + 1:
            raise Violation("a wait fell two phases behind its barrier")

    def producer(pw):
        g = 0
        for u in range(units):
            for c in range(NCH):
                s = g % S
                par = ((g // S) & 1) ^ 1
                while not a_empty[s].done(par):
                    yield
                expect_phase(a_empty[s], par, g // S - 1 if g >= S else -1)
                if stage_readers[s]:
                    raise Violation("producer overwrote a stage an MMA still reads")
                if stage_owner[s] != g:
                    stage_owner[s] = g
                    stage_writes[s] = 0
                stage_writes[s] += 1
                yield
                a_full[s].arrive()
                g += 1

    def issue(s, g, tile):
        if stage_owner[s] != g or stage_writes[s] != PW:
            raise Violation("MMA read a stage before every producer wrote it")
        st = tile_state.get(tile)
        if st is not None and st[1] in ("ready",):
            raise Violation("MMA overwrote an accumulator tile the epilogue has not read")
        stage_readers[s] += 1
        pipe.append(("mma", s, tile))

    def mma():
        g = 0
        macc, mpar = 0, 0
        pre_full = pre_acc = False
        for it in range(units):
            acc = macc
            acc_par = mpar ^ 1
            macc += 1
            if macc == NACC:
                macc, mpar = 0, mpar ^ 1
            if split:
                bars = [0, 1]
                first_bar = 0
            else:
                bars = [acc * U + t for t in range(U)]
                first_bar = acc * U + U - 1
            if not pre_acc:
                while not acc_empty[first_bar].done(acc_par):
                    yield
            pre_acc = False
            for b in (bars if not split else [0]):
                st = tile_state.get(b)
                if st is not None and st[1] != "read":
                    raise Violation("accumulator tile reused before the epilogue read it")
            if split:
                s0 = g % S
                for c in range(NCH):
                    s = (g + c) % S
                    par = ((g + c) // S) & 1
                    if not (c == 0 and pre_full):
                        while not a_full[s].done(par):
                            yield
                    tile_state[0] = (it, "mma")
                    issue(s, g + c, 0)
                    yield
                pipe.append(("commit", ("acc_full", 0)))
                while not acc_empty[1].done(acc_par):
                    yield
                st = tile_state.get(1)
                if st is not None and st[1] != "read":
                    raise Violation("accumulator half B reused before the epilogue read it")
                for c in range(NCH):
                    s = (g + c) % S
                    tile_state[1] = (it, "mma")
                    issue(s, g + c, 1)
                    pipe.append(("commit", ("a_empty", s)))
                    yield
                g += NCH
                pre_full = a_full[g % S].done((g // S) & 1)
                pre_acc = acc_empty[0].done(mpar ^ 1)
                pipe.append(("commit", ("acc_full", 1)))
                yield
                continue
            for c in range(NCH):
                s = g % S
                par = (g // S) & 1
                if not pre_full:
                    while not a_full[s].done(par):
                        yield
                for t in range(U):
                    b = acc * U + t
                    tile_state[b] = (it, "mma")
                    issue(s, g, b)
                    if c == NCH - 1:
                        pipe.append(("commit", ("acc_full", b)))
                    yield
                g += 1
                pre_full = a_full[g % S].done((g // S) & 1)
                if c == NCH - 1:
                    pre_acc = acc_empty[macc * U + U - 1].done(mpar ^ 1)
                pipe.append(("commit", ("a_empty", s)))
                yield

    def epilogue(ew):
        eacc, epar = 0, 0
        for it in range(units):
            acc, par = eacc, epar
            eacc += 1
            if eacc == NACC:
                eacc, epar = 0, epar ^ 1
            bars = [0, 1] if split else [acc * U + t for t in range(U)]
            for b in bars:
                while not acc_full[b].done(par):
                    yield
                st = tile_state.get(b)
                if st is None or st[0] != it or st[1] not in ("ready", "read"):
                    raise Violation("epilogue read an accumulator before its MMAs completed")
                yield
                acc_empty[b].arrive()
                if acc_empty[b].pending == EW:  # phase just completed: all warps read it
                    tile_state[b] = (it, "read")

    def complete_one():
        kind, *rest = pipe.pop(0)
        if kind == "mma":
            s, tile = rest
            stage_readers[s] -= 1
            st = tile_state[tile]
            # a tile is ready only when its committing MMAs are done: mark
            # progress; the commit below publishes it
            tile_state[tile] = (st[0], "mma")
        else:
            which, idx = rest[0]
            if which == "a_empty":
                a_empty[idx].arrive()
            else:
                st = tile_state[idx]
                tile_state[idx] = (st[0], "ready")
                acc_full[idx].arrive()

    actors = [producer(i) for i in range(PW)] + [mma()] + [epilogue(i) for i in range(EW)]
    alive = list(range(len(actors)))
    ticks = 0
    while alive or pipe:
        ticks += 1
        if ticks > max_ticks:
            raise Violation("no progress: deadlock")
        if pipe and (not alive or rng.random() < 0.3):
            complete_one()
            continue
        k = rng.choice(alive)
        try:
            next(actors[k])
        except StopIteration:
            alive.remove(k)
    return ticks


SHAPES = [
    # S, NACC, U, NCH, units, PW, EW, split
    (4, 2, 2, 1, 9, 3, 2, False),   # conv3d / conv2d: two tiles a unit, one chunk
    (4, 4, 1, 1, 11, 2, 2, False),  # single-tile units
    (3, 2, 2, 4, 7, 3, 2, False),   # several chunks a unit (C_in 64), pooled-like
    (2, 2, 2, 3, 6, 2, 3, False),   # fewer stages than chunks
    (1, 4, 1, 2, 5, 2, 2, False),   # one stage
    (4, 1, 1, 4, 7, 3, 2, True),    # parity-class split schedule (NCH <= S)
    (4, 1, 1, 1, 9, 2, 2, True),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_protocol_random_interleavings(shape):
    S, NACC, U, NCH, units, PW, EW, split = shape
    for seed in range(60):
        run_model(S, NACC, U, NCH, units, PW, EW, split, seed)


def test_model_catches_a_planted_race():
    """The checker is not vacuous: a producer that does not wait for the
    stage to be free (planted here, in the model only) is caught."""
    caught = False
    orig = Barrier.done

    def eager(self, parity):  # producers stop waiting for the stage to be free
        return True if self.name == "a_empty" else orig(self, parity)

    Barrier.done = eager
    try:
        for seed in range(40):
            try:
                run_model(1, 2, 2, 2, 6, 2, 2, False, seed)
            except Violation:
                caught = True
                break
    finally:
        Barrier.done = orig
    assert caught


def test_model_catches_a_skipped_accumulator_wait():
    """Planted in the model only: the MMA role does not wait for the
    epilogue to free an accumulator, and the checker reports the reuse."""
    orig = Barrier.done
    msgs = set()

    def eager(self, parity):
        return True if self.count == 2 and self.name == "" and self.pending == 2 else orig(self, parity)

    Barrier.done = eager  # acc_empty barriers have EW = 2 arrivals here
    try:
        for seed in range(60):
            try:
                run_model(4, 2, 2, 1, 12, 3, 2, False, seed)
            except Violation as e:
                msgs.add(str(e))
    finally:
        Barrier.done = orig
    assert any("accumulator" in m for m in msgs), msgs
