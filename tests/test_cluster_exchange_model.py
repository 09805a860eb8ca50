"""Exhaustive check of the cluster schedule's pipelined exchange protocol, on the CPU.

Each CTA of a cluster walks the same rows. In iteration i it posts row i's slice totals into
exchange slot i mod 3, waits at the cluster barrier for row i - 1, reads row i - 1's slot from
every CTA, and arrives for row i. The first iteration only posts and arrives. After the last row
it waits and reads once more, then passes the final barrier (arrive, wait). The hardware barrier
completes phase k once every CTA has arrived k + 1 times, and a CTA's k-th wait returns only then.

This model runs every interleaving of those steps for small clusters and row counts. It checks
that every read finds the value posted for the row being read, never a later row's. With two
slots instead of three, the same search finds an interleaving where a fast CTA overwrites a slot
before a slow one reads it. That is why the kernel rotates over three slots."""
import functools

import pytest


def _program(rows, stop_at=None):
    """The per-CTA step list of the kernel's loop: (op, row). stop_at: the row whose exchange
    reports a timed-out wait; every CTA reads the same flag, skips the arrive and leaves the loop."""
    steps = []
    for i in range(rows + 1):
        if i < rows:
            steps.append(("post", i))
        if i > 0:
            steps.append(("wait", None))
            steps.append(("read", i - 1))
            if i - 1 == stop_at:
                break
        if i < rows:
            steps.append(("arrive", None))
    steps += [("arrive", None), ("wait", None)]          # the final barrier
    return tuple(steps)


def _violation(ctas, rows, nslots, stop_at=None):
    """True if some interleaving lets a CTA read a slot that no longer holds the row it wants."""
    prog = _program(rows, stop_at)

    @functools.lru_cache(maxsize=None)
    def search(pcs, arrivals, waits, slots):
        done = True
        for c in range(ctas):
            pc = pcs[c]
            if pc == len(prog):
                continue
            done = False
            op, row = prog[pc]
            a, w, sl = list(arrivals), list(waits), [list(x) for x in slots]
            if op == "post":
                sl[c][row % nslots] = row
            elif op == "arrive":
                a[c] += 1
            elif op == "wait":
                # the CTA's w[c]-th wait returns once every CTA has arrived w[c] + 1 times
                if min(arrivals) < waits[c] + 1:
                    continue                                 # blocked
                w[c] += 1
            elif op == "read":
                if any(sl[p][row % nslots] != row for p in range(ctas)):
                    return True
            npcs = pcs[:c] + (pc + 1,) + pcs[c + 1:]
            if search(npcs, tuple(a), tuple(w), tuple(tuple(x) for x in sl)):
                return True
        if not done and all(pcs[c] == len(prog) or prog[pcs[c]][0] == "wait" and
                            min(arrivals) < waits[c] + 1 for c in range(ctas)):
            raise AssertionError("deadlock at %r" % (pcs,))
        return False

    start = tuple([None] * nslots for _ in range(ctas))
    return search((0,) * ctas, (0,) * ctas, (0,) * ctas, tuple(tuple(x) for x in start))


@pytest.mark.parametrize("ctas,rows", [(2, 1), (2, 2), (2, 5), (3, 4), (4, 3)])
def test_three_slots_never_lose_a_row(ctas, rows):
    assert not _violation(ctas, rows, 3)


@pytest.mark.parametrize("stop_at", [0, 1, 3])
def test_joint_stop_reaches_the_final_barrier(stop_at):
    # a deadlock raises inside the search
    assert not _violation(3, 4, 3, stop_at)


def test_two_slots_would_race():
    assert _violation(2, 4, 2)


def test_program_alternates_arrive_and_wait():
    # the hardware barrier needs arrive, wait, arrive, wait, ... from every thread
    for rows in range(0, 6):
        for stop_at in [None] + list(range(rows)):
            ops = [op for op, _ in _program(rows, stop_at) if op in ("arrive", "wait")]
            assert ops == ["arrive", "wait"] * (len(ops) // 2)


# ---- the exchanges that are not pipelined --------------------------------------------------
# The FP8 kernels with a weight offset or fp32 input exchange twice per row, each exchange a
# post, an arrive, a wait and a read of every CTA's slot: first the slice sums (slots rotating
# over three), then the slice maxima of |y| (slots rotating over two). A timed-out wait is
# shared through the first exchange; every CTA then leaves the loop before the second. After
# the loop every CTA passes the final barrier.

def _program_unpipelined(rows, slots, stop_at=None):
    """Per-CTA step list: (op, channel, row). `slots` gives each exchange's slot count, in order."""
    steps = []
    for i in range(rows):
        for ch in range(len(slots)):
            steps += [("post", ch, i), ("arrive", ch, None), ("wait", ch, None), ("read", ch, i)]
            if ch == 0 and i == stop_at:
                break
        if i == stop_at:
            break
    steps += [("arrive", None, None), ("wait", None, None)]     # the final barrier
    return tuple(steps)


def _violation_unpipelined(ctas, rows, slots, stop_at=None):
    prog = _program_unpipelined(rows, slots, stop_at)

    @functools.lru_cache(maxsize=None)
    def search(pcs, arrivals, waits, sl):
        done = True
        for c in range(ctas):
            pc = pcs[c]
            if pc == len(prog):
                continue
            done = False
            op, ch, row = prog[pc]
            a, w = list(arrivals), list(waits)
            s = [[list(x) for x in per_cta] for per_cta in sl]
            if op == "post":
                s[c][ch][row % slots[ch]] = row
            elif op == "arrive":
                a[c] += 1
            elif op == "wait":
                if min(arrivals) < waits[c] + 1:
                    continue                                 # blocked
                w[c] += 1
            elif op == "read":
                if any(s[p][ch][row % slots[ch]] != row for p in range(ctas)):
                    return True
            npcs = pcs[:c] + (pc + 1,) + pcs[c + 1:]
            key = tuple(tuple(tuple(x) for x in per_cta) for per_cta in s)
            if search(npcs, tuple(a), tuple(w), key):
                return True
        if not done and all(pcs[c] == len(prog) or prog[pcs[c]][0] == "wait" and
                            min(arrivals) < waits[c] + 1 for c in range(ctas)):
            raise AssertionError("deadlock at %r" % (pcs,))
        return False

    start = tuple(tuple(tuple([None] * n) for n in slots) for _ in range(ctas))
    return search((0,) * ctas, (0,) * ctas, (0,) * ctas, start)


@pytest.mark.parametrize("ctas,rows", [(2, 1), (2, 3), (2, 5), (3, 3), (4, 2)])
def test_two_unpipelined_exchanges_never_lose_a_row(ctas, rows):
    # sums over three slots, maxima over two: a slot is written again only after every CTA has
    # passed a later barrier, so after its reads
    assert not _violation_unpipelined(ctas, rows, (3, 2))


@pytest.mark.parametrize("stop_at", [0, 2])
def test_unpipelined_joint_stop_reaches_the_final_barrier(stop_at):
    assert not _violation_unpipelined(3, 4, (3, 2), stop_at)


@pytest.mark.parametrize("ctas,rows", [(2, 4), (3, 3)])
def test_one_unpipelined_exchange_never_loses_a_row(ctas, rows):
    # one exchange per row over three slots (the W16 kernel's row maximum rides with its sums)
    assert not _violation_unpipelined(ctas, rows, (3,))


def test_unpipelined_single_slot_would_race():
    # the rotation is what makes it safe: one slot per exchange loses a row
    assert _violation_unpipelined(2, 3, (1,))
