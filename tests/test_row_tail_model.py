"""Exhaustive check of the CTA-per-row schedule's dynamic row tail, on the CPU.

P row processors hand out rows as the kernel's ring refills do. Processor p first takes rows
p, p + P, ... below rows_static. When it hands out its last static row it also takes a ticket
from the launch's counter, one call ahead. Later calls turn that ticket into the row
rows_static + t and take the next ticket, until a ticket lands past the last row. Each atomic
add on the counter is one step of the model, and every interleaving of the processors' steps is
searched. The holder of the last ticket, (rows - rows_static) + P - 1, sets the counter back to
0 for the next launch.

The search checks that every row is handed out exactly once, that the reset is the counter's
last access, and that the counter ends at 0. With the last ticket off by one, it finds the
counter left dirty or a reset before other processors' atomics."""
import functools

import pytest


def _search(P, rows, rows_static, last_ticket=None):
    """Returns None when every interleaving is correct, else a description of the first failure."""
    last = (rows - rows_static) + P - 1 if last_ticket is None else last_ticket

    # processor state: (pc, next_static, have_ahead, ahead, exhausted, r)
    def start(p):
        return ("call", p, False, 0, False, -1)

    def steps(st, ctr):
        """The processor's next step: (new state, new counter, emitted row or None, event)."""
        pc, ns, ha, ah, ex, r = st
        if pc == "call":
            if ex:
                return ("done", ns, ha, ah, ex, r), ctr, None, None
            if ns < rows_static:
                r = ns
                ns += P
                if ns >= rows_static:
                    return ("ahead", ns, ha, ah, ex, r), ctr, None, None
                return ("call", ns, ha, ah, ex, r), ctr, r, None
            if ha:
                return take(ns, ah, ctr, atomic=False)
            return ("take", ns, ha, ah, ex, r), ctr, None, None
        if pc == "take":
            return take(ns, ctr, ctr + 1, atomic=True)
        if pc == "ahead":                                 # one atomic: the ticket for next time
            return ("call", ns, True, ctr, ex, r), ctr + 1, r, "atomic"
        raise AssertionError(pc)

    def take(ns, t, ctr, atomic):
        event = "atomic" if atomic else None
        r = rows_static + t
        if r >= rows:
            if t == last:
                return ("done", ns, False, 0, True, -1), 0, None, "reset" if not atomic else "atomic+reset"
            return ("done", ns, False, 0, True, -1), ctr, None, event
        return ("ahead", ns, False, 0, False, r), ctr, None, event

    @functools.lru_cache(maxsize=None)
    def dfs(states, ctr, handed, reset):
        if all(s[0] == "done" for s in states):
            if sorted(handed) != list(range(rows)):
                return "rows handed out %r" % (sorted(handed),)
            if ctr != 0:
                return "counter left at %d" % ctr
            return None
        for i, st in enumerate(states):
            if st[0] == "done":
                continue
            nst, nctr, row, event = steps(st, ctr)
            if event and event.startswith("atomic") and reset:
                return "atomic after the reset"
            nreset = reset or (event is not None and event.endswith("reset"))
            nhanded = handed + ((row,) if row is not None else ())
            if len(set(nhanded)) != len(nhanded):
                return "row %d handed out twice" % row
            err = dfs(states[:i] + (nst,) + states[i + 1:], nctr, tuple(sorted(nhanded)), nreset)
            if err:
                return err
        return None

    return dfs(tuple(start(p) for p in range(P)), 0, (), False)


@pytest.mark.parametrize("P,rows,rows_static", [
    (1, 3, 2), (2, 5, 3), (2, 6, 6), (3, 7, 4), (3, 5, 0), (3, 2, 0), (4, 9, 6), (3, 8, 8),
])
def test_every_row_once_and_the_counter_comes_back_clean(P, rows, rows_static):
    assert _search(P, rows, rows_static) is None


@pytest.mark.parametrize("delta", [-1, 1])
def test_an_off_by_one_last_ticket_is_caught(delta):
    P, rows, rows_static = 3, 7, 4
    good = (rows - rows_static) + P - 1
    assert _search(P, rows, rows_static, last_ticket=good + delta) is not None
