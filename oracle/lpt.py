"""Pure-Python oracle of the LPT assignment (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference leg may use this module.

DMuon docs, "架构设计" §3.1 "分区（全局 LPT）": one global
longest-processing-time greedy pass over all work units, with Graham's
bound of at most 4/3 - 1/(3R) times the optimum on R identical slots.
Reading of the greedy's tie rules (the page gives none): items are taken in
descending size, equal sizes by ascending index; each goes to the slot with
the smallest current load, equal loads to the lowest slot index.  With these
rules the assignment is unique, so implementations can be compared bit for
bit.
"""

from __future__ import annotations


def lpt_assign(sizes, n_slots):
    """Assign each item to a slot.  Returns (slot per item, load per slot)."""
    n_slots = int(n_slots)
    sizes = [int(s) for s in sizes]
    if n_slots < 1:
        raise ValueError("need at least one slot")
    if any(s < 0 for s in sizes):
        raise ValueError("item sizes must be non-negative")
    order = sorted(range(len(sizes)), key=lambda i: (-sizes[i], i))
    loads = [0] * n_slots
    slot_of = [-1] * len(sizes)
    for i in order:
        best = 0
        for j in range(1, n_slots):
            if loads[j] < loads[best]:
                best = j
        slot_of[i] = best
        loads[best] += sizes[i]
    return slot_of, loads


def graham_bound(n_slots):
    """Worst-case ratio of the LPT makespan to the optimum on n_slots slots."""
    return 4.0 / 3.0 - 1.0 / (3.0 * n_slots)
