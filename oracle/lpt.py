"""Pure-Python oracle of the LPT assignments (test infrastructure only).

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

``lpt_assign_layered`` adds the two constraints the same section builds into
the algorithm: (1) same-layer concurrency -- the parameters of one layer go
to different owner slots; (2) small-parameter merging -- within a layer, the
parameters below a threshold (5e6 elements by default) form one unit that
shares one owner.  Readings taken: a unit is placed on the least-loaded slot
that holds no unit of its layer yet (ties: lowest index), and on the
least-loaded slot overall when every slot already holds one; units are taken
in descending size, ties by their first item's index; items with a negative
layer id belong to no layer (never merged, never constrained).
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


SMALL_PARAM_THRESHOLD = 5_000_000


def lpt_assign_layered(sizes, layers, n_slots, small_threshold=SMALL_PARAM_THRESHOLD):
    """Layer-aware LPT.  Returns (slot per item, load per slot)."""
    n_slots = int(n_slots)
    sizes = [int(s) for s in sizes]
    layers = [int(x) for x in layers]
    if n_slots < 1:
        raise ValueError("need at least one slot")
    if len(layers) != len(sizes):
        raise ValueError("one layer id per item")
    if any(s < 0 for s in sizes):
        raise ValueError("item sizes must be non-negative")
    units = []          # each: [size, first item, items, layer]
    small_unit = {}     # layer -> index of its merged unit
    for i, (size, layer) in enumerate(zip(sizes, layers)):
        if layer >= 0 and size < small_threshold:
            if layer in small_unit:
                u = units[small_unit[layer]]
                u[0] += size
                u[2].append(i)
                continue
            small_unit[layer] = len(units)
        units.append([size, i, [i], layer])
    order = sorted(range(len(units)), key=lambda k: (-units[k][0], units[k][1]))
    loads = [0] * n_slots
    holds = [set() for _ in range(n_slots)]
    slot_of = [-1] * len(sizes)
    for k in order:
        size, _, items, layer = units[k]
        free = [j for j in range(n_slots) if layer < 0 or layer not in holds[j]]
        pool = free if free else list(range(n_slots))
        best = pool[0]
        for j in pool[1:]:
            if loads[j] < loads[best]:
                best = j
        loads[best] += size
        if layer >= 0:
            holds[best].add(layer)
        for i in items:
            slot_of[i] = best
    return slot_of, loads
