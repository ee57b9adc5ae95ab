"""Split plans restated in plain Python integers -- the oracle's plan.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A plan cuts each row's KV list into tiles of ``tile`` entries and groups
consecutive tiles into splits.  A split is one unit of work whose partial
(out, lse) the combine merges in split order.  Both policies below return, per
row, the split boundaries in tile units: ``[0, e_1, ..., n_tiles]`` (an empty
row has the single empty split ``[0, 0]``), plus the work list: every
(row, split) pair as ``row * max_splits + split``, rows in batch order.

INVARIANT -- FlashMLA issue #212, "Question": the split count of a row derives
only from that row's own length and fixed constants.  Our rule (the constants
are ours; the page prints none):

    n_tiles  = ceil(L / tile)
    tps      = max(min_tps, ceil(n_tiles / max_splits))   # tiles per split
    n_splits = max(1, ceil(n_tiles / tps))
    split s covers tiles [s * tps, min((s + 1) * tps, n_tiles))

BALANCED -- same page, "Where it comes from": a batch-wide block quota

    payload = ceil(total / num_parts) + fixed_overhead,
    total   = sum over rows of (n_tiles + fixed_overhead),

then rows are packed greedily, in batch order, into parts of ``payload``
tiles, each split costing its tiles plus ``fixed_overhead``; a row is cut
wherever a part fills up.  This is our re-derivation of the quoted quota line
and the prose describing the packing loop; ``fixed_overhead`` and
``num_parts`` are inputs here (the library reports the values it used).
"""

from __future__ import annotations

# Split constants per kernel variant: (tile entries, min tiles per split,
# max splits per row).  These are restated independently of the library;
# tests/test_abi_load.py checks that the library reports the same numbers.
VARIANT_CONSTANTS = {
    "fma": (64, 16, 64),
    "mla": (64, 8, 32),
    "gqa_tc": (64, 16, 64),
}

BALANCED_FIXED_OVERHEAD = 2


def ceil_div(a, b):
    return -(-a // b)


def plan_invariant(lengths, tile, min_tps, max_splits):
    """Per-row boundaries (tile units) under the INVARIANT rule."""
    bounds = []
    for L in lengths:
        L = int(L)
        n_tiles = ceil_div(L, tile)
        tps = max(min_tps, ceil_div(n_tiles, max_splits))
        n_splits = max(1, ceil_div(n_tiles, tps))
        bounds.append([min(s * tps, n_tiles) for s in range(n_splits)] + [n_tiles])
    return bounds


def plan_balanced(lengths, tile, max_splits, num_parts, fixed_overhead):
    """Per-row boundaries (tile units) under the batch-wide BALANCED quota."""
    n_tiles = [ceil_div(int(L), tile) for L in lengths]
    total = sum(n + fixed_overhead for n in n_tiles)
    payload = ceil_div(total, max(1, num_parts)) + fixed_overhead
    # the quota is raised, where needed, so that the longest row fits in the
    # split budget: full parts of payload - fixed_overhead tiles cut it into
    # at most max_splits pieces
    longest = max(n_tiles, default=0)
    payload = max(payload, ceil_div(longest, max(1, max_splits - 1)) + fixed_overhead)
    bounds = []
    room = payload  # tiles still free in the current part
    for n in n_tiles:
        cuts = [0]
        begin = 0
        while True:
            rest = n - begin
            if rest + fixed_overhead <= room:
                # the rest of the row fits in this part
                room -= rest + fixed_overhead
                break
            take = room - fixed_overhead
            if take > 0 and len(cuts) < max_splits:
                # fill this part with the row's next `take` tiles and cut there
                begin += take
                cuts.append(begin)
            # open a new part
            room = payload
            if len(cuts) == max_splits:
                # split budget exhausted: the last split takes the rest
                room = max(0, room - (n - begin) - fixed_overhead)
                break
        cuts.append(n)
        bounds.append(cuts)
    return bounds


SORT_KEYS = 256


def work_list(bounds, max_splits):
    """Every (row, split) pair as ``row * max_splits + split``: items with more
    tiles first (key = tile count capped at 255), rows and splits in batch
    order within a key.  The order only decides which CTA takes an item; an
    implementation may order items of equal key differently."""
    items = [(b * max_splits + s, cuts[s + 1] - cuts[s])
             for b, cuts in enumerate(bounds) for s in range(len(cuts) - 1)]
    items.sort(key=lambda it: -min(it[1], SORT_KEYS - 1))  # stable: batch order within a key
    return [slot for slot, _ in items]


def work_key(bounds, max_splits, slot):
    """Sort key of a work item (its tile count, capped)."""
    b, s = divmod(slot, max_splits)
    return min(bounds[b][s + 1] - bounds[b][s], SORT_KEYS - 1)
