"""Oracle: splitting heavy items into pieces along their KV blocks (test infrastructure only).

db-SP blog, scenario 1: the greedy cannot reach a perfect balance, partly because an
item's load cannot be divided; the closing remark of the page points at splitting the
load further. An item (b, h, q-block) whose row holds L dense blocks is cut here into k
pieces along its KV blocks; each piece is an item of its own for the greedy, its
attention result is a partial (O, m, l) over its blocks, and the partials of one item
are combined with the running-maximum rescale of the 6D attention notes, section 2.1
(step 3 of the ring loop and the final division), so the split result equals the
unsplit one up to rounding.

Readings where nothing fixes the rule (applied identically on the GPU):
* an item is split when its load L exceeds ``max_piece_load`` T, into
  k = min(ceil(L / T), max_pieces) pieces; otherwise k = 1 (kept whole);
* piece j of k takes the dense blocks whose rank in the row (column order, within
  the causal limit) lies in [floor(j L / k), floor((j + 1) L / k)), so piece loads
  differ by at most one and add up to L;
* units: first every whole item in item order, then the pieces of the split items
  in (item, j) order; the pieces of split item s use partial slots
  split_off[s] .. split_off[s + 1] - 1, and unit n_whole + slot is that piece;
* ``unit_pk`` packs j | k << 16; a whole item has j = 0, k = 1 and slot -1.
"""

import numpy as np


def split_counts(load, max_piece_load, max_pieces):
    """k for one item: 1 when load <= T, else min(ceil(load / T), max_pieces)."""
    load, t, p = int(load), int(max_piece_load), int(max_pieces)
    if load <= t:
        return 1
    return min((load + t - 1) // t, p)


def piece_range(load, j, k):
    """Dense-rank range [lo, hi) of piece j of k of a row with `load` dense blocks."""
    load, j, k = int(load), int(j), int(k)
    return (j * load) // k, ((j + 1) * load) // k


def split_plan(loads, max_piece_load, max_pieces):
    """The unit table of a split plan, by explicit loops over the items.

    loads: int sequence [n] (dense blocks per item); max_piece_load >= 1; max_pieces >= 1.
    Returns a dict of int64 arrays: unit_item, unit_pk, unit_slot, unit_load (length
    U = n_whole + n_slots), split_item [n_split], split_off [n_split + 1], and the
    counts (U, n_whole, n_split, n_slots).
    """
    loads = [int(x) for x in loads]
    assert max_piece_load >= 1 and max_pieces >= 1
    ks = [split_counts(x, max_piece_load, max_pieces) for x in loads]
    whole = [i for i, k in enumerate(ks) if k == 1]
    split = [i for i, k in enumerate(ks) if k > 1]
    unit_item, unit_pk, unit_slot, unit_load = [], [], [], []
    for i in whole:
        unit_item.append(i)
        unit_pk.append(0 | (1 << 16))
        unit_slot.append(-1)
        unit_load.append(loads[i])
    split_off = [0]
    for i in split:
        k = ks[i]
        for j in range(k):
            lo, hi = piece_range(loads[i], j, k)
            unit_item.append(i)
            unit_pk.append(j | (k << 16))
            unit_slot.append(split_off[-1] + j)
            unit_load.append(hi - lo)
        split_off.append(split_off[-1] + k)
    n_whole, n_split, n_slots = len(whole), len(split), split_off[-1]
    as64 = lambda a: np.asarray(a, dtype=np.int64)
    return {
        "unit_item": as64(unit_item),
        "unit_pk": as64(unit_pk),
        "unit_slot": as64(unit_slot),
        "unit_load": as64(unit_load),
        "split_item": as64(split),
        "split_off": as64(split_off),
        "counts": (n_whole + n_slots, n_whole, n_split, n_slots),
    }


def piece_columns(dense_cols, load, j, k):
    """The KV-block columns of piece j of k, from the row's dense columns in order."""
    lo, hi = piece_range(load, j, k)
    return list(dense_cols[lo:hi])


def auto_piece_load(total_load, n_workers):
    """Default T: half the mean load per worker, ceil(ceil(total / m) / 2), at least 1.

    An item heavier than that is what keeps LPT away from the mean (its makespan is
    at least the largest item); pieces of at most half the mean leave LPT within
    half a mean of it.
    """
    mean = -(-int(total_load) // int(n_workers))
    return max(1, -(-mean // 2))
