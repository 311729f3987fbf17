"""Oracle: longest-processing-time-first (LPT) planning with a stay-in-place bonus.

Test infrastructure only.

db-SP blog, scenario 1: balancing heads over identical machines is the
identical-machines scheduling problem (minimise the makespan). The greedy the page
uses repeatedly hands the longest remaining job to the machine that is currently
least loaded. The page shows that it is not optimal -- loads [8, 7, 6, 5, 4] on two
machines give [8+5+4, 7+6] (makespan 17) where [8+7, 6+5+4] reaches 15 -- and
states its guarantee: the greedy's makespan is at most (4m-1)/(3m) times the
optimum on m machines.

db-SP blog, scenario 2, third bullet: when Q-blocks are rebalanced the same greedy
is run, except that a Q-block placed on the machine it already lives on is treated
as if its load were somewhat smaller.

Readings where the page is silent (each is applied identically on the GPU):
* equal loads are taken in increasing item id (a stable sort on descending load);
* among equally attractive machines the lowest index wins;
* the bonus is an integer ``stay_bonus`` subtracted from the home machine's
  current load only when choosing; the machine then accrues the item's true load
  (the work does not shrink). ``home=None`` means no bonus.
* the worklist lists, for each machine in index order, its items in the order
  the greedy assigned them (CSR: ``offsets[m+1]``, ``worklist[n]``).
"""

import itertools

import numpy as np


def lpt_order(loads):
    """Item ids sorted by load descending, equal loads by id ascending."""
    loads = [int(x) for x in loads]
    return sorted(range(len(loads)), key=lambda i: (-loads[i], i))


def lpt_plan(loads, n_workers, home=None, stay_bonus=0):
    """Textbook LPT with the stay bonus; numpy argmin per item.

    loads: int sequence [n]; n_workers: m >= 1; home: int sequence [n] or None.
    Returns dict with worker_of [n], offsets [m+1], worklist [n] (int64 arrays),
    worker_loads [m] (true accumulated loads) and makespan.
    """
    loads = np.asarray(loads, dtype=np.int64)
    n = loads.shape[0]
    m = int(n_workers)
    assert m >= 1
    if home is not None:
        home = np.asarray(home, dtype=np.int64)
    L = np.zeros(m, dtype=np.int64)
    worker_of = np.full(n, -1, dtype=np.int64)
    per_worker = [[] for _ in range(m)]
    idx = np.arange(m)
    for i in lpt_order(loads):
        key = L.copy()
        if home is not None:
            key = key - stay_bonus * (idx == home[i])
        p = int(np.argmin(key))  # first minimum: lowest index among ties
        worker_of[i] = p
        L[p] += loads[i]
        per_worker[p].append(i)
    offsets = np.zeros(m + 1, dtype=np.int64)
    for p in range(m):
        offsets[p + 1] = offsets[p] + len(per_worker[p])
    worklist = np.array([i for p in range(m) for i in per_worker[p]], dtype=np.int64)
    return {
        "worker_of": worker_of,
        "offsets": offsets,
        "worklist": worklist,
        "worker_loads": L,
        "makespan": int(L.max()) if m else 0,
    }


def lpt_plan_loops(loads, n_workers, home=None, stay_bonus=0):
    """Same greedy written with plain Python loops (for tiny cross-checks)."""
    loads = [int(x) for x in loads]
    m = int(n_workers)
    L = [0] * m
    worker_of = [-1] * len(loads)
    for i in lpt_order(loads):
        best, best_key = -1, None
        for p in range(m):
            key = L[p]
            if home is not None and int(home[i]) == p:
                key -= stay_bonus
            if best_key is None or key < best_key:
                best, best_key = p, key
        worker_of[i] = best
        L[best] += loads[i]
    return worker_of, L


def brute_force_opt(loads, n_workers):
    """Optimal makespan by trying every assignment of n items to m machines.

    Only for tiny instances (m**n assignments). Exact integer arithmetic.
    """
    loads = np.asarray(loads, dtype=np.int64)
    n, m = loads.shape[0], int(n_workers)
    if n == 0:
        return 0
    assign = np.array(list(itertools.product(range(m), repeat=n)), dtype=np.int8)
    per_machine = np.stack([(assign == p).astype(np.int64) @ loads for p in range(m)], axis=1)
    return int(per_machine.max(axis=1).min())
