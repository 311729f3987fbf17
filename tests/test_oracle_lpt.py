"""Pins for oracle.lpt: the page's counter-example, the page's worst-case bound on
brute-forced tiny instances, Graham's tight family, and the bonus special cases."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import lpt
from conftest import load_golden


def test_page_counterexample():
    g = load_golden("lpt_counterexample.json")
    plan = lpt.lpt_plan(g["loads"], g["n_workers"])
    parts = [[g["loads"][i] for i in plan["worklist"][plan["offsets"][p]:plan["offsets"][p + 1]]]
             for p in range(g["n_workers"])]
    assert parts == g["lpt_partition_by_worker"]
    assert plan["makespan"] == g["lpt_makespan"]
    assert plan["worker_loads"].tolist() == [17, 13]
    assert plan["worker_of"].tolist() == [0, 1, 1, 0, 0]
    assert lpt.brute_force_opt(g["loads"], g["n_workers"]) == g["opt_makespan"]
    assert sum(g["opt_partition"][0]) == g["opt_makespan"]


def test_loop_version_matches_numpy_version():
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(0, 30))
        m = int(rng.integers(1, 9))
        loads = rng.integers(0, 25, n)
        home = rng.integers(0, m, n)
        bonus = int(rng.integers(0, 30))
        for h, b in [(None, 0), (home, bonus)]:
            a = lpt.lpt_plan(loads, m, h, b)
            wo, L = lpt.lpt_plan_loops(loads, m, h, b)
            assert a["worker_of"].tolist() == wo
            assert a["worker_loads"].tolist() == L


def test_worst_case_bound_on_brute_forced_instances():
    """db-SP blog, scenario 1: LPT <= (4m-1)/(3m) * OPT."""
    rng = np.random.default_rng(0)
    worst = {}
    for seed in range(240):
        m = [2, 3, 4][seed % 3]
        n = int(rng.integers(m + 1, 9))
        loads = rng.integers(1, 21, n)
        got = lpt.lpt_plan(loads, m)["makespan"]
        opt = lpt.brute_force_opt(loads, m)
        assert opt <= got
        assert Fraction(got, opt) <= Fraction(4 * m - 1, 3 * m)
        worst[m] = max(worst.get(m, Fraction(1)), Fraction(got, opt))
    assert all(v >= 1 for v in worst.values())


@pytest.mark.parametrize("m", [2, 3, 4])
def test_graham_tight_family(m):
    """Graham's tight instance: 2m+1 jobs 2m-1, 2m-1, 2m-2, 2m-2, ..., m+1, m+1, m, m, m.
    LPT's makespan is 4m-1, the optimum is 3m: the page's bound is attained."""
    loads = []
    for t in range(2 * m - 1, m, -1):
        loads += [t, t]
    loads += [m, m, m]
    got = lpt.lpt_plan(loads, m)["makespan"]
    assert got == 4 * m - 1
    assert lpt.brute_force_opt(loads, m) == 3 * m
    assert Fraction(got, 3 * m) == Fraction(4 * m - 1, 3 * m)


def test_bonus_zero_equals_no_home():
    rng = np.random.default_rng(11)
    loads = rng.integers(0, 40, 300)
    home = rng.integers(0, 17, 300)
    a = lpt.lpt_plan(loads, 17)
    b = lpt.lpt_plan(loads, 17, home, 0)
    for k in ("worker_of", "offsets", "worklist", "worker_loads"):
        np.testing.assert_array_equal(a[k], b[k])


def test_huge_bonus_keeps_everything_home():
    rng = np.random.default_rng(12)
    loads = rng.integers(1, 40, 200)
    home = rng.integers(0, 9, 200)
    plan = lpt.lpt_plan(loads, 9, home, int(loads.sum()) + 1)
    np.testing.assert_array_equal(plan["worker_of"], home)
    # true loads are accrued: each worker holds the sum of its home items
    for p in range(9):
        assert plan["worker_loads"][p] == loads[home == p].sum()


def test_more_workers_than_items():
    loads = [5, 9, 9, 1, 0, 3]
    plan = lpt.lpt_plan(loads, 10)
    order = lpt.lpt_order(loads)
    assert order == [1, 2, 0, 5, 3, 4]
    for rank, i in enumerate(order):
        assert plan["worker_of"][i] == rank
    assert plan["offsets"].tolist() == [0, 1, 2, 3, 4, 5, 6, 6, 6, 6, 6]


def test_csr_invariants():
    rng = np.random.default_rng(5)
    loads = rng.integers(0, 64, 1000)
    plan = lpt.lpt_plan(loads, 37)
    off, wl, wo = plan["offsets"], plan["worklist"], plan["worker_of"]
    assert off[0] == 0 and off[-1] == 1000 and (np.diff(off) >= 0).all()
    assert sorted(wl.tolist()) == list(range(1000))
    for p in range(37):
        items = wl[off[p]:off[p + 1]]
        assert (wo[items] == p).all()
        assert plan["worker_loads"][p] == loads[items].sum()
        # assignment order: heaviest first, equal loads by id
        keys = [(-loads[i], i) for i in items]
        assert keys == sorted(keys)
    # the greedy's balance guarantee: no worker exceeds the least-loaded one by
    # more than the largest item
    assert plan["worker_loads"].max() - plan["worker_loads"].min() <= loads.max()


def test_empty_input():
    plan = lpt.lpt_plan([], 4)
    assert plan["offsets"].tolist() == [0, 0, 0, 0, 0]
    assert plan["worklist"].size == 0
