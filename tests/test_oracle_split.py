"""Pins for oracle.split: a hand-worked table, the partition of every row's dense
blocks, balanced piece loads against brute force, the piece-size bound implied by
the split rule, and split-then-merge attention equal to the unsplit attention."""

import itertools

import numpy as np
import pytest

from oracle import attention as OA
from oracle import merge as OM
from oracle import split as OS


def test_hand_worked_table():
    # loads [5, 12, 0, 30], T = 8, at most 3 pieces: item 1 -> 2 pieces (6 + 6), item 3 ->
    # ceil(30 / 8) = 4 capped at 3 pieces (10 + 10 + 10); items 0 and 2 stay whole
    t = OS.split_plan([5, 12, 0, 30], 8, 3)
    assert t["counts"] == (7, 2, 2, 5)
    assert t["unit_item"].tolist() == [0, 2, 1, 1, 3, 3, 3]
    assert t["unit_load"].tolist() == [5, 0, 6, 6, 10, 10, 10]
    assert t["unit_slot"].tolist() == [-1, -1, 0, 1, 2, 3, 4]
    assert t["unit_pk"].tolist() == [1 << 16, 1 << 16, 2 << 16, 1 | 2 << 16, 3 << 16, 1 | 3 << 16, 2 | 3 << 16]
    assert t["split_item"].tolist() == [1, 3]
    assert t["split_off"].tolist() == [0, 2, 5]
    # an uneven cut: 7 blocks in min(ceil(7 / 2), 3) = 3 pieces by floor(j * 7 / 3):
    # ranks [0, 2), [2, 4), [4, 7)
    t = OS.split_plan([7], 2, 3)
    assert t["unit_load"].tolist() == [2, 2, 3]
    assert [OS.piece_range(7, j, 3) for j in range(3)] == [(0, 2), (2, 4), (4, 7)]


def test_pieces_partition_every_row():
    rng = np.random.default_rng(0)
    for _ in range(200):
        nk = int(rng.integers(1, 40))
        row = rng.random(nk) < rng.random()
        cols = np.flatnonzero(row)
        load = len(cols)
        for k in range(1, 7):
            got = []
            for j in range(k):
                got += OS.piece_columns(cols, load, j, k)
            assert got == cols.tolist()  # in order, each dense block exactly once


def test_piece_loads_are_the_most_even_split():
    """Brute force over every way to cut L ordered blocks into k runs: the oracle's
    loads reach the minimum possible max - min spread, and they add up to L."""
    for load in range(0, 13):
        for k in range(1, 6):
            sizes = [b - a for a, b in (OS.piece_range(load, j, k) for j in range(k))]
            assert sum(sizes) == load and min(sizes) >= 0
            best = min(max(c) - min(c) for c in itertools.product(range(load + 1), repeat=k) if sum(c) == load)
            assert max(sizes) - min(sizes) == best


def test_split_rule_bounds_the_pieces():
    rng = np.random.default_rng(1)
    loads = rng.integers(0, 300, 500)
    for t_max, p_max in ((1, 1000), (7, 1000), (50, 1000), (50, 3), (299, 2)):
        tab = OS.split_plan(loads, t_max, p_max)
        n_whole, n_split = tab["counts"][1], tab["counts"][2]
        assert n_whole + n_split == len(loads)
        for i, x in enumerate(loads):
            k = OS.split_counts(x, t_max, p_max)
            assert (k == 1) == (x <= t_max) or (k == 1 and p_max == 1)
            assert 1 <= k <= p_max
            if k > 1 and p_max >= -(-x // t_max):
                assert -(-x // k) <= t_max  # uncapped: every piece fits under T
        # units of one item carry its whole load; slots run 0 .. n_slots - 1 in order
        for i in tab["split_item"]:
            sel = tab["unit_item"] == i
            assert tab["unit_load"][sel].sum() == loads[i]
        pieces = tab["unit_slot"][tab["unit_slot"] >= 0]
        assert pieces.tolist() == list(range(tab["counts"][3]))


def test_auto_piece_load():
    assert OS.auto_piece_load(34971, 152) == 116  # ceil(34971 / 152) = 231 -> 116
    assert OS.auto_piece_load(0, 8) == 1
    assert OS.auto_piece_load(10, 1) == 5


@pytest.mark.parametrize("causal", [False, True])
def test_split_attention_equals_unsplit(causal):
    """Every split item's pieces, each attended as a partial over its own blocks and
    combined by the merge, give the unsplit attention of that item."""
    rng = np.random.default_rng(2 + causal)
    B, H, S, d, block = 1, 2, 64, 8, 8
    nq = S // block
    mask = (rng.random((B, H, nq, nq)) < 0.6).astype(np.uint8)
    if causal:
        for qb in range(nq):
            mask[:, :, qb, qb] = 1
    q, k, v = (rng.standard_normal((B, H, S, d)) for _ in range(3))
    ref_o, ref_lse = OA.attention(q, k, v, mask, block, causal)
    for b, h, qb in itertools.product(range(B), range(H), range(nq)):
        limit = qb + 1 if causal else nq
        cols = np.flatnonzero(mask[b, h, qb, :limit])
        load = len(cols)
        for kk in (2, 3):
            o_parts, m_parts, l_parts = [], [], []
            for j in range(kk):
                sub = np.zeros_like(mask)
                sub[b, h, qb, OS.piece_columns(cols, load, j, kk)] = 1
                o_p, m_p, l_p = OA.attention_partials(q, k, v, sub, block, causal)
                rows = slice(qb * block, (qb + 1) * block)
                o_parts.append(o_p[b, h, rows])
                m_parts.append(m_p[b, h, rows])
                l_parts.append(l_p[b, h, rows])
            o, lse = OM.merge_partials(np.stack(o_parts), np.stack(m_parts), np.stack(l_parts))
            rows = slice(qb * block, (qb + 1) * block)
            np.testing.assert_allclose(o, ref_o[b, h, rows], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, ref_lse[b, h, rows], rtol=0, atol=1e-12)


def test_automatic_piece_load_bounds_the_slots():
    """With T = auto_piece_load(total, m), an item of L > T dense blocks makes at most
    ceil(L / T) < 2 L / T pieces, so all pieces together number fewer than
    2 total / T <= 4 m: the capacity the split path allocates by default."""
    rng = np.random.default_rng(7)
    for _ in range(300):
        m = int(rng.integers(1, 300))
        n = int(rng.integers(1, 3000))
        kind = rng.integers(0, 3)
        if kind == 0:
            loads = rng.integers(0, 200, n)
        elif kind == 1:  # a few very heavy items
            loads = rng.integers(0, 3, n)
            loads[rng.integers(0, n, 3)] = rng.integers(1000, 100000, 3)
        else:  # every item just above the automatic T
            t0 = OS.auto_piece_load(n * 50, m)
            loads = np.full(n, t0 + 1)
        total = int(loads.sum())
        t = OS.auto_piece_load(total, m)
        tab = OS.split_plan(loads, t, 10**6)
        assert tab["counts"][3] < 4 * m or total == 0
