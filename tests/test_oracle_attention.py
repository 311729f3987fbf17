"""Pins for oracle.attention: library attention (torch SDPA in fp64) on masks that
reduce to dense or causal attention, closed forms, and structural invariants."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, causal=False, scale=None, attn_mask=None):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.float64)
    out = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), is_causal=causal, scale=scale,
        attn_mask=None if attn_mask is None else torch.from_numpy(attn_mask))
    return out.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_is_dense_attention(causal):
    B, H, S, d, blk = 2, 3, 96, 16, 32
    q, k, v = (_rand((B, H, S, d), s) for s in (1, 2, 3))
    mask = np.ones((B, H, S // blk, S // blk), dtype=np.uint8)
    o, lse = A.attention(q, k, v, mask, blk, causal)
    np.testing.assert_allclose(o, _sdpa(q, k, v, causal=causal), rtol=0, atol=1e-12)
    # LSE against an independent closed form: log of the softmax denominator
    s = np.einsum("bhqd,bhkd->bhqk", q, k) / math.sqrt(d)
    if causal:
        s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
    ref = np.log(np.exp(s).sum(-1))
    np.testing.assert_allclose(lse, ref, rtol=1e-12, atol=1e-12)


def test_general_mask_matches_sdpa_with_element_mask():
    B, H, S, d, blk = 1, 2, 128, 32, 32
    q, k, v = (_rand((B, H, S, d), s) for s in (4, 5, 6))
    rng = np.random.default_rng(9)
    mask = (rng.random((B, H, 4, 4)) < 0.5).astype(np.uint8)
    mask[..., np.arange(4), np.arange(4)] = 1
    el = np.repeat(np.repeat(mask != 0, blk, axis=2), blk, axis=3)
    o, _ = A.attention(q, k, v, mask, blk, False)
    np.testing.assert_allclose(o, _sdpa(q, k, v, attn_mask=el), atol=1e-12)


def test_single_block_per_row_is_softmax_over_that_block():
    B, H, S, d, blk = 1, 1, 128, 8, 32
    q, k, v = (_rand((B, H, S, d), s) for s in (7, 8, 9))
    nQ = S // blk
    pick = [2, 0, 3, 1]
    mask = np.zeros((B, H, nQ, nQ), dtype=np.uint8)
    for i, j in enumerate(pick):
        mask[0, 0, i, j] = 1
    o, _ = A.attention(q, k, v, mask, blk, False)
    for i, j in enumerate(pick):
        rows, cols = slice(i * blk, (i + 1) * blk), slice(j * blk, (j + 1) * blk)
        ref = _sdpa(q[:, :, rows], k[:, :, cols], v[:, :, cols])
        np.testing.assert_allclose(o[:, :, rows], ref, atol=1e-12)


def test_constant_keys_give_uniform_weights():
    """All keys equal: every admissible key has the same score, so O is the mean of
    the admissible V rows and LSE = score + ln(count)."""
    B, H, S, d, blk = 1, 1, 64, 4, 16
    q = _rand((B, H, S, d), 1)
    k = np.broadcast_to(_rand((1, 1, 1, d), 2), (B, H, S, d)).copy()
    v = _rand((B, H, S, d), 3)
    mask = np.array([[1, 0, 1, 0], [0, 1, 0, 0], [1, 1, 1, 1], [0, 0, 1, 1]], np.uint8)[None, None]
    for causal in (False, True):
        o, lse = A.attention(q, k, v, mask, blk, causal, scale=0.5)
        for r in range(S):
            qb = r // blk
            keys = [c for c in range(S) if mask[0, 0, qb, c // blk] and (not causal or c <= r)]
            if not keys:
                assert lse[0, 0, r] == -np.inf and (o[0, 0, r] == 0).all()
                continue
            np.testing.assert_allclose(o[0, 0, r], v[0, 0, keys].mean(0), atol=1e-12)
            score = 0.5 * q[0, 0, r] @ k[0, 0, 0]
            assert abs(lse[0, 0, r] - (score + math.log(len(keys)))) < 1e-12


def test_empty_rows_and_partials():
    B, H, S, d, blk = 1, 1, 64, 8, 16
    q, k, v = (_rand((B, H, S, d), s) for s in (1, 2, 3))
    mask = np.zeros((1, 1, 4, 4), np.uint8)
    mask[0, 0, 1, 2] = 1
    r = A.attention_item(q, k, v, mask, 0, 0, 0, blk, False)
    assert (r["o"] == 0).all() and (r["lse"] == -np.inf).all()
    assert (r["m"] == -np.inf).all() and (r["l"] == 0).all() and (r["o_unnorm"] == 0).all()
    r = A.attention_item(q, k, v, mask, 0, 0, 1, blk, False)
    np.testing.assert_allclose(r["o_unnorm"] / r["l"][:, None], r["o"], atol=1e-13)
    np.testing.assert_allclose(r["m"] + np.log(r["l"]), r["lse"], atol=1e-13)


def test_causal_skips_blocks_above_the_diagonal():
    B, H, S, d, blk = 1, 2, 96, 8, 32
    q, k, v = (_rand((B, H, S, d), s) for s in (1, 2, 3))
    full = np.ones((B, H, 3, 3), np.uint8)
    lower = np.tril(full[0, 0])[None, None].repeat(2, axis=1)
    a = A.attention(q, k, v, full, blk, True)
    b = A.attention(q, k, v, lower, blk, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_permuting_heads_permutes_outputs():
    B, H, S, d, blk = 1, 4, 64, 8, 16
    q, k, v = (_rand((B, H, S, d), s) for s in (1, 2, 3))
    mask = (np.random.default_rng(4).random((B, H, 4, 4)) < 0.6).astype(np.uint8)
    perm = [2, 0, 3, 1]
    o, lse = A.attention(q, k, v, mask, blk, False)
    op, lp = A.attention(q[:, perm], k[:, perm], v[:, perm], mask[:, perm], blk, False)
    np.testing.assert_array_equal(op, o[:, perm])
    np.testing.assert_array_equal(lp, lse[:, perm])


@pytest.mark.parametrize("causal", [False, True])
def test_admissible_key_item_matches_sdpa(causal):
    """The long-sequence form (sum over the admissible keys only) against torch SDPA with
    the element mask, including a row with no dense block and, when causal, a row whose
    only blocks lie above the diagonal."""
    B, H, S, d, blk = 1, 2, 256, 16, 32
    nQ = S // blk
    q, k, v = (_rand((B, H, S, d), s) for s in (31, 32, 33))
    rng = np.random.default_rng(34)
    mask = (rng.random((B, H, nQ, nQ)) < 0.3).astype(np.uint8)
    mask[0, 0, 3] = 0                 # no dense block at all
    mask[0, 1, 2] = 0
    mask[0, 1, 2, 5:] = 1             # only blocks above the diagonal (empty when causal)
    el = np.repeat(np.repeat(mask != 0, blk, axis=2), blk, axis=3)
    if causal:
        el &= np.tril(np.ones((S, S), bool))
    for h in range(H):
        for qb in range(nQ):
            rows = slice(qb * blk, (qb + 1) * blk)
            r = A.attention_item_keys(q[0, h, rows], k[0, h], v[0, h], mask[0, h, qb], blk, qb, causal)
            live = el[0, h, rows].any(-1)
            if live.any():
                ref = _sdpa(q[0, h, rows][live][None], k[0, h][None], v[0, h][None],
                            attn_mask=el[0, h, rows][live][None])[0]
                np.testing.assert_allclose(r["o"][live], ref, rtol=0, atol=1e-12)
            assert (r["o"][~live] == 0).all() and (r["lse"][~live] == -np.inf).all()
            assert (r["m"][~live] == -np.inf).all() and (r["l"][~live] == 0).all()
