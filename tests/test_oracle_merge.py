"""Pins for oracle.merge: merging shard partials reproduces the unsharded attention
(the identity the ring loop of the 6D attention notes §2.1 relies on)."""

import numpy as np
import pytest

from oracle import attention as A
from oracle import merge as M
from load_balancing_gb300 import workloads as W


def _problem(causal, seed=0):
    B, H, S, d, blk = 1, 2, 256, 16, 32
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((B, H, S, d)) for _ in range(3))
    nQ = S // blk
    mask = (rng.random((B, H, nQ, nQ)) < 0.5).astype(np.uint8)
    mask[..., np.arange(nQ), np.arange(nQ)] = 1
    if causal:
        mask = mask * np.tril(np.ones((nQ, nQ), np.uint8))
    return q, k, v, mask, blk


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("n_shards", [1, 2, 4, 8])
def test_merge_of_shards_equals_unsharded(causal, layout, n_shards):
    q, k, v, mask, blk = _problem(causal)
    o_ref, lse_ref = A.attention(q, k, v, mask, blk, causal)
    sm = W.shard_masks(mask, n_shards, layout)
    parts = [A.attention_partials(q, k, v, sm[s], blk, causal) for s in range(n_shards)]
    o_p = np.stack([p[0] for p in parts]).reshape(n_shards, -1, q.shape[-1])
    m_p = np.stack([p[1] for p in parts]).reshape(n_shards, -1)
    l_p = np.stack([p[2] for p in parts]).reshape(n_shards, -1)
    o, lse = M.merge_partials(o_p, m_p, l_p)
    np.testing.assert_allclose(o.reshape(o_ref.shape), o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(lse_ref.shape), lse_ref, rtol=0, atol=1e-12)
    assert np.isfinite(o).all()


def test_single_shard_is_identity_and_empty_rows_stay_clean():
    rng = np.random.default_rng(2)
    o = rng.standard_normal((1, 5, 4))
    m = rng.standard_normal((1, 5))
    l = rng.random((1, 5)) + 0.5
    m[0, 2], l[0, 2], o[0, 2] = -np.inf, 0.0, 0.0
    out, lse = M.merge_partials(o, m, l)
    live = [0, 1, 3, 4]
    np.testing.assert_allclose(out[live], o[0, live] / l[0, live][:, None], atol=1e-15)
    np.testing.assert_allclose(lse[live], m[0, live] + np.log(l[0, live]), atol=1e-15)
    assert (out[2] == 0).all() and lse[2] == -np.inf


def test_all_empty_shards():
    o = np.zeros((3, 2, 4))
    m = np.full((3, 2), -np.inf)
    l = np.zeros((3, 2))
    out, lse = M.merge_partials(o, m, l)
    assert (out == 0).all() and (lse == -np.inf).all()


def test_shard_order_does_not_matter():
    q, k, v, mask, blk = _problem(True, seed=3)
    sm = W.shard_masks(mask, 4, "striped")
    parts = [A.attention_partials(q, k, v, sm[s], blk, True) for s in range(4)]
    o_p = np.stack([p[0] for p in parts]).reshape(4, -1, q.shape[-1])
    m_p = np.stack([p[1] for p in parts]).reshape(4, -1)
    l_p = np.stack([p[2] for p in parts]).reshape(4, -1)
    a = M.merge_partials(o_p, m_p, l_p)
    perm = [3, 1, 0, 2]
    b = M.merge_partials(o_p[perm], m_p[perm], l_p[perm])
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)
