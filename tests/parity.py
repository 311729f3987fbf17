"""Shared tolerances and comparison helpers for the GPU parity tests.

Tolerances for bf16 outputs against the fp64 oracle: max |dO| <= 2e-2 and
mean |dO| <= 2e-3; LSE within 1e-3 absolute (natural-log units). Integer outputs
(loads, worklists) must be bit-exact.
"""

import numpy as np
import torch

from oracle import attention as A

TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE = 1e-3


def to64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_rows_close(o, o_ref, lse=None, lse_ref=None, what=""):
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= TOL_MAX, f"{what}: max |dO| = {err.max():.3e}"
    assert err.mean() <= TOL_MEAN, f"{what}: mean |dO| = {err.mean():.3e}"
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        empty = ~np.isfinite(lse_ref)
        assert (lse[empty] == -np.inf).all(), f"{what}: empty rows must have LSE = -inf"
        assert np.isfinite(lse[~empty]).all(), f"{what}: non-finite LSE on a live row"
        if (~empty).any():
            d = np.abs(lse[~empty] - lse_ref[~empty]).max()
            assert d <= TOL_LSE, f"{what}: max |dLSE| = {d:.3e}"
    return float(err.max()), float(err.mean())


def oracle_item(q, k, v, mask, b, h, qb, block, causal, scale=None):
    """Oracle for one item from torch tensors on any device (copies one head)."""
    qh = to64(q[b, h, qb * block:(qb + 1) * block])[None, None]
    kh = to64(k[b, h])[None, None]
    vh = to64(v[b, h])[None, None]
    mrow = np.asarray(mask[b, h, qb])[None, None, None, :]
    # attention_item reads rows qb*block.. of q: give it a q whose row 0 is the item
    S = kh.shape[2]
    qfull = np.zeros((1, 1, S, qh.shape[-1]))
    qfull[0, 0, qb * block:(qb + 1) * block] = qh[0, 0]
    mfull = np.zeros((1, 1, mask.shape[2], mask.shape[3]), dtype=np.uint8)
    mfull[0, 0, qb] = mrow[0, 0, 0]
    return A.attention_item(qfull, kh, vh, mfull, 0, 0, qb, block, causal, scale)


def sample_items(mask_np, n_random, n_heavy, seed, whole_heads=()):
    """Item ids for sampled parity: given whole heads, n_random uniform items and the
    n_heavy items with the largest dense-block counts."""
    B, H, nQ, _ = mask_np.shape
    loads = (mask_np != 0).sum(-1).reshape(-1)
    rng = np.random.default_rng(seed)
    items = set(rng.choice(loads.size, size=min(n_random, loads.size), replace=False).tolist())
    items |= set(np.argsort(-loads, kind="stable")[:n_heavy].tolist())
    for (b, h) in whole_heads:
        base = (b * H + h) * nQ
        items |= set(range(base, base + nQ))
    return sorted(items)


def check_items(w, mask_np, q, k, v, out, lse, items, scale=None):
    """Sampled parity: every item of ``items`` against the oracle over its admissible
    keys, copying each head's K and V to the host once."""
    by_head = {}
    for item in items:
        bh, qb = divmod(int(item), w.nQ)
        by_head.setdefault(bh, []).append(qb)
    for bh, qbs in sorted(by_head.items()):
        b, h = divmod(bh, w.H)
        kh, vh = to64(k[b, h]), to64(v[b, h])
        for qb in qbs:
            rows = slice(qb * w.block, (qb + 1) * w.block)
            r = A.attention_item_keys(to64(q[b, h, rows]), kh, vh, mask_np[b, h, qb], w.block, qb, w.causal,
                                      scale)
            assert_rows_close(to64(out[b, h, rows]), r["o"], to64(lse[b, h, rows]), r["lse"],
                              what=f"{w.name} item {bh * w.nQ + qb}")

