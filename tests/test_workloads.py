"""Input generators: determinism, the structural properties each workload promises,
and the dense-block counts the workloads are sized for."""

import numpy as np
import pytest

from load_balancing_gb300 import workloads as W


@pytest.mark.parametrize("name", ["tiny", "llm", "video", "sharded"])
def test_masks_deterministic_and_shaped(name):
    w = W.WORKLOADS[name]
    a, b = W.make_mask(w), W.make_mask(w)
    assert a.dtype == np.uint8 and a.shape == (w.B, w.H, w.nQ, w.nK)
    np.testing.assert_array_equal(a, b)
    assert a.flags["C_CONTIGUOUS"]
    d = np.arange(w.nQ)
    assert (a[..., d, d] == 1).all(), "diagonal must be dense"
    if w.causal:
        assert (np.triu(a, 1) == 0).all()


def test_dense_block_counts():
    tiny = W.make_mask(W.WORKLOADS["tiny"]).sum()
    assert 40 <= tiny <= 100  # 2 heads x (8 + 0.5 x 56) ~ 72
    llm = int(W.make_mask(W.WORKLOADS["llm"]).sum())
    # 16 global heads: 64 + 0.9 x 2016 each (~1878); 16 local heads: 310 each
    assert abs(llm - (16 * (64 + 0.9 * 2016) + 16 * 310)) < 600
    video = int(W.make_mask(W.WORKLOADS["video"]).sum())
    assert 60_000 < video < 170_000
    sharded = int(W.make_mask(W.WORKLOADS["sharded"]).sum())
    assert sharded == 16 * 256 * 257 // 2 == 526_336


def test_video_structure():
    w = W.WORKLOADS["video"]
    m = W.make_mask(w)
    i = np.arange(w.nQ)[:, None]
    j = np.arange(w.nK)[None, :]
    same_frame = (i // 8) == (j // 8)
    same_offset = (i % 8) == (j % 8)
    assert (m[0, :12][:, same_frame] == 1).all()
    assert (m[0, 12:][:, same_offset] == 1).all()


def test_imbalance_rows_have_per_head_constant_count():
    w = W.custom("imb_small", 1, 6, 128 * 64, 128, 128, False, 5, 105, "lognormal",
                 mu=np.log(0.1), sigma=1.0, lo=0.01, hi=0.6)
    m = W.make_mask(w)
    rows = m.sum(-1)
    for h in range(w.H):
        assert (rows[0, h] == rows[0, h, 0]).all()
        assert 1 <= rows[0, h, 0] <= int(round(0.6 * w.nK))
    d = np.arange(w.nQ)
    assert (m[..., d, d] == 1).all()


def test_shard_masks_partition_columns():
    w = W.WORKLOADS["tiny"]
    m = W.make_mask(w)
    for layout in ("contiguous", "striped"):
        sm = W.shard_masks(m, 4, layout)
        np.testing.assert_array_equal(sm.sum(0), m)
        cols = W.shard_columns(w.nK, 4, layout)
        assert sorted(np.concatenate(cols).tolist()) == list(range(w.nK))


def test_qkv_bf16_values_and_determinism():
    import torch

    w = W.WORKLOADS["tiny"]
    q, k, v = W.make_qkv(w)
    assert q.dtype == torch.bfloat16 and q.shape == (w.B, w.H, w.S, w.d)
    q2, _, _ = W.make_qkv(w)
    assert torch.equal(q, q2)
    assert abs(float(q.float().std()) - 1.0) < 0.05
    small = W.custom("s", 1, 2, 256, 64, 64, True, 1, 2)
    a = W.make_qkv(small)[0]
    b = W.make_qkv(small)[0]
    assert torch.equal(a, b)


def test_perturbed_mask():
    w = W.WORKLOADS["llm"]
    m0 = W.make_mask(w)
    m1 = W.perturb_mask(m0, 0.02, 1, w.causal)
    assert np.array_equal(m1, W.perturb_mask(m0, 0.02, 1, w.causal))  # seeded
    nq = w.nQ
    upper = np.triu(np.ones((nq, nq), dtype=bool), 1)
    assert not m1[..., upper].any()  # causal clip kept
    lower = ~upper
    changed = (m0 != m1)[..., lower].mean()
    assert 0.015 < changed < 0.025
