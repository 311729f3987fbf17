"""Dense-block lists and the attention producers that read them, on the GPU.

dbsp_dense_block_lists must equal the oracle's lists bit for bit (every row, the causal
lists too, 16-byte and byte paths, rows of one to several 512-column chunks).
dbsp_block_sparse_attn_fwd_listed must give the same output as the kernel that scans the
mask rows (bit for bit: the same tiles in the same order), and so match the oracle
element by element; out-of-range counts or indices set DBSP_ERR_INVALID_ARG without a
fault.
"""

import numpy as np
import pytest
import torch

from load_balancing_gb300 import dbsp
from load_balancing_gb300 import path as P
from load_balancing_gb300 import workloads as W
from oracle import attention as A
from oracle import loads as OL
from parity import assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check_lists(mask_np, causal, mask=None):
    mask = torch.from_numpy(mask_np).to(DEV) if mask is None else mask
    counts, cols = dbsp.dbsp_dense_block_lists(mask, causal)
    assert dbsp.dbsp_device_status() == 0
    ref = OL.dense_block_lists(mask_np, causal)
    c = counts.cpu().numpy().reshape(-1)
    k = cols.cpu().numpy().view(np.uint16).reshape(len(ref), -1)
    np.testing.assert_array_equal(c, [len(x) for x in ref])
    for r, x in enumerate(ref):
        np.testing.assert_array_equal(k[r, :len(x)], x, err_msg=f"row {r}")


@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 3, 5, 7), (1, 2, 64, 64), (1, 1, 70, 1536),
                                   (1, 1, 33, 4112), (1, 2, 300, 300), (2, 1, 128, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("density", [0.0, 0.35, 1.0])
def test_dense_block_lists(built_library, cuda_device, shape, causal, density):
    if causal and shape[2] != shape[3]:
        pytest.skip("causal lists need a square mask")
    rng = np.random.default_rng(abs(hash((shape, causal, density))) % 2**32)
    vals = rng.integers(1, 256, shape).astype(np.uint8)  # any non-zero byte is dense
    _check_lists(np.where(rng.random(shape) < density, vals, 0).astype(np.uint8), causal)


@pytest.mark.parametrize("name", ["tiny", "llm", "video", "sharded"])
def test_dense_block_lists_of_workload_masks(built_library, cuda_device, name):
    w = W.WORKLOADS[name]
    _check_lists(W.make_mask(w), w.causal)


def test_dense_block_lists_unaligned_mask_takes_byte_path(built_library, cuda_device):
    rng = np.random.default_rng(5)
    mask_np = (rng.random((1, 2, 48, 48)) < 0.5).astype(np.uint8)
    buf = torch.zeros(mask_np.size + 1, dtype=torch.uint8, device=DEV)
    buf[1:] = torch.from_numpy(mask_np.reshape(-1)).to(DEV)
    _check_lists(mask_np, False, mask=buf[1:].view(mask_np.shape))


def _run_both(q, k, v, mask, block, causal, p, lists, **kw):
    out0, lse0 = P.attention(q, k, v, mask, block, causal, p, **kw)
    out1, lse1 = P.attention(q, k, v, mask, block, causal, p, lists=lists, **kw)
    torch.cuda.synchronize()
    assert dbsp.dbsp_device_status() == 0
    return out0, lse0, out1, lse1


@pytest.mark.parametrize("block,d", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_listed_attention_equals_scanning_kernel(built_library, cuda_device, block, d, causal):
    w = W.custom(f"lists_{block}_{d}_{int(causal)}", 2, 3, 5 * block, d, block, causal, 11, 111, "bernoulli",
                 p=0.45, numpy_qkv=True)
    mask_np = W.make_mask(w)
    mask_np[0, 0, 1, :] = 0  # an item with no dense block at all
    q, k, v = W.make_qkv(w, "cpu")
    mask = torch.from_numpy(mask_np).to(DEV)
    lists = P.dense_lists(mask, causal)
    for m in (1, 7, 200):
        p = P.plan(mask, m)
        out0, lse0, out1, lse1 = _run_both(q.to(DEV), k.to(DEV), v.to(DEV), mask, block, causal, p, lists)
        assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal)
    assert_rows_close(to64(out1), o_ref, to64(lse1), lse_ref, what=f"listed b{block} d{d} c{causal}")


def test_listed_attention_on_the_llm_workload(built_library, cuda_device):
    w = W.WORKLOADS["llm"]
    mask_np = W.make_mask(w)
    q, k, v = W.make_qkv(w, DEV)
    mask = torch.from_numpy(mask_np).to(DEV)
    p = P.plan(mask, P.default_workers() - 1)
    out0, lse0, out1, lse1 = _run_both(q, k, v, mask, w.block, w.causal, p, P.dense_lists(mask, w.causal))
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_listed_partial_mode_equals_scanning_kernel(built_library, cuda_device):
    w = W.custom("lists_partial", 1, 2, 6 * 128, 128, 128, True, 12, 112, "bernoulli", p=0.6, numpy_qkv=True)
    mask_np = W.make_mask(w)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w, "cpu"))
    mask = torch.from_numpy(mask_np).to(DEV)
    p = P.plan(mask, 5)
    lists = P.dense_lists(mask, True)
    res = []
    for use in (False, True):
        o = torch.full(q.shape, 7.0, dtype=torch.float32, device=DEV)
        mm = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
        ll = torch.empty_like(mm)
        fn = dbsp.dbsp_block_sparse_attn_fwd_listed if use else dbsp.dbsp_block_sparse_attn_fwd
        extra = (lists[0], lists[1]) if use else ()
        fn(q, k, v, mask, w.block, True, p.worker_offsets, p.worklist, 5, *extra, o_part=o, m_part=mm, l_part=ll)
        torch.cuda.synchronize()
        assert dbsp.dbsp_device_status() == 0
        res.append((o, mm, ll))
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_out_of_range_lists_are_reported(built_library, cuda_device):
    """A count above the row's limit, or an index at or past it, sets
    DBSP_ERR_INVALID_ARG; the launch ends normally and the next call is clean."""
    w = W.custom("lists_bad", 1, 2, 4 * 128, 128, 128, True, 13, 113, "bernoulli", p=0.6, numpy_qkv=True)
    mask_np = W.make_mask(w)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w, "cpu"))
    mask = torch.from_numpy(mask_np).to(DEV)
    p = P.plan(mask, 3)
    counts, cols = P.dense_lists(mask, True)
    bad_count = counts.clone()
    bad_count.view(-1)[1] = 3  # row qb = 1 of a causal mask admits 2 blocks
    P.attention(q, k, v, mask, w.block, True, p, lists=(bad_count, cols))
    assert dbsp.dbsp_device_status() == dbsp.DBSP_ERR_INVALID_ARG
    bad_cols = cols.clone()
    c = counts.view(-1).cpu().numpy()
    r = next(i for i in range(c.size) if c[i] >= 1 and i % w.nQ < w.nK - 1)
    bad_cols.view(-1, w.nK)[r, 0] = r % w.nQ + 1  # row qb admits blocks 0..qb
    P.attention(q, k, v, mask, w.block, True, p, lists=(counts, bad_cols))
    assert dbsp.dbsp_device_status() == dbsp.DBSP_ERR_INVALID_ARG
    out, lse = P.attention(q, k, v, mask, w.block, True, p, lists=(counts, cols))
    assert dbsp.dbsp_device_status() == dbsp.DBSP_OK
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, w.block, True)
    assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what="listed after the bad lists")


@pytest.mark.parametrize("kind", ["empty", "dense", "one_block"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block,d", [(128, 128), (64, 64)])
def test_listed_attention_degenerate_masks(built_library, cuda_device, kind, causal, block, d):
    """Degenerate masks through the listed producers: every item empty (the producers
    write O = 0 and LSE = -inf, and no MMA runs at all), every block dense, and a sequence
    of a single block (nQ = nK = 1). Bit-identical to the scanning kernel and, element by
    element, the oracle's."""
    nb = 1 if kind == "one_block" else 4
    B, H = 2, 3
    mask_np = (np.zeros if kind == "empty" else np.ones)((B, H, nb, nb), dtype=np.uint8)
    rng = np.random.default_rng(nb * 10 + int(causal) + block)
    shape = (B, H, nb * block, d)
    q, k, v = (torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16) for _ in range(3))
    mask = torch.from_numpy(mask_np).to(DEV)
    p = P.plan(mask, 5, causal=causal)
    out0, lse0, out1, lse1 = _run_both(q.to(DEV), k.to(DEV), v.to(DEV), mask, block, causal, p,
                                       P.dense_lists(mask, causal))
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal)
    assert_rows_close(to64(out1), o_ref, to64(lse1), lse_ref, what=f"listed {kind} c{causal} b{block}")
    if kind == "empty":
        assert not out1.any() and torch.isneginf(lse1).all()
