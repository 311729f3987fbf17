"""dbsp_block_mask_loads on the GPU: bit-exact against the oracle."""

import numpy as np
import pytest
import torch

from load_balancing_gb300 import workloads as W
from oracle import loads as OL

pytestmark = pytest.mark.gpu


def _run(mask_np, with_head=True):
    from load_balancing_gb300 import dbsp

    dev = torch.device("cuda:0")
    B, H, nQ, nK = mask_np.shape
    mask = torch.from_numpy(mask_np).to(dev)
    row = torch.full((B, H, nQ), -7, dtype=torch.int32, device=dev)
    col = torch.full((B, H, nK), -7, dtype=torch.int32, device=dev)
    head = torch.full((B, H), -7, dtype=torch.int32, device=dev) if with_head else None
    dbsp.dbsp_block_mask_loads(mask, row, col, head)
    assert dbsp.dbsp_device_status() == 0
    return row.cpu().numpy(), col.cpu().numpy(), None if head is None else head.cpu().numpy()


@pytest.mark.parametrize("name", W.ORDER)
def test_workload_masks(built_library, cuda_device, name):
    mask = W.make_mask(W.WORKLOADS[name])
    row, col, head = _run(mask)
    r, c, h = OL.block_mask_loads(mask)
    np.testing.assert_array_equal(row, r)
    np.testing.assert_array_equal(col, c)
    np.testing.assert_array_equal(head, h)


@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 3, 5, 7), (1, 2, 16, 48), (1, 1, 300, 16),
                                   (2, 2, 1000, 33), (1, 1, 4, 16384), (3, 1, 2048, 64), (1, 5, 9, 8),
                                   # rows streamed through shared memory: a ragged last stage, 96 units
                                   # per row (a quarter of the threads idle), 256 units per row, and
                                   # bands long enough that per-thread byte counters are flushed
                                   (1, 2, 37, 4096), (1, 1, 70, 1536), (1, 1, 8192, 1024),
                                   (1, 1, 2048, 4096), (1, 1, 131072, 16), (1, 1, 3, 4112),
                                   # 8 bands of 188 rows per head, 6 stages of 32 rows each, the
                                   # last band shorter and ragged
                                   (2, 2, 1500, 512),
                                   # several 1 MB heads of 8 ranks; rows of 65 units whose stages
                                   # end ragged (15 rows per stage)
                                   (2, 3, 1024, 1024), (1, 5, 1000, 1040)])
@pytest.mark.parametrize("density", [0.0, 0.3, 1.0])
def test_random_masks(built_library, cuda_device, shape, density):
    rng = np.random.default_rng(hash((shape, density)) % 2**32)
    vals = rng.integers(1, 256, shape).astype(np.uint8)  # any non-zero byte is dense
    mask = np.where(rng.random(shape) < density, vals, 0).astype(np.uint8)
    row, col, head = _run(mask, with_head=shape[0] != 3)
    r, c, h = OL.block_mask_loads(mask)
    np.testing.assert_array_equal(row, r)
    np.testing.assert_array_equal(col, c)
    if head is not None:
        np.testing.assert_array_equal(head, h)


def test_unaligned_mask_pointer_takes_byte_path(built_library, cuda_device):
    from load_balancing_gb300 import dbsp

    rng = np.random.default_rng(3)
    mask_np = (rng.random((1, 2, 64, 64)) < 0.5).astype(np.uint8)
    buf = torch.zeros(mask_np.size + 1, dtype=torch.uint8, device="cuda:0")
    buf[1:] = torch.from_numpy(mask_np.reshape(-1)).cuda()
    mask = buf[1:].view(1, 2, 64, 64)  # 1-byte offset: the 16-byte vector path is not allowed
    row = torch.empty((1, 2, 64), dtype=torch.int32, device="cuda:0")
    col = torch.empty_like(row)
    dbsp.dbsp_block_mask_loads(mask, row, col)
    r, c, _ = OL.block_mask_loads(mask_np)
    np.testing.assert_array_equal(row.cpu().numpy(), r)
    np.testing.assert_array_equal(col.cpu().numpy(), c)


@pytest.mark.parametrize("name", W.ORDER)
def test_kv_block_loads(built_library, cuda_device, name):
    from load_balancing_gb300 import dbsp

    mask_np = W.make_mask(W.WORKLOADS[name])
    B, H, nQ, nK = mask_np.shape
    row = torch.empty((B, H, nQ), dtype=torch.int32, device="cuda:0")
    col = torch.empty((B, H, nK), dtype=torch.int32, device="cuda:0")
    dbsp.dbsp_block_mask_loads(torch.from_numpy(mask_np).cuda(), row, col)
    kv = torch.full((nK,), -3, dtype=torch.int32, device="cuda:0")
    dbsp.dbsp_kv_block_loads(col, kv)
    assert dbsp.dbsp_device_status() == 0
    np.testing.assert_array_equal(kv.cpu().numpy(), OL.kv_block_loads(mask_np))


@pytest.mark.parametrize("shape", [(1, 2, 16, 16), (2, 3, 64, 64), (1, 1, 1024, 1024), (1, 2, 300, 300),
                                   (1, 1, 4112, 4112), (1, 1, 33, 33), (1, 2, 2048, 2048)])
def test_causal_loads_count_only_blocks_on_or_below_the_diagonal(built_library, cuda_device, shape):
    """dbsp_block_mask_loads_causal on masks that are NOT clipped to the diagonal equals
    the oracle's loads of the same masks clipped to it (6D notes §2.3: the blocks after
    a Q block's diagonal are skipped): streamed rows (16 and 64 KV blocks, 1024 with the
    unrolled path, 2048 over 8 ranks of 256 rows), byte rows (300, 33) and 16-byte
    register rows (4112)."""
    from load_balancing_gb300 import dbsp

    rng = np.random.default_rng(sum(shape))
    vals = rng.integers(1, 256, shape).astype(np.uint8)
    mask_np = np.where(rng.random(shape) < 0.5, vals, 0).astype(np.uint8)
    dev = torch.device("cuda:0")
    B, H, nQ, nK = shape
    mask = torch.from_numpy(mask_np).to(dev)
    row = torch.full((B, H, nQ), -7, dtype=torch.int32, device=dev)
    col = torch.full((B, H, nK), -7, dtype=torch.int32, device=dev)
    head = torch.full((B, H), -7, dtype=torch.int32, device=dev)
    dbsp.dbsp_block_mask_loads_causal(mask, row, col, head)
    assert dbsp.dbsp_device_status() == 0
    clipped = np.where(np.tril(np.ones((nQ, nK), dtype=bool)), mask_np, 0).astype(np.uint8)
    r, c, h = OL.block_mask_loads(clipped)
    np.testing.assert_array_equal(row.cpu().numpy(), r)
    np.testing.assert_array_equal(col.cpu().numpy(), c)
    np.testing.assert_array_equal(head.cpu().numpy(), h)


@pytest.mark.parametrize("shape,n_shards", [((1, 2, 16, 64), 8), ((2, 1, 7, 48), 3), ((1, 1, 5, 33), 4),
                                            ((1, 3, 256, 256), 8)])
def test_shard_masks(built_library, cuda_device, shape, n_shards):
    """dbsp_shard_masks: shard s keeps exactly the columns j with shard_of[j] == s (16-byte
    and byte paths); a shard index out of range clears its column and is reported."""
    from load_balancing_gb300 import dbsp

    rng = np.random.default_rng(sum(shape) + n_shards)
    mask_np = rng.integers(0, 3, shape).astype(np.uint8)
    shard_np = rng.integers(0, n_shards, shape[-1]).astype(np.int32)
    dev = torch.device("cuda:0")
    out = dbsp.dbsp_shard_masks(torch.from_numpy(mask_np).to(dev), torch.from_numpy(shard_np).to(dev), n_shards)
    assert dbsp.dbsp_device_status() == 0
    ref = np.stack([np.where(shard_np == s, mask_np, 0) for s in range(n_shards)]).astype(np.uint8)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    bad = shard_np.copy()
    bad[1] = n_shards  # outside [0, n_shards)
    out = dbsp.dbsp_shard_masks(torch.from_numpy(mask_np).to(dev), torch.from_numpy(bad).to(dev), n_shards)
    assert dbsp.dbsp_device_status() == dbsp.DBSP_ERR_INVALID_ARG
    ref = np.stack([np.where(bad == s, mask_np, 0) for s in range(n_shards)]).astype(np.uint8)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
