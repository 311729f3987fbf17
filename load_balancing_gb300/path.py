"""The whole hot path as one call: mask loads -> LPT plan -> attention (-> merge).

This module only allocates output tensors with torch and chains the C-ABI calls of
``dbsp``; every step runs in the library's kernels.
"""

from dataclasses import dataclass

import torch

from . import dbsp


@dataclass
class Plan:
    row_loads: torch.Tensor
    col_loads: torch.Tensor
    head_loads: torch.Tensor
    worker_of: torch.Tensor
    worker_offsets: torch.Tensor
    worklist: torch.Tensor
    worker_loads: torch.Tensor
    n_workers: int


def default_workers(device=None):
    """One persistent worker per SM of the device."""
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


def alloc_plan(B, H, nQ, nK, n_workers, device):
    i32 = dict(dtype=torch.int32, device=device)
    n = B * H * nQ
    return Plan(torch.empty((B, H, nQ), **i32), torch.empty((B, H, nK), **i32), torch.empty((B, H), **i32),
                torch.empty(n, **i32), torch.empty(n_workers + 1, **i32), torch.empty(n, **i32),
                torch.empty(n_workers, dtype=torch.int64, device=device), n_workers)


def plan(mask, n_workers, home=None, stay_bonus=0, out=None, stream=None, block_cost=1, item_cost=0):
    """Loads of ``mask`` [B,H,nQ,nK] (uint8, CUDA) and the LPT worklist over (b,h,qb) items.

    The default plans on dense-block counts, as the pages do; ``block_cost`` and
    ``item_cost`` plan on ``row_load * block_cost + item_cost`` instead.
    """
    B, H, nQ, nK = mask.shape
    p = out or alloc_plan(B, H, nQ, nK, n_workers, mask.device)
    dbsp.dbsp_block_mask_loads(mask, p.row_loads, p.col_loads, p.head_loads, stream=stream)
    if block_cost == 1 and item_cost == 0:
        dbsp.dbsp_plan_lpt(p.row_loads.view(-1), n_workers, p.worker_of, p.worker_offsets, p.worklist,
                           p.worker_loads, home=home, stay_bonus=stay_bonus, stream=stream)
    else:
        dbsp.dbsp_plan_lpt_cost(p.row_loads.view(-1), n_workers, block_cost, item_cost, p.worker_of,
                                p.worker_offsets, p.worklist, p.worker_loads, home=home, stay_bonus=stay_bonus,
                                stream=stream)
    return p


@dataclass
class ShardPlan:
    kv_loads: torch.Tensor       # int32 [nK]: dense blocks of each KV block over all heads
    shard_of: torch.Tensor       # int32 [nK]: shard of each KV block
    shard_offsets: torch.Tensor  # int32 [n_shards + 1]: CSR over shards
    shard_blocks: torch.Tensor   # int32 [nK]: KV blocks grouped by shard
    shard_loads: torch.Tensor    # int64 [n_shards]: dense blocks per shard
    n_shards: int


def plan_kv_shards(mask, n_shards, stream=None):
    """LPT assignment of KV blocks to ``n_shards`` sequence shards (shared by every head).

    db-SP blog, scenario 2: KV blocks are balanced by their column loads, here summed
    over all heads because every head is split the same way. Mask loads, the sum over
    heads and the LPT all run in the library's kernels.
    """
    B, H, nQ, nK = mask.shape
    dev = mask.device
    i32 = dict(dtype=torch.int32, device=dev)
    row = torch.empty((B, H, nQ), **i32)
    col = torch.empty((B, H, nK), **i32)
    dbsp.dbsp_block_mask_loads(mask, row, col, None, stream=stream)
    kv = torch.empty(nK, **i32)
    dbsp.dbsp_kv_block_loads(col, kv, stream=stream)
    sp = ShardPlan(kv, torch.empty(nK, **i32), torch.empty(n_shards + 1, **i32), torch.empty(nK, **i32),
                   torch.empty(n_shards, dtype=torch.int64, device=dev), n_shards)
    dbsp.dbsp_plan_lpt(kv, n_shards, sp.shard_of, sp.shard_offsets, sp.shard_blocks, sp.shard_loads,
                       stream=stream)
    return sp


def shard_masks_from_plan(mask, sp):
    """uint8 [n_shards, B, H, nQ, nK]: ``mask`` restricted to each shard's KV blocks."""
    owned = sp.shard_of.view(1, -1) == torch.arange(sp.n_shards, device=mask.device, dtype=torch.int32).view(-1, 1)
    return mask.unsqueeze(0) * owned.to(torch.uint8).view(sp.n_shards, 1, 1, 1, -1)


def attention(q, k, v, mask, block, causal, p, out=None, lse=None, scale=0.0, cta_timing=None,
              stream=None):
    """Final-mode attention over plan ``p``; returns (out bf16, lse fp32)."""
    B, H, S, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, block, causal, p.worker_offsets, p.worklist,
                                    p.n_workers, out=out, lse=lse, scale=scale, cta_timing=cta_timing,
                                    stream=stream)
    return out, lse


def attention_partial(q, k, v, mask, block, causal, p, o_part, m_part, l_part, scale=0.0, stream=None):
    """Partial-mode attention (one KV shard, expressed by ``mask``) into caller buffers."""
    dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, block, causal, p.worker_offsets, p.worklist,
                                    p.n_workers, o_part=o_part, m_part=m_part, l_part=l_part,
                                    scale=scale, stream=stream)


# Planning loads of a shard's partial pass: a dense block counts 8, an item 1 (an item
# without dense blocks costs its output rows, about an eighth of a block's MMA time).
SHARD_BLOCK_COST = 8
SHARD_ITEM_COST = 1


def sharded_attention(q, k, v, shard_masks, block, causal, n_workers, scale=0.0, stream=None):
    """Per-shard partials (each shard planned on its own loads) merged into (out, lse)."""
    n_sh = shard_masks.shape[0]
    B, H, S, d = q.shape
    dev = q.device
    o_parts = torch.empty((n_sh, B, H, S, d), dtype=torch.float32, device=dev)
    m_parts = torch.empty((n_sh, B, H, S), dtype=torch.float32, device=dev)
    l_parts = torch.empty((n_sh, B, H, S), dtype=torch.float32, device=dev)
    for s in range(n_sh):
        # a shard leaves many items without dense blocks: an item cost spreads them
        ps = plan(shard_masks[s], n_workers, stream=stream, block_cost=SHARD_BLOCK_COST, item_cost=SHARD_ITEM_COST)
        attention_partial(q, k, v, shard_masks[s], block, causal, ps, o_parts[s], m_parts[s], l_parts[s],
                          scale=scale, stream=stream)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    dbsp.dbsp_merge_partials(o_parts.view(n_sh, -1, d), m_parts.view(n_sh, -1), l_parts.view(n_sh, -1),
                             out.view(-1, d), lse.view(-1), stream=stream)
    return out, lse, (o_parts, m_parts, l_parts)
