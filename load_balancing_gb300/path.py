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


def plan(mask, n_workers, home=None, stay_bonus=0, out=None, stream=None):
    """Loads of ``mask`` [B,H,nQ,nK] (uint8, CUDA) and the LPT worklist over (b,h,qb) items."""
    B, H, nQ, nK = mask.shape
    p = out or alloc_plan(B, H, nQ, nK, n_workers, mask.device)
    dbsp.dbsp_block_mask_loads(mask, p.row_loads, p.col_loads, p.head_loads, stream=stream)
    dbsp.dbsp_plan_lpt(p.row_loads.view(-1), n_workers, p.worker_of, p.worker_offsets, p.worklist,
                       p.worker_loads, home=home, stay_bonus=stay_bonus, stream=stream)
    return p


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


def sharded_attention(q, k, v, shard_masks, block, causal, n_workers, scale=0.0, stream=None):
    """Per-shard partials (each shard planned on its own loads) merged into (out, lse)."""
    n_sh = shard_masks.shape[0]
    B, H, S, d = q.shape
    dev = q.device
    o_parts = torch.empty((n_sh, B, H, S, d), dtype=torch.float32, device=dev)
    m_parts = torch.empty((n_sh, B, H, S), dtype=torch.float32, device=dev)
    l_parts = torch.empty((n_sh, B, H, S), dtype=torch.float32, device=dev)
    for s in range(n_sh):
        ps = plan(shard_masks[s], n_workers, stream=stream)
        attention_partial(q, k, v, shard_masks[s], block, causal, ps, o_parts[s], m_parts[s], l_parts[s],
                          scale=scale, stream=stream)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    dbsp.dbsp_merge_partials(o_parts.view(n_sh, -1, d), m_parts.view(n_sh, -1), l_parts.view(n_sh, -1),
                             out.view(-1, d), lse.view(-1), stream=stream)
    return out, lse, (o_parts, m_parts, l_parts)
