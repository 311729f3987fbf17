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


def _mask_loads(mask, row_loads, col_loads, head_loads, causal, stream):
    # causal: count only the blocks on or below the diagonal, the ones causal attention
    # computes (a mask need not be clipped to the diagonal beforehand)
    fn = dbsp.dbsp_block_mask_loads_causal if causal else dbsp.dbsp_block_mask_loads
    fn(mask, row_loads, col_loads, head_loads, stream=stream)


def plan(mask, n_workers, home=None, stay_bonus=0, out=None, stream=None, block_cost=1, item_cost=0, causal=False):
    """Loads of ``mask`` [B,H,nQ,nK] (uint8, CUDA) and the LPT worklist over (b,h,qb) items.

    The default plans on dense-block counts, as the pages do; ``block_cost`` and
    ``item_cost`` plan on ``row_load * block_cost + item_cost`` instead. With ``causal``
    the loads count only the blocks on or below the diagonal (pass it for causal
    attention unless the mask is already clipped to the diagonal).
    """
    B, H, nQ, nK = mask.shape
    p = out or alloc_plan(B, H, nQ, nK, n_workers, mask.device)
    _mask_loads(mask, p.row_loads, p.col_loads, p.head_loads, causal, stream)
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


def shard_masks_from_plan(mask, sp, stream=None):
    """uint8 [n_shards, B, H, nQ, nK]: ``mask`` restricted to each shard's KV blocks (one kernel)."""
    return dbsp.dbsp_shard_masks(mask, sp.shard_of, sp.n_shards, stream=stream)


def dense_lists(mask, causal=False, out=None, stream=None):
    """(counts int32 [B,H,nQ], cols int16 [B,H,nQ,nK]): every row's dense KV blocks, for
    ``attention(..., lists=...)``. With ``causal`` only the blocks on or below the diagonal."""
    counts, cols = (None, None) if out is None else out
    return dbsp.dbsp_dense_block_lists(mask, causal, counts, cols, stream=stream)


def attention(q, k, v, mask, block, causal, p, out=None, lse=None, scale=0.0, cta_timing=None,
              stream=None, lists=None):
    """Final-mode attention over plan ``p``; returns (out bf16, lse fp32). With ``lists``
    (from ``dense_lists`` of the same mask and causal flag) the kernel reads each item's
    dense blocks from them instead of scanning its mask row; the output is the same."""
    B, H, S, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if lists is not None:
        dbsp.dbsp_block_sparse_attn_fwd_listed(q, k, v, mask, block, causal, p.worker_offsets, p.worklist,
                                               p.n_workers, lists[0], lists[1], out=out, lse=lse, scale=scale,
                                               cta_timing=cta_timing, stream=stream)
    else:
        dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, block, causal, p.worker_offsets, p.worklist,
                                        p.n_workers, out=out, lse=lse, scale=scale, cta_timing=cta_timing,
                                        stream=stream)
    return out, lse


class PipelinedSteps:
    """Consecutive batches with the next batch's mask loads and plan hidden behind the
    current batch's attention.

    The attention kernel fills every SM it runs on (one persistent CTA per SM holds the
    whole register file), so a plan launched beside it would find no room. Here the
    attention runs on ``n_workers`` = SM count - 1 workers and the remaining SM takes the
    mask loads, the LPT plan and the dense-block lists of the next batch meanwhile, on a
    side stream, into the second of two plan buffers. ``prime`` plans the first batch;
    each ``step`` then runs one batch's attention on ``stream`` (reading its dense-block
    lists) and plans the next one beside it. The plan waits for everything enqueued on
    ``stream`` before the step (so it never overwrites a plan that an earlier attention
    still reads), and ``stream`` waits for the plan at the end of the step. Results are
    those of ``plan`` + ``attention`` on each batch. ``causal`` is the attention's: loads,
    plans and lists then count only the blocks on or below the diagonal, the ones it computes.
    """

    def __init__(self, B, H, nQ, nK, device, causal=False, n_workers=None, use_lists=True):
        self.n_workers = n_workers or max(1, default_workers(device) - 1)
        self.plans = [alloc_plan(B, H, nQ, nK, self.n_workers, device) for _ in range(2)]
        self.causal = bool(causal)
        self.lists = [(torch.empty((B, H, nQ), dtype=torch.int32, device=device),
                       torch.empty((B, H, nQ, nK), dtype=torch.int16, device=device)) for _ in range(2)] \
            if use_lists else None
        self._side = torch.cuda.Stream(device, priority=0)
        self._cur = 0

    def _plan(self, mask, i, stream):
        plan(mask, self.n_workers, out=self.plans[i], stream=stream, causal=self.causal)
        if self.lists is not None:
            dense_lists(mask, self.causal, out=self.lists[i], stream=stream)

    def prime(self, mask, stream=None):
        """Plans the first batch (on ``stream``)."""
        self._plan(mask, self._cur, stream or torch.cuda.current_stream(mask.device))

    def step(self, q, k, v, mask, block, causal, next_mask=None, out=None, lse=None, scale=0.0,
             cta_timing=None, stream=None, events=None):
        """Attention of the primed batch (``mask`` must be the mask it was planned from)
        beside the loads and plan of ``next_mask`` (none when it is None). ``events``, if
        given, are four CUDA events recorded at the step's start, the attention's end (both
        on ``stream``), the plan's end (side stream) and the step's end (``stream``).
        Returns (out, lse)."""
        if bool(causal) != self.causal:
            raise ValueError("causal differs from the one the batches are planned for")
        st = stream or torch.cuda.current_stream(q.device)
        e = events or [torch.cuda.Event() for _ in range(4)]
        e[0].record(st)
        B, H, S, d = q.shape
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
        attention(q, k, v, mask, block, causal, self.plans[self._cur], out=out, lse=lse, scale=scale,
                  cta_timing=cta_timing, stream=st,
                  lists=None if self.lists is None else self.lists[self._cur])
        e[1].record(st)
        self._side.wait_event(e[0])
        if next_mask is not None:
            self._plan(next_mask, 1 - self._cur, self._side)
        e[2].record(self._side)
        st.wait_event(e[2])
        e[3].record(st)
        self._cur = 1 - self._cur
        return out, lse


def attention_partial(q, k, v, mask, block, causal, p, o_part, m_part, l_part, scale=0.0, stream=None):
    """Partial-mode attention (one KV shard, expressed by ``mask``) into caller buffers."""
    dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, block, causal, p.worker_offsets, p.worklist,
                                    p.n_workers, o_part=o_part, m_part=m_part, l_part=l_part,
                                    scale=scale, stream=stream)


# Planning cost of one item, in dense blocks. Besides its dense blocks an item costs its
# Q tile, its mask-row scan and its epilogue. A least-squares fit of per-CTA busy time
# (cta_timing) to items and blocks per CTA, over the CTAs of three worklists on the
# LLM-heads workload, gives 2.88 us per item and 0.683 us per block: 4.2 blocks per item.
ITEM_COST_BLOCKS = 4
PLAN_BLOCK_COST_SCALE = 8  # block cost at which a measured item/block ratio is rounded
# A shard's partial pass leaves many items with few or no dense blocks; planned on dense
# blocks alone, every empty item lands on the same (least-loaded) worker. Shard passes
# therefore plan on row_load + ITEM_COST_BLOCKS. Whole-mask plans keep the pages' dense-
# block loads: there the item cost gained nothing measurable.
SHARD_BLOCK_COST = 1
SHARD_ITEM_COST = ITEM_COST_BLOCKS


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
        ps = plan(shard_masks[s], n_workers, stream=stream, block_cost=SHARD_BLOCK_COST, item_cost=SHARD_ITEM_COST,
                  causal=bool(causal))
        attention_partial(q, k, v, shard_masks[s], block, causal, ps, o_parts[s], m_parts[s], l_parts[s],
                          scale=scale, stream=stream)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    dbsp.dbsp_merge_partials(o_parts.view(n_sh, -1, d), m_parts.view(n_sh, -1), l_parts.view(n_sh, -1),
                             out.view(-1, d), lse.view(-1), stream=stream)
    return out, lse, (o_parts, m_parts, l_parts)


@dataclass
class SplitPlan:
    """Heavy items split along their KV blocks, and the LPT worklist over the units."""
    row_loads: torch.Tensor      # int32 [B, H, nQ]
    col_loads: torch.Tensor      # int32 [B, H, nK]
    head_loads: torch.Tensor     # int32 [B, H]
    unit_item: torch.Tensor      # int32 [n_items * max_pieces]
    unit_pk: torch.Tensor        # int32: j | k << 16
    unit_slot: torch.Tensor      # int32: partial slot of a piece, -1 for a whole item
    unit_load: torch.Tensor      # int32: dense blocks of the unit
    split_item: torch.Tensor     # int32 [n_items]
    split_off: torch.Tensor      # int32 [n_items + 1]
    counts: torch.Tensor         # int32 [5]: units, whole items, split items, slots, T
    worker_of: torch.Tensor      # int32 [n_items * max_pieces], per unit
    worker_offsets: torch.Tensor  # int32 [n_workers + 1]
    worklist: torch.Tensor       # int32: unit ids grouped by worker
    worker_loads: torch.Tensor   # int64 [n_workers]
    o_piece: torch.Tensor        # fp32 [max_slots, block, d]
    m_piece: torch.Tensor        # fp32 [max_slots, block]
    l_piece: torch.Tensor        # fp32 [max_slots, block]
    n_workers: int
    max_pieces: int
    max_slots: int


def alloc_split_plan(B, H, nQ, nK, n_workers, block, d, max_pieces, max_slots, device):
    i32 = dict(dtype=torch.int32, device=device)
    n = B * H * nQ
    cap = n * max_pieces
    return SplitPlan(torch.empty((B, H, nQ), **i32), torch.empty((B, H, nK), **i32), torch.empty((B, H), **i32),
                     torch.empty(cap, **i32), torch.empty(cap, **i32), torch.empty(cap, **i32),
                     torch.empty(cap, **i32), torch.empty(n, **i32), torch.empty(n + 1, **i32),
                     torch.zeros(5, **i32), torch.empty(cap, **i32), torch.empty(n_workers + 1, **i32),
                     torch.empty(cap, **i32), torch.empty(n_workers, dtype=torch.int64, device=device),
                     torch.empty((max(max_slots, 1), block, d), dtype=torch.float32, device=device),
                     torch.empty((max(max_slots, 1), block), dtype=torch.float32, device=device),
                     torch.empty((max(max_slots, 1), block), dtype=torch.float32, device=device),
                     n_workers, max_pieces, max_slots)


def plan_split(mask, n_workers, block, d, max_piece_load=0, max_pieces=4, max_slots=None, block_cost=1,
               item_cost=0, out=None, stream=None, causal=False):
    """Mask loads -> split plan -> LPT over the units, all on the device (no host sync).

    ``max_piece_load`` T <= 0 selects half the mean load per worker. With that choice a
    split item of load L > T makes at most ceil(L / T) < 2 L / T pieces, so all pieces
    together number fewer than 2 total / T <= 4 n_workers: the default ``max_slots``.
    With a fixed T the default is the worst case n_items * max_pieces; the piece buffers
    take max_slots * block * (d + 2) * 4 bytes, so pass a smaller ``max_slots`` for large
    problems (a plan that needs more pieces reports DBSP_ERR_UNSUPPORTED on the device).
    ``causal`` counts only the blocks on or below the diagonal, as in ``plan``.
    """
    B, H, nQ, nK = mask.shape
    n = B * H * nQ
    if max_slots is None:
        max_slots = n * max_pieces if max_piece_load > 0 else min(n * max_pieces, 4 * n_workers)
    sp = out or alloc_split_plan(B, H, nQ, nK, n_workers, block, d, max_pieces, max_slots, mask.device)
    _mask_loads(mask, sp.row_loads, sp.col_loads, sp.head_loads, causal, stream)
    dbsp.dbsp_split_plan(sp.row_loads.view(-1), n_workers, max_piece_load, max_pieces, sp.max_slots, sp.unit_item,
                         sp.unit_pk, sp.unit_slot, sp.unit_load, sp.split_item, sp.split_off, sp.counts,
                         stream=stream)
    dbsp.dbsp_plan_lpt_cost_n(sp.unit_load, sp.counts[:1], n_workers, block_cost, item_cost, sp.worker_of,
                              sp.worker_offsets, sp.worklist, sp.worker_loads, stream=stream)
    return sp


def attention_split(q, k, v, mask, block, causal, sp, out=None, lse=None, scale=0.0, cta_timing=None,
                    stream=None):
    """Attention over a split plan: whole items written directly, pieces merged; returns (out, lse)."""
    B, H, S, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    dbsp.dbsp_block_sparse_attn_fwd_units(q, k, v, mask, block, causal, sp.worker_offsets, sp.worklist,
                                          sp.n_workers, sp.unit_item, sp.unit_pk, sp.unit_slot, out, lse,
                                          sp.o_piece, sp.m_piece, sp.l_piece, scale=scale, cta_timing=cta_timing,
                                          stream=stream)
    dbsp.dbsp_merge_pieces(sp.o_piece, sp.m_piece, sp.l_piece, sp.split_item, sp.split_off, sp.counts, out, lse,
                           block=block, stream=stream)
    return out, lse
