"""Heavy items split along their KV blocks, on the GPU: the unit table and the LPT over
units bit-exact against the oracle, and split attention (pieces merged) against the
fp64 oracle's unsplit attention."""

import numpy as np
import pytest
import torch

from load_balancing_gb300 import dbsp
from load_balancing_gb300 import path as P
from load_balancing_gb300 import workloads as W
from oracle import attention as A
from oracle import lpt as OP
from oracle import split as OS
from parity import assert_rows_close, oracle_item, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _split_table(loads, m, t, p, max_slots=None):
    n = len(loads)
    cap = max(1, n * p)
    i32 = dict(dtype=torch.int32, device=DEV)
    lt = torch.as_tensor(np.asarray(loads, dtype=np.int32)).to(DEV)
    out = {k: torch.full((cap,), -7, **i32) for k in ("unit_item", "unit_pk", "unit_slot", "unit_load")}
    out["split_item"] = torch.full((max(1, n),), -7, **i32)
    out["split_off"] = torch.full((n + 1,), -7, **i32)
    out["counts"] = torch.full((5,), -7, **i32)
    dbsp.dbsp_split_plan(lt, m, t, p, cap if max_slots is None else max_slots, out["unit_item"], out["unit_pk"],
                         out["unit_slot"], out["unit_load"], out["split_item"], out["split_off"], out["counts"])
    status = dbsp.dbsp_device_status()
    return {k: v.cpu().numpy() for k, v in out.items()}, status


@pytest.mark.parametrize("t,p", [(1, 4), (5, 2), (50, 7), (0, 4), (0, 1), (10**6, 3)])
def test_split_table_bit_exact(built_library, cuda_device, t, p):
    rng = np.random.default_rng(t + 13 * p)
    for n, hi, m in ((0, 1, 4), (1, 9, 1), (37, 40, 5), (3000, 130, 152), (20000, 64, 152)):
        loads = rng.integers(0, hi, n)
        got, status = _split_table(loads, m, t, p)
        assert status == 0
        t_eff = t if t > 0 else OS.auto_piece_load(int(loads.sum()), m)
        ref = OS.split_plan(loads, t_eff, p)
        U, n_whole, n_split, n_slots = ref["counts"]
        assert got["counts"].tolist() == [U, n_whole, n_split, n_slots, t_eff]
        for key in ("unit_item", "unit_pk", "unit_slot", "unit_load"):
            np.testing.assert_array_equal(got[key][:U], ref[key], err_msg=key)
        np.testing.assert_array_equal(got["split_item"][:n_split], ref["split_item"])
        np.testing.assert_array_equal(got["split_off"][:n_split + 1], ref["split_off"])


def test_split_table_errors(built_library, cuda_device):
    got, status = _split_table([3, -1, 2], 2, 1, 4)
    assert status == dbsp.DBSP_ERR_INVALID_ARG and got["counts"][:4].tolist() == [0, 0, 0, 0]
    got, status = _split_table([30, 30, 30], 2, 10, 4, max_slots=5)  # 9 pieces needed
    assert status == dbsp.DBSP_ERR_UNSUPPORTED and got["counts"][:4].tolist() == [0, 0, 0, 0]


def test_lpt_over_units_with_device_count(built_library, cuda_device):
    rng = np.random.default_rng(5)
    for n, hi, m, t, p in ((2000, 128, 152, 0, 4), (300, 64, 7, 9, 3), (5, 3, 4, 1, 2)):
        loads = rng.integers(0, hi, n)
        mask = torch.zeros((1, 1, n, 1), dtype=torch.uint8, device=DEV)  # loads come from `loads` below
        cap = n * p
        i32 = dict(dtype=torch.int32, device=DEV)
        lt = torch.as_tensor(loads.astype(np.int32)).to(DEV)
        tab = [torch.empty(cap, **i32) for _ in range(4)]
        si, so, cnt = torch.empty(n, **i32), torch.empty(n + 1, **i32), torch.zeros(5, **i32)
        dbsp.dbsp_split_plan(lt, m, t, p, cap, *tab, si, so, cnt)
        wo, off, wl = torch.empty(cap, **i32), torch.empty(m + 1, **i32), torch.empty(cap, **i32)
        wload = torch.empty(m, dtype=torch.int64, device=DEV)
        dbsp.dbsp_plan_lpt_cost_n(tab[3], cnt[:1], m, 1, 0, wo, off, wl, wload)
        assert dbsp.dbsp_device_status() == 0
        t_eff = t if t > 0 else OS.auto_piece_load(int(loads.sum()), m)
        ref_tab = OS.split_plan(loads, t_eff, p)
        U = ref_tab["counts"][0]
        ref = OP.lpt_plan(ref_tab["unit_load"], m)
        np.testing.assert_array_equal(wo.cpu().numpy()[:U], ref["worker_of"])
        np.testing.assert_array_equal(off.cpu().numpy(), ref["offsets"])
        np.testing.assert_array_equal(wl.cpu().numpy()[:U], ref["worklist"])
        np.testing.assert_array_equal(wload.cpu().numpy(), ref["worker_loads"])
        del mask


def _small(block, d, causal, B=2, H=3, nblocks=6, seed=3, density=0.6):
    w = W.custom(f"split_{block}_{d}_{int(causal)}", B, H, nblocks * block, d, block, causal, seed, seed + 100,
                 "bernoulli", p=density, numpy_qkv=True)
    mask_np = W.make_mask(w)
    mask_np[0, 0, 1, :] = 0  # an item with no dense block
    return w, mask_np


@pytest.mark.parametrize("block,d", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("t,p,n_workers", [(1, 8, 7), (2, 3, 200), (0, 4, 3)])
def test_split_attention_small(built_library, cuda_device, block, d, causal, t, p, n_workers):
    w, mask_np = _small(block, d, causal)
    q, k, v = W.make_qkv(w, "cpu")
    mask = torch.from_numpy(mask_np).to(DEV)
    sp = P.plan_split(mask, n_workers, block, d, max_piece_load=t, max_pieces=p)
    out, lse = P.attention_split(q.to(DEV), k.to(DEV), v.to(DEV), mask, block, causal, sp)
    assert dbsp.dbsp_device_status() == 0
    counts = sp.counts.cpu().numpy()
    if t == 1:
        assert counts[2] > 0  # items were split
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal)
    assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what=f"split b{block} d{d} c{causal} t{t} p{p}")


def test_split_without_splits_equals_plain_path(built_library, cuda_device):
    w, mask_np = _small(128, 128, True)
    q, k, v = (x.to(DEV) for x in W.make_qkv(w, "cpu"))
    mask = torch.from_numpy(mask_np).to(DEV)
    sp = P.plan_split(mask, 5, 128, 128, max_piece_load=10**6, max_pieces=4)
    out_s, lse_s = P.attention_split(q, k, v, mask, 128, True, sp)
    p = P.plan(mask, 5)
    out_p, lse_p = P.attention(q, k, v, mask, 128, True, p)
    assert dbsp.dbsp_device_status() == 0
    assert sp.counts.cpu().numpy()[2] == 0
    assert torch.equal(out_s, out_p) and torch.equal(lse_s, lse_p)


def test_hand_made_units_with_empty_pieces(built_library, cuda_device):
    """More pieces than dense blocks leaves pieces empty ((m, l) = (-inf, 0), O never
    read); the merge still gives the unsplit result."""
    block, d, causal = 128, 128, True
    w, mask_np = _small(block, d, causal, B=1, H=1, nblocks=4)
    q, k, v = W.make_qkv(w, "cpu")
    mask = torch.from_numpy(mask_np).to(DEV)
    loads = (mask_np != 0).sum(-1).reshape(-1)
    items = list(range(loads.size))
    unit_item, unit_pk, unit_slot, split_item, split_off = [], [], [], [], [0]
    for i in items:  # every item in loads + 2 pieces
        kk = int(loads[i]) + 2
        split_item.append(i)
        for j in range(kk):
            unit_item.append(i)
            unit_pk.append(j | (kk << 16))
            unit_slot.append(split_off[-1] + j)
        split_off.append(split_off[-1] + kk)
    n_units = len(unit_item)
    i32 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32)).to(DEV)
    m = 3
    wl = i32(list(range(n_units)))
    off = i32([(n_units * r) // m for r in range(m + 1)])
    slots = split_off[-1]
    o_piece = torch.full((slots, block, d), float("nan"), dtype=torch.float32, device=DEV)
    m_piece = torch.empty((slots, block), dtype=torch.float32, device=DEV)
    l_piece = torch.empty((slots, block), dtype=torch.float32, device=DEV)
    out = torch.empty((1, 1, w.S, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((1, 1, w.S), dtype=torch.float32, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    dbsp.dbsp_block_sparse_attn_fwd_units(qd, kd, vd, mask, block, causal, off, wl, m, i32(unit_item), i32(unit_pk),
                                          i32(unit_slot), out, lse, o_piece, m_piece, l_piece)
    counts = i32([n_units, 0, len(split_item), slots, 1])
    dbsp.dbsp_merge_pieces(o_piece, m_piece, l_piece, i32(split_item), i32(split_off), counts, out, lse,
                           block=block)
    assert dbsp.dbsp_device_status() == 0
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal)
    assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what="hand-made units")
    # an out-of-range slot is reported and its unit skipped
    bad_slot = list(unit_slot)
    bad_slot[0] = slots + 5
    dbsp.dbsp_block_sparse_attn_fwd_units(qd, kd, vd, mask, block, causal, off, wl, m, i32(unit_item),
                                          i32(unit_pk), i32(bad_slot), out, lse, o_piece, m_piece, l_piece)
    assert dbsp.dbsp_device_status() == dbsp.DBSP_ERR_INVALID_ARG
    # slots beyond the piece buffers' capacity (or beyond counts[3]) are reported, not read
    bad_off = list(split_off)
    bad_off[-1] = slots + 3
    bad_counts = i32([n_units, 0, len(split_item), slots + 3, 1])
    dbsp.dbsp_merge_pieces(o_piece, m_piece, l_piece, i32(split_item), i32(bad_off), bad_counts, out, lse,
                           block=block)
    assert dbsp.dbsp_device_status() == dbsp.DBSP_ERR_INVALID_ARG
    dbsp.dbsp_merge_pieces(o_piece, m_piece, l_piece, i32(split_item), i32(bad_off), counts, out, lse, block=block)
    assert dbsp.dbsp_device_status() == dbsp.DBSP_ERR_INVALID_ARG


def test_long_causal_heads_sampled(built_library, cuda_device):
    """Two fully causal heads of 16,384 tokens on one worker per SM: the heavy rows are
    split (automatic piece load); sampled items, heaviest included, against the oracle."""
    w = W.custom("long_causal", 1, 2, 16384, 128, 128, True, 6, 106, "causal_full")
    mask_np = W.make_mask(w)
    q, k, v = W.make_qkv(w, DEV)
    mask = torch.from_numpy(mask_np).to(DEV)
    m = P.default_workers()
    sp = P.plan_split(mask, m, w.block, w.d)
    out, lse = P.attention_split(q, k, v, mask, w.block, w.causal, sp)
    assert dbsp.dbsp_device_status() == 0
    counts = sp.counts.cpu().numpy()
    assert counts[2] > 0 and counts[4] == OS.auto_piece_load(int(mask_np.sum()), m)
    nq = w.nQ
    for item in (0, 1, nq // 2, nq - 2, nq - 1, nq + 3, 2 * nq - 1):
        b, h, qb = 0, item // nq, item % nq
        r = oracle_item(q, k, v, mask_np, b, h, qb, w.block, w.causal)
        rows = slice(qb * w.block, (qb + 1) * w.block)
        assert_rows_close(to64(out[b, h, rows]), r["o"], to64(lse[b, h, rows]), r["lse"], what=f"item {item}")
