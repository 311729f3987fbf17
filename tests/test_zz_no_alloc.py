"""The allocation-free split attention entry point, on the GPU, through the C ABI.

dbsp_block_sparse_attn_fwd_split_noalloc is for callers that cannot allocate device
memory where they run attention: a serving runtime whose memory pool was reserved up
front and must not grow, or a host thread that may not call cudaMalloc because that
call synchronises the device. It does what dbsp_block_sparse_attn_fwd_units followed
by dbsp_merge_pieces do, but keeps the pieces in the library's own static device
scratch instead of buffers the caller allocates.

Two calls in a row, each on a different split plan (so the second call's pieces land
in scratch the first call left behind), are compared with the existing entry points
run on caller-allocated piece buffers, at the tolerances of every attention parity
test: max |dO| <= 2e-2, mean |dO| <= 2e-3, |dLSE| <= 1e-3. A plan whose pieces would
not fit the scratch is refused before the GPU is touched.

This file sorts last so that a run stopping at the first failure has run every other
test before it.
"""

import pytest
import torch

from load_balancing_gb300 import dbsp
from load_balancing_gb300 import path as P
from load_balancing_gb300 import workloads as W
from parity import assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _problem(block=128, d=128, causal=True, B=2, H=3, nblocks=6, seed=3):
    w = W.custom(f"noalloc_{block}_{d}_{int(causal)}", B, H, nblocks * block, d, block, causal, seed, seed + 100,
                 "bernoulli", p=0.6, numpy_qkv=True)
    mask_np = W.make_mask(w)
    mask_np[0, 0, 1, :] = 0  # an item with no dense block
    q, k, v = (x.to(DEV) for x in W.make_qkv(w, "cpu"))
    return w, torch.from_numpy(mask_np).to(DEV), q, k, v


def _no_alloc(q, k, v, mask, w, sp):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.S), float("nan"), dtype=torch.float32, device=DEV)
    dbsp.dbsp_block_sparse_attn_fwd_split_noalloc(q, k, v, mask, w.block, w.causal, sp.worker_offsets, sp.worklist,
                                                  sp.n_workers, sp.unit_item, sp.unit_pk, sp.unit_slot,
                                                  sp.split_item, sp.split_off, sp.counts, sp.max_slots, out, lse)
    return out, lse


@pytest.mark.parametrize("block,d,causal", [(128, 128, True), (64, 64, False)])
def test_no_alloc_matches_split_path_twice(built_library, cuda_device, block, d, causal):
    w, mask, q, k, v = _problem(block, d, causal)
    plans = [P.plan_split(mask, 7, block, d, max_piece_load=1, max_pieces=4),
             P.plan_split(mask, 5, block, d, max_piece_load=2, max_pieces=3)]
    for i, sp in enumerate(plans):
        assert sp.counts.cpu().numpy()[2] > 0  # items were split: the pieces use the scratch
        out_ref, lse_ref = P.attention_split(q, k, v, mask, block, causal, sp)
        out, lse = _no_alloc(q, k, v, mask, w, sp)
        assert dbsp.dbsp_device_status() == 0
        assert_rows_close(to64(out), to64(out_ref), to64(lse), to64(lse_ref), what=f"no-alloc call {i + 1}")


def test_no_alloc_refuses_a_plan_beyond_the_scratch(built_library, cuda_device):
    w, mask, q, k, v = _problem()
    sp = P.plan_split(mask, 7, 128, 128, max_piece_load=1, max_pieces=4)
    too_many = dbsp.DBSP_NOALLOC_SCRATCH_BYTES // (128 * 130 * 4) + 1
    out = torch.empty_like(q)
    lib = dbsp.library()
    st = lib.dbsp_block_sparse_attn_fwd_split_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), mask.data_ptr(), w.B, w.H, w.S, w.d, w.block, 1, 0.0,
        sp.worker_offsets.data_ptr(), sp.worklist.data_ptr(), sp.n_workers, sp.unit_item.data_ptr(),
        sp.unit_pk.data_ptr(), sp.unit_slot.data_ptr(), sp.unit_item.numel(), sp.split_item.data_ptr(),
        sp.split_off.data_ptr(), sp.counts.data_ptr(), too_many, out.data_ptr(), None, None, None)
    assert st == dbsp.DBSP_ERR_INVALID_ARG
    with pytest.raises(ValueError, match="scratch"):
        dbsp.dbsp_block_sparse_attn_fwd_split_noalloc(q, k, v, mask, w.block, w.causal, sp.worker_offsets,
                                                      sp.worklist, sp.n_workers, sp.unit_item, sp.unit_pk,
                                                      sp.unit_slot, sp.split_item, sp.split_off, sp.counts,
                                                      too_many, out)
