"""PipelinedSteps on the GPU: batch i's attention beside batch i+1's loads and plan.

Three batches with different masks and Q values go through prime + three steps. Each
step's plan buffer must hold the oracle's loads and LPT worklist for its batch (over SM
count - 1 workers); each step's output must equal, bit for bit, the serial path's
(plan then attention on the caller's stream) on the same inputs, since an item's result
does not depend on the worker that computes it, and match the oracle's attention
element by element (max |dO| <= 2e-2, mean |dO| <= 2e-3, |dLSE| <= 1e-3).
"""

import numpy as np
import pytest
import torch

from load_balancing_gb300 import dbsp
from load_balancing_gb300 import path as P
from load_balancing_gb300 import workloads as W
from oracle import attention as A
from oracle import loads as OL
from oracle import lpt as OP
from parity import assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _masks(w, n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        m = (rng.random((w.B, w.H, w.nQ, w.nK)) < 0.3 + 0.25 * i).astype(np.uint8)
        if w.causal:
            m = np.where(np.tril(np.ones((w.nQ, w.nK), dtype=bool)), m, 0).astype(np.uint8)
        m[..., np.arange(w.nQ), np.arange(w.nQ)] = 1
        out.append(m)
    return out


@pytest.mark.parametrize("lists", [True, False])
@pytest.mark.parametrize("causal", [True, False])
def test_pipelined_steps_match_serial_and_oracle(built_library, cuda_device, causal, lists):
    w = W.custom(f"pipe_{int(causal)}", 1, 3, 6 * 128, 128, 128, causal, 7, 117, "bernoulli", p=0.5,
                 numpy_qkv=True)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w, "cpu"))
    masks_np = _masks(w, 3, 41 + int(causal))
    masks = [torch.from_numpy(m).to(DEV) for m in masks_np]
    rng = np.random.default_rng(9)
    qs = [q] + [torch.from_numpy(rng.standard_normal(q.shape).astype(np.float32)).to(torch.bfloat16).to(DEV)
                for _ in range(2)]
    pipe = P.PipelinedSteps(w.B, w.H, w.nQ, w.nK, DEV, causal=causal, use_lists=lists)
    m = pipe.n_workers
    assert m == P.default_workers(DEV) - 1
    st = torch.cuda.Stream(DEV, priority=-1)
    outs = []
    with torch.cuda.stream(st):
        pipe.prime(masks[0], stream=st)
        for i in range(3):
            plan_i = pipe.plans[pipe._cur]
            o, l = pipe.step(qs[i], k, v, masks[i], w.block, w.causal, next_mask=masks[i + 1] if i < 2 else None,
                             stream=st)
            st.synchronize()
            # the plan this step's attention read
            r, _, _ = OL.block_mask_loads(masks_np[i])
            ref = OP.lpt_plan(r.reshape(-1), m)
            np.testing.assert_array_equal(plan_i.worklist.cpu().numpy(), np.asarray(ref["worklist"]))
            np.testing.assert_array_equal(plan_i.worker_offsets.cpu().numpy(), np.asarray(ref["offsets"]))
            outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    assert dbsp.dbsp_device_status() == 0
    for i in range(3):
        o_ser, l_ser = P.attention(qs[i], k, v, masks[i], w.block, w.causal, P.plan(masks[i], m + 1))
        torch.cuda.synchronize()
        assert torch.equal(outs[i][0], o_ser) and torch.equal(outs[i][1], l_ser)
        o_ref, lse_ref = A.attention(to64(qs[i]), to64(k), to64(v), masks_np[i], w.block, w.causal)
        assert_rows_close(to64(outs[i][0]), o_ref, to64(outs[i][1]), lse_ref, what=f"pipelined step {i}")


def test_pipelined_step_rejects_a_different_causal_flag(built_library, cuda_device):
    """The batches are planned (loads, LPT, lists) for one causal setting; a step asked
    for the other raises before it launches anything, and the pipeline stays usable."""
    w = W.custom("pipe_flag", 1, 2, 3 * 128, 128, 128, True, 8, 118, "bernoulli", p=0.5, numpy_qkv=True)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w, "cpu"))
    mask_np = W.make_mask(w)
    mask = torch.from_numpy(mask_np).to(DEV)
    pipe = P.PipelinedSteps(w.B, w.H, w.nQ, w.nK, DEV, causal=True)
    pipe.prime(mask)
    with pytest.raises(ValueError):
        pipe.step(q, k, v, mask, w.block, False)
    o, l = pipe.step(q, k, v, mask, w.block, True)
    torch.cuda.synchronize()
    assert dbsp.dbsp_device_status() == 0
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, w.block, True)
    assert_rows_close(to64(o), o_ref, to64(l), lse_ref, what="pipelined step after a rejected flag")
