"""The hot path captured as one CUDA graph, as the benchmark times it, on the GPU.

Mask loads, the LPT plan and attention are launched with programmatic stream
serialization: each kernel may start while the previous one finishes and waits
(griddepcontrol.wait) before it touches the previous kernel's results. Captured in one
CUDA graph and replayed, each launch must still see the results of the one before.
The test changes the mask and Q in place between replays, so that stale loads, a
stale plan or a stale mask row would show: after every replay the loads and the
worklist are bit-exact against the oracle's, and the output matches the oracle's
attention element by element (max |dO| <= 2e-2, mean |dO| <= 2e-3, |dLSE| <= 1e-3).
A split-path graph (units attention, then the piece merge) is checked the same way.
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
    for _ in range(n):
        m = (rng.random((w.B, w.H, w.nQ, w.nK)) < 0.55).astype(np.uint8)
        if w.causal:
            m = np.where(np.tril(np.ones((w.nQ, w.nK), dtype=bool)), m, 0).astype(np.uint8)
        m[..., np.arange(w.nQ), np.arange(w.nQ)] = 1
        out.append(m)
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_step_graph_sees_each_launchs_inputs(built_library, cuda_device, causal):
    w = W.custom(f"graph_step_{int(causal)}", 1, 3, 6 * 128, 128, 128, causal, 7, 107, "bernoulli", p=0.5,
                 numpy_qkv=True)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w, "cpu"))
    masks = _masks(w, 3, 31 + int(causal))
    m = 5
    mask = torch.from_numpy(masks[0]).to(DEV)
    pb = P.alloc_plan(w.B, w.H, w.nQ, w.nK, m, DEV)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=DEV)
    side = torch.cuda.Stream(DEV)

    def step(st):
        dbsp.dbsp_block_mask_loads(mask, pb.row_loads, pb.col_loads, pb.head_loads, stream=st)
        dbsp.dbsp_plan_lpt(pb.row_loads.view(-1), m, pb.worker_of, pb.worker_offsets, pb.worklist, pb.worker_loads,
                           stream=st)
        dbsp.dbsp_block_sparse_attn_fwd(q, k, v, mask, w.block, w.causal, pb.worker_offsets, pb.worklist, m,
                                        out=out, lse=lse, stream=st)

    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        step(side)  # warm-up outside the capture
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            step(side)
    torch.cuda.current_stream().wait_stream(side)
    rng = np.random.default_rng(5)
    for i, mask_np in enumerate(masks):
        mask.copy_(torch.from_numpy(mask_np))
        if i:  # new Q values too
            q_np = rng.standard_normal(q.shape).astype(np.float32)
            q.copy_(torch.from_numpy(q_np).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        assert dbsp.dbsp_device_status() == 0
        r, c, h = OL.block_mask_loads(mask_np)
        np.testing.assert_array_equal(pb.row_loads.cpu().numpy(), r)
        np.testing.assert_array_equal(pb.col_loads.cpu().numpy(), c)
        ref = OP.lpt_plan(r.reshape(-1), m)
        np.testing.assert_array_equal(pb.worklist.cpu().numpy(), np.asarray(ref["worklist"]))
        np.testing.assert_array_equal(pb.worker_offsets.cpu().numpy(), np.asarray(ref["offsets"]))
        o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, w.block, w.causal)
        assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what=f"graph replay {i}")


def test_split_graph_sees_each_launchs_inputs(built_library, cuda_device):
    """Units attention followed by the piece merge, captured and replayed after the Q
    values change: the merge must read the pieces of the same replay."""
    w = W.custom("graph_split", 1, 2, 8 * 128, 128, 128, True, 9, 109, "bernoulli", p=0.7, numpy_qkv=True)
    q, k, v = (t.to(DEV) for t in W.make_qkv(w, "cpu"))
    mask_np = _masks(w, 1, 77)[0]
    mask = torch.from_numpy(mask_np).to(DEV)
    sp = P.plan_split(mask, 7, w.block, w.d, max_piece_load=2, max_pieces=3)
    torch.cuda.synchronize()
    assert sp.counts.cpu().numpy()[2] > 0  # items were split
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=DEV)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        P.attention_split(q, k, v, mask, w.block, w.causal, sp, out=out, lse=lse, stream=side)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            P.attention_split(q, k, v, mask, w.block, w.causal, sp, out=out, lse=lse, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    rng = np.random.default_rng(8)
    for i in range(2):
        q_np = rng.standard_normal(q.shape).astype(np.float32)
        q.copy_(torch.from_numpy(q_np).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        assert dbsp.dbsp_device_status() == 0
        o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, w.block, w.causal)
        assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what=f"split graph replay {i}")
