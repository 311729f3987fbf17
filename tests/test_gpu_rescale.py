"""The online softmax's rescaling step and an explicit softmax scale, on the GPU.

6D attention notes §2.1, step 3: when a later chunk of keys raises a row's maximum, the
running sum and the unnormalised output are multiplied by exp(m_old - m_new) before the
new chunk is added. The kernel applies that factor to its TMEM accumulator only when a
row's maximum grows by more than 2^8 (8 in log2 units), which N(0, 1) inputs with the
default scale never reach. Here the keys of later KV-blocks are scaled up (seeded ramp,
rounded to bf16), and each case first checks on the host, in fp64, that a good share of
the rows does grow by more than 8.5 log2 units after its first dense block; the GPU
output is then compared with the fp64 oracle element by element (max |dO| <= 2e-2, mean
|dO| <= 2e-3, |dLSE| <= 1e-3) in final, partial and split (unit) mode, for every
(block, d) pair the kernel implements, causal and not. Separate cases pass an explicit
softmax scale.
"""

import math

import numpy as np
import pytest
import torch

from load_balancing_gb300 import dbsp
from load_balancing_gb300 import path as P
from load_balancing_gb300 import workloads as W
from oracle import attention as A
from parity import assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LOG2E = 1.0 / math.log(2.0)


def _problem(block, d, causal, seed, nblocks=6, density=0.6, H=2):
    w = W.custom(f"rescale_{block}_{d}_{int(causal)}", 1, H, nblocks * block, d, block, causal, seed, seed + 100,
                 "bernoulli", p=density, numpy_qkv=True)
    mask_np = W.make_mask(w)
    q, k, v = W.make_qkv(w, "cpu")
    return w, mask_np, q, k, v


def _grown_rows(q, k, mask_np, block, causal, scale, margin=8.5):
    """(rows whose running maximum, in log2 units over the dense blocks in column order,
    grows by more than ``margin`` after the first dense block; live rows)."""
    q64, k64 = to64(q), to64(k)
    B, H, nQ, nK = mask_np.shape
    grown = live = 0
    for b in range(B):
        for h in range(H):
            for qb in range(nQ):
                cols = [j for j in range(nK) if mask_np[b, h, qb, j] and (not causal or j <= qb)]
                if not cols:
                    continue
                qr = q64[b, h, qb * block:(qb + 1) * block]
                run = None
                jumped = np.zeros(block, dtype=bool)
                for j in cols:
                    s = qr @ k64[b, h, j * block:(j + 1) * block].T * scale * LOG2E
                    if causal and j == qb:
                        s = np.where(np.tril(np.ones((block, block), bool)), s, -np.inf)
                    mx = s.max(axis=1)
                    if run is None:
                        run = mx
                    else:
                        jumped |= mx > run + margin
                        run = np.maximum(run, mx)
                grown += int(jumped.sum())
                live += block
    return grown, live


@pytest.mark.parametrize("block,d", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", ["final", "partial"])
def test_rescale_elementwise(built_library, cuda_device, block, d, causal, mode):
    w, mask_np, q, k, v = _problem(block, d, causal, seed=40 + block + d)
    k = W.ramp_key_blocks(k, block, 1.5)
    scale = 1.0 / math.sqrt(d)
    grown, live = _grown_rows(q, k, mask_np, block, causal, scale)
    assert grown >= 0.2 * live, f"only {grown} of {live} rows reach the rescaling step"
    mask = torch.from_numpy(mask_np).to(DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    p = P.plan(mask, 5)
    if mode == "final":
        out, lse = P.attention(qd, kd, vd, mask, block, causal, p)
        assert dbsp.dbsp_device_status() == 0
        o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal)
        assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what=f"rescale b{block} d{d} c{causal}")
    else:
        shape = (w.B, w.H, w.S)
        o_part = torch.empty(shape + (d,), dtype=torch.float32, device=DEV)
        m_part = torch.empty(shape, dtype=torch.float32, device=DEV)
        l_part = torch.empty(shape, dtype=torch.float32, device=DEV)
        P.attention_partial(qd, kd, vd, mask, block, causal, p, o_part, m_part, l_part)
        assert dbsp.dbsp_device_status() == 0
        o_ref, m_ref, l_ref = A.attention_partials(to64(q), to64(k), to64(v), mask_np, block, causal)
        live_rows = np.isfinite(m_ref)
        m_g, l_g, o_g = to64(m_part), to64(l_part), to64(o_part)
        assert (m_g[~live_rows] == -np.inf).all() and (l_g[~live_rows] == 0).all()
        # m is the true row maximum; l and O are relative to it (the kernel's lagging
        # reference maximum must have been folded out)
        assert np.abs(m_g[live_rows] - m_ref[live_rows]).max() <= 1e-3
        assert (np.abs(l_g[live_rows] / l_ref[live_rows] - 1) <= 1e-2).all()
        norm = lambda o, l: np.where(live_rows[..., None], o / np.where(live_rows, l, 1)[..., None], 0)
        assert_rows_close(norm(o_g, l_g), norm(o_ref, l_ref), what=f"rescale partial b{block} d{d} c{causal}")


@pytest.mark.parametrize("block,d", [(128, 128), (64, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_split_units(built_library, cuda_device, block, d, causal):
    """Pieces of split items rescale within their own dense blocks, and the merge folds
    the pieces' maxima (unit variant of the kernel, then the piece merge)."""
    w, mask_np, q, k, v = _problem(block, d, causal, seed=60 + block, nblocks=8, density=0.7)
    k = W.ramp_key_blocks(k, block, 1.5)
    grown, live = _grown_rows(q, k, mask_np, block, causal, 1.0 / math.sqrt(d))
    assert grown >= 0.2 * live
    mask = torch.from_numpy(mask_np).to(DEV)
    sp = P.plan_split(mask, 7, block, d, max_piece_load=3, max_pieces=3)
    out, lse = P.attention_split(q.to(DEV), k.to(DEV), v.to(DEV), mask, block, causal, sp)
    assert dbsp.dbsp_device_status() == 0
    assert sp.counts.cpu().numpy()[2] > 0  # items were split
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal)
    assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what=f"rescale split b{block} d{d} c{causal}")


@pytest.mark.parametrize("scale", [0.05, 0.3, 1.0])
@pytest.mark.parametrize("block,d,causal", [(128, 128, True), (64, 64, False), (128, 64, False)])
def test_explicit_scale(built_library, cuda_device, scale, block, d, causal):
    """The ``scale`` argument replaces 1/sqrt(d); scale 1.0 with d >= 64 also drives rows
    through the rescaling step without any key ramp."""
    w, mask_np, q, k, v = _problem(block, d, causal, seed=80 + block + d)
    mask = torch.from_numpy(mask_np).to(DEV)
    p = P.plan(mask, 6)
    out, lse = P.attention(q.to(DEV), k.to(DEV), v.to(DEV), mask, block, causal, p, scale=scale)
    assert dbsp.dbsp_device_status() == 0
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, block, causal, scale=scale)
    assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what=f"scale {scale} b{block} d{d} c{causal}")
    if scale == 1.0:
        grown, live = _grown_rows(q, k, mask_np, block, causal, scale)
        assert grown > 0
