"""dbsp_merge_partials on the GPU against the oracle's fold (6D attention notes §2.1)."""

import numpy as np
import pytest
import torch

from oracle import merge as OM
from parity import assert_rows_close

pytestmark = pytest.mark.gpu


def _partials(n, rows, d, seed, empty_frac=0.2):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((n, rows, d)).astype(np.float32) * 3
    m = (rng.standard_normal((n, rows)) * 4).astype(np.float32)
    l = (rng.random((n, rows)) * 50 + 0.5).astype(np.float32)
    empty = rng.random((n, rows)) < empty_frac
    m[empty], l[empty], o[empty] = -np.inf, 0.0, 0.0
    if rows > 3:
        m[:, 3], l[:, 3], o[:, 3] = -np.inf, 0.0, 0.0  # a row with no live partial
    return o, m, l


@pytest.mark.parametrize("n,rows,d", [(1, 1000, 128), (3, 777, 64), (8, 4096, 128), (5, 100, 4),
                                      (2, 513, 12), (16, 64, 1024), (9, 300, 64)])
def test_merge_matches_oracle(built_library, cuda_device, n, rows, d):
    from load_balancing_gb300 import dbsp

    o, m, l = _partials(n, rows, d, seed=n * 1000 + d)
    dev = torch.device("cuda:0")
    out = torch.empty((rows, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    dbsp.dbsp_merge_partials(torch.from_numpy(o).to(dev), torch.from_numpy(m).to(dev),
                             torch.from_numpy(l).to(dev), out, lse)
    assert dbsp.dbsp_device_status() == 0
    o_ref, lse_ref = OM.merge_partials(o, m, l)
    # merged values are weighted means of O_k / scale: compare relative to their size
    scale = max(1.0, float(np.abs(o_ref).max()))
    assert_rows_close(out.double().cpu().numpy() / scale, o_ref / scale, lse.double().cpu().numpy(), lse_ref,
                      what="merge")


def test_merge_without_lse(built_library, cuda_device):
    from load_balancing_gb300 import dbsp

    o, m, l = _partials(4, 300, 128, seed=5)
    dev = torch.device("cuda:0")
    out = torch.empty((300, 128), dtype=torch.bfloat16, device=dev)
    dbsp.dbsp_merge_partials(torch.from_numpy(o).to(dev), torch.from_numpy(m).to(dev),
                             torch.from_numpy(l).to(dev), out, None)
    o_ref, _ = OM.merge_partials(o, m, l)
    scale = max(1.0, float(np.abs(o_ref).max()))
    assert_rows_close(out.double().cpu().numpy() / scale, o_ref / scale, what="merge no lse")


def test_empty_partials_are_not_read(built_library, cuda_device):
    """An empty partial's O rows may hold anything (the attention kernel leaves them
    unwritten): NaN there must not reach the merged output."""
    from load_balancing_gb300 import dbsp

    o, m, l = _partials(11, 500, 64, seed=77, empty_frac=0.4)
    o_dirty = o.copy()
    o_dirty[~np.isfinite(m)] = np.nan
    dev = torch.device("cuda:0")
    out = torch.empty((500, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(500, dtype=torch.float32, device=dev)
    dbsp.dbsp_merge_partials(torch.from_numpy(o_dirty).to(dev), torch.from_numpy(m).to(dev),
                             torch.from_numpy(l).to(dev), out, lse)
    o_ref, lse_ref = OM.merge_partials(o, m, l)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    scale = max(1.0, float(np.abs(o_ref).max()))
    assert_rows_close(got / scale, o_ref / scale, lse.double().cpu().numpy(), lse_ref, what="merge dirty")
