"""A pipeline wait that runs out, on the GPU, without a fault.

The attention kernel bounds every mbarrier wait; when one runs out the CTA records
DBSP_ERR_TIMEOUT in the device error word, every role leaves its loop, copies and MMAs
in flight are waited for (bounded) and TMEM is freed. To make a wait run out, a test
build of the library (compiled with -DDBSP_WAIT_TEST: 20 ms waits, and the V producer
of CTA 0 issues neither the arrival nor the copy of its first tile, so no copy is left
in flight) runs in a child process next to the product library:
  * the test build reports DBSP_ERR_TIMEOUT, twice in a row (the word is cleared and
    set again), and the items of every other CTA still match the oracle;
  * the product library, on the same stream of the same process, then returns
    DBSP_OK and the whole output matches the oracle: the context stays usable.
The streaming mask-loads kernel is tested the same way: in the test build its CTA
(0, 0) leaves out the first of its shared-memory stages (arrival and copy), so its
bounded stage wait runs out; the other heads' loads are still exact, and the product
library then returns exact loads for every head.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def _child(test_lib):
    import numpy as np
    import torch

    from load_balancing_gb300 import dbsp
    from load_balancing_gb300 import path as P
    from load_balancing_gb300 import workloads as W
    from oracle import attention as A
    from parity import assert_rows_close, to64

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = W.WORKLOADS["tiny"]
    mask_np = W.make_mask(w)
    q, k, v = W.make_qkv(w, "cpu")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    mask = torch.from_numpy(mask_np).to(dev)
    o_ref, lse_ref = A.attention(to64(q), to64(k), to64(v), mask_np, w.block, w.causal)
    m = 4
    product = dbsp.library()
    report = {}

    p = P.plan(mask, m)  # planned by the product library: the test build's loads time out too
    torch.cuda.synchronize()
    assert dbsp.dbsp_device_status() == dbsp.DBSP_OK
    dbsp._lib = dbsp.open_library(test_lib)
    off = p.worker_offsets.cpu().numpy()
    wl = p.worklist.cpu().numpy()
    statuses = []
    for _ in range(2):
        out = torch.zeros_like(qd)
        lse = torch.zeros((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        P.attention(qd, kd, vd, mask, w.block, w.causal, p, out=out, lse=lse)
        statuses.append(dbsp.dbsp_device_status())
        for item in wl[off[1]:off[m]]:  # items of CTAs 1..m-1
            bh, qb = divmod(int(item), w.nQ)
            b, h = divmod(bh, w.H)
            rows = slice(qb * w.block, (qb + 1) * w.block)
            assert_rows_close(to64(out[b, h, rows]), o_ref[b, h, rows], to64(lse[b, h, rows]),
                              lse_ref[b, h, rows], what=f"test build, item {item}")
    report["test_build_status"] = statuses
    report["cta0_items"] = int(off[1] - off[0])

    dbsp._lib = product
    out, lse = P.attention(qd, kd, vd, mask, w.block, w.causal, P.plan(mask, m))
    report["product_status"] = dbsp.dbsp_device_status()
    assert_rows_close(to64(out), o_ref, to64(lse), lse_ref, what="product build after the timeouts")
    print("WAIT_TEST " + json.dumps(report))


def test_bounded_wait_runs_out(built_library, cuda_device):
    from load_balancing_gb300 import build as lbuild

    test_lib = lbuild.build_wait_test()
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([HERE, os.path.dirname(HERE), env.get("PYTHONPATH", "")])
    code = f"import test_gpu_wait_timeout as t; t._child({test_lib!r})"
    r = subprocess.run([sys.executable, "-c", code], cwd=HERE, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, f"child failed:\n{r.stdout}\n{r.stderr}"
    line = [x for x in r.stdout.splitlines() if x.startswith("WAIT_TEST ")][-1]
    report = json.loads(line[len("WAIT_TEST "):])
    from load_balancing_gb300 import dbsp

    assert report["cta0_items"] > 0
    assert report["test_build_status"] == [dbsp.DBSP_ERR_TIMEOUT, dbsp.DBSP_ERR_TIMEOUT]
    assert report["product_status"] == dbsp.DBSP_OK


def _loads_child(test_lib):
    import numpy as np
    import torch

    from load_balancing_gb300 import dbsp
    from oracle import loads as OL

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # 4096 x 64 per head: 8 ranks of 512 rows each, two 16 KB stages per rank, so the
    # second stage of CTA (0, 0) is still in flight when its first wait gives up
    B, H, nQ, nK = 1, 2, 4096, 64
    rng = np.random.default_rng(12)
    mask_np = (rng.random((B, H, nQ, nK)) < 0.4).astype(np.uint8)
    mask = torch.from_numpy(mask_np).to(dev)
    r_ref, c_ref, h_ref = OL.block_mask_loads(mask_np)
    product = dbsp.library()
    report = {}

    def run():
        row = torch.full((B, H, nQ), -7, dtype=torch.int32, device=dev)
        col = torch.full((B, H, nK), -7, dtype=torch.int32, device=dev)
        head = torch.full((B, H), -7, dtype=torch.int32, device=dev)
        dbsp.dbsp_block_mask_loads(mask, row, col, head)
        return row.cpu().numpy(), col.cpu().numpy(), head.cpu().numpy(), dbsp.dbsp_device_status()

    dbsp._lib = dbsp.open_library(test_lib)
    row, col, head, st = run()
    report["test_build_status"] = st
    # CTA (0, 0) holds rows 0..511 of head 0; the other ranks' rows and head 1 are exact
    report["other_rows_exact"] = bool((row[0, 0, 512:] == r_ref[0, 0, 512:]).all())
    report["other_head_exact"] = bool((row[:, 1] == r_ref[:, 1]).all() and (col[:, 1] == c_ref[:, 1]).all()
                                      and (head[:, 1] == h_ref[:, 1]).all())
    dbsp._lib = product
    row, col, head, st = run()
    report["product_status"] = st
    report["product_exact"] = bool((row == r_ref).all() and (col == c_ref).all() and (head == h_ref).all())
    print("WAIT_TEST " + json.dumps(report))


def test_bounded_stage_wait_of_mask_loads_runs_out(built_library, cuda_device):
    from load_balancing_gb300 import build as lbuild

    test_lib = lbuild.build_wait_test()
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([HERE, os.path.dirname(HERE), env.get("PYTHONPATH", "")])
    code = f"import test_gpu_wait_timeout as t; t._loads_child({test_lib!r})"
    r = subprocess.run([sys.executable, "-c", code], cwd=HERE, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, f"child failed:\n{r.stdout}\n{r.stderr}"
    line = [x for x in r.stdout.splitlines() if x.startswith("WAIT_TEST ")][-1]
    report = json.loads(line[len("WAIT_TEST "):])
    from load_balancing_gb300 import dbsp

    assert report["test_build_status"] == dbsp.DBSP_ERR_TIMEOUT
    assert report["other_rows_exact"]
    assert report["other_head_exact"]
    assert report["product_status"] == dbsp.DBSP_OK
    assert report["product_exact"]
