"""dbsp_plan_lpt on the GPU: bit-exact against the oracle's textbook LPT."""

import numpy as np
import pytest
import torch

from load_balancing_gb300 import workloads as W
from oracle import loads as OL
from oracle import lpt as OP
from conftest import load_golden

pytestmark = pytest.mark.gpu


def _plan(loads, m, home=None, bonus=0, check_status=True):
    from load_balancing_gb300 import dbsp

    dev = torch.device("cuda:0")
    loads_t = torch.as_tensor(np.asarray(loads, dtype=np.int32)).to(dev)
    n = loads_t.numel()
    wo = torch.full((n,), -5, dtype=torch.int32, device=dev)
    off = torch.full((m + 1,), -5, dtype=torch.int32, device=dev)
    wl = torch.full((n,), -5, dtype=torch.int32, device=dev)
    wload = torch.full((m,), -5, dtype=torch.int64, device=dev)
    home_t = None if home is None else torch.as_tensor(np.asarray(home, dtype=np.int32)).to(dev)
    dbsp.dbsp_plan_lpt(loads_t, m, wo, off, wl, wload, home=home_t, stay_bonus=bonus)
    status = dbsp.dbsp_device_status()
    if check_status:
        assert status == 0
    return {"worker_of": wo.cpu().numpy(), "offsets": off.cpu().numpy(), "worklist": wl.cpu().numpy(),
            "worker_loads": wload.cpu().numpy(), "status": status}


def _assert_same(got, ref):
    for key in ("worker_of", "offsets", "worklist", "worker_loads"):
        np.testing.assert_array_equal(got[key], np.asarray(ref[key]), err_msg=key)


def test_page_counterexample(built_library, cuda_device):
    g = load_golden("lpt_counterexample.json")
    got = _plan(g["loads"], g["n_workers"])
    assert got["worker_loads"].tolist() == [17, 13]
    assert got["worker_of"].tolist() == [0, 1, 1, 0, 0]
    _assert_same(got, OP.lpt_plan(g["loads"], 2))


@pytest.mark.parametrize("name", W.ORDER)
def test_workload_item_sets(built_library, cuda_device, name):
    mask = W.make_mask(W.WORKLOADS[name])
    row = OL.block_mask_loads(mask)[0].reshape(-1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for m in sorted({1, 7, 32, sms, 1024}):
        _assert_same(_plan(row, m), OP.lpt_plan(row, m))


@pytest.mark.parametrize("m", [1, 2, 3, 31, 32, 33, 64, 100, 257, 513, 1024])
def test_random_instances_with_bonus(built_library, cuda_device, m):
    rng = np.random.default_rng(m)
    for n in (0, 1, 5, 33, 1000):
        loads = rng.integers(0, 100, n)
        _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))
        home = rng.integers(0, m, n)
        bonus = int(rng.integers(0, 150))
        _assert_same(_plan(loads, m, home, bonus), OP.lpt_plan(loads, m, home, bonus))


@pytest.mark.parametrize("name", ["llm", "video", "sharded"])
def test_plan_reuse_with_bonus(built_library, cuda_device, name):
    """The plan-reuse scenario (db-SP blog, scenario 2, third bullet): the next mask flips
    2 % of the blocks and its plan takes the previous plan as home. Bonuses from 1 up to
    past the loads' spread, bit-exact."""
    w = W.WORKLOADS[name]
    mask0 = W.make_mask(w)
    mask1 = W.perturb_mask(mask0, 0.02, 1, w.causal)
    row0 = OL.block_mask_loads(mask0)[0].reshape(-1)
    row1 = OL.block_mask_loads(mask1)[0].reshape(-1)
    m = torch.cuda.get_device_properties(0).multi_processor_count - 1
    home = np.asarray(OP.lpt_plan(row0, m)["worker_of"])
    for bonus in (1, 2, 4, 8, 32, 100, 1000):
        _assert_same(_plan(row1, m, home, bonus), OP.lpt_plan(row1, m, home, bonus))


@pytest.mark.parametrize("m", [2, 5, 64, 151, 1024])
def test_batched_bonus_random_homes(built_library, cuda_device, m):
    """Random homes, zero loads at the tail, bonuses small and large against the loads,
    from a handful of items to 9,000."""
    rng = np.random.default_rng(100 + m)
    for n in (7, 500, 4096, 8192, 9000):
        loads = rng.integers(0, 60, n)
        loads[rng.random(n) < 0.05] = 0
        home = rng.integers(0, m, n)
        for bonus in (1, 3, 17, 90):
            _assert_same(_plan(loads, m, home, bonus), OP.lpt_plan(loads, m, home, bonus))


def test_static_home_schedule_and_huge_bonus(built_library, cuda_device):
    rng = np.random.default_rng(9)
    n, m = 4096, 148
    loads = rng.integers(1, 64, n)
    home = (np.arange(n) * m) // n  # contiguous static schedule
    for bonus in (0, 5, 64, int(loads.sum()) + 1):
        _assert_same(_plan(loads, m, home, bonus), OP.lpt_plan(loads, m, home, bonus))


@pytest.mark.parametrize("m", [1, 7, 152, 1024])
def test_bonus_above_total_load_keeps_every_item_home(built_library, cuda_device, m):
    """A bonus above the total load makes every lowered home key the smallest, so every
    item stays at home, ranked by the LPT order (the plan takes a one-warp path for it);
    a bonus equal to the total load still takes the general greedy. Both bit-exact."""
    rng = np.random.default_rng(21 + m)
    n = 3000
    loads = rng.integers(0, 80, n)
    home = rng.integers(0, m, n)
    total = int(loads.sum())
    for bonus in (total + 1, 1 << 20):
        got = _plan(loads, m, home, bonus)
        _assert_same(got, OP.lpt_plan(loads, m, home, bonus))
        np.testing.assert_array_equal(got["worker_of"], home)
    _assert_same(_plan(loads, m, home, total), OP.lpt_plan(loads, m, home, total))
    # more items than the staged order holds: the order lives in the worklist
    n2 = 50000
    loads2 = rng.integers(1, 3000, n2)
    home2 = rng.integers(0, m, n2)
    got = _plan(loads2, m, home2, 1 << 30)
    _assert_same(got, OP.lpt_plan(loads2, m, home2, 1 << 30))


def test_large_loads_take_comparison_sort(built_library, cuda_device):
    rng = np.random.default_rng(4)
    loads = rng.integers(0, 5_000_000, 3000)
    loads[::7] = loads[3]  # plenty of ties
    _assert_same(_plan(loads, 37), OP.lpt_plan(loads, 37))


@pytest.mark.parametrize("n,hi,m", [(50000, 100, 148), (3000, 20000, 64), (2000, 4097, 1000)])
def test_unstaged_counting_paths(built_library, cuda_device, n, hi, m):
    """Beyond the shared-memory staging limits (n > 45056 or a load > 4095) the kernel
    sorts through global memory; the result must not change."""
    rng = np.random.default_rng(n + hi)
    loads = rng.integers(0, hi, n)
    loads[0] = hi - 1
    _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))


def test_zero_loads_and_single_worker(built_library, cuda_device):
    rng = np.random.default_rng(12)
    loads = rng.integers(0, 3, 5000)  # long runs of 0, 1, 2
    for m in (1, 2, 5, 148):
        _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))
    _assert_same(_plan(np.zeros(100, dtype=np.int64), 7), OP.lpt_plan(np.zeros(100, dtype=np.int64), 7))


def test_more_workers_than_items(built_library, cuda_device):
    loads = [5, 9, 9, 1, 0, 3]
    _assert_same(_plan(loads, 10), OP.lpt_plan(loads, 10))


def test_bad_inputs_set_device_status(built_library, cuda_device):
    got = _plan([3, -1, 2], 2, check_status=False)
    assert got["status"] == 1
    assert (got["offsets"] == 0).all()
    got = _plan([3, 1, 2], 2, home=[0, 5, 1], bonus=1, check_status=False)
    assert got["status"] == 1
    big = np.full(20000, 40000)
    got = _plan(big, 4, check_status=False)
    assert got["status"] == 2
    # the error word is cleared by the read: a good call afterwards is clean
    _assert_same(_plan([1, 2, 3], 2), OP.lpt_plan([1, 2, 3], 2))


@pytest.mark.parametrize("m,lo,hi", [(64, 1800, 2048), (300, 20000, 32768)])
def test_key_width_boundary(built_library, cuda_device, m, lo, hi):
    """Worker keys are 32-bit while total / m + max_load < 2^20 and 64-bit beyond;
    instances on both sides of that bound give the textbook LPT."""
    rng = np.random.default_rng(m)
    mean = (lo + hi - 1) / 2
    for target in ((1 << 20) * 0.97, (1 << 20) * 1.03):
        n = int((target - (hi - 1)) * m / mean)
        loads = rng.integers(lo, hi, n)
        loads[0] = hi - 1
        _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))



@pytest.mark.parametrize("m", [1, 2, 3, 33, 152, 1024])
def test_bucket_ring_edges(built_library, cuda_device, m):
    """Loads far apart (one huge item among tiny ones, long runs of equal loads) make
    the least-loaded worker win many picks in a row and move workers across the whole
    load ring; the plan stays the textbook LPT."""
    rng = np.random.default_rng(m + 77)
    for n in (2, 9, 300, 3000):
        loads = rng.choice(np.array([0, 1, 2, 1000]), n, p=[0.2, 0.4, 0.3, 0.1])
        _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))
        loads = rng.integers(0, 64, n)
        loads[: max(1, n // 50)] = 2047
        _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))


@pytest.mark.parametrize("bc,ic", [(1, 0), (1, 1), (8, 1), (16, 3), (1000, 7)])
def test_cost_model_is_lpt_on_transformed_loads(built_library, cuda_device, bc, ic):
    """dbsp_plan_lpt_cost plans on loads * block_cost + item_cost: the textbook LPT of
    the transformed loads (the order of the items is unchanged)."""
    from load_balancing_gb300 import dbsp

    dev = torch.device("cuda:0")
    rng = np.random.default_rng(bc * 31 + ic)
    for n, m, hi in ((1, 3, 5), (500, 7, 40), (4096, 152, 33), (3000, 300, 3)):
        loads = rng.integers(0, hi, n)
        loads[rng.random(n) < 0.3] = 0  # many items without dense blocks
        lt = torch.as_tensor(loads.astype(np.int32)).to(dev)
        wo = torch.empty(n, dtype=torch.int32, device=dev)
        off = torch.empty(m + 1, dtype=torch.int32, device=dev)
        wl = torch.empty(n, dtype=torch.int32, device=dev)
        wload = torch.empty(m, dtype=torch.int64, device=dev)
        dbsp.dbsp_plan_lpt_cost(lt, m, bc, ic, wo, off, wl, wload)
        assert dbsp.dbsp_device_status() == 0
        got = {"worker_of": wo.cpu().numpy(), "offsets": off.cpu().numpy(), "worklist": wl.cpu().numpy(),
               "worker_loads": wload.cpu().numpy()}
        _assert_same(got, OP.lpt_plan(loads.astype(np.int64) * bc + ic, m))


def test_item_cost_spreads_empty_items(built_library, cuda_device):
    """With block costs only, every item without dense blocks goes to the least-loaded
    worker; with an item cost the empty items are spread so that the planning loads
    balance to within one item."""
    from load_balancing_gb300 import dbsp

    dev = torch.device("cuda:0")
    loads = np.zeros(1000, dtype=np.int32)
    loads[:50] = 10
    m = 20
    lt = torch.as_tensor(loads).to(dev)
    counts, wloads = [], []
    for bc, ic in ((1, 0), (8, 1)):
        wo = torch.empty(1000, dtype=torch.int32, device=dev)
        off = torch.empty(m + 1, dtype=torch.int32, device=dev)
        wl = torch.empty(1000, dtype=torch.int32, device=dev)
        wload = torch.empty(m, dtype=torch.int64, device=dev)
        dbsp.dbsp_plan_lpt_cost(lt, m, bc, ic, wo, off, wl, wload)
        counts.append(np.bincount(wo.cpu().numpy(), minlength=m))
        wloads.append(wload.cpu().numpy())
    assert counts[0].max() >= 950  # the zero loads pile onto one worker
    assert counts[1].max() <= 100  # spread over the workers
    assert wloads[1].max() - wloads[1].min() <= 10 * 8 + 1  # planning loads within one item


@pytest.mark.parametrize("m,wmaxes", [(1, (0, 1, 2047)), (152, (511, 512, 818, 819, 2047)),
                                      (1024, (127, 128, 255, 256))])
def test_bucket_ring_limits(built_library, cuda_device, m, wmaxes):
    """The load-bucket greedy runs while the ring (2 wmax + 1 buckets of ceil(m / 32)
    words) and each batch's window fit their shared-memory budgets; instances on both
    sides of those limits, with long runs, ties and zero loads, give the textbook LPT."""
    rng = np.random.default_rng(m)
    for wmax in wmaxes:
        for n in (m // 2 + 1, 4 * m + 3, 20000):
            loads = rng.integers(0, wmax + 1, n)
            loads[rng.random(n) < 0.2] = max(0, wmax // 3)  # a long run of equal loads
            loads[0] = wmax
            _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))


def test_causal_plan_of_an_unclipped_mask(built_library, cuda_device):
    """path.plan(causal=True) on a causal mask that still holds blocks above the diagonal
    plans exactly what the oracle's LPT gives for the loads of the mask clipped to the
    diagonal (the blocks causal attention computes); without the flag the plan differs."""
    from load_balancing_gb300 import path as P

    rng = np.random.default_rng(21)
    shape = (1, 4, 48, 48)
    mask_np = (rng.random(shape) < 0.5).astype(np.uint8)
    mask = torch.from_numpy(mask_np).to("cuda:0")
    clipped = np.where(np.tril(np.ones(shape[2:], dtype=bool)), mask_np, 0).astype(np.uint8)
    row, _, _ = OL.block_mask_loads(clipped)
    ref = OP.lpt_plan(row.reshape(-1), 9)
    p = P.plan(mask, 9, causal=True)
    got = {"worker_of": p.worker_of.cpu().numpy(), "offsets": p.worker_offsets.cpu().numpy(),
           "worklist": p.worklist.cpu().numpy(), "worker_loads": p.worker_loads.cpu().numpy()}
    _assert_same(got, ref)
    q = P.plan(mask, 9)
    assert not np.array_equal(q.worker_loads.cpu().numpy(), got["worker_loads"])


@pytest.mark.parametrize("n,hi,m", [(8191, 60, 152), (8192, 60, 152), (46000, 30, 152), (46085, 30, 152)])
def test_worklist_assembled_in_shared_memory(built_library, cuda_device, n, hi, m):
    """From 8,192 items up to what fits the kernel's dynamic shared memory (46,084
    int32), the worklist is assembled in shared memory and copied out; either side of
    both limits the plan is the oracle's."""
    rng = np.random.default_rng(n)
    loads = rng.integers(0, hi, n)
    _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))


def _runs_in_id_order(rng, n, values):
    """Loads in runs of one value in id order, of random lengths (1 to 700), so that the
    stable scatter's groups of 256 ids meet runs that start and end mid-group."""
    out = np.empty(n, dtype=np.int64)
    i = 0
    while i < n:
        r = int(rng.integers(1, 700))
        out[i:i + r] = rng.choice(values)
        i += r
    return out


@pytest.mark.parametrize("n", [22528, 22529, 30000, 45056])
@pytest.mark.parametrize("m", [7, 152, 1024])
@pytest.mark.parametrize("shape", ["spread", "sparse", "id_runs"])
def test_staged_plans_with_many_or_few_runs(built_library, cuda_device, n, m, shape):
    """Staged plans on both sides of the 22,528-item limit for keeping the sorted loads:
    beyond it a position's load comes from the table of runs of equal load. Loads spread
    over [0, 2047] (short runs, few empty bins), a handful of loads far apart (long runs,
    hundreds of empty bins between them) and runs of one load in id order (the scatter's
    groups of one load) all give the oracle's LPT."""
    rng = np.random.default_rng(n * 7 + m)
    # the largest load that keeps the bucket ring (R >= 2 wmax + 1 buckets, R a power of two:
    # R <= 4,096 and R * ceil(m / 32) <= 10,240 words), which the table of runs serves
    wmax = {7: 2047, 152: 1023, 1024: 127}[m]
    if shape == "spread":
        loads = rng.integers(0, wmax + 1, n)
    elif shape == "sparse":
        loads = rng.choice(np.array([0, 3, wmax // 4, wmax // 2 + 1, wmax]), n)
    else:
        loads = _runs_in_id_order(rng, n, rng.integers(0, wmax + 1, 40))
    loads[n // 3] = wmax
    _assert_same(_plan(loads, m), OP.lpt_plan(loads, m))


@pytest.mark.parametrize("n", [16383, 16384, 20001])
def test_large_plans_with_homes_and_unaligned_loads(built_library, cuda_device, n):
    """From 16,384 items up the kernel keeps 8 reads in flight per thread and prefetches
    the loads and homes into L2 (16-byte aligned arrays only). Plans with homes and a
    bonus, and plans whose loads start 4 bytes past a 16-byte boundary (no prefetch, no
    16-byte reads), on both sides of that limit, are the oracle's."""
    from load_balancing_gb300 import dbsp

    rng = np.random.default_rng(n)
    m = 152
    loads = rng.integers(0, 90, n)
    home = rng.integers(0, m, n)
    for bonus in (0, 3):
        _assert_same(_plan(loads, m, home, bonus), OP.lpt_plan(loads, m, home, bonus))
    dev = torch.device("cuda:0")
    buf = torch.zeros(n + 1, dtype=torch.int32, device=dev)
    buf[1:] = torch.as_tensor(loads.astype(np.int32)).to(dev)
    shifted = buf[1:]  # 4-byte aligned only
    assert shifted.data_ptr() % 16 != 0
    wo = torch.full((n,), -5, dtype=torch.int32, device=dev)
    off = torch.full((m + 1,), -5, dtype=torch.int32, device=dev)
    wl = torch.full((n,), -5, dtype=torch.int32, device=dev)
    wload = torch.full((m,), -5, dtype=torch.int64, device=dev)
    dbsp.dbsp_plan_lpt(shifted, m, wo, off, wl, wload)
    assert dbsp.dbsp_device_status() == 0
    got = {"worker_of": wo.cpu().numpy(), "offsets": off.cpu().numpy(), "worklist": wl.cpu().numpy(),
           "worker_loads": wload.cpu().numpy()}
    _assert_same(got, OP.lpt_plan(loads, m))
