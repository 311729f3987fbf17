"""The C-ABI library: it builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "dbsp.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DBSP_API\s+[\w\s\*]+?\b(dbsp_\w+)\s*\(", text)))


def test_header_declares_the_path(built_library):
    names = declared_symbols()
    for required in ("dbsp_block_mask_loads", "dbsp_plan_lpt", "dbsp_block_sparse_attn_fwd",
                     "dbsp_merge_partials", "dbsp_device_status", "dbsp_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(built_library):
    lib = ctypes.CDLL(built_library)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_uses_the_same_names(built_library):
    from load_balancing_gb300 import dbsp

    for name in declared_symbols():
        if name in ("dbsp_status_string", "dbsp_last_error_string"):
            continue
        assert callable(getattr(dbsp, name)), name


def test_status_strings(built_library):
    from load_balancing_gb300 import dbsp

    lib = dbsp.library()
    assert lib.dbsp_status_string(0) == b"ok"
    assert b"timed out" in lib.dbsp_status_string(4)
    assert lib.dbsp_status_string(99) == b"unknown status"


FAKE = 1 << 20  # never dereferenced: validation fails first


@pytest.mark.parametrize("args,expect", [
    ((None, 1, 1, 1, 1, FAKE, FAKE, None, None), 1),            # null mask
    ((FAKE, 0, 1, 1, 1, FAKE, FAKE, None, None), 1),            # B = 0
    ((FAKE, 1, 1, 1, 1, None, FAKE, None, None), 1),            # null row loads
    ((FAKE, 1, 1, 8, 20000, FAKE, FAKE, None, None), 2),        # nK beyond the kernel
    ((FAKE, 1, 1, 131073, 8, FAKE, FAKE, None, None), 2),       # nQ beyond the kernel
    ((FAKE, 1, 1, 1, 1, FAKE + 2, FAKE, None, None), 1),        # misaligned int32 output
    ((FAKE, 70000, 1, 1, 1, FAKE, FAKE, None, None), 1),        # B*H beyond the grid
])
def test_mask_loads_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_block_mask_loads(*args) == expect
    # the causal variant checks the same, and first that the mask is square
    assert dbsp.library().dbsp_block_mask_loads_causal(*args) == (expect if args[3] == args[4] else 1)


def test_causal_mask_loads_need_a_square_mask(built_library):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_block_mask_loads_causal(FAKE, 1, 1, 8, 16, FAKE, FAKE, None, None) == 1


@pytest.mark.parametrize("args,expect", [
    ((FAKE, None, 10, 0, 0, FAKE, FAKE, FAKE, None, None), 1),       # no workers
    ((FAKE, None, 10, 1025, 0, FAKE, FAKE, FAKE, None, None), 1),    # too many workers
    ((FAKE, None, -1, 4, 0, FAKE, FAKE, FAKE, None, None), 1),       # negative n
    ((FAKE, None, 10, 4, -3, FAKE, FAKE, FAKE, None, None), 1),      # negative bonus
    ((None, None, 10, 4, 0, FAKE, FAKE, FAKE, None, None), 1),       # null loads
    ((FAKE, None, 10, 4, 0, FAKE, None, FAKE, None, None), 1),       # null offsets
    ((FAKE, None, 3_000_000, 1000, 0, FAKE, FAKE, FAKE, None, None), 1),  # n*m overflow
])
def test_plan_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_plan_lpt(*args) == expect


@pytest.mark.parametrize("bc,ic,expect", [(0, 0, 1), (-2, 0, 1), (70000, 0, 1), (1, -1, 1), (1, 1 << 25, 1)])
def test_plan_cost_host_validation(built_library, bc, ic, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_plan_lpt_cost(FAKE, None, 10, 4, 0, bc, ic, FAKE, FAKE, FAKE, None, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, 2, 8, FAKE, None), 1),      # null column loads
    ((FAKE, 0, 8, FAKE, None), 1),      # no groups
    ((FAKE, 2, 0, FAKE, None), 1),      # no columns
    ((FAKE, 2, 8, None, None), 1),      # null output
    ((FAKE + 2, 2, 8, FAKE, None), 1),  # misaligned input
])
def test_kv_block_loads_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_kv_block_loads(*args) == expect


def _attn_args(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, mask=FAKE, B=1, H=1, S=256, d=128, block=128, causal=0, scale=0.0,
             off=FAKE, wl=FAKE, nw=4, out=FAKE, lse=None, op=None, mp=None, lp=None, tim=None, st=None)
    a.update(kw)
    return tuple(a.values())


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1),
    (dict(d=96), 2),
    (dict(block=32), 2),
    (dict(S=200), 2),
    (dict(nw=0), 1),
    (dict(out=None), 1),                          # neither mode
    (dict(op=FAKE, mp=FAKE, lp=FAKE), 1),         # both modes
    (dict(out=None, op=FAKE, mp=FAKE), 1),        # partial mode missing l
    (dict(q=FAKE + 8), 1),                        # q not 16-byte aligned
    (dict(B=70000, H=70000), 1),                  # rows overflow
])
def test_attention_host_validation(built_library, kw, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_block_sparse_attn_fwd(*_attn_args(**kw)) == expect


@pytest.mark.parametrize("args,expect", [
    ((FAKE, FAKE, FAKE, 0, 10, 128, FAKE, None, None), 1),
    ((FAKE, FAKE, FAKE, 2, 10, 130, FAKE, None, None), 1),
    ((FAKE, FAKE, FAKE, 2, -1, 128, FAKE, None, None), 1),
    ((FAKE + 4, FAKE, FAKE, 2, 10, 128, FAKE, None, None), 1),
    ((FAKE, FAKE, FAKE, 2, 0, 128, FAKE, None, None), 0),        # nothing to do
])
def test_merge_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_merge_partials(*args) == expect


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from load_balancing_gb300 import dbsp

    monkeypatch.setattr(dbsp, "_lib", None)
    monkeypatch.setattr(dbsp, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dbsp.library()


@pytest.mark.parametrize("args,expect", [
    ((FAKE, 10, 0, 0, 4, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),       # no workers
    ((FAKE, -1, 4, 0, 4, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),       # negative n
    ((FAKE, 10, 4, 0, 0, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),       # no pieces
    ((FAKE, 10, 4, 0, 1025, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),    # too many pieces
    ((FAKE, 10, 4, 0, 4, -1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),       # negative capacity
    ((FAKE, 10, 4, 0, 4, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None), 1),       # null counts
    ((None, 10, 4, 0, 4, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),       # null loads
    ((FAKE, 3_000_000, 4, 0, 1000, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None), 1),  # n*P overflow
])
def test_split_plan_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_split_plan(*args) == expect


def test_units_and_pieces_host_validation(built_library):
    from load_balancing_gb300 import dbsp

    lib = dbsp.library()
    base = [FAKE, FAKE, FAKE, FAKE, 1, 2, 512, 128, 128, 1, 0.0, FAKE, FAKE, 4]
    tail = [FAKE, FAKE, FAKE, 16, FAKE, FAKE, FAKE, FAKE, FAKE, 4, None, None]
    assert lib.dbsp_block_sparse_attn_fwd_units(*base, None, *tail[1:]) == 1      # null unit table
    bad = list(tail)
    bad[4] = None                                                                   # no final output
    assert lib.dbsp_block_sparse_attn_fwd_units(*base, *bad) == 1
    bad = list(tail)
    bad[9] = -1                                                                     # negative slot capacity
    assert lib.dbsp_block_sparse_attn_fwd_units(*base, *bad) == 1
    # the units entry shares the plain entry's shape checks
    assert lib.dbsp_block_sparse_attn_fwd_units(*base[:7], 96, *base[8:], *tail) == 2  # d = 96
    assert lib.dbsp_merge_pieces(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 1, 2, 512, 96, 128, FAKE, None, None) == 1
    assert lib.dbsp_merge_pieces(FAKE, FAKE, FAKE, None, FAKE, FAKE, 8, 1, 2, 512, 128, 128, FAKE, None, None) == 1
    assert lib.dbsp_merge_pieces(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 1, 2, 512, 128, 128, FAKE, None,
                                 None) == 1  # negative slot capacity
    assert lib.dbsp_plan_lpt_cost_n(FAKE, None, 10, 4, 1, 0, FAKE, FAKE, FAKE, None, None) == 1


@pytest.mark.parametrize("args,expect", [
    ((None, 1, 1, 4, 16, FAKE, 2, FAKE, None), 1),        # null mask
    ((FAKE, 1, 1, 4, 16, None, 2, FAKE, None), 1),        # null shard_of
    ((FAKE, 1, 1, 4, 16, FAKE, 0, FAKE, None), 1),        # no shards
    ((FAKE, 1, 1, 4, 16, FAKE, 70000, FAKE, None), 1),    # too many shards
    ((FAKE, 1, 1, 4, 16, FAKE + 2, 2, FAKE, None), 1),    # misaligned shard_of
    ((FAKE, 70000, 70000, 4, 16, FAKE, 2, FAKE, None), 1),  # mask too large
])
def test_shard_masks_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_shard_masks(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, 1, 2, 4, 4, 0, FAKE, FAKE, None), 1),               # no mask
    ((FAKE, 0, 2, 4, 4, 0, FAKE, FAKE, None), 1),               # B < 1
    ((FAKE, 1, 2, 4, 6, 1, FAKE, FAKE, None), 1),               # causal needs nQ == nK
    ((FAKE, 4, 4, 46341, 46341, 0, FAKE, FAKE, None), 1),       # mask bytes overflow int
    ((FAKE, 1, 1, 4, 65537, 0, FAKE, FAKE, None), 2),           # column indices are 16-bit
    ((FAKE, 1, 2, 4, 4, 0, FAKE + 2, FAKE, None), 1),           # counts not 4-byte aligned
    ((FAKE, 1, 2, 4, 4, 0, FAKE, FAKE + 1, None), 1),           # cols not 2-byte aligned
    ((FAKE, 1, 2, 4, 4, 0, None, FAKE, None), 1),               # no counts
])
def test_dense_block_lists_host_validation(built_library, args, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_dense_block_lists(*args) == expect


def _listed_args(dense_n=FAKE, dense_cols=FAKE, **kw):
    a = list(_attn_args(**kw))
    # the listed entry takes the lists after n_workers (q .. nw are the first 14 arguments)
    return tuple(a[:14] + [dense_n, dense_cols] + a[14:])


@pytest.mark.parametrize("lists,kw,expect", [
    (dict(dense_n=None), {}, 1),
    (dict(dense_cols=None), {}, 1),
    (dict(dense_n=FAKE + 2), {}, 1),                 # counts not 4-byte aligned
    (dict(dense_cols=FAKE + 1), {}, 1),              # indices not 2-byte aligned
    ({}, dict(q=None), 1),                           # the attention's own checks follow
    ({}, dict(d=96), 2),
    ({}, dict(out=None), 1),
])
def test_listed_attention_host_validation(built_library, lists, kw, expect):
    from load_balancing_gb300 import dbsp

    assert dbsp.library().dbsp_block_sparse_attn_fwd_listed(*_listed_args(**lists, **kw)) == expect
