"""Thin ctypes binding of libdbsp.so (declared in include/dbsp.h).

Argument marshalling only: each function checks that the torch tensors it is given
have the dtype, device and contiguity the C ABI expects, passes their pointers and
the current CUDA stream, and raises ``DbspError`` on a non-zero status. All
computation happens in the library's CUDA kernels. If the library has not been
built the first call raises; there is no fallback.
"""

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdbsp.so")
_lib = None

DBSP_OK = 0
DBSP_ERR_INVALID_ARG = 1
DBSP_ERR_UNSUPPORTED = 2
DBSP_ERR_CUDA = 3
DBSP_ERR_TIMEOUT = 4
DBSP_MAX_WORKERS = 1024

_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64

_SIGNATURES = {
    "dbsp_status_string": (ctypes.c_char_p, [_i32]),
    "dbsp_last_error_string": (ctypes.c_char_p, []),
    "dbsp_block_mask_loads": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "dbsp_block_mask_loads_causal": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "dbsp_shard_masks": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]),
    "dbsp_dense_block_lists": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "dbsp_kv_block_loads": (_i32, [_vp, _i32, _i32, _vp, _vp]),
    "dbsp_plan_lpt": (_i32, [_vp, _vp, _i32, _i32, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp]),
    "dbsp_plan_lpt_cost": (_i32, [_vp, _vp, _i32, _i32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp,
                                  _vp, _vp, _vp]),
    "dbsp_block_sparse_attn_fwd": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                          ctypes.c_float, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp,
                                          _vp, _vp]),
    "dbsp_block_sparse_attn_fwd_listed": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                                 ctypes.c_float, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp,
                                                 _vp, _vp, _vp, _vp]),
    "dbsp_merge_partials": (_i32, [_vp, _vp, _vp, _i32, _i64, _i32, _vp, _vp, _vp]),
    "dbsp_plan_lpt_cost_n": (_i32, [_vp, _vp, _i32, _i32, ctypes.c_int32, ctypes.c_int32, _vp, _vp, _vp, _vp,
                                    _vp]),
    "dbsp_split_plan": (_i32, [_vp, _i32, _i32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp, _vp,
                               _vp, _vp, _vp, _vp, _vp]),
    "dbsp_block_sparse_attn_fwd_units": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                                ctypes.c_float, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp,
                                                _vp, _vp, _vp, _i32, _vp, _vp]),
    "dbsp_merge_pieces": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "dbsp_device_status": (_i32, [_vp]),
    "dbsp_block_sparse_attn_fwd_split_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                                        ctypes.c_float, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp,
                                                        _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
}
DBSP_NOALLOC_SCRATCH_BYTES = 16 << 20


class DbspError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        lib = library()
        msg = lib.dbsp_status_string(status).decode()
        extra = lib.dbsp_last_error_string().decode() if status == DBSP_ERR_CUDA else ""
        super().__init__(f"{where}: status {status} ({msg}){': ' + extra if extra else ''}")


def open_library(path):
    """Loads a build of the library at ``path`` and declares every entry point's types."""
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def library():
    """The loaded libdbsp.so (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libdbsp.so is not built ({_LIB_PATH}); run "
                               "load_balancing_gb300.build.build() or __graft_entry__.build()")
        _lib = open_library(_LIB_PATH)
    return _lib


def library_path():
    return _LIB_PATH


def _check(status, where):
    if status != DBSP_OK:
        raise DbspError(status, where)


def _ptr(t, dtype, name, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dbsp_block_mask_loads(mask, row_loads, col_loads, head_loads=None, stream=None):
    """mask uint8 [B,H,nQ,nK] -> row_loads int32 [B,H,nQ], col_loads [B,H,nK], head_loads [B,H]."""
    B, H, nQ, nK = mask.shape
    st = library().dbsp_block_mask_loads(
        _ptr(mask, torch.uint8, "mask"), B, H, nQ, nK, _ptr(row_loads, torch.int32, "row_loads"),
        _ptr(col_loads, torch.int32, "col_loads"), _ptr(head_loads, torch.int32, "head_loads", True),
        _stream(stream))
    _check(st, "dbsp_block_mask_loads")


def dbsp_block_mask_loads_causal(mask, row_loads, col_loads, head_loads=None, stream=None):
    """As dbsp_block_mask_loads, counting only the blocks on or below the diagonal (nQ == nK)."""
    B, H, nQ, nK = mask.shape
    st = library().dbsp_block_mask_loads_causal(
        _ptr(mask, torch.uint8, "mask"), B, H, nQ, nK, _ptr(row_loads, torch.int32, "row_loads"),
        _ptr(col_loads, torch.int32, "col_loads"), _ptr(head_loads, torch.int32, "head_loads", True),
        _stream(stream))
    _check(st, "dbsp_block_mask_loads_causal")


def dbsp_shard_masks(mask, shard_of, n_shards, out=None, stream=None):
    """mask uint8 [B,H,nQ,nK], shard_of int32 [nK] -> uint8 [n_shards,B,H,nQ,nK]: each shard's KV blocks only."""
    B, H, nQ, nK = mask.shape
    if out is None:
        out = torch.empty((n_shards, B, H, nQ, nK), dtype=torch.uint8, device=mask.device)
    st = library().dbsp_shard_masks(_ptr(mask, torch.uint8, "mask"), B, H, nQ, nK,
                                    _ptr(shard_of, torch.int32, "shard_of"), int(n_shards),
                                    _ptr(out, torch.uint8, "out"), _stream(stream))
    _check(st, "dbsp_shard_masks")
    return out


def dbsp_kv_block_loads(col_loads, kv_loads, stream=None):
    """col_loads int32 [..., nK] (every leading dim a group) -> kv_loads int32 [nK], summed over groups."""
    nK = col_loads.shape[-1]
    groups = col_loads.numel() // nK
    st = library().dbsp_kv_block_loads(_ptr(col_loads, torch.int32, "col_loads"), groups, nK,
                                       _ptr(kv_loads, torch.int32, "kv_loads"), _stream(stream))
    _check(st, "dbsp_kv_block_loads")


def dbsp_plan_lpt(loads, n_workers, worker_of, worker_offsets, worklist, worker_loads=None,
                  home=None, stay_bonus=0, stream=None):
    """LPT plan: loads int32 [n] -> worker_of [n], worker_offsets [m+1], worklist [n], worker_loads int64 [m]."""
    n = loads.numel()
    st = library().dbsp_plan_lpt(
        _ptr(loads, torch.int32, "loads"), _ptr(home, torch.int32, "home", True), n, n_workers,
        int(stay_bonus), _ptr(worker_of, torch.int32, "worker_of"),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        _ptr(worker_loads, torch.int64, "worker_loads", True), _stream(stream))
    _check(st, "dbsp_plan_lpt")


def dbsp_plan_lpt_cost(loads, n_workers, block_cost, item_cost, worker_of, worker_offsets, worklist,
                       worker_loads=None, home=None, stay_bonus=0, stream=None):
    """LPT plan over planning loads ``loads * block_cost + item_cost`` (same outputs as dbsp_plan_lpt)."""
    n = loads.numel()
    st = library().dbsp_plan_lpt_cost(
        _ptr(loads, torch.int32, "loads"), _ptr(home, torch.int32, "home", True), n, n_workers,
        int(stay_bonus), int(block_cost), int(item_cost), _ptr(worker_of, torch.int32, "worker_of"),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        _ptr(worker_loads, torch.int64, "worker_loads", True), _stream(stream))
    _check(st, "dbsp_plan_lpt_cost")


def dbsp_block_sparse_attn_fwd(q, k, v, mask, block, causal, worker_offsets, worklist, n_workers,
                               out=None, lse=None, o_part=None, m_part=None, l_part=None,
                               scale=0.0, cta_timing=None, stream=None):
    """Block-sparse attention forward over a CSR worklist (final or partial mode)."""
    B, H, S, d = q.shape
    st = library().dbsp_block_sparse_attn_fwd(
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        _ptr(mask, torch.uint8, "mask"), B, H, S, d, block, int(bool(causal)), float(scale),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        n_workers, _ptr(out, torch.bfloat16, "out", True), _ptr(lse, torch.float32, "lse", True),
        _ptr(o_part, torch.float32, "o_part", True), _ptr(m_part, torch.float32, "m_part", True),
        _ptr(l_part, torch.float32, "l_part", True), _ptr(cta_timing, torch.int64, "cta_timing", True),
        _stream(stream))
    _check(st, "dbsp_block_sparse_attn_fwd")


def dbsp_dense_block_lists(mask, causal=False, counts=None, cols=None, stream=None):
    """Dense-block lists of every mask row: counts int32 [B,H,nQ], cols int16 [B,H,nQ,nK]
    (the KV-block indices as 16-bit words, ascending; entries past the count unwritten)."""
    B, H, nQ, nK = mask.shape
    if counts is None:
        counts = torch.empty((B, H, nQ), dtype=torch.int32, device=mask.device)
    if cols is None:
        cols = torch.empty((B, H, nQ, nK), dtype=torch.int16, device=mask.device)
    st = library().dbsp_dense_block_lists(
        _ptr(mask, torch.uint8, "mask"), B, H, nQ, nK, int(bool(causal)), _ptr(counts, torch.int32, "counts"),
        _ptr(cols, torch.int16, "cols"), _stream(stream))
    _check(st, "dbsp_dense_block_lists")
    return counts, cols


def dbsp_block_sparse_attn_fwd_listed(q, k, v, mask, block, causal, worker_offsets, worklist, n_workers,
                                      dense_n, dense_cols, out=None, lse=None, o_part=None, m_part=None,
                                      l_part=None, scale=0.0, cta_timing=None, stream=None):
    """dbsp_block_sparse_attn_fwd reading each item's dense blocks from dbsp_dense_block_lists."""
    B, H, S, d = q.shape
    st = library().dbsp_block_sparse_attn_fwd_listed(
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        _ptr(mask, torch.uint8, "mask"), B, H, S, d, block, int(bool(causal)), float(scale),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        n_workers, _ptr(dense_n, torch.int32, "dense_n"), _ptr(dense_cols, torch.int16, "dense_cols"),
        _ptr(out, torch.bfloat16, "out", True), _ptr(lse, torch.float32, "lse", True),
        _ptr(o_part, torch.float32, "o_part", True), _ptr(m_part, torch.float32, "m_part", True),
        _ptr(l_part, torch.float32, "l_part", True), _ptr(cta_timing, torch.int64, "cta_timing", True),
        _stream(stream))
    _check(st, "dbsp_block_sparse_attn_fwd_listed")


def dbsp_merge_partials(o_parts, m_parts, l_parts, out, lse=None, stream=None):
    """o_parts fp32 [n, rows, d], m/l fp32 [n, rows] -> out bf16 [rows, d], lse fp32 [rows]."""
    n, rows, d = o_parts.shape
    st = library().dbsp_merge_partials(
        _ptr(o_parts, torch.float32, "o_parts"), _ptr(m_parts, torch.float32, "m_parts"),
        _ptr(l_parts, torch.float32, "l_parts"), n, rows, d, _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse", True), _stream(stream))
    _check(st, "dbsp_merge_partials")


def dbsp_plan_lpt_cost_n(loads, n_items_dev, n_workers, block_cost, item_cost, worker_of, worker_offsets,
                         worklist, worker_loads=None, stream=None):
    """LPT over the first ``n_items_dev[0]`` (device int32) of ``loads`` (capacity loads.numel())."""
    st = library().dbsp_plan_lpt_cost_n(
        _ptr(loads, torch.int32, "loads"), _ptr(n_items_dev, torch.int32, "n_items_dev"), loads.numel(),
        n_workers, int(block_cost), int(item_cost), _ptr(worker_of, torch.int32, "worker_of"),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        _ptr(worker_loads, torch.int64, "worker_loads", True), _stream(stream))
    _check(st, "dbsp_plan_lpt_cost_n")


def dbsp_split_plan(loads, n_workers, max_piece_load, max_pieces, max_slots, unit_item, unit_pk, unit_slot,
                    unit_load, split_item, split_off, counts, stream=None):
    """Unit table of heavy items split along their KV blocks (int32 outputs, counts [5])."""
    st = library().dbsp_split_plan(
        _ptr(loads, torch.int32, "loads"), loads.numel(), n_workers, int(max_piece_load), int(max_pieces),
        int(max_slots), _ptr(unit_item, torch.int32, "unit_item"), _ptr(unit_pk, torch.int32, "unit_pk"),
        _ptr(unit_slot, torch.int32, "unit_slot"), _ptr(unit_load, torch.int32, "unit_load"),
        _ptr(split_item, torch.int32, "split_item"), _ptr(split_off, torch.int32, "split_off"),
        _ptr(counts, torch.int32, "counts"), _stream(stream))
    _check(st, "dbsp_split_plan")


def dbsp_block_sparse_attn_fwd_units(q, k, v, mask, block, causal, worker_offsets, worklist, n_workers,
                                     unit_item, unit_pk, unit_slot, out, lse, o_piece, m_piece, l_piece,
                                     scale=0.0, cta_timing=None, stream=None):
    """Attention over a worklist of units: whole items to out/lse, pieces to o/m/l_piece slots."""
    B, H, S, d = q.shape
    st = library().dbsp_block_sparse_attn_fwd_units(
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        _ptr(mask, torch.uint8, "mask"), B, H, S, d, block, int(bool(causal)), float(scale),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        n_workers, _ptr(unit_item, torch.int32, "unit_item"), _ptr(unit_pk, torch.int32, "unit_pk"),
        _ptr(unit_slot, torch.int32, "unit_slot"), unit_item.numel(), _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse", True), _ptr(o_piece, torch.float32, "o_piece"),
        _ptr(m_piece, torch.float32, "m_piece"), _ptr(l_piece, torch.float32, "l_piece"),
        m_piece.shape[0] if m_piece.dim() == 2 else m_piece.numel() // block,
        _ptr(cta_timing, torch.int64, "cta_timing", True), _stream(stream))
    _check(st, "dbsp_block_sparse_attn_fwd_units")


def dbsp_merge_pieces(o_piece, m_piece, l_piece, split_item, split_off, counts, out, lse=None, block=128,
                      stream=None):
    """Combine the pieces of every split item into out bf16 [B,H,S,d] (and lse fp32 [B,H,S]).

    The piece buffers' capacity (slots) is taken from ``m_piece`` ([max_slots, block])."""
    B, H, S, d = out.shape
    max_slots = m_piece.shape[0] if m_piece.dim() == 2 else m_piece.numel() // block
    st = library().dbsp_merge_pieces(
        _ptr(o_piece, torch.float32, "o_piece"), _ptr(m_piece, torch.float32, "m_piece"),
        _ptr(l_piece, torch.float32, "l_piece"), _ptr(split_item, torch.int32, "split_item"),
        _ptr(split_off, torch.int32, "split_off"), _ptr(counts, torch.int32, "counts"), max_slots, B, H, S, d,
        block,
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse", True), _stream(stream))
    _check(st, "dbsp_merge_pieces")


def dbsp_block_sparse_attn_fwd_split_noalloc(q, k, v, mask, block, causal, worker_offsets, worklist, n_workers,
                                             unit_item, unit_pk, unit_slot, split_item, split_off, counts,
                                             max_slots, out, lse=None, scale=0.0, cta_timing=None, stream=None):
    """Split attention (units, then the piece merge) with the pieces in the library's static
    device scratch: nothing is allocated. ``max_slots`` is the piece capacity of the split
    plan; max_slots * block * (d + 2) * 4 bytes must fit DBSP_NOALLOC_SCRATCH_BYTES."""
    B, H, S, d = q.shape
    need = max_slots * block * (d + 2) * 4
    if need > DBSP_NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"max_slots={max_slots} needs {need} bytes of piece scratch; the static scratch holds "
                         f"{DBSP_NOALLOC_SCRATCH_BYTES}")
    st = library().dbsp_block_sparse_attn_fwd_split_noalloc(
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        _ptr(mask, torch.uint8, "mask"), B, H, S, d, block, int(bool(causal)), float(scale),
        _ptr(worker_offsets, torch.int32, "worker_offsets"), _ptr(worklist, torch.int32, "worklist"),
        n_workers, _ptr(unit_item, torch.int32, "unit_item"), _ptr(unit_pk, torch.int32, "unit_pk"),
        _ptr(unit_slot, torch.int32, "unit_slot"), unit_item.numel(), _ptr(split_item, torch.int32, "split_item"),
        _ptr(split_off, torch.int32, "split_off"), _ptr(counts, torch.int32, "counts"), int(max_slots),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse", True),
        _ptr(cta_timing, torch.int64, "cta_timing", True), _stream(stream))
    _check(st, "dbsp_block_sparse_attn_fwd_split_noalloc")


def dbsp_device_status(stream=None):
    """Synchronise the stream and return (and clear) the device error word."""
    return library().dbsp_device_status(_stream(stream))
