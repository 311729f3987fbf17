"""Seeded synthetic inputs for the block-sparse attention path.

This module only *generates inputs*: block masks, Q/K/V tensors and KV-shard
column restrictions. It computes nothing of the method itself (no loads, no
planning, no softmax), so both the CUDA path and the CPU oracle can consume what
it makes. It imports neither.

The workloads are synthetic stand-ins shaped like the ones the source pages talk
about (db-SP blog, scenario 1: LLM heads that look globally or locally, video
heads that look within a frame or across frames; DSP notes: spatial and temporal
stages of video transformers). No dataset is involved.

Masks use ``numpy.random.default_rng(seed)`` (PCG64). Q/K/V are N(0, 1) rounded to
bf16 (round-to-nearest-even): the tiny workload draws them with numpy, larger ones
with ``torch.randn`` on a seeded generator on the requested device.
"""

from dataclasses import dataclass, field
import math

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    d: int
    block: int
    causal: bool
    mask_seed: int
    qkv_seed: int
    kind: str
    extra: dict = field(default_factory=dict)

    @property
    def nQ(self):
        return self.S // self.block

    @property
    def nK(self):
        return self.S // self.block

    @property
    def n_items(self):
        return self.B * self.H * self.nQ

    def describe(self):
        return (f"{self.name}: B={self.B} H={self.H} S={self.S} d={self.d} "
                f"block={self.block} causal={int(self.causal)} mask={self.kind}")


WORKLOADS = {
    # 8x8 block mask per head, Bernoulli(0.5), diagonal forced, non-causal.
    "tiny": Workload("tiny", 1, 2, 512, 64, 64, False, 0, 100, "bernoulli",
                     {"p": 0.5}),
    # LLM heads: 16 "global" heads Bernoulli(0.9) below the diagonal, 16 "local"
    # heads = sliding window of 4 blocks (diagonal included) plus block-0 sink.
    "llm": Workload("llm", 1, 32, 8192, 128, 128, True, 2, 102, "llm",
                    {"p_global": 0.9, "window": 4, "n_global": 16}),
    # Video-DiT heads: 16 frames x 1024 tokens; 12 spatial heads keep same-frame
    # blocks, 12 temporal heads keep equal in-frame offsets; each head ORs in
    # Bernoulli(rho_h) with rho_h ~ U[0.05, 0.40].
    "video": Workload("video", 1, 24, 16384, 128, 128, False, 3, 103, "video",
                      {"frames": 16, "tokens_per_frame": 1024, "n_spatial": 12,
                       "rho_lo": 0.05, "rho_hi": 0.40}),
    # Sharded-KV merge: full causal mask; 8 contiguous or 8 striped KV shards.
    "sharded": Workload("sharded", 1, 16, 32768, 128, 128, True, 4, 104, "causal_full",
                        {"n_shards": 8}),
    # Imbalance stress: per-head density lognormal(ln 0.1, 1) clipped to
    # [1%, 60%]; each row keeps the diagonal plus uniformly drawn blocks.
    "imbalance": Workload("imbalance", 1, 40, 131072, 128, 128, False, 5, 105, "lognormal",
                          {"mu": math.log(0.1), "sigma": 1.0, "lo": 0.01, "hi": 0.60}),
}

ORDER = ["tiny", "llm", "video", "sharded", "imbalance"]


def custom(name, B, H, S, d, block, causal, mask_seed, qkv_seed, kind="bernoulli", **extra):
    """A workload with explicit sizes (for multi-tile / ragged parity cases)."""
    return Workload(name, B, H, S, d, block, causal, mask_seed, qkv_seed, kind, dict(extra))


def _force_diagonal(m):
    n = min(m.shape[-2], m.shape[-1])
    idx = np.arange(n)
    m[..., idx, idx] = 1
    return m


def _causal_clip(m):
    nQ, nK = m.shape[-2], m.shape[-1]
    keep = np.arange(nK)[None, :] <= np.arange(nQ)[:, None]
    return m * keep.astype(m.dtype)


def make_mask(w):
    """uint8 block mask [B, H, nQ, nK] for workload ``w`` (seeded)."""
    rng = np.random.default_rng(w.mask_seed)
    B, H, nQ, nK = w.B, w.H, w.nQ, w.nK
    x = w.extra
    if w.kind == "bernoulli":
        m = (rng.random((B, H, nQ, nK)) < x.get("p", 0.5)).astype(np.uint8)
        if x.get("diag", True):
            m = _force_diagonal(m)
    elif w.kind == "llm":
        m = np.zeros((B, H, nQ, nK), dtype=np.uint8)
        i = np.arange(nQ)[:, None]
        j = np.arange(nK)[None, :]
        local = ((j <= i) & (j > i - x["window"])) | (j == 0)
        for b in range(B):
            for h in range(H):
                if h < x["n_global"]:
                    g = (rng.random((nQ, nK)) < x["p_global"]) & (j < i)
                    m[b, h] = (g | (j == i)).astype(np.uint8)
                else:
                    m[b, h] = local.astype(np.uint8)
    elif w.kind == "video":
        per_frame = x["tokens_per_frame"] // w.block
        i = np.arange(nQ)[:, None]
        j = np.arange(nK)[None, :]
        spatial = (i // per_frame) == (j // per_frame)
        temporal = (i % per_frame) == (j % per_frame)
        rho = rng.uniform(x["rho_lo"], x["rho_hi"], size=(B, H))
        m = np.zeros((B, H, nQ, nK), dtype=np.uint8)
        for b in range(B):
            for h in range(H):
                base = spatial if h < x["n_spatial"] else temporal
                extra = rng.random((nQ, nK)) < rho[b, h]
                m[b, h] = (base | extra).astype(np.uint8)
    elif w.kind == "causal_full":
        tril = np.tril(np.ones((nQ, nK), dtype=np.uint8))
        m = np.broadcast_to(tril, (B, H, nQ, nK)).copy()
    elif w.kind == "lognormal":
        rho = np.clip(rng.lognormal(mean=x["mu"], sigma=x["sigma"], size=(B, H)),
                      x["lo"], x["hi"])
        keep = np.maximum(1, np.rint(rho * nK)).astype(np.int64)
        m = np.zeros((B, H, nQ, nK), dtype=np.uint8)
        diag = np.arange(min(nQ, nK))
        for b in range(B):
            for h in range(H):
                # uniform choice without replacement: the k_h smallest of i.i.d.
                # uniform keys per row, with the diagonal forced first
                keys = rng.random((nQ, nK))
                keys[diag, diag] = -1.0
                k = int(keep[b, h])
                sel = np.argpartition(keys, k - 1, axis=1)[:, :k]
                np.put_along_axis(m[b, h], sel, 1, axis=1)
    else:
        raise ValueError(f"unknown mask kind {w.kind!r}")
    if w.causal:
        m = _causal_clip(m)
    return np.ascontiguousarray(m, dtype=np.uint8)


def perturb_mask(mask, frac, seed, causal):
    """The next step's mask: every block flipped (dense <-> empty) with probability
    ``frac``, seeded; blocks above the diagonal stay empty when ``causal``."""
    rng = np.random.default_rng(seed)
    flip = rng.random(mask.shape) < frac
    m = np.where(flip, 1 - (mask != 0), mask != 0).astype(np.uint8)
    if causal:
        m = _causal_clip(m)
    return np.ascontiguousarray(m)


def shard_columns(nK, n_shards, layout):
    """KV-block column ids of each shard.

    contiguous: shard s owns blocks [s*nK/n, (s+1)*nK/n); striped: blocks j with
    j mod n == s (the block-granular reading of striping, 6D attention notes §2.3).
    """
    if layout == "contiguous":
        edges = [(s * nK) // n_shards for s in range(n_shards + 1)]
        return [np.arange(edges[s], edges[s + 1]) for s in range(n_shards)]
    if layout == "striped":
        return [np.arange(s, nK, n_shards) for s in range(n_shards)]
    raise ValueError(layout)


def shard_masks(mask, n_shards, layout):
    """uint8 [n_shards, B, H, nQ, nK]: ``mask`` restricted to each shard's columns."""
    nK = mask.shape[-1]
    out = np.zeros((n_shards,) + mask.shape, dtype=np.uint8)
    for s, cols in enumerate(shard_columns(nK, n_shards, layout)):
        out[s][..., cols] = mask[..., cols]
    return out


def make_qkv_numpy(w):
    """(q, k, v) as numpy float32 arrays holding bf16-representable values.

    N(0, 1) from ``default_rng(qkv_seed)``, rounded to bf16 with torch (RNE).
    """
    import torch

    rng = np.random.default_rng(w.qkv_seed)
    shape = (w.B, w.H, w.S, w.d)
    out = []
    for _ in range(3):
        x = rng.standard_normal(shape, dtype=np.float32)
        out.append(torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy())
    return tuple(out)


def make_qkv(w, device="cpu"):
    """(q, k, v) bf16 torch tensors [B, H, S, d] on ``device``.

    The tiny workload (and any workload with ``extra['numpy_qkv']``) uses the numpy
    stream so that its values are identical on every machine; the others use
    ``torch.randn`` with a generator seeded by ``qkv_seed`` on ``device``.
    """
    import torch

    if w.name == "tiny" or w.extra.get("numpy_qkv", False):
        return tuple(torch.from_numpy(a).to(torch.bfloat16).to(device) for a in make_qkv_numpy(w))
    g = torch.Generator(device=device)
    g.manual_seed(w.qkv_seed)
    shape = (w.B, w.H, w.S, w.d)
    return tuple(torch.randn(shape, generator=g, device=device, dtype=torch.float32)
                 .to(torch.bfloat16) for _ in range(3))


def ramp_key_blocks(k, block, step):
    """Keys of KV-block j multiplied by (1 + step * j), rounded to bf16 (RNE).

    Later KV-blocks then score higher, so a query row's running maximum keeps growing
    from one dense block to the next: inputs that drive the online softmax through its
    rescaling step. ``k`` is a bf16 tensor [B, H, S, d]; the result is a new one.
    """
    import torch

    S = k.shape[2]
    factor = 1.0 + step * (torch.arange(S, device=k.device, dtype=torch.float32) // block)
    return (k.float() * factor.view(1, 1, S, 1)).to(torch.bfloat16)

