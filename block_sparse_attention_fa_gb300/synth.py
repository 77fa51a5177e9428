"""Seeded synthetic inputs for block-sparse attention workloads.

This module only draws random numbers and lays out workload descriptions
(shapes, segment ids, ALiBi slopes).  It holds none of the attention
arithmetic: both the CUDA path and the CPU oracle consume what it produces,
so the two always see bit-identical inputs.

Workloads (all tensors are ``[B, H, T, D]`` contiguous, ``D`` innermost):

* ``grouped_fp32``   -- grouped variate attention, fp32, B=1 H=4 D=128,
  8 groups x 17 variates = 136 tokens, segment id = token // 17
  (TiRex2 PR "perf: expose FlexAttention loader override", sections
  "Performance characterization" and "Variate-attention layer": one target
  plus 16 covariates per window, embedding 512 over four heads).
* ``grouped_bf16``   -- the same group structure at scale, bf16,
  4096 groups x 17 = 69632 tokens.
* ``document_bf16``  -- document packing, bf16, B=4 H=16 D=64 T=8192,
  document lengths uniform in [256, 2048], the last one truncated
  (FlexAttention Guide, "Production Engineering", item 1).
* ``causal_softcap_bf16`` -- causal + tanh soft-cap C=50, bf16, B=8 H=16
  D=128 T=4096, inputs scaled by 2 so that the cap is active (FlexAttention
  Guide, "The Problem" soft-capping formula and the implementation script).
* ``window_alibi_gqa_bf16`` -- causal sliding window 1024 + ALiBi, GQA
  32 query / 8 KV heads, D=128, T=32768.

Reading of the ALiBi slopes: the slopes form the geometric sequence
``2^(-8 (h+1) / H)`` over 0-based query heads ``h`` (Press et al., as cited
by the FlexAttention Guide); a literal 0-based ``2^(-8h/H)`` would give
head 0 the slope 1 and no head the slope ``2^-8``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

BLOCK = 128


def standard_normal(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """fp32 N(0, scale^2) samples from numpy's PCG64 stream for ``seed``."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=int(np.prod(shape)), dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x.reshape(shape)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value (ties to even), kept in fp32.

    The result is exactly representable in bf16, so converting it to a bf16
    tensor is lossless and the oracle sees the very values the GPU sees.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def group_segments(T: int, group: int) -> np.ndarray:
    """Segment id ``t // group`` for every token (one variate group each)."""
    return (np.arange(T, dtype=np.int64) // group).astype(np.int32)


def document_segments(seed: int, B: int, T: int, lo: int = 256, hi: int = 2048) -> np.ndarray:
    """Per batch row, documents of length U{lo..hi} packed until T tokens.

    Lengths are drawn from a seeded stream until they cover ``T``; the last
    document is truncated.  Ids are 0, 1, 2, ... in packing order, so every
    row is non-decreasing.
    """
    rng = np.random.default_rng(seed)
    seg = np.empty((B, T), dtype=np.int32)
    for b in range(B):
        pos, doc = 0, 0
        while pos < T:
            n = int(rng.integers(lo, hi + 1))
            seg[b, pos:min(T, pos + n)] = doc
            pos += n
            doc += 1
    return seg


def tree_table(seed: int, B: int, context: int, n_tree: int) -> np.ndarray:
    """Attend tables of speculative-decoding candidate trees (tree attention).

    Per batch row, a tree of ``n_tree`` draft tokens: node 0 is the root and
    node k > 0 hangs under a parent drawn uniformly from [0, k).  The queries
    are the tree nodes (q_len = n_tree), the keys the ``context`` tokens
    followed by the tree nodes (kv_len = context + n_tree).  Query k sees every
    context key and the tree keys of its ancestors and itself.  Returns bool
    [B, n_tree, context + n_tree].
    """
    rng = np.random.default_rng(seed)
    t = np.zeros((B, n_tree, context + n_tree), dtype=bool)
    t[:, :, :context] = True
    for b in range(B):
        parent = [-1] + [int(rng.integers(0, k)) for k in range(1, n_tree)]
        for k in range(n_tree):
            a = k
            while a >= 0:
                t[b, k, context + a] = True
                a = parent[a]
    return t


def pack_table(table: np.ndarray) -> np.ndarray:
    """A bool attend table [batch, q_len, kv_len] in the C ABI's packed form:
    int32 [batch, q_len, ceil(kv_len / 32)], bit j % 32 (least significant
    first) of word j // 32."""
    t = np.asarray(table, dtype=bool)
    if t.ndim == 2:
        t = t[None]
    pad = (-t.shape[2]) % 32
    t = np.concatenate([t, np.zeros(t.shape[:2] + (pad,), bool)], axis=2)
    bits = t.reshape(t.shape[0], t.shape[1], -1, 32).astype(np.uint64)
    words = (bits << np.arange(32, dtype=np.uint64)).sum(axis=3).astype(np.uint32)
    return words.view(np.int32)


def alibi_slopes(H: int) -> np.ndarray:
    """Geometric ALiBi slopes ``2^(-8 (h+1) / H)`` for query heads h = 0..H-1."""
    h = np.arange(H, dtype=np.float64)
    return np.exp2(-8.0 * (h + 1.0) / H).astype(np.float32)


def composite_slopes(H: int) -> np.ndarray:
    """Slopes ``linspace(0.1, 0.8, H)``, as the guide's composite ALiBi +
    soft-cap example draws them."""
    return np.linspace(0.1, 0.8, H, dtype=np.float64).astype(np.float32)


@dataclasses.dataclass
class Workload:
    """A seeded synthetic attention problem (shapes, mask and score_mod)."""

    name: str
    dtype: str                 # "bf16" or "fp32"
    B: int
    Hq: int
    Hkv: int
    T: int
    D: int
    mask: str                  # "full" | "causal" | "sliding_window" | "document" | "prefix_lm"
    score: str = "none"        # "none" | "softcap" | "alibi" | "rel_bias"
    window: int = 0
    prefix_len: int = 0
    softcap: float = 0.0
    group: int = 0             # document mask from token // group
    doc_lo: int = 256
    doc_hi: int = 2048
    rel_max: int = 0
    input_scale: float = 1.0
    seed: int = 0
    groups: Optional[int] = None   # number of independent windows (grouped workloads)
    q_len: Optional[int] = None    # query rows when they differ from T (decoding shapes)
    tree: int = 0                  # table mask: candidate trees of this many tokens after T - tree context keys

    @property
    def Tq(self) -> int:
        return self.q_len or self.T

    @property
    def kv_len(self) -> int:
        return self.T

    def segments(self) -> Optional[np.ndarray]:
        """int32 [Bs, T] segment ids for document masks, else None."""
        if self.mask != "document":
            return None
        if self.group > 0:
            return group_segments(self.T, self.group)[None, :].copy()
        return document_segments(self.seed + 1000, self.B, self.T, self.doc_lo, self.doc_hi)

    def table(self) -> Optional[np.ndarray]:
        """bool [B, Tq, T] attend table for table masks (candidate trees)."""
        if self.mask != "table":
            return None
        return tree_table(self.seed + 3000, self.B, self.T - self.tree, self.tree)

    def slopes(self) -> Optional[np.ndarray]:
        if self.score == "alibi":
            return alibi_slopes(self.Hq)
        if self.score == "alibi_softcap":
            return composite_slopes(self.Hq)
        return None

    def rel_bias(self) -> Optional[np.ndarray]:
        """fp32 [Hq, 2R+1] relative-position bias table (seeded)."""
        if self.score != "rel_bias":
            return None
        return standard_normal(self.seed + 2000, (self.Hq, 2 * self.rel_max + 1), 0.5)

    def qkv(self):
        """(q, k, v) fp32 numpy arrays; bf16 workloads are pre-rounded to bf16."""
        q = standard_normal(self.seed * 3 + 0, (self.B, self.Hq, self.Tq, self.D), self.input_scale)
        k = standard_normal(self.seed * 3 + 1, (self.B, self.Hkv, self.T, self.D), self.input_scale)
        v = standard_normal(self.seed * 3 + 2, (self.B, self.Hkv, self.T, self.D), self.input_scale)
        if self.dtype == "bf16":
            q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
        return q, k, v

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (for downscaled parity cases)."""
        return dataclasses.replace(self, **kw)


# Decoding shapes for the split-KV forward (fa_fwd_decode): a few query rows
# per (batch, query head) against a long key/value sequence; every key
# visible.  GQA 32 / 8 and T = 32768 as the window workload.
DECODE_WORKLOADS = {
    "decode_gqa_bf16": Workload(
        name="decode_gqa_bf16", dtype="bf16", B=8, Hq=32, Hkv=8, T=32768, D=128,
        mask="full", seed=6, q_len=1),
    "decode_spec4_bf16": Workload(
        name="decode_spec4_bf16", dtype="bf16", B=8, Hq=32, Hkv=8, T=32768, D=128,
        mask="full", seed=7, q_len=4),
    # tree attention: a 4-token candidate tree per sequence after 32768
    # context tokens, its tokens querying the context and their ancestors
    "decode_tree_bf16": Workload(
        name="decode_tree_bf16", dtype="bf16", B=8, Hq=32, Hkv=8, T=32768 + 4, D=128,
        mask="table", seed=9, q_len=4, tree=4),
}

WORKLOADS = {
    "grouped_fp32": Workload(
        name="grouped_fp32", dtype="fp32", B=1, Hq=4, Hkv=4, T=136, D=128,
        mask="document", group=17, seed=1, groups=8),
    "grouped_bf16": Workload(
        name="grouped_bf16", dtype="bf16", B=1, Hq=4, Hkv=4, T=69632, D=128,
        mask="document", group=17, seed=2, groups=4096),
    "document_bf16": Workload(
        name="document_bf16", dtype="bf16", B=4, Hq=16, Hkv=16, T=8192, D=64,
        mask="document", seed=3),
    "causal_softcap_bf16": Workload(
        name="causal_softcap_bf16", dtype="bf16", B=8, Hq=16, Hkv=16, T=4096, D=128,
        mask="causal", score="softcap", softcap=50.0, input_scale=2.0, seed=4),
    "window_alibi_softcap_bf16": Workload(
        name="window_alibi_softcap_bf16", dtype="bf16", B=2, Hq=8, Hkv=8, T=4096, D=64,
        mask="sliding_window", window=512, score="alibi_softcap", softcap=50.0, seed=8),
    "window_alibi_gqa_bf16": Workload(
        name="window_alibi_gqa_bf16", dtype="bf16", B=1, Hq=32, Hkv=8, T=32768, D=128,
        mask="sliding_window", window=1024, score="alibi", seed=5),
}
