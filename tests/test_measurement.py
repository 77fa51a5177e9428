"""The benchmark's work counts, checked on small cases without a GPU.

bench.py reports visited-tile FLOPs (4 r c D per visited tile per (b, hq)),
algorithmic bytes and the decoding bytes; these tests recount them by brute
force from the oracle's BlockMask and from the tensor shapes, so that a
roofline fraction is only ever algorithmic work over time.  Also the packed
table layout the tests and bench hand to the C ABI.
"""
import numpy as np
import pytest

import bench
import oracle
from block_sparse_attention_fa_gb300 import synth


@pytest.mark.parametrize("mask,kw,T", [("causal", {}, 300), ("sliding_window", {"window": 100}, 520),
                                       ("full", {}, 129), ("document", {"doc_lo": 20, "doc_hi": 90}, 400)])
def test_visited_flops_is_the_tile_sum(mask, kw, T):
    w = synth.Workload(name="m", dtype="bf16", B=2, Hq=4, Hkv=2, T=T, D=64, mask=mask, seed=3, **kw)
    seg = w.segments()
    bm = oracle.block_mask(mask=mask, B=seg.shape[0] if seg is not None else 1, H=1, q_len=T, kv_len=T,
                           window=w.window, seg=seg)
    total = 0
    nq = bm["kv_num_blocks"].shape[-1]
    for b in range(bm["kv_num_blocks"].shape[0]):
        for qb in range(nq):
            r = min(128, T - 128 * qb)
            for key in ("kv", "full_kv"):
                n = bm[f"{key}_num_blocks"][b, 0, qb]
                for kb in bm[f"{key}_indices"][b, 0, qb, :n]:
                    c = min(128, T - 128 * int(kb))
                    total += 4 * r * c * w.D
    reps = (w.B // bm["kv_num_blocks"].shape[0]) * w.Hq
    assert bench.visited_flops(w, bm) == pytest.approx(total * reps, rel=1e-12)


def test_byte_counts():
    w = synth.WORKLOADS["causal_softcap_bf16"]
    # Q, K, V read and O written in bf16, lse in fp32
    assert bench.algorithmic_bytes(w) == 8 * 4096 * 128 * 2 * (16 + 16 + 16 + 16) + 8 * 16 * 4096 * 4
    d = synth.DECODE_WORKLOADS["decode_gqa_bf16"]
    # K and V once per (b, kv head); Q and O per query row; lse
    assert bench.decode_bytes(d) == 2 * 8 * 8 * 32768 * 128 * 2 + 2 * 8 * 32 * 1 * 128 * 2 + 8 * 32 * 1 * 4


def test_pack_table_bit_layout():
    rng = np.random.default_rng(1)
    t = rng.random((2, 5, 70)) < 0.5
    w = synth.pack_table(t).view(np.uint32)
    assert w.shape == (2, 5, 3)
    for b in range(2):
        for i in range(5):
            for j in range(70):
                assert bool((int(w[b, i, j // 32]) >> (j % 32)) & 1) == t[b, i, j]
            for j in range(70, 96):                      # padding bits are clear
                assert not (int(w[b, i, j // 32]) >> (j % 32)) & 1
