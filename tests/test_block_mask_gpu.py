"""GPU BlockMask builder vs the oracle's brute-force tile scan: bit-exact on
every array (counts, ascending indices, -1 padding), through the C ABI; and
the transposed lists (fa_block_mask_build_cols) bit-exact against a
brute-force transpose of the oracle's lists."""
import numpy as np
import pytest

import oracle
from block_sparse_attention_fa_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import torch
    from block_sparse_attention_fa_gb300 import fa as fam
    assert torch.cuda.is_available()
    fam.load_library()
    return fam


def transpose_lists(want):
    """The transposed BlockMask by brute force from the oracle's lists: for
    each kv block, the q-blocks whose row lists it as partial / full,
    ascending, -1 padded."""
    B, H, nq, nkv = want["kv_indices"].shape
    out = {"q_num_blocks": np.zeros((B, H, nkv), np.int32), "q_indices": np.full((B, H, nkv, nq), -1, np.int32),
           "full_q_num_blocks": np.zeros((B, H, nkv), np.int32),
           "full_q_indices": np.full((B, H, nkv, nq), -1, np.int32)}
    for b in range(B):
        for h in range(H):
            for src_n, src_i, dst_n, dst_i in (("kv_num_blocks", "kv_indices", "q_num_blocks", "q_indices"),
                                               ("full_kv_num_blocks", "full_kv_indices", "full_q_num_blocks",
                                                "full_q_indices")):
                cols = [[] for _ in range(nkv)]
                for qb in range(nq):
                    for kb in want[src_i][b, h, qb, :want[src_n][b, h, qb]]:
                        cols[kb].append(qb)
                for kb in range(nkv):
                    out[dst_n][b, h, kb] = len(cols[kb])
                    out[dst_i][b, h, kb, :len(cols[kb])] = cols[kb]
    return out


def _check_cols(fa, bm, want, label):
    import torch
    got = {k: v.cpu().numpy() for k, v in bm.cols().items()}
    fa.default_workspace(torch.device("cuda")).check()
    exp = transpose_lists(want)
    for key in exp:
        np.testing.assert_array_equal(got[key], exp[key], err_msg=f"{label} transposed {key}")


def _build_both(fa, mask, B, H, q_len, kv_len, window=0, prefix_len=0, seg=None):
    import torch
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    bm = fa.block_mask(mask, B, H, q_len, kv_len, window=window, prefix_len=prefix_len, seg_ids=seg_t)
    fa.default_workspace(torch.device("cuda")).check()
    got = bm.numpy()
    want = oracle.block_mask(mask=mask, B=B, H=H, q_len=q_len, kv_len=kv_len, window=window,
                             prefix_len=prefix_len, seg=seg)
    for key in want:
        np.testing.assert_array_equal(got[key], want[key], err_msg=f"{mask} {key}")
    _check_cols(fa, bm, want, mask)
    return got


@pytest.mark.parametrize("T", [1, 17, 127, 128, 129, 136, 300, 1000, 2049])
@pytest.mark.parametrize("mask,kw", [
    ("full", {}), ("causal", {}), ("sliding_window", {"window": 0}), ("sliding_window", {"window": 127}),
    ("sliding_window", {"window": 128}), ("sliding_window", {"window": 300}),
    ("prefix_lm", {"prefix_len": 0}), ("prefix_lm", {"prefix_len": 200}), ("prefix_lm", {"prefix_len": 5000}),
])
def test_builder_matches_bruteforce(fa, T, mask, kw):
    _build_both(fa, mask, 1, 1, T, T, **kw)


@pytest.mark.parametrize("q_len,kv_len", [(200, 333), (333, 200), (64, 1000), (1000, 64)])
@pytest.mark.parametrize("mask,kw", [("full", {}), ("causal", {}), ("sliding_window", {"window": 100}),
                                     ("prefix_lm", {"prefix_len": 150})])
def test_builder_rectangular(fa, q_len, kv_len, mask, kw):
    _build_both(fa, mask, 1, 1, q_len, kv_len, **kw)


@pytest.mark.parametrize("T,lo,hi,B,H", [(136, 17, 17, 1, 4), (1000, 1, 40, 2, 1), (3000, 100, 700, 3, 2),
                                         (2048, 128, 128, 1, 1), (5000, 1, 5000, 2, 3)])
def test_builder_documents(fa, T, lo, hi, B, H):
    seg = synth.document_segments(T + lo + hi, B, T, lo, hi)
    _build_both(fa, "document", B, H, T, T, seg=seg)


def test_builder_shared_segments_broadcast(fa):
    seg = synth.group_segments(700, 17)[None, :].copy()
    _build_both(fa, "document", 3, 2, 700, 700, seg=seg)


def test_builder_rejects_unsorted_segments(fa):
    import torch
    seg = np.zeros((2, 500), np.int32)
    seg[1, 300:] = 1
    seg[1, 400] = 0                       # not non-decreasing in batch row 1
    bm = fa.block_mask("document", 2, 1, 500, 500, seg_ids=torch.from_numpy(seg).cuda())
    with pytest.raises(fa.FAError) as ei:
        fa.default_workspace(torch.device("cuda")).check()
    assert ei.value.status == fa.ERR_DEVICE_CHECK
    assert "row 1" in str(ei.value)
    fa.default_workspace(torch.device("cuda")).check()      # cleared


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_builder_full_size_workloads(fa, name):
    w = synth.WORKLOADS[name]
    seg = w.segments()
    got = _build_both(fa, w.mask, seg.shape[0] if seg is not None else 1, 1, w.T, w.T,
                      window=w.window, prefix_len=w.prefix_len, seg=seg)
    if name == "causal_softcap_bf16":
        assert got["full_kv_num_blocks"].sum() == 496 and got["kv_num_blocks"].sum() == 32
    if name == "window_alibi_gqa_bf16":
        assert got["full_kv_num_blocks"].sum() == 1764 and got["kv_num_blocks"].sum() == 504
    if name == "grouped_bf16":
        assert got["full_kv_num_blocks"].sum() == 0 and got["kv_num_blocks"].sum() == 1568


def _tables():
    """(name, bool table [batch, q_len, kv_len]): candidate trees behind a
    context, the window predicate as a table, and random blocky tables with
    empty, full and partial tiles (ragged edges included)."""
    rng = np.random.default_rng(9)
    out = [("tree", synth.tree_table(3, 2, 300, 40)), ("tree_long", synth.tree_table(4, 1, 1000, 129))]
    i, j = np.meshgrid(np.arange(700), np.arange(700), indexing="ij")
    out.append(("window", ((i >= j) & (i - j <= 150))[None]))
    for q_len, kv_len in [(300, 333), (128, 256), (1, 129), (257, 31)]:
        coarse = rng.random((2, (q_len + 63) // 64, (kv_len + 63) // 64))
        t = np.repeat(np.repeat(coarse, 64, 1), 64, 2)[:, :q_len, :kv_len]
        dense = rng.random((2, q_len, kv_len)) < 0.5
        out.append((f"blocky {q_len}x{kv_len}", np.where(t < 0.3, False, np.where(t > 0.7, True, dense))))
    return out


@pytest.mark.parametrize("name,table", _tables(), ids=[n for n, _ in _tables()])
@pytest.mark.parametrize("H", [1, 3])
def test_builder_tables(fa, name, table, H):
    """Lookup-table masks: each batch row's own table, bits read per tile."""
    import torch
    Bt, q_len, kv_len = table.shape
    tab = torch.from_numpy(synth.pack_table(table)).cuda()
    bm = fa.block_mask("table", Bt, H, q_len, kv_len, table=tab)
    fa.default_workspace(torch.device("cuda")).check()
    got = bm.numpy()
    want = oracle.block_mask(mask="table", B=Bt, H=H, q_len=q_len, kv_len=kv_len, table=table)
    for key in want:
        np.testing.assert_array_equal(got[key], want[key], err_msg=f"{name} {key}")
    _check_cols(fa, bm, want, name)
