"""GPU split-KV decoding forward (fa_fwd_decode) vs the fp64 oracle, element
by element, through the C ABI.

The oracle is the plain definition of the result for any (q_len, kv_len); the
decoding path must reach it for every mask, score_mod, split count and row
grouping it accepts, with the bf16 tolerances of the prefill forward
(max-abs 2e-2, rel-L2 5e-3, lse 1e-3).  The full-size decoding workloads (the
bench's shapes and split choice) are compared on every row.
"""
import numpy as np
import pytest

from block_sparse_attention_fa_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from block_sparse_attention_fa_gb300 import fa
    assert torch.cuda.is_available()
    fa.load_library()


def _case(mask="full", score="none", B=2, Hq=8, Hkv=2, q_len=3, kv_len=1000, D=128, seed=21, **kw):
    return synth.Workload(name="decode_case", dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, T=kv_len, D=D, mask=mask,
                          score=score, seed=seed, q_len=q_len, **kw)


def _run(w, num_splits=0, per_head=False, out_fp32=False):
    import torch
    from block_sparse_attention_fa_gb300 import fa
    q, k, v = w.qkv()
    qd, kd, vd = parity.to_device(w, q, k, v)
    table = w.table()
    tab = torch.from_numpy(synth.pack_table(table)).cuda() if table is not None else None
    bm = fa.block_mask(w.mask, tab.shape[0] if tab is not None else 1, w.Hq if per_head else 1, w.Tq, w.T,
                       window=w.window, prefix_len=w.prefix_len, table=tab)
    o, lse = fa.fwd_decode(qd, kd, vd, bm, num_splits=num_splits, out_fp32=out_fp32,
                           **parity.score_kwargs_gpu(w))
    fa.default_workspace(qd.device).check()
    torch.cuda.synchronize()
    if table is not None:
        import oracle
        o_ref, lse_ref = oracle.fwd(q, k, v, mask="table", table=table, **parity.score_kwargs_oracle(w))
    else:
        o_ref, lse_ref = parity.run_oracle(w, q, k, v, None)
    return (o.double().cpu().numpy(), lse.double().cpu().numpy()), (o_ref, lse_ref)


def _check(w, **kw):
    (o, lse), (o_ref, lse_ref) = _run(w, **kw)
    return parity.compare(o, o_ref, lse, lse_ref, "bf16", label=w.name)


MASKS = [("full", {}), ("causal", {}), ("sliding_window", {"window": 40}), ("prefix_lm", {"prefix_len": 300})]
SCORES = [("none", {}), ("softcap", {"softcap": 5.0}), ("alibi", {}), ("rel_bias", {"rel_max": 40}),
          ("alibi_softcap", {"softcap": 4.0})]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,mkw", MASKS)
@pytest.mark.parametrize("score,skw", SCORES)
def test_masks_and_scores(D, mask, mkw, score, skw):
    """kv_len 1000 leaves a ragged tail tile; splits 1, 3 and the library's
    choice rotate over the cases."""
    splits = {"none": 1, "softcap": 3, "alibi": 0, "rel_bias": 5, "alibi_softcap": 2}[score]
    _check(_case(mask, score, D=D, **mkw, **skw), num_splits=splits)


@pytest.mark.parametrize("Hq,Hkv,q_len", [(1, 1, 1), (4, 4, 1), (8, 2, 1), (32, 8, 1), (16, 4, 4), (4, 1, 4),
                                          (2, 2, 16), (8, 8, 7)])
def test_row_groups(Hq, Hkv, q_len):
    """Rows per group from 1 to the maximum of 16 (Hq / Hkv x q_len)."""
    _check(_case("causal", "alibi", B=1, Hq=Hq, Hkv=Hkv, q_len=q_len, kv_len=777, D=128))


@pytest.mark.parametrize("splits", [1, 2, 7, 9, 64, 256])
def test_split_counts(splits):
    """More splits than visited tiles leaves empty splits (max -inf, sum 0)
    that the merge must ignore; 9 tiles over 2 or 7 splits are uneven."""
    _check(_case("full", "softcap", softcap=20.0, kv_len=1100, D=64), num_splits=splits)


def test_per_head_block_mask():
    """A BlockMask with H = Hq: each row group is one query head."""
    _check(_case("sliding_window", "rel_bias", Hq=4, Hkv=2, q_len=8, kv_len=600, window=200, rel_max=64),
           per_head=True, num_splits=4)


@pytest.mark.parametrize("kv_len", [1, 2, 127, 128, 129, 4099])
def test_lengths(kv_len):
    _check(_case("full", "none", B=1, Hq=8, Hkv=4, q_len=2, kv_len=kv_len, D=128))


def test_empty_rows():
    """Raw-index window of 0 against a single key: rows 1.. see nothing."""
    w = _case("sliding_window", "none", B=1, Hq=2, Hkv=1, q_len=5, kv_len=1, window=0, D=64)
    (o, lse), (o_ref, lse_ref) = _run(w, num_splits=2)
    assert np.isneginf(lse_ref).sum() == 2 * 4
    parity.compare(o, o_ref, lse, lse_ref, "bf16", label="empty rows")


def test_fp32_output():
    w = _case("full", "softcap", softcap=30.0, B=1, Hq=8, Hkv=2, q_len=2, kv_len=2000, input_scale=2.0)
    (o, lse), (o_ref, lse_ref) = _run(w, out_fp32=True)
    parity.compare(o, o_ref, lse, lse_ref, "bf16", label="fp32 out")


def test_matches_prefill_forward():
    """The decoding and prefill paths agree on the same call (same BlockMask),
    and each agrees with the fp64 oracle."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = _case("prefix_lm", "alibi", B=2, Hq=8, Hkv=2, q_len=4, kv_len=3000, prefix_len=1000)
    q, k, v = w.qkv()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = fa.block_mask(w.mask, 1, 1, w.Tq, w.T, prefix_len=w.prefix_len)
    o1, l1 = fa.fwd_decode(qd, kd, vd, bm, num_splits=6, out_fp32=True, **parity.score_kwargs_gpu(w))
    o2, l2 = fa.fwd(qd, kd, vd, bm, out_fp32=True, **parity.score_kwargs_gpu(w))
    torch.cuda.synchronize()
    assert float((o1 - o2).abs().max()) < 1e-2
    assert float((l1 - l2).abs().max()) < 1e-3
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, None)
    for o, lse, label in ((o1, l1, "decode"), (o2, l2, "prefill")):
        parity.compare(o.double().cpu().numpy(), o_ref, lse.double().cpu().numpy(), lse_ref, "bf16",
                       label=f"{label} vs oracle")


def test_unsupported_shapes_are_errors():
    import torch
    from block_sparse_attention_fa_gb300 import fa
    q = torch.zeros((1, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 256, 128), dtype=torch.bfloat16, device="cuda")
    bm = fa.block_mask("full", 1, 1, 1, 256)
    with pytest.raises(fa.FAError) as ei:           # 32 query heads on one kv head: 32 rows
        fa.fwd_decode(q, k, k, bm)
    assert ei.value.status == fa.ERR_UNSUPPORTED
    q2 = torch.zeros((1, 1, 200, 128), dtype=torch.bfloat16, device="cuda")
    bm2 = fa.block_mask("full", 1, 1, 200, 256)
    with pytest.raises(fa.FAError) as ei:           # two q-blocks
        fa.fwd_decode(q2, k, k, bm2)
    assert ei.value.status == fa.ERR_UNSUPPORTED


@pytest.mark.parametrize("name", sorted(synth.DECODE_WORKLOADS))
def test_full_size_decode_workloads(name):
    """The bench's decoding shapes, split count chosen by the library, every
    row against the oracle (each row reads the whole 32768-key sequence)."""
    _check(synth.DECODE_WORKLOADS[name])


@pytest.mark.parametrize("q_len,Hq,Hkv,splits", [(4, 8, 2, 0), (16, 4, 4, 3), (3, 16, 4, 7)])
def test_tree_attention_tables(q_len, Hq, Hkv, splits):
    """Speculative-decoding verification: the draft tree's tokens query the
    context and their ancestors through a lookup-table mask."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    table = synth.tree_table(41 + q_len, 2, 1500, q_len)
    w = _case("table", "alibi", B=2, Hq=Hq, Hkv=Hkv, q_len=q_len, kv_len=1500 + q_len, D=128)
    q, k, v = w.qkv()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = fa.block_mask("table", 2, 1, q_len, w.T, table=torch.from_numpy(synth.pack_table(table)).cuda())
    o, lse = fa.fwd_decode(qd, kd, vd, bm, num_splits=splits, **parity.score_kwargs_gpu(w))
    fa.default_workspace(qd.device).check()
    import oracle
    o_ref, lse_ref = oracle.fwd(q, k, v, mask="table", table=table, **parity.score_kwargs_oracle(w))
    parity.compare(o.double().cpu().numpy(), o_ref, lse.double().cpu().numpy(), lse_ref, "bf16", label="tree")
