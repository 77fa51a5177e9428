"""GPU backward (fa_bwd) vs the fp64 oracle's gradients, element by element.

The forward runs first (bf16 O and lse, as a training step keeps them), then
the backward with a seeded bf16 upstream gradient dO.  Both sides see the
same bf16-valued q, k, v and dO.  Tolerances: the GPU rounds P and dS to bf16
for their products (as the forward rounds P) and forms Delta from the bf16 O,
so each gradient is held to rel-L2 <= 1e-2 and max-abs <= 2e-2 of its largest
reference entry (at least 2e-2).
"""
import numpy as np
import pytest

import oracle
from block_sparse_attention_fa_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS_FRAC = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from block_sparse_attention_fa_gb300 import fa
    assert torch.cuda.is_available()
    fa.load_library()


def _compare(got, ref, label):
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), f"{label}: non-finite"
    err = np.abs(got - ref)
    bound = MAX_ABS_FRAC * max(1.0, float(np.abs(ref).max()))
    assert err.max() <= bound, f"{label}: max abs {err.max():.3e} > {bound:.3e}"
    denom = np.linalg.norm(ref)
    if denom > 0:
        rel = np.linalg.norm(got - ref) / denom
        assert rel <= REL_L2, f"{label}: rel L2 {rel:.3e}"


def _run(w, q_len=None, table=None, per_head=False, seed=77):
    import torch
    from block_sparse_attention_fa_gb300 import fa
    q_len = q_len or w.T
    _, k, v = w.qkv()
    q = synth.round_to_bf16(synth.standard_normal(seed, (w.B, w.Hq, q_len, w.D), w.input_scale))
    g = synth.round_to_bf16(synth.standard_normal(seed + 1, (w.B, w.Hq, q_len, w.D)))
    qd, kd, vd = parity.to_device(w, q, k, v)
    gd = torch.from_numpy(g).cuda().to(torch.bfloat16)
    seg = w.segments()
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    tab = torch.from_numpy(synth.pack_table(table)).cuda() if table is not None else None
    Bm = seg.shape[0] if seg is not None else (tab.shape[0] if tab is not None else 1)
    bm = fa.block_mask(w.mask, Bm, w.Hq if per_head else 1, q_len, w.T, window=w.window,
                       prefix_len=w.prefix_len, seg_ids=seg_t, table=tab)
    kw = parity.score_kwargs_gpu(w)
    o, lse = fa.fwd(qd, kd, vd, bm, **kw)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, gd, bm, **kw)
    fa.default_workspace(qd.device).check()
    torch.cuda.synchronize()
    okw = dict(parity.mask_kwargs(w, seg), **parity.score_kwargs_oracle(w))
    if table is not None:
        okw["table"] = table
    rq, rk, rv = oracle.bwd(q, k, v, g, **okw)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _compare(got.cpu().numpy(), ref, f"{w.mask}/{w.score} {name}")


def _case(mask, score="none", B=2, Hq=4, Hkv=2, T=300, D=128, **kw):
    return synth.Workload(name="bwd", dtype="bf16", B=B, Hq=Hq, Hkv=Hkv, T=T, D=D, mask=mask, score=score,
                          seed=31, **kw)


MASKS = [("full", {}), ("causal", {}), ("sliding_window", {"window": 100}), ("prefix_lm", {"prefix_len": 170}),
         ("document", {"doc_lo": 20, "doc_hi": 180})]
SCORES = [("none", {}), ("softcap", {"softcap": 5.0}), ("alibi", {}), ("rel_bias", {"rel_max": 40}),
          ("alibi_softcap", {"softcap": 4.0})]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,mkw", MASKS)
@pytest.mark.parametrize("score,skw", SCORES)
def test_masks_and_scores(D, mask, mkw, score, skw):
    _run(_case(mask, score, D=D, **mkw, **skw))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 1), (8, 2)])
def test_gqa_sums_over_the_group(Hq, Hkv):
    _run(_case("causal", "alibi", B=1, Hq=Hq, Hkv=Hkv, T=400))


@pytest.mark.parametrize("T", [1, 17, 128, 129, 513])
def test_lengths(T):
    _run(_case("causal", B=1, Hq=2, Hkv=2, T=T, D=64))


def test_rectangular_with_empty_rows():
    """q_len > kv_len + window: the last rows attend to nothing and must get
    zero gradient; their q-blocks are empty."""
    _run(_case("sliding_window", B=1, Hq=2, Hkv=1, T=130, window=100), q_len=700)


def test_tree_table_and_per_head_mask():
    table = synth.tree_table(23, 2, 500, 60)
    _run(_case("table", "softcap", T=560, softcap=8.0), q_len=60, table=table)
    _run(_case("sliding_window", "rel_bias", T=300, window=64, rel_max=30), per_head=True)


def test_window_alibi_softcap_workload():
    """The guide's composite example workload at full size (B 2, H 8, 4096
    tokens, D 64, window 512, ALiBi then soft-cap)."""
    w = synth.WORKLOADS["window_alibi_softcap_bf16"]
    _run(w)


def test_causal_softcap_full_length():
    """The causal soft-cap workload's sequence length, input scale and cap
    (T 4096, inputs x2, C 50) on two heads of one batch row, all rows."""
    w = synth.WORKLOADS["causal_softcap_bf16"].scaled(B=1, Hq=2, Hkv=2)
    _run(w)
