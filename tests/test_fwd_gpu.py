"""GPU forward vs the fp64 oracle, element by element, through the C ABI.

Small and downscaled cases are compared on every output row; the full-size
workloads (the bench's shapes and launch configuration) on sampled rows that
the oracle computes one by one (q-block edges, the ragged tail, seeded random
rows).  Tolerances: bf16 max-abs 2e-2 and rel-L2 5e-3, fp32 max-abs 1e-4.
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


def _case(dtype, mask, score="none", B=1, Hq=4, Hkv=4, T=300, D=128, seed=11, **kw):
    return synth.Workload(name="case", dtype=dtype, B=B, Hq=Hq, Hkv=Hkv, T=T, D=D, mask=mask, score=score,
                          seed=seed, **kw)


def _check_full(w, out_fp32=False, max_abs=None):
    q, k, v = w.qkv()
    seg = w.segments()
    o, lse = parity.run_gpu(w, q, k, v, seg, out_fp32=out_fp32)
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, seg)
    return parity.compare(o, o_ref, lse, lse_ref, w.dtype, max_abs=max_abs, label=w.name)


MASKS = [("full", {}), ("causal", {}), ("sliding_window", {"window": 150}), ("prefix_lm", {"prefix_len": 170}),
         ("document", {"doc_lo": 20, "doc_hi": 180})]
SCORES = [("none", {}), ("softcap", {"softcap": 5.0}), ("alibi", {}), ("rel_bias", {"rel_max": 40}),
          ("alibi_softcap", {"softcap": 4.0})]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,mkw", MASKS)
@pytest.mark.parametrize("score,skw", SCORES)
def test_masks_and_scores(dtype, D, mask, mkw, score, skw):
    w = _case(dtype, mask, score, B=2, Hq=2, Hkv=2, T=300, D=D, input_scale=1.0, **mkw, **skw)
    _check_full(w)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (8, 1)])
def test_gqa_ratios(dtype, Hq, Hkv):
    _check_full(_case(dtype, "causal", "alibi", B=1, Hq=Hq, Hkv=Hkv, T=400, D=128))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [1, 17, 127, 128, 129, 136, 640])
def test_lengths(dtype, T):
    _check_full(_case(dtype, "causal", B=1, Hq=2, Hkv=2, T=T, D=64))
    _check_full(_case(dtype, "full", B=1, Hq=2, Hkv=1, T=T, D=128))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("q_len,kv_len,mask,kw", [
    (200, 333, "causal", {}), (333, 200, "full", {}), (700, 130, "sliding_window", {"window": 100}),
    (260, 500, "prefix_lm", {"prefix_len": 300}),
])
def test_rectangular_and_empty_rows(dtype, q_len, kv_len, mask, kw):
    """Tq != Tkv.  The window case leaves rows i > kv_len - 1 + W with no key
    at all, so whole q-blocks are empty: O = 0 and lse = -inf."""
    w = _case(dtype, mask, B=1, Hq=2, Hkv=2, T=q_len, D=128, **kw)
    q, _, _ = w.qkv()
    _, k, v = w.scaled(T=kv_len).qkv()
    o, lse = parity.run_gpu(w, q, k, v, None)
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, None)
    parity.compare(o, o_ref, lse, lse_ref, dtype, label=f"{mask} {q_len}x{kv_len}")
    if mask == "sliding_window":
        assert np.isneginf(lse_ref).any()


@pytest.mark.parametrize("name,small", [
    ("grouped_fp32", {}),
    ("grouped_bf16", {"T": 64 * 17 + 5}),
    ("document_bf16", {"B": 2, "Hq": 3, "Hkv": 3, "T": 1500, "doc_lo": 40, "doc_hi": 400}),
    ("causal_softcap_bf16", {"B": 2, "Hq": 2, "Hkv": 2, "T": 900}),
    ("window_alibi_gqa_bf16", {"Hq": 8, "Hkv": 2, "T": 2000, "window": 300}),
])
def test_downscaled_workloads_full_compare(name, small):
    w = synth.WORKLOADS[name].scaled(**small)
    if name == "causal_softcap_bf16":
        # bf16 output alone can miss max-abs 2e-2 at |O| >= 8 (half a unit is
        # 2^-5 there): fp32 output meets the literal bound, bf16 output the
        # bound plus its own rounding.
        _check_full(w, out_fp32=True)
        q, k, v = w.qkv()
        o, lse = parity.run_gpu(w, q, k, v, None)
        o_ref, lse_ref = parity.run_oracle(w, q, k, v, None)
        o2, r2 = o.reshape(-1, w.D), o_ref.reshape(-1, w.D)
        excess = np.abs(o2 - r2) - (parity.BF16_MAX_ABS + parity.bf16_output_floor(r2, o2))
        assert excess.max() <= 0, f"bf16 output over the bound by {excess.max():.3e}"
    else:
        _check_full(w)


def _check_sampled(w, rows, out_fp32):
    q, k, v = w.qkv()
    seg = w.segments()
    o, lse = parity.run_gpu(w, q, k, v, seg, out_fp32=out_fp32)
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, seg, rows=rows)
    return parity.compare(o.reshape(-1, w.D)[rows], o_ref, lse.reshape(-1)[rows], lse_ref, w.dtype, label=w.name)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_full_size_workloads_sampled_rows(name):
    """The full-size workloads in the bench's launch configuration."""
    w = synth.WORKLOADS[name]
    edges = [0, 1, 127, 128, 129, w.T // 2, w.T - 129, w.T - 128, w.T - 2, w.T - 1]
    rows = parity.sample_rows(w, n_random=2048 if w.T > 10000 else 4096, seed=7, extra_q=edges)
    _check_sampled(w, rows, out_fp32=(name == "causal_softcap_bf16"))


def test_causal_softcap_bf16_output_floor():
    """The bf16-output run of the soft-cap workload: its error stays within
    max-abs 2e-2 plus half a bf16 unit of the reference value."""
    w = synth.WORKLOADS["causal_softcap_bf16"]
    rows = parity.sample_rows(w, n_random=4096, seed=3, extra_q=[0, 1, 2, 3, 4, 5])
    q, k, v = w.qkv()
    o, lse = parity.run_gpu(w, q, k, v, None)
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, None, rows=rows)
    got = o.reshape(-1, w.D)[rows]
    excess = np.abs(got - o_ref) - (parity.BF16_MAX_ABS + parity.bf16_output_floor(o_ref, got))
    print(f"bf16-output soft-cap: max abs {np.abs(got - o_ref).max():.4e}, worst excess over the bound {excess.max():.4e}")
    assert excess.max() <= 0, f"bf16 output over the bound by {excess.max():.3e}"
    assert np.linalg.norm(got - o_ref) / np.linalg.norm(o_ref) <= parity.BF16_REL_L2
    np.testing.assert_allclose(lse.reshape(-1)[rows], lse_ref, atol=parity.LSE_TOL["bf16"])


def test_timeout_is_reported_and_context_survives():
    """A loader that skips its first K tile leaves the consumers' bounded
    waits to run out: the call reports FA_ERR_TIMEOUT through the workspace,
    nothing faults, and the next normal call is correct."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = _case("bf16", "causal", B=1, Hq=2, Hkv=2, T=256, D=128)
    q, k, v = w.qkv()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = fa.block_mask("causal", 1, 1, 256, 256)
    ws = fa.Workspace()
    fa.fwd(qd, kd, vd, bm, workspace=ws, timeout_ms=50, debug_flags=fa.DEBUG_DROP_FIRST_LOAD)
    with pytest.raises(fa.FAError) as ei:
        ws.check()
    assert ei.value.status == fa.ERR_TIMEOUT
    ws.check()                                            # flags were cleared
    o, lse = fa.fwd(qd, kd, vd, bm, workspace=ws)
    ws.check()
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, None)
    parity.compare(o.double().cpu().numpy(), o_ref, lse.double().cpu().numpy(), lse_ref, "bf16")
    torch.cuda.synchronize()


def test_runs_on_a_side_stream():
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = _case("bf16", "sliding_window", "alibi", B=1, Hq=4, Hkv=2, T=600, D=128, window=200)
    q, k, v = w.qkv()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qd, kd, vd = parity.to_device(w, q, k, v)
        bm = fa.block_mask("sliding_window", 1, 1, 600, 600, window=200)
        o, lse = fa.fwd(qd, kd, vd, bm, **parity.score_kwargs_gpu(w))
    s.synchronize()
    o_ref, lse_ref = parity.run_oracle(w, q, k, v, None)
    parity.compare(o.double().cpu().numpy(), o_ref, lse.double().cpu().numpy(), lse_ref, "bf16")


@pytest.mark.parametrize("name", ["causal_softcap_bf16", "document_bf16", "grouped_bf16"])
def test_repeated_launches_are_bitwise_identical(name):
    """Each row's tiles are reduced in a fixed order, so two launches on the
    same inputs must agree bit for bit (a race between pipeline roles would
    show up here as a difference)."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = synth.WORKLOADS[name]
    q, k, v = w.qkv()
    seg = w.segments()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = parity.gpu_block_mask(w, seg)
    skw = parity.score_kwargs_gpu(w)
    outs = []
    for _ in range(3):
        o, lse = fa.fwd(qd, kd, vd, bm, **skw)
        outs.append((o.clone(), lse.clone()))
    fa.default_workspace(qd.device).check()
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(lse, outs[0][1])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("case", ["tree", "tree_short_tail", "square"])
def test_table_masks(dtype, D, case):
    """Lookup-table masks: candidate trees behind a context (tree attention,
    q_len = tree size; in the short-tail case the last kv tile's second half
    lies wholly past kv_len) and a random blocky square table; each batch row
    reads its own table."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    if case == "tree":
        table = synth.tree_table(17, 2, 700, 150)
    elif case == "tree_short_tail":
        table = synth.tree_table(18, 2, 500, 60)
    else:
        rng = np.random.default_rng(5)
        coarse = rng.random((2, 6, 6))
        t = np.repeat(np.repeat(coarse, 64, 1), 64, 2)[:, :333, :333]
        table = np.where(t < 0.3, False, np.where(t > 0.7, True, rng.random((2, 333, 333)) < 0.4))
    Bt, q_len, kv_len = table.shape
    w = _case(dtype, "table", "alibi_softcap", B=2, Hq=4, Hkv=2, T=kv_len, D=D, softcap=6.0)
    _, k, v = w.qkv()
    q = synth.standard_normal(99, (2, 4, q_len, D))
    if dtype == "bf16":
        q = synth.round_to_bf16(q)
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = fa.block_mask("table", Bt, 1, q_len, kv_len, table=torch.from_numpy(synth.pack_table(table)).cuda())
    o, lse = fa.fwd(qd, kd, vd, bm, **parity.score_kwargs_gpu(w))
    fa.default_workspace(qd.device).check()
    import oracle
    o_ref, lse_ref = oracle.fwd(q, k, v, mask="table", table=table, **parity.score_kwargs_oracle(w))
    parity.compare(o.double().cpu().numpy(), o_ref, lse.double().cpu().numpy(), lse_ref, dtype, label=case)
