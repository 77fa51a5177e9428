"""Pins for the fp64 CPU oracle (no GPU).

Each test fixes the oracle to something other than itself: closed forms
derived by hand, the pages' printed facts (tests/golden/page_facts.json),
reductions to simpler cases, an independent library computation (torch CPU
float64) for the unmasked textbook case, and invariants.  Together they are
chosen so that a dropped scale, a flipped sign, a wrong index direction or
an off-by-one window edge fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from block_sparse_attention_fa_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def _rand(shape, seed, scale=1.0):
    return synth.standard_normal(seed, shape, scale)


# ---------------------------------------------------------------- closed forms

def test_softcap_closed_form():
    # D = 1, scale = 2 ln 2, q = k0 = 1: s0 = 2 ln 2; with C = 2, s0 / C = ln 2 and
    # tanh(ln 2) = (4 - 1) / (4 + 1) = 3/5, so the capped score is 6/5.  k1 = 0 gives 0.
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.array([1.0, 0.0], np.float32).reshape(1, 1, 2, 1)
    v = np.array([1.0, 0.0], np.float32).reshape(1, 1, 2, 1)
    o, lse = oracle.fwd(q, k, v, score="softcap", softcap=2.0, scale=2.0 * math.log(2.0))
    assert o[0, 0, 0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-1.2)), abs=1e-14)
    assert lse[0, 0, 0] == pytest.approx(math.log(math.exp(1.2) + 1.0), abs=1e-14)


def test_softcap_limits():
    q, k, v = (_rand((1, 2, 40, 16), s, 3.0) for s in (1, 2, 3))
    o_none, l_none = oracle.fwd(q, k, v, mask="causal")
    o_big, l_big = oracle.fwd(q, k, v, mask="causal", score="softcap", softcap=1e30)
    np.testing.assert_allclose(o_big, o_none, atol=1e-12)
    np.testing.assert_allclose(l_big, l_none, atol=1e-12)
    # |C tanh(s / C)| < C: with every key masked but itself the lse of row 0 is the capped score
    C = 2.0
    _, l_cap = oracle.fwd(q, k, v, mask="causal", score="softcap", softcap=C)
    assert np.all(np.abs(l_cap[..., 0]) <= C)
    s00 = (q[..., 0, :].astype(np.float64) * k[..., 0, :]).sum(-1) / 4.0
    np.testing.assert_allclose(l_cap[..., 0], C * np.tanh(s00 / C), atol=1e-12)


def test_alibi_then_softcap_closed_form():
    """The composite score_mod of the guide's 'Implementation' script: bias
    first, then the cap.  q = 0 makes every raw score 0, so the causal row
    i = 2 sees u_j = -slope (2 - j); with slope = C ln 2 and C = 1 the capped
    scores are C tanh(-ln 4), C tanh(-ln 2), 0 = -15/17, -3/5, 0
    (tanh(ln a) = (a^2 - 1) / (a^2 + 1)).  Capping first and adding the bias
    after would give -2 ln 2, -ln 2, 0 instead."""
    C = 1.0
    q = np.zeros((1, 1, 3, 1), np.float32)
    k = np.ones((1, 1, 3, 1), np.float32)
    v = np.array([1.0, 2.0, 4.0], np.float32).reshape(1, 1, 3, 1)
    slopes = np.array([C * math.log(2.0)], np.float32)
    o, lse = oracle.fwd(q, k, v, mask="causal", score="alibi_softcap", slopes=slopes, softcap=C)
    sl = float(slopes[0]) / C                       # the float32 slope, in units of C
    w = [math.exp(C * math.tanh(-2.0 * sl)), math.exp(C * math.tanh(-sl)), 1.0]
    assert math.tanh(-2.0 * math.log(2.0)) == pytest.approx(-15.0 / 17.0, abs=1e-15)
    assert math.tanh(-math.log(2.0)) == pytest.approx(-3.0 / 5.0, abs=1e-15)
    assert o[0, 0, 2, 0] == pytest.approx((w[0] * 1 + w[1] * 2 + w[2] * 4) / sum(w), abs=1e-7)
    assert lse[0, 0, 2] == pytest.approx(math.log(sum(w)), abs=1e-7)
    assert o[0, 0, 2, 0] == pytest.approx((math.exp(-15 / 17) + 2 * math.exp(-0.6) + 4) /
                                          (math.exp(-15 / 17) + math.exp(-0.6) + 1), abs=1e-6)
    cap_first = [0.25, 0.5, 1.0]
    assert abs(o[0, 0, 2, 0] - (0.25 + 1.0 + 4.0) / sum(cap_first)) > 0.1


def test_alibi_then_softcap_reductions():
    """Zero slopes give the plain soft-cap; a cap of 1e30 gives plain ALiBi."""
    q, k, v = (_rand((1, 3, 50, 16), s, 2.0) for s in (11, 12, 13))
    slopes = np.array([0.1, 0.45, 0.8], np.float32)
    o_c, l_c = oracle.fwd(q, k, v, mask="sliding_window", window=20, score="alibi_softcap",
                          slopes=np.zeros(3, np.float32), softcap=3.0)
    o_s, l_s = oracle.fwd(q, k, v, mask="sliding_window", window=20, score="softcap", softcap=3.0)
    np.testing.assert_allclose(o_c, o_s, atol=1e-13)
    np.testing.assert_allclose(l_c, l_s, atol=1e-13)
    o_c, l_c = oracle.fwd(q, k, v, mask="causal", score="alibi_softcap", slopes=slopes, softcap=1e30)
    o_a, l_a = oracle.fwd(q, k, v, mask="causal", score="alibi", slopes=slopes)
    np.testing.assert_allclose(o_c, o_a, atol=1e-12)
    np.testing.assert_allclose(l_c, l_a, atol=1e-12)


def test_composite_facts_of_the_page():
    f = GOLDEN["composite_score_mod"]
    assert f["order"] == ["alibi_bias", "softcap"] and f["softcap_C"] == GOLDEN["softcap_C"]["value"]


def test_table_mask_equal_to_causal_is_causal():
    """A lookup table holding the causal predicate gives the causal result."""
    q, k, v = (_rand((2, 2, 37, 8), s) for s in (21, 22, 23))
    table = np.tril(np.ones((37, 37), bool))
    o_t, l_t = oracle.fwd(q, k, v, mask="table", table=table, score="alibi", slopes=np.array([0.3, 0.7], np.float32))
    o_c, l_c = oracle.fwd(q, k, v, mask="causal", score="alibi", slopes=np.array([0.3, 0.7], np.float32))
    np.testing.assert_array_equal(o_t, o_c)
    np.testing.assert_array_equal(l_t, l_c)


def test_table_mask_tree_closed_form():
    """Tree attention with q = 0 (all scores equal): each tree query averages
    V over the context and its ancestors-or-self.  Tree parents 0 <- 1 <- 3,
    0 <- 2; one context key."""
    table = np.zeros((1, 4, 5), bool)
    table[0, :, 0] = True                           # the context key
    for node, anc in enumerate([[0], [0, 1], [0, 2], [0, 1, 3]]):
        for a in anc:
            table[0, node, 1 + a] = True
    q = np.zeros((1, 1, 4, 1), np.float32)
    k = np.ones((1, 1, 5, 1), np.float32)
    v = np.array([1.0, 2.0, 4.0, 8.0, 16.0], np.float32).reshape(1, 1, 5, 1)
    o, lse = oracle.fwd(q, k, v, mask="table", table=table)
    np.testing.assert_allclose(o[0, 0, :, 0], [(1 + 2) / 2, (1 + 2 + 4) / 3, (1 + 2 + 8) / 3, (1 + 2 + 4 + 16) / 4],
                               atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.log([2, 3, 3, 4]), atol=1e-14)


def test_table_mask_per_batch_and_tree_generator():
    """Each batch row reads its own table; the generated trees give every
    query its context, itself and its root, and only ancestors otherwise."""
    t = synth.tree_table(5, 2, 6, 9)
    assert t.shape == (2, 9, 15)
    assert t[:, :, :6].all() and all(t[b, k, 6 + k] and t[b, k, 6] for b in range(2) for k in range(9))
    assert not np.triu(t[:, :, 6:], 1).any()        # no node sees a later node
    q, k, v = (_rand((2, 1, 9, 4), s) for s in (31, 32, 33))
    k, v = _rand((2, 1, 15, 4), 34), _rand((2, 1, 15, 4), 35)
    o, _ = oracle.fwd(q, k, v, mask="table", table=t)
    for b in range(2):
        ob, _ = oracle.fwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], mask="table", table=t[b])
        np.testing.assert_array_equal(o[b], ob[0])


def test_table_block_mask_matches_the_closed_form_kind():
    """The brute-force BlockMask of a table holding the sliding-window
    predicate equals that of the sliding-window kind, bit for bit."""
    T, W = 700, 150
    i, j = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
    table = (i >= j) & (i - j <= W)
    a = oracle.block_mask(mask="table", B=1, H=1, q_len=T, kv_len=T, table=table)
    b = oracle.block_mask(mask="sliding_window", B=1, H=1, q_len=T, kv_len=T, window=W)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_alibi_closed_form_and_sign():
    # q = 0 makes every raw score 0, so the weights are exp(-slope |i - j|).  With
    # slope = ln 2 and the causal row i = 2: 2^-2, 2^-1, 1 -> 1/7, 2/7, 4/7.
    q = np.zeros((1, 1, 3, 1), np.float32)
    k = np.ones((1, 1, 3, 1), np.float32)
    v = np.array([1.0, 2.0, 4.0], np.float32).reshape(1, 1, 3, 1)
    slopes = np.array([math.log(2.0)], np.float32)
    o, lse = oracle.fwd(q, k, v, mask="causal", score="alibi", slopes=slopes)
    assert o[0, 0, 2, 0] == pytest.approx((1 * 1 + 2 * 2 + 4 * 4) / 7.0, abs=1e-6)   # = 3
    assert lse[0, 0, 2] == pytest.approx(math.log(7.0 / 4.0), abs=1e-6)
    assert o[0, 0, 1, 0] == pytest.approx((1 * 1 + 2 * 2) / 3.0, abs=1e-6)
    assert o[0, 0, 0, 0] == pytest.approx(1.0, abs=1e-12)


def test_alibi_uses_query_head():
    q = np.zeros((1, 2, 2, 1), np.float32)
    k = np.ones((1, 1, 2, 1), np.float32)
    v = np.array([0.0, 1.0], np.float32).reshape(1, 1, 2, 1)
    slopes = np.array([0.0, math.log(3.0)], np.float32)
    o, _ = oracle.fwd(q, k, v, mask="full", score="alibi", slopes=slopes)
    assert o[0, 0, 0, 0] == pytest.approx(0.5, abs=1e-12)          # head 0: slope 0, uniform
    assert o[0, 1, 0, 0] == pytest.approx(1.0 / 4.0, abs=1e-6)     # head 1: weights 1, 1/3


def test_rel_bias_closed_form():
    # table over r = i - j clamped to [-1, 1]: r = -1 -> ln 1, 0 -> ln 2, +1 -> ln 4
    q = np.zeros((1, 1, 3, 1), np.float32)
    k = np.ones((1, 1, 3, 1), np.float32)
    v = np.array([1.0, 10.0, 100.0], np.float32).reshape(1, 1, 3, 1)
    table = np.log(np.array([[1.0, 2.0, 4.0]], np.float64)).astype(np.float32)
    o, _ = oracle.fwd(q, k, v, mask="full", score="rel_bias", rel_bias=table, rel_max=1)
    # row 0: r = 0, -1, -2 -> clamp -1 : weights 2, 1, 1 (/4)
    assert o[0, 0, 0, 0] == pytest.approx((2 * 1 + 1 * 10 + 1 * 100) / 4.0, rel=1e-6)
    # row 1: r = 1, 0, -1 : weights 4, 2, 1 (/7)
    assert o[0, 0, 1, 0] == pytest.approx((4 * 1 + 2 * 10 + 1 * 100) / 7.0, rel=1e-6)
    # row 2: r = 2 -> clamp 1, 1, 0 : weights 4, 4, 2 (/10)
    assert o[0, 0, 2, 0] == pytest.approx((4 * 1 + 4 * 10 + 2 * 100) / 10.0, rel=1e-6)


def test_sliding_window_edge_is_inclusive():
    # page code: q_idx >= kv_idx and (q_idx - kv_idx) <= W.  q = 0 -> uniform weights.
    fact = GOLDEN["sliding_window_edge"]
    assert fact["inclusive"] is True
    W = 2
    T = 8
    q = np.zeros((1, 1, T, 1), np.float32)
    k = np.ones((1, 1, T, 1), np.float32)
    v = np.arange(T, dtype=np.float32).reshape(1, 1, T, 1)
    o, lse = oracle.fwd(q, k, v, mask="sliding_window", window=W)
    assert o[0, 0, 5, 0] == pytest.approx((3 + 4 + 5) / 3.0, abs=1e-12)
    assert lse[0, 0, 5] == pytest.approx(math.log(3.0), abs=1e-12)
    assert o[0, 0, 1, 0] == pytest.approx(0.5, abs=1e-12)


def test_document_and_prefix_closed_forms():
    T = 6
    q = np.zeros((1, 1, T, 1), np.float32)
    k = np.ones((1, 1, T, 1), np.float32)
    v = np.arange(T, dtype=np.float32).reshape(1, 1, T, 1)
    seg = np.array([0, 0, 1, 1, 1, 2], np.int32)
    o, _ = oracle.fwd(q, k, v, mask="document", seg=seg)
    np.testing.assert_allclose(o[0, 0, :, 0], [0.5, 0.5, 3, 3, 3, 5], atol=1e-12)
    o, _ = oracle.fwd(q, k, v, mask="prefix_lm", prefix_len=2)
    # row 0: {0, 1}; row 1: {0, 1}; row 2: {0, 1, 2}; row 4: {0..4}
    np.testing.assert_allclose(o[0, 0, :, 0], [0.5, 0.5, 1.0, 1.5, 2.0, 2.5], atol=1e-12)


def test_causal_row0_attends_to_itself():
    q, k, v = (_rand((2, 3, 50, 32), s) for s in (4, 5, 6))
    o, lse = oracle.fwd(q, k, v, mask="causal")
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=0)
    s00 = (q[:, :, 0].astype(np.float64) * k[:, :, 0]).sum(-1) / math.sqrt(32)
    np.testing.assert_allclose(lse[:, :, 0], s00, atol=1e-12)


# ---------------------------------------------------- the unmasked textbook case

def test_unmasked_equals_library_softmax_attention():
    torch = pytest.importorskip("torch")
    q, k, v = (_rand((2, 3, 37, 24), s) for s in (7, 8, 9))
    o, lse = oracle.fwd(q, k, v)
    tq, tk, tv = (torch.from_numpy(x).double() for x in (q, k, v))
    s = tq @ tk.transpose(-1, -2) / math.sqrt(24)
    ref = torch.softmax(s, dim=-1) @ tv
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def test_lse_normalises_masked_rows():
    torch = pytest.importorskip("torch")
    q, k, v = (_rand((1, 2, 30, 8), s) for s in (10, 11, 12))
    _, lse = oracle.fwd(q, k, v, mask="sliding_window", window=5)
    s = torch.from_numpy(q).double() @ torch.from_numpy(k).double().transpose(-1, -2) / math.sqrt(8)
    i = torch.arange(30)[:, None]
    j = torch.arange(30)[None, :]
    s = s.masked_fill(~((i >= j) & (i - j <= 5)), float("-inf"))
    total = torch.exp(s - torch.from_numpy(lse)[..., None]).sum(-1)
    np.testing.assert_allclose(total.numpy(), 1.0, atol=1e-12)


# ------------------------------------------------------------------ reductions

def test_group_mask_is_independent_per_group_attention():
    G, n = 5, 17
    T = G * n
    q, k, v = (_rand((1, 2, T, 16), s) for s in (13, 14, 15))
    seg = synth.group_segments(T, n)
    o, lse = oracle.fwd(q, k, v, mask="document", seg=seg)
    for g in range(G):
        sl = slice(g * n, (g + 1) * n)
        og, lg = oracle.fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl])
        np.testing.assert_allclose(o[:, :, sl], og, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], lg, atol=1e-13)


def test_mask_reductions():
    T = 45
    q, k, v = (_rand((1, 2, T, 8), s) for s in (16, 17, 18))
    causal = oracle.fwd(q, k, v, mask="causal")
    full = oracle.fwd(q, k, v, mask="full")
    for got, want in [
        (oracle.fwd(q, k, v, mask="sliding_window", window=T - 1), causal),
        (oracle.fwd(q, k, v, mask="sliding_window", window=10**6), causal),
        (oracle.fwd(q, k, v, mask="prefix_lm", prefix_len=0), causal),
        (oracle.fwd(q, k, v, mask="prefix_lm", prefix_len=T), full),
        (oracle.fwd(q, k, v, mask="document", seg=np.zeros(T, np.int32)), full),
        (oracle.fwd(q, k, v, mask="causal", score="alibi", slopes=np.zeros(2, np.float32)), causal),
        (oracle.fwd(q, k, v, mask="causal", score="rel_bias",
                    rel_bias=np.zeros((2, 7), np.float32), rel_max=3), causal),
    ]:
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_array_equal(got[1], want[1])
    # a narrower window differs from causal
    assert not np.allclose(oracle.fwd(q, k, v, mask="sliding_window", window=3)[0], causal[0])


def test_gqa_equals_repeated_kv():
    q = _rand((2, 8, 33, 16), 19)
    k, v = (_rand((2, 2, 33, 16), s) for s in (20, 21))
    o, lse = oracle.fwd(q, k, v, mask="causal")
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    o2, lse2 = oracle.fwd(q, kr, vr, mask="causal")
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_constant_v_gives_constant_output():
    q, k = (_rand((1, 2, 40, 8), s) for s in (22, 23))
    v = np.full((1, 2, 40, 8), 1.75, np.float32)
    o, _ = oracle.fwd(q, k, v, mask="prefix_lm", prefix_len=7)
    np.testing.assert_allclose(o, 1.75, atol=1e-14)


def test_rows_subset_matches_full():
    q, k, v = (_rand((2, 4, 20, 8), s) for s in (24, 25, 26))
    o, lse = oracle.fwd(q, k, v, mask="causal")
    rows = np.array([0, 5, 19, 20 * 4 + 3, 2 * 4 * 20 - 1], np.int64)
    o2, l2 = oracle.fwd(q, k, v, mask="causal", rows=rows)
    np.testing.assert_array_equal(o.reshape(-1, 8)[rows], o2)
    np.testing.assert_array_equal(lse.reshape(-1)[rows], l2)


def test_fully_masked_row_is_zero_with_minus_inf_lse():
    # a window of -1 admits no pair at all (i >= j and i - j <= -1 is never true)
    q, k, v = (_rand((1, 1, 4, 4), s) for s in (27, 28, 29))
    o, lse = oracle.fwd(q, k, v, mask="sliding_window", window=-1)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))
    # a document row whose id appears among no keys of a shorter kv range
    seg = np.array([0, 1, 1, 1], np.int32)
    o, lse = oracle.fwd(q, k, v, mask="document", seg=seg)
    assert np.isfinite(lse).all()


# ------------------------------------------------------------ the tile scan

def _dense_pred(mask, T, window=0, prefix_len=0, seg=None):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    if mask == "full":
        return np.ones((T, T), bool)
    if mask == "causal":
        return i >= j
    if mask == "sliding_window":
        return (i >= j) & (i - j <= window)
    if mask == "prefix_lm":
        return (j < prefix_len) | (i >= j)
    if mask == "document":
        return seg[:, None] == seg[None, :]
    raise ValueError(mask)


@pytest.mark.parametrize("mask,kw", [
    ("full", {}), ("causal", {}), ("sliding_window", {"window": 11}),
    ("prefix_lm", {"prefix_len": 13}), ("document", {}),
])
@pytest.mark.parametrize("T", [8, 37, 64, 70])
def test_block_mask_classification_on_small_tiles(mask, kw, T):
    block = 8
    seg = None
    if mask == "document":
        seg = np.sort(np.random.default_rng(T).integers(0, 6, T)).astype(np.int32)
        kw = {"seg": seg}
    bm = oracle.block_mask(mask=mask, B=1, H=1, q_len=T, kv_len=T, block=block, **kw)
    pred = _dense_pred(mask, T, **{k: v for k, v in kw.items()})
    n = (T + block - 1) // block
    for qb in range(n):
        part = set(bm["kv_indices"][0, 0, qb, : bm["kv_num_blocks"][0, 0, qb]].tolist())
        full = set(bm["full_kv_indices"][0, 0, qb, : bm["full_kv_num_blocks"][0, 0, qb]].tolist())
        assert not part & full
        assert np.all(bm["kv_indices"][0, 0, qb, bm["kv_num_blocks"][0, 0, qb]:] == -1)
        assert np.all(bm["full_kv_indices"][0, 0, qb, bm["full_kv_num_blocks"][0, 0, qb]:] == -1)
        for kb in range(n):
            tile = pred[qb * block:(qb + 1) * block, kb * block:(kb + 1) * block]
            complete = tile.shape == (block, block)
            if not tile.any():
                assert kb not in part and kb not in full
            elif complete and tile.all():
                assert kb in full
            else:
                assert kb in part


def test_block_mask_skip_fractions_from_the_pages():
    T = GOLDEN["causal_skip_fraction"]["T"]
    nq = T // GOLDEN["tile_size"]["value"]
    bm = oracle.block_mask(mask="causal", B=1, H=1, q_len=T, kv_len=T)
    visited = int(bm["kv_num_blocks"].sum() + bm["full_kv_num_blocks"].sum())
    assert visited == nq * (nq + 1) // 2 == 2080          # lower triangle incl. diagonal
    assert int(bm["kv_num_blocks"].sum()) == nq           # only the diagonal is partial
    assert abs((1 - visited / nq**2) - GOLDEN["causal_skip_fraction"]["about"]) < 0.01

    W = GOLDEN["sliding_window_skip_fraction"]["W"]
    bm = oracle.block_mask(mask="sliding_window", window=W, B=1, H=1, q_len=T, kv_len=T)
    full = int(bm["full_kv_num_blocks"].sum())
    part = int(bm["kv_num_blocks"].sum())
    # q-blocks 0..7 visit qb full + 1 diagonal; later ones 7 full + 2 partial
    assert (full, part) == (28 + 56 * 7, 8 + 56 * 2) == (420, 120)
    assert 1 - (full + part) / nq**2 > GOLDEN["sliding_window_skip_fraction"]["more_than"]


def test_block_mask_broadcast_and_tail():
    # B > 1 document masks give per-batch rows; a tail tile is never full
    seg = np.stack([np.zeros(300, np.int32), (np.arange(300) // 150).astype(np.int32)])
    bm = oracle.block_mask(mask="document", B=2, H=3, q_len=300, kv_len=300, seg=seg)
    assert bm["kv_num_blocks"].shape == (2, 3, 3)
    np.testing.assert_array_equal(bm["kv_num_blocks"][0, 0], [1, 1, 3])
    np.testing.assert_array_equal(bm["full_kv_num_blocks"][0, 0], [2, 2, 0])
    for h in range(3):
        np.testing.assert_array_equal(bm["kv_indices"][1, h], bm["kv_indices"][1, 0])


# ------------------------------------------------------------------ backward

def _quantized(shape, seed, scale=1.0):
    """Values on a 2^-8 grid, so that adding +-2^-10 is exact in float32."""
    return np.round(_rand(shape, seed, scale) * 256.0) / 256.0


def _fd_grads(fwd_kw, q, k, v, g, eps=2.0 ** -10):
    """Central differences of sum(O * g) through the oracle's forward."""
    def loss(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, **fwd_kw)
        return float((o * g).sum())
    out = []
    for which in range(3):
        arrs = [q.copy(), k.copy(), v.copy()]
        grad = np.zeros(arrs[which].shape)
        for idx in np.ndindex(arrs[which].shape):
            a = [x.copy() for x in arrs]
            a[which][idx] += eps
            up = loss(*a)
            a[which][idx] -= 2 * eps
            dn = loss(*a)
            grad[idx] = (up - dn) / (2 * eps)
        out.append(grad)
    return out


BWD_MASKS = [("full", {}), ("causal", {}), ("sliding_window", {"window": 2}),
             ("table", {"table": np.array([[1, 0, 1, 0, 0, 1], [0, 0, 0, 0, 0, 0], [1, 1, 1, 1, 0, 0],
                                           [0, 1, 0, 1, 1, 1]], bool)})]
BWD_SCORES = [("none", {}), ("softcap", {"softcap": 1.5}), ("alibi", {"slopes": np.array([0.3, 0.9], np.float32)}),
              ("rel_bias", {"rel_max": 2, "rel_bias": np.array([[0.5, -1.0, 0.25, 2.0, -0.5],
                                                                [1.0, 0.0, -0.75, 0.5, 0.125]], np.float32)}),
              ("alibi_softcap", {"softcap": 1.5, "slopes": np.array([0.3, 0.9], np.float32)})]


@pytest.mark.parametrize("mask,mkw", BWD_MASKS, ids=[m for m, _ in BWD_MASKS])
@pytest.mark.parametrize("score,skw", BWD_SCORES, ids=[s for s, _ in BWD_SCORES])
def test_backward_matches_finite_differences(mask, mkw, score, skw):
    """dq, dk, dv of sum(O * dO) against central differences of the forward,
    GQA (2 query heads on 1 kv head), Tq != Tkv; the table leaves row 1 with
    no key (its gradients are zero)."""
    q = _quantized((1, 2, 4, 3), 41, 1.5)
    k = _quantized((1, 1, 6, 3), 42, 1.5)
    v = _quantized((1, 1, 6, 3), 43)
    g = _rand((1, 2, 4, 3), 44)
    kw = {"mask": mask, "score": score, **mkw, **skw}
    dq, dk, dv = oracle.bwd(q, k, v, g, **kw)
    fq, fk, fv = _fd_grads(kw, q, k, v, g)
    np.testing.assert_allclose(dq, fq, atol=2e-6)
    np.testing.assert_allclose(dk, fk, atol=2e-6)
    np.testing.assert_allclose(dv, fv, atol=2e-6)


def test_backward_invariants():
    """Softmax rows sum to one: sum_j dv_j = sum_i dO_i over the rows that
    attend; and with every key equal, S does not depend on q: dq = 0."""
    q, k, v, g = (_rand((1, 2, 30, 8), s).astype(np.float32) for s in (51, 52, 53, 54))
    _, dk, dv = oracle.bwd(q, k, v, g, mask="causal")
    np.testing.assert_allclose(dv.sum(axis=2), g.astype(np.float64).sum(axis=2), atol=1e-12)
    k_eq = np.repeat(k[:, :, :1], 30, axis=2)
    dq, _, _ = oracle.bwd(q, k_eq, v, g, mask="full")
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)


def test_backward_gqa_is_the_sum_over_the_group():
    """dK, dV of a shared kv head equal the sums of the per-head gradients with
    K and V repeated for every query head."""
    q, g = _rand((1, 4, 20, 8), 61), _rand((1, 4, 20, 8), 62)
    k, v = _rand((1, 2, 20, 8), 63), _rand((1, 2, 20, 8), 64)
    dq, dk, dv = oracle.bwd(q, k, v, g, mask="sliding_window", window=5, score="alibi",
                            slopes=np.array([0.1, 0.2, 0.3, 0.4], np.float32))
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq2, dk2, dv2 = oracle.bwd(q, kr, vr, g, mask="sliding_window", window=5, score="alibi",
                               slopes=np.array([0.1, 0.2, 0.3, 0.4], np.float32))
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(1, 2, 2, 20, 8).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(1, 2, 2, 20, 8).sum(axis=2), atol=1e-12)
