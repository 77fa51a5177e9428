"""The tanh polynomial the soft-cap kernels evaluate on the FMA pipe: its
header matches a fresh Remez derivation, and the folded form the forward
evaluates (coefficients scaled by the cap and the score scale), carried out
in fp32 on the CPU, stays within 2e-5 relative error of C tanh(s / C)."""
import importlib.util
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "block_sparse_attention_fa_gb300", "csrc")


def _gen():
    spec = importlib.util.spec_from_file_location("gen_poly", os.path.join(CSRC, "gen_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def tanh_header():
    text = open(os.path.join(CSRC, "tanh_poly.h")).read()
    c = [float(v) for v in re.findall(r"kTanhC\d = ([-0-9.e]+)f;", text)]
    U = float(re.search(r"kTanhRange = ([-0-9.e]+)f;", text).group(1))
    return c, U


def test_tanh_header_matches_derivation():
    g = _gen()
    c, maxerr = g.tanh_coeffs()
    hc, U = tanh_header()
    assert U == g.TANH_RANGE
    np.testing.assert_allclose(hc, np.float32(c), rtol=0, atol=1e-7)
    assert maxerr < 1e-5


def test_softcap_polynomial_as_the_kernel_folds_it():
    """x = s * Q(s^2) with Q_k = C log2(e) a c_k a^(2k), a = scale / C: the
    capped score in base-2 units, in fp32, within 2e-5 relative of
    C tanh(scale s / C) log2(e) wherever |scale s / C| <= U."""
    hc, U = tanh_header()
    log2e = 1.4426950408889634
    for C, scale in [(50.0, 128 ** -0.5), (5.0, 64 ** -0.5), (1.0, 1.0)]:
        a = np.float32(scale / C)
        Q = [np.float32(C * log2e * a * ck * float(a) ** (2 * k)) for k, ck in enumerate(hc)]
        s = np.linspace(-U / a, U / a, 400001).astype(np.float32)
        w = (s * s).astype(np.float32)
        q = Q[4]
        for k in (3, 2, 1, 0):
            q = np.float32(np.float64(q) * np.float64(w) + np.float64(Q[k]))
        x = (s * q).astype(np.float64)
        want = C * np.tanh(np.float64(scale) * s / C) * log2e
        nz = np.abs(want) > 0
        assert np.max(np.abs(x[nz] - want[nz]) / np.abs(want[nz])) < 2e-5


def tanh2_header():
    text = open(os.path.join(CSRC, "tanh2_poly.h")).read()
    c = [float(v) for v in re.findall(r"kTanh2C\d = ([-0-9.e]+)f;", text)]
    U = float(re.search(r"kTanh2Range = ([-0-9.e]+)f;", text).group(1))
    return c, U


def test_tanh2_header_matches_derivation():
    g = _gen()
    c, maxerr = g.tanh_coeffs(g.TANH2_DEGREE, g.TANH2_RANGE)
    hc, U = tanh2_header()
    assert U == g.TANH2_RANGE == 0.5
    np.testing.assert_allclose(hc, np.float32(c), rtol=0, atol=1e-7)
    assert maxerr < 3e-5


def test_softcap_degree2_tier_as_the_kernel_folds_it():
    """The degree-2 tier the forward uses where every |scale s / C| <= 1/2:
    x Q(x^2) + nm with Q_k = C log2(e) a c_k a^(2k), evaluated in fp32 with
    fused multiply-adds, stays within 5e-5 relative of C tanh(a x) log2(e);
    the capped row max taken from the raw max equals the max of the capped
    scores (the cap is increasing), so the largest element's argument is 0."""
    hc, U = tanh2_header()
    log2e = 1.4426950408889634
    for C, scale in [(50.0, 128 ** -0.5), (20.0, 64 ** -0.5), (1.0, 1.0)]:
        a = np.float32(scale / C)
        Q = [np.float32(C * log2e * a * ck * float(a) ** (2 * k)) for k, ck in enumerate(hc)]
        x = np.linspace(-U / a, U / a, 200001).astype(np.float32)
        w = (x * x).astype(np.float32)
        q = np.float32(np.float64(w) * np.float64(Q[2]) + np.float64(Q[1])).astype(np.float32)
        q = np.float32(np.float64(q) * np.float64(w) + np.float64(Q[0])).astype(np.float32)
        got = (np.float64(x) * np.float64(q))
        want = C * np.tanh(np.float64(a) * x) * log2e
        nz = np.abs(want) > 0
        assert np.max(np.abs(got[nz] - want[nz]) / np.abs(want[nz])) < 5e-5
        # monotonic: the capped value of the largest raw score is the largest capped value
        assert np.all(np.diff(got) >= 0)
