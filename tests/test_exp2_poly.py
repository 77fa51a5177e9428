"""The polynomials evaluated on the FMA pipe.  For 2^x: its header matches a fresh Remez
derivation, and the evaluation scheme (round-to-integer by adding 1.5*2^23,
degree-3 polynomial on [-1/2, 1/2], integer add into the exponent field),
carried out in fp32 on the CPU, stays within 1e-4 relative error of exp2
over the range the softmax feeds it."""
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


def header_coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    return [float(v) for v in re.findall(r"kExp2C\d = ([-0-9.e]+)f;", text)]


def test_header_matches_derivation():
    c, maxerr = _gen().exp2_coeffs(3)
    np.testing.assert_allclose(header_coeffs(), np.float32(c), rtol=0, atol=1e-7)
    assert maxerr < 1e-4


def eval_like_device(x):
    c = np.float32(header_coeffs())
    x = np.float32(x)
    shift = np.float32(12582912.0)
    t = (x + shift).astype(np.float32)
    n = (t - shift).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(c[3])
    for ck in (c[2], c[1], c[0]):
        p = np.float32(np.float64(p) * np.float64(f) + np.float64(ck))      # one rounding, as fma
    bits = p.view(np.int32) + (t.view(np.int32) << np.int32(23))
    return bits.astype(np.int32).view(np.float32)


def test_relative_error_over_the_softmax_range():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2_000_001, dtype=np.float32),
                        np.float32([-125.0, -0.5, 0.5, 0.0, -1e-7, 7.999])])
    got = eval_like_device(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 1e-4, rel.max()


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
