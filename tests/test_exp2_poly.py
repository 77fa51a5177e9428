"""The polynomial 2^x used on the FMA pipe: its header matches a fresh Remez
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
    spec = importlib.util.spec_from_file_location("gen_exp2_poly", os.path.join(CSRC, "gen_exp2_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def header_coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    return [float(v) for v in re.findall(r"kExp2C\d = ([-0-9.e]+)f;", text)]


def test_header_matches_derivation():
    c, maxerr, _ = _gen().remez(3)
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
