"""Helpers shared by the GPU parity tests, the smoke check and the benchmark.

They feed the same seeded inputs (``synth``) to the CUDA path (through the
C-ABI binding) and to the fp64 oracle, and compare the results with the
tolerances the forward is held to:
  bf16 inputs: max |O - O_ref| <= 2e-2 and ||O - O_ref||_2 / ||O_ref||_2 <= 5e-3
  fp32 inputs: max |O - O_ref| <= 1e-4
and the logsumexp within 1e-3 (bf16) / 1e-4 (fp32); rows that attend to
nothing must give O = 0 and lse = -inf on both sides.
"""
from __future__ import annotations

import numpy as np

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
FP32_MAX_ABS = 1e-4
LSE_TOL = {"bf16": 1e-3, "fp32": 1e-4}


def to_device(w, q, k, v):
    import torch
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return tuple(torch.from_numpy(x).to("cuda").to(dt).contiguous() for x in (q, k, v))


def score_kwargs_gpu(w):
    import torch
    kw = {"score": w.score}
    if w.score in ("softcap", "alibi_softcap"):
        kw["softcap"] = w.softcap
    if w.score in ("alibi", "alibi_softcap"):
        kw["alibi_slopes"] = torch.from_numpy(w.slopes()).cuda()
    if w.score == "rel_bias":
        kw["rel_bias"] = torch.from_numpy(w.rel_bias()).cuda()
        kw["rel_max"] = w.rel_max
    return kw


def score_kwargs_oracle(w):
    kw = {"score": w.score}
    if w.score in ("softcap", "alibi_softcap"):
        kw["softcap"] = w.softcap
    if w.score in ("alibi", "alibi_softcap"):
        kw["slopes"] = w.slopes()
    if w.score == "rel_bias":
        kw["rel_bias"] = w.rel_bias()
        kw["rel_max"] = w.rel_max
    return kw


def mask_kwargs(w, seg):
    kw = {"mask": w.mask}
    if w.mask == "sliding_window":
        kw["window"] = w.window
    elif w.mask == "prefix_lm":
        kw["prefix_len"] = w.prefix_len
    elif w.mask == "document":
        kw["seg"] = seg
    return kw


def gpu_block_mask(w, seg, q_len=None, kv_len=None):
    import torch
    from block_sparse_attention_fa_gb300 import fa
    q_len = q_len or w.T
    kv_len = kv_len or w.kv_len
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    B = seg.shape[0] if seg is not None else 1
    return fa.block_mask(w.mask, B, 1, q_len, kv_len, window=w.window, prefix_len=w.prefix_len,
                         seg_ids=seg_t)


def run_gpu(w, q, k, v, seg, out_fp32=False):
    """(o, lse) as float64 numpy arrays from the CUDA path."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    qd, kd, vd = to_device(w, q, k, v)
    bm = gpu_block_mask(w, seg, q.shape[2], k.shape[2])
    o, lse = fa.fwd(qd, kd, vd, bm, out_fp32=out_fp32, **score_kwargs_gpu(w))
    fa.default_workspace(qd.device).check()
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def run_oracle(w, q, k, v, seg, rows=None):
    import oracle
    return oracle.fwd(q, k, v, rows=rows, **mask_kwargs(w, seg), **score_kwargs_oracle(w))


def compare(o, o_ref, lse, lse_ref, dtype, max_abs=None, label=""):
    """Assert the tolerances; returns the measured errors."""
    o = np.asarray(o, np.float64).reshape(-1, o_ref.shape[-1])
    o_ref = np.asarray(o_ref, np.float64).reshape(o.shape)
    lse = np.asarray(lse, np.float64).reshape(-1)
    lse_ref = np.asarray(lse_ref, np.float64).reshape(-1)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{label}: fully masked rows differ"
    assert np.all(o[empty] == 0.0), f"{label}: fully masked rows must be 0"
    assert np.all(np.isfinite(o)), f"{label}: non-finite output"
    err = np.abs(o - o_ref)
    max_err = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(o_ref))
    rel_l2 = float(np.linalg.norm(o - o_ref) / denom) if denom > 0 else 0.0
    lse_err = float(np.abs(lse[~empty] - lse_ref[~empty]).max()) if (~empty).any() else 0.0
    if dtype == "bf16":
        limit = BF16_MAX_ABS if max_abs is None else max_abs
        assert max_err <= limit, f"{label}: max abs {max_err:.3e} > {limit}"
        assert rel_l2 <= BF16_REL_L2, f"{label}: rel L2 {rel_l2:.3e} > {BF16_REL_L2}"
    else:
        limit = FP32_MAX_ABS if max_abs is None else max_abs
        assert max_err <= limit, f"{label}: max abs {max_err:.3e} > {limit}"
    assert lse_err <= LSE_TOL[dtype], f"{label}: lse err {lse_err:.3e} > {LSE_TOL[dtype]}"
    return {"max_abs": max_err, "rel_l2": rel_l2, "lse_max_abs": lse_err}


def bf16_half_ulp(x):
    """Half a unit in the last place of bf16 at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def bf16_output_floor(o_ref, o_gpu):
    """The rounding a bf16 output may add on top of the 2e-2 bound: half a
    unit at the larger of |O_ref| and |O| (the two can sit on either side of
    a power of two, where the unit doubles)."""
    return bf16_half_ulp(np.maximum(np.abs(o_ref), np.abs(o_gpu)))


def sample_rows(w, n_random, seed=0, extra_q=()):
    """Flat row indices: n_random seeded random rows over all (b, h, i), plus
    every head's rows i in `extra_q` (q-block edges, the tail)."""
    rng = np.random.default_rng(seed)
    total = w.B * w.Hq * w.T
    rows = set(rng.choice(total, size=min(n_random, total), replace=False).tolist())
    for b in range(w.B):
        for h in range(w.Hq):
            for i in extra_q:
                if 0 <= i < w.T:
                    rows.add((b * w.Hq + h) * w.T + i)
    return np.array(sorted(rows), np.int64)
