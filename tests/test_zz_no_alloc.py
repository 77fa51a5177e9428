"""fa_fwd_noalloc, the forward for callers that cannot allocate device memory
(code inside an allocator's hooks, processes whose device memory a framework
owns outright, paths that must not risk cudaMalloc's implicit device
synchronisation).  Its scratch is a static device array instead of a caller
workspace; its output must agree with fa_fwd's on the same inputs, call after
call.  Collected last on purpose, and self-contained so that it passes both
alone in a fresh process and after the other tests."""
import numpy as np
import pytest

from block_sparse_attention_fa_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,mask,score,kw", [
    ("bf16", "causal", "alibi", {}),
    ("bf16", "sliding_window", "softcap", {"window": 200, "softcap": 5.0}),
    ("fp32", "document", "none", {"doc_lo": 30, "doc_hi": 200}),
])
def test_noalloc_matches_fa_fwd_on_two_calls_in_a_row(dtype, mask, score, kw):
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = synth.Workload(name="noalloc", dtype=dtype, B=2, Hq=4, Hkv=2, T=700, D=128, mask=mask, score=score,
                       seed=31, **kw)
    q, k, v = w.qkv()
    seg = w.segments()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = parity.gpu_block_mask(w, seg)
    skw = parity.score_kwargs_gpu(w)
    ref_o, ref_lse = fa.fwd(qd, kd, vd, bm, **skw)
    fa.default_workspace(qd.device).check()
    limit = parity.BF16_MAX_ABS if dtype == "bf16" else parity.FP32_MAX_ABS
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        fa.fwd_noalloc(qd, kd, vd, bm, out=out, lse=lse, **skw)
        torch.cuda.synchronize()
        diff = (out.double() - ref_o.double()).abs().max().item()
        assert diff <= limit, diff
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=parity.LSE_TOL[dtype])
