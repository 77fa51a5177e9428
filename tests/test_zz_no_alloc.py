"""fa_fwd_noalloc, the forward for callers that cannot allocate device memory
(code inside an allocator's hooks, processes whose device memory a framework
owns outright, paths that must not risk cudaMalloc's implicit device
synchronisation).  Its scratch is a static device array instead of a caller
workspace.  It runs the same kernel as fa_fwd, so its output must equal
fa_fwd's bit for bit, call after call, and agree with the fp64 oracle within
the forward's tolerances; and after a first call it must allocate no device
memory at all.  Collected last on purpose, and self-contained so that it
passes both alone in a fresh process and after the other tests."""
import gc

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
    o_or, lse_or = parity.run_oracle(w, q, k, v, seg)
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        fa.fwd_noalloc(qd, kd, vd, bm, out=out, lse=lse, **skw)
        torch.cuda.synchronize()
        # the same kernel on the same inputs: identical bits
        assert torch.equal(out.view(torch.int16 if dtype == "bf16" else torch.int32),
                           ref_o.view(torch.int16 if dtype == "bf16" else torch.int32))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        # and the oracle's result within the forward's tolerances
        parity.compare(out.double().cpu().numpy(), o_or, lse.double().cpu().numpy(), lse_or, dtype,
                       label=f"noalloc {dtype} {mask} {score}")


def test_noalloc_allocates_no_device_memory():
    """After a first call (which looks up the static array's address), further
    calls change neither the caching allocator's count nor the device's free
    memory."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = synth.Workload(name="noalloc_mem", dtype="bf16", B=1, Hq=4, Hkv=4, T=1000, D=64, mask="causal",
                       score="softcap", softcap=20.0, seed=32)
    q, k, v = w.qkv()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = parity.gpu_block_mask(w, None)
    skw = parity.score_kwargs_gpu(w)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=qd.device)
    fa.fwd_noalloc(qd, kd, vd, bm, out=out, lse=lse, **skw)
    torch.cuda.synchronize()
    first = out.clone()
    gc.collect()
    torch.cuda.synchronize()
    # the caching allocator's cumulative count of allocations (frees of other
    # tests' garbage do not move it) and the device's free memory
    n_alloc0 = torch.cuda.memory_stats()["allocation.all.allocated"]
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        fa.fwd_noalloc(qd, kd, vd, bm, out=out, lse=lse, **skw)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == n_alloc0
    assert free1 >= free0, (free0, free1)
    assert torch.equal(out.view(torch.int16), first.view(torch.int16))


def test_noalloc_rejected_call_leaves_the_array_alone():
    """A call the argument checks reject returns an error and launches
    nothing; the next good call still gives the right answer."""
    import ctypes
    import torch
    from block_sparse_attention_fa_gb300 import fa
    w = synth.Workload(name="noalloc_rej", dtype="bf16", B=1, Hq=2, Hkv=2, T=300, D=128, mask="causal",
                       score="none", seed=33)
    q, k, v = w.qkv()
    qd, kd, vd = parity.to_device(w, q, k, v)
    bm = parity.gpu_block_mask(w, None)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=qd.device)
    lib = fa.load_library()
    a = fa.FwdArgs()
    a.dtype, a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = fa.BF16, 1, 2, 2, 300, 300, 96   # head dim 96: unsupported
    a.q, a.k, a.v, a.o, a.lse = qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr()
    st = lib.fa_fwd_noalloc(ctypes.byref(a), ctypes.byref(bm.struct), None, None)
    assert st == fa.ERR_UNSUPPORTED, lib.fa_last_error()
    fa.fwd_noalloc(qd, kd, vd, bm, out=out, lse=lse)
    torch.cuda.synchronize()
    o_or, lse_or = parity.run_oracle(w, q, k, v, None)
    parity.compare(out.double().cpu().numpy(), o_or, lse.double().cpu().numpy(), lse_or, "bf16",
                   label="noalloc after a rejected call")
