"""C-ABI checks that need no GPU: the library loads, exports every function
include/fa.h declares, the ctypes structs match the header's layout, and
argument validation rejects bad calls before anything is launched."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    from block_sparse_attention_fa_gb300 import build, fa as fam
    try:
        build.build()
    except RuntimeError as e:  # no CUDA toolkit on this host
        pytest.skip(str(e))
    fam.load_library()
    return fam


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted([
        "fa_block_mask_build", "fa_block_mask_build_cols", "fa_block_mask_shape", "fa_block_mask_size", "fa_bwd",
        "fa_bwd_rowstats_bytes", "fa_decode_partials_bytes", "fa_decode_splits", "fa_fwd",
        "fa_fwd_decode", "fa_fwd_noalloc", "fa_last_error", "fa_version", "fa_workspace_bytes",
        "fa_workspace_check"])


def test_library_exports_every_declared_symbol(fa):
    lib = fa.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(fa.SYMBOLS) == set(declared_functions())
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (fa_\w+)", out))
    assert set(declared_functions()) <= exported


def test_struct_layout_matches_header(fa, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "fa.h"
#define F(T, m) printf(#T "." #m " %zu\n", offsetof(T, m));
int main(void) {
  printf("fa_mask_desc %zu\nfa_block_mask %zu\nfa_score_desc %zu\nfa_fwd_args %zu\nfa_bwd_args %zu\n"
         "fa_block_mask_cols %zu\n",
         sizeof(fa_mask_desc), sizeof(fa_block_mask), sizeof(fa_score_desc), sizeof(fa_fwd_args),
         sizeof(fa_bwd_args), sizeof(fa_block_mask_cols));
  F(fa_bwd_args, scale) F(fa_bwd_args, q) F(fa_bwd_args, dout) F(fa_bwd_args, lse) F(fa_bwd_args, rowstats)
  F(fa_bwd_args, timeout_ms) F(fa_block_mask_cols, q_indices) F(fa_block_mask_cols, full_q_indices)
  F(fa_mask_desc, seg_ids) F(fa_mask_desc, table) F(fa_mask_desc, table_batch)
  F(fa_block_mask, kv_num_blocks) F(fa_block_mask, full_kv_indices)
  F(fa_block_mask, mask) F(fa_score_desc, alibi_slopes) F(fa_score_desc, rel_max)
  F(fa_fwd_args, scale) F(fa_fwd_args, q) F(fa_fwd_args, lse) F(fa_fwd_args, timeout_ms)
  F(fa_fwd_args, flags) F(fa_fwd_args, debug_flags)
  return 0;
}''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], capture_output=True,
                                                               text=True, check=True).stdout.split("\n") if line)
    got = {k: int(v) for k, v in got.items()}
    assert got["fa_mask_desc"] == ctypes.sizeof(fa.MaskDesc)
    assert got["fa_block_mask"] == ctypes.sizeof(fa.BlockMaskStruct)
    assert got["fa_score_desc"] == ctypes.sizeof(fa.ScoreDesc)
    assert got["fa_fwd_args"] == ctypes.sizeof(fa.FwdArgs)
    assert got["fa_bwd_args"] == ctypes.sizeof(fa.BwdArgs)
    assert got["fa_block_mask_cols"] == ctypes.sizeof(fa.BlockMaskColsStruct)
    pairs = {"fa_mask_desc": fa.MaskDesc, "fa_block_mask": fa.BlockMaskStruct,
             "fa_score_desc": fa.ScoreDesc, "fa_fwd_args": fa.FwdArgs, "fa_bwd_args": fa.BwdArgs,
             "fa_block_mask_cols": fa.BlockMaskColsStruct}
    for key, off in got.items():
        if "." in key:
            t, m = key.split(".")
            assert getattr(pairs[t], m).offset == off, key


def test_shape_query(fa):
    lib = fa.load_library()
    nq, nkv, ne = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    assert lib.fa_block_mask_shape(2, 3, 300, 129, ctypes.byref(nq), ctypes.byref(nkv), ctypes.byref(ne)) == fa.OK
    assert (nq.value, nkv.value, ne.value) == (3, 2, 2 * 3 * 3 * 2)
    assert lib.fa_block_mask_shape(0, 1, 1, 1, None, None, None) == fa.ERR_INVALID_ARG
    assert b"extents" in lib.fa_last_error()
    assert lib.fa_workspace_bytes() >= 16
    assert b"sm_103a" in lib.fa_version()


FAKE = 0x10000  # a 16-byte aligned non-NULL address; never dereferenced (validation fails first)


def _bm(fa, **kw):
    s = fa.BlockMaskStruct()
    s.B, s.H, s.q_len, s.kv_len = 1, 1, 256, 256
    s.block_q = s.block_kv = 128
    s.nq, s.nkv = 2, 2
    s.kv_num_blocks = s.kv_indices = s.full_kv_num_blocks = s.full_kv_indices = FAKE
    s.mask.kind = fa.MASK_KINDS["causal"]
    for k, v in kw.items():
        if k.startswith("mask_"):
            setattr(s.mask, k[5:], v)
        else:
            setattr(s, k, v)
    return s


def _args(fa, **kw):
    a = fa.FwdArgs()
    a.dtype, a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = fa.BF16, 1, 4, 4, 256, 256, 128
    a.q = a.k = a.v = a.o = a.lse = FAKE
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,status,text", [
    ({"block_q": 64}, "ERR_UNSUPPORTED", b"128"),
    ({"nq": 3}, "ERR_INVALID_ARG", b"nq"),
    ({"kv_indices": None}, "ERR_INVALID_ARG", b"non-NULL"),
    ({"mask_kind": 9}, "ERR_INVALID_ARG", b"mask kind"),
    ({"mask_kind": 2, "mask_window": -1}, "ERR_INVALID_ARG", b"window"),
    ({"mask_kind": 4, "mask_prefix_len": -5}, "ERR_INVALID_ARG", b"prefix"),
    ({"mask_kind": 3}, "ERR_INVALID_ARG", b"seg_ids"),
    ({"mask_kind": 3, "mask_seg_ids": FAKE, "mask_seg_batch": 2}, "ERR_INVALID_ARG", b"seg_batch"),
    ({"mask_kind": 3, "mask_seg_ids": FAKE, "mask_seg_batch": 1, "kv_len": 200, "nkv": 2},
     "ERR_UNSUPPORTED", b"q_len == kv_len"),
    ({"mask_kind": 5}, "ERR_INVALID_ARG", b"needs a table"),
    ({"mask_kind": 5, "mask_table": FAKE + 2, "mask_table_batch": 1}, "ERR_INVALID_ARG", b"aligned"),
    ({"mask_kind": 5, "mask_table": FAKE, "mask_table_batch": 2}, "ERR_INVALID_ARG", b"table_batch"),
])
def test_block_mask_build_rejects(fa, kw, status, text):
    lib = fa.load_library()
    bm = _bm(fa, **kw)
    st = lib.fa_block_mask_build(ctypes.byref(bm), ctypes.c_void_p(FAKE), None)
    assert st == getattr(fa, status)
    assert text in lib.fa_last_error()


def test_block_mask_build_needs_workspace(fa):
    lib = fa.load_library()
    assert lib.fa_block_mask_build(ctypes.byref(_bm(fa)), None, None) == fa.ERR_INVALID_ARG


@pytest.mark.parametrize("kw,bmkw,score,status,text", [
    ({"D": 96}, {}, None, "ERR_UNSUPPORTED", b"head dim"),
    ({"Hkv": 3}, {}, None, "ERR_INVALID_ARG", b"multiple"),
    ({"dtype": 7}, {}, None, "ERR_INVALID_ARG", b"dtype"),
    ({"q": FAKE + 8}, {}, None, "ERR_INVALID_ARG", b"aligned"),
    ({"o": None}, {}, None, "ERR_INVALID_ARG", b"non-NULL"),
    ({"q_len": 300}, {}, None, "ERR_INVALID_ARG", b"built for"),
    ({"B": 2}, {"B": 3}, None, "ERR_INVALID_ARG", b"block mask B"),
    ({}, {"H": 2}, None, "ERR_INVALID_ARG", b"block mask H"),
    ({"flags": 4}, {}, None, "ERR_INVALID_ARG", b"flags"),
    ({"dtype": 1, "flags": 1}, {}, None, "ERR_INVALID_ARG", b"bf16 inputs only"),
    ({}, {}, {"kind": 1, "softcap": 0.0}, "ERR_INVALID_ARG", b"softcap"),
    ({}, {}, {"kind": 2}, "ERR_INVALID_ARG", b"alibi"),
    ({}, {}, {"kind": 3, "rel_max": 2}, "ERR_INVALID_ARG", b"relative bias"),
    ({}, {}, {"kind": 8}, "ERR_INVALID_ARG", b"score kind"),
])
def test_fwd_rejects(fa, kw, bmkw, score, status, text):
    lib = fa.load_library()
    a = _args(fa, **kw)
    bm = _bm(fa, **bmkw)
    sc = fa.ScoreDesc()
    for k, v in (score or {}).items():
        setattr(sc, k, v)
    st = lib.fa_fwd(ctypes.byref(a), ctypes.byref(bm), ctypes.byref(sc), ctypes.c_void_p(FAKE), None)
    assert st == getattr(fa, status), lib.fa_last_error()
    assert text in lib.fa_last_error()


def test_fwd_rejects_null_args(fa):
    lib = fa.load_library()
    assert lib.fa_fwd(None, None, None, None, None) == fa.ERR_INVALID_ARG
    a = _args(fa)
    assert lib.fa_fwd(ctypes.byref(a), ctypes.byref(_bm(fa)), None, None, None) == fa.ERR_INVALID_ARG
    assert b"workspace" in lib.fa_last_error()


def _partials_ok(fa, a, splits):
    return fa.load_library().fa_decode_partials_bytes(ctypes.byref(a), splits)


@pytest.mark.parametrize("kw,bmkw,splits,status,text", [
    ({"dtype": 1}, {}, 1, "ERR_UNSUPPORTED", b"bf16"),
    ({}, {}, 1, "ERR_UNSUPPORTED", b"q_len <= 128"),
    ({"q_len": 1, "kv_len": 1}, {"q_len": 1, "nq": 1, "mask_kind": 3, "mask_seg_ids": FAKE, "mask_seg_batch": 1,
                    "kv_len": 1, "nkv": 1}, 1, "ERR_UNSUPPORTED", b"document"),
    ({"q_len": 1, "Hq": 32, "Hkv": 1}, {"q_len": 1, "nq": 1}, 1, "ERR_UNSUPPORTED", b"at most 16"),
    ({"q_len": 8, "Hq": 4, "Hkv": 1}, {"q_len": 8, "nq": 1}, 1, "ERR_UNSUPPORTED", b"at most 16"),
    ({"q_len": 1}, {"q_len": 1, "nq": 1}, 300, "ERR_INVALID_ARG", b"num_splits"),
    ({"q_len": 1}, {"q_len": 1, "nq": 1}, -1, "ERR_INVALID_ARG", b"num_splits"),
    ({"q_len": 1, "debug_flags": 1}, {"q_len": 1, "nq": 1}, 1, "ERR_UNSUPPORTED", b"debug"),
])
def test_decode_rejects(fa, kw, bmkw, splits, status, text):
    lib = fa.load_library()
    a = _args(fa, **kw)
    bm = _bm(fa, **bmkw)
    st = lib.fa_fwd_decode(ctypes.byref(a), ctypes.byref(bm), None, splits, ctypes.c_void_p(FAKE), 1 << 40,
                           ctypes.c_void_p(FAKE), None)
    assert st == getattr(fa, status), lib.fa_last_error()
    assert text in lib.fa_last_error()


def test_decode_partials_checks(fa):
    lib = fa.load_library()
    a = _args(fa, q_len=2, Hq=8, Hkv=2)
    bm = _bm(fa, q_len=2, nq=1)
    need = lib.fa_decode_partials_bytes(ctypes.byref(a), 5)
    assert need == 1 * 8 * 2 * 5 * (128 + 2) * 4
    assert lib.fa_decode_partials_bytes(ctypes.byref(a), 0) == 0
    assert lib.fa_fwd_decode(ctypes.byref(a), ctypes.byref(bm), None, 5, None, need, ctypes.c_void_p(FAKE),
                             None) == fa.ERR_INVALID_ARG
    assert b"partials" in lib.fa_last_error()
    assert lib.fa_fwd_decode(ctypes.byref(a), ctypes.byref(bm), None, 5, ctypes.c_void_p(FAKE + 4), need,
                             ctypes.c_void_p(FAKE), None) == fa.ERR_INVALID_ARG
    assert lib.fa_fwd_decode(ctypes.byref(a), ctypes.byref(bm), None, 5, ctypes.c_void_p(FAKE), need - 4,
                             ctypes.c_void_p(FAKE), None) == fa.ERR_INVALID_ARG
    assert b"needed" in lib.fa_last_error()


def test_decode_split_choice(fa):
    """The automatic split count lies in [1, nkv] and grows with the length."""
    lib = fa.load_library()
    a = _args(fa, q_len=1, B=1, Hq=8, Hkv=8, kv_len=32768)
    short = _bm(fa, q_len=1, nq=1, kv_len=256, nkv=2)
    long_ = _bm(fa, q_len=1, nq=1, kv_len=32768, nkv=256)
    s_short = lib.fa_decode_splits(ctypes.byref(a), ctypes.byref(short))
    s_long = lib.fa_decode_splits(ctypes.byref(a), ctypes.byref(long_))
    assert 1 <= s_short <= 2
    assert s_short <= s_long <= 256
    assert lib.fa_decode_splits(None, ctypes.byref(long_)) == 0


def _bwd_args(fa, **kw):
    a = fa.BwdArgs()
    a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = 1, 4, 4, 256, 256, 128
    a.q = a.k = a.v = a.o = a.dout = a.lse = a.dq = a.dk = a.dv = a.rowstats = FAKE
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,bmkw,status,text", [
    ({"D": 96}, {}, "ERR_UNSUPPORTED", b"head dim"),
    ({"Hkv": 3}, {}, "ERR_INVALID_ARG", b"multiple"),
    ({"dout": None}, {}, "ERR_INVALID_ARG", b"non-NULL"),
    ({"o": FAKE + 8}, {}, "ERR_INVALID_ARG", b"16-byte"),
    ({"dk": FAKE + 4}, {}, "ERR_INVALID_ARG", b"16-byte"),
    ({"rowstats": FAKE + 8}, {}, "ERR_INVALID_ARG", b"16-byte"),
    ({"lse": FAKE + 2}, {}, "ERR_INVALID_ARG", b"4-byte"),
    ({"q_len": 300}, {}, "ERR_INVALID_ARG", b"built for"),
    ({}, {"H": 2}, "ERR_INVALID_ARG", b"block mask H"),
])
def test_bwd_rejects(fa, kw, bmkw, status, text):
    lib = fa.load_library()
    cols = fa.BlockMaskColsStruct(FAKE, FAKE, FAKE, FAKE)
    st = lib.fa_bwd(ctypes.byref(_bwd_args(fa, **kw)), ctypes.byref(_bm(fa, **bmkw)), ctypes.byref(cols), None,
                    ctypes.c_void_p(FAKE), None)
    assert st == getattr(fa, status), lib.fa_last_error()
    assert text in lib.fa_last_error()


def test_bwd_needs_cols_and_workspace(fa):
    lib = fa.load_library()
    cols = fa.BlockMaskColsStruct(FAKE, FAKE, FAKE, FAKE)
    st = lib.fa_bwd(ctypes.byref(_bwd_args(fa)), ctypes.byref(_bm(fa)), None, None, ctypes.c_void_p(FAKE), None)
    assert st == fa.ERR_INVALID_ARG and b"transposed" in lib.fa_last_error()
    st = lib.fa_bwd(ctypes.byref(_bwd_args(fa)), ctypes.byref(_bm(fa)), ctypes.byref(cols), None, None, None)
    assert st == fa.ERR_INVALID_ARG and b"workspace" in lib.fa_last_error()
    st = lib.fa_block_mask_build_cols(ctypes.byref(_bm(fa)), None, ctypes.c_void_p(FAKE), None)
    assert st == fa.ERR_INVALID_ARG and b"transposed" in lib.fa_last_error()
    assert lib.fa_bwd_rowstats_bytes(2, 3, 300) == 2 * 2 * 3 * 3 * 128 * 4
    assert lib.fa_bwd_rowstats_bytes(0, 3, 300) == 0


def test_binding_rejects_wrong_tensors_before_the_library(fa):
    """The Python wrappers check dtypes and shapes of what they pass on (CPU
    tensors here: the check fails before any CUDA call)."""
    import torch
    q = torch.zeros((1, 2, 4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.bwd(q, q, q, q, torch.zeros(1), q, None)
    with pytest.raises(ValueError):
        fa.fwd_decode(q, q, q, None)
    with pytest.raises(ValueError):
        fa.fwd_decode(q.float(), q, q, None)


def test_binding_rejects_bad_forward_tensors(fa):
    """fwd and fwd_noalloc share one check of everything they hand to the C
    ABI as raw pointers (CPU tensors and wrong shapes fail before any CUDA
    call); so does block_mask for the segment ids."""
    import torch

    class _BM:
        q_len, kv_len = 4, 4

    q = torch.zeros((1, 2, 4, 64), dtype=torch.bfloat16)
    lse = torch.zeros((1, 2, 4))
    for call in (lambda **kw: fa.fwd(q, q, q, _BM(), **kw),
                 lambda **kw: fa.fwd_noalloc(q, q, q, _BM(), out=q, lse=lse, **kw)):
        with pytest.raises(ValueError, match="CUDA"):
            call()
    with pytest.raises(ValueError, match="share a dtype"):
        fa.fwd(q, q.float(), q, _BM())
    with pytest.raises(ValueError, match="seg_ids"):
        fa.block_mask("document", 1, 1, 4, 4, seg_ids=torch.zeros((1, 4), dtype=torch.int64))


def test_block_mask_size_in_bytes(fa):
    """fa_block_mask_size: nq, nkv and the bytes of each index array."""
    lib = fa.load_library()
    nq, nkv, nb = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    assert lib.fa_block_mask_size(2, 3, 300, 129, ctypes.byref(nq), ctypes.byref(nkv), ctypes.byref(nb)) == fa.OK
    assert (nq.value, nkv.value, nb.value) == (3, 2, 4 * 2 * 3 * 3 * 2)
    assert lib.fa_block_mask_size(1, 1, 69632, 69632, None, None, ctypes.byref(nb)) == fa.OK
    assert nb.value == 4 * 544 * 544
    assert lib.fa_block_mask_size(1, 0, 1, 1, None, None, None) == fa.ERR_INVALID_ARG
