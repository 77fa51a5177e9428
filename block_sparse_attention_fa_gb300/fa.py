"""Thin ctypes binding over the C ABI in ``include/fa.h``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_lib/libfa_gb300.so``.  PyTorch supplies device memory and the
current stream.  If the library is missing or fails to load this module
raises; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libfa_gb300.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK = range(6)
BF16, FP32 = 0, 1
MASK_KINDS = {"full": 0, "causal": 1, "sliding_window": 2, "document": 3, "prefix_lm": 4, "table": 5}
SCORE_KINDS = {"none": 0, "softcap": 1, "alibi": 2, "rel_bias": 3, "alibi_softcap": 4}
OUT_FP32 = 1
DEBUG_DROP_FIRST_LOAD = 1
BLOCK = 128

SYMBOLS = ("fa_workspace_bytes", "fa_block_mask_shape", "fa_block_mask_size", "fa_block_mask_build", "fa_fwd",
           "fa_fwd_noalloc", "fa_fwd_decode", "fa_decode_partials_bytes", "fa_decode_splits", "fa_bwd",
           "fa_block_mask_build_cols", "fa_bwd_rowstats_bytes", "fa_workspace_check", "fa_last_error", "fa_version")


class FAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"fa status {status}: {msg}")
        self.status = status


class MaskDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32), ("prefix_len", ctypes.c_int32),
                ("seg_batch", ctypes.c_int32), ("seg_ids", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("table_batch", ctypes.c_int32)]


class BlockMaskStruct(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("block_q", ctypes.c_int32), ("block_kv", ctypes.c_int32),
                ("nq", ctypes.c_int32), ("nkv", ctypes.c_int32),
                ("kv_num_blocks", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
                ("full_kv_num_blocks", ctypes.c_void_p), ("full_kv_indices", ctypes.c_void_p),
                ("mask", MaskDesc)]


class ScoreDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                ("rel_bias", ctypes.c_void_p), ("rel_max", ctypes.c_int32)]


class FwdArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("B", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("q_len", ctypes.c_int32), ("kv_len", ctypes.c_int32),
                ("D", ctypes.c_int32), ("scale", ctypes.c_float),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("timeout_ms", ctypes.c_uint32), ("flags", ctypes.c_uint32),
                ("debug_flags", ctypes.c_uint32)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("D", ctypes.c_int32), ("scale", ctypes.c_float),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("o", ctypes.c_void_p),
                ("dout", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("dq", ctypes.c_void_p),
                ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p), ("rowstats", ctypes.c_void_p),
                ("timeout_ms", ctypes.c_uint32)]


class BlockMaskColsStruct(ctypes.Structure):
    _fields_ = [("q_num_blocks", ctypes.c_void_p), ("q_indices", ctypes.c_void_p),
                ("full_q_num_blocks", ctypes.c_void_p), ("full_q_indices", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run `python -m block_sparse_attention_fa_gb300.build`)")
    h = ctypes.CDLL(path)
    h.fa_workspace_bytes.restype = ctypes.c_size_t
    h.fa_workspace_bytes.argtypes = []
    h.fa_block_mask_shape.restype = ctypes.c_int
    h.fa_block_mask_shape.argtypes = [ctypes.c_int32] * 4 + [ctypes.POINTER(ctypes.c_int32)] * 2 + \
        [ctypes.POINTER(ctypes.c_int64)]
    h.fa_block_mask_size.restype = ctypes.c_int
    h.fa_block_mask_size.argtypes = [ctypes.c_int32] * 4 + [ctypes.POINTER(ctypes.c_int32)] * 2 + \
        [ctypes.POINTER(ctypes.c_size_t)]
    h.fa_block_mask_build.restype = ctypes.c_int
    h.fa_block_mask_build.argtypes = [ctypes.POINTER(BlockMaskStruct), ctypes.c_void_p, ctypes.c_void_p]
    h.fa_fwd.restype = ctypes.c_int
    h.fa_fwd.argtypes = [ctypes.POINTER(FwdArgs), ctypes.POINTER(BlockMaskStruct),
                         ctypes.POINTER(ScoreDesc), ctypes.c_void_p, ctypes.c_void_p]
    h.fa_fwd_noalloc.restype = ctypes.c_int
    h.fa_fwd_noalloc.argtypes = [ctypes.POINTER(FwdArgs), ctypes.POINTER(BlockMaskStruct),
                                 ctypes.POINTER(ScoreDesc), ctypes.c_void_p]
    h.fa_fwd_decode.restype = ctypes.c_int
    h.fa_fwd_decode.argtypes = [ctypes.POINTER(FwdArgs), ctypes.POINTER(BlockMaskStruct),
                                ctypes.POINTER(ScoreDesc), ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                ctypes.c_void_p, ctypes.c_void_p]
    h.fa_decode_partials_bytes.restype = ctypes.c_size_t
    h.fa_decode_partials_bytes.argtypes = [ctypes.POINTER(FwdArgs), ctypes.c_int32]
    h.fa_decode_splits.restype = ctypes.c_int32
    h.fa_decode_splits.argtypes = [ctypes.POINTER(FwdArgs), ctypes.POINTER(BlockMaskStruct)]
    h.fa_block_mask_build_cols.restype = ctypes.c_int
    h.fa_block_mask_build_cols.argtypes = [ctypes.POINTER(BlockMaskStruct), ctypes.POINTER(BlockMaskColsStruct),
                                           ctypes.c_void_p, ctypes.c_void_p]
    h.fa_bwd_rowstats_bytes.restype = ctypes.c_size_t
    h.fa_bwd_rowstats_bytes.argtypes = [ctypes.c_int32] * 3
    h.fa_bwd.restype = ctypes.c_int
    h.fa_bwd.argtypes = [ctypes.POINTER(BwdArgs), ctypes.POINTER(BlockMaskStruct),
                         ctypes.POINTER(BlockMaskColsStruct), ctypes.POINTER(ScoreDesc), ctypes.c_void_p,
                         ctypes.c_void_p]
    h.fa_workspace_check.restype = ctypes.c_int
    h.fa_workspace_check.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    h.fa_last_error.restype = ctypes.c_char_p
    h.fa_last_error.argtypes = []
    h.fa_version.restype = ctypes.c_char_p
    h.fa_version.argtypes = []
    _lib = h
    return h


def _check(status: int):
    if status != OK:
        raise FAError(status, load_library().fa_last_error().decode())


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class Workspace:
    """fa_workspace_bytes() zero-filled device bytes for status flags."""

    def __init__(self, device=None):
        n = load_library().fa_workspace_bytes()
        self.tensor = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())

    def check(self, stream=None):
        """Synchronise and raise FAError if a kernel flagged a device-side failure."""
        _check(load_library().fa_workspace_check(self.ptr, _stream_ptr(stream)))


_default_ws = {}


def default_workspace(device, stream=None) -> Workspace:
    """The binding's workspace for (device, stream).  Launches that may run
    concurrently must not share a workspace (the forward keeps its work
    queue there), so each stream gets its own."""
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    if stream is None:
        stream = torch.cuda.current_stream(idx)
    key = (idx, stream.cuda_stream)
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device("cuda", idx))
    return _default_ws[key]


class BlockMask:
    """A BlockMask over 128 x 128 tiles (device int32 arrays + the mask_mod)."""

    def __init__(self, B, H, q_len, kv_len, mask, window, prefix_len, seg_ids, device, table=None):
        lib = load_library()
        nq, nkv, ne = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        _check(lib.fa_block_mask_shape(B, H, q_len, kv_len, ctypes.byref(nq), ctypes.byref(nkv), ctypes.byref(ne)))
        self.B, self.H, self.q_len, self.kv_len = B, H, q_len, kv_len
        self.nq, self.nkv = nq.value, nkv.value
        self.mask, self.window, self.prefix_len = mask, window, prefix_len
        self.seg_ids = seg_ids
        self.table = table
        self.kv_num_blocks = torch.empty((B, H, self.nq), dtype=torch.int32, device=device)
        self.kv_indices = torch.empty((B, H, self.nq, self.nkv), dtype=torch.int32, device=device)
        self.full_kv_num_blocks = torch.empty((B, H, self.nq), dtype=torch.int32, device=device)
        self.full_kv_indices = torch.empty((B, H, self.nq, self.nkv), dtype=torch.int32, device=device)
        s = BlockMaskStruct()
        s.B, s.H, s.q_len, s.kv_len = B, H, q_len, kv_len
        s.block_q = s.block_kv = BLOCK
        s.nq, s.nkv = self.nq, self.nkv
        s.kv_num_blocks = self.kv_num_blocks.data_ptr()
        s.kv_indices = self.kv_indices.data_ptr()
        s.full_kv_num_blocks = self.full_kv_num_blocks.data_ptr()
        s.full_kv_indices = self.full_kv_indices.data_ptr()
        s.mask.kind = MASK_KINDS[mask]
        s.mask.window = window
        s.mask.prefix_len = prefix_len
        if seg_ids is not None:
            s.mask.seg_batch = seg_ids.shape[0]
            s.mask.seg_ids = seg_ids.data_ptr()
        if table is not None:
            s.mask.table_batch = table.shape[0]
            s.mask.table = table.data_ptr()
        self.struct = s

    def rebuild(self, stream=None, workspace: Optional["Workspace"] = None):
        """Run fa_block_mask_build again into this BlockMask's own buffers
        (e.g. after the segment ids changed in place); capturable in a CUDA
        graph since it allocates nothing."""
        ws = workspace or default_workspace(self.kv_num_blocks.device, stream)
        _check(load_library().fa_block_mask_build(ctypes.byref(self.struct), ws.ptr, _stream_ptr(stream)))
        return self

    def cols(self, stream=None, workspace: Optional["Workspace"] = None, rebuild: bool = False) -> dict:
        """The transposed lists (fa_block_mask_build_cols: the q-blocks that
        visit each kv block), built on first use and kept with the mask."""
        if getattr(self, "_cols", None) is None or rebuild:
            dev = self.kv_num_blocks.device
            if getattr(self, "_cols", None) is None:
                t = {"q_num_blocks": torch.empty((self.B, self.H, self.nkv), dtype=torch.int32, device=dev),
                     "q_indices": torch.empty((self.B, self.H, self.nkv, self.nq), dtype=torch.int32, device=dev),
                     "full_q_num_blocks": torch.empty((self.B, self.H, self.nkv), dtype=torch.int32, device=dev),
                     "full_q_indices": torch.empty((self.B, self.H, self.nkv, self.nq), dtype=torch.int32,
                                                   device=dev)}
                cs = BlockMaskColsStruct()
                for k, v in t.items():
                    setattr(cs, k, v.data_ptr())
                self._cols, self._cols_struct = t, cs
            ws = workspace or default_workspace(dev, stream)
            _check(load_library().fa_block_mask_build_cols(ctypes.byref(self.struct), ctypes.byref(self._cols_struct),
                                                           ws.ptr, _stream_ptr(stream)))
        return self._cols

    def visited_tiles(self) -> int:
        return int(self.kv_num_blocks.sum().item() + self.full_kv_num_blocks.sum().item())

    def numpy(self) -> dict:
        return {k: getattr(self, k).cpu().numpy() for k in
                ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices")}


def block_mask(mask: str, B: int, H: int, q_len: int, kv_len: int, *, window: int = 0, prefix_len: int = 0,
               seg_ids: Optional[torch.Tensor] = None, table: Optional[torch.Tensor] = None, device=None,
               stream=None, workspace: Optional[Workspace] = None) -> BlockMask:
    """Build a BlockMask (fa_block_mask_build) for a built-in mask_mod.

    mask "table": ``table`` is the packed lookup table of the C ABI, a CUDA
    int32 tensor [table_batch, q_len, ceil(kv_len / 32)] whose bit j % 32 of
    word j // 32 in row i says whether query i attends to key j."""
    if table is not None:
        if table.dim() == 2:
            table = table[None]
        if table.dtype != torch.int32 or not table.is_cuda or tuple(table.shape[1:]) != (q_len, (kv_len + 31) // 32):
            raise ValueError("table must be a CUDA int32 tensor [batch, q_len, ceil(kv_len / 32)]")
        table = table.contiguous()
        device = table.device
    if seg_ids is not None:
        if seg_ids.dim() == 1:
            seg_ids = seg_ids[None]
        if seg_ids.dtype != torch.int32 or not seg_ids.is_cuda or seg_ids.dim() != 2:
            raise ValueError("seg_ids must be a CUDA int32 tensor [seg_batch, kv_len]")
        if seg_ids.shape[1] != kv_len or seg_ids.shape[0] not in (1, B):
            raise ValueError(f"seg_ids must hold kv_len={kv_len} ids per row and 1 or B={B} rows "
                             f"(got {tuple(seg_ids.shape)})")
        seg_ids = seg_ids.contiguous()
        device = seg_ids.device
    device = torch.device(device or "cuda")
    bm = BlockMask(B, H, q_len, kv_len, mask, window, prefix_len, seg_ids, device, table=table)
    ws = workspace or default_workspace(device, stream)
    _check(load_library().fa_block_mask_build(ctypes.byref(bm.struct), ws.ptr, _stream_ptr(stream)))
    return bm


def _check_fwd_tensors(q, k, v, out, lse, out_fp32, alibi_slopes, rel_bias, rel_max, bm):
    """The shapes, dtypes and placement fa_fwd / fa_fwd_noalloc read and write
    through raw pointers, which the C ABI cannot see: anything wrong here
    would become an out-of-bounds device access, so it is rejected first."""
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"unsupported dtype {q.dtype}")
    for t in (k, v):
        if t.dtype != q.dtype:
            raise ValueError("q, k and v must share a dtype")
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dim() == 4):
            raise ValueError("q, k, v must be contiguous CUDA tensors [B, H, T, D]")
    B, Hq, Tq, D = q.shape
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("k and v must have the same shape")
    if k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, kv_len, D] with q's B and D")
    if out_fp32 and q.dtype != torch.bfloat16:
        raise ValueError("out_fp32 applies to bf16 inputs only")
    want = torch.float32 if (out_fp32 or q.dtype == torch.float32) else torch.bfloat16
    if out.dtype != want or not out.is_cuda or not out.is_contiguous() or tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must be a contiguous CUDA {want} tensor of q's shape")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Tq):
        raise ValueError("lse must be a contiguous CUDA float32 tensor [B, Hq, q_len]")
    if alibi_slopes is not None:
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_cuda or not alibi_slopes.is_contiguous() \
                or alibi_slopes.numel() < Hq:
            raise ValueError("alibi_slopes must be a contiguous CUDA float32 tensor of at least Hq entries")
    if rel_bias is not None:
        if rel_bias.dtype != torch.float32 or not rel_bias.is_cuda or not rel_bias.is_contiguous() \
                or rel_bias.numel() < Hq * (2 * rel_max + 1):
            raise ValueError("rel_bias must be a contiguous CUDA float32 tensor [Hq, 2 rel_max + 1]")
    if bm.q_len != Tq or bm.kv_len != k.shape[2]:
        raise ValueError(f"the BlockMask was built for ({bm.q_len}, {bm.kv_len}), not ({Tq}, {k.shape[2]})")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, bm: BlockMask, *, score: str = "none",
        softcap: float = 0.0, alibi_slopes: Optional[torch.Tensor] = None,
        rel_bias: Optional[torch.Tensor] = None, rel_max: int = 0, scale: Optional[float] = None,
        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
        workspace: Optional[Workspace] = None, stream=None, timeout_ms: int = 0, debug_flags: int = 0,
        out_fp32: bool = False):
    """Block-sparse attention forward (fa_fwd); returns (o, lse).

    ``out_fp32`` writes O in fp32 for bf16 inputs (FA_OUT_FP32)."""
    dt = {torch.bfloat16: BF16, torch.float32: FP32}.get(q.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, T, D]")
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    _check_fwd_tensors(q, k, v, out, lse, out_fp32, alibi_slopes, rel_bias, rel_max, bm)
    a = FwdArgs()
    a.dtype, a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = dt, B, Hq, Hkv, Tq, Tkv, D
    a.scale = 0.0 if scale is None else float(scale)
    a.q, a.k, a.v, a.o, a.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr()
    a.timeout_ms, a.debug_flags = timeout_ms, debug_flags
    a.flags = OUT_FP32 if out_fp32 else 0
    sc = ScoreDesc()
    sc.kind = SCORE_KINDS[score]
    sc.softcap = softcap
    if alibi_slopes is not None:
        sc.alibi_slopes = alibi_slopes.data_ptr()
    if rel_bias is not None:
        sc.rel_bias = rel_bias.data_ptr()
        sc.rel_max = rel_max
    ws = workspace or default_workspace(q.device, stream)
    _check(load_library().fa_fwd(ctypes.byref(a), ctypes.byref(bm.struct), ctypes.byref(sc), ws.ptr,
                                 _stream_ptr(stream)))
    return out, lse


def fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, bm: BlockMask, *, out: torch.Tensor,
                lse: torch.Tensor, score: str = "none", softcap: float = 0.0,
                alibi_slopes: Optional[torch.Tensor] = None, rel_bias: Optional[torch.Tensor] = None,
                rel_max: int = 0, scale: Optional[float] = None, stream=None, out_fp32: bool = False):
    """fa_fwd_noalloc: the forward for callers that cannot allocate device
    memory.  The caller passes preallocated `out` and `lse`; no workspace is
    taken (the library's scratch is a static device array)."""
    dt = {torch.bfloat16: BF16, torch.float32: FP32}.get(q.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {q.dtype}")
    _check_fwd_tensors(q, k, v, out, lse, out_fp32, alibi_slopes, rel_bias, rel_max, bm)
    B, Hq, Tq, D = q.shape
    a = FwdArgs()
    a.dtype, a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = dt, B, Hq, k.shape[1], Tq, k.shape[2], D
    a.scale = 0.0 if scale is None else float(scale)
    a.q, a.k, a.v, a.o, a.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr()
    a.flags = OUT_FP32 if out_fp32 else 0
    sc = ScoreDesc()
    sc.kind = SCORE_KINDS[score]
    sc.softcap = softcap
    if alibi_slopes is not None:
        sc.alibi_slopes = alibi_slopes.data_ptr()
    if rel_bias is not None:
        sc.rel_bias = rel_bias.data_ptr()
        sc.rel_max = rel_max
    _check(load_library().fa_fwd_noalloc(ctypes.byref(a), ctypes.byref(bm.struct), ctypes.byref(sc),
                                         _stream_ptr(stream)))
    return out, lse


def _score_desc(score, softcap, alibi_slopes, rel_bias, rel_max) -> ScoreDesc:
    sc = ScoreDesc()
    sc.kind = SCORE_KINDS[score]
    sc.softcap = softcap
    if alibi_slopes is not None:
        sc.alibi_slopes = alibi_slopes.data_ptr()
    if rel_bias is not None:
        sc.rel_bias = rel_bias.data_ptr()
        sc.rel_max = rel_max
    return sc


def decode_args(q: torch.Tensor, k: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, v: torch.Tensor = None,
                scale: Optional[float] = None, out_fp32: bool = False) -> FwdArgs:
    """The fa_fwd_args of a bf16 decoding call (shapes taken from q and k)."""
    B, Hq, Tq, D = q.shape
    a = FwdArgs()
    a.dtype, a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = BF16, B, Hq, k.shape[1], Tq, k.shape[2], D
    a.scale = 0.0 if scale is None else float(scale)
    a.q, a.k, a.o, a.lse = q.data_ptr(), k.data_ptr(), out.data_ptr(), lse.data_ptr()
    a.v = (v if v is not None else k).data_ptr()
    a.flags = OUT_FP32 if out_fp32 else 0
    return a


def decode_splits(q: torch.Tensor, k: torch.Tensor, bm: BlockMask) -> int:
    """The split count fa_fwd_decode picks for num_splits=0 on this device."""
    a = decode_args(q, k, q, q)
    return int(load_library().fa_decode_splits(ctypes.byref(a), ctypes.byref(bm.struct)))


def decode_partials(q: torch.Tensor, num_splits: int) -> torch.Tensor:
    """fp32 scratch for fa_fwd_decode: [B, Hq, q_len, num_splits, D + 2]."""
    B, Hq, Tq, D = q.shape
    return torch.empty((B, Hq, Tq, num_splits, D + 2), dtype=torch.float32, device=q.device)


def fwd_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, bm: BlockMask, *, score: str = "none",
               softcap: float = 0.0, alibi_slopes: Optional[torch.Tensor] = None,
               rel_bias: Optional[torch.Tensor] = None, rel_max: int = 0, scale: Optional[float] = None,
               num_splits: int = 0, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               partials: Optional[torch.Tensor] = None, workspace: Optional[Workspace] = None, stream=None,
               timeout_ms: int = 0, out_fp32: bool = False):
    """Split-KV decoding forward (fa_fwd_decode) for bf16 q of at most 128
    rows; returns (o, lse).  ``num_splits`` 0 lets the library choose;
    ``partials`` (see decode_partials) is allocated when not given."""
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("fwd_decode takes bf16 q, k, v")
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dim() == 4):
            raise ValueError("q, k, v must be contiguous CUDA tensors [B, H, T, D]")
    B, Hq, Tq, D = q.shape
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    want = torch.float32 if out_fp32 else torch.bfloat16
    if out.dtype != want or not out.is_cuda or not out.is_contiguous() or tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must be a contiguous CUDA {want} tensor of q's shape")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Tq):
        raise ValueError("lse must be a contiguous CUDA float32 tensor [B, Hq, q_len]")
    a = decode_args(q, k, out, lse, v=v, scale=scale, out_fp32=out_fp32)
    a.timeout_ms = timeout_ms
    lib = load_library()
    if num_splits == 0:
        num_splits = int(lib.fa_decode_splits(ctypes.byref(a), ctypes.byref(bm.struct))) or 1
    if partials is None:
        partials = decode_partials(q, num_splits)
    if partials.dtype != torch.float32 or not partials.is_cuda or not partials.is_contiguous():
        raise ValueError("partials must be a contiguous CUDA float32 tensor (see decode_partials)")
    sc = _score_desc(score, softcap, alibi_slopes, rel_bias, rel_max)
    ws = workspace or default_workspace(q.device, stream)
    _check(lib.fa_fwd_decode(ctypes.byref(a), ctypes.byref(bm.struct), ctypes.byref(sc), num_splits,
                             ctypes.c_void_p(partials.data_ptr()), partials.numel() * partials.element_size(),
                             ws.ptr, _stream_ptr(stream)))
    return out, lse


def bwd_rowstats(q: torch.Tensor) -> torch.Tensor:
    """fp32 scratch for fa_bwd: fa_bwd_rowstats_bytes() bytes as a flat tensor."""
    B, Hq, Tq, _ = q.shape
    n = load_library().fa_bwd_rowstats_bytes(B, Hq, Tq) // 4
    return torch.empty(n, dtype=torch.float32, device=q.device)


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, bm: BlockMask, *, score: str = "none", softcap: float = 0.0,
        alibi_slopes: Optional[torch.Tensor] = None, rel_bias: Optional[torch.Tensor] = None, rel_max: int = 0,
        scale: Optional[float] = None, dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
        dv: Optional[torch.Tensor] = None, rowstats: Optional[torch.Tensor] = None,
        workspace: Optional[Workspace] = None, stream=None, timeout_ms: int = 0):
    """Backward of fwd (fa_bwd) for bf16 q, k, v, the forward's bf16 o and
    its lse, and the upstream gradient dout; returns fp32 (dq, dk, dv).  The
    BlockMask's transposed lists are built on first use (BlockMask.cols)."""
    for t in (q, k, v, o, dout):
        if t.dtype != torch.bfloat16 or not (t.is_cuda and t.is_contiguous() and t.dim() == 4):
            raise ValueError("q, k, v, o and dout must be contiguous CUDA bf16 tensors [B, H, T, D]")
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    if tuple(k.shape) != tuple(v.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, kv_len, D] with q's B and D")
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty((B, Hq, Tq, D), **f32) if dq is None else dq
    dk = torch.empty((B, Hkv, Tkv, D), **f32) if dk is None else dk
    dv = torch.empty((B, Hkv, Tkv, D), **f32) if dv is None else dv
    rowstats = bwd_rowstats(q) if rowstats is None else rowstats
    for name, t, shape in (("lse", lse, (B, Hq, Tq)), ("dq", dq, (B, Hq, Tq, D)), ("dk", dk, (B, Hkv, Tkv, D)),
                           ("dv", dv, (B, Hkv, Tkv, D))):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape {shape}")
    need = load_library().fa_bwd_rowstats_bytes(B, Hq, Tq)
    if rowstats.dtype != torch.float32 or not rowstats.is_cuda or not rowstats.is_contiguous() \
            or rowstats.numel() * 4 < need:
        raise ValueError(f"rowstats must be a contiguous CUDA float32 tensor of at least {need} bytes")
    if bm.q_len != Tq or bm.kv_len != Tkv:
        raise ValueError(f"the BlockMask was built for ({bm.q_len}, {bm.kv_len}), not ({Tq}, {Tkv})")
    a = BwdArgs()
    a.B, a.Hq, a.Hkv, a.q_len, a.kv_len, a.D = B, Hq, Hkv, Tq, Tkv, D
    a.scale = 0.0 if scale is None else float(scale)
    a.q, a.k, a.v, a.o, a.dout = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr()
    a.lse, a.dq, a.dk, a.dv = lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    a.rowstats = rowstats.data_ptr()
    a.timeout_ms = timeout_ms
    sc = _score_desc(score, softcap, alibi_slopes, rel_bias, rel_max)
    ws = workspace or default_workspace(q.device, stream)
    bm.cols(stream=stream, workspace=ws)
    _check(load_library().fa_bwd(ctypes.byref(a), ctypes.byref(bm.struct), ctypes.byref(bm._cols_struct),
                                 ctypes.byref(sc), ws.ptr, _stream_ptr(stream)))
    return dq, dk, dv


def version() -> str:
    return load_library().fa_version().decode()
