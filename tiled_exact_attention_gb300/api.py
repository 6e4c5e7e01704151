"""Python entry points with the same names as the C ABI (argument marshalling only).

Tensors are torch CUDA tensors: Q, O ``[b, sq, hq, d]``, K, V ``[b, skv, hkv, d]``
(head dimension contiguous), LSE fp32 ``[b, hq, sq]``.  PyTorch provides the
device memory and the current stream; every step of the computation runs in
libfa.so.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import (FA_BF16, FA_FP16, FA_OFFSET_BOTTOM_RIGHT, BwdArgs, E4m3Args, FwdArgs, KvcacheArgs, QuantArgs,
                   SplitkvE4m3Args, VarlenArgs, check)

_DT = {torch.bfloat16: FA_BF16, torch.float16: FA_FP16}


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _strides(t: torch.Tensor):
    s = t.stride()
    return (ctypes.c_int64 * 3)(s[0], s[1], s[2])


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [b, s, h, d]")
        if t.dtype not in _DT:
            raise ValueError(f"{name} must be bf16 or fp16")
        if t.stride(3) != 1:
            raise ValueError(f"{name} must have a contiguous head dimension")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share a dtype")
    if k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("inconsistent q/k/v shapes")


def make_args(q, k, v, o, lse, *, causal: bool, scale: float | None, q_pos_offset: int | None,
              window=None, softcap: float = 0.0) -> FwdArgs:
    """Fill `fa_fwd_args`.  window = (left, right) turns on the sliding window (-1 leaves a side open);
    softcap = c > 0 caps every scaled score s to c * tanh(s / c)."""
    _check_qkv(q, k, v)
    b, sq, hq, d = q.shape
    skv, hkv = k.shape[1], k.shape[2]
    a = FwdArgs()
    a.dtype = _DT[q.dtype]
    a.b, a.sq, a.skv, a.hq, a.hkv, a.d = b, sq, skv, hq, hkv, d
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.o, a.lse = o.data_ptr(), lse.data_ptr()
    a.q_strides, a.k_strides, a.v_strides, a.o_strides = _strides(q), _strides(k), _strides(v), _strides(o)
    a.causal = 1 if causal else 0
    a.q_pos_offset = FA_OFFSET_BOTTOM_RIGHT if q_pos_offset is None else int(q_pos_offset)
    a.scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    if window is not None:
        a.local = 1
        a.window_left, a.window_right = int(window[0]), int(window[1])
    a.softcap = float(softcap)
    return a


def _outputs(q, out, lse):
    b, sq, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, hq, sq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_cuda or out.stride(3) != 1:
        raise ValueError("out must match q")
    if lse.shape != (b, hq, sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [b, hq, sq]")
    return out, lse


def fa_fwd(q, k, v, *, causal: bool = False, scale: float | None = None, q_pos_offset: int | None = None,
           out=None, lse=None, stream=None, window=None, softcap: float = 0.0):
    """Forward pass; returns (O, LSE)."""
    out, lse = _outputs(q, out, lse)
    a = make_args(q, k, v, out, lse, causal=causal, scale=scale, q_pos_offset=q_pos_offset, window=window,
                  softcap=softcap)
    check(_lib.load().fa_fwd(ctypes.byref(a), _stream_handle(stream)), "fa_fwd")
    return out, lse


def fa_num_splits_heuristic(units: int, slots: int, num_kv_blocks: int, max_splits: int = 128) -> int:
    return int(_lib.load().fa_num_splits_heuristic(units, slots, num_kv_blocks, max_splits))


def fa_splitkv_default_splits(q, k, v, *, causal=False, scale=None, q_pos_offset=None, window=None,
                              softcap: float = 0.0) -> int:
    out, lse = _outputs(q, None, None)
    a = make_args(q, k, v, out, lse, causal=causal, scale=scale, q_pos_offset=q_pos_offset, window=window,
                  softcap=softcap)
    return int(_lib.load().fa_splitkv_default_splits(ctypes.byref(a)))


def fa_splitkv_workspace_size(q, k, v, num_splits: int = 0, *, causal=False, scale=None,
                              q_pos_offset=None, window=None, softcap: float = 0.0) -> int:
    out, lse = _outputs(q, None, None)
    a = make_args(q, k, v, out, lse, causal=causal, scale=scale, q_pos_offset=q_pos_offset, window=window,
                  softcap=softcap)
    return int(_lib.load().fa_splitkv_workspace_size(ctypes.byref(a), num_splits))


def fa_fwd_splitkv(q, k, v, *, causal: bool = False, scale: float | None = None, q_pos_offset: int | None = None,
                   num_splits: int = 0, workspace=None, out=None, lse=None, stream=None, return_splits=False,
                   window=None, softcap: float = 0.0):
    """Split-KV forward + combine; returns (O, LSE) (and the split count if asked)."""
    out, lse = _outputs(q, out, lse)
    a = make_args(q, k, v, out, lse, causal=causal, scale=scale, q_pos_offset=q_pos_offset, window=window,
                  softcap=softcap)
    lib = _lib.load()
    need = int(lib.fa_splitkv_workspace_size(ctypes.byref(a), int(num_splits)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    used = ctypes.c_int32(0)
    check(lib.fa_fwd_splitkv(ctypes.byref(a), int(num_splits), ctypes.c_void_p(workspace.data_ptr()),
                             workspace.numel() * workspace.element_size(), ctypes.byref(used),
                             _stream_handle(stream)), "fa_fwd_splitkv")
    if return_splits:
        return out, lse, int(used.value)
    return out, lse


def fa_fwd_splitkv_noalloc(q, k, v, *, causal: bool = False, scale: float | None = None,
                           q_pos_offset: int | None = None, num_splits: int = 0, out=None, lse=None, stream=None,
                           return_splits=False, window=None, softcap: float = 0.0):
    """Split-KV forward that uses the library's built-in scratch instead of a workspace."""
    out, lse = _outputs(q, out, lse)
    a = make_args(q, k, v, out, lse, causal=causal, scale=scale, q_pos_offset=q_pos_offset, window=window,
                  softcap=softcap)
    used = ctypes.c_int32(0)
    check(_lib.load().fa_fwd_splitkv_noalloc(ctypes.byref(a), int(num_splits), ctypes.byref(used),
                                             _stream_handle(stream)), "fa_fwd_splitkv_noalloc")
    if return_splits:
        return out, lse, int(used.value)
    return out, lse


def make_kvcache_args(q, k, v, o, lse, *, block_table=None, seqlens_k=None, cu_seqlens_k=None,
                      max_seqlen_k: int = 0, scale: float | None = None, window_left=None,
                      softcap: float = 0.0) -> KvcacheArgs:
    """Fill `fa_kvcache_args`.  q, o: [b, hq, d]; paged k/v: [num_pages, page_size, hkv, d] with
    block_table [b, n] and seqlens_k [b] (int32); packed k/v: [total_k, hkv, d] with cu_seqlens_k [b + 1].
    window_left (not None) keeps only the last window_left + 1 keys of each sequence."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", o)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in _DT or t.stride(-1) != 1:
            raise ValueError(f"{name} must be a CUDA bf16/fp16 tensor with a contiguous last dimension")
    if q.dim() != 3 or o.shape != q.shape:
        raise ValueError("q and out must be [b, hq, d]")
    b, hq, d = q.shape
    a = KvcacheArgs()
    a.dtype = _DT[q.dtype]
    a.b, a.hq, a.d = b, hq, d
    a.q = q.data_ptr()
    a.q_strides = (ctypes.c_int64 * 2)(q.stride(0), q.stride(1))
    a.k, a.v = k.data_ptr(), v.data_ptr()
    if block_table is not None:
        if k.dim() != 4 or v.shape != k.shape or seqlens_k is None:
            raise ValueError("paged cache: k, v [num_pages, page_size, hkv, d] and seqlens_k are required")
        for t in (block_table, seqlens_k):
            if t.dtype != torch.int32 or not t.is_cuda:
                raise ValueError("block_table and seqlens_k must be CUDA int32 tensors")
        a.num_pages, a.page_size, a.hkv = k.shape[0], k.shape[1], k.shape[2]
        a.k_strides = (ctypes.c_int64 * 3)(k.stride(0), k.stride(1), k.stride(2))
        a.v_strides = (ctypes.c_int64 * 3)(v.stride(0), v.stride(1), v.stride(2))
        a.block_table = block_table.data_ptr()
        a.block_table_stride = block_table.stride(0)
        a.seqlens_k = seqlens_k.data_ptr()
    else:
        if k.dim() != 3 or v.shape != k.shape or cu_seqlens_k is None:
            raise ValueError("packed keys: k, v [total_k, hkv, d] and cu_seqlens_k are required")
        if cu_seqlens_k.dtype != torch.int32 or not cu_seqlens_k.is_cuda:
            raise ValueError("cu_seqlens_k must be a CUDA int32 tensor")
        a.num_pages, a.page_size, a.hkv = k.shape[0], 0, k.shape[1]
        a.k_strides = (ctypes.c_int64 * 3)(0, k.stride(0), k.stride(1))
        a.v_strides = (ctypes.c_int64 * 3)(0, v.stride(0), v.stride(1))
        a.cu_seqlens_k = cu_seqlens_k.data_ptr()
    a.max_seqlen_k = int(max_seqlen_k)
    a.o = o.data_ptr()
    a.o_strides = (ctypes.c_int64 * 2)(o.stride(0), o.stride(1))
    a.lse = lse.data_ptr()
    a.scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    if window_left is not None:
        a.local, a.window_left = 1, int(window_left)
    a.softcap = float(softcap)
    return a


def fa_fwd_kvcache(q, k, v, *, block_table=None, seqlens_k=None, cu_seqlens_k=None, max_seqlen_k=None,
                   scale=None, num_splits: int = 0, workspace=None, out=None, lse=None, stream=None,
                   return_splits=False, window_left=None, softcap: float = 0.0):
    """Decode one query row per sequence against a paged or packed KV cache; returns (O [b, hq, d], LSE [b, hq])."""
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    if max_seqlen_k is None:
        lens = seqlens_k if block_table is not None else (cu_seqlens_k[1:] - cu_seqlens_k[:-1])
        max_seqlen_k = int(lens.max().item()) if lens.numel() else 0
    a = make_kvcache_args(q, k, v, out, lse, block_table=block_table, seqlens_k=seqlens_k,
                          cu_seqlens_k=cu_seqlens_k, max_seqlen_k=max_seqlen_k, scale=scale,
                          window_left=window_left, softcap=softcap)
    lib = _lib.load()
    if workspace is None:
        need = int(lib.fa_kvcache_workspace_size(ctypes.byref(a), int(num_splits)))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    used = ctypes.c_int32(0)
    check(lib.fa_fwd_kvcache(ctypes.byref(a), int(num_splits), ctypes.c_void_p(workspace.data_ptr()),
                             workspace.numel() * workspace.element_size(), ctypes.byref(used),
                             _stream_handle(stream)), "fa_fwd_kvcache")
    if return_splits:
        return out, lse, int(used.value)
    return out, lse


def make_varlen_args(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int, causal: bool,
                     scale: float | None, window=None, softcap: float = 0.0) -> VarlenArgs:
    """Fill `fa_varlen_args`.  q, o: [total_q, hq, d]; k, v: [total_k, hkv, d]; lse: fp32 [hq, total_q];
    cu_seqlens_q / cu_seqlens_k: CUDA int32 [b + 1] prefix sums."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", o)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in _DT or t.dim() != 3 \
                or t.stride(2) != 1:
            raise ValueError(f"{name} must be a CUDA bf16/fp16 [rows, heads, d] tensor with contiguous d")
    if q.dtype != k.dtype or q.dtype != v.dtype or o.dtype != q.dtype:
        raise ValueError("q, k, v, out must share a dtype")
    if k.shape != v.shape or q.shape[2] != k.shape[2] or o.shape != q.shape:
        raise ValueError("inconsistent q/k/v/out shapes")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA int32 vector")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold b + 1 >= 2 entries")
    total_q, hq, d = q.shape
    total_k, hkv = k.shape[0], k.shape[1]
    if lse.shape != (hq, total_q) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [hq, total_q]")
    a = VarlenArgs()
    a.dtype = _DT[q.dtype]
    a.b = cu_seqlens_q.numel() - 1
    a.hq, a.hkv, a.d = hq, hkv, d
    a.total_q, a.total_k, a.max_seqlen_q = total_q, total_k, int(max_seqlen_q)
    a.q, a.k, a.v, a.o, a.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()
    a.q_strides = (ctypes.c_int64 * 2)(q.stride(0), q.stride(1))
    a.k_strides = (ctypes.c_int64 * 2)(k.stride(0), k.stride(1))
    a.v_strides = (ctypes.c_int64 * 2)(v.stride(0), v.stride(1))
    a.o_strides = (ctypes.c_int64 * 2)(o.stride(0), o.stride(1))
    a.cu_seqlens_q, a.cu_seqlens_k = cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr()
    a.causal = 1 if causal else 0
    if window is not None:
        a.local = 1
        a.window_left, a.window_right = int(window[0]), int(window[1])
    a.scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    a.softcap = float(softcap)
    return a


def fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int | None = None, causal: bool = False,
                  scale: float | None = None, window=None, out=None, lse=None, stream=None, softcap: float = 0.0):
    """Forward pass over packed variable-length sequences; returns (O [total_q, hq, d], LSE [hq, total_q]).
    max_seqlen_q defaults to the longest sequence (read back from the device once)."""
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    if max_seqlen_q is None:
        lens = cu_seqlens_q[1:] - cu_seqlens_q[:-1]
        max_seqlen_q = int(lens.max().item()) if lens.numel() else 0
    a = make_varlen_args(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=max_seqlen_q, causal=causal,
                         scale=scale, window=window, softcap=softcap)
    check(_lib.load().fa_fwd_varlen(ctypes.byref(a), _stream_handle(stream)), "fa_fwd_varlen")
    return out, lse


def make_bwd_args(q, k, v, o, lse, dout, dq, dk, dv, *, causal: bool, scale: float | None,
                  q_pos_offset: int | None, window=None, softcap: float = 0.0) -> BwdArgs:
    """Fill `fa_bwd_args` from [b, s, h, d] tensors (lse fp32 [b, hq, sq])."""
    _check_qkv(q, k, v)
    for name, t, like in (("o", o, q), ("dout", dout, q), ("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.shape != like.shape or t.dtype != q.dtype \
                or t.stride(3) != 1:
            raise ValueError(f"{name} must be a CUDA tensor shaped and typed like its forward counterpart")
    b, sq, hq, d = q.shape
    if lse.shape != (b, hq, sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [b, hq, sq]")
    a = BwdArgs()
    a.dtype = _DT[q.dtype]
    a.b, a.sq, a.skv, a.hq, a.hkv, a.d = b, sq, k.shape[1], hq, k.shape[2], d
    a.q, a.k, a.v, a.o, a.dout, a.lse = (t.data_ptr() for t in (q, k, v, o, dout, lse))
    a.dq, a.dk, a.dv = dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    a.q_strides, a.k_strides, a.v_strides = _strides(q), _strides(k), _strides(v)
    a.o_strides, a.do_strides = _strides(o), _strides(dout)
    a.dq_strides, a.dk_strides, a.dv_strides = _strides(dq), _strides(dk), _strides(dv)
    a.causal = 1 if causal else 0
    a.q_pos_offset = FA_OFFSET_BOTTOM_RIGHT if q_pos_offset is None else int(q_pos_offset)
    a.scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    if window is not None:
        a.local = 1
        a.window_left, a.window_right = int(window[0]), int(window[1])
    a.softcap = float(softcap)
    return a


def fa_bwd_workspace_size(q, k, v, *, causal: bool = False, scale: float | None = None,
                          q_pos_offset: int | None = None, window=None, softcap: float = 0.0) -> int:
    """Device workspace bytes fa_bwd needs for these shapes (D and L * log2(e) per padded row)."""
    b, sq, hq, _ = q.shape
    lse = torch.empty((b, hq, sq), dtype=torch.float32, device=q.device)
    a = make_bwd_args(q, k, v, q, lse, q, q, k, v, causal=causal, scale=scale, q_pos_offset=q_pos_offset,
                      window=window, softcap=softcap)
    return int(_lib.load().fa_bwd_workspace_size(ctypes.byref(a)))


def fa_bwd(q, k, v, o, lse, dout, *, causal: bool = False, scale: float | None = None,
           q_pos_offset: int | None = None, window=None, dq=None, dk=None, dv=None, workspace=None, stream=None,
           softcap: float = 0.0):
    """Backward pass for the forward call with the same arguments; returns (dQ, dK, dV)."""
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    a = make_bwd_args(q, k, v, o, lse, dout, dq, dk, dv, causal=causal, scale=scale, q_pos_offset=q_pos_offset,
                      window=window, softcap=softcap)
    lib = _lib.load()
    if workspace is None:
        need = int(lib.fa_bwd_workspace_size(ctypes.byref(a)))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    check(lib.fa_bwd(ctypes.byref(a), ctypes.c_void_p(workspace.data_ptr()),
                     workspace.numel() * workspace.element_size(), _stream_handle(stream)), "fa_bwd")
    return dq, dk, dv


def fa_quantize_e4m3(x, *, per_head: bool = False, transpose: bool = False, stream=None):
    """e4m3 codes (torch.uint8) of a [b, s, h, d] bf16/fp16 tensor and their descales (fp32).
    Codes are [b, s, h, d], or [b, h, d, s_pad] (s_pad = s rounded up to 16) with transpose=True;
    descales are [b, h, ceil(s / 128)] per 128-row block, or [b, h] with per_head=True."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype not in _DT or x.dim() != 4 or x.stride(3) != 1:
        raise ValueError("x must be a CUDA bf16/fp16 [b, s, h, d] tensor with contiguous d")
    b, s, h, d = x.shape
    if transpose:
        sp = (s + 15) // 16 * 16
        out = torch.zeros((b, h, d, sp), dtype=torch.uint8, device=x.device)
        ost = (out.stride(0), out.stride(1), out.stride(2))
    else:
        out = torch.empty((b, s, h, d), dtype=torch.uint8, device=x.device)
        ost = (out.stride(0), out.stride(1), out.stride(2))
    ds = torch.empty((b, h) if per_head else (b, h, (s + 127) // 128), dtype=torch.float32, device=x.device)
    a = QuantArgs()
    a.dtype = _DT[x.dtype]
    a.b, a.s, a.h, a.d = b, s, h, d
    a.x = x.data_ptr()
    a.x_strides = _strides(x)
    a.out = out.data_ptr()
    a.out_strides = (ctypes.c_int64 * 3)(*ost)
    a.transpose, a.per_head = int(bool(transpose)), int(bool(per_head))
    a.descale = ds.data_ptr()
    check(_lib.load().fa_quantize_e4m3(ctypes.byref(a), _stream_handle(stream)), "fa_quantize_e4m3")
    return out, ds


def quantize_qkv_e4m3(q, k, v, stream=None):
    """The inputs fa_fwd_e4m3 expects: (q8, q_descale), (k8, k_descale) per 128-row block, and V
    transposed with one descale per (batch, head)."""
    return (fa_quantize_e4m3(q, stream=stream), fa_quantize_e4m3(k, stream=stream),
            fa_quantize_e4m3(v, per_head=True, transpose=True, stream=stream))


def fa_fwd_e4m3(q8, q_descale, k8, k_descale, vt8, v_descale, *, causal: bool = False, scale: float | None = None,
                q_pos_offset: int | None = None, window=None, out=None, lse=None, stream=None):
    """Forward pass on e4m3 inputs (see fa_quantize_e4m3); returns (O bf16 [b, sq, hq, d], LSE [b, hq, sq])."""
    for name, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 4 \
                or t.stride(3) != 1:
            raise ValueError(f"{name} must be a CUDA uint8 4-D tensor with a contiguous last dimension")
    b, sq, hq, d = q8.shape
    skv, hkv = k8.shape[1], k8.shape[2]
    if k8.shape != (b, skv, hkv, d) or vt8.shape[:3] != (b, hkv, d) or vt8.shape[3] < skv:
        raise ValueError("inconsistent q8 / k8 / vt8 shapes")
    if out is None:
        out = torch.empty((b, sq, hq, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((b, hq, sq), dtype=torch.float32, device=q8.device)
    a = E4m3Args()
    a.b, a.sq, a.skv, a.hq, a.hkv, a.d = b, sq, skv, hq, hkv, d
    a.q, a.k, a.vt = q8.data_ptr(), k8.data_ptr(), vt8.data_ptr()
    a.q_descale, a.k_descale, a.v_descale = q_descale.data_ptr(), k_descale.data_ptr(), v_descale.data_ptr()
    a.o, a.lse = out.data_ptr(), lse.data_ptr()
    a.q_strides = (ctypes.c_int64 * 3)(q8.stride(0), q8.stride(1), q8.stride(2))
    a.k_strides = (ctypes.c_int64 * 3)(k8.stride(0), k8.stride(1), k8.stride(2))
    a.vt_strides = (ctypes.c_int64 * 3)(vt8.stride(0), vt8.stride(1), vt8.stride(2))
    a.o_strides = _strides(out)
    a.causal = 1 if causal else 0
    a.q_pos_offset = FA_OFFSET_BOTTOM_RIGHT if q_pos_offset is None else int(q_pos_offset)
    a.scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    if window is not None:
        a.local = 1
        a.window_left, a.window_right = int(window[0]), int(window[1])
    check(_lib.load().fa_fwd_e4m3(ctypes.byref(a), _stream_handle(stream)), "fa_fwd_e4m3")
    return out, lse


def make_splitkv_e4m3_args(q, k8, k_descale, v8, v_descale, o, lse, *, scale=None) -> SplitkvE4m3Args:
    """Fill `fa_splitkv_e4m3_args`: q, o [b, hq, d] bf16/fp16; k8, v8 e4m3 codes (torch.uint8) [b, skv, hkv, d];
    k_descale [b, hkv, ceil(skv / 128)], v_descale [b, hkv] (fa_quantize_e4m3, V with per_head=True)."""
    if not isinstance(q, torch.Tensor) or not q.is_cuda or q.dtype not in _DT or q.dim() != 3 or q.stride(2) != 1:
        raise ValueError("q must be a CUDA bf16/fp16 [b, hq, d] tensor with contiguous d")
    for name, t in (("k8", k8), ("v8", v8)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 4 \
                or t.stride(3) != 1:
            raise ValueError(f"{name} must be a CUDA uint8 [b, skv, hkv, d] tensor with contiguous d")
    b, hq, d = q.shape
    skv, hkv = k8.shape[1], k8.shape[2]
    if k8.shape != (b, skv, hkv, d) or v8.shape != k8.shape or o.shape != q.shape:
        raise ValueError("inconsistent q / k8 / v8 / out shapes")
    a = SplitkvE4m3Args()
    a.dtype = _DT[q.dtype]
    a.b, a.skv, a.hq, a.hkv, a.d = b, skv, hq, hkv, d
    a.q = q.data_ptr()
    a.q_strides = (ctypes.c_int64 * 2)(q.stride(0), q.stride(1))
    a.k, a.v = k8.data_ptr(), v8.data_ptr()
    a.k_strides = (ctypes.c_int64 * 3)(k8.stride(0), k8.stride(1), k8.stride(2))
    a.v_strides = (ctypes.c_int64 * 3)(v8.stride(0), v8.stride(1), v8.stride(2))
    a.k_descale, a.v_descale = k_descale.data_ptr(), v_descale.data_ptr()
    a.o = o.data_ptr()
    a.o_strides = (ctypes.c_int64 * 2)(o.stride(0), o.stride(1))
    a.lse = lse.data_ptr()
    a.scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    return a


def fa_fwd_splitkv_e4m3(q, k8, k_descale, v8, v_descale, *, scale=None, num_splits: int = 0, workspace=None,
                        out=None, lse=None, stream=None, return_splits=False):
    """Decode one query row per (batch, head) against e4m3 keys and values; returns (O [b, hq, d], LSE [b, hq])."""
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    a = make_splitkv_e4m3_args(q, k8, k_descale, v8, v_descale, out, lse, scale=scale)
    lib = _lib.load()
    if workspace is None:
        need = int(lib.fa_splitkv_e4m3_workspace_size(ctypes.byref(a), int(num_splits)))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    used = ctypes.c_int32(0)
    check(lib.fa_fwd_splitkv_e4m3(ctypes.byref(a), int(num_splits), ctypes.c_void_p(workspace.data_ptr()),
                                  workspace.numel() * workspace.element_size(), ctypes.byref(used),
                                  _stream_handle(stream)), "fa_fwd_splitkv_e4m3")
    if return_splits:
        return out, lse, int(used.value)
    return out, lse


def fa_splitkv_combine(o_part, lse_part, out, lse=None, stream=None):
    """Merge fp32 partials o_part [ns, b, hq, sq, d], lse_part [ns, b, hq, sq] into out [b, sq, hq, d]."""
    ns, b, hq, sq, d = o_part.shape
    if not (o_part.is_cuda and lse_part.is_cuda and out.is_cuda):
        raise ValueError("tensors must be on the GPU")
    if o_part.dtype != torch.float32 or lse_part.dtype != torch.float32 or not o_part.is_contiguous() \
            or not lse_part.is_contiguous() or lse_part.shape != (ns, b, hq, sq):
        raise ValueError("partials must be contiguous fp32")
    if out.dtype not in _DT or out.shape != (b, sq, hq, d) or out.stride(3) != 1:
        raise ValueError("out must be [b, sq, hq, d] bf16/fp16")
    st = _strides(out)
    lp = ctypes.c_void_p(lse.data_ptr()) if lse is not None else ctypes.c_void_p(0)
    check(_lib.load().fa_splitkv_combine(ctypes.c_void_p(o_part.data_ptr()), ctypes.c_void_p(lse_part.data_ptr()),
                                         ns, b, hq, sq, d, _DT[out.dtype], ctypes.c_void_p(out.data_ptr()), st, lp,
                                         _stream_handle(stream)), "fa_splitkv_combine")
    return out, lse


def fa_sync_status(stream=None) -> int:
    """Synchronise the stream; return the status code (0 = ok, 4 = a device wait timed out)."""
    return int(_lib.load().fa_sync_status(_stream_handle(stream)))


def fa_selftest_wait_timeout(stream=None) -> None:
    check(_lib.load().fa_selftest_wait_timeout(_stream_handle(stream)), "fa_selftest_wait_timeout")


def fa_version() -> int:
    return int(_lib.load().fa_version())
