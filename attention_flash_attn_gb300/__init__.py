"""GB300 (sm_103a) fused attention with tanh soft-capping, a learnable sink, GQA and
causal / sliding-window / packed-segment masks.

Thin Python binding over the C ABI of ``libattn_gb300.so`` (include/attn_gb300.h):
PyTorch supplies device memory and the current stream; every step of the forward and
backward runs in the library's CUDA kernels.  The names follow the C entry points.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _capi
from ._capi import AttnArgs, AttnError, lib  # noqa: F401

__all__ = ["attn_fwd", "attn_fwd_noalloc", "attn_bwd", "attn_meta", "attn_check_device_status", "attn_path_name",
           "attn_launch_counter", "attn_profile_next_main_kernel", "attn_profile_next_aux_kernels", "AttnError",
           "build_args"]

_DTYPES = {torch.bfloat16: _capi.ATTN_DTYPE_BF16, torch.float32: _capi.ATTN_DTYPE_F32}
_ws_cache: dict = {}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _on_device(where: str, device: torch.device, tensors):
    """Every tensor the library will read or write must live on the CUDA device of q: a host
    pointer handed to a kernel would fault the GPU instead of failing the call."""
    if device.type != "cuda":
        raise ValueError(f"{where}: q, k, v must be CUDA tensors")
    for t in tensors:
        if t is not None and t.device != device:
            raise ValueError(f"{where}: every tensor must be on {device} (got one on {t.device})")


def _dense(where: str, name: str, t: torch.Tensor, shape, dtype):
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{where}: {name} must be a contiguous {dtype} tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def build_args(q, k, v, *, causal=False, window=0, softcap=0.0, sink=None, scale=None,
               bias=None, seg_q=None, seg_k=None, cu_seqlens=None, off_by_one=False, kv_splits=0,
               cu_seqlens_k=None, meta=None):
    """Fill an ``attn_args`` from tensors.  Returns (args, tensors kept alive).
    cu_seqlens_k: key boundaries of the cu_seqlens sequences (varlen with Sq != Sk per sequence).
    off_by_one: the off-by-one softmax (an extra column of logit 0 per row, no gradient).
    kv_splits: split-KV forward into that many key shares per query tile (0 / 1: off).
    meta: mask metadata from attn_meta for these same arguments (or None)."""
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share dtype bfloat16 or float32")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, S, H, D]")
    for t in (q, k, v):
        if t.stride(-1) != 1:
            raise ValueError("the head dimension must be contiguous")
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must both be [B, Sk, Hkv, D] with q's B and D")
    a = AttnArgs()
    a.dtype = _DTYPES[q.dtype]
    a.B, a.Sq, a.Sk, a.Hq, a.Hkv, a.D = B, Sq, Sk, Hq, Hkv, D
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.q_stride_b, a.q_stride_s, a.q_stride_h = q.stride(0), q.stride(1), q.stride(2)
    a.k_stride_b, a.k_stride_s, a.k_stride_h = k.stride(0), k.stride(1), k.stride(2)
    a.v_stride_b, a.v_stride_s, a.v_stride_h = v.stride(0), v.stride(1), v.stride(2)
    keep = [q, k, v]
    if bias is not None:
        if (bias.dtype != q.dtype or bias.dim() != 4 or tuple(bias.shape[2:]) != (Sq, Sk)
                or bias.shape[0] not in (1, B) or bias.shape[1] not in (1, Hq)):
            raise ValueError("bias must be [1|B, 1|Hq, Sq, Sk] in the dtype of q")
        if bias.stride(-1) != 1 or bias.stride(-2) != Sk:
            raise ValueError("bias rows must be dense [Sq, Sk]")
        a.bias = bias.data_ptr()
        a.bias_stride_b = 0 if bias.shape[0] == 1 else bias.stride(0)
        a.bias_stride_h = 0 if bias.shape[1] == 1 else bias.stride(1)
        keep.append(bias)
    if seg_q is not None:
        if seg_k is None and Sq != Sk:
            raise ValueError("seg_k [B, Sk] is required when Sq != Sk")
        seg_k = seg_q if seg_k is None else seg_k
        if tuple(seg_q.shape) != (B, Sq) or tuple(seg_k.shape) != (B, Sk):
            raise ValueError("seg_q must be [B, Sq] and seg_k [B, Sk]")
        seg_q, seg_k = seg_q.to(torch.int32).contiguous(), seg_k.to(torch.int32).contiguous()
        a.seg_q, a.seg_k = seg_q.data_ptr(), seg_k.data_ptr()
        keep += [seg_q, seg_k]
    elif seg_k is not None:
        raise ValueError("seg_k needs seg_q")
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a 1-D tensor of nseq + 1 boundaries")
        cu = cu_seqlens.to(torch.int32).contiguous()
        a.cu_seqlens, a.nseq = cu.data_ptr(), cu.numel() - 1
        keep.append(cu)
    if cu_seqlens_k is not None:
        cuk = cu_seqlens_k.to(torch.int32).contiguous()
        if cu_seqlens is None or cuk.numel() != a.nseq + 1:
            raise ValueError("cu_seqlens_k needs cu_seqlens with the same number of sequences")
        a.cu_seqlens_k = cuk.data_ptr()
        keep.append(cuk)
    a.causal = int(bool(causal))
    a.window = int(window)
    a.softcap = float(softcap)
    if sink is not None:
        if sink.numel() != Hq:
            raise ValueError("sink must hold one logit per query head [Hq]")
        sink = sink.to(torch.float32).contiguous()
        a.sink = sink.data_ptr()
        keep.append(sink)
    a.scale = float(D ** -0.5 if scale is None else scale)
    a.softmax_type = _capi.ATTN_SOFTMAX_OFF_BY_ONE if off_by_one else _capi.ATTN_SOFTMAX_DEFAULT
    a.kv_splits = int(kv_splits)
    if meta is not None:
        if meta.dtype != torch.uint8 or not meta.is_contiguous():
            raise ValueError("meta must be the contiguous uint8 buffer attn_meta returns")
        need = lib().attn_meta_size(ctypes.byref(a))
        if meta.numel() < need:
            raise ValueError(f"meta holds {meta.numel()} bytes; these arguments need {need}")
        a.meta = meta.data_ptr()
        keep.append(meta)
    return a, keep


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _workspace(device, nbytes: int) -> torch.Tensor:
    """Per (device, stream) workspace, zero-filled when (re)allocated."""
    key = (device.index, _stream(device))
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _check(status: int, where: str):
    if status != _capi.ATTN_OK:
        raise AttnError(status, where)


def _fwd_outputs(where, q, keep, out, lse):
    """O [B, Sq, Hq, D] in q's dtype and LSE [B, Hq, Sq] float32: the caller's (checked) or new."""
    B, Sq, Hq, D = q.shape
    _on_device(where, q.device, keep + [out, lse])
    if out is not None:
        _dense(where, "out", out, (B, Sq, Hq, D), q.dtype)
    if lse is not None:
        _dense(where, "lse", lse, (B, Hq, Sq), torch.float32)
    O = torch.empty((B, Sq, Hq, D), dtype=q.dtype, device=q.device) if out is None else out
    LSE = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device) if lse is None else lse
    return O, LSE


def attn_fwd(q, k, v, *, causal=False, window=0, softcap=0.0, sink=None, scale=None,
             bias=None, seg_q=None, seg_k=None, cu_seqlens=None, off_by_one=False, kv_splits=0,
             cu_seqlens_k=None, meta=None, out=None, lse=None):
    """Forward: returns (O [B,Sq,Hq,D] in q's dtype, LSE [B,Hq,Sq] float32)."""
    a, keep = build_args(q, k, v, causal=causal, window=window, softcap=softcap, sink=sink,
                         scale=scale, bias=bias, seg_q=seg_q, seg_k=seg_k, cu_seqlens=cu_seqlens,
                         off_by_one=off_by_one, kv_splits=kv_splits, cu_seqlens_k=cu_seqlens_k,
                         meta=meta)
    O, LSE = _fwd_outputs("attn_fwd", q, keep, out, lse)
    L = lib()
    need = L.attn_fwd_workspace_size(ctypes.byref(a))
    if need == 0:
        _check(_capi.ATTN_ERR_INVALID, "attn_fwd")
    ws = _workspace(q.device, need)
    _check(L.attn_fwd(ctypes.byref(a), O.data_ptr(), LSE.data_ptr(), ws.data_ptr(), ws.numel(),
                      _stream(q.device)), "attn_fwd")
    del keep
    return O, LSE


def attn_fwd_noalloc(q, k, v, *, causal=False, window=0, softcap=0.0, sink=None, scale=None,
                     bias=None, seg_q=None, seg_k=None, cu_seqlens=None, off_by_one=False, kv_splits=0,
                     cu_seqlens_k=None, out=None, lse=None):
    """attn_fwd with the library's built-in scratch instead of a workspace (for callers that
    cannot allocate device memory; see include/attn_gb300.h).  Returns (O, LSE)."""
    a, keep = build_args(q, k, v, causal=causal, window=window, softcap=softcap, sink=sink,
                         scale=scale, bias=bias, seg_q=seg_q, seg_k=seg_k, cu_seqlens=cu_seqlens,
                         off_by_one=off_by_one, kv_splits=kv_splits, cu_seqlens_k=cu_seqlens_k)
    O, LSE = _fwd_outputs("attn_fwd_noalloc", q, keep, out, lse)
    _check(lib().attn_fwd_noalloc(ctypes.byref(a), O.data_ptr(), LSE.data_ptr(), _stream(q.device)),
           "attn_fwd_noalloc")
    del keep
    return O, LSE


def attn_bwd(q, k, v, O, LSE, dO, *, causal=False, window=0, softcap=0.0, sink=None, scale=None,
             bias=None, seg_q=None, seg_k=None, cu_seqlens=None, off_by_one=False, kv_splits=0,
             cu_seqlens_k=None, meta=None):
    """Backward: returns (dQ, dK, dV, dbias or None, dsink or None).  (kv_splits, a forward
    setting, is accepted and ignored so that one set of keyword arguments serves both.)"""
    a, keep = build_args(q, k, v, causal=causal, window=window, softcap=softcap, sink=sink,
                         scale=scale, bias=bias, seg_q=seg_q, seg_k=seg_k, cu_seqlens=cu_seqlens,
                         off_by_one=off_by_one, kv_splits=kv_splits, cu_seqlens_k=cu_seqlens_k,
                         meta=meta)
    _on_device("attn_bwd", q.device, keep + [O, LSE, dO])
    B, Sq, Hq, D = q.shape
    _dense("attn_bwd", "O", O, (B, Sq, Hq, D), q.dtype)
    _dense("attn_bwd", "dO", dO, (B, Sq, Hq, D), q.dtype)
    _dense("attn_bwd", "LSE", LSE, (B, Hq, Sq), torch.float32)
    L = lib()
    need = L.attn_bwd_workspace_size(ctypes.byref(a))
    if need == 0:
        _check(_capi.ATTN_ERR_INVALID, "attn_bwd")
    dQ = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    dK = torch.empty(k.shape, dtype=q.dtype, device=q.device)
    dV = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    dbias = None
    if bias is not None:
        dbias = torch.empty((bias.shape[0], bias.shape[1], q.shape[1], k.shape[1]),
                            dtype=q.dtype, device=q.device)
    dsink = torch.empty((q.shape[2],), dtype=torch.float32, device=q.device) if sink is not None else None
    ws = _workspace(q.device, need)
    _check(L.attn_bwd(ctypes.byref(a), O.data_ptr(), LSE.data_ptr(), dO.data_ptr(), dQ.data_ptr(),
                      dK.data_ptr(), dV.data_ptr(), _ptr(dbias), _ptr(dsink), ws.data_ptr(),
                      ws.numel(), _stream(q.device)), "attn_bwd")
    del keep
    return dQ, dK, dV, dbias, dsink


def attn_meta(q, k, v, *, out=None, **kw) -> Optional[torch.Tensor]:
    """Mask metadata for these arguments (segments / cu_seqlens), built once on the current
    stream to be passed as ``meta=`` to attn_fwd and attn_bwd with the same arguments; None
    when the arguments need none.  ``out``: a uint8 buffer to rebuild it into (reused when it
    is large enough)."""
    kw.pop("meta", None)
    kw.pop("kv_splits", None)
    a, keep = build_args(q, k, v, **kw)
    _on_device("attn_meta", q.device, keep + [out])
    if out is not None and (out.dtype != torch.uint8 or not out.is_contiguous()):
        raise ValueError("attn_meta: out must be a contiguous uint8 buffer")
    L = lib()
    need = L.attn_meta_size(ctypes.byref(a))
    if need == 0:
        return None
    buf = out if out is not None and out.numel() >= need else torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(L.attn_meta_build(ctypes.byref(a), buf.data_ptr(), buf.numel(), _stream(q.device)), "attn_meta_build")
    del keep
    return buf


def attn_check_device_status(device=None) -> int:
    """Synchronise and read/clear the device status word of this stream's workspace."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws = _ws_cache.get((device.index, _stream(device)))
    if ws is None:
        return _capi.ATTN_OK
    return lib().attn_check_device_status(ws.data_ptr(), _stream(device))


def attn_path_name(q, k, v, **kw) -> str:
    a, keep = build_args(q, k, v, **kw)
    return lib().attn_path_name(ctypes.byref(a)).decode()


def attn_launch_counter() -> int:
    return int(lib().attn_launch_counter())


def attn_profile_next_main_kernel(ev_start: "torch.cuda.Event", ev_end: "torch.cuda.Event"):
    """Have the next attn_fwd / attn_bwd of this thread record the two events around its
    main kernel, on the call's stream."""
    lib().attn_profile_next_main_kernel(ctypes.c_void_p(ev_start.cuda_event),
                                        ctypes.c_void_p(ev_end.cuda_event))


def attn_profile_next_aux_kernels(pre_start, pre_end, post_start, post_end):
    """Have the next attn_bwd of this thread record the four events around its preprocess and
    postprocess kernels, on the call's stream."""
    lib().attn_profile_next_aux_kernels(*(ctypes.c_void_p(e.cuda_event) for e in (pre_start, pre_end, post_start,
                                                                                    post_end)))
