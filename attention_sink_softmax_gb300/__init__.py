"""GB300 (sm_103a) sink attention: causal / sliding-window GQA attention with
one learnable sink logit per query head, forward and full backward.

The computation is the one on the page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、
超稳定！" (nmedialink.com): sections "GPT-OSS中的带注意力槽的注意力机制" and
"数学公式深入解读" (the sink joins the softmax denominator and adds no value
row) and "反向传播的实现" (the sink gradient). All of it runs in libsinkattn,
a C-ABI CUDA library (include/sink_attn.h); the functions below, named like
the C entry points, only marshal torch tensors into pointers and sizes. Torch
provides device memory and streams.

Tensors: padded q/o/dout [B, N, H_q, d] and k/v [B, N, H_kv, d], or packed
[T, H, d] with int32 ``cu_seqlens`` [num_seqs + 1] on the device; sinks [H_q]
fp32; lse [H_q, T] fp32. dtype bf16 or fp32, d = 64 or 128 (decode: 64).

The ``_ex`` forms carry ``o_lo`` (bf16 only): the part of O that its rounding
to bf16 dropped, written by the forward and used by the backward to form
D = dO . O from about 16 bits of O instead of the stored 8 (see "Precision of
D" in include/sink_attn.h). ``sink_attention`` uses them for bf16.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _abi
from ._abi import SinkAttnError, SinkAttnParams, lib, status_str  # noqa: F401

__all__ = [
    "SinkAttnParams", "SinkAttnError", "make_params", "sink_attn_workspace_bytes",
    "sink_attn_fwd", "sink_attn_bwd", "sink_attn_bwd_preprocess", "sink_attn_bwd_main",
    "sink_attn_bwd_prepare",
    "sink_attn_fwd_ex", "sink_attn_bwd_ex", "sink_attn_bwd_preprocess_ex",
    "sink_attn_set_wait_limit_ns", "sink_attn_set_deterministic",
    "sink_attn_testing_withhold_load",
    "sink_attn_fetch_device_error", "sink_attn_bwd_preprocess_noalloc",
    "sink_attn_noalloc_scratch_bytes", "sink_attn_status_str", "sink_attn_kernel_launches",
    "sink_attn_version", "make_decode_params", "sink_attn_decode_workspace_bytes",
    "sink_attn_decode",
    "sink_attention", "SinkAttentionFunction",
]

_DTYPES = {torch.bfloat16: _abi.SINK_BF16, torch.float32: _abi.SINK_FP32}


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _need_cuda(name: str, t: Optional[torch.Tensor], dtype=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")


def make_params(q: torch.Tensor, k: torch.Tensor, cu_seqlens: Optional[torch.Tensor] = None,
                max_seqlen: Optional[int] = None, causal: bool = True, window: int = 0,
                softmax_scale: Optional[float] = None) -> SinkAttnParams:
    """sink_attn_params_t from tensor shapes.

    Packed input needs ``max_seqlen`` (an upper bound on every sequence's
    length); if it is None it is read from ``cu_seqlens``, which synchronises.
    """
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    p = SinkAttnParams()
    if q.dim() == 4:
        if cu_seqlens is not None:
            raise ValueError("cu_seqlens is for the packed [T, H, d] layout")
        B, N, h_q, d = q.shape
        p.batch, p.max_seqlen, p.total_tokens = B, N, B * N
        h_kv = k.shape[2]
    elif q.dim() == 3:
        T, h_q, d = q.shape
        h_kv = k.shape[1]
        if cu_seqlens is None:
            p.batch, p.max_seqlen, p.total_tokens = (1 if T > 0 else 0), T, T
        else:
            nseq = cu_seqlens.numel() - 1
            if max_seqlen is None:
                c = cu_seqlens.to("cpu", torch.int64)
                max_seqlen = int((c[1:] - c[:-1]).max()) if nseq > 0 else 0
            p.batch, p.max_seqlen, p.total_tokens = nseq, int(max_seqlen), T
    else:
        raise ValueError("q must be [B, N, H, d] or [T, H, d]")
    p.h_q, p.h_kv, p.head_dim = h_q, h_kv, d
    p.dtype = _DTYPES[q.dtype]
    p.softmax_scale = float(softmax_scale) if softmax_scale is not None else 0.0
    p.causal = 1 if causal else 0
    p.window = int(window) if window else 0
    return p


def _check_qkv(q, k, v):
    _need_cuda("q", q)
    _need_cuda("k", k, q.dtype)
    _need_cuda("v", v, q.dtype)
    if k.shape != v.shape or k.dim() != q.dim() or k.shape[:-2] != q.shape[:-2]:
        raise ValueError("k and v must match q's layout with H_kv heads")


def sink_attn_workspace_bytes(params: SinkAttnParams, is_bwd: bool) -> int:
    return int(lib().sink_attn_workspace_bytes(ctypes.byref(params), 1 if is_bwd else 0))


def _workspace(params, is_bwd, device, workspace):
    need = sink_attn_workspace_bytes(params, is_bwd)
    if need == 0:
        raise SinkAttnError(_abi.SINK_ERR_INVALID_ARG, "sink_attn_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    return workspace


def sink_attn_fwd(q, k, v, sinks, cu_seqlens=None, *, max_seqlen=None, causal=True, window=0,
                  softmax_scale=None, out=None, lse=None, workspace=None, stream=None,
                  params=None):
    """Forward: returns (o, lse). See sink_attn_fwd in include/sink_attn.h."""
    _check_qkv(q, k, v)
    _need_cuda("sinks", sinks, torch.float32)
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    p = params or make_params(q, k, cu_seqlens, max_seqlen, causal, window, softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((p.h_q, p.total_tokens), dtype=torch.float32, device=q.device)
    workspace = _workspace(p, False, q.device, workspace)
    st = lib().sink_attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(sinks),
                             _ptr(cu_seqlens), _ptr(out), _ptr(lse), _ptr(workspace),
                             workspace.numel(), _stream(stream, q.device))
    _abi.check(st, "sink_attn_fwd")
    return out, lse


def _check_o_lo(o_lo, o):
    _need_cuda("o_lo", o_lo, o.dtype)
    if o.dtype != torch.bfloat16:
        raise ValueError("o_lo is for bf16 outputs only")
    if o_lo.shape != o.shape or o_lo.device != o.device:
        raise ValueError("o_lo must have o's shape and device")


def sink_attn_fwd_ex(q, k, v, sinks, cu_seqlens=None, *, max_seqlen=None, causal=True, window=0,
                     softmax_scale=None, out=None, o_lo=None, lse=None, workspace=None,
                     stream=None, params=None):
    """Forward that also writes o_lo = bf16(O - bf16(O)) (bf16 only): returns
    (o, o_lo, lse). See sink_attn_fwd_ex in include/sink_attn.h."""
    _check_qkv(q, k, v)
    _need_cuda("sinks", sinks, torch.float32)
    if q.dtype != torch.bfloat16:
        raise ValueError("sink_attn_fwd_ex writes o_lo for bf16 inputs only")
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    p = params or make_params(q, k, cu_seqlens, max_seqlen, causal, window, softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if o_lo is None:
        o_lo = torch.empty_like(q)
    _check_o_lo(o_lo, out)
    if lse is None:
        lse = torch.empty((p.h_q, p.total_tokens), dtype=torch.float32, device=q.device)
    workspace = _workspace(p, False, q.device, workspace)
    st = lib().sink_attn_fwd_ex(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(sinks),
                                _ptr(cu_seqlens), _ptr(out), _ptr(o_lo), _ptr(lse), _ptr(workspace),
                                workspace.numel(), _stream(stream, q.device))
    _abi.check(st, "sink_attn_fwd_ex")
    return out, o_lo, lse


def sink_attn_bwd_ex(q, k, v, sinks, o, o_lo, lse, dout, cu_seqlens=None, *, max_seqlen=None,
                     causal=True, window=0, softmax_scale=None, dq=None, dk=None, dv=None,
                     dsinks=None, workspace=None, stream=None, params=None):
    """Full backward with D formed from o + o_lo: returns (dq, dk, dv, dsinks).
    See sink_attn_bwd_ex in include/sink_attn.h."""
    _check_qkv(q, k, v)
    _need_cuda("o", o, q.dtype)
    _check_o_lo(o_lo, o)
    _need_cuda("dout", dout, q.dtype)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("sinks", sinks, torch.float32)
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    p = params or make_params(q, k, cu_seqlens, max_seqlen, causal, window, softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dsinks = torch.empty_like(sinks) if dsinks is None else dsinks
    workspace = _workspace(p, True, q.device, workspace)
    st = lib().sink_attn_bwd_ex(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(sinks),
                                _ptr(cu_seqlens), _ptr(o), _ptr(o_lo), _ptr(lse), _ptr(dout),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dsinks), _ptr(workspace),
                                workspace.numel(), _stream(stream, q.device))
    _abi.check(st, "sink_attn_bwd_ex")
    return dq, dk, dv, dsinks


def sink_attn_bwd(q, k, v, sinks, o, lse, dout, cu_seqlens=None, *, max_seqlen=None,
                  causal=True, window=0, softmax_scale=None, dq=None, dk=None, dv=None,
                  dsinks=None, workspace=None, stream=None, params=None):
    """Full backward: returns (dq, dk, dv, dsinks). See sink_attn_bwd in include/sink_attn.h."""
    _check_qkv(q, k, v)
    _need_cuda("o", o, q.dtype)
    _need_cuda("dout", dout, q.dtype)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("sinks", sinks, torch.float32)
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    p = params or make_params(q, k, cu_seqlens, max_seqlen, causal, window, softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dsinks = torch.empty_like(sinks) if dsinks is None else dsinks
    workspace = _workspace(p, True, q.device, workspace)
    st = lib().sink_attn_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(sinks),
                             _ptr(cu_seqlens), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(dsinks), _ptr(workspace), workspace.numel(),
                             _stream(stream, q.device))
    _abi.check(st, "sink_attn_bwd")
    return dq, dk, dv, dsinks


def sink_attn_bwd_preprocess(params, sinks, o, lse, dout, *, delta=None, dsinks=None,
                             workspace=None, stream=None):
    """Backward step 1: returns (delta [H_q, T] fp32, dsinks [H_q] fp32)."""
    _need_cuda("o", o)
    _need_cuda("dout", dout, o.dtype)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("sinks", sinks, torch.float32)
    if delta is None:
        delta = torch.empty((params.h_q, params.total_tokens), dtype=torch.float32, device=o.device)
    dsinks = torch.empty_like(sinks) if dsinks is None else dsinks
    workspace = _workspace(params, True, o.device, workspace)
    st = lib().sink_attn_bwd_preprocess(ctypes.byref(params), _ptr(sinks), _ptr(o), _ptr(lse),
                                        _ptr(dout), _ptr(delta), _ptr(dsinks), _ptr(workspace),
                                        workspace.numel(), _stream(stream, o.device))
    _abi.check(st, "sink_attn_bwd_preprocess")
    return delta, dsinks


def sink_attn_bwd_preprocess_ex(params, sinks, o, o_lo, lse, dout, *, delta=None, dsinks=None,
                                workspace=None, stream=None):
    """Backward step 1 with delta = dout . (o + o_lo): returns (delta, dsinks)."""
    _need_cuda("o", o)
    _check_o_lo(o_lo, o)
    _need_cuda("dout", dout, o.dtype)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("sinks", sinks, torch.float32)
    if delta is None:
        delta = torch.empty((params.h_q, params.total_tokens), dtype=torch.float32, device=o.device)
    dsinks = torch.empty_like(sinks) if dsinks is None else dsinks
    workspace = _workspace(params, True, o.device, workspace)
    st = lib().sink_attn_bwd_preprocess_ex(ctypes.byref(params), _ptr(sinks), _ptr(o), _ptr(o_lo),
                                           _ptr(lse), _ptr(dout), _ptr(delta), _ptr(dsinks),
                                           _ptr(workspace), workspace.numel(),
                                           _stream(stream, o.device))
    _abi.check(st, "sink_attn_bwd_preprocess_ex")
    return delta, dsinks


def sink_attn_bwd_main(params, q, k, v, lse, delta, dout, cu_seqlens=None, *, dq=None, dk=None,
                       dv=None, workspace=None, stream=None, prepared=False):
    """Backward step 2: returns (dq, dk, dv). prepared=True (sink_attn_bwd_main_ex
    with SINK_BWD_PREPARED) skips the preparation pass, which
    sink_attn_bwd_prepare must already have run on the same workspace."""
    _check_qkv(q, k, v)
    _need_cuda("dout", dout, q.dtype)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("delta", delta, torch.float32)
    if prepared and workspace is None:
        raise ValueError("prepared=True needs the workspace sink_attn_bwd_prepare filled")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    workspace = _workspace(params, True, q.device, workspace)
    st = lib().sink_attn_bwd_main_ex(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(cu_seqlens), _ptr(lse), _ptr(delta), _ptr(dout),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                     workspace.numel(),
                                     _abi.SINK_BWD_PREPARED if prepared else 0,
                                     _stream(stream, q.device))
    _abi.check(st, "sink_attn_bwd_main_ex")
    return dq, dk, dv


def sink_attn_bwd_prepare(params, q, k, *, workspace, stream=None):
    """The backward's preparation pass on its own (f16 copies of q and k, the
    zeroed dQ accumulator, into `workspace`); it depends on q and k alone, so
    it can run on a second stream while the forward runs. Follow it with
    sink_attn_bwd_main(..., workspace=workspace, prepared=True), ordered after
    it (an event). Returns the workspace."""
    _check_qkv(q, k, k)
    workspace = _workspace(params, True, q.device, workspace)
    st = lib().sink_attn_bwd_prepare(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(workspace),
                                     workspace.numel(), _stream(stream, q.device))
    _abi.check(st, "sink_attn_bwd_prepare")
    return workspace


def sink_attn_bwd_preprocess_noalloc(params, sinks, o, lse, dout, *, delta=None, dsinks=None,
                                     stream=None):
    """Backward step 1 with the library's fixed scratch instead of a workspace.

    For callers that cannot obtain scratch device memory; see
    sink_attn_bwd_preprocess_noalloc in include/sink_attn.h for the size limit
    and the rule that overlapping calls race. Returns (delta, dsinks); pass
    preallocated ``delta``/``dsinks`` to allocate nothing here either.
    """
    _need_cuda("o", o)
    _need_cuda("dout", dout, o.dtype)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("sinks", sinks, torch.float32)
    if delta is None:
        delta = torch.empty((params.h_q, params.total_tokens), dtype=torch.float32, device=o.device)
    dsinks = torch.empty_like(sinks) if dsinks is None else dsinks
    # the kernels write delta [h_q, T] and dsinks [h_q]: a smaller buffer would be overrun
    _need_cuda("delta", delta, torch.float32)
    _need_cuda("dsinks", dsinks, torch.float32)
    if tuple(delta.shape) != (params.h_q, params.total_tokens) or dsinks.numel() != params.h_q:
        raise ValueError(f"delta must be [{params.h_q}, {params.total_tokens}] and dsinks "
                         f"[{params.h_q}]")
    for name, t in (("dout", dout), ("lse", lse), ("sinks", sinks), ("delta", delta),
                    ("dsinks", dsinks)):
        if t.device != o.device:
            raise ValueError(f"{name} is on {t.device}, o on {o.device}")
    # the library looks up its scratch array on the current device: make it o's
    with torch.cuda.device(o.device):
        st = lib().sink_attn_bwd_preprocess_noalloc(ctypes.byref(params), _ptr(sinks), _ptr(o),
                                                    _ptr(lse), _ptr(dout), _ptr(delta),
                                                    _ptr(dsinks), _stream(stream, o.device))
    _abi.check(st, "sink_attn_bwd_preprocess_noalloc")
    return delta, dsinks


def sink_attn_noalloc_scratch_bytes() -> int:
    return int(lib().sink_attn_noalloc_scratch_bytes())


def make_decode_params(q: torch.Tensor, k_cache: torch.Tensor, max_seqlen: int, window: int = 0,
                       softmax_scale: Optional[float] = None) -> SinkAttnParams:
    """sink_attn_params_t for sink_attn_decode: q [B, H_q, d], k_cache [T, H_kv, d];
    ``max_seqlen`` bounds every context length."""
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if q.dim() != 3 or k_cache.dim() != 3:
        raise ValueError("q must be [B, H_q, d] and the cache [T, H_kv, d]")
    p = SinkAttnParams()
    p.batch, p.h_q, p.head_dim = q.shape
    p.total_tokens, p.h_kv = k_cache.shape[0], k_cache.shape[1]
    p.max_seqlen = int(max_seqlen)
    p.dtype = _DTYPES[q.dtype]
    p.softmax_scale = float(softmax_scale) if softmax_scale is not None else 0.0
    p.causal = 1
    p.window = int(window) if window else 0
    return p


def sink_attn_decode_workspace_bytes(params: SinkAttnParams) -> int:
    return int(lib().sink_attn_decode_workspace_bytes(ctypes.byref(params)))


def sink_attn_decode(q, k_cache, v_cache, sinks, kv_start, kv_len, *, max_seqlen=None, window=0,
                     softmax_scale=None, out=None, lse=None, workspace=None, stream=None,
                     params=None):
    """Decode: one query per entry against a key/value cache; returns (o, lse).
    See sink_attn_decode in include/sink_attn.h. ``max_seqlen`` None reads the
    largest of ``kv_len`` (synchronises)."""
    _need_cuda("q", q)
    _need_cuda("k_cache", k_cache, q.dtype)
    _need_cuda("v_cache", v_cache, q.dtype)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    _need_cuda("sinks", sinks, torch.float32)
    _need_cuda("kv_start", kv_start, torch.int32)
    _need_cuda("kv_len", kv_len, torch.int32)
    if params is None:
        if max_seqlen is None:  # synchronises: pass max_seqlen or params inside a graph capture
            max_seqlen = int(kv_len.max()) if kv_len.numel() else 0
        params = make_decode_params(q, k_cache, max_seqlen, window, softmax_scale)
    p = params
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((p.h_q, p.batch), dtype=torch.float32, device=q.device)
    need = sink_attn_decode_workspace_bytes(p)
    if need == 0:
        raise SinkAttnError(_abi.SINK_ERR_INVALID_ARG, "sink_attn_decode_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    st = lib().sink_attn_decode(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sinks),
                                _ptr(kv_start), _ptr(kv_len), _ptr(out), _ptr(lse), _ptr(workspace),
                                workspace.numel(), _stream(stream, q.device))
    _abi.check(st, "sink_attn_decode")
    return out, lse


def sink_attn_fetch_device_error(workspace: torch.Tensor, stream=None):
    """(status, flags) of the device flag word in ``workspace``; synchronises the stream."""
    flags = ctypes.c_uint32(0)
    st = lib().sink_attn_fetch_device_error(_ptr(workspace), workspace.numel(),
                                            _stream(stream, workspace.device), ctypes.byref(flags))
    return int(st), int(flags.value)


def sink_attn_status_str(status: int) -> str:
    return status_str(status)


def sink_attn_set_wait_limit_ns(limit_ns: int) -> int:
    """Limit of every bounded wait inside the kernels, for calls made after this
    one (process-wide); 0 restores the default of 2 s. Returns the previous limit."""
    return int(lib().sink_attn_set_wait_limit_ns(int(limit_ns)))


def sink_attn_set_deterministic(on: bool) -> bool:
    """Reproducible dq for backward calls made after this one (process-wide):
    the 64-wide bf16 backward then runs as a key-owning dK/dV kernel and a
    query-owning dQ kernel with no reduce-adds. Slower; off by default. The
    workspace size depends on it. Returns the previous setting."""
    return bool(lib().sink_attn_set_deterministic(1 if on else 0))


def sink_attn_testing_withhold_load(on: bool) -> None:
    """Test hook (include/sink_attn_testing.h): when on, the 64-wide tensor-core
    forward and backward stop loading after their first stage, so that their
    bounded waits run out and the call reports SINK_ERR_TIMEOUT. Tests only."""
    lib().sink_attn_testing_withhold_load(1 if on else 0)


def sink_attn_kernel_launches() -> int:
    """Kernels libsinkattn has enqueued in this process so far."""
    return int(lib().sink_attn_kernel_launches())


def sink_attn_version() -> int:
    return int(lib().sink_attn_version())


class SinkAttentionFunction(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run in libsinkattn. With bf16
    inputs the forward also writes o_lo, which the backward uses to form D."""

    @staticmethod
    def forward(ctx, q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, softmax_scale):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        sinks = sinks.contiguous()
        p = make_params(q, k, cu_seqlens, max_seqlen, causal, window, softmax_scale)
        if q.dtype == torch.bfloat16:
            o, o_lo, lse = sink_attn_fwd_ex(q, k, v, sinks, cu_seqlens, params=p)
        else:
            (o, lse), o_lo = sink_attn_fwd(q, k, v, sinks, cu_seqlens, params=p), None
        ctx.save_for_backward(q, k, v, sinks, o, o_lo, lse, cu_seqlens)
        ctx.params = p
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, sinks, o, o_lo, lse, cu = ctx.saved_tensors
        if o_lo is not None:
            dq, dk, dv, ds = sink_attn_bwd_ex(q, k, v, sinks, o, o_lo, lse, do.contiguous(), cu,
                                              params=ctx.params)
        else:
            dq, dk, dv, ds = sink_attn_bwd(q, k, v, sinks, o, lse, do.contiguous(), cu,
                                           params=ctx.params)
        return dq, dk, dv, ds, None, None, None, None, None


def sink_attention(q, k, v, sinks, cu_seqlens=None, max_seqlen=None, causal=True, window=0,
                   softmax_scale=None):
    """Differentiable sink attention (gradients for q, k, v and sinks)."""
    return SinkAttentionFunction.apply(q, k, v, sinks, cu_seqlens, max_seqlen, causal, window,
                                       softmax_scale)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
