"""Ulysses sequence parallelism around sink attention.

Page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！" (nmedialink.com),
section "结合Flash Attention V3的序列并行技术" and Fig. 8: with the sequence
split over P ranks, one all-to-all before attention turns each rank's token
shard of every head into every token of a shard of the heads; attention runs
unchanged on those heads; one all-to-all after it turns the output back into
token shards. Attention itself needs no communication, because heads are
independent, and each head's sink travels with its head.

Layout (per rank r of the process group, P ranks):
  q [..., n, H_q, d], k/v [..., n, H_kv, d]: this rank's n = N / P tokens of
  every head, tokens [r n, (r + 1) n) of the full sequence (packed [n, H, d]
  with ``cu_seqlens`` describing the full N tokens, or padded [B, n, H, d]);
  sinks [H_q]: every head's sink (a replicated parameter).
After the first all-to-all rank r holds all N tokens of query heads
[r H_q / P, (r + 1) H_q / P) and key/value heads [r H_kv / P, (r + 1) H_kv / P):
with contiguous head shards the grouped-query mapping h -> h // (H_q / H_kv)
is the same inside the shard, so the local attention is the ordinary call.
H_q and H_kv must be divisible by P.

The all-to-all is one ``torch.distributed.all_to_all_single`` per tensor (NCCL
between GPUs, gloo in the CPU tests; no multicast). The backward is the same
exchange in reverse around the local backward. The sink gradient of rank r
holds its own heads' entries and zeros elsewhere, so the usual sum of a
replicated parameter's gradient over the group gives the full dS_h.

The local attention is a pair of callables (``local``); the default runs the
library's C ABI (the extended entry points for bf16, which keep o_lo for D).
"""
from __future__ import annotations

from typing import Callable, NamedTuple, Optional

import torch
import torch.distributed as dist


class LocalAttention(NamedTuple):
    """forward(q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale)
    -> (o, saved); backward(saved, do) -> (dq, dk, dv, dsinks). Tensors are one
    rank's full-sequence head shard."""
    forward: Callable
    backward: Callable


def _library_forward(q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale):
    from . import make_params, sink_attn_fwd, sink_attn_fwd_ex
    p = make_params(q, k, cu_seqlens, max_seqlen, causal, window, scale)
    if q.dtype == torch.bfloat16:
        o, o_lo, lse = sink_attn_fwd_ex(q, k, v, sinks, cu_seqlens, params=p)
    else:
        (o, lse), o_lo = sink_attn_fwd(q, k, v, sinks, cu_seqlens, params=p), None
    return o, (q, k, v, sinks, cu_seqlens, o, o_lo, lse, p)


def _library_backward(saved, do):
    from . import sink_attn_bwd, sink_attn_bwd_ex
    q, k, v, sinks, cu, o, o_lo, lse, p = saved
    if o_lo is not None:
        return sink_attn_bwd_ex(q, k, v, sinks, o, o_lo, lse, do, cu, params=p)
    return sink_attn_bwd(q, k, v, sinks, o, lse, do, cu, params=p)


LIBRARY = LocalAttention(_library_forward, _library_backward)


def _exchange(x: torch.Tensor, group) -> torch.Tensor:
    """all_to_all_single along dim 0 (equal splits). gloo takes CPU tensors
    only, so a CUDA tensor on a gloo group goes through host memory."""
    staged = x.is_cuda and dist.get_backend(group) == "gloo"
    src = x.cpu() if staged else x.contiguous()
    out = torch.empty_like(src)
    dist.all_to_all_single(out, src, group=group)
    return out.to(x.device) if staged else out


def seq_to_heads(x: torch.Tensor, group=None) -> torch.Tensor:
    """[..., n, H, d] token shard of every head -> [..., P n, H / P, d], every
    token of this rank's head shard (the all-to-all before attention)."""
    P = dist.get_world_size(group)
    *pre, n, H, d = x.shape
    if H % P:
        raise ValueError(f"{H} heads do not split over {P} ranks")
    y = x.reshape(*pre, n, P, H // P, d)
    y = y.movedim(-3, 0).contiguous()          # [P, ..., n, H/P, d]: chunk s goes to rank s
    y = _exchange(y, group)                    # [P, ..., n, H/P, d]: chunk s came from rank s
    y = y.movedim(0, -4)                       # [..., P, n, H/P, d]
    return y.reshape(*pre, P * n, H // P, d)


def heads_to_seq(y: torch.Tensor, group=None) -> torch.Tensor:
    """Inverse of seq_to_heads: [..., P n, H / P, d] -> [..., n, H, d]."""
    P = dist.get_world_size(group)
    *pre, N, Hl, d = y.shape
    if N % P:
        raise ValueError(f"{N} tokens do not split over {P} ranks")
    n = N // P
    x = y.reshape(*pre, P, n, Hl, d).movedim(-4, 0).contiguous()  # chunk s: rank s's tokens
    x = _exchange(x, group)                                         # chunk s: head shard s
    x = x.movedim(0, -3)                                            # [..., n, P, Hl, d]
    return x.reshape(*pre, n, P * Hl, d)


def _head_slice(H: int, group) -> slice:
    P, r = dist.get_world_size(group), dist.get_rank(group)
    return slice(r * H // P, (r + 1) * H // P)


class _Ulysses(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale, group, local):
        hs = _head_slice(q.shape[-2], group)
        qh, kh, vh = (seq_to_heads(t, group) for t in (q, k, v))
        o, saved = local.forward(qh, kh, vh, sinks[hs].contiguous(), cu_seqlens, max_seqlen,
                                 causal, window, scale)
        ctx.saved = saved
        ctx.local, ctx.group, ctx.hs, ctx.n_sinks = local, group, hs, sinks.shape[0]
        return heads_to_seq(o, group)

    @staticmethod
    def backward(ctx, do):
        doh = seq_to_heads(do.contiguous(), ctx.group)
        dq, dk, dv, ds = ctx.local.backward(ctx.saved, doh)
        ctx.saved = None
        dsinks = torch.zeros(ctx.n_sinks, dtype=ds.dtype, device=ds.device)
        dsinks[ctx.hs] = ds
        return (heads_to_seq(dq, ctx.group), heads_to_seq(dk, ctx.group),
                heads_to_seq(dv, ctx.group), dsinks, None, None, None, None, None, None, None)


def ulysses_sink_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, sinks: torch.Tensor,
                           cu_seqlens: Optional[torch.Tensor] = None,
                           max_seqlen: Optional[int] = None, causal: bool = True, window: int = 0,
                           softmax_scale: Optional[float] = None, group=None,
                           local: LocalAttention = LIBRARY) -> torch.Tensor:
    """Sink attention over a sequence split across the ranks of ``group``
    (see the module docstring for the layout); differentiable in q, k, v and
    sinks. ``cu_seqlens``/``max_seqlen`` describe the full sequence (packed
    layout); pass ``max_seqlen`` to avoid reading ``cu_seqlens`` on the host."""
    P = dist.get_world_size(group)
    if q.shape[-2] % P or k.shape[-2] % P:
        raise ValueError(f"H_q = {q.shape[-2]} and H_kv = {k.shape[-2]} must split over {P} ranks")
    if k.shape != v.shape or k.shape[:-2] != q.shape[:-2]:
        raise ValueError("k and v must match q's token layout")
    return _Ulysses.apply(q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, softmax_scale,
                          group, local)
