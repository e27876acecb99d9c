"""Seeded synthetic inputs for sink attention (no attention arithmetic here).

This module only draws random tensors with the shapes, dtypes and value
distributions of the workloads below; it is shared by the CUDA library's tests
and benchmark and by the oracle's tests, and imports neither.

The workloads stand in for the attention layers of the GPT-OSS-20B model that
the page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！" (nmedialink.com)
trains: sinks that stabilise sliding-window training (section "FlashAttentionV3
对注意力槽的支持"), responses up to 16k and prompts up to 8k tokens (section
"内存高效训练：大模型时代的基石"), padding removed and sequences packed (section
"结合Flash Attention V3的序列并行技术"). The head layout (64 query heads, 8
key/value heads, head size 64, window 128) is GPT-OSS-20B's; the page does not
print it. The RL tasks' data (GSM8K, ReTool, VerifyIf) is not used: these
seeded normal draws stand in for it.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Workload:
    name: str
    batch: int            # number of sequences
    seqlen: int           # N for the padded layout, longest sequence when packed
    h_q: int
    h_kv: int
    head_dim: int
    dtype: torch.dtype    # dtype of q, k, v, o, dout, dq, dk, dv
    causal: bool
    window: int           # 0 = no window; W > 0 = keys i-W+1 .. i
    seed: int
    scale: Optional[float] = None        # None = 1/sqrt(head_dim)
    qk_gain: float = 1.0                 # Q and K are drawn N(0,1) times this
    sink_dist: str = "normal"            # "normal" = N(0,1); "uniform10" = U[-10, 10]
    lengths: Optional[list] = None       # packed layout when set
    windows: list = field(default_factory=list)  # extra layer calls on the same batch (packed case)

    @property
    def packed(self) -> bool:
        return self.lengths is not None

    @property
    def total_tokens(self) -> int:
        return sum(self.lengths) if self.packed else self.batch * self.seqlen


def _packed_lengths(seed: int, nseq: int, lo: int, hi: int) -> list:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (nseq,), generator=g)]


def workload(index: int) -> Workload:
    """The workloads: 0 tiny fp32 check; 1 full-causal GPT-OSS-20B layer;
    2 sliding-window layer; 3 packed variable-length rollouts; 4 long context;
    5 the same layer with 128-wide heads (half as many)."""
    if index == 0:
        return Workload("tiny_fp32_causal_B1_N128_Hq4_Hkv1_d64", 1, 128, 4, 1, 64, torch.float32,
                        True, 0, seed=0)
    if index == 1:
        return Workload("causal_B2_N8192_Hq64_Hkv8_d64_bf16", 2, 8192, 64, 8, 64, torch.bfloat16,
                        True, 0, seed=1, scale=0.125)
    if index == 2:
        return Workload("window128_B4_N8192_Hq64_Hkv8_d64_bf16", 4, 8192, 64, 8, 64, torch.bfloat16,
                        True, 128, seed=2, scale=0.125)
    if index == 3:
        lengths = _packed_lengths(3, 48, 256, 8192)
        return Workload("packed48_U256-8192_Hq64_Hkv8_d64_bf16_causal+window128", len(lengths),
                        max(lengths), 64, 8, 64, torch.bfloat16, True, 0, seed=3, scale=0.125,
                        lengths=lengths, windows=[0, 128])
    if index == 4:
        return Workload("causal_B1_N32768_Hq64_Hkv8_d64_bf16_qk4_sinkU10", 1, 32768, 64, 8, 64,
                        torch.bfloat16, True, 0, seed=4, scale=0.125, qk_gain=4.0,
                        sink_dist="uniform10")
    if index == 5:
        # the 128-wide head variant at the same FLOP count as workload 1
        return Workload("causal_B2_N8192_Hq32_Hkv4_d128_bf16", 2, 8192, 32, 4, 128, torch.bfloat16,
                        True, 0, seed=5, scale=1.0 / 128 ** 0.5)
    raise ValueError(f"no workload {index}")


def make_inputs(w: Workload, *, device: str = "cpu", seed: Optional[int] = None) -> dict:
    """q, k, v, dout (w.dtype), sinks (fp32) and cu_seqlens (int32 or None).

    Values are drawn in fp32 from a CPU torch.Generator seeded with w.seed (or
    ``seed``) in the order q, k, v, sinks, dout, then cast to w.dtype, so the
    same seed gives the same tensors on every machine. Padded layout: q
    [B, N, H_q, d], k/v [B, N, H_kv, d]; packed layout: [T, H, d].
    """
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    if w.packed:
        T = w.total_tokens
        qshape, kshape = (T, w.h_q, w.head_dim), (T, w.h_kv, w.head_dim)
    else:
        qshape = (w.batch, w.seqlen, w.h_q, w.head_dim)
        kshape = (w.batch, w.seqlen, w.h_kv, w.head_dim)

    def normal(shape, gain=1.0):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if gain != 1.0:
            t.mul_(gain)
        return t.to(w.dtype)

    q = normal(qshape, w.qk_gain)
    k = normal(kshape, w.qk_gain)
    v = normal(kshape)
    if w.sink_dist == "normal":
        sinks = torch.randn(w.h_q, generator=g, dtype=torch.float32)
    elif w.sink_dist == "uniform10":
        sinks = torch.rand(w.h_q, generator=g, dtype=torch.float32) * 20.0 - 10.0
    else:
        raise ValueError(w.sink_dist)
    dout = normal(qshape)
    cu = None
    if w.packed:
        cu = torch.zeros(len(w.lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(w.lengths, dtype=torch.int64), 0).to(torch.int32)
    out = dict(q=q, k=k, v=v, sinks=sinks, dout=dout, cu_seqlens=cu)
    if device != "cpu":
        out = {key: (t.to(device) if t is not None else None) for key, t in out.items()}
    return out


def random_problem(seed: int, lengths, h_q: int, h_kv: int, head_dim: int,
                   dtype=torch.bfloat16, packed: bool = True, sink_scale: float = 1.0,
                   qk_gain: float = 1.0) -> dict:
    """Small seeded problem for parity tests: q, k, v, dout, sinks, cu_seqlens.

    ``lengths`` lists the sequence lengths; with ``packed`` False they must be
    equal and the padded [B, N, H, d] layout is returned (cu_seqlens None).
    """
    g = torch.Generator().manual_seed(seed)
    T = int(sum(lengths))
    if packed:
        qshape, kshape = (T, h_q, head_dim), (T, h_kv, head_dim)
    else:
        assert len(set(lengths)) == 1
        qshape = (len(lengths), lengths[0], h_q, head_dim)
        kshape = (len(lengths), lengths[0], h_kv, head_dim)
    q = (torch.randn(qshape, generator=g) * qk_gain).to(dtype)
    k = (torch.randn(kshape, generator=g) * qk_gain).to(dtype)
    v = torch.randn(kshape, generator=g).to(dtype)
    sinks = torch.randn(h_q, generator=g) * sink_scale
    dout = torch.randn(qshape, generator=g).to(dtype)
    cu = None
    if packed:
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, sinks=sinks, dout=dout, cu_seqlens=cu)


@dataclass
class DecodeWorkload:
    """Decode: `batch` newest tokens, each against its own `ctx`-token context in
    a shared key/value cache (contexts back to back)."""
    name: str
    batch: int
    ctx: int
    h_q: int
    h_kv: int
    head_dim: int
    dtype: torch.dtype
    window: int
    seed: int
    scale: float = 0.125

    @property
    def cache_tokens(self) -> int:
        return self.batch * self.ctx


def decode_workload() -> DecodeWorkload:
    """Streaming inference on the GPT-OSS-20B layer shape: 8 sequences whose
    contexts are 32768 tokens (the long-context workload's length)."""
    return DecodeWorkload("decode_B8_ctx32768_Hq64_Hkv8_d64_bf16", 8, 32768, 64, 8, 64,
                          torch.bfloat16, 0, 7)


def make_decode_inputs(w: DecodeWorkload, *, device: str = "cpu") -> dict:
    """q [batch, h_q, d], k/v cache [batch * ctx, h_kv, d] ~ N(0,1) in w.dtype,
    sinks [h_q] ~ N(0,1) fp32, kv_start / kv_len int32 [batch]."""
    g = torch.Generator().manual_seed(w.seed)
    T = w.cache_tokens
    q = torch.randn(w.batch, w.h_q, w.head_dim, generator=g).to(w.dtype)
    k = torch.randn(T, w.h_kv, w.head_dim, generator=g).to(w.dtype)
    v = torch.randn(T, w.h_kv, w.head_dim, generator=g).to(w.dtype)
    sinks = torch.randn(w.h_q, generator=g).float()
    kv_start = torch.arange(w.batch, dtype=torch.int32) * w.ctx
    kv_len = torch.full((w.batch,), w.ctx, dtype=torch.int32)
    out = dict(q=q, k=k, v=v, sinks=sinks, kv_start=kv_start, kv_len=kv_len)
    return {n: t.to(device) for n, t in out.items()}
