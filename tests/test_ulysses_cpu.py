"""Ulysses sequence parallelism (attention_sink_softmax_gb300.ulysses) on two
gloo ranks on the CPU: the sequence is split over the ranks, the wrapper's
all-to-alls move it to head shards and back, and the local attention is the
fp64 oracle (passed in by this test; the product code never imports it). The
sharded forward and backward must equal the oracle on the unsharded problem:
each rank's output and input gradients are its token shard of the full
result, and the sink gradients summed over the ranks are the full dS_h."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from attention_sink_softmax_gb300 import inputs
from attention_sink_softmax_gb300.ulysses import (LocalAttention, heads_to_seq, seq_to_heads,
                                                  ulysses_sink_attention)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_local():
    """The oracle as the local attention: fp64 on CPU tensors."""
    def fwd(q, k, v, sinks, cu, max_seqlen, causal, window, scale):
        kw = dict(scale=scale, causal=causal, window=window,
                  cu_seqlens=cu.numpy() if cu is not None else None)
        o, _ = oracle.forward(q, k, v, sinks, **kw)
        return torch.from_numpy(o), (q, k, v, sinks, kw)

    def bwd(saved, do):
        q, k, v, sinks, kw = saved
        dq, dk, dv, ds = oracle.backward(q, k, v, sinks, do, **kw)
        return tuple(torch.from_numpy(np.asarray(x)) for x in (dq, dk, dv, ds))
    return LocalAttention(fwd, bwd)


CASES = {
    # packed: two sequences over 512 tokens, causal and window 64
    "packed_causal": dict(lengths=[300, 212], packed=True, window=0),
    "packed_window": dict(lengths=[300, 212], packed=True, window=64),
    # padded [B, N, H, d], the sequence dimension split
    "padded_causal": dict(lengths=[256, 256], packed=False, window=0),
}


def _rank(rank, ws, port, case, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    c = CASES[case]
    prob = inputs.random_problem(41, c["lengths"], 8, 2, 64, dtype=torch.float64,
                                 packed=c["packed"], sink_scale=2.0)
    scale = 1 / math.sqrt(64)
    cu = prob["cu_seqlens"]
    sd = 0 if c["packed"] else 1  # token dimension
    N = prob["q"].shape[sd]
    n = N // ws
    shard = lambda t: t.narrow(sd, rank * n, n).contiguous()
    # the all-to-all pair is an exact permutation of the data
    x = shard(prob["q"])
    assert torch.equal(heads_to_seq(seq_to_heads(x)), x)
    q, k, v = (shard(prob[n_]).requires_grad_() for n_ in ("q", "k", "v"))
    sinks = prob["sinks"].double().requires_grad_()
    o = ulysses_sink_attention(q, k, v, sinks, cu, max_seqlen=max(c["lengths"]), causal=True,
                               window=c["window"], softmax_scale=scale, local=_oracle_local())
    o.backward(shard(prob["dout"]))
    torch.save({"o": o.detach(), "dq": q.grad, "dk": k.grad, "dv": v.grad, "ds": sinks.grad},
               os.path.join(outdir, f"{case}_r{rank}.pt"))
    dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
def test_ulysses_two_ranks_equals_unsharded_oracle(case, tmp_path):
    ws = 2
    mp.spawn(_rank, args=(ws, _free_port(), case, str(tmp_path)), nprocs=ws, join=True)
    got = [torch.load(os.path.join(tmp_path, f"{case}_r{r}.pt")) for r in range(ws)]
    c = CASES[case]
    prob = inputs.random_problem(41, c["lengths"], 8, 2, 64, dtype=torch.float64,
                                 packed=c["packed"], sink_scale=2.0)
    kw = dict(scale=1 / 8, causal=True, window=c["window"],
              cu_seqlens=prob["cu_seqlens"].numpy() if prob["cu_seqlens"] is not None else None)
    o, _ = oracle.forward(prob["q"], prob["k"], prob["v"], prob["sinks"], **kw)
    dq, dk, dv, ds = oracle.backward(prob["q"], prob["k"], prob["v"], prob["sinks"],
                                     prob["dout"], **kw)
    sd = 0 if c["packed"] else 1
    for name, full in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        cat = torch.cat([g[name] for g in got], dim=sd).numpy()
        np.testing.assert_allclose(cat, full, rtol=0, atol=1e-12, err_msg=name)
    # each rank's sink gradient covers its own heads; their sum is dS_h
    total = sum(g["ds"] for g in got).numpy()
    np.testing.assert_allclose(total, ds, rtol=0, atol=1e-12)
    assert torch.all(got[0]["ds"][4:] == 0) and torch.all(got[1]["ds"][:4] == 0)


def test_ulysses_rejects_heads_that_do_not_split(tmp_path):
    ws = 2
    mp.spawn(_reject_rank, args=(ws, _free_port()), nprocs=ws, join=True)


def _reject_rank(rank, ws, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    q = torch.zeros(16, 6, 64, dtype=torch.float64)
    k = torch.zeros(16, 3, 64, dtype=torch.float64)  # 3 key/value heads over 2 ranks
    with pytest.raises(ValueError):
        ulysses_sink_attention(q, k, k, torch.zeros(6), local=_oracle_local())
    dist.destroy_process_group()
