"""Ulysses sequence parallelism with the library's kernels as the local
attention: two ranks (fresh processes, gloo for the all-to-alls through host
memory) share the one GPU for their local kernels, which are independent of
each other. The sharded forward and backward are checked element by element
against the fp64 oracle on the unsharded problem, at the bf16 tolerance."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from attention_sink_softmax_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


LENGTHS = [700, 324]  # packed, 1024 tokens split over 2 ranks


def _rank(rank, ws, port, window, outdir):
    from attention_sink_softmax_gb300.ulysses import ulysses_sink_attention
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    torch.cuda.set_device(0)
    prob = inputs.random_problem(51, LENGTHS, 16, 4, 64, dtype=torch.bfloat16, sink_scale=2.0)
    n = sum(LENGTHS) // ws
    d = {k: v.cuda() for k, v in prob.items()}
    shard = lambda t: t[rank * n:(rank + 1) * n].contiguous()
    q, k, v = (shard(d[x]).requires_grad_() for x in ("q", "k", "v"))
    sinks = d["sinks"].clone().requires_grad_()
    o = ulysses_sink_attention(q, k, v, sinks, d["cu_seqlens"], max_seqlen=max(LENGTHS),
                               causal=True, window=window, softmax_scale=0.125)
    o.backward(shard(d["dout"]))
    torch.cuda.synchronize()
    torch.save({n_: t.detach().cpu() for n_, t in (("o", o), ("dq", q.grad), ("dk", k.grad),
                                                    ("dv", v.grad), ("ds", sinks.grad))},
               os.path.join(outdir, f"w{window}_r{rank}.pt"))
    dist.destroy_process_group()


@pytest.mark.parametrize("window", [0, 128])
def test_ulysses_two_ranks_on_the_gpu_match_the_oracle(window, tmp_path):
    ws = 2
    mp.spawn(_rank, args=(ws, _free_port(), window, str(tmp_path)), nprocs=ws, join=True)
    got = [torch.load(os.path.join(tmp_path, f"w{window}_r{r}.pt")) for r in range(ws)]
    prob = inputs.random_problem(51, LENGTHS, 16, 4, 64, dtype=torch.bfloat16, sink_scale=2.0)
    kw = dict(scale=0.125, causal=True, window=window, cu_seqlens=prob["cu_seqlens"].numpy())
    o, _ = oracle.forward(prob["q"], prob["k"], prob["v"], prob["sinks"], **kw)
    dq, dk, dv, ds = oracle.backward(prob["q"], prob["k"], prob["v"], prob["sinks"],
                                     prob["dout"], **kw)
    for name, ref in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        cat = torch.cat([g[name] for g in got], dim=0)
        assert_close(name, cat, ref, torch.bfloat16)
    assert_close("dS_h", sum(g["ds"] for g in got), ds, torch.bfloat16, rounds_output=False)
