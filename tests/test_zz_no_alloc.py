"""sink_attn_bwd_preprocess_noalloc: backward step 1 for callers that cannot
allocate device memory (they are handed inputs and outputs only, e.g. a plugin
inside a framework that owns all device memory). It keeps its scratch in a
fixed array inside the library; these tests check it against the workspace
entry point, sink_attn_bwd_preprocess, through the C ABI, on consecutive calls
that share that array: the same kernels in the same order, so the results are
equal bit for bit. dS_h is also checked against the oracle.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import attention_sink_softmax_gb300 as sa
from attention_sink_softmax_gb300 import _abi, inputs
import math

import oracle
from parity import assert_close


def test_scratch_limit_rejected_before_launch():
    p = _abi.SinkAttnParams()
    p.batch, p.max_seqlen, p.total_tokens = 1, 10_000_000, 10_000_000
    p.h_q, p.h_kv, p.head_dim, p.dtype, p.causal = 64, 8, 64, _abi.SINK_BF16, 1
    nul = ctypes.c_void_p(0)
    st = _abi.lib().sink_attn_bwd_preprocess_noalloc(ctypes.byref(p), *([nul] * 6), nul)
    assert st == _abi.SINK_ERR_SCRATCH_LIMIT
    assert "no-allocation" in sa.sink_attn_status_str(st)
    assert sa.sink_attn_noalloc_scratch_bytes() == 1 << 20


def test_noalloc_validates_like_the_workspace_entry_point():
    """The same field checks and status codes as sink_attn_bwd_preprocess: too
    many query heads is unsupported (a grid dimension), not a launch failure."""
    p = _abi.SinkAttnParams()
    p.batch, p.max_seqlen, p.total_tokens = 1, 1, 1
    p.h_q, p.h_kv, p.head_dim, p.dtype, p.causal = 70000, 1, 64, _abi.SINK_BF16, 1
    nul = ctypes.c_void_p(0)
    assert _abi.lib().sink_attn_bwd_preprocess_noalloc(ctypes.byref(p), *([nul] * 6), nul) == \
        _abi.SINK_ERR_UNSUPPORTED
    p.h_q, p.total_tokens = 64, 1 << 30  # T * h_q * d beyond the index range
    p.max_seqlen = 1 << 30
    assert _abi.lib().sink_attn_bwd_preprocess_noalloc(ctypes.byref(p), *([nul] * 6), nul) == \
        _abi.SINK_ERR_INVALID_ARG
    p.h_q, p.h_kv, p.total_tokens, p.max_seqlen = 8, 3, 16, 16  # h_q not a multiple of h_kv
    assert _abi.lib().sink_attn_bwd_preprocess_noalloc(ctypes.byref(p), *([nul] * 6), nul) == \
        _abi.SINK_ERR_INVALID_ARG


def _forward(seed, lengths, h_q, h_kv):
    prob = inputs.random_problem(seed, lengths, h_q, h_kv, 64, dtype=torch.bfloat16,
                                 sink_scale=2.0)
    d = {k: v.cuda() for k, v in prob.items()}
    o, lse = sa.sink_attn_fwd(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"],
                              max_seqlen=max(lengths))
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=max(lengths))
    return p, d, o, lse


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    # two different problems back to back: the second call reuses the array
    # that the first one filled
    for seed, lengths, h_q, h_kv in ((1, [300, 77], 8, 2), (2, [1000, 1, 2047], 16, 4)):
        p, d, o, lse = _forward(seed, lengths, h_q, h_kv)
        ref_delta, ref_ds = sa.sink_attn_bwd_preprocess(p, d["sinks"], o, lse, d["dout"])
        delta = torch.full_like(ref_delta, float("nan"))
        ds = torch.full_like(ref_ds, float("nan"))
        sa.sink_attn_bwd_preprocess_noalloc(p, d["sinks"], o, lse, d["dout"], delta=delta, dsinks=ds)
        torch.cuda.synchronize()
        assert torch.equal(delta, ref_delta)
        assert torch.equal(ds, ref_ds)
        # and the sink gradient against the oracle (inputs of ordinary spread: the
        # stored bf16 O in D stays well inside the tolerance)
        prob = {k: v.cpu() for k, v in d.items()}
        _, _, _, rds = oracle.backward(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"],
                                       scale=1 / math.sqrt(64), causal=True, window=0,
                                       cu_seqlens=prob["cu_seqlens"].numpy())
        assert_close("dS_h", ds, rds, torch.bfloat16, rounds_output=False)
