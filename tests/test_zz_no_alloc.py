"""sink_attn_bwd_preprocess_noalloc: backward step 1 for callers that cannot
allocate device memory (they are handed inputs and outputs only, e.g. a plugin
inside a framework that owns all device memory). It keeps its scratch in a
fixed array inside the library; these tests check it against the workspace
entry point, sink_attn_bwd_preprocess, through the C ABI, on consecutive calls
that share that array.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import attention_sink_softmax_gb300 as sa
from attention_sink_softmax_gb300 import _abi, inputs
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
        assert_close("delta", delta, ref_delta.cpu().double().numpy(), torch.bfloat16,
                     rounds_output=False)
        assert_close("dS_h", ds, ref_ds.cpu().double().numpy(), torch.bfloat16, rounds_output=False)
