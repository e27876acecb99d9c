"""Conditions found on the device, reported through the workspace's flag word
(sink_attn_fetch_device_error) without faulting or hanging the GPU:

  - cu_seqlens that is not a valid packing (it lives in device memory, so only
    the kernels can check it): every kernel checks its sequence's bounds before
    any load or store and skips a bad sequence;
  - a bounded wait that runs out: the test hook withholds the producer's loads
    after its first stage, the wait limit is lowered to a few milliseconds, the
    kernel reports SINK_ERR_TIMEOUT and returns; a normal call on the same
    stream afterwards is correct.
"""
import math

import numpy as np
import pytest
import torch

import attention_sink_softmax_gb300 as sa
from attention_sink_softmax_gb300 import _abi, inputs
from parity import assert_close, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 7.0


def _bad_seqlens_case(cu_list, total, dtype, head_dim):
    """Forward and backward on packed inputs of `total` tokens with the given
    cu_seqlens; returns (fwd status, fwd flags, bwd status, bwd flags, o)."""
    prob = inputs.random_problem(31, [total], 4, 2, head_dim, dtype=dtype, packed=True)
    d = {k: v.to(DEV) for k, v in prob.items()}
    cu = torch.tensor(cu_list, dtype=torch.int32, device=DEV)
    p = sa.make_params(d["q"], d["k"], cu, max_seqlen=total)
    wf = torch.empty(sa.sink_attn_workspace_bytes(p, False), dtype=torch.uint8, device=DEV)
    wb = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device=DEV)
    o = torch.full_like(d["q"], SENTINEL)
    lse = torch.full((4, total), SENTINEL, device=DEV)
    if dtype == torch.bfloat16:
        o_lo = torch.zeros_like(d["q"])
        sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], cu, out=o, o_lo=o_lo, lse=lse,
                            workspace=wf, params=p)
    else:
        sa.sink_attn_fwd(d["q"], d["k"], d["v"], d["sinks"], cu, out=o, lse=lse, workspace=wf,
                         params=p)
    fst, fflags = sa.sink_attn_fetch_device_error(wf)
    sa.sink_attn_bwd(d["q"], d["k"], d["v"], d["sinks"], o, lse, d["dout"], cu, workspace=wb,
                     params=p)
    bst, bflags = sa.sink_attn_fetch_device_error(wb)
    torch.cuda.synchronize()
    return fst, fflags, bst, bflags, o.cpu(), lse.cpu()


@pytest.mark.parametrize("dtype,head_dim", [(torch.bfloat16, 64), (torch.bfloat16, 128),
                                            (torch.float32, 64)])
@pytest.mark.parametrize("cu_list,untouched", [
    ([0, 100, 500], (100, 400)),   # the last sequence ends past total_tokens
    ([0, 300, 200], (300, 400)),   # cu_seqlens decreases
    ([8, 100, 400], (0, 100)),     # cu_seqlens[0] != 0
    ([0, -5, 400], (0, 400)),      # a negative boundary: both sequences are invalid
])
def test_bad_cu_seqlens_flagged_and_skipped(dtype, head_dim, cu_list, untouched):
    fst, fflags, bst, bflags, o, lse = _bad_seqlens_case(cu_list, 400, dtype, head_dim)
    assert fst == _abi.SINK_ERR_DEVICE and fflags & _abi.SINK_FLAG_BAD_SEQLENS, (fst, fflags)
    assert bst == _abi.SINK_ERR_DEVICE and bflags & _abi.SINK_FLAG_BAD_SEQLENS, (bst, bflags)
    a, b = untouched
    # rows that only an invalid sequence covers are left as they were
    assert torch.all(o[a:b].float() == SENTINEL)
    assert torch.all(lse[:, a:b] == SENTINEL)


def test_valid_packing_raises_no_flag():
    fst, fflags, bst, bflags, o, _ = _bad_seqlens_case([0, 100, 400], 400, torch.bfloat16, 64)
    assert (fst, fflags, bst, bflags) == (_abi.SINK_OK, 0, _abi.SINK_OK, 0)
    assert torch.all(torch.isfinite(o.float()))


def test_bounded_wait_gives_up_and_the_next_call_is_correct():
    """The forward's and the backward's producers withhold their loads after the
    first stage; with a 5 ms wait limit the consumers give up, the call reports
    SINK_ERR_TIMEOUT, and the same stream then runs a correct step."""
    prob = inputs.random_problem(32, [600, 300], 8, 2, 64, dtype=torch.bfloat16, packed=True)
    d = {k: v.to(DEV) for k, v in prob.items()}
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=600)
    wf = torch.empty(sa.sink_attn_workspace_bytes(p, False), dtype=torch.uint8, device=DEV)
    wb = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device=DEV)
    prev = sa.sink_attn_set_wait_limit_ns(5_000_000)
    sa.sink_attn_testing_withhold_load(True)
    try:
        o, o_lo, lse = sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"],
                                           params=p, workspace=wf)
        st, flags = sa.sink_attn_fetch_device_error(wf)
        assert st == _abi.SINK_ERR_TIMEOUT and flags & _abi.SINK_FLAG_TIMEOUT, (st, flags)
        sa.sink_attn_bwd_ex(d["q"], d["k"], d["v"], d["sinks"], o, o_lo, lse, d["dout"],
                            d["cu_seqlens"], params=p, workspace=wb)
        st, flags = sa.sink_attn_fetch_device_error(wb)
        assert st == _abi.SINK_ERR_TIMEOUT and flags & _abi.SINK_FLAG_TIMEOUT, (st, flags)
    finally:
        sa.sink_attn_testing_withhold_load(False)
        sa.sink_attn_set_wait_limit_ns(prev)
    torch.cuda.synchronize()
    # the context is usable and the next step is correct
    got = gpu_fwd_bwd(d["q"], d["k"], d["v"], d["sinks"], d["dout"], d["cu_seqlens"], params=p)
    torch.cuda.synchronize()
    ref = oracle_fwd_bwd(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"], scale=0.125,
                         causal=True, window=0, cu_seqlens=prob["cu_seqlens"])
    for name, g, r in zip(("O", "LSE", "dQ", "dK", "dV", "dS_h"), got, ref):
        assert_close(name, g, r, torch.bfloat16, rounds_output=name not in ("LSE", "dS_h"))
