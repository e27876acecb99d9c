"""The backward's preparation pass issued on its own (sink_attn_bwd_prepare)
on a second, lower-priority stream while the forward runs, then
sink_attn_bwd_main with SINK_BWD_PREPARED: the same gradients as the one-call
backward (dK, dV bit for bit; dQ, whose fp32 reduce-adds land in a varying
order, within the bf16 tolerance of the oracle), for both backward modes and
for the paths that need no preparation."""
import math

import pytest
import torch

import attention_sink_softmax_gb300 as sa
from attention_sink_softmax_gb300 import inputs
from parity import assert_close, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


def _split_step(d, p, side):
    """fwd on the current stream with the preparation on `side`; then the
    backward steps with the prepared workspace."""
    main = torch.cuda.current_stream()
    ws = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device="cuda")
    ready = torch.cuda.Event()
    ready.record(main)
    side.wait_event(ready)
    sa.sink_attn_bwd_prepare(p, d["q"], d["k"], workspace=ws, stream=side)
    prepared = torch.cuda.Event()
    prepared.record(side)
    o, o_lo, lse = sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], params=p)
    delta, ds = sa.sink_attn_bwd_preprocess_ex(p, d["sinks"], o, o_lo, lse, d["dout"], workspace=ws)
    main.wait_event(prepared)
    dq, dk, dv = sa.sink_attn_bwd_main(p, d["q"], d["k"], d["v"], lse, delta, d["dout"],
                                       d["cu_seqlens"], workspace=ws, prepared=True)
    return o, lse, dq, dk, dv, ds


def _one_call(d, p):
    o, o_lo, lse = sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], params=p)
    dq, dk, dv, ds = sa.sink_attn_bwd_ex(d["q"], d["k"], d["v"], d["sinks"], o, o_lo, lse, d["dout"],
                                         d["cu_seqlens"], params=p)
    return o, lse, dq, dk, dv, ds


@pytest.mark.parametrize("head_dim,deterministic", [(64, False), (64, True), (128, False)])
def test_prepared_backward_matches_the_one_call_backward(head_dim, deterministic):
    prob = inputs.random_problem(23, [700, 333], 8, 2, head_dim, dtype=torch.bfloat16, packed=True,
                                 sink_scale=2.0)
    d = {k: (v.cuda() if v is not None else None) for k, v in prob.items()}
    scale = 1.0 / math.sqrt(head_dim)
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=700, causal=True, window=0,
                       softmax_scale=scale)
    side = torch.cuda.Stream(priority=0)
    prev = sa.sink_attn_set_deterministic(deterministic)
    try:
        ref = _one_call(d, p)
        got = _split_step(d, p, side)
        torch.cuda.synchronize()
    finally:
        sa.sink_attn_set_deterministic(prev)
    for i in (0, 1, 3, 4, 5):  # O, LSE, dK, dV, dS_h
        assert torch.equal(got[i], ref[i]), i
    if deterministic or head_dim == 128:
        assert torch.equal(got[2], ref[2])
    oracle = oracle_fwd_bwd(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"], scale=scale,
                            causal=True, window=0, cu_seqlens=prob["cu_seqlens"])
    assert_close("dQ", got[2], oracle[2].reshape(tuple(got[2].shape)), torch.bfloat16)


def test_prepared_workspace_reused_over_steps():
    """Several steps on one workspace: each step's preparation is ordered after
    the previous step's backward (the accumulator it zeroes is the one that
    backward read), and every step's dQ matches the oracle."""
    prob = inputs.random_problem(29, [512, 384], 8, 2, 64, dtype=torch.bfloat16, packed=True)
    d = {k: (v.cuda() if v is not None else None) for k, v in prob.items()}
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=512, causal=True, window=0,
                       softmax_scale=0.125)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=0)
    ws = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device="cuda")
    oracle = oracle_fwd_bwd(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"], scale=0.125,
                            causal=True, window=0, cu_seqlens=prob["cu_seqlens"])
    done = torch.cuda.Event()
    done.record(main)
    for _ in range(3):
        side.wait_event(done)
        sa.sink_attn_bwd_prepare(p, d["q"], d["k"], workspace=ws, stream=side)
        prepared = torch.cuda.Event()
        prepared.record(side)
        o, o_lo, lse = sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], params=p)
        delta, _ = sa.sink_attn_bwd_preprocess_ex(p, d["sinks"], o, o_lo, lse, d["dout"], workspace=ws)
        main.wait_event(prepared)
        dq, _, _ = sa.sink_attn_bwd_main(p, d["q"], d["k"], d["v"], lse, delta, d["dout"],
                                         d["cu_seqlens"], workspace=ws, prepared=True)
        done = torch.cuda.Event()
        done.record(main)
        torch.cuda.synchronize()
        assert_close("dQ", dq, oracle[2].reshape(tuple(dq.shape)), torch.bfloat16)


@pytest.mark.parametrize("prep_det,main_det", [(True, False), (False, True)])
def test_reproducible_setting_may_change_between_prepare_and_main(prep_det, main_det):
    """The workspace layout is the same in both backward modes, and the
    preparation always zeroes the accumulator, so flipping
    sink_attn_set_deterministic between the two calls still gives correct
    gradients."""
    prob = inputs.random_problem(31, [640, 200], 8, 2, 64, dtype=torch.bfloat16, packed=True,
                                 sink_scale=2.0)
    d = {k: (v.cuda() if v is not None else None) for k, v in prob.items()}
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=640, causal=True, window=0,
                       softmax_scale=0.125)
    ws = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device="cuda")
    prev = sa.sink_attn_set_deterministic(prep_det)
    try:
        sa.sink_attn_bwd_prepare(p, d["q"], d["k"], workspace=ws)
        o, o_lo, lse = sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], params=p)
        delta, ds = sa.sink_attn_bwd_preprocess_ex(p, d["sinks"], o, o_lo, lse, d["dout"], workspace=ws)
        sa.sink_attn_set_deterministic(main_det)
        dq, dk, dv = sa.sink_attn_bwd_main(p, d["q"], d["k"], d["v"], lse, delta, d["dout"],
                                           d["cu_seqlens"], workspace=ws, prepared=True)
        torch.cuda.synchronize()
    finally:
        sa.sink_attn_set_deterministic(prev)
    oracle = oracle_fwd_bwd(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"], scale=0.125,
                            causal=True, window=0, cu_seqlens=prob["cu_seqlens"])
    for name, g, r in (("dQ", dq, oracle[2]), ("dK", dk, oracle[3]), ("dV", dv, oracle[4])):
        assert_close(name, g, r.reshape(tuple(g.shape)), torch.bfloat16)
