"""GPU parity of libsinkattn against the fp64 oracle, element by element, on
seeded inputs that span several tiles with ragged tails, plus edge cases.

All calls go through the C ABI (via the ctypes binding). bf16 runs through the
extended entry points (o_lo kept from the forward for D), fp32 through the
plain ones; the plain bf16 entry points are checked on their own below."""
import math

import numpy as np
import pytest
import torch

import attention_sink_softmax_gb300 as sa
from attention_sink_softmax_gb300 import _abi, inputs
from parity import assert_close, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(prob, *, causal=True, window=0, scale=None, max_seqlen=None):
    d = {k: (v.to(DEV) if v is not None else None) for k, v in prob.items()}
    out = gpu_fwd_bwd(d["q"], d["k"], d["v"], d["sinks"], d["dout"], d["cu_seqlens"],
                      max_seqlen=max_seqlen, causal=causal, window=window, softmax_scale=scale)
    torch.cuda.synchronize()
    return out


def _check(prob, dtype, *, causal=True, window=0, scale=None, got=None):
    hd = prob["q"].shape[-1]
    sc = scale if scale is not None else 1.0 / math.sqrt(hd)
    if got is None:
        got = _run(prob, causal=causal, window=window, scale=scale)
    ref = oracle_fwd_bwd(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"], scale=sc,
                         causal=causal, window=window, cu_seqlens=prob["cu_seqlens"])
    for name, g, r in zip(("O", "LSE", "dQ", "dK", "dV"), got[:5], ref[:5]):
        assert_close(name, g, r.reshape(tuple(g.shape)), dtype, rounds_output=(name != "LSE"))
    assert_close("dS_h", got[5], ref[5], dtype, rounds_output=False)
    return got


def test_tiny_fp32_workload_full_oracle():
    """B=1, N=128, H_q=4, H_kv=1, d=64, fp32, causal, seed 0: every output."""
    w = inputs.workload(0)
    prob = inputs.make_inputs(w)
    _check(prob, torch.float32)


CASES = [
    # lengths, h_q, h_kv, packed, causal, window
    ([300, 300], 8, 2, False, True, 0),        # padded, 3 tiles + ragged tail (a 1-tile CTA)
    ([512, 512], 4, 2, False, True, 0),        # padded, 4 whole tiles, two 2-tile CTAs per sequence
    ([1, 127, 129, 255, 300], 4, 1, True, True, 0),
    ([517], 8, 8, True, True, 128),            # MHA, window 128
    ([640, 33], 8, 1, True, True, 1),          # MQA, window 1 (diagonal only)
    ([200, 385], 4, 2, True, True, 200),
    ([200], 4, 1, True, False, 0),             # no mask (the page's pseudocode)
    ([5, 0, 7, 130], 4, 2, True, True, 0),     # an empty sequence in the middle
    ([333, 190], 6, 2, True, True, 0),         # group of 3: the forward's odd-group CTAs
    ([700], 5, 1, True, True, 4096),           # group of 5, window longer than the sequence
    ([900, 260], 14, 2, True, True, 640),      # group of 7, window 640
    ([700, 301], 6, 2, True, True, 256),       # window 256 (the multi-tile forward's limit), group of 3
    ([513, 129], 8, 2, True, True, 256),       # window 256, pairs of query heads, ragged tails
    ([600, 77], 8, 2, True, True, 257),        # just above it: two row tiles per CTA, both bounds
    ([2100, 700, 3], 4, 2, True, True, 0),     # causal pairs: 17 row tiles, one CTA of one tile
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lengths,h_q,h_kv,packed,causal,window", CASES)
def test_small_parity(dtype, lengths, h_q, h_kv, packed, causal, window):
    prob = inputs.random_problem(11, lengths, h_q, h_kv, 64, dtype=dtype, packed=packed,
                                 sink_scale=2.0)
    _check(prob, dtype, causal=causal, window=window)


D128_CASES = [
    # lengths, h_q, h_kv, causal, window
    ([300, 129], 4, 2, True, 0),     # several tiles and ragged tails
    ([517], 6, 2, True, 200),        # group of 3, window
    ([200, 1], 2, 1, False, 0),      # no mask
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lengths,h_q,h_kv,causal,window", D128_CASES)
def test_head_dim_128_parity(dtype, lengths, h_q, h_kv, causal, window):
    """head_dim 128: in bf16 the forward on the tensor cores (one 128-row tile
    per CTA, two 64-column atoms per tile) and the backward's dQ and dK/dV
    tensor-core kernels; the fp32 path on the CUDA cores."""
    prob = inputs.random_problem(21, lengths, h_q, h_kv, 128, dtype=dtype, packed=True,
                                 sink_scale=2.0)
    _check(prob, dtype, causal=causal, window=window)


def test_large_logits_and_extreme_sinks():
    """Q, K scaled x4 (logit std ~16) with sinks in [-10, 10], and sinks of
    +-30 that make rows sink-dominated or sink-negligible."""
    prob = inputs.random_problem(5, [777], 8, 2, 64, dtype=torch.bfloat16, qk_gain=4.0)
    prob["sinks"] = torch.linspace(-10, 10, 8)
    _check(prob, torch.bfloat16, scale=0.125)
    # logits of std ~1 with sinks of +-30: the +30 heads are sink-dominated
    prob = inputs.random_problem(5, [777], 8, 2, 64, dtype=torch.bfloat16)
    prob["sinks"] = torch.tensor([30.0, -30.0] * 4)
    o, lse, *_ = _check(prob, torch.bfloat16, scale=0.125)
    assert float(o[:, 0::2].abs().max()) < 2e-2
    assert float((lse[0::2] - 30.0).abs().max()) < 1e-3


def test_minus_infinity_sink_is_standard_attention():
    """S_h = -inf takes no probability mass (section "标准注意力机制回顾" form)."""
    for dtype in (torch.bfloat16, torch.float32):
        prob = inputs.random_problem(12, [300, 77], 8, 2, 64, dtype=dtype)
        prob["sinks"] = torch.full((8,), float("-inf"))
        got = _check(prob, dtype, window=100)
        assert torch.all(got[5] == 0)


def test_window_wider_than_sequence_equals_causal():
    prob = inputs.random_problem(3, [300, 41], 8, 2, 64)
    a = _run(prob, window=0)
    b = _run(prob, window=4096)
    for x, y in zip(a, b):
        torch.testing.assert_close(x, y, rtol=0, atol=0)


def test_packed_single_sequence_equals_padded():
    prob = inputs.random_problem(4, [384, 384], 8, 2, 64, packed=False)
    a = _run(prob)
    packed = {k: (v.reshape(-1, *v.shape[2:]) if k in ("q", "k", "v", "dout") else v)
              for k, v in prob.items()}
    packed["cu_seqlens"] = torch.tensor([0, 384, 768], dtype=torch.int32)
    b = _run(packed)
    for x, y in zip(a[:1] + a[2:5], b[:1] + b[2:5]):
        torch.testing.assert_close(x.reshape(y.shape), y, rtol=0, atol=0)
    torch.testing.assert_close(a[1], b[1], rtol=0, atol=0)
    torch.testing.assert_close(a[5], b[5], rtol=0, atol=0)


def test_sink_gradient_is_deterministic():
    prob = inputs.random_problem(6, [1000, 531], 8, 2, 64)
    first = _run(prob)[5]
    for _ in range(3):
        torch.testing.assert_close(_run(prob)[5], first, rtol=0, atol=0)


def test_plain_entry_points_without_o_lo():
    """sink_attn_fwd / sink_attn_bwd (no o_lo): O, LSE and dV are bit for bit
    those of the extended path (the forward is the same kernel and dV does not
    involve D); dQ, dK and dS_h use D from the stored bf16 O and still meet the
    stated tolerance on inputs of ordinary spread."""
    prob = inputs.random_problem(13, [300, 517], 8, 2, 64, dtype=torch.bfloat16, packed=True,
                                 sink_scale=2.0)
    d = {k: v.to(DEV) for k, v in prob.items()}
    kw = dict(max_seqlen=517)
    o, lse = sa.sink_attn_fwd(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], **kw)
    plain = (o, lse) + sa.sink_attn_bwd(d["q"], d["k"], d["v"], d["sinks"], o, lse, d["dout"],
                                         d["cu_seqlens"], **kw)
    ext = _run(prob, max_seqlen=517)
    for i in (0, 1, 4):
        assert torch.equal(plain[i], ext[i]), ("O", "LSE", "dQ", "dK", "dV")[i]
    _check(prob, torch.bfloat16, got=plain)


def test_o_lo_is_the_rounding_residual_of_o():
    """o_lo = bf16(O - bf16(O)): o + o_lo is closer to the exact O than o by
    about the 8 more bits it carries, and o_lo is within half a bf16 ulp of o."""
    prob = inputs.random_problem(14, [400], 8, 2, 64, dtype=torch.bfloat16, packed=True)
    d = {k: v.to(DEV) for k, v in prob.items()}
    o, o_lo, lse = sa.sink_attn_fwd_ex(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"],
                                       max_seqlen=400)
    ro, _ = oracle_fwd_bwd(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["dout"],
                           scale=0.125, causal=True, window=0, cu_seqlens=prob["cu_seqlens"],
                           backward=False)
    o64, lo64 = o.double().cpu().numpy(), o_lo.double().cpu().numpy()
    err_hi = np.abs(o64 - ro).max()
    err_both = np.abs(o64 + lo64 - ro).max()
    assert err_both < err_hi / 16, (err_hi, err_both)
    assert np.all(np.abs(lo64) <= 2.0 ** -8 * np.abs(o64) + 1e-30)


@pytest.mark.parametrize("window", [0, 128])
def test_deterministic_mode_gives_reproducible_dq(window):
    """sink_attn_set_deterministic(1): the 64-wide backward as a dK/dV kernel
    and a query-owning dQ kernel. dq is then the same bit for bit on every run
    and within tolerance of the oracle (large logits included); dk, dv and
    dS_h equal the default path's bit for bit (the same kernels compute them)."""
    for gain in (1.0, 4.0):
        prob = inputs.random_problem(15, [700, 300], 8, 2, 64, dtype=torch.bfloat16, packed=True,
                                     sink_scale=2.0, qk_gain=gain)
        default = _run(prob, window=window, scale=0.125)
        prev = sa.sink_attn_set_deterministic(True)
        try:
            runs = [_run(prob, window=window, scale=0.125) for _ in range(3)]
        finally:
            sa.sink_attn_set_deterministic(prev)
        for r in runs[1:]:
            for x, y in zip(r, runs[0]):
                assert torch.equal(x, y)
        for i in (0, 1, 3, 4, 5):  # O, LSE, dK, dV, dS_h
            assert torch.equal(runs[0][i], default[i]), i
        _check(prob, torch.bfloat16, window=window, scale=0.125, got=runs[0])


def test_empty_input():
    q = torch.empty(0, 4, 64, dtype=torch.bfloat16, device=DEV)
    k = torch.empty(0, 1, 64, dtype=torch.bfloat16, device=DEV)
    sinks = torch.randn(4, device=DEV)
    cu = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = sa.sink_attn_fwd(q, k, k, sinks, cu, max_seqlen=0)
    dq, dk, dv, ds = sa.sink_attn_bwd(q, k, k, sinks, o, lse, q, cu, max_seqlen=0)
    torch.cuda.synchronize()
    assert o.numel() == 0 and lse.numel() == 0
    assert torch.all(ds == 0)
    o, o_lo, lse = sa.sink_attn_fwd_ex(q, k, k, sinks, cu, max_seqlen=0)
    dq, dk, dv, ds = sa.sink_attn_bwd_ex(q, k, k, sinks, o, o_lo, lse, q, cu, max_seqlen=0)
    torch.cuda.synchronize()
    assert torch.all(ds == 0)


def test_sequence_longer_than_max_seqlen_is_flagged():
    """Rows past max_seqlen are not computed and the device flag reports it."""
    prob = inputs.random_problem(8, [100, 300], 4, 1, 64)
    d = {k: v.to(DEV) for k, v in prob.items()}
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=256)
    ws = torch.empty(sa.sink_attn_workspace_bytes(p, False), dtype=torch.uint8, device=DEV)
    sa.sink_attn_fwd(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], params=p, workspace=ws)
    st, flags = sa.sink_attn_fetch_device_error(ws)
    assert st == _abi.SINK_ERR_DEVICE and flags == 2
    st, flags = sa.sink_attn_fetch_device_error(ws)  # cleared by the read
    assert st == _abi.SINK_OK and flags == 0


def test_host_pointer_rejected_before_launch():
    prob = inputs.random_problem(9, [64], 4, 1, 64)
    d = {k: (v.to(DEV) if v is not None else None) for k, v in prob.items()}
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=64)
    ws = torch.empty(sa.sink_attn_workspace_bytes(p, False), dtype=torch.uint8, device=DEV)
    host_q = prob["q"].contiguous()
    o = torch.empty_like(d["q"])
    lse = torch.empty(4, 64, device=DEV)
    st = _abi.lib().sink_attn_fwd(
        __import__("ctypes").byref(p), sa._ptr(host_q), sa._ptr(d["k"]), sa._ptr(d["v"]),
        sa._ptr(d["sinks"]), sa._ptr(d["cu_seqlens"]), sa._ptr(o), sa._ptr(lse), sa._ptr(ws),
        ws.numel(), sa._stream(None, d["q"].device))
    assert st == _abi.SINK_ERR_INVALID_ARG


def test_autograd_wrapper_matches_direct_calls():
    prob = inputs.random_problem(10, [333], 8, 2, 64)
    d = {k: (v.to(DEV) if v is not None else None) for k, v in prob.items()}
    q = d["q"].clone().requires_grad_()
    k = d["k"].clone().requires_grad_()
    v = d["v"].clone().requires_grad_()
    s = d["sinks"].clone().requires_grad_()
    o = sa.sink_attention(q, k, v, s, d["cu_seqlens"], max_seqlen=333)
    o.backward(d["dout"])
    ref = _run(prob)
    torch.testing.assert_close(o.detach(), ref[0], rtol=0, atol=0)
    for g, r in zip((q.grad, k.grad, v.grad, s.grad), ref[2:]):
        torch.testing.assert_close(g, r, rtol=0, atol=0)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_training_step_under_cuda_graph_capture_matches_eager(head_dim):
    """The forward and backward entry points only enqueue work on the caller's
    stream (no synchronisation, no allocation), so a training step captured in
    a CUDA graph and replayed gives the eager results: bit for bit for O, LSE,
    dK, dV and dS_h; dQ at d = 64 comes from fp32 reduce-adds whose order
    varies, so it may differ in the last bf16 place."""
    prob = inputs.random_problem(8, [300, 517], 8, 2, head_dim, dtype=torch.bfloat16, packed=True)
    d = {k: v.to(DEV) for k, v in prob.items()}
    p = sa.make_params(d["q"], d["k"], d["cu_seqlens"], max_seqlen=517)
    wf = torch.empty(sa.sink_attn_workspace_bytes(p, False), dtype=torch.uint8, device=DEV)
    wb = torch.empty(sa.sink_attn_workspace_bytes(p, True), dtype=torch.uint8, device=DEV)
    args = (d["q"], d["k"], d["v"], d["sinks"])

    def step(outs, stream):
        o, lse, dq, dk, dv, ds, o_lo = outs
        sa.sink_attn_fwd_ex(*args, d["cu_seqlens"], out=o, o_lo=o_lo, lse=lse, workspace=wf,
                            params=p, stream=stream)
        sa.sink_attn_bwd_ex(*args, o, o_lo, lse, d["dout"], d["cu_seqlens"], dq=dq, dk=dk, dv=dv,
                            dsinks=ds, workspace=wb, params=p, stream=stream)

    def alloc():
        return (torch.empty_like(d["q"]), torch.empty(8, d["q"].shape[0], device=DEV),
                torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
                torch.empty_like(d["sinks"]), torch.empty_like(d["q"]))

    eager = alloc()
    step(eager, torch.cuda.current_stream())
    torch.cuda.synchronize()
    graphed = alloc()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        step(graphed, torch.cuda.current_stream())
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV", "dS_h", "o_lo"), eager, graphed):
        if name == "dQ" and head_dim == 64:
            torch.testing.assert_close(b.float(), a.float(), rtol=1e-2, atol=1e-2)
        else:
            assert torch.equal(a, b), name
    assert sa.sink_attn_fetch_device_error(wb)[0] == _abi.SINK_OK
