"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (the same C-ABI calls on the full inputs).

The GPU computes the whole problem; the oracle computes exact sub-problems it
can finish in seconds, and the GPU outputs they cover are compared element by
element:
  - one (sequence, key/value head) unit: all its rows and keys (its query
    heads' O, LSE, dQ; its dK, dV), since units are independent;
  - under a causal mask, the first R rows of a sequence are the whole problem
    of length R (O, LSE, dQ of those rows);
  - rows [N-R, N) evaluated over all keys give O, LSE, dQ of those rows and
    dK, dV of keys >= N-R exactly, since only those rows see those keys;
  - dS_h = -sum over all rows of P_sink * (dO . O) from the oracle's O and LSE
    (the page's simplified sink-gradient equation).
The bf16 path is the extended one (o_lo kept from the forward for D); every
test prints the per-tensor max-abs and relative L2 errors it measured.
"""
import math

import numpy as np
import pytest
import torch

import attention_sink_softmax_gb300 as sa
import oracle
from attention_sink_softmax_gb300 import inputs
from parity import assert_close, gpu_fwd_bwd

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gpu(w, prob, window):
    d = {k: (v.to(DEV) if v is not None else None) for k, v in prob.items()}
    out = gpu_fwd_bwd(d["q"], d["k"], d["v"], d["sinks"], d["dout"], d["cu_seqlens"],
                      max_seqlen=w.seqlen, causal=w.causal, window=window, softmax_scale=w.scale)
    torch.cuda.synchronize()
    out = [t.cpu() for t in out]
    del d
    torch.cuda.empty_cache()
    return out


def _print(rep):
    for name, r in rep.items():
        print(f"{name}: max-abs {r['max_abs']:.3e} rel-L2 {r['rel_l2']:.3e} "
              f"max-abs beyond one output ulp {r['max_abs_beyond_rounding']:.3e}")


def _sink_grad_from_forward(o, lse, dout, sinks_h):
    """-sum_t exp(S_h - LSE_t) (dO_t . O_t) for one head; o, dout [T, d], lse [T]."""
    D = np.einsum("td,td->t", np.asarray(dout, np.float64), o)
    return -float(np.sum(np.exp(sinks_h - lse) * D))


def _unit(prob, b, hk, g, padded):
    """Tensors of sequence b restricted to key/value head hk and its query heads."""
    hs = slice(hk * g, (hk + 1) * g)
    if padded:
        return (prob["q"][b, :, hs], prob["k"][b, :, hk:hk + 1], prob["v"][b, :, hk:hk + 1],
                prob["sinks"][hs], prob["dout"][b, :, hs])
    cu = prob["cu_seqlens"]
    a, e = int(cu[b]), int(cu[b + 1])
    return (prob["q"][a:e, hs], prob["k"][a:e, hk:hk + 1], prob["v"][a:e, hk:hk + 1],
            prob["sinks"][hs], prob["dout"][a:e, hs])


def _check_unit(w, got, prob, b, hk, window, report, tag, dsink_batches=()):
    g = w.h_q // w.h_kv
    padded = not w.packed
    q, k, v, s, do = _unit(prob, b, hk, g, padded)
    kw = dict(scale=w.scale, causal=w.causal, window=window)
    o, lse = oracle.forward(q, k, v, s, **kw)
    dq, dk, dv, ds = oracle.backward(q, k, v, s, do, **kw)
    go, glse, gdq, gdk, gdv, gds = got
    hs = slice(hk * g, (hk + 1) * g)
    if padded:
        N = w.seqlen
        tsl = slice(b * N, (b + 1) * N)
        sel = lambda t: t[b, :, hs]
        selk = lambda t: t[b, :, hk:hk + 1]
    else:
        cu = prob["cu_seqlens"]
        tsl = slice(int(cu[b]), int(cu[b + 1]))
        sel = lambda t: t[tsl, hs]
        selk = lambda t: t[tsl, hk:hk + 1]
    assert_close(f"{tag} O", sel(go), o, w.dtype, report)
    assert_close(f"{tag} LSE", glse[hs, tsl], lse, w.dtype, report, rounds_output=False)
    assert_close(f"{tag} dQ", sel(gdq), dq, w.dtype, report)
    assert_close(f"{tag} dK", selk(gdk), dk, w.dtype, report)
    assert_close(f"{tag} dV", selk(gdv), dv, w.dtype, report)
    if dsink_batches is not None:
        total = ds.copy()
        for b2 in dsink_batches:
            q2, k2, v2, s2, do2 = _unit(prob, b2, hk, g, padded)
            o2, lse2 = oracle.forward(q2, k2, v2, s2, **kw)
            for hh in range(g):
                total[hh] += _sink_grad_from_forward(o2[:, hh], lse2[hh], do2[:, hh].to(torch.float64), float(s2[hh]))
        assert_close(f"{tag} dS_h", gds[hs], total, w.dtype, report, rounds_output=False)


def test_full_causal_B2_N8192():
    w = inputs.workload(1)
    prob = inputs.make_inputs(w)
    got = _gpu(w, prob, w.window)
    rep = {}
    _check_unit(w, got, prob, b=1, hk=5, window=0, report=rep, tag="cfg1 b1 hk5", dsink_batches=[0])
    _print(rep)


def test_sliding_window_B4_N8192():
    w = inputs.workload(2)
    prob = inputs.make_inputs(w)
    got = _gpu(w, prob, w.window)
    rep = {}
    _check_unit(w, got, prob, b=2, hk=1, window=128, report=rep, tag="cfg2 b2 hk1",
                dsink_batches=[0, 1, 3])
    _check_unit(w, got, prob, b=0, hk=6, window=128, report=rep, tag="cfg2 b0 hk6", dsink_batches=None)
    _print(rep)


def test_packed_variable_length_both_layers():
    w = inputs.workload(3)
    prob = inputs.make_inputs(w)
    lengths = np.array(w.lengths)
    picks = [int(np.argmin(lengths)), int(np.argsort(lengths)[len(lengths) // 2]), int(np.argmax(lengths))]
    rep = {}
    for window in w.windows:
        got = _gpu(w, prob, window)
        for s in picks:
            _check_unit(w, got, prob, b=s, hk=7, window=window, report=rep,
                        tag=f"cfg3 win{window} seq{s} len{lengths[s]}", dsink_batches=None)
        if window > 0:
            # dS_h of query head 0 summed over all 48 sequences
            g = w.h_q // w.h_kv
            cu = prob["cu_seqlens"].numpy()
            o, lse = oracle.forward(prob["q"][:, 0:1], prob["k"][:, 0:1], prob["v"][:, 0:1],
                                    prob["sinks"][0:1], scale=w.scale, window=window,
                                    cu_seqlens=cu)
            exp = _sink_grad_from_forward(o[:, 0], lse[0], prob["dout"][:, 0].to(torch.float64),
                                          float(prob["sinks"][0]))
            assert_close("cfg3 dS_h head0", got[5][0:1], np.array([exp]), w.dtype, rep,
                         rounds_output=False)
    _print(rep)


def test_long_context_N32768_prefix_and_suffix():
    w = inputs.workload(4)
    prob = inputs.make_inputs(w)
    got = _gpu(w, prob, 0)
    go, glse, gdq, gdk, gdv, gds = got
    rep = {}
    g = w.h_q // w.h_kv
    N = w.seqlen
    kw = dict(scale=w.scale, causal=True, window=0)
    for hk in (0, 7):
        hs = slice(hk * g, (hk + 1) * g)
        q, k, v, s, do = _unit(prob, 0, hk, g, True)
        # prefix rows [0, R): the causal prefix is the whole problem of length R
        R = 1024
        o, lse = oracle.forward(q[:R], k[:R], v[:R], s, **kw)
        dq, _, _, _ = oracle.backward(q[:R], k[:R], v[:R], s, do[:R], **kw)
        assert_close(f"cfg4 hk{hk} O prefix", go[0, :R, hs], o, w.dtype, rep)
        assert_close(f"cfg4 hk{hk} LSE prefix", glse[hs, :R], lse, w.dtype, rep, rounds_output=False)
        assert_close(f"cfg4 hk{hk} dQ prefix", gdq[0, :R, hs], dq, w.dtype, rep)
        # suffix rows [N-R2, N) over all keys
        R2 = 384
        o, lse = oracle.forward(q, k, v, s, row_begin=N - R2, **kw)
        dq, dk, dv, _ = oracle.backward(q, k, v, s, do, row_begin=N - R2, **kw)
        assert_close(f"cfg4 hk{hk} O suffix", go[0, N - R2:, hs], o[N - R2:], w.dtype, rep)
        assert_close(f"cfg4 hk{hk} LSE suffix", glse[hs, N - R2:], lse[:, N - R2:], w.dtype, rep,
                     rounds_output=False)
        assert_close(f"cfg4 hk{hk} dQ suffix", gdq[0, N - R2:, hs], dq[N - R2:], w.dtype, rep)
        assert_close(f"cfg4 hk{hk} dK suffix", gdk[0, N - R2:, hk:hk + 1], dk[N - R2:], w.dtype, rep)
        assert_close(f"cfg4 hk{hk} dV suffix", gdv[0, N - R2:, hk:hk + 1], dv[N - R2:], w.dtype, rep)
    # dS_h of two heads (the largest and the smallest sink) over all rows, checked
    # as one vector (the relative L2 bound is defined on the dS_h tensor)
    heads = [int(torch.argmax(prob["sinks"])), int(torch.argmin(prob["sinks"]))]
    exps = []
    for h in heads:
        hk = h // g
        o, lse = oracle.forward(prob["q"][0, :, h:h + 1], prob["k"][0, :, hk:hk + 1],
                                prob["v"][0, :, hk:hk + 1], prob["sinks"][h:h + 1], **kw)
        exps.append(_sink_grad_from_forward(o[:, 0], lse[0], prob["dout"][0, :, h].to(torch.float64),
                                            float(prob["sinks"][h])))
    assert_close("cfg4 dS_h", gds[heads], np.array(exps), w.dtype, rep, rounds_output=False)
    _print(rep)


def test_head_dim_128_causal_B2_N8192():
    """Workload 5 (head_dim 128, 32/4 heads): one (sequence, key/value head)
    unit whole, plus the causal prefix and the last rows of another head."""
    w = inputs.workload(5)
    prob = inputs.make_inputs(w)
    got = _gpu(w, prob, w.window)
    rep = {}
    _check_unit(w, got, prob, b=0, hk=3, window=0, report=rep, tag="cfg5 b0 hk3", dsink_batches=[1])
    go, glse, gdq, gdk, gdv, _ = got
    g = w.h_q // w.h_kv
    N = w.seqlen
    kw = dict(scale=w.scale, causal=True, window=0)
    hk = 0
    hs = slice(hk * g, (hk + 1) * g)
    q, k, v, s, do = _unit(prob, 1, hk, g, True)
    R = 512
    o, lse = oracle.forward(q[:R], k[:R], v[:R], s, **kw)
    dq, _, _, _ = oracle.backward(q[:R], k[:R], v[:R], s, do[:R], **kw)
    assert_close("cfg5 b1 hk0 O prefix", go[1, :R, hs], o, w.dtype, rep)
    assert_close("cfg5 b1 hk0 dQ prefix", gdq[1, :R, hs], dq, w.dtype, rep)
    R2 = 256
    o, lse = oracle.forward(q, k, v, s, row_begin=N - R2, **kw)
    dq, dk, dv, _ = oracle.backward(q, k, v, s, do, row_begin=N - R2, **kw)
    assert_close("cfg5 b1 hk0 O suffix", go[1, N - R2:, hs], o[N - R2:], w.dtype, rep)
    assert_close("cfg5 b1 hk0 LSE suffix", glse[hs, N + N - R2:], lse[:, N - R2:], w.dtype, rep,
                 rounds_output=False)
    assert_close("cfg5 b1 hk0 dQ suffix", gdq[1, N - R2:, hs], dq[N - R2:], w.dtype, rep)
    assert_close("cfg5 b1 hk0 dK suffix", gdk[1, N - R2:, hk:hk + 1], dk[N - R2:], w.dtype, rep)
    assert_close("cfg5 b1 hk0 dV suffix", gdv[1, N - R2:, hk:hk + 1], dv[N - R2:], w.dtype, rep)
    _print(rep)
