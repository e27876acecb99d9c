"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Every check compares the oracle with something other than itself: the page's
invariant, closed forms, a hand-derived worked example, torch's own
scaled_dot_product_attention (a library routine) with the sink expressed as an
extra key, and central finite differences. Citations refer to the page
"惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！" (nmedialink.com) by section.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, T, h_q, h_kv, d, sink_scale=1.0):
    q = rng.standard_normal((T, h_q, d))
    k = rng.standard_normal((T, h_kv, d))
    v = rng.standard_normal((T, h_kv, d))
    sinks = sink_scale * rng.standard_normal(h_q)
    dout = rng.standard_normal((T, h_q, d))
    return q, k, v, sinks, dout


def _mask(L, causal, window):
    """Boolean [L, L] matrix of allowed (row, key) pairs."""
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    if not causal:
        return np.ones((L, L), dtype=bool)
    m = j <= i
    if window > 0:
        m &= j >= i - window + 1
    return m


def _sdpa_with_virtual_sink_key(q, k, v, sinks, dout, cu, scale, causal, window):
    """Sink attention expressed through torch.nn.functional.scaled_dot_product_attention.

    The sink is one extra key whose score is S_h and whose value row is zero
    (section "GPT-OSS中的带注意力槽的注意力机制": the sink joins the softmax but
    contributes no value). It is realised as a zero key/value row plus an
    additive float mask whose last column holds S_h, so torch's own softmax,
    matmuls and autograd produce the forward and every gradient.
    """
    T, h_q, d = q.shape
    h_kv = k.shape[1]
    g = h_q // h_kv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    ts = torch.tensor(sinks, requires_grad=True)
    outs, lses = [], []
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        qs = tq[a:b].permute(1, 0, 2)  # [H, L, d]
        ks = tk[a:b].permute(1, 0, 2).repeat_interleave(g, dim=0)
        vs = tv[a:b].permute(1, 0, 2).repeat_interleave(g, dim=0)
        zero = torch.zeros(h_q, 1, d, dtype=torch.float64)
        k_ext = torch.cat([ks, zero], dim=1)
        v_ext = torch.cat([vs, zero], dim=1)
        allowed = torch.tensor(_mask(L, causal, window))
        content = torch.zeros(L, L, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
        mask = torch.cat([content.expand(h_q, L, L), ts.view(h_q, 1, 1).expand(h_q, L, 1)], dim=2)
        from torch.nn.attention import SDPBackend, sdpa_kernel
        with sdpa_kernel(SDPBackend.MATH):
            o = torch.nn.functional.scaled_dot_product_attention(
                qs.unsqueeze(0), k_ext.unsqueeze(0), v_ext.unsqueeze(0),
                attn_mask=mask.unsqueeze(0), scale=scale)[0]
        outs.append(o.permute(1, 0, 2))
        scores = scale * (qs @ k_ext.transpose(1, 2)) + mask
        lses.append(torch.logsumexp(scores, dim=-1))
    O = torch.cat(outs, 0)
    lse = torch.cat(lses, 1)
    (O * torch.tensor(dout)).sum().backward()
    return (O.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(),
            tv.grad.numpy(), ts.grad.numpy())


CASES = [
    # (lengths, h_q, h_kv, d, causal, window)
    ([37], 4, 2, 16, True, 0),
    ([9, 30, 1, 17], 4, 1, 8, True, 0),
    ([40], 2, 2, 8, True, 5),
    ([12, 25], 6, 3, 8, True, 1),
    ([21], 2, 1, 8, False, 0),
    ([19, 6], 4, 2, 128, True, 7),   # the 128-wide head of the variants
]


@pytest.mark.parametrize("lengths,h_q,h_kv,d,causal,window", CASES)
def test_matches_sdpa_with_sink_as_zero_value_key(lengths, h_q, h_kv, d, causal, window):
    rng = np.random.default_rng(7)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v, sinks, dout = _rand_problem(rng, int(cu[-1]), h_q, h_kv, d, sink_scale=2.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.forward(q, k, v, sinks, scale=scale, causal=causal, window=window, cu_seqlens=cu)
    dq, dk, dv, ds = oracle.backward(q, k, v, sinks, dout, scale=scale, causal=causal,
                                     window=window, cu_seqlens=cu)
    ro, rlse, rdq, rdk, rdv, rds = _sdpa_with_virtual_sink_key(q, k, v, sinks, dout, cu, scale,
                                                               causal, window)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, rdq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, rdk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, rdv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ds, rds, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0)])
def test_sink_to_minus_infinity_is_standard_attention(causal, window):
    """Section "标准注意力机制回顾": with S_h -> -inf the sink takes no mass and the
    result is plain softmax attention, here torch's scaled_dot_product_attention."""
    rng = np.random.default_rng(3)
    T, h, d = 33, 3, 16
    q, k, v, _, _ = _rand_problem(rng, T, h, h, d)
    sinks = np.full(h, -1e300)
    o, _ = oracle.forward(q, k, v, sinks, causal=causal, window=window)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).permute(1, 0, 2), torch.tensor(k).permute(1, 0, 2),
        torch.tensor(v).permute(1, 0, 2), is_causal=causal).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_row_probabilities_sum_to_one_and_row_identity():
    """Section "GPT-OSS中的带注意力槽的注意力机制": sum_j P_ij + P_sink = 1 per row.
    Softmax shift invariance: the combined-row gradient sums to 0."""
    rng = np.random.default_rng(11)
    cu = np.array([0, 50, 64], dtype=np.int32)
    q, k, v, sinks, dout = _rand_problem(rng, 64, 4, 2, 8, sink_scale=3.0)
    for window in (0, 7):
        for seq in range(2):
            for head in range(4):
                L = cu[seq + 1] - cu[seq]
                for i in range(L):
                    first, p, dz = oracle.row(q, k, v, sinks, seq=seq, head=head, i=i, dout=dout,
                                              window=window, cu_seqlens=cu)
                    n = len(p) - 1
                    assert n == (i + 1 if window == 0 else min(i + 1, window))
                    assert first == i + 1 - n
                    assert abs(p.sum() - 1.0) < 1e-12
                    assert np.all(p > 0)
                    assert abs(dz.sum()) < 1e-12


def test_sink_gradient_is_sum_of_row_terms():
    """Section "反向传播的实现", simplified form: dL/dS_h = sum over rows of
    -P_{i,h} * sum_j P_ij * upstream_ij, i.e. the sum of each row's sink entry."""
    rng = np.random.default_rng(5)
    cu = np.array([0, 20, 45], dtype=np.int32)
    q, k, v, sinks, dout = _rand_problem(rng, 45, 2, 1, 8)
    _, _, _, ds = oracle.backward(q, k, v, sinks, dout, cu_seqlens=cu)
    o, _ = oracle.forward(q, k, v, sinks, cu_seqlens=cu)
    for head in range(2):
        acc = 0.0
        for seq in range(2):
            for i in range(cu[seq + 1] - cu[seq]):
                _, p, dz = oracle.row(q, k, v, sinks, seq=seq, head=head, i=i, dout=dout,
                                      cu_seqlens=cu)
                row_tok = cu[seq] + i
                # the row term equals -P_{i,h} * (dO_i . O_i)
                assert abs(dz[-1] + p[-1] * np.dot(dout[row_tok, head], o[row_tok, head])) < 1e-12
                acc += dz[-1]
        assert abs(acc - ds[head]) < 1e-12


def _loss(q, k, v, sinks, dout, **kw):
    o, _ = oracle.forward(q, k, v, sinks, **kw)
    return float(np.sum(o * dout))


@pytest.mark.parametrize("lengths,h_q,h_kv,window", [([7], 2, 1, 0), ([5, 11], 2, 2, 3), ([16], 4, 2, 0)])
def test_central_finite_differences_every_input(lengths, h_q, h_kv, window):
    """Every gradient, including dL/dS_h, against central differences in fp64."""
    rng = np.random.default_rng(13)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    d = 4
    q, k, v, sinks, dout = _rand_problem(rng, int(cu[-1]), h_q, h_kv, d)
    kw = dict(scale=0.7, window=window, cu_seqlens=cu)
    grads = oracle.backward(q, k, v, sinks, dout, **kw)
    h = 1e-6
    for name, arr, g in zip("qkvs", (q, k, v, sinks), grads):
        num = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for idx in range(flat.size):
            save = flat[idx]
            flat[idx] = save + h
            lp = _loss(q, k, v, sinks, dout, **kw)
            flat[idx] = save - h
            lm = _loss(q, k, v, sinks, dout, **kw)
            flat[idx] = save
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=2e-8, err_msg=f"d{name}")


def test_closed_form_single_key():
    """N = 1: the row sees one key, so O_0 = sigmoid(S_00 - S_h) v_0,
    LSE = log(e^S_00 + e^S_h), dL/dS_h = -sigmoid(S_h - S_00) (dO_0 . O_0)."""
    rng = np.random.default_rng(17)
    d = 8
    for _ in range(5):
        q, k, v, sinks, dout = _rand_problem(rng, 1, 1, 1, d, sink_scale=3.0)
        scale = 0.3
        s00 = scale * float(q[0, 0] @ k[0, 0])
        sh = float(sinks[0])
        sig = 1.0 / (1.0 + math.exp(-(s00 - sh)))
        o, lse = oracle.forward(q, k, v, sinks, scale=scale)
        np.testing.assert_allclose(o[0, 0], sig * v[0, 0], rtol=0, atol=1e-14)
        assert abs(lse[0, 0] - (max(s00, sh) + math.log1p(math.exp(-abs(s00 - sh))))) < 1e-13
        dq, dk, dv, ds = oracle.backward(q, k, v, sinks, dout, scale=scale)
        D = float(dout[0, 0] @ o[0, 0])
        assert abs(ds[0] - (-(1.0 - sig) * D)) < 1e-13
        np.testing.assert_allclose(dv[0, 0], sig * dout[0, 0], rtol=0, atol=1e-14)
        dz = sig * (1 - sig) * float(dout[0, 0] @ v[0, 0])
        np.testing.assert_allclose(dq[0, 0], scale * dz * k[0, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(dk[0, 0], scale * dz * q[0, 0], rtol=0, atol=1e-13)


def test_closed_form_equal_logits():
    """q = 0 makes every score 0, so P_ij = 1 / (n + e^S_h) (section "数学公式深入
    解读", equation for P_ij) and O_i is the sum of the visible values times that."""
    rng = np.random.default_rng(19)
    T, h, d = 20, 2, 8
    _, k, v, sinks, _ = _rand_problem(rng, T, h, 1, d)
    q = np.zeros((T, h, d))
    o, lse = oracle.forward(q, k, v, sinks)
    for hh in range(h):
        for i in range(T):
            n = i + 1
            pij = 1.0 / (n + math.exp(sinks[hh]))
            np.testing.assert_allclose(o[i, hh], pij * v[: i + 1, 0].sum(0), rtol=0, atol=1e-13)
            assert abs(lse[hh, i] - math.log(n + math.exp(sinks[hh]))) < 1e-13


def test_sink_to_plus_infinity():
    """A dominant sink takes all the mass: O -> 0 and LSE -> S_h."""
    rng = np.random.default_rng(23)
    q, k, v, _, _ = _rand_problem(rng, 16, 2, 1, 8)
    sinks = np.array([200.0, 300.0])
    o, lse = oracle.forward(q, k, v, sinks)
    assert np.max(np.abs(o)) < 1e-60
    np.testing.assert_allclose(lse, np.repeat(sinks[:, None], 16, 1), rtol=0, atol=1e-12)


def test_window_one_is_diagonal_sigmoid_and_wide_window_is_causal():
    rng = np.random.default_rng(29)
    T, d = 24, 8
    q, k, v, sinks, dout = _rand_problem(rng, T, 2, 1, d)
    o1, _ = oracle.forward(q, k, v, sinks, window=1)
    for h in range(2):
        for i in range(T):
            s = float(q[i, h] @ k[i, 0]) / math.sqrt(d)
            sig = 1.0 / (1.0 + math.exp(-(s - sinks[h])))
            np.testing.assert_allclose(o1[i, h], sig * v[i, 0], rtol=0, atol=1e-14)
    oc, lc = oracle.forward(q, k, v, sinks)
    ow, lw = oracle.forward(q, k, v, sinks, window=T)
    np.testing.assert_array_equal(oc, ow)
    np.testing.assert_array_equal(lc, lw)
    gc = oracle.backward(q, k, v, sinks, dout)
    gw = oracle.backward(q, k, v, sinks, dout, window=T + 5)
    for a, b in zip(gc, gw):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("c", [7.5, -40.0])
def test_adding_a_constant_to_every_logit_of_a_row_changes_only_the_lse(c):
    """Softmax shift invariance at the logit level (section "数学公式深入解读":
    P_ij and P_{i,h} share one denominator): a column c / scale appended to Q
    against a column of ones appended to K adds c to every score, and c is
    added to S_h; then O and P_sink (hence dS_h) are unchanged and LSE grows by
    exactly c."""
    rng = np.random.default_rng(31)
    q, k, v, sinks, dout = _rand_problem(rng, 23, 4, 2, 8)
    cu = np.array([0, 9, 23], np.int32)
    kw = dict(scale=0.3, causal=True, window=0, cu_seqlens=cu)
    o, lse = oracle.forward(q, k, v, sinks, **kw)
    ds = oracle.backward(q, k, v, sinks, dout, **kw)[3]

    def extend(x, value):
        return np.concatenate([x, np.full(x.shape[:2] + (1,), value)], axis=2)

    q2, k2, v2, dout2 = extend(q, c / 0.3), extend(k, 1.0), extend(v, 0.0), extend(dout, 0.0)
    o2, lse2 = oracle.forward(q2, k2, v2, sinks + c, **kw)
    ds2 = oracle.backward(q2, k2, v2, sinks + c, dout2, **kw)[3]
    np.testing.assert_allclose(o2[..., :8], o, rtol=0, atol=1e-12)
    assert np.all(o2[..., 8] == 0)
    np.testing.assert_allclose(lse2, lse + c, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ds2, ds, rtol=0, atol=1e-11)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(31)
    T, h_q, h_kv, d = 19, 6, 2, 8
    g = h_q // h_kv
    q, k, v, sinks, dout = _rand_problem(rng, T, h_q, h_kv, d)
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    o, lse = oracle.forward(q, k, v, sinks, window=4)
    orr, lser = oracle.forward(q, kr, vr, sinks, window=4)
    np.testing.assert_allclose(o, orr, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lser, rtol=0, atol=1e-14)
    dq, dk, dv, ds = oracle.backward(q, k, v, sinks, dout, window=4)
    dqr, dkr, dvr, dsr = oracle.backward(q, kr, vr, sinks, dout, window=4)
    np.testing.assert_allclose(dq, dqr, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dkr.reshape(T, h_kv, g, d).sum(2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dvr.reshape(T, h_kv, g, d).sum(2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(ds, dsr, rtol=0, atol=1e-13)


def test_packed_sequences_are_independent_and_padded_layout_matches():
    rng = np.random.default_rng(37)
    lengths = [5, 1, 13, 8]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, sinks, dout = _rand_problem(rng, T, 2, 1, 8)
    o, lse = oracle.forward(q, k, v, sinks, cu_seqlens=cu)
    dq, dk, dv, ds = oracle.backward(q, k, v, sinks, dout, cu_seqlens=cu)
    ds_sum = np.zeros_like(ds)
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        os_, ls_ = oracle.forward(q[a:b], k[a:b], v[a:b], sinks)
        np.testing.assert_array_equal(o[a:b], os_)
        np.testing.assert_array_equal(lse[:, a:b], ls_)
        g = oracle.backward(q[a:b], k[a:b], v[a:b], sinks, dout[a:b])
        np.testing.assert_array_equal(dq[a:b], g[0])
        np.testing.assert_array_equal(dk[a:b], g[1])
        np.testing.assert_array_equal(dv[a:b], g[2])
        ds_sum += g[3]
    np.testing.assert_allclose(ds, ds_sum, rtol=0, atol=1e-14)
    # padded [B, N, H, d] equals packed with equal lengths
    B, N = 3, 7
    q4, k4, v4, _, do4 = _rand_problem(rng, B * N, 2, 1, 8)
    o4, l4 = oracle.forward(q4.reshape(B, N, 2, 8), k4.reshape(B, N, 1, 8), v4.reshape(B, N, 1, 8), sinks)
    cu4 = np.arange(0, (B + 1) * N, N, dtype=np.int32)
    op, lp = oracle.forward(q4, k4, v4, sinks, cu_seqlens=cu4)
    np.testing.assert_array_equal(o4.reshape(B * N, 2, 8), op)
    np.testing.assert_array_equal(l4, lp)


def test_row_range_gives_exact_rows_and_complete_late_keys():
    rng = np.random.default_rng(41)
    T = 40
    q, k, v, sinks, dout = _rand_problem(rng, T, 4, 2, 8)
    o, lse = oracle.forward(q, k, v, sinks)
    dq, dk, dv, _ = oracle.backward(q, k, v, sinks, dout)
    r0 = 25
    o2, l2 = oracle.forward(q, k, v, sinks, row_begin=r0)
    np.testing.assert_array_equal(o2[r0:], o[r0:])
    np.testing.assert_array_equal(l2[:, r0:], lse[:, r0:])
    assert np.all(o2[:r0] == 0)
    dq2, dk2, dv2, _ = oracle.backward(q, k, v, sinks, dout, row_begin=r0)
    np.testing.assert_allclose(dq2[r0:], dq[r0:], rtol=0, atol=1e-14)
    # keys j >= r0 are seen only by rows >= r0 under the causal mask
    np.testing.assert_allclose(dk2[r0:], dk[r0:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv2[r0:], dv[r0:], rtol=0, atol=1e-14)


def test_hand_worked_example_fixture():
    with open(os.path.join(GOLDEN, "hand_worked_example.json"), encoding="utf-8") as f:
        fx = json.load(f)
    env = {"e": math.e, "log": math.log, "exp": math.exp}
    exp = {key: np.array([eval(expr, {"__builtins__": {}}, env) for expr, _ in vals])
           for key, vals in fx["expected"].items()}
    for key, vals in fx["expected"].items():
        np.testing.assert_allclose(exp[key], [v for _, v in vals], rtol=0, atol=1e-15)
    su = fx["setup"]
    q, k, v, dout = (np.array(su[n]) for n in ("q", "k", "v", "dout"))
    sinks = np.array(su["sinks"])
    o, lse = oracle.forward(q, k, v, sinks, scale=su["scale"])
    dq, dk, dv, ds = oracle.backward(q, k, v, sinks, dout, scale=su["scale"])
    np.testing.assert_allclose(o.reshape(-1), exp["o"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse.reshape(-1), exp["lse"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dq.reshape(-1), exp["dq"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dk.reshape(-1), exp["dk"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dv.reshape(-1), exp["dv"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ds, exp["dsinks"], rtol=0, atol=1e-15)


def test_rejects_invalid_arguments():
    q = np.zeros((4, 2, 8))
    k = np.zeros((4, 1, 8))
    with pytest.raises(ValueError):
        oracle.forward(q, k, k, np.zeros(2), causal=False, window=3)
    with pytest.raises(ValueError):
        oracle.forward(q, k, k, np.zeros(2), cu_seqlens=np.array([0, 3, 2, 4], dtype=np.int32))
    with pytest.raises(ValueError):
        oracle.forward(np.zeros((4, 3, 8)), k[:, :1].repeat(2, 1), k[:, :1].repeat(2, 1), np.zeros(3))


# ----------------------------------------------------------------------------- decode
def _decode_problem(rng, lengths, h_q, h_kv, d, sink_scale=1.0):
    """A shared cache holding every context back to back, one query per context."""
    T = int(sum(lengths)) + 3
    k = rng.standard_normal((T, h_kv, d))
    v = rng.standard_normal((T, h_kv, d))
    q = rng.standard_normal((len(lengths), h_q, d))
    sinks = sink_scale * rng.standard_normal(h_q)
    starts = np.concatenate([[2], 2 + np.cumsum(lengths)[:-1]]).astype(np.int64)
    return q, k, v, sinks, starts, np.asarray(lengths, dtype=np.int64)


@pytest.mark.parametrize("window", [0, 5])
def test_decode_with_sink_at_minus_infinity_is_sdpa_of_one_query(window):
    """S_h -> -inf: the newest token attends like plain softmax attention
    (torch's scaled_dot_product_attention) over its context or window."""
    rng = np.random.default_rng(31)
    q, k, v, _, starts, lens = _decode_problem(rng, [1, 9, 40], 4, 2, 16)
    sinks = np.full(4, -1e30)
    o, lse = oracle.decode(q, k, v, sinks, starts, lens, scale=0.25, window=window)
    for b, (s0, n) in enumerate(zip(starts, lens)):
        lo = max(0, n - window) if window else 0
        kk = torch.tensor(k[s0 + lo:s0 + n]).repeat_interleave(2, dim=1).permute(1, 0, 2)
        vv = torch.tensor(v[s0 + lo:s0 + n]).repeat_interleave(2, dim=1).permute(1, 0, 2)
        qq = torch.tensor(q[b])[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=0.25)[:, 0]
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_decode_window_one_is_a_sigmoid_of_the_newest_key():
    """Window 1: one key j against the sink: O = sigmoid(s - S_h) v_j, and
    LSE = log(exp(s) + exp(S_h))."""
    rng = np.random.default_rng(32)
    q, k, v, sinks, starts, lens = _decode_problem(rng, [5, 12], 2, 1, 8)
    o, lse = oracle.decode(q, k, v, sinks, starts, lens, scale=0.5, window=1)
    for b, (s0, n) in enumerate(zip(starts, lens)):
        j = s0 + n - 1
        for h in range(2):
            s = 0.5 * float(q[b, h] @ k[j, 0])
            sig = 1.0 / (1.0 + math.exp(-(s - sinks[h])))
            np.testing.assert_allclose(o[b, h], sig * v[j, 0], rtol=1e-12, atol=1e-14)
            assert lse[h, b] == pytest.approx(math.log(math.exp(s) + math.exp(sinks[h])), rel=1e-13)


def test_decode_equals_the_row_routine_on_every_prefix():
    """Streaming one sequence token by token gives each row of the training
    forward: checked against the oracle's separate single-row routine
    (combined probabilities over the row's keys and the sink)."""
    rng = np.random.default_rng(33)
    L, h_q, h_kv, d = 24, 4, 2, 8
    q, k, v, sinks, dout = _rand_problem(rng, L, h_q, h_kv, d)
    cu = np.array([0, L], dtype=np.int32)
    for window in (0, 6):
        o, lse = oracle.decode(q, k, v, sinks, np.zeros(L, np.int64), np.arange(1, L + 1),
                               scale=0.3, window=window)
        for i in range(L):
            for h in range(h_q):
                first, p, _ = oracle.row(q, k, v, sinks, seq=0, head=h, i=i, scale=0.3, causal=True,
                                         window=window, cu_seqlens=cu)
                keys = np.arange(first, first + len(p) - 1)
                np.testing.assert_allclose(o[i, h], p[:-1] @ v[keys, h // 2], rtol=1e-12, atol=1e-14)
                # LSE from the sink's probability: P_sink = exp(S_h - LSE)
                assert lse[h, i] == pytest.approx(sinks[h] - math.log(p[-1]), rel=1e-12, abs=1e-12)
