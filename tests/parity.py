"""Helpers for GPU-vs-oracle parity tests.

Tolerances. The workloads state: bf16 inputs with fp32 accumulation reach
max-abs error <= 2e-2 and relative L2 error <= 1e-2 on O, dQ, dK, dV and dS_h;
fp32 inputs reach max-abs error <= 1e-4. The reference is the fp64 oracle on
the exact fp64 widening of the inputs the GPU received.

A bf16 output cannot sit closer to the exact value than its own rounding (one
ulp of a value in [8, 16) is 0.0625), so the max-abs bound is applied to the
error beyond the output format's rounding:
  - bf16 tensors (O, dQ, dK, dV):  |gpu - ref| <= 2e-2 + 2^-8 |ref|
    (2^-8 |ref| bounds one bf16 ulp of ref);
  - dS_h (fp32) is computed from the stored bf16 O through D_i = dO_i . O_i,
    so the rounding of O propagates:  |gpu - ref| <= 2e-2 + 2^-8 sum_i
    P_sink,i sum_c |dO_ic O_ic|  (2^-9 bounds bf16 rounding of each O_ic; the
    extra factor 2 covers fp32 accumulation).
  - dQ and dK likewise see the rounding of O through D: dS_ij = P_ij (dP_ij -
    D_i), so with |dD_i| <= delta_i = 2^-8 sum_c |dO_ic O_ic|:
      |dQ_ic error| <= scale delta_i sum_j P_ij |k_jc|
      |dK_jc error| <= scale sum_(h,i) P_ij delta_i |q_ic|
    Both sums are attention-shaped and come from the oracle itself:
    sum_j P_ij |k_jc| is the forward output with V := |K|, and
    sum_i P_ij x_i is the dV output of the backward with dout := x.
    When attention is sharp (large logits) dP_ij - D_i cancels and this term
    dominates; for diffuse attention it is negligible and tests may skip it
    (which only makes them stricter).
For fp32 inputs the same forms are used with 2^-22 in place of 2^-8. The
relative L2 bound applies unchanged. LSE (fp32, not named in the stated
bounds) is held to the bounds of O.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {
    torch.bfloat16: dict(max_abs=2e-2, rel_l2=1e-2, fmt=2.0 ** -8),
    torch.float32: dict(max_abs=1e-4, rel_l2=1e-4, fmt=2.0 ** -22),
}


def _np(x):
    if torch.is_tensor(x):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    got, ref = _np(got), _np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if not np.all(np.isfinite(got)):
        return float("inf"), float("inf")
    err = np.abs(got - ref)
    denom = np.linalg.norm(ref.reshape(-1))
    rel = float(np.linalg.norm(err.reshape(-1)) / denom) if denom > 0 else float(np.linalg.norm(err))
    return (float(err.max()) if err.size else 0.0), rel


def assert_close(name, got, ref, dtype, report=None, allowance=None, rounds_output=True):
    """Checks got against ref; ``allowance`` (broadcastable to ref) is extra
    absolute slack for propagated input-format rounding; bf16/fp32 tensor
    outputs also get one output-format ulp (``rounds_output``)."""
    tol = TOL[dtype]
    g, r = _np(got), _np(ref)
    ma, rel = errors(g, r)
    bound = np.full(r.shape, tol["max_abs"])
    if rounds_output:
        bound = bound + tol["fmt"] * np.abs(r)
    if allowance is not None:
        bound = bound + np.asarray(allowance, dtype=np.float64)
    excess = np.abs(g - r) - bound if r.size else np.zeros(0)
    worst = int(np.argmax(excess)) if r.size else 0
    if report is not None:
        report[name] = dict(max_abs=ma, rel_l2=rel,
                            max_abs_beyond_rounding=float(np.max(np.abs(g - r) - (bound - tol["max_abs"])))
                            if r.size else 0.0)
    if r.size:
        assert excess.reshape(-1)[worst] <= 0, (
            f"{name}: |err| {np.abs(g - r).reshape(-1)[worst]:.3e} at |ref| "
            f"{np.abs(r).reshape(-1)[worst]:.3e} exceeds {bound.reshape(-1)[worst]:.3e} "
            f"(max-abs {ma:.3e}, rel-L2 {rel:.3e})")
    assert rel <= tol["rel_l2"], f"{name}: relative L2 error {rel:.3e} > {tol['rel_l2']}"


def dsink_allowance(o_ref, lse_ref, dout, sinks, dtype):
    """Per head: fmt * sum_t P_sink(h, t) * sum_c |dO_tc O_tc| over packed rows.

    o_ref, dout [T, H, d]; lse_ref [H, T]; sinks [H]."""
    o = _np(o_ref)
    do = _np(dout).reshape(o.shape)
    lse = _np(lse_ref)
    s = _np(sinks)
    mag = np.einsum("thd->ht", np.abs(do * o))
    psink = np.exp(s[:, None] - lse)
    return TOL[dtype]["fmt"] * np.sum(psink * mag, axis=1)


def assert_dsinks_close(name, got, ref, dtype, o_ref, lse_ref, dout, sinks, report=None,
                        extra_allowance=None):
    allow = dsink_allowance(o_ref, lse_ref, dout, sinks, dtype)
    if extra_allowance is not None:
        allow = allow + extra_allowance
    assert_close(name, got, ref, dtype, report, allowance=allow, rounds_output=False)


def oracle_fwd_bwd(q, k, v, sinks, dout, *, scale, causal, window, cu_seqlens=None,
                   row_begin=0, row_end=1 << 30, backward=True):
    """Oracle on CPU copies (exact fp64 widening) of the given tensors."""
    cu = cu_seqlens.cpu().numpy() if cu_seqlens is not None else None
    kw = dict(scale=scale, causal=causal, window=window, cu_seqlens=cu,
              row_begin=row_begin, row_end=row_end)
    o, lse = oracle.forward(q.cpu(), k.cpu(), v.cpu(), sinks.cpu(), **kw)
    if not backward:
        return o, lse
    dq, dk, dv, ds = oracle.backward(q.cpu(), k.cpu(), v.cpu(), sinks.cpu(), dout.cpu(), **kw)
    return o, lse, dq, dk, dv, ds


def d_rounding_allowances(q, k, v, sinks, dout, o_ref, *, scale, causal, window, dtype,
                          cu_seqlens=None, row_begin=0, row_end=1 << 30):
    """(allow_dq, allow_dk) for the rounding of the stored O propagated through D.

    q/dout/o_ref share a layout ([T, H_q, d] or [B, N, H_q, d]); k/v likewise
    with H_kv heads. Rows outside [row_begin, row_end) contribute nothing.
    """
    fmt = TOL[dtype]["fmt"]
    qn, kn = _np(q), _np(k)
    delta = fmt * np.sum(np.abs(_np(dout) * _np(o_ref)), axis=-1, keepdims=True)
    cu = cu_seqlens.cpu().numpy() if torch.is_tensor(cu_seqlens) else cu_seqlens
    kw = dict(scale=scale, causal=causal, window=window, cu_seqlens=cu,
              row_begin=row_begin, row_end=row_end)
    pk, _ = oracle.forward(qn, kn, np.abs(kn), _np(sinks), **kw)
    allow_dq = scale * delta * pk
    _, _, pq, _ = oracle.backward(qn, kn, _np(v), _np(sinks), delta * np.abs(qn), **kw)
    allow_dk = scale * pq
    return allow_dq, allow_dk
