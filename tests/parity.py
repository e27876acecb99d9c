"""Helpers for GPU-vs-oracle parity tests.

Tolerances. The workloads state: bf16 inputs with fp32 accumulation reach
max-abs error <= 2e-2 and relative L2 error <= 1e-2 on O, dQ, dK, dV and dS_h;
fp32 inputs reach max-abs error <= 1e-4. The reference is the fp64 oracle on
the exact fp64 widening of the inputs the GPU received.

One reading is applied to the max-abs bound: a value stored in bf16 cannot sit
closer to the exact value than its own rounding (one ulp of a value in
[8, 16) is 0.0625), so for tensors stored in the input dtype (O, dQ, dK, dV)
the bound is |gpu - ref| <= max_abs + fmt |ref|, with fmt = 2^-8 for bf16
(one bf16 ulp of ref is at most 2^-8 |ref|) and 2^-22 for fp32. dS_h and LSE
are fp32 outputs and get no such term. The relative L2 bound applies
unchanged. LSE (fp32, not named in the stated bounds) is held to the bounds of
O.

The bf16 path under test is the extended one (sink_attn_fwd_ex /
sink_attn_bwd_ex): the forward also returns o_lo, the part of O that its bf16
rounding dropped, and the backward forms D = dO . (o + o_lo), so no term for
the stored O's rounding is needed anywhere.
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


def assert_close(name, got, ref, dtype, report=None, rounds_output=True):
    """Checks got against ref element by element: max-abs bound (plus one
    output-format ulp for tensors stored in the input dtype, ``rounds_output``)
    and relative L2 bound."""
    tol = TOL[dtype]
    g, r = _np(got), _np(ref)
    ma, rel = errors(g, r)
    bound = np.full(r.shape, tol["max_abs"])
    if rounds_output:
        bound = bound + tol["fmt"] * np.abs(r)
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


def gpu_fwd_bwd(q, k, v, sinks, dout, cu_seqlens=None, **kw):
    """Forward + backward through the C ABI on the given device tensors: the
    extended entry points for bf16 (o_lo kept between them), the plain ones
    for fp32. Returns (o, lse, dq, dk, dv, dsinks)."""
    import attention_sink_softmax_gb300 as sa
    if q.dtype == torch.bfloat16:
        o, o_lo, lse = sa.sink_attn_fwd_ex(q, k, v, sinks, cu_seqlens, **kw)
        dq, dk, dv, ds = sa.sink_attn_bwd_ex(q, k, v, sinks, o, o_lo, lse, dout, cu_seqlens, **kw)
    else:
        o, lse = sa.sink_attn_fwd(q, k, v, sinks, cu_seqlens, **kw)
        dq, dk, dv, ds = sa.sink_attn_bwd(q, k, v, sinks, o, lse, dout, cu_seqlens, **kw)
    return o, lse, dq, dk, dv, ds
