"""fp64 CPU oracle for softmax attention with one learnable sink logit per head.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package. It shares no code with the CUDA library ``attention_sink_softmax_gb300``
and neither imports the other.

The arithmetic lives in ``sink_oracle.c`` (plain C, fp64, OpenMP over
independent units); this module only compiles it with gcc and marshals numpy
arrays. Every function follows the page "惊爆！GPT-OSS-20B强化学习，训练速度
狂飙、超稳定！" (nmedialink.com): the forward from sections "GPT-OSS中的带注意力
槽的注意力机制" and "数学公式深入解读", the backward from section "反向传播的实现".

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sink_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsink_oracle.so")
_lock = threading.Lock()
_lib = None

_DP = ctypes.POINTER(ctypes.c_double)
_IP = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile ``sink_oracle.c`` into ``oracle/_build/libsink_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                           os.path.getmtime(os.path.join(_HERE, "sink_oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            common = [ctypes.c_int, _IP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_double, ctypes.c_int, ctypes.c_int]
            lib.sink_oracle_forward.argtypes = common + [ctypes.c_int, ctypes.c_int] + [_DP] * 6
            lib.sink_oracle_forward.restype = ctypes.c_int
            lib.sink_oracle_backward.argtypes = common + [ctypes.c_int, ctypes.c_int] + [_DP] * 9
            lib.sink_oracle_backward.restype = ctypes.c_int
            lib.sink_oracle_row.argtypes = common + [_DP] * 5 + [ctypes.c_int] * 3 + [
                _DP, _DP, ctypes.POINTER(ctypes.c_int)]
            lib.sink_oracle_row.restype = ctypes.c_int
            lib.sink_oracle_num_threads.argtypes = []
            lib.sink_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """Exact conversion to a contiguous fp64 numpy array (bf16/fp32 widen exactly)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_DP)


def _shape(q, k, cu_seqlens):
    """Returns (q, k viewed as [T, H, d], cu_seqlens) for padded [B,N,H,d] or packed [T,H,d] input."""
    if q.ndim == 4:
        B, N = q.shape[0], q.shape[1]
        if cu_seqlens is None:
            cu_seqlens = np.arange(0, (B + 1) * N, N, dtype=np.int32)
        q = q.reshape(B * N, q.shape[2], q.shape[3])
        k = k.reshape(B * N, k.shape[2], k.shape[3])
    elif cu_seqlens is None:
        cu_seqlens = np.array([0, q.shape[0]], dtype=np.int32)
    return q, k, _i32(cu_seqlens)


def num_threads() -> int:
    return _load().sink_oracle_num_threads()


def forward(q, k, v, sinks, *, scale=None, causal=True, window=0, cu_seqlens=None,
            row_begin=0, row_end=1 << 30):
    """O and LSE of sink attention in fp64.

    q [B,N,H_q,d] or [T,H_q,d]; k, v with H_kv heads; sinks [H_q].
    Returns (o with q's shape, lse [H_q, T]).
    """
    qs = q.shape
    q, k, v, sinks = _f64(q), _f64(k), _f64(v), _f64(sinks)
    q, k, cu = _shape(q, k, cu_seqlens)
    v = v.reshape(k.shape)
    T, h_q, d = q.shape
    h_kv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((T, h_q, d), dtype=np.float64)
    lse = np.zeros((h_q, T), dtype=np.float64)
    rc = _load().sink_oracle_forward(len(cu) - 1, cu.ctypes.data_as(_IP), h_q, h_kv, d,
                                     float(scale), int(causal), int(window),
                                     int(row_begin), int(row_end),
                                     _p(q), _p(k), _p(v), _p(sinks), _p(o), _p(lse))
    if rc != 0:
        raise ValueError("sink_oracle_forward: invalid argument")
    return o.reshape(qs), lse


def backward(q, k, v, sinks, dout, *, scale=None, causal=True, window=0, cu_seqlens=None,
             row_begin=0, row_end=1 << 30):
    """dQ, dK, dV, dS_h of sink attention for the loss L = sum(O * dout), in fp64."""
    qs, ks = q.shape, k.shape
    q, k, v, sinks, dout = _f64(q), _f64(k), _f64(v), _f64(sinks), _f64(dout)
    q, k, cu = _shape(q, k, cu_seqlens)
    v = v.reshape(k.shape)
    dout = dout.reshape(q.shape)
    T, h_q, d = q.shape
    h_kv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dsinks = np.zeros(h_q, dtype=np.float64)
    rc = _load().sink_oracle_backward(len(cu) - 1, cu.ctypes.data_as(_IP), h_q, h_kv, d,
                                      float(scale), int(causal), int(window),
                                      int(row_begin), int(row_end),
                                      _p(q), _p(k), _p(v), _p(sinks), _p(dout),
                                      _p(dq), _p(dk), _p(dv), _p(dsinks))
    if rc != 0:
        raise ValueError("sink_oracle_backward: invalid argument")
    return dq.reshape(qs), dk.reshape(ks), dv.reshape(ks), dsinks


def row(q, k, v, sinks, *, seq, head, i, dout=None, scale=None, causal=True, window=0,
        cu_seqlens=None):
    """One row in full: (first_key, p, dz).

    p = combined probabilities over the row's allowed keys followed by the sink
    (so p[-1] is P_{i,h}); dz = gradient of L = sum(O * dout) with respect to the
    combined score row (dz[-1] is the row's term of dL/dS_h), or None without dout.
    """
    q, k, v, sinks = _f64(q), _f64(k), _f64(v), _f64(sinks)
    q, k, cu = _shape(q, k, cu_seqlens)
    v = v.reshape(k.shape)
    T, h_q, d = q.shape
    h_kv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    Lmax = int(np.max(np.diff(cu))) if len(cu) > 1 else 0
    p = np.zeros(Lmax + 1, dtype=np.float64)
    dz = np.zeros(Lmax + 1, dtype=np.float64)
    if dout is not None:
        dout = _f64(dout).reshape(q.shape)
    first = ctypes.c_int(0)
    n = _load().sink_oracle_row(len(cu) - 1, cu.ctypes.data_as(_IP), h_q, h_kv, d,
                                float(scale), int(causal), int(window),
                                _p(q), _p(k), _p(v), _p(sinks),
                                _p(dout) if dout is not None else None,
                                int(seq), int(head), int(i), _p(p), _p(dz), ctypes.byref(first))
    if n < 0:
        raise ValueError("sink_oracle_row: invalid argument")
    return first.value, p[: n + 1].copy(), (dz[: n + 1].copy() if dout is not None else None)


def decode(q, k_cache, v_cache, sinks, kv_start, kv_len, *, scale=None, window=0):
    """Decode oracle: query b (q [B, H_q, d]) is the last token of the context
    k_cache / v_cache [kv_start[b] : kv_start[b] + kv_len[b]] ([T, H_kv, d]);
    returns (o [B, H_q, d], lse [H_q, B]) in fp64.

    No arithmetic of its own: for each query it evaluates row kv_len[b] - 1 of
    the forward above on that context (the query placed in that row), which is
    what a streaming decoder computes for the newest token.
    """
    q, k_cache, v_cache, sinks = _f64(q), _f64(k_cache), _f64(v_cache), _f64(sinks)
    B, h_q, d = q.shape
    h_kv = k_cache.shape[1]
    o = np.zeros((B, h_q, d), dtype=np.float64)
    lse = np.zeros((h_q, B), dtype=np.float64)
    starts = np.asarray(kv_start, dtype=np.int64).reshape(-1)
    lens = np.asarray(kv_len, dtype=np.int64).reshape(-1)
    for b in range(B):
        s0, n = int(starts[b]), int(lens[b])
        if n < 1 or s0 < 0 or s0 + n > k_cache.shape[0]:
            raise ValueError("decode: context outside the cache")
        qq = np.zeros((n, h_q, d), dtype=np.float64)
        qq[n - 1] = q[b]
        ob, lb = forward(qq, k_cache[s0:s0 + n], v_cache[s0:s0 + n], sinks, scale=scale, causal=True,
                         window=window, cu_seqlens=np.array([0, n], dtype=np.int32),
                         row_begin=n - 1, row_end=n)
        o[b] = ob[n - 1]
        lse[:, b] = lb[:, n - 1]
    return o, lse
