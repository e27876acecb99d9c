"""Host-side checks of libsinkattn that need no GPU: the library loads, exports
every entry point include/*.h declares, and rejects invalid arguments before
touching the device."""
import ctypes
import glob
import os
import re

import pytest

import attention_sink_softmax_gb300 as sa
from attention_sink_softmax_gb300 import _abi
from attention_sink_softmax_gb300 import build as sa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    sa_build.build()
    return _abi.lib()


def _declared_functions():
    names = []
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"SINK_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert set(_abi.EXPORTS) | set(_abi.TESTING_EXPORTS) == set(declared)
    assert len(declared) >= 8
    for name in declared:
        assert hasattr(L, name), f"libsinkattn does not export {name}"


def test_status_strings_and_version(L):
    assert sa.sink_attn_status_str(0) == "ok"
    for st in range(7):
        assert isinstance(sa.sink_attn_status_str(st), str)
    assert sa.sink_attn_status_str(99) == "unknown status"
    assert sa.sink_attn_version() >= 200


def _params(**kw):
    p = _abi.SinkAttnParams()
    base = dict(batch=2, max_seqlen=8192, total_tokens=16384, h_q=64, h_kv=8, head_dim=64,
                dtype=_abi.SINK_BF16, softmax_scale=0.125, causal=1, window=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


def test_workspace_sizes(L):
    p = _params()
    fwd = sa.sink_attn_workspace_bytes(p, False)
    bwd = sa.sink_attn_workspace_bytes(p, True)
    assert fwd >= 256 and fwd % 256 == 0
    # the backward holds at least delta [h_q, T] fp32
    assert bwd >= 256 + 4 * 64 * 16384
    assert sa.sink_attn_workspace_bytes(_params(h_q=63), True) == 0
    assert sa.sink_attn_workspace_bytes(_params(head_dim=96), True) == 0
    # head_dim 128: delta and the dS_h partials, no fp32 dQ accumulator (CUDA-core backward)
    d128 = sa.sink_attn_workspace_bytes(_params(head_dim=128), True)
    assert 256 + 4 * 64 * 16384 <= d128 < bwd


@pytest.mark.parametrize("kw,status", [
    (dict(h_q=63), _abi.SINK_ERR_INVALID_ARG),          # h_q not a multiple of h_kv
    (dict(causal=0, window=128), _abi.SINK_ERR_INVALID_ARG),
    (dict(head_dim=96), _abi.SINK_ERR_UNSUPPORTED),
    (dict(head_dim=32), _abi.SINK_ERR_UNSUPPORTED),
    (dict(dtype=7), _abi.SINK_ERR_INVALID_ARG),
    (dict(total_tokens=100), _abi.SINK_ERR_INVALID_ARG),  # padded: T != B * N
    (dict(batch=-1), _abi.SINK_ERR_INVALID_ARG),
    (dict(causal=2), _abi.SINK_ERR_INVALID_ARG),
])
def test_invalid_params_rejected_before_launch(L, kw, status):
    p = _params(**kw)
    nul = ctypes.c_void_p(0)
    st = L.sink_attn_fwd(ctypes.byref(p), *([nul] * 7), nul, 0, nul)
    assert st == status
    st = L.sink_attn_bwd(ctypes.byref(p), *([nul] * 12), nul, 0, nul)
    assert st == status


def test_missing_workspace_rejected(L):
    p = _params()
    nul = ctypes.c_void_p(0)
    assert L.sink_attn_fwd(ctypes.byref(p), *([nul] * 7), nul, 0, nul) == _abi.SINK_ERR_WORKSPACE
    assert L.sink_attn_bwd(ctypes.byref(p), *([nul] * 12), nul, 0, nul) == _abi.SINK_ERR_WORKSPACE
    assert L.sink_attn_fetch_device_error(nul, 0, nul, None) == _abi.SINK_ERR_WORKSPACE


def test_split_preparation_entry_points_validate(L):
    """sink_attn_bwd_prepare / sink_attn_bwd_main_ex: unknown option bits and
    a missing workspace are rejected before anything touches the device."""
    p = _params()
    nul = ctypes.c_void_p(0)
    assert L.sink_attn_bwd_main_ex(ctypes.byref(p), *([nul] * 10), nul, 0, 2, nul) == \
        _abi.SINK_ERR_INVALID_ARG
    assert L.sink_attn_bwd_main_ex(ctypes.byref(p), *([nul] * 10), nul, 0,
                                   _abi.SINK_BWD_PREPARED, nul) == _abi.SINK_ERR_WORKSPACE
    assert L.sink_attn_bwd_prepare(ctypes.byref(p), nul, nul, nul, 0, nul) == _abi.SINK_ERR_WORKSPACE
    bad = _params(h_kv=3)  # 64 query heads do not group over 3
    assert L.sink_attn_bwd_prepare(ctypes.byref(bad), nul, nul, nul, 0, nul) == \
        _abi.SINK_ERR_INVALID_ARG


def test_host_memory_workspace_rejected(L):
    """A host buffer is never handed to a kernel: the call fails up front."""
    p = _params()
    buf = ctypes.create_string_buffer(1 << 20)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    nul = ctypes.c_void_p(0)
    st = L.sink_attn_fwd(ctypes.byref(p), *([nul] * 7), ctypes.c_void_p(addr), 1 << 19, nul)
    assert st == _abi.SINK_ERR_WORKSPACE


def test_python_layer_rejects_cpu_tensors(L):
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sa.sink_attn_fwd(q, k, k, torch.zeros(2))


def test_decode_workspace_and_validation(L):
    p = _params(batch=8, max_seqlen=32768, total_tokens=262144)
    need = sa.sink_attn_decode_workspace_bytes(p)
    # header + a chunk counter per (query, key/value head) + 64 chunks x 8
    # queries x 64 heads x (m, l, o[64]) fp32
    assert need >= 256 + 4 * 8 * 8 + 4 * 64 * 8 * 64 * 66 and need % 256 == 0
    assert sa.sink_attn_decode_workspace_bytes(_params(causal=0)) == 0
    assert sa.sink_attn_decode_workspace_bytes(_params(head_dim=128)) == 0
    nul = ctypes.c_void_p(0)
    assert L.sink_attn_decode(ctypes.byref(_params(causal=0)), *([nul] * 8), nul, 0, nul) == \
        _abi.SINK_ERR_INVALID_ARG
    assert L.sink_attn_decode(ctypes.byref(p), *([nul] * 8), nul, 0, nul) == _abi.SINK_ERR_WORKSPACE


def test_wait_limit_setter_round_trip(L):
    prev = sa.sink_attn_set_wait_limit_ns(5_000_000)
    try:
        assert prev == 2_000_000_000
        assert sa.sink_attn_set_wait_limit_ns(0) == 5_000_000
        assert sa.sink_attn_set_wait_limit_ns(0) == 2_000_000_000
    finally:
        sa.sink_attn_set_wait_limit_ns(0)


def test_flag_bits_match_the_header(L):
    text = open(os.path.join(ROOT, "include", "sink_attn.h"), encoding="utf-8").read()
    for name in ("SINK_FLAG_TIMEOUT", "SINK_FLAG_SEQ_TOO_LONG", "SINK_FLAG_BAD_SEQLENS",
                 "SINK_BWD_PREPARED"):
        m = re.search(rf"#define {name} (\d+)u", text)
        assert m and int(m.group(1)) == getattr(_abi, name)
