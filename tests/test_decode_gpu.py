"""GPU parity of sink_attn_decode (one query per entry against a key/value
cache, split over keys, merged with the sink counted once) against the fp64
oracle, and the training-versus-inference consistency check: streaming a
sequence token by token through the decode path must reproduce the training
forward's per-token log-normaliser and output (the page's Fig. 4 diagnostic,
section "纠正训练与推理不一致问题", restated as a kernel-consistency test).

All calls go through the C ABI (via the ctypes binding)."""
import numpy as np
import pytest
import torch

import attention_sink_softmax_gb300 as sa
import oracle
from attention_sink_softmax_gb300 import _abi, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _problem(seed, lengths, h_q, h_kv, dtype, sink_scale=2.0, gap=3):
    """A shared cache with every context back to back (and a few rows between
    them), one query per context."""
    g = torch.Generator().manual_seed(seed)
    T = int(sum(lengths)) + gap * (len(lengths) + 1)
    k = torch.randn(T, h_kv, 64, generator=g).to(dtype)
    v = torch.randn(T, h_kv, 64, generator=g).to(dtype)
    q = torch.randn(len(lengths), h_q, 64, generator=g).to(dtype)
    sinks = (sink_scale * torch.randn(h_q, generator=g)).float()
    starts, s = [], gap
    for n in lengths:
        starts.append(s)
        s += n + gap
    return q, k, v, sinks, torch.tensor(starts, dtype=torch.int32), torch.tensor(lengths, dtype=torch.int32)


def _run(q, k, v, sinks, starts, lens, window, scale=None):
    d = [t.to(DEV) for t in (q, k, v, sinks, starts, lens)]
    o, lse = sa.sink_attn_decode(*d, window=window, softmax_scale=scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


CASES = [
    # lengths, h_q, h_kv
    ([1, 7, 129, 300, 1000], 8, 2),
    ([2048, 33], 8, 1),       # MQA-like group of 8
    ([513, 64], 16, 1),       # group of 16: two query heads per warp
    ([100, 257], 4, 4),       # MHA
    ([300, 77], 32, 1),       # group of 32: the CUDA-core kernel for bf16 too
    ([77, 1500], 12, 1),      # group of 12: two 8-head blocks, four of them padding
    ([250, 3], 6, 2),         # group of 3
    ([700, 5, 2100], 64, 8),  # the served model's 64 / 8 heads, ragged contexts
    ([333, 90], 10, 5),       # 5 key/value heads (5 warps), group of 2
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("window", [0, 128])
@pytest.mark.parametrize("lengths,h_q,h_kv", CASES)
def test_decode_parity(dtype, window, lengths, h_q, h_kv):
    q, k, v, sinks, starts, lens = _problem(7, lengths, h_q, h_kv, dtype)
    o, lse = _run(q, k, v, sinks, starts, lens, window)
    o_ref, lse_ref = oracle.decode(q, k, v, sinks, starts.numpy(), lens.numpy(), scale=0.125,
                                   window=window)
    assert_close("decode O", o, o_ref, dtype)
    assert_close("decode LSE", lse, lse_ref, dtype, rounds_output=False)


@pytest.mark.parametrize("window", [0, 100])
def test_decode_reads_nothing_outside_the_context(window):
    """Every cache row outside the contexts holds NaN, and the last context
    ends at the cache's last row (its final 32-key box runs past the cache):
    the result must match the oracle computed on the clean cache."""
    q, k, v, sinks, starts, lens = _problem(11, [45, 1000, 33], 8, 2, torch.bfloat16, gap=1)
    lens[-1] = k.shape[0] - int(starts[-1])  # the last context runs to the end of the cache
    o_ref, lse_ref = oracle.decode(q, k, v, sinks, starts.numpy(), lens.numpy(), scale=0.125,
                                   window=window)
    inside = torch.zeros(k.shape[0], dtype=torch.bool)
    for st, n in zip(starts.tolist(), lens.tolist()):
        inside[st:st + n] = True
    assert not inside.all()
    k_bad, v_bad = k.clone(), v.clone()
    k_bad[~inside] = float("nan")
    v_bad[~inside] = float("nan")
    o, lse = _run(q, k_bad, v_bad, sinks, starts, lens, window)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert_close("decode O (NaN outside the contexts)", o, o_ref, torch.bfloat16)
    assert_close("decode LSE (NaN outside the contexts)", lse, lse_ref, torch.bfloat16,
                 rounds_output=False)


def test_decode_full_size_sampled_queries():
    """The benchmarked shape: 8 queries, 32768-token contexts, 64/8 heads, bf16;
    every query's output checked against the oracle for two of the queries."""
    w = inputs.decode_workload()
    prob = inputs.make_decode_inputs(w)
    o, lse = _run(prob["q"], prob["k"], prob["v"], prob["sinks"], prob["kv_start"], prob["kv_len"],
                  w.window, w.scale)
    pick = [0, w.batch - 1]
    o_ref, lse_ref = oracle.decode(prob["q"][pick], prob["k"], prob["v"], prob["sinks"],
                                   prob["kv_start"][pick].numpy(), prob["kv_len"][pick].numpy(),
                                   scale=w.scale, window=w.window)
    assert_close("decode O (full size)", o[pick], o_ref, torch.bfloat16)
    assert_close("decode LSE (full size)", lse[:, pick], lse_ref, torch.bfloat16, rounds_output=False)


@pytest.mark.parametrize("window", [0, 128])
def test_training_and_inference_paths_agree_token_by_token(window):
    """One 1000-token sequence: the training forward (tensor cores, all rows at
    once) and the decode path (each token against its own prefix) give the same
    per-token sink log-probability log P_sink = S_h - LSE (the log-probability
    mass the page's sink takes) to 2e-3, and outputs that each meet the
    oracle's tolerance. The outputs differ from each other by the two paths'
    own roundings (the training path multiplies V by P rounded to bf16, the
    decode path by fp32 P; both round O to bf16, each about 2.5e-3 relative
    L2 from the exact result), so their gap is held to the sum, 5e-3."""
    L, h_q, h_kv = 1000, 8, 2
    g = torch.Generator().manual_seed(5)
    q = torch.randn(L, h_q, 64, generator=g).bfloat16()
    k = torch.randn(L, h_kv, 64, generator=g).bfloat16()
    v = torch.randn(L, h_kv, 64, generator=g).bfloat16()
    sinks = (2.0 * torch.randn(h_q, generator=g)).float()
    cu = torch.tensor([0, L], dtype=torch.int32)
    qd, kd, vd, sd, cud = (t.to(DEV) for t in (q, k, v, sinks, cu))
    o_tr, lse_tr = sa.sink_attn_fwd(qd, kd, vd, sd, cud, max_seqlen=L, window=window)
    starts = torch.zeros(L, dtype=torch.int32, device=DEV)
    lens = torch.arange(1, L + 1, dtype=torch.int32, device=DEV)
    o_inf, lse_inf = sa.sink_attn_decode(qd, kd, vd, sd, starts, lens, max_seqlen=L, window=window)
    torch.cuda.synchronize()
    logp_tr = (sd[:, None] - lse_tr).cpu().double()
    logp_inf = (sd[:, None] - lse_inf).cpu().double()
    gap = (logp_tr - logp_inf).abs()
    assert float(gap.max()) <= 2e-3, f"max |log P_sink gap| {float(gap.max()):.3e}"
    rel = float((o_tr.float() - o_inf.float()).norm() / o_tr.float().norm())
    assert rel <= 5e-3, f"output rel-L2 gap {rel:.3e}"
    # both against the oracle
    o_ref, lse_ref = oracle.forward(q, k, v, sinks, scale=0.125, window=window,
                                    cu_seqlens=np.array([0, L], dtype=np.int32))
    assert_close("train O", o_tr.cpu(), o_ref, torch.bfloat16)
    assert_close("infer O", o_inf.cpu(), o_ref, torch.bfloat16)
    assert_close("infer LSE", lse_inf.cpu(), lse_ref, torch.bfloat16, rounds_output=False)
    print({"window": window, "max_logp_sink_gap": float(gap.max()), "mean_logp_sink_gap": float(gap.mean()),
           "o_rel_gap": rel})


def test_invalid_context_flags_and_yields_the_empty_row():
    """A context longer than max_seqlen (or past the cache) reads no key: o = 0,
    lse = S_h, and the flag word reports SINK_ERR_DEVICE."""
    q, k, v, sinks, starts, lens = _problem(9, [10, 20], 4, 1, torch.bfloat16)
    lens_bad = lens.clone()
    lens_bad[1] = 40  # > max_seqlen below, and past the next context
    d = [t.to(DEV) for t in (q, k, v, sinks, starts, lens_bad)]
    p = sa.make_decode_params(d[0], d[1], max_seqlen=20)
    ws = torch.empty(sa.sink_attn_decode_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    o, lse = sa.sink_attn_decode(*d, params=p, workspace=ws)
    st, flags = sa.sink_attn_fetch_device_error(ws)
    assert st == _abi.SINK_ERR_DEVICE and flags != 0
    assert torch.all(o[1].float() == 0)
    np.testing.assert_allclose(lse[:, 1].cpu().numpy(), sinks.numpy(), rtol=1e-6)
    o_ref, lse_ref = oracle.decode(q[:1], k, v, sinks, starts[:1].numpy(), lens[:1].numpy(), scale=0.125)
    assert_close("decode O (valid query)", o[:1].cpu(), o_ref, torch.bfloat16)


def test_decode_rejects_host_pointers():
    q, k, v, sinks, starts, lens = _problem(3, [5], 4, 1, torch.bfloat16)
    d = [t.to(DEV) for t in (q, k, v, sinks)]
    with pytest.raises(ValueError):
        sa.sink_attn_decode(*d, starts, lens.to(DEV))  # kv_start left on the host


def test_decode_under_cuda_graph_capture_matches_eager():
    """The C-ABI call only enqueues work on the caller's stream, so a run of
    decode calls captured into a CUDA graph and replayed gives the eager
    result bit for bit."""
    q, k, v, sinks, starts, lens = _problem(13, [700, 64, 2000], 16, 2, torch.bfloat16)
    d = [t.to(DEV) for t in (q, k, v, sinks, starts, lens)]
    p = sa.make_decode_params(d[0], d[1], max_seqlen=2000)
    ws = torch.empty(sa.sink_attn_decode_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    o_e, lse_e = sa.sink_attn_decode(*d, params=p, workspace=ws)
    torch.cuda.synchronize()
    o_g, lse_g = torch.empty_like(o_e), torch.empty_like(lse_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        sa.sink_attn_decode(*d, params=p, out=o_g, lse=lse_g, workspace=ws,
                            stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e)
    assert sa.sink_attn_fetch_device_error(ws)[0] == _abi.SINK_OK


def test_decode_empty_batch_and_empty_cache():
    """No query: nothing is enqueued and the call succeeds. An empty cache:
    every context is invalid, so every query gets the empty row (o = 0,
    lse = S_h) and the flag word reports it."""
    sinks = torch.randn(8).float().to(DEV)
    k = torch.randn(10, 2, 64).bfloat16().to(DEV)
    q0 = torch.empty(0, 8, 64, dtype=torch.bfloat16, device=DEV)
    z = torch.empty(0, dtype=torch.int32, device=DEV)
    o, lse = sa.sink_attn_decode(q0, k, k, sinks, z, z, max_seqlen=10)
    torch.cuda.synchronize()
    assert o.shape == (0, 8, 64) and lse.shape == (8, 0)
    q = torch.randn(2, 8, 64).bfloat16().to(DEV)
    k0 = torch.empty(0, 2, 64, dtype=torch.bfloat16, device=DEV)
    starts = torch.zeros(2, dtype=torch.int32, device=DEV)
    lens = torch.ones(2, dtype=torch.int32, device=DEV)
    p = sa.make_decode_params(q, k0, max_seqlen=4)
    ws = torch.empty(sa.sink_attn_decode_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    o, lse = sa.sink_attn_decode(q, k0, k0, sinks, starts, lens, params=p, workspace=ws)
    st, flags = sa.sink_attn_fetch_device_error(ws)
    assert st == _abi.SINK_ERR_DEVICE and flags != 0
    assert torch.all(o.float() == 0)
    torch.testing.assert_close(lse, sinks[:, None].expand(8, 2), rtol=1e-6, atol=1e-6)
