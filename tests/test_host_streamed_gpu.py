"""Host-resident prompts (B = 1, pinned host tensors) go through the device in
segments on three streams (copy in / compute / copy out).  The chunked kernel hands
its fp32 state between calls exactly as between chunks and the segments are whole
chunks, so the result must equal one device-side call bit for bit."""
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
from kimi_delta_attention_gated_gb300.inputs import make_inputs, make_logit_inputs

pytestmark = pytest.mark.gpu


def _host(d, names):
    return {n: d[n].cpu().pin_memory() for n in names if d.get(n) is not None}


@pytest.mark.parametrize("gated", [False, True])
def test_streamed_equals_single_call(gated):
    T = 2 * kda.HOST_SEGMENT + 500  # three segments, a ragged last one
    d = make_inputs("long" if gated else "prefill", device="cuda", T=T, H=4, B=1)
    s0 = torch.randn((1, 4, 128, 128), device="cuda") * 0.02
    kw = dict(scale=d["scale"])
    if gated:
        kw.update(gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
    ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, **kw)
    h = _host(d, ["q", "k", "v", "g", "beta", "gate"])
    kwh = dict(scale=d["scale"])
    if gated:
        kwh.update(gate=h["gate"], norm_w=d["norm_w"].cpu(), eps=d["eps"])
    out = kda.chunk_fwd(h["q"], h["k"], h["v"], h["g"], h["beta"], s0.cpu(), **kwh)
    torch.cuda.synchronize()
    assert all(t.device.type == "cpu" for t in out)
    for a, b in zip(out, ref):
        assert torch.equal(a, b.cpu())


def test_streamed_logits_equals_single_call():
    T = 3 * kda.HOST_SEGMENT
    d = make_logit_inputs("prefill", device="cuda", T=T, H=3)
    args = (d["g_logits"], d["beta_logits"], d["A_log"])
    ref = kda.chunk_fwd_logits(d["q"], d["k"], d["v"], *args, dt_bias=d["dt_bias"], scale=d["scale"])
    h = _host(d, ["q", "k", "v", "g_logits", "beta_logits"])
    out = kda.chunk_fwd_logits(h["q"], h["k"], h["v"], h["g_logits"], h["beta_logits"], d["A_log"].cpu(),
                               dt_bias=d["dt_bias"].cpu(), scale=d["scale"])
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b.cpu())


def test_streamed_into_caller_buffers():
    T = 2 * kda.HOST_SEGMENT
    d = make_inputs("prefill", device="cuda", T=T, H=2)
    ref_o, ref_s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"])
    h = _host(d, ["q", "k", "v", "g", "beta"])
    o_h = torch.empty((1, T, 2, 128)).pin_memory()
    s_h = torch.empty((1, 2, 128, 128)).pin_memory()
    o, s = kda.chunk_fwd(h["q"], h["k"], h["v"], h["g"], h["beta"], scale=d["scale"], o=o_h, final_state=s_h)
    assert o.data_ptr() == o_h.data_ptr() and s.data_ptr() == s_h.data_ptr()
    assert torch.equal(o_h, ref_o.cpu()) and torch.equal(s_h, ref_s.cpu())


def test_c_entry_pageable_batch_small_segments():
    """kda_chunk_fwd_host called directly with pageable numpy buffers: B = 2 sequences,
    256-token segments (five of them, the last ragged), an initial state, the gated norm
    writing y as well as o.  Equal bit for bit to one device call."""
    import ctypes
    import numpy as np
    from kimi_delta_attention_gated_gb300 import _load
    B, T, H = 2, 1100, 3
    d = make_inputs("long", device="cuda", T=T, H=H, B=B)
    s0 = torch.randn((B, H, 128, 128), device="cuda") * 0.02
    ref_o, ref_s, ref_y = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, scale=d["scale"],
                                        gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
    bf = lambda t: np.ascontiguousarray(t.view(torch.int16).cpu().numpy())  # bf16 bits, pageable
    f32 = lambda t: np.ascontiguousarray(t.float().cpu().numpy())
    q, k, v, gate = bf(d["q"]), bf(d["k"]), bf(d["v"]), bf(d["gate"])
    g, beta, nw, s0h = f32(d["g"]), f32(d["beta"]), f32(d["norm_w"]), f32(s0)
    o = np.zeros((B, T, H, 128), np.float32)
    y = np.zeros((B, T, H * 128), np.float32)
    fs = np.zeros((B, H, 128, 128), np.float32)
    lib = _load()
    need = lib.kda_chunk_fwd_host_workspace_size(B, H, 128, 128, 256)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.kda_chunk_fwd_host(p(q), p(k), p(v), 0, p(g), p(beta), p(s0h), p(fs), p(o), 1, B, T, H, 128, 128, 64,
                                d["scale"], 1, p(gate), 0, p(nw), d["eps"], p(y), 256, ctypes.c_void_p(ws.data_ptr()),
                                need, 0, st)
    assert rc == 0, lib.kda_last_error()
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(o, ref_o.cpu().numpy())
    assert np.array_equal(y, ref_y.cpu().numpy())
    assert np.array_equal(fs, ref_s.cpu().numpy())


def test_c_entry_empty_prompt_hands_the_state_through():
    import ctypes
    import numpy as np
    from kimi_delta_attention_gated_gb300 import _load
    lib = _load()
    s0 = np.random.default_rng(0).standard_normal((1, 2, 128, 128)).astype(np.float32)
    fs = np.zeros_like(s0)
    need = lib.kda_chunk_fwd_host_workspace_size(1, 2, 128, 128, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    o = np.zeros((1, 0, 2, 128), np.float32)
    rc = lib.kda_chunk_fwd_host(None, None, None, 0, None, None, p(s0), p(fs), p(o), 1, 1, 0, 2, 128, 128, 64,
                                0.088, 1, None, 0, None, 1e-5, None, 0, ctypes.c_void_p(ws.data_ptr()), need, 0,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.kda_last_error()
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(fs, s0)
