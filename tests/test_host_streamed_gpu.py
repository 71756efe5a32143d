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
