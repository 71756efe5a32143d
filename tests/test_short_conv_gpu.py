"""GPU parity of the short convolution (kda_short_conv_fwd through the Python binding)
against the fp64 oracle on the same seeded inputs: dense and varlen (an empty
sequence, sequences shorter than the filter, sequences crossing 64-token tiles),
filter widths 2-4, bias, bf16 and fp32 in/out, decode steps with the state updated
in place, and the full conv_prefill workload on a sample of channels.

Tolerance: the kernel sums W products in fp32 and applies SiLU with a fast
exponential, so fp32 outputs sit within a few 1e-7 of the oracle (bound 1e-5 of
the output's rms); bf16 outputs add one rounding, at most 2^-9 relative
(bound 2^-8 relative + 1e-6).  The carried state is a copy of inputs: exact."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_conv_inputs

pytestmark = pytest.mark.gpu

FP32_OUT_TOL = 1e-5


def run_oracle(d, act="silu", channels=slice(None)):
    x = d["x"].float().cpu().numpy()[..., channels]
    w = d["weight"].double().cpu().numpy()[channels]
    b = None if d["bias"] is None else d["bias"].double().cpu().numpy()[channels]
    s0 = None if d["conv_state"] is None else d["conv_state"].double().cpu().numpy()[..., channels]
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].numpy()
    return oracle.short_conv(x, w, b, s0, cu_seqlens=cu, activation=act)


def check(y, sf, yr, sr, y_bf16):
    y = y.double().cpu().numpy()
    assert np.all(np.isfinite(y))
    if y_bf16:
        assert np.all(np.abs(y - yr) <= 2.0 ** -8 * np.abs(yr) + 1e-6)
    else:
        rms = max(float(np.sqrt(np.mean(yr * yr))), 1e-30) if yr.size else 1.0
        assert (np.abs(y - yr).max() / rms if yr.size else 0.0) <= FP32_OUT_TOL
    if sf is not None:
        assert np.array_equal(sf.double().cpu().numpy(), sr)


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_dense(W, out):
    d = make_conv_inputs(B=3, T=150, D=512, W=W, state=True, bias=(W == 3))
    dev = {k: (v.cuda() if torch.is_tensor(v) and k != "cu_seqlens" else v) for k, v in d.items()}
    y, sf = kda.short_conv(dev["x"], dev["weight"], dev["bias"], dev["conv_state"],
                           out_dtype=torch.bfloat16 if out == "bf16" else torch.float32)
    torch.cuda.synchronize()
    yr, sr = run_oracle(d)
    check(y, sf, yr, sr, out == "bf16")


def test_fp32_input_no_activation():
    d = make_conv_inputs(B=2, T=70, D=264, W=4, state=False)
    x32 = d["x"].float() * 1.37  # values that bf16 cannot hold
    d32 = dict(d, x=x32)
    y, sf = kda.short_conv(x32.cuda(), d["weight"].cuda(), activation=None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr, sr = oracle.short_conv(x32.numpy(), d["weight"].double().numpy(), activation=None)
    check(y, sf, yr, sr, False)
    assert d32["x"].dtype == torch.float32


def test_varlen_edges():
    lengths = [130, 0, 2, 1, 64, 65, 3, 200]
    d = make_conv_inputs(D=256, W=4, lengths=lengths, state=True, bias=True)
    dev = {k: (v.cuda() if torch.is_tensor(v) and k != "cu_seqlens" else v) for k, v in d.items()}
    y, sf = kda.short_conv(dev["x"], dev["weight"], dev["bias"], dev["conv_state"], cu_seqlens=d["cu_seqlens"],
                           out_dtype=torch.float32)
    torch.cuda.synchronize()
    yr, sr = run_oracle(d)
    check(y, sf, yr, sr, False)


def test_varlen_zero_state_and_no_state_out():
    d = make_conv_inputs(D=128, W=4, lengths=[5, 77, 1], state=False)
    y, sf = kda.short_conv(d["x"].cuda(), d["weight"].cuda(), cu_seqlens=d["cu_seqlens"],
                           output_final_state=False)
    torch.cuda.synchronize()
    assert sf is None
    yr, _ = run_oracle(d)
    check(y, None, yr, None, True)


def test_decode_steps_in_place():
    """Three decode steps, the state updated in place, against the oracle run over
    the three tokens at once (the state carries the history)."""
    B, D, W = 37, 384, 4
    d = make_conv_inputs(B=B, T=3, D=D, W=W, state=True)
    state = d["conv_state"].clone().cuda()
    w = d["weight"].cuda()
    ys = []
    for t in range(3):
        y, s_out = kda.short_conv(d["x"][:, t:t + 1].contiguous().cuda(), w, None, state, final_state=state,
                                  out_dtype=torch.float32)
        assert s_out.data_ptr() == state.data_ptr()
        ys.append(y)
    torch.cuda.synchronize()
    yr, sr = run_oracle(d)
    check(torch.cat(ys, 1), state, yr, sr, False)


def test_empty_prompt_hands_state_through():
    d = make_conv_inputs(B=2, T=0, D=64, W=4, state=True)
    y, sf = kda.short_conv(d["x"].cuda(), d["weight"].cuda(), None, d["conv_state"].cuda())
    torch.cuda.synchronize()
    assert y.shape == (2, 0, 64)
    assert torch.equal(sf.cpu(), d["conv_state"])


def test_conv_prefill_full_size_sampled():
    """The benchmarked workload (B=1, T=8192, D=36864) in the launch configuration the
    benchmark times; the oracle checks every token of 1024 sampled channels (the
    convolution is depthwise, so channels are independent)."""
    d = make_conv_inputs("conv_prefill", device="cuda")
    y = torch.empty_like(d["x"])
    yk, sf = kda.short_conv(d["x"], d["weight"], None, None, y=y)
    torch.cuda.synchronize()
    assert yk.data_ptr() == y.data_ptr()
    ch = np.sort(np.random.default_rng(0).choice(d["D"], 1024, replace=False))
    dc = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}
    yr, sr = run_oracle(dc, channels=ch)
    check(y[..., torch.from_numpy(ch).cuda()], sf[..., torch.from_numpy(ch).cuda()], yr, sr, True)
