"""GPU parity of the decode step with the q, k, v short convolutions fused ahead of it
(kda_recurrent_step_conv through the Python binding's ``conv=`` argument) against the
fp64 oracle composed the way the layer composes the two steps: oracle.short_conv (+ SiLU)
on each raw projection with its history, then oracle.recurrent on the convolved q, k, v
(and oracle.gated_rmsnorm, oracle.gates where the case uses them).

Tolerances: the kernel convolves in fp32 and keeps the result in fp32, so o, the state
and y sit at the decode path's own fp32 level (max|diff| / rms <= 1e-4, as the plain
decode tests); the new histories are copies of inputs and must match exactly."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_decode_conv_inputs
from tests.gpu_helpers import FP32_TOL, np32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


def conv_oracle(d, units=None):
    """(q, k, v convolved [U, 128] fp64 each, new histories [3][B, W-1, D] fp64) for the
    units (b, h) given, or all units in (b, h) order."""
    B, H = d["q"].shape[:2]
    D = H * 128
    outs, hists = [], []
    for f, name in enumerate(("q", "k", "v")):
        x = np32(d[name]).reshape(B, 1, D)
        s0 = None if d["conv_state"] is None else np32(d["conv_state"][f]).astype(np.float64)
        y, sf = oracle.short_conv(x, np32(d["conv_weight"][f]).astype(np.float64), None, s0, activation="silu")
        y = y.reshape(B, H, 128)
        outs.append(y if units is None else np.stack([y[b, h] for b, h in units]))
        hists.append(sf)
    return outs, hists


def step_oracle(d, units=None):
    """Oracle o [U, 128], final state [U, 128, 128], y [U, 128] (or None) over the units."""
    B, H = d["q"].shape[:2]
    if units is None:
        units = [(b, h) for b in range(B) for h in range(H)]
    (qc, kc, vc), hists = conv_oracle(d, units)
    bs = np.array([u[0] for u in units])
    hs = np.array([u[1] for u in units])
    if "g_logits" in d:
        g, beta = oracle.gates(np32(d["g_logits"]), np32(d["A_log"]), np32(d["beta_logits"]),
                               np32(d["dt_bias"]), d["g_lower_bound"])
    else:
        g, beta = np32(d["g"]).astype(np.float64), np32(d["beta"]).astype(np.float64)
    g, beta = g[bs, hs], beta[bs, hs]
    s0 = np32(d["initial_state"])[bs, hs].astype(np.float64)
    col = lambda a: a[:, None, None]  # each unit is its own batch row: one token, one head
    o, s = oracle.recurrent(col(qc), col(kc), col(vc), col(g), beta[:, None, None], s0[:, None], scale=d["scale"])
    o = o[:, 0, 0]
    y = None
    if d.get("gate") is not None:
        y = oracle.gated_rmsnorm(o[:, None], np32(d["gate"])[bs, hs][:, None], np32(d["norm_w"]), eps=d["eps"])
        y = y.reshape(-1, 128)
    return o, s[:, 0], y, hists


def to_cuda(d):
    out = {}
    for n, t in d.items():
        if torch.is_tensor(t):
            out[n] = t.cuda()
        elif isinstance(t, tuple):
            out[n] = tuple(x.cuda() for x in t)
        else:
            out[n] = t
    return out


def run(d, *, norm=True, in_place=False, out_dtype=torch.float32):
    """The fused step on d (device tensors).  Returns (o, state, y or None, histories)."""
    state = d["initial_state"]
    hist_out = d["conv_state"] if in_place else None
    conv = (d["conv_weight"], d["conv_state"], hist_out)
    kw = dict(state_out=state if in_place else None, out_dtype=out_dtype, conv=conv)
    if norm:
        kw.update(gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
    if "g_logits" in d:
        res = kda.recurrent_step_logits(d["q"], d["k"], d["v"], d["g_logits"], d["beta_logits"], d["A_log"], state,
                                        dt_bias=d["dt_bias"], g_lower_bound=d["g_lower_bound"], **kw)
    else:
        res = kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, **kw)
    torch.cuda.synchronize()
    if norm:
        o, s, y, h = res
    else:
        (o, s, h), y = res, None
    return o, s, y, h


def check(d_ref, res, units=None):
    o, s, y, h = res
    oo, so, yo, ho = step_oracle(d_ref, units)
    if units is not None:
        bs = [u[0] for u in units]
        hs = [u[1] for u in units]
        o, s = o[bs, hs], s[bs, hs]
        y = None if y is None else y.view(-1, d_ref["H"], 128)[bs, hs]
    else:
        o, s = o.reshape(-1, 128), s.reshape(-1, 128, 128)
        y = None if y is None else y.reshape(-1, 128)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL
    if y is not None:
        assert rel_err(y, yo) <= FP32_TOL
    for f in range(3):
        assert np.array_equal(h[f].double().cpu().numpy(), ho[f]), f"history {f} is not the shifted input"


@pytest.mark.parametrize("W", [2, 3, 4])
def test_decode_conv_small(W):
    d = make_decode_conv_inputs(B=3, H=4, W=W)
    res = run(to_cuda(d))
    check(d, res)


def test_decode_conv_zero_history_logits_no_norm():
    """No history (the first token of each sequence), gates from bf16 logits, no norm."""
    d = make_decode_conv_inputs(B=2, H=5, W=4, history=False, logits=True)
    res = run(to_cuda(d), norm=False)
    check(d, res)


def test_decode_conv_in_place_many_units_per_cta():
    """State and histories updated in place; 7 x 97 units, several per CTA of the
    persistent kernel; fp32 raw inputs (values bf16 cannot hold)."""
    d = make_decode_conv_inputs(B=7, H=97, W=4, logits=True, seed=11)
    for n in ("q", "k", "v"):
        d[n] = d[n].float() * 1.37
    dev = to_cuda(d)
    hist_ptrs = [t.data_ptr() for t in dev["conv_state"]]
    s_ptr = dev["initial_state"].data_ptr()
    o, s, y, h = run(dev, in_place=True)
    assert s.data_ptr() == s_ptr and [t.data_ptr() for t in h] == hist_ptrs
    check(d, (o, s, y, h))


def test_decode_conv_matches_unfused_path():
    """The fused step against the two-call path of the library (short_conv with fp32
    output, then recurrent_step): the same fp32 arithmetic up to summation order."""
    d = to_cuda(make_decode_conv_inputs(B=4, H=6, W=4))
    o, s, y, h = run(d)
    B, H = 4, 6
    conv_out = []
    for f, n in enumerate(("q", "k", "v")):
        yc, sf = kda.short_conv(d[n].reshape(B, 1, H * 128), d["conv_weight"][f], None, d["conv_state"][f],
                                out_dtype=torch.float32)
        conv_out.append(yc.reshape(B, H, 128))
        assert torch.equal(sf, h[f])
    o2, s2, y2 = kda.recurrent_step(*conv_out, d["g"], d["beta"], d["initial_state"], gate=d["gate"],
                                    norm_w=d["norm_w"], eps=d["eps"])
    torch.cuda.synchronize()
    assert rel_err(o, o2.double().cpu().numpy()) <= 1e-5
    assert rel_err(s, s2.double().cpu().numpy()) <= 1e-5
    assert rel_err(y, y2.double().cpu().numpy()) <= 1e-5


def test_decode_conv_full_size_in_place_sampled():
    """B=256, H=96 (the fused decode workload the benchmark times: 1.6 GB of state, three
    histories of 3 x 12288 channels per sequence) in place; sampled units against the oracle."""
    d = make_decode_conv_inputs(B=256, H=96, W=4, device="cuda")
    ref = {n: (t.cpu() if torch.is_tensor(t) else tuple(x.cpu() for x in t) if isinstance(t, tuple) else t)
           for n, t in d.items()}
    o, s, y, h = run(d, in_place=True)
    rng = np.random.default_rng(1)
    units = [(int(b), int(hh)) for b, hh in zip(rng.integers(0, 256, 64), rng.integers(0, 96, 64))]
    units += [(0, 0), (255, 95)]
    oo, so, yo, ho = step_oracle(ref, units)
    bs = [u[0] for u in units]
    hs = [u[1] for u in units]
    assert rel_err(o[bs, hs], oo) <= FP32_TOL
    assert rel_err(s[bs, hs], so) <= FP32_TOL
    assert rel_err(y.view(256, 96, 128)[bs, hs], yo) <= FP32_TOL
    for f in range(3):
        assert np.array_equal(h[f].double().cpu().numpy(), ho[f])


def test_decode_conv_rejects_unsupported():
    d = to_cuda(make_decode_conv_inputs(B=2, H=2, W=4))
    with pytest.raises(kda.KDAError):  # K = 64 is not built with the fused convolutions
        q = d["q"][..., :64].contiguous()
        kda.recurrent_step(q, q, d["v"], d["g"][..., :64].contiguous(), d["beta"], None,
                           conv=(d["conv_weight"], d["conv_state"]))
