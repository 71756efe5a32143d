"""Pins for the fp64 short-convolution oracle (the causal depthwise conv + SiLU
applied to q, k and v before the delta rule).

What the pins rest on (nnterp encyclopedia "Kimi-Linear", section "Printout":
Conv1d(12288, 12288, kernel_size=4, padding=3, groups=12288, bias=False); Kimi-K3
atlas "gate-project (decode, P = 1000)", section "Code": ShortConvolution(...,
kernel_size=4, activation='silu')):
  * library routines: torch's conv1d with exactly the printed configuration
    (depthwise, padding W-1, first T outputs kept) and numpy's convolve;
  * closed forms: the identity filter, the impulse response (tap order), SiLU;
  * structure: split-halves with the state handed across, varlen == separate runs.
Each pin is also run against planted mistakes (flipped taps, a dropped tap, the
activation before the sum, the state read newest-first) that must fail one of them.
"""
import numpy as np
import pytest
import torch

import oracle

RTOL = 1e-12


def oracle_runner(x, w, bias=None, state=None, act="silu"):
    return oracle.short_conv(x, w, bias, state, activation=act)


def silu(z):
    return z / (1.0 + np.exp(-z))


def mutant_runner(kind):
    """numpy re-implementation of the definition with one planted mistake."""
    def run(x, w, bias=None, state=None, act="silu"):
        x = np.asarray(x, dtype=np.float64)
        B, T, D = x.shape
        W = w.shape[1]
        y = np.zeros_like(x)
        sf = np.zeros((B, W - 1, D))
        for b in range(B):
            hist = np.zeros((W - 1, D)) if state is None else np.array(state[b], dtype=np.float64)
            if kind == "state_newest_first":
                hist = hist[::-1].copy()
            ww = w[:, ::-1] if kind == "flipped_taps" else w
            for t in range(T):
                win = np.concatenate([hist, x[b, t][None]], 0)  # [W, D], oldest first
                terms = ww.T * win
                if kind == "dropped_tap":
                    terms = terms[1:]
                if kind == "act_before_sum":
                    z = silu(terms).sum(0) if act == "silu" else terms.sum(0)
                else:
                    z = terms.sum(0)
                    z = silu(z) if act == "silu" else z
                if bias is not None:
                    z = z + bias
                y[b, t] = z
                hist = win[1:]
            sf[b] = hist
        return y, sf
    return run


def _data(B=2, T=9, D=12, W=4, seed=0):
    r = np.random.default_rng(seed)
    x = r.standard_normal((B, T, D)).astype(np.float32)
    w = r.uniform(-0.5, 0.5, (D, W))
    s0 = r.standard_normal((B, W - 1, D))
    return x, w, s0


def pin_torch_conv1d(run):
    """torch.nn.functional.conv1d with the printed configuration, in float64."""
    x, w, _ = _data()
    B, T, D = x.shape
    W = w.shape[1]
    ref = torch.nn.functional.conv1d(torch.from_numpy(x.astype(np.float64)).transpose(1, 2),
                                     torch.from_numpy(w)[:, None, :], padding=W - 1, groups=D)[..., :T]
    ref = ref.transpose(1, 2).numpy()
    y, _ = run(x, w, act=None)
    return np.allclose(y, ref, rtol=RTOL, atol=1e-13) and np.allclose(run(x, w)[0], silu(ref), rtol=RTOL, atol=1e-13)


def pin_numpy_convolve_with_state(run):
    """Per channel: the state prepended to the sequence, a 'valid' true convolution
    with the reversed filter (numpy convolve flips its kernel)."""
    x, w, s0 = _data(seed=1)
    y, sf = run(x, w, state=s0, act=None)
    B, T, D = x.shape
    W = w.shape[1]
    ok = True
    for b in range(B):
        for c in range(D):
            ext = np.concatenate([s0[b, :, c], x[b, :, c].astype(np.float64)])
            ref = np.convolve(ext, w[c, ::-1], mode="valid")
            ok &= np.allclose(y[b, :, c], ref, rtol=RTOL, atol=1e-13)
            ok &= np.allclose(sf[b, :, c], ext[-(W - 1):], rtol=0, atol=0)
    return ok


def pin_identity_filter(run):
    """weight = [0, .., 0, 1]: y = x (no activation), y = silu(x) with it."""
    x, _, _ = _data(seed=2)
    D = x.shape[2]
    w = np.zeros((D, 4))
    w[:, 3] = 1.0
    y0, _ = run(x, w, act=None)
    y1, _ = run(x, w)
    return np.array_equal(y0, x.astype(np.float64)) and np.allclose(y1, silu(x.astype(np.float64)), rtol=RTOL)


def pin_impulse_response(run):
    """A unit impulse at t = 0 from a zero state reads the taps newest-first:
    y[t][c] = weight[c][W-1-t] for t < W, then 0."""
    D, W, T = 5, 4, 7
    x = np.zeros((1, T, D), dtype=np.float32)
    x[0, 0] = 1.0
    w = np.arange(1, D * W + 1, dtype=np.float64).reshape(D, W)
    y, _ = run(x, w, act=None)
    ref = np.zeros((1, T, D))
    for t in range(W):
        ref[0, t] = w[:, W - 1 - t]
    return np.array_equal(y, ref)


def pin_state_taps(run):
    """A zero input after a one-hot state (slot j, oldest first) reads tap j at t = 0,
    and the state moves up by one slot."""
    D, W = 3, 4
    x = np.zeros((1, 1, D), dtype=np.float32)
    w = np.arange(1, D * W + 1, dtype=np.float64).reshape(D, W)
    ok = True
    for j in range(W - 1):
        s = np.zeros((1, W - 1, D))
        s[0, j] = 1.0
        y, sf = run(x, w, state=s, act=None)
        ok &= np.array_equal(y[0, 0], w[:, j])
        ok &= np.array_equal(sf[0, W - 2], np.zeros(D)) and (j == 0 or np.array_equal(sf[0, j - 1], np.ones(D)))
    return ok


def pin_split_halves(run):
    x, w, s0 = _data(T=11, seed=3)
    y, sf = run(x, w, state=s0)
    y1, s1 = run(x[:, :4], w, state=s0)
    y2, s2 = run(x[:, 4:], w, state=s1)
    return np.allclose(np.concatenate([y1, y2], 1), y, rtol=RTOL, atol=1e-13) and np.allclose(s2, sf, rtol=0, atol=0)


def pin_bias(run):
    x, w, _ = _data(seed=4)
    bias = np.linspace(-1, 1, x.shape[2])
    y0, _ = run(x, w, act=None)
    yb, _ = run(x, w, bias=bias, act=None)
    return np.allclose(yb - y0, np.broadcast_to(bias, y0.shape), rtol=0, atol=1e-12)


PINS = [pin_torch_conv1d, pin_numpy_convolve_with_state, pin_identity_filter, pin_impulse_response,
        pin_state_taps, pin_split_halves, pin_bias]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    assert pin(oracle_runner)


@pytest.mark.parametrize("kind", ["flipped_taps", "dropped_tap", "act_before_sum", "state_newest_first"])
def test_pins_catch_mutant(kind):
    run = mutant_runner(kind)
    assert not all(p(run) for p in PINS), f"no pin catches the '{kind}' mistake"


def test_mutant_harness_is_faithful():
    """Without a planted mistake the numpy harness passes every pin."""
    run = mutant_runner("none")
    assert all(p(run) for p in PINS)


def test_varlen_equals_separate_runs():
    x, w, _ = _data(B=1, T=13, seed=5)
    cu = [0, 5, 5, 13]
    s0 = np.random.default_rng(6).standard_normal((3, 3, x.shape[2]))
    y, sf = oracle.short_conv(x, w, None, s0, cu_seqlens=cu)
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        yn, sn = oracle.short_conv(x[:, a:b], w, None, s0[n:n + 1])
        assert np.allclose(y[:, a:b], yn, rtol=0, atol=0)
        assert np.allclose(sf[n], sn[0], rtol=0, atol=0)
    assert np.array_equal(sf[1], s0[1])  # an empty sequence hands its state through
