"""GPU tests of the split tensor-core prefill (mode "split", a workspace given): the state-independent
pre-pass over every chunk and head, then the per-head chain kernel.  The two forms run the
same products at the same split-bf16 precision; the split form accumulates the R/O product's
hi and lo parts in separate TMEM columns and adds them afterwards, so its fp32 sums differ
from the fused kernel's only in their order.  Every case is checked against the fp64 oracle
(max|diff| / rms(oracle) <= 5e-3) and, where no chunk needs the exact decay-range fallback,
against the fused form to 1e-3 of rms (five times tighter); the full-size prefill workload is
compared with the fused form, which its own full-size test checks against the oracle."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_inputs, make_logit_inputs
from tests.gpu_helpers import PARITY, assert_bf16_close, np32, oracle_run, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


def both(d, **kw):
    """The same call through the fused form (no workspace) and the split form."""
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("initial_state"))
    kw = dict(scale=d["scale"], chunk=64, cu_seqlens=d.get("cu_seqlens"), **kw)
    fused = kda.chunk_fwd(*args, workspace=None, mode="tensor", **kw)
    split = kda.chunk_fwd(*args, workspace="auto", mode="split", **kw)
    kda.device_status()
    return fused, split


def assert_agrees(a, b):
    """The split form's outputs against the fused form's: within 1e-3 of the fused one's rms
    (both carry about 6e-5 of split-bf16 error; they differ in fp32 summation order), plus
    one bf16 ulp where the output is bf16 (the two may round a value to neighbouring bf16s)."""
    for x, y in zip(a, b):
        if x is None:
            assert y is None
            continue
        assert x.dtype == y.dtype and x.shape == y.shape
        xf, yf = x.double(), y.double()
        assert torch.isfinite(yf).all()
        rms = float(torch.sqrt(torch.mean(xf * xf)))
        ulp = 2.0 ** -7 * xf.abs() if x.dtype == torch.bfloat16 else 0.0
        assert bool(((yf - xf).abs() <= ulp + 1e-3 * rms).all())


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 333])
def test_split_matches_fused(T):
    d = make_inputs("varlen", device="cuda", lengths=[T], H=3)  # one sequence with an initial state
    fused, split = both(d)
    assert_agrees(fused, split)
    oo, so = oracle_run(d)
    assert rel_err(split[0], oo) <= PARITY
    assert rel_err(split[1], so) <= PARITY


def test_split_matches_fused_varlen_with_empty_sequences():
    d = make_inputs("varlen", device="cuda", lengths=[0, 70, 1, 0, 128, 191], H=2)
    fused, split = both(d)
    assert_agrees(fused, split)
    oo, so = oracle_run(d)
    assert rel_err(split[0], oo) <= PARITY
    assert rel_err(split[1], so) <= PARITY


@pytest.mark.parametrize("gdt,odt", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32)])
def test_split_matches_fused_with_norm(gdt, odt):
    d = make_inputs("long", device="cuda", B=2, T=150, H=3)
    gate = d["gate"].to(gdt)
    fused, split = both(d, gate=gate, norm_w=d["norm_w"], eps=d["eps"], out_dtype=odt)
    assert_agrees(fused, split)
    oo, so = oracle_run(d)
    yo = oracle.gated_rmsnorm(oo, np32(gate), np32(d["norm_w"]), eps=d["eps"])
    if odt == torch.float32:
        assert rel_err(split[2], yo) <= PARITY
    else:
        assert_bf16_close(split[2], yo, 5e-4)


def test_split_matches_fused_norm_without_o():
    d = make_inputs("long", device="cuda", B=1, T=190, H=2)
    fused, split = both(d, gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"], return_o=False)
    assert fused[0] is None and split[0] is None
    assert_agrees(fused, split)


def test_split_matches_fused_gate_logits():
    d = make_logit_inputs("prefill", device="cuda", T=300, H=3)
    args = (d["q"], d["k"], d["v"], d["g_logits"], d["beta_logits"], d["A_log"])
    kw = dict(dt_bias=d["dt_bias"], g_lower_bound=d["g_lower_bound"], scale=d["scale"])
    fused = kda.chunk_fwd_logits(*args, workspace=None, mode="tensor", **kw)
    split = kda.chunk_fwd_logits(*args, workspace="auto", mode="split", **kw)
    kda.device_status()
    assert_agrees(fused, split)
    g, beta = oracle.gates(np32(d["g_logits"]), np32(d["A_log"]), np32(d["beta_logits"]), np32(d["dt_bias"]),
                           d["g_lower_bound"])
    oo, so = oracle.recurrent(np32(d["q"]), np32(d["k"]), np32(d["v"]), g, beta, scale=d["scale"])
    assert rel_err(split[0], oo) <= PARITY
    assert rel_err(split[1], so) <= PARITY


def test_split_matches_fused_prefill_workload_full_size():
    """The benchmark's prefill (B=1, T=8192, H=96) through both forms."""
    d = make_inputs("prefill", device="cuda")
    fused, split = both(d)
    assert_agrees(fused, split)


def test_split_fallback_every_chunk():
    """g = -5 everywhere: every chunk's decay range is far beyond the fast grams' limit, so
    the pre-pass forms A and P exactly and the chain kernel Kg from exp(gamma - G)."""
    d = make_inputs("prefill", device="cuda", T=200, H=2, g_const=-5.0)
    _, split = both(d)
    oo, so = oracle_run(d)
    assert rel_err(split[0], oo) <= PARITY
    assert rel_err(split[1], so) <= PARITY


def test_split_fallback_mixed_chunks():
    """Strong decay on some tokens only: fast and exact chunks side by side."""
    d = make_inputs("prefill", device="cuda", T=448, H=2)
    g = d["g"].clone()
    g[:, 64:128] = -5.0
    g[:, 300:310, :, :40] = -5.0
    d["g"] = g
    _, split = both(d)
    oo, so = oracle_run(d)
    assert rel_err(split[0], oo) <= PARITY
    assert rel_err(split[1], so) <= PARITY


def test_split_workspace_tensor_and_reuse():
    """A caller-owned workspace, reused by two calls in a row with different shapes."""
    a = make_inputs("prefill", device="cuda", T=260, H=4)
    b = make_inputs("varlen", device="cuda", lengths=[100, 33, 300], H=4)
    ws = torch.empty(max(kda.workspace_size(1, 260, 4), kda.workspace_size(1, 433, 4, 3)), dtype=torch.uint8,
                     device="cuda")
    for d in (a, b, a):
        out = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("initial_state"), scale=d["scale"],
                            cu_seqlens=d.get("cu_seqlens"), workspace=ws, mode="split")
        ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("initial_state"), scale=d["scale"],
                            cu_seqlens=d.get("cu_seqlens"), workspace=None, mode="tensor")
        assert_agrees(ref, out)
    kda.device_status()


def test_split_rejects_a_small_workspace():
    d = make_inputs("prefill", device="cuda", T=128, H=2)
    ws = torch.empty(kda.workspace_size(1, 128, 2) - 16, dtype=torch.uint8, device="cuda")
    for mode in ("tensor", "split"):
        with pytest.raises(kda.KDAError):
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], workspace=ws, mode=mode)
    with pytest.raises(kda.KDAError):  # the split form has nowhere to put its operands without one
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], mode="split")
