"""GPU tests of the concurrent tensor-core prefill (a workspace given, mode "tensor"): the
fused kernel runs one CTA per (sequence, head) while a pre-pass on the SMs it leaves idle
forms chunks' T diag(beta) and P ahead of it; a fused CTA takes a chunk's operands from the
pre-pass when their flag is set as it gets there and forms them itself otherwise, never
waiting.  The pre-pass computes those operands with the fused kernel's own arithmetic, in
the same order, so the concurrent form must give the fused form's bits whichever chunks it
took from where; each case also checks the oracle, and that the pre-pass was used
(prepass_hits) where it must have been: few heads, long prompts."""
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_inputs, make_logit_inputs
from tests.gpu_helpers import PARITY, np32, oracle_run, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


def both(d, **kw):
    """The same call through the fused form and the concurrent form; returns (fused,
    concurrent, chunks the concurrent call took from the pre-pass)."""
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("initial_state"))
    kw = dict(scale=d["scale"], chunk=64, mode="tensor", cu_seqlens=d.get("cu_seqlens"), **kw)
    fused = kda.chunk_fwd(*args, workspace=None, **kw)
    kda.prepass_hits()
    conc = kda.chunk_fwd(*args, workspace="auto", **kw)
    hits = kda.prepass_hits()
    kda.device_status()
    return fused, conc, hits


def assert_same(a, b):
    for x, y in zip(a, b):
        if x is None:
            assert y is None
            continue
        assert torch.equal(x, y)


def test_few_heads_long_prompt_takes_the_prepass():
    """4 heads x 64 chunks on a GPU of far more SMs: the pre-pass runs well ahead, so most
    chunks after the first few come from it."""
    d = make_inputs("prefill", device="cuda", T=4096, H=4)
    fused, conc, hits = both(d)
    assert_same(fused, conc)
    assert hits >= 4 * 64 // 2, hits
    oo, so = oracle_run(d, heads=[0, 3])
    assert rel_err(conc[0][:, :, [0, 3]], oo) <= PARITY
    assert rel_err(conc[1][:, [0, 3]], so) <= PARITY


def test_prefill_workload_full_size():
    """The benchmark's prefill (B=1, T=8192, H=96): same bits as the fused form."""
    d = make_inputs("prefill", device="cuda")
    fused, conc, hits = both(d)
    assert_same(fused, conc)
    assert 0 <= hits <= 96 * 128


@pytest.mark.parametrize("T", [1, 64, 65, 333])
def test_short_prompts_with_initial_state(T):
    d = make_inputs("varlen", device="cuda", lengths=[T], H=3)
    fused, conc, _ = both(d)
    assert_same(fused, conc)
    oo, so = oracle_run(d)
    assert rel_err(conc[0], oo) <= PARITY
    assert rel_err(conc[1], so) <= PARITY


def test_varlen_with_empty_sequences():
    d = make_inputs("varlen", device="cuda", lengths=[0, 700, 1, 0, 1280, 191], H=2)
    fused, conc, hits = both(d)
    assert_same(fused, conc)
    assert hits > 0
    oo, so = oracle_run(d)
    assert rel_err(conc[0], oo) <= PARITY
    assert rel_err(conc[1], so) <= PARITY


@pytest.mark.parametrize("gdt,odt", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32)])
def test_with_norm(gdt, odt):
    d = make_inputs("long", device="cuda", B=2, T=1500, H=3)
    gate = d["gate"].to(gdt)
    fused, conc, hits = both(d, gate=gate, norm_w=d["norm_w"], eps=d["eps"], out_dtype=odt)
    assert_same(fused, conc)
    assert hits > 0


def test_gate_logits():
    d = make_logit_inputs("prefill", device="cuda", T=2000, H=3)
    args = (d["q"], d["k"], d["v"], d["g_logits"], d["beta_logits"], d["A_log"])
    kw = dict(dt_bias=d["dt_bias"], g_lower_bound=d["g_lower_bound"], scale=d["scale"], mode="tensor")
    fused = kda.chunk_fwd_logits(*args, workspace=None, **kw)
    kda.prepass_hits()
    conc = kda.chunk_fwd_logits(*args, workspace="auto", **kw)
    hits = kda.prepass_hits()
    kda.device_status()
    assert_same(fused, conc)
    assert hits > 0
    g, beta = oracle.gates(np32(d["g_logits"]), np32(d["A_log"]), np32(d["beta_logits"]), np32(d["dt_bias"]),
                           d["g_lower_bound"])
    oo, so = oracle.recurrent(np32(d["q"]), np32(d["k"]), np32(d["v"]), g, beta, scale=d["scale"])
    assert rel_err(conc[0], oo) <= PARITY
    assert rel_err(conc[1], so) <= PARITY


def test_wide_decay_chunks_keep_their_exact_path():
    """Strong decay on some chunks: those take the fused kernel's exact path even when the
    pre-pass has formed their operands; the others may come from the pre-pass."""
    d = make_inputs("prefill", device="cuda", T=2048, H=2)
    g = d["g"].clone()
    g[:, 640:704] = -5.0
    g[:, 1300:1310, :, :40] = -5.0
    d["g"] = g
    fused, conc, _ = both(d)
    assert_same(fused, conc)
    oo, so = oracle_run(d)
    assert rel_err(conc[0], oo) <= PARITY
    assert rel_err(conc[1], so) <= PARITY


def test_many_heads_run_the_fused_form_alone():
    """As many units as SMs or more: no SM is left for a pre-pass, the workspace is unused."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d = make_inputs("prefill", device="cuda", T=128, H=sms)
    fused, conc, hits = both(d)
    assert_same(fused, conc)
    assert hits == 0
