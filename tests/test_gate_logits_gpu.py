"""GPU parity of the fused gate prologue (kda_chunk_fwd_logits, kda_recurrent_step_logits):
g = max(lb, -exp(A_log) softplus(z + dt_bias)) and beta = sigmoid(b) computed inside the
kernels from bf16 / fp32 logits, against the oracle (oracle.gates, then the fp64
recurrence) on the same seeded logits.  Covers the tensor-core and fp32 chunked
paths, varlen with partial chunks (padding must stay an identity step), a chunk
whose decay range forces the exact fallback, the decode step with the gated norm,
and the full-size prefill in the benchmark's launch configuration (sampled heads).
Tolerance: the same 5e-3 max|diff| / rms bound as the g/beta paths."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from tests.gpu_helpers import PARITY, rel_err
from kimi_delta_attention_gated_gb300.inputs import make_logit_inputs

pytestmark = pytest.mark.gpu


def np32(t):
    return t.detach().float().cpu().numpy()


def oracle_from_logits(d, heads=None):
    hs = slice(None) if heads is None else list(heads)
    g, beta = oracle.gates(np32(d["g_logits"])[:, :, hs], np32(d["A_log"])[hs], np32(d["beta_logits"])[:, :, hs],
                           np32(d["dt_bias"])[hs], d["g_lower_bound"])
    s0 = d.get("initial_state")
    s0 = None if s0 is None else np32(s0)[:, hs].astype(np.float64)
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].numpy()
    return oracle.recurrent(np32(d["q"])[:, :, hs], np32(d["k"])[:, :, hs], np32(d["v"])[:, :, hs], g, beta, s0,
                            scale=d["scale"], cu_seqlens=cu)


def dev(d):
    return {k: (v.cuda() if torch.is_tensor(v) and k != "cu_seqlens" else v) for k, v in d.items()}


def run_chunk(d, mode, chunk=64):
    x = dev(d)
    return kda.chunk_fwd_logits(x["q"], x["k"], x["v"], x["g_logits"], x["beta_logits"], x["A_log"],
                                x["initial_state"], dt_bias=x["dt_bias"], g_lower_bound=x["g_lower_bound"],
                                scale=x["scale"], chunk=chunk, cu_seqlens=d["cu_seqlens"], mode=mode)


@pytest.mark.parametrize("mode", ["tensor", "fp32"])
@pytest.mark.parametrize("ldt", [torch.bfloat16, torch.float32])
def test_prefill_logits(mode, ldt):
    d = make_logit_inputs("prefill", T=200, H=4, logits_dtype=ldt)
    o, sf = run_chunk(d, mode)
    torch.cuda.synchronize()
    ro, rs = oracle_from_logits(d)
    assert rel_err(o, ro) <= PARITY
    assert rel_err(sf, rs) <= PARITY


@pytest.mark.parametrize("mode", ["tensor", "fp32"])
def test_varlen_partial_chunks(mode):
    d = make_logit_inputs("varlen", H=3, lengths=[70, 1, 129, 64, 33])
    o, sf = run_chunk(d, mode)
    torch.cuda.synchronize()
    ro, rs = oracle_from_logits(d)
    assert rel_err(o, ro) <= PARITY
    assert rel_err(sf, rs) <= PARITY


@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float32])
def test_prefill_logits_with_gated_norm(gdt):
    """The gates-from-logits tensor kernel with the fused sigmoid-gated RMSNorm (its own
    compiled instance), varlen with partial chunks, bf16 or fp32 gate: o, y and the final
    states against the oracle (y = the oracle's gated norm of the oracle's o)."""
    d = make_logit_inputs("varlen", H=3, lengths=[70, 1, 129, 64, 33])
    B, T, H, V = d["v"].shape
    gen = torch.Generator().manual_seed(2024)
    gate = torch.randn((B, T, H, V), generator=gen).to(gdt)
    norm_w = 1 + 0.1 * torch.randn(V, generator=gen)
    x = dev(d)
    o, sf, y = kda.chunk_fwd_logits(x["q"], x["k"], x["v"], x["g_logits"], x["beta_logits"], x["A_log"],
                                    x["initial_state"], dt_bias=x["dt_bias"], g_lower_bound=x["g_lower_bound"],
                                    scale=x["scale"], cu_seqlens=d["cu_seqlens"], mode="tensor",
                                    gate=gate.cuda(), norm_w=norm_w.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    ro, rs = oracle_from_logits(d)
    ry = oracle.gated_rmsnorm(ro, np32(gate), np32(norm_w), 1e-5)
    assert rel_err(o, ro) <= PARITY
    assert rel_err(y, ry) <= PARITY
    assert rel_err(sf, rs) <= PARITY


def test_wide_decay_takes_exact_fallback():
    """Large logits with A = 16 drive g to the -5 floor on every channel: a chunk's decay
    range is 320 > 80, so the tensor kernel computes its grams exactly (reading g from
    the logits there too)."""
    d = make_logit_inputs("prefill", T=130, H=2, z_mean=3.0)
    d["A_log"] = torch.full_like(d["A_log"], float(np.log(16.0)))
    o, sf = run_chunk(d, "tensor")
    torch.cuda.synchronize()
    ro, rs = oracle_from_logits(d)
    assert rel_err(o, ro) <= PARITY
    assert rel_err(sf, rs) <= PARITY


def test_decode_step_logits_with_norm():
    d = make_logit_inputs("decode", B=19, H=5)
    x = dev(d)
    sq = lambda t: t.squeeze(1).contiguous()
    state = x["initial_state"].clone()
    o, s_out, y = kda.recurrent_step_logits(sq(x["q"]), sq(x["k"]), sq(x["v"]), sq(x["g_logits"]),
                                            sq(x["beta_logits"]), x["A_log"], state, dt_bias=x["dt_bias"],
                                            gate=sq(x["gate"]), norm_w=x["norm_w"], eps=d["eps"], state_out=state)
    torch.cuda.synchronize()
    ro, rs = oracle_from_logits(d)
    ry = oracle.gated_rmsnorm(ro, np32(d["gate"]), np32(d["norm_w"]), d["eps"])
    assert rel_err(o, ro[:, 0]) <= PARITY
    assert rel_err(s_out, rs) <= PARITY
    assert rel_err(y, ry[:, 0]) <= PARITY


def test_full_size_prefill_logits_sampled():
    """B=1 T=8192 H=96 bf16 logits, the launch the benchmark times; the oracle checks 3 heads."""
    d = make_logit_inputs("prefill", device="cuda")
    o, sf = kda.chunk_fwd_logits(d["q"], d["k"], d["v"], d["g_logits"], d["beta_logits"], d["A_log"], None,
                                 dt_bias=d["dt_bias"], g_lower_bound=d["g_lower_bound"], scale=d["scale"])
    torch.cuda.synchronize()
    heads = [0, 47, 95]
    dc = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}
    ro, rs = oracle_from_logits(dc, heads)
    assert rel_err(o[:, :, heads], ro) <= PARITY
    assert rel_err(sf[:, heads], rs) <= PARITY
