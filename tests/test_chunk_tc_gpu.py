"""GPU parity of the tensor-core chunked prefill (tcgen05) against the fp64 oracle.

Full-size workloads run in the launch configuration the benchmark uses and are
compared on sampled heads (the oracle recomputes those heads in full); small
cases are compared element by element.  Bar: max|diff| / rms(oracle) <= 5e-3 for
the outputs and, separately, the final states."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_inputs
from tests.gpu_helpers import PARITY, assert_bf16_close, np32, oracle_run, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


def run_tc(d, **kw):
    return kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("initial_state"), scale=d["scale"],
                         chunk=64, mode="tensor", cu_seqlens=d.get("cu_seqlens"), **kw)


def test_tc_small_ragged_with_state():
    d = make_inputs("prefill", device="cuda", B=2, T=200, H=3)
    d["initial_state"] = 0.02 * torch.randn(2, 3, 128, 128, device="cuda")
    o, s = run_tc(d)
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY


@pytest.mark.parametrize("T", [1, 64, 65, 127, 128, 300])
def test_tc_lengths(T):
    d = make_inputs("prefill", device="cuda", B=1, T=T, H=2)
    o, s = run_tc(d)
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY


def test_tc_prefill_workload_full_size_sampled():
    """B=1, T=8192, H=96, d=128, zero initial state, fp32 outputs: the benchmark's call."""
    d = make_inputs("prefill", device="cuda")
    o = torch.empty(1, 8192, 96, 128, device="cuda")
    fs = torch.empty(1, 96, 128, 128, device="cuda")
    kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, scale=d["scale"], chunk=64, o=o,
                  final_state=fs, mode="auto")
    torch.cuda.synchronize()
    heads = [0, 17, 48, 95]
    oo, so = oracle_run(d, heads=heads)
    assert rel_err(o[:, :, heads], oo) <= PARITY
    assert rel_err(fs[:, heads], so) <= PARITY
    assert torch.isfinite(o).all() and torch.isfinite(fs).all()


def test_tc_varlen_workload_full_size_sampled():
    """8 packed sequences, lengths log-uniform in [512, 16384], initial states N(0, 0.02^2)."""
    d = make_inputs("varlen", device="cuda")
    o, s = run_tc(d)
    torch.cuda.synchronize()
    heads = [3, 60]
    oo, so = oracle_run(d, heads=heads)
    assert rel_err(o[:, :, heads], oo) <= PARITY
    for n in range(d["N"]):
        assert rel_err(s[n, heads], so[n]) <= PARITY, f"sequence {n}"


def test_tc_long_workload_full_size_sampled_with_norm():
    """B=2, T=65536, H=96 with the fused sigmoid-gated RMSNorm (o not materialised)."""
    d = make_inputs("long", device="cuda")
    _, s, y = run_tc(d, gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"], return_o=False)
    torch.cuda.synchronize()
    heads = [5, 77]
    oo, so = oracle_run(d, heads=heads)
    gate = np32(d["gate"][:, :, heads])
    yo = oracle.gated_rmsnorm(oo, gate, np32(d["norm_w"]), eps=d["eps"])
    y_h = y.view(2, 65536, 96, 128)[:, :, heads].reshape(2, 65536, len(heads) * 128)
    assert rel_err(y_h, yo) <= PARITY
    assert rel_err(s[:, heads], so) <= PARITY


def test_tc_matches_fp32_chunk_path():
    d = make_inputs("prefill", device="cuda", T=512, H=4)
    o1, s1 = run_tc(d)
    o2, s2 = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], chunk=64, mode="fp32")
    assert rel_err(o1, o2) <= PARITY
    assert rel_err(s1, s2) <= PARITY


def test_tc_decay_range_fallback_everywhere():
    """g = -5 on every token: every chunk exceeds the factorised range and takes the exact gram."""
    d = make_inputs("prefill", device="cuda", T=200, H=2, g_const=-5.0)
    o, s = run_tc(d)
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY


def test_tc_decay_range_fallback_mixed():
    """Only the second chunk is beyond the range: both gram paths meet in one sequence."""
    d = make_inputs("prefill", device="cuda", T=256, H=2)
    d["g"][:, 64:128] = -4.0
    o, s = run_tc(d)
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY


def test_tc_varlen_edges_and_empty_sequences():
    lengths = [0, 5, 64, 130, 1, 0, 257]
    d = make_inputs("prefill", device="cuda", lengths=lengths, H=2)
    d["initial_state"] = 0.02 * torch.randn(len(lengths), 2, 128, 128, device="cuda")
    o, s = run_tc(d)
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY
    assert torch.equal(s[0], d["initial_state"][0]) and torch.equal(s[5], d["initial_state"][5])


def test_tc_split_halves_in_place_state():
    d = make_inputs("prefill", device="cuda", T=384, H=2)
    sl = lambda a, b: (d["q"][:, a:b], d["k"][:, a:b], d["v"][:, a:b], d["g"][:, a:b], d["beta"][:, a:b])
    o, s = kda.chunk_fwd(*sl(0, 384), scale=d["scale"], mode="tensor")
    state = torch.zeros(1, 2, 128, 128, device="cuda")
    o1, _ = kda.chunk_fwd(*sl(0, 192), state, scale=d["scale"], mode="tensor", final_state=state)
    o2, s2 = kda.chunk_fwd(*sl(192, 384), state, scale=d["scale"], mode="tensor", final_state=state)
    assert rel_err(torch.cat([o1, o2], 1), o) <= PARITY
    assert rel_err(s2, s) <= PARITY


def test_tc_fused_norm_and_o_together():
    d = make_inputs("long", device="cuda", B=1, T=333, H=3)
    o, s, y = run_tc(d, gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
    oo, so = oracle_run(d)
    yo = oracle.gated_rmsnorm(oo, np32(d["gate"]), np32(d["norm_w"]), eps=d["eps"])
    assert rel_err(o, oo) <= PARITY
    assert rel_err(y, yo) <= PARITY
    assert rel_err(s, so) <= PARITY


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16])
def test_tc_fused_norm_gate_dtypes_bf16_out(gdt):
    """The fused-norm instance with an fp32 or bf16 gate, o and y in bf16 (ragged tail)."""
    d = make_inputs("long", device="cuda", B=1, T=333, H=3)
    gate = d["gate"].to(gdt)
    o, s, y = run_tc(d, gate=gate, norm_w=d["norm_w"], eps=d["eps"], out_dtype=torch.bfloat16)
    oo, so = oracle_run(d)
    yo = oracle.gated_rmsnorm(oo, np32(gate), np32(d["norm_w"]), eps=d["eps"])
    assert o.dtype == torch.bfloat16 and y.dtype == torch.bfloat16
    # bf16 outputs: within the rounding to bf16 (half an ulp, 2^-9 relative) plus the
    # fp32 path's own error, element by element
    for a, ref in ((o, oo), (y, yo)):
        a = a.double().cpu().numpy().reshape(ref.shape)
        rms = np.sqrt((ref ** 2).mean())
        assert np.all(np.abs(a - ref) <= 2.0 ** -8 * np.abs(ref) + 5e-4 * rms)
    assert rel_err(s, so) <= PARITY


def test_tc_bf16_output():
    """bf16 o from the tensor path, element by element: four full chunks and a 7-token
    tail, so the full-chunk and the ragged store paths both write bf16."""
    d = make_inputs("prefill", device="cuda", T=263, H=2)
    o, s = run_tc(d, out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    oo, so = oracle_run(d)
    assert_bf16_close(o, oo, 5e-4)
    assert rel_err(s, so) <= PARITY


def test_tc_qk_norm_off():
    d = make_inputs("prefill", device="cuda", T=100, H=2)
    o, s = run_tc(d, use_qk_l2norm=False)
    q, k, v, g, beta = (np32(d[n]) for n in ("q", "k", "v", "g", "beta"))
    oo, so = oracle.recurrent(q, k, v, g, beta, scale=d["scale"], use_qk_l2norm=False)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY


def test_tc_frozen_state_closed_form():
    """beta = 0 and g = 0: the state never changes and o_t = scale * S0^T q^_t exactly in
    real arithmetic (no oracle involved); the tensor path must reproduce it."""
    d = make_inputs("prefill", device="cuda", T=200, H=3)
    d["beta"] = torch.zeros_like(d["beta"])
    d["g"] = torch.zeros_like(d["g"])
    s0 = 0.02 * torch.randn(1, 3, 128, 128, device="cuda", dtype=torch.float64)
    d["initial_state"] = s0.float()
    o, s = run_tc(d)
    qh = d["q"].double()
    qh = qh / torch.sqrt((qh * qh).sum(-1, keepdim=True) + 1e-6)
    ref = d["scale"] * torch.einsum("bthk,bhkv->bthv", qh, d["initial_state"].double())
    assert rel_err(o, ref) <= PARITY
    assert torch.equal(s, d["initial_state"])


def test_tc_pure_decay_closed_form():
    """beta = 0: S_t = Diag(exp sum_{s<=t} g_s) S0 and o_t = scale * S0^T (exp(G_t) * q^_t)
    (closed form of the decay-only recurrence); chunks cross and the tail is ragged."""
    d = make_inputs("prefill", device="cuda", T=150, H=2)
    d["beta"] = torch.zeros_like(d["beta"])
    d["initial_state"] = 0.02 * torch.randn(1, 2, 128, 128, device="cuda")
    o, s = run_tc(d)
    G = torch.cumsum(d["g"].double(), dim=1)  # [B,T,H,K]
    qh = d["q"].double()
    qh = qh / torch.sqrt((qh * qh).sum(-1, keepdim=True) + 1e-6)
    s0 = d["initial_state"].double()
    ref_o = d["scale"] * torch.einsum("bthk,bhkv->bthv", qh * torch.exp(G), s0)
    ref_s = torch.exp(G[:, -1])[..., None] * s0  # [B,H,K,1] * [B,H,K,V]
    assert rel_err(o, ref_o) <= PARITY
    assert rel_err(s, ref_s) <= PARITY


def test_tc_varlen_many_sequences():
    """More sequences than the host-side longest-first ordering covers (64): the kernel
    takes them in index order."""
    r = np.random.default_rng(11)
    lengths = [int(x) for x in r.integers(0, 200, 100)]
    d = make_inputs("prefill", device="cuda", lengths=lengths, H=1)
    o, s = run_tc(d)
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= PARITY
    assert rel_err(s, so) <= PARITY
