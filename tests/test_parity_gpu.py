"""GPU parity of the CUDA paths against the fp64 oracle, through the C ABI.

Decode step (fused gated norm), the token-by-token form, the fp32 chunked path and
the standalone gated norm.  The bar: max|diff| / rms(oracle) <= 5e-3 for outputs and
final states; the fp32 paths are also held to 1e-4 against each other."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_helpers import FP32_TOL, PARITY, assert_bf16_close, np32, oracle_run, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


def norm_oracle(o, d):
    return oracle.gated_rmsnorm(o, np32(d["gate"]), np32(d["norm_w"]), eps=d["eps"])


# --------------------------------------------------------------------------- decode


def decode_inputs(B, H, K=128, V=128, seed=3):
    w = WORKLOADS["decode"]
    d = make_inputs(w, device="cuda", B=B, H=H, seed=seed)
    d = {k: (v.squeeze(1) if torch.is_tensor(v) and v.dim() >= 3 and k not in ("initial_state",) else v)
         for k, v in d.items()}
    return d


def decode_oracle(d, units=None):
    """Oracle for one token per sequence; units = list of (b, h) or None for all."""
    q, k, v, g, beta = (np32(d[n]) for n in ("q", "k", "v", "g", "beta"))
    s0 = np32(d["initial_state"]).astype(np.float64)
    gate = np32(d["gate"])
    if units is not None:
        bs = np.array([u[0] for u in units])
        hs = np.array([u[1] for u in units])
        sel = lambda x: x[bs, hs][:, None]  # each unit becomes its own batch row, one head
        q, k, v, g, beta, s0, gate = sel(q), sel(k), sel(v), sel(g), sel(beta), sel(s0), sel(gate)
    o, s = oracle.recurrent(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], s0, scale=d["scale"])
    y = oracle.gated_rmsnorm(o[:, 0], gate, np32(d["norm_w"]), eps=d["eps"])
    return o[:, 0], s, y


def test_decode_small_matches_oracle():
    d = decode_inputs(B=3, H=4)
    o, s, y = kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                 gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"])
    torch.cuda.synchronize()
    oo, so, yo = decode_oracle(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL
    assert rel_err(y.view(3, 4, 128), yo.reshape(3, 4, 128)) <= FP32_TOL


def test_decode_full_size_in_place_sampled():
    """The decode workload at full size (B=256, H=96, d=128, state 1.6 GB) with the state
    updated in place, in the launch configuration the benchmark times; sampled units
    against the oracle."""
    d = decode_inputs(B=256, H=96)
    s_in = d["initial_state"].clone()
    state = d["initial_state"]
    y = torch.empty(256, 96 * 128, device="cuda")
    o, s, y = kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, gate=d["gate"],
                                 norm_w=d["norm_w"], eps=d["eps"], state_out=state, y=y, return_o=True)
    torch.cuda.synchronize()
    assert s.data_ptr() == state.data_ptr()
    rng = np.random.default_rng(0)
    units = [(int(b), int(h)) for b, h in zip(rng.integers(0, 256, 96), rng.integers(0, 96, 96))]
    units += [(0, 0), (255, 95)]
    d_ref = dict(d, initial_state=s_in)
    oo, so, yo = decode_oracle(d_ref, units)
    bs = [u[0] for u in units]
    hs = [u[1] for u in units]
    assert rel_err(o[bs, hs], oo[:, 0]) <= FP32_TOL
    assert rel_err(s[bs, hs], so[:, 0]) <= FP32_TOL
    assert rel_err(y.view(256, 96, 128)[bs, hs], yo.reshape(-1, 128)) <= FP32_TOL


def test_decode_zero_state_and_no_norm():
    d = decode_inputs(B=2, H=3)
    o, s = kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], None)
    torch.cuda.synchronize()
    dz = dict(d, initial_state=torch.zeros_like(d["initial_state"]))
    oo, so, _ = decode_oracle(dz)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


def test_decode_fp32_inputs_bf16_outputs_and_many_units_per_cta():
    """fp32 q, k, v and gate (staged rows of 512 bytes instead of 256) and bf16 outputs;
    5 x 97 units, more than one per CTA of the persistent decode kernel on most GPUs
    with few SMs and exactly its stride pattern on the others."""
    d = decode_inputs(B=5, H=97)
    f32 = {n: d[n].float() for n in ("q", "k", "v", "gate")}
    o, s, y = kda.recurrent_step(f32["q"], f32["k"], f32["v"], d["g"], d["beta"], d["initial_state"],
                                 gate=f32["gate"], norm_w=d["norm_w"], eps=d["eps"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert o.dtype == torch.bfloat16 and y.dtype == torch.bfloat16
    oo, so, yo = decode_oracle(d)
    assert rel_err(s, so) <= FP32_TOL
    # bf16 outputs: the oracle's values, rounded to bf16 once (half an ulp, 2^-9 relative)
    for got, ref in ((o.float(), oo), (y.float().view(5, 97, 128), yo.reshape(5, 97, 128))):
        got = got.cpu().double().numpy()
        ref = np.asarray(ref, np.float64)
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * rms)


@pytest.mark.parametrize("K,V", [(32, 32), (64, 64), (128, 64), (64, 128)])
def test_decode_other_head_sizes(K, V):
    torch.manual_seed(0)
    B, H = 3, 2
    q = torch.randn(B, H, K, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, H, K, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, H, V, device="cuda").to(torch.bfloat16)
    g = -torch.rand(B, H, K, device="cuda")
    beta = torch.rand(B, H, device="cuda")
    s0 = 0.1 * torch.randn(B, H, K, V, device="cuda")
    o, s = kda.recurrent_step(q, k, v, g, beta, s0, scale=K ** -0.5)
    oo, so = oracle.recurrent(np32(q)[:, None], np32(k)[:, None], np32(v)[:, None], np32(g)[:, None],
                              np32(beta)[:, None], np32(s0), scale=K ** -0.5)
    assert rel_err(o, oo[:, 0]) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


# --------------------------------------------------------------------------- token-by-token form


@pytest.mark.parametrize("K,V,T", [(32, 32, 64), (128, 128, 37), (64, 128, 20)])
def test_recurrent_fwd_matches_oracle(K, V, T):
    torch.manual_seed(1)
    B, H = 2, 3
    q = torch.randn(B, T, H, K, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, T, H, K, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, T, H, V, device="cuda").to(torch.bfloat16)
    g = -torch.rand(B, T, H, K, device="cuda")
    beta = torch.rand(B, T, H, device="cuda")
    s0 = 0.05 * torch.randn(B, H, K, V, device="cuda")
    o, s = kda.recurrent_fwd(q, k, v, g, beta, s0, scale=K ** -0.5)
    oo, so = oracle.recurrent(np32(q), np32(k), np32(v), np32(g), np32(beta), np32(s0), scale=K ** -0.5)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


def test_recurrent_fwd_states_and_norm():
    d = make_inputs("tiny", device="cuda", T=40)
    gate = torch.randn(1, 40, 2, 32, device="cuda").to(torch.bfloat16)
    w = 1 + 0.1 * torch.randn(32, device="cuda")
    o, s, st, y = kda.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                                    output_states=True, gate=gate, norm_w=w)
    oo, so, sto = oracle_run(d, return_states=True)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(st, sto) <= FP32_TOL
    assert rel_err(st[:, -1], so) <= FP32_TOL
    yo = oracle.gated_rmsnorm(oo, np32(gate), np32(w), eps=1e-5)
    assert rel_err(y, yo) <= FP32_TOL


def test_recurrent_fwd_varlen_with_empty_sequences():
    lengths = [5, 0, 19, 1, 0, 33]
    d = make_inputs("tiny", device="cuda", lengths=lengths)
    s0 = 0.1 * torch.randn(len(lengths), 2, 32, 32, device="cuda")
    d["initial_state"] = s0
    o, s = kda.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, scale=d["scale"],
                             cu_seqlens=d["cu_seqlens"])
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL
    # an empty sequence hands its initial state through unchanged
    assert torch.equal(s[1], s0[1]) and torch.equal(s[4], s0[4])


# --------------------------------------------------------------------------- fp32 chunked path


def test_tiny_workload_chunk_fp32():
    """The tiny workload exactly (B=1, T=64, H=2, d=32, chunk 16, zero initial state)."""
    d = make_inputs("tiny", device="cuda")
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], chunk=16, mode="fp32")
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 200])
def test_chunk_fp32_ragged_and_chunks(chunk, T):
    d = make_inputs("prefill", device="cuda", T=T, H=2, B=2)
    d["initial_state"] = 0.02 * torch.randn(2, 2, 128, 128, device="cuda")
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], scale=d["scale"],
                         chunk=chunk, mode="fp32")
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


def test_chunk_fp32_equals_recurrent_fp32():
    """spec internal check: GPU chunked and GPU token-by-token, both fp32, within 1e-4."""
    d = make_inputs("prefill", device="cuda", T=300, H=3)
    d["initial_state"] = 0.02 * torch.randn(1, 3, 128, 128, device="cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"])
    o1, s1 = kda.chunk_fwd(*args, scale=d["scale"], chunk=64, mode="fp32")
    o2, s2 = kda.recurrent_fwd(*args, scale=d["scale"])
    assert rel_err(o1, o2) <= FP32_TOL
    assert rel_err(s1, s2) <= FP32_TOL


def test_chunk_fp32_stress_min_decay():
    """g = -5 everywhere (the gate lower bound): every factor exp(G_i - G_j) underflows fast."""
    d = make_inputs("prefill", device="cuda", T=150, H=2, g_const=-5.0)
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], chunk=64, mode="fp32")
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


def test_chunk_fp32_varlen_edges():
    lengths = [0, 5, 64, 130, 1, 0]
    d = make_inputs("prefill", device="cuda", lengths=lengths, H=2)
    d["initial_state"] = 0.02 * torch.randn(len(lengths), 2, 128, 128, device="cuda")
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], scale=d["scale"],
                         chunk=64, mode="fp32", cu_seqlens=d["cu_seqlens"])
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= FP32_TOL
    assert rel_err(s, so) <= FP32_TOL


def test_chunk_fp32_empty_prompt_passes_state_through():
    d = make_inputs("prefill", device="cuda", T=0, H=2)
    s0 = torch.randn(1, 2, 128, 128, device="cuda")
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, scale=d["scale"], mode="fp32")
    assert o.numel() == 0
    assert torch.equal(s, s0)


def test_chunk_fp32_split_halves_and_in_place_state():
    d = make_inputs("prefill", device="cuda", T=256, H=2)
    args = lambda a, b: (d["q"][:, a:b], d["k"][:, a:b], d["v"][:, a:b], d["g"][:, a:b], d["beta"][:, a:b])
    o, s = kda.chunk_fwd(*args(0, 256), scale=d["scale"], mode="fp32")
    state = torch.zeros(1, 2, 128, 128, device="cuda")
    o1, _ = kda.chunk_fwd(*args(0, 100), state, scale=d["scale"], mode="fp32", final_state=state)
    o2, s2 = kda.chunk_fwd(*args(100, 256), state, scale=d["scale"], mode="fp32", final_state=state)
    assert s2.data_ptr() == state.data_ptr()
    assert rel_err(torch.cat([o1, o2], 1), o) <= FP32_TOL
    assert rel_err(s2, s) <= FP32_TOL


def test_chunk_fp32_fused_norm_without_o():
    d = make_inputs("long", device="cuda", T=100, H=3, B=2)
    o_ref, s_ref = oracle_run(d)
    _, s, y = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], mode="fp32",
                            gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"], return_o=False)
    assert rel_err(y, norm_oracle(o_ref, d)) <= FP32_TOL
    assert rel_err(s, s_ref) <= FP32_TOL


def test_chunk_fp32_bf16_outputs():
    """bf16 o from the fp32 chunked path, element by element, over three full chunks and
    a 37-token tail."""
    d = make_inputs("prefill", device="cuda", T=229, H=2)
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], mode="fp32",
                         out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    oo, so = oracle_run(d)
    assert_bf16_close(o, oo, FP32_TOL)
    assert rel_err(s, so) <= FP32_TOL


# --------------------------------------------------------------------------- gated norm


@pytest.mark.parametrize("V", [32, 64, 128])
def test_gated_rmsnorm_kernel(V):
    torch.manual_seed(2)
    o = torch.randn(33, 5, V, device="cuda")
    gate = torch.randn(33, 5, V, device="cuda").to(torch.bfloat16)
    w = 1 + 0.1 * torch.randn(V, device="cuda")
    y = kda.gated_rmsnorm(o, gate, w, 1e-5)
    yo = oracle.gated_rmsnorm(np32(o), np32(gate), np32(w), 1e-5)
    assert rel_err(y, yo) <= FP32_TOL
    y_in_place = o.clone()
    kda.gated_rmsnorm(y_in_place, gate, w, 1e-5, y=y_in_place.view(33, 5 * V))
    assert rel_err(y_in_place.view(33, 5 * V), yo) <= FP32_TOL


def test_gated_rmsnorm_zero_rows():
    o = torch.zeros(0, 3, 128, device="cuda")
    y = kda.gated_rmsnorm(o, o.to(torch.bfloat16), torch.ones(128, device="cuda"))
    assert y.shape == (0, 384)


def test_launch_count_and_host_inputs_round_trip():
    """Host (pinned) inputs go through the same kernels and come back to the host."""
    before = kda.launch_count()
    d = make_inputs("tiny")
    pinned = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in d.items() if k != "initial_state"}
    o, s = kda.chunk_fwd(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"], scale=d["scale"],
                         chunk=16)
    assert o.device.type == "cpu" and s.device.type == "cpu"
    assert kda.launch_count() > before
    oo, so = oracle_run(d)
    assert rel_err(o, oo) <= FP32_TOL
