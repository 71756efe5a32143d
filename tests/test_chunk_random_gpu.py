"""Seeded random sweep of the tensor-core prefill against the fp64 oracle.

Each case takes the form (the fused kernel, the concurrent form with a workspace, or the
split form) and the inputs (g and beta given, the same with the fused sigmoid-gated
RMSNorm, gates from logits, or both) from its seed, every pair twice, and draws the rest:
1-4 sequences of 0-400 tokens packed as varlen (so empty sequences, single tokens, ragged
tails and several whole chunks all occur), 1-6 heads, an initial state or none, fp32 or
bf16 outputs, and an fp32 or bf16 gate and logits.
Bar, as for the other parity tests: fp32 outputs and the final states within
max|diff| / rms(oracle) <= 5e-3; bf16 outputs element by element within their rounding
to bf16 plus 5e-4 rms (the fp32 path's own error)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
import oracle
from kimi_delta_attention_gated_gb300.inputs import make_inputs, make_logit_inputs
from tests.gpu_helpers import PARITY, assert_bf16_close, np32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kimi_delta_attention_gated_gb300 import build
    build.build()


def draw(seed):
    rng = np.random.default_rng(7000 + seed)
    n = int(rng.integers(1, 5))
    lengths = [int(x) for x in rng.integers(0, 401, n)]
    if n > 1 and rng.random() < 0.4:
        lengths[int(rng.integers(0, n))] = 0
    if sum(lengths) == 0:
        lengths[0] = 1
    # every (form, inputs) pair twice over 24 seeds; the rest drawn
    return dict(lengths=lengths, H=int(rng.integers(1, 7)), state=bool(rng.random() < 0.5),
                form=("fused", "concurrent", "split")[seed % 3],
                kind=("g", "norm", "logits", "logits+norm")[(seed // 3) % 4],
                out=(torch.float32, torch.bfloat16)[int(rng.integers(0, 2))],
                xdt=(torch.float32, torch.bfloat16)[int(rng.integers(0, 2))])


def check(a, ref, out_dtype):
    if out_dtype == torch.bfloat16:
        assert a.dtype == torch.bfloat16
        assert_bf16_close(a, ref, 5e-4)
    else:
        assert rel_err(a, ref) <= PARITY


@pytest.mark.parametrize("seed", range(24))
def test_random_case(seed):
    c = draw(seed)
    H, logits, norm = c["H"], c["kind"].startswith("logits"), c["kind"].endswith("norm")
    d = (make_logit_inputs("prefill", "cuda", lengths=c["lengths"], H=H, seed=seed, logits_dtype=c["xdt"])
         if logits else make_inputs("prefill", "cuda", lengths=c["lengths"], H=H, seed=seed))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(500 + seed)
    N, T, V = len(c["lengths"]), d["T"], d["V"]
    s0 = 0.02 * torch.randn((N, H, 128, V), generator=gen, device="cuda") if c["state"] else None
    kw = dict(scale=d["scale"], chunk=64, cu_seqlens=d["cu_seqlens"], out_dtype=c["out"],
              mode="split" if c["form"] == "split" else "tensor",
              workspace=None if c["form"] == "fused" else "auto")
    gate = norm_w = None
    if norm:
        gate = torch.randn((1, T, H, V), generator=gen, device="cuda").to(c["xdt"])
        norm_w = 1.0 + 0.1 * torch.randn((V,), generator=gen, device="cuda")
        kw.update(gate=gate, norm_w=norm_w, eps=d["eps"])
    if logits:
        res = kda.chunk_fwd_logits(d["q"], d["k"], d["v"], d["g_logits"], d["beta_logits"], d["A_log"], s0,
                                   dt_bias=d["dt_bias"], g_lower_bound=d["g_lower_bound"], **kw)
        g, beta = oracle.gates(np32(d["g_logits"]), np32(d["A_log"]), np32(d["beta_logits"]), np32(d["dt_bias"]),
                               d["g_lower_bound"])
    else:
        res = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], s0, **kw)
        g, beta = np32(d["g"]), np32(d["beta"])
    torch.cuda.synchronize()
    kda.device_status()
    oo, so = oracle.recurrent(np32(d["q"]), np32(d["k"]), np32(d["v"]), g, beta,
                              None if s0 is None else np32(s0).astype(np.float64), scale=d["scale"],
                              cu_seqlens=d["cu_seqlens"].cpu().numpy().astype(np.int64))
    check(res[0], oo, c["out"])
    assert rel_err(res[1], so) <= PARITY, c
    if norm:
        check(res[2], oracle.gated_rmsnorm(oo, np32(gate), np32(norm_w), eps=d["eps"]), c["out"])
