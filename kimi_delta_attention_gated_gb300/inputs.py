"""Seeded synthetic inputs for the KDA core, shaped like the Kimi-K3 KDA layers.

This module draws random numbers and nothing else: it holds none of the method's
arithmetic and serves both the CUDA path and the fp64 oracle (which receive the
same bits).  The shapes come from the Kimi-K3 config (96 KDA heads of 128
features, gate lower bound -5; atlas page "final-block-state", config.json
excerpt) and the decode shapes from the atlas page "gate-project (decode,
P = 1000)".  The decay recipe mirrors the layer's parameters shown on that page
(per-head A_log = log U(1, 16), a softplus of the decay logits, the lower bound
-5): g = max(-5, -exp(A_h) * softplus(z)) with z ~ N(-4, 1).

Workloads (names used by the tests and the benchmark):
  tiny      B=1  T=64     H=2   d=32   chunk 16  zero initial state
  prefill   B=1  T=8192   H=96  d=128  chunk 64  zero initial state
  varlen    8 sequences, lengths log-uniform in [512, 16384], H=96, d=128,
            initial state N(0, 0.02^2) per sequence
  decode    B=256 one token each, H=96, d=128, state N(0, 0.02^2),
            gate logits N(0,1), norm weight 1 + N(0, 0.1^2), eps 1e-5
  long      B=2  T=65536  H=96  d=128  chunk 64, zero initial state, gated norm

Short-convolution inputs (make_conv_inputs): x is the q, k and v projections side by
side, D = 3 * 96 * 128 = 36864 channels of N(0, 1) values in bf16; the filter is
Conv1d's default initialisation for a depthwise filter of 4 taps, U(-1/2, 1/2)
(bound 1/sqrt(fan_in), fan_in = 4); the conv state N(0, 1) (earlier inputs).
  conv_prefill  B=1   T=8192  D=36864  W=4, zero state
  conv_decode   B=256 T=1     D=36864  W=4, state given (updated in place)

Decode with the convolutions fused (make_decode_conv_inputs): the decode workload's
g, beta (or logits), state, gate and norm weight, with q, k, v replaced by the raw
projections (N(0, 1) in bf16, [B, H, 128] each), three filters [H*128, W] drawn as
above and three histories [B, W-1, H*128] of N(0, 1) values rounded to bf16 (earlier
raw inputs), each held in fp32.
  decode_conv   B=256 H=96 d=128 W=4, histories given (updated in place)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

GATE_LOWER_BOUND = -5.0
NORM_EPS = 1e-5


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    T: int
    H: int
    K: int
    V: int
    chunk: int
    n_seqs: int = 0            # > 0: varlen, packed as B = 1
    init_state_std: float = 0.0
    gated_norm: bool = False
    decode: bool = False
    len_range: tuple = field(default=(512, 16384))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.K)


WORKLOADS = {
    "tiny": Workload("tiny", 0, B=1, T=64, H=2, K=32, V=32, chunk=16),
    "prefill": Workload("prefill", 1, B=1, T=8192, H=96, K=128, V=128, chunk=64),
    "varlen": Workload("varlen", 2, B=1, T=0, H=96, K=128, V=128, chunk=64, n_seqs=8,
                       init_state_std=0.02),
    "decode": Workload("decode", 3, B=256, T=1, H=96, K=128, V=128, chunk=64,
                       init_state_std=0.02, gated_norm=True, decode=True),
    "long": Workload("long", 4, B=2, T=65536, H=96, K=128, V=128, chunk=64, gated_norm=True),
}


def varlen_lengths(n_seqs: int, lo: int, hi: int, gen: torch.Generator) -> list:
    """Lengths floor(exp(U(ln lo, ln hi))), clamped to [lo, hi]."""
    u = torch.rand(n_seqs, generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).floor().long()
    return [int(x) for x in lens.clamp(lo, hi)]


def _unit_rows_bf16(shape, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    return x.to(torch.bfloat16)


def make_inputs(w: Workload | str, device="cpu", *, T: int | None = None, H: int | None = None,
                B: int | None = None, lengths: list | None = None, g_const: float | None = None,
                seed: int | None = None) -> dict:
    """Draw one seeded input set.  Optional overrides shrink a workload for tests.

    Returns a dict of torch tensors on ``device``:
      q, k [B,T,H,K] bf16 (rows of unit L2 norm before rounding), v [B,T,H,V] bf16,
      g [B,T,H,K] fp32, beta [B,T,H] fp32, initial_state [N,H,K,V] fp32 or None,
      gate [B,T,H,V] bf16 and norm_w [V] fp32 when the workload has the gated norm,
      cu_seqlens (int32, host) for varlen, plus the scalars.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    cu = None
    if w.n_seqs or lengths is not None:
        if lengths is None:
            cpu_gen = torch.Generator()
            cpu_gen.manual_seed(1000 + (w.seed if seed is None else seed))
            lengths = varlen_lengths(w.n_seqs, w.len_range[0], w.len_range[1], cpu_gen)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        B, T = 1, int(cu[-1])
        N = len(lengths)
    else:
        N = B
    K, V = w.K, w.V
    q = _unit_rows_bf16((B, T, H, K), gen, device)
    k = _unit_rows_bf16((B, T, H, K), gen, device)
    v = torch.randn((B, T, H, V), generator=gen, device=device).to(torch.bfloat16)
    # Per-head A_h = log U(1, 16); decay logits z ~ N(-4, 1).
    a_log = torch.log(torch.empty(H, device=device).uniform_(1.0, 16.0, generator=gen))
    z = torch.randn((B, T, H, K), generator=gen, device=device) - 4.0
    g = torch.clamp(-torch.exp(a_log)[:, None] * torch.nn.functional.softplus(z), min=GATE_LOWER_BOUND)
    if g_const is not None:
        g = torch.full_like(g, float(g_const))
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen, device=device))
    s0 = None
    if w.init_state_std > 0:
        s0 = torch.randn((N, H, K, V), generator=gen, device=device) * w.init_state_std
    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), initial_state=s0,
               cu_seqlens=cu, B=B, T=T, H=H, K=K, V=V, N=N, chunk=w.chunk, scale=w.scale,
               eps=NORM_EPS, workload=w.name)
    if w.gated_norm:
        out["gate"] = torch.randn((B, T, H, V), generator=gen, device=device).to(torch.bfloat16)
        out["norm_w"] = 1.0 + 0.1 * torch.randn((V,), generator=gen, device=device)
    return out


def make_logit_inputs(w: Workload | str, device="cpu", *, T: int | None = None, H: int | None = None,
                      B: int | None = None, lengths: list | None = None, seed: int | None = None,
                      z_mean: float = -4.0, logits_dtype=torch.bfloat16) -> dict:
    """make_inputs(...) with the decay and write strength given as the layer's logits
    instead of g and beta: g_logits [B,T,H,K] ~ N(z_mean, 1), beta_logits [B,T,H] ~ N(0, 1)
    (both in ``logits_dtype``), A_log [H] = log U(1, 16), dt_bias [H,K] ~ U(-1/2, 1/2),
    lower bound -5.  q, k, v, the states and the norm inputs are drawn as in make_inputs
    (the same seed gives the same q, k, v)."""
    d = make_inputs(w, device, T=T, H=H, B=B, lengths=lengths, seed=seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(10_000 + (WORKLOADS[w].seed if isinstance(w, str) else w.seed) + (seed or 0))
    Bq, Tq, Hq, K = d["q"].shape
    z = torch.randn((Bq, Tq, Hq, K), generator=gen, device=device) + z_mean
    b = torch.randn((Bq, Tq, Hq), generator=gen, device=device)
    d.pop("g")
    d.pop("beta")
    d.update(g_logits=z.to(logits_dtype).contiguous(), beta_logits=b.to(logits_dtype).contiguous(),
             A_log=torch.log(torch.empty(Hq, device=device).uniform_(1.0, 16.0, generator=gen)),
             dt_bias=torch.empty((Hq, K), device=device).uniform_(-0.5, 0.5, generator=gen),
             g_lower_bound=GATE_LOWER_BOUND)
    return d


CONV_WORKLOADS = {
    "conv_prefill": dict(seed=5, B=1, T=8192, D=3 * 96 * 128, W=4, state=False),
    "conv_decode": dict(seed=6, B=256, T=1, D=3 * 96 * 128, W=4, state=True),
}


def make_conv_inputs(w: str | None = None, device="cpu", *, B: int | None = None, T: int | None = None,
                     D: int | None = None, W: int | None = None, lengths: list | None = None,
                     state: bool | None = None, bias: bool = False, seed: int | None = None) -> dict:
    """Seeded inputs for the short convolution: x [B,T,D] bf16, weight [D,W] fp32,
    bias [D] or None, conv_state [N,W-1,D] fp32 or None, cu_seqlens (host int32) for varlen."""
    cfg = dict(CONV_WORKLOADS[w]) if w else dict(seed=7, B=1, T=64, D=256, W=4, state=False)
    B = cfg["B"] if B is None else B
    T = cfg["T"] if T is None else T
    D = cfg["D"] if D is None else D
    W = cfg["W"] if W is None else W
    state = cfg["state"] if state is None else state
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg["seed"] if seed is None else seed)
    cu = None
    N = B
    if lengths is not None:
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        B, T, N = 1, int(cu[-1]), len(lengths)
    x = torch.randn((B, T, D), generator=gen, device=device).to(torch.bfloat16)
    weight = torch.empty((D, W), device=device).uniform_(-W ** -0.5, W ** -0.5, generator=gen)
    b = torch.empty((D,), device=device).uniform_(-W ** -0.5, W ** -0.5, generator=gen) if bias else None
    s0 = torch.randn((N, W - 1, D), generator=gen, device=device) if state else None
    return dict(x=x, weight=weight, bias=b, conv_state=s0, cu_seqlens=cu, B=B, T=T, D=D, W=W, N=N)


def make_decode_conv_inputs(B: int = 256, H: int = 96, W: int = 4, *, device="cpu", seed: int = 8,
                            history: bool = True, logits: bool = False) -> dict:
    """Seeded inputs of one decode step with the short convolutions fused: the decode
    workload's inputs at [B, H, 128] (make_logit_inputs' with ``logits``), q, k, v
    replaced by raw projections, plus conv_weight (three [H*128, W] fp32) and
    conv_state (three [B, W-1, H*128] fp32, or None without ``history``)."""
    make = make_logit_inputs if logits else make_inputs
    d = make("decode", device, B=B, H=H, seed=seed)
    d = {n: (t.squeeze(1) if torch.is_tensor(t) and t.dim() >= 3 and n != "initial_state" else t)
         for n, t in d.items()}
    gen = torch.Generator(device=device)
    gen.manual_seed(30_000 + seed)
    D = H * d["K"]
    d["q"], d["k"], d["v"] = (torch.randn((B, H, d["K"]), generator=gen, device=device).to(torch.bfloat16)
                              for _ in range(3))
    d["conv_weight"] = tuple(torch.empty((D, W), device=device).uniform_(-W ** -0.5, W ** -0.5, generator=gen)
                             for _ in range(3))
    d["conv_state"] = tuple(torch.randn((B, W - 1, D), generator=gen, device=device).to(torch.bfloat16).float()
                            for _ in range(3)) if history else None
    d["W"] = W
    return d
