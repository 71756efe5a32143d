"""Shared helpers for the GPU parity tests: move seeded inputs to the device, run the
fp64 oracle on (a sample of) the same bits, and measure max|diff| / rms(oracle)."""
import numpy as np
import torch

import oracle

PARITY = 5e-3      # bf16 q/k/v, fp32 state: max|diff| / rms(oracle), outputs and final state
FP32_TOL = 1e-4    # fp32 paths against each other / against the oracle


def rel_err(a, ref):
    a = np.asarray(a.detach().float().cpu().numpy() if torch.is_tensor(a) else a, np.float64)
    ref = np.asarray(ref.detach().double().cpu().numpy() if torch.is_tensor(ref) else ref, np.float64)
    assert a.shape == ref.shape, (a.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert np.all(np.isfinite(a)), "non-finite values in the CUDA result"
    return float(np.abs(a - ref).max()) / max(rms, 1e-30)


def to_dev(d, device="cuda"):
    out = {}
    for k, v in d.items():
        out[k] = v.to(device) if torch.is_tensor(v) and k != "cu_seqlens" else v
    return out


def np32(t):
    return t.detach().float().cpu().numpy()


def oracle_run(d, heads=None, seqs=None, return_states=False):
    """Oracle on inputs dict d (any device), optionally restricted to some heads / sequences.
    Returns (o [B,T,H',V], final [N',H',K,V][, states])."""
    hs = slice(None) if heads is None else list(heads)
    q, k, v, g, beta = (np32(d[n])[:, :, hs] for n in ("q", "k", "v", "g", "beta"))
    s0 = d.get("initial_state")
    s0 = None if s0 is None else np32(s0)[:, hs].astype(np.float64)
    cu = d.get("cu_seqlens")
    if cu is not None:
        cu = cu.cpu().numpy().astype(np.int64)
    if seqs is not None:
        if cu is None:  # dense batch rows
            q, k, v, g, beta = (x[seqs] for x in (q, k, v, g, beta))
            if s0 is not None:
                s0 = s0[seqs]
        else:
            raise ValueError("sample varlen inputs by slicing cu_seqlens in the test")
    return oracle.recurrent(q, k, v, g, beta, s0, scale=d["scale"], cu_seqlens=cu,
                            return_states=return_states)


def assert_bf16_close(a, ref, c):
    """A bf16 output against the fp64 oracle, element by element: within the rounding to
    bf16 (half an ulp is 2^-9 relative; 2^-8 leaves a factor two) plus c * rms(oracle)
    for the path's own fp32 error before the rounding."""
    a = np.asarray(a.detach().double().cpu().numpy() if torch.is_tensor(a) else a, np.float64)
    ref = np.asarray(ref, np.float64)
    a = a.reshape(ref.shape)
    assert np.all(np.isfinite(a)), "non-finite values in the CUDA result"
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = 2.0 ** -8 * np.abs(ref) + c * rms
    excess = np.abs(a - ref) - bound
    worst = int(np.argmax(excess))
    assert excess.flat[worst] <= 0, (f"element {np.unravel_index(worst, ref.shape)}: got {a.flat[worst]!r}, "
                                     f"oracle {ref.flat[worst]!r}, bound {bound.flat[worst]!r}")
