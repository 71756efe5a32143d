"""GPU unit test of the logit -> gate conversions the kernels share (kda_internal.cuh):
g = max(lower, -exp(A_log) * softplus(z + dt_bias)) and beta = sigmoid(b), evaluated on
the device through tests/csrc/gate_probe.cu and compared, element by element, with the
same formulas in fp64 (softplus through numpy's log1p).  Reading of the combining line:
Kimi-K3 atlas "gate-project (decode, P = 1000)", section "Code" (A_log, dt_bias,
gate_lower_bound, b_proj)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "gate_probe.cu")
CSRC = os.path.join(ROOT, "kimi_delta_attention_gated_gb300", "csrc")
OUT = os.path.join(ROOT, "_build", "libgate_probe.so")


@pytest.fixture(scope="module")
def probe():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    deps = [SRC, os.path.join(CSRC, "kda_internal.cuh")]
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < max(os.path.getmtime(d) for d in deps):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", "-I", CSRC, "-I", os.path.join(ROOT, "include"), SRC, "-o", OUT],
                       check=True)
    lib = ctypes.CDLL(OUT)
    lib.gate_probe.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p]
    lib.gate_probe.restype = ctypes.c_int
    return lib


def run(probe, x, a_h, lower):
    xd = torch.tensor(x, dtype=torch.float32, device="cuda")
    g = torch.empty_like(xd)
    b = torch.empty_like(xd)
    assert probe.gate_probe(xd.data_ptr(), xd.numel(), a_h, lower, g.data_ptr(), b.data_ptr(),
                            torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    return xd.double().cpu().numpy(), g.double().cpu().numpy(), b.double().cpu().numpy()


def softplus64(x):
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


@pytest.mark.parametrize("a_h", [1.0, 16.0])
def test_softplus_gate_relative_accuracy(probe, a_h):
    """Across logits from -20 to 20 (the decay logits of the workloads sit near -4, where
    e^z is small) g keeps fp32-level relative accuracy: at most 4e-6 of |g|, the error of
    the fast exponential for arguments up to 20, with no floor (lower = -inf)."""
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-20.0, 20.0, 40001), rng.normal(-4.0, 1.0, 100000)]).astype(np.float32)
    xs, g, _ = run(probe, x, a_h, float("-inf"))
    ref = -a_h * softplus64(xs)
    rel = np.abs(g - ref) / np.abs(ref)
    assert rel.max() <= 4e-6, f"max relative error {rel.max():.3e} at z = {xs[rel.argmax()]}"


def test_gate_floor_and_beta(probe):
    """The lower bound is a floor on g, applied exactly; beta = sigmoid(b) to within
    fp32 rounding of the fast exponential and divide (absolute 5e-7 on values in (0, 1))."""
    x = np.linspace(-12.0, 12.0, 24001).astype(np.float32)
    xs, g, b = run(probe, x, 16.0, -5.0)
    raw = -16.0 * softplus64(xs)
    ref = np.maximum(-5.0, raw)
    assert (g >= -5.0).all()                               # the floor is never crossed
    clearly_below = raw < -5.0 * (1 + 1e-5)                # floored whatever the rounding
    assert clearly_below.any() and (g[clearly_below] == -5.0).all()
    assert (np.abs(g - ref) <= 4e-6 * np.abs(ref)).all()
    assert np.abs(b - 1.0 / (1.0 + np.exp(-xs))).max() <= 5e-7
