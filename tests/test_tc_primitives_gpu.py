"""GPU unit test of the tcgen05 building blocks (operand layouts, A in TMEM, negate,
accumulate) that the tensor-core prefill kernel is built from.  The probe kernel in
tests/csrc/tc_primitives.cu is compiled here with nvcc for sm_103a."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "tc_primitives.cu")
CSRC = os.path.join(ROOT, "kimi_delta_attention_gated_gb300", "csrc")
OUT = os.path.join(ROOT, "_build", "libtc_primitives.so")


@pytest.fixture(scope="module")
def probe():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < max(os.path.getmtime(SRC),
                                                               os.path.getmtime(os.path.join(CSRC, "kda_tc_ptx.cuh"))):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", "-I", CSRC, SRC, "-o", OUT], check=True)
    lib = ctypes.CDLL(OUT)
    lib.tc_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                             ctypes.c_void_p]
    lib.tc_probe.restype = ctypes.c_int
    return lib


CASES = {  # which: (K, N, negate second half)
    0: (128, 64, False),
    1: (64, 64, False),
    2: (64, 128, False),
    3: (64, 64, False),
    4: (128, 64, True),
    5: (64, 128, False),
}


def test_bounded_wait_reports_timeout(probe):
    """A wait on an mbarrier that nothing arrives on gives up after its poll bound and
    reports it; the context stays usable (the next launch still computes correctly)."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    A = torch.zeros(128, 128, device="cuda", dtype=torch.bfloat16)
    D = torch.zeros(128, 64, device="cuda")
    rc = probe.tc_probe(6, A.data_ptr(), A.data_ptr(), D.data_ptr(), err.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(err.item()) == 2
    test_tc_primitive(probe, 0)


@pytest.mark.parametrize("which", sorted(CASES))
def test_tc_primitive(probe, which):
    K, N, neg = CASES[which]
    g = torch.Generator(device="cuda")
    g.manual_seed(100 + which)
    A = torch.randn(128, 128, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(128, 128, device="cuda", generator=g).to(torch.bfloat16)
    D = torch.full((128, N), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe(which, A.data_ptr(), B.data_ptr(), D.data_ptr(), err.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(err.item()) == 0, "mbarrier wait timed out"
    a, b = A.double()[:, :K], B.double()[:N, :K]
    if neg:
        ref = a[:, :64] @ b[:, :64].T - a[:, 64:] @ b[:, 64:].T
    else:
        ref = a @ b.T
    diff = (D.double() - ref).abs().max().item()
    assert diff <= 1e-3 * ref.abs().max().item(), f"case {which}: max diff {diff}"
