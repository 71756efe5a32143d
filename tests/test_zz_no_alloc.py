"""GPU test of kda_chunk_fwd_noalloc, the prefill entry point that allocates nothing.

It serves callers that cannot hand the library a workspace (a fixed operator or plugin
interface that passes only tensors, a path where device allocation is not allowed): its
scratch is a fixed array in the library's own device memory.  The test calls it through
the C ABI twice in a row, on two different prompts (so the second call finds the first
one's contents in the shared array), and compares each result with kda_chunk_fwd given a
workspace, within the parity tolerance of the other tests; a call too large for the array
must be refused.  This file is collected last so that a failure here leaves every other
test already run."""
import ctypes

import pytest
import torch

import kimi_delta_attention_gated_gb300 as kda
from kimi_delta_attention_gated_gb300.inputs import make_inputs
from tests.gpu_helpers import PARITY, rel_err

pytestmark = pytest.mark.gpu
BF16, F32, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    from kimi_delta_attention_gated_gb300 import build
    build.build()
    return kda._load()


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(lib, d, o, fs):
    cu = d.get("cu_seqlens")
    cu_d = None if cu is None else cu.to("cuda", torch.int32)
    cu_h = None if cu is None else cu.to(torch.int32).contiguous()
    n_seqs = 0 if cu is None else cu.numel() - 1
    st = torch.cuda.current_stream().cuda_stream
    return lib.kda_chunk_fwd_noalloc(
        ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), BF16, ptr(d["g"]), ptr(d["beta"]), ptr(d.get("initial_state")),
        ptr(fs), ptr(o), F32, ptr(cu_d), ptr(cu_h), n_seqs, d["B"], d["T"], d["H"], d["K"], d["V"], 64,
        d["scale"], 1, None, BF16, None, 1e-5, None, 1, ctypes.c_void_p(st))


def test_noalloc_matches_workspace_entry_two_calls(lib):
    prompts = [make_inputs("varlen", device="cuda", lengths=[200, 0, 331], H=8),
               make_inputs("prefill", device="cuda", T=520, H=6)]
    for d in prompts:
        o = torch.empty((d["B"], d["T"], d["H"], d["V"]), device="cuda")
        fs = torch.empty((d["N"], d["H"], d["K"], d["V"]), device="cuda")
        assert call_noalloc(lib, d, o, fs) == 0, lib.kda_last_error()
        ws = torch.empty(kda.workspace_size(d["B"], d["T"], d["H"], 0 if d["cu_seqlens"] is None else d["N"]),
                         dtype=torch.uint8, device="cuda")
        ref_o, ref_s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("initial_state"),
                                     scale=d["scale"], cu_seqlens=d.get("cu_seqlens"), mode="tensor", workspace=ws)
        torch.cuda.synchronize()
        assert rel_err(o, ref_o) <= PARITY
        assert rel_err(fs, ref_s) <= PARITY
    kda.device_status()


def test_noalloc_refuses_a_call_beyond_its_array(lib):
    """8192 tokens at 96 heads need 129 x 96 blobs of 32 KiB, more than the fixed 64 MiB."""
    d = make_inputs("prefill", device="cuda", T=8192, H=96)
    o = torch.empty((1, 8192, 96, 128), device="cuda")
    fs = torch.empty((1, 96, 128, 128), device="cuda")
    assert call_noalloc(lib, d, o, fs) == UNSUPPORTED
    assert b"fixed workspace" in lib.kda_last_error()
