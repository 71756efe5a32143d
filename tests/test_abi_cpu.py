"""CPU checks of the C ABI: libkda loads, exports every symbol include/*.h declares,
and rejects bad arguments on the host with a defined status before launching
anything.  No test here touches a GPU: the device pointers are fake aligned
addresses that validation never dereferences."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED = 0, 1, 2
BF16, F32 = 0, 1
FAKE = 0x10000000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    from kimi_delta_attention_gated_gb300 import build as b
    b.build()
    from kimi_delta_attention_gated_gb300 import _load
    return _load()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names.update(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for fn in ("kda_chunk_fwd", "kda_recurrent_fwd", "kda_recurrent_step", "kda_gated_rmsnorm",
               "kda_short_conv_fwd", "kda_device_status", "kda_set_wait_limit"):
        assert fn in names


def test_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, f"libkda does not export {missing}"


def test_version_and_status_strings(lib):
    assert lib.kda_version() >= 10000
    lib.kda_status_string.restype = ctypes.c_char_p
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(1) == b"KDA_ERR_INVALID_ARG"
    assert lib.kda_status_string(99) == b"KDA_ERR_UNKNOWN"


SPAN = 1 << 24  # fake tensors of one call lie this far apart, so that none overlaps another


def fake(i):
    return FAKE + i * SPAN


def chunk_call(lib, **over):
    a = dict(q=fake(0), k=fake(1), v=fake(2), qkv=BF16, g=fake(3), beta=fake(4), s0=None, sT=None, o=fake(5),
             odt=F32, cu=None, cu_host=None, n_seqs=0, B=1, T=64, H=2, K=128, V=128, chunk=64, scale=0.088,
             l2=1, gate=None, gdt=BF16, w=None, eps=1e-5, y=None, ws=None, ws_bytes=0, mode=0)
    a.update(over)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["qkv"], a["g"], a["beta"], a["s0"], a["sT"], a["o"],
                             a["odt"], a["cu"], a["cu_host"], a["n_seqs"], a["B"], a["T"], a["H"], a["K"],
                             a["V"], a["chunk"], a["scale"], a["l2"], a["gate"], a["gdt"], a["w"], a["eps"],
                             a["y"], a["ws"], a["ws_bytes"], a["mode"], None)


def cu_host(values):
    arr = np.asarray(values, np.int32)
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), INVALID),
    (dict(beta=None), INVALID),
    (dict(o=None), INVALID),                       # o may be NULL only with the gated norm
    (dict(K=100), UNSUPPORTED),
    (dict(V=256), UNSUPPORTED),
    (dict(chunk=48), UNSUPPORTED),
    (dict(qkv=7), UNSUPPORTED),
    (dict(odt=3), UNSUPPORTED),
    (dict(q=FAKE + 4), INVALID),                   # misaligned
    (dict(o=FAKE + 8), INVALID),
    (dict(H=0), INVALID),
    (dict(T=-1), INVALID),
    (dict(B=0), INVALID),
    (dict(mode=9), INVALID),
    (dict(mode=1, K=32, V=32), UNSUPPORTED),       # tensor path only at K = V = 128
    (dict(mode=1, chunk=32), UNSUPPORTED),
    (dict(mode=1, qkv=F32), UNSUPPORTED),
    (dict(gate=FAKE), INVALID),                    # gate without norm_w / y
    (dict(gate=FAKE, w=FAKE, y=FAKE, eps=0.0), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(cu=FAKE, n_seqs=0), INVALID),
    (dict(cu=FAKE, n_seqs=2, B=2), INVALID),       # varlen needs B == 1
    (dict(cu_host=FAKE), INVALID),                 # host copy without the device array
])
def test_chunk_fwd_rejects(lib, over, code):
    assert chunk_call(lib, **over) == code
    assert lib.kda_last_error()


@pytest.mark.parametrize("over,what", [
    (dict(o=fake(0) + 4096), b"o must not overlap q"),             # o inside q
    (dict(o=fake(3) - 16), b"o must not overlap g"),               # o runs into g
    (dict(gate=fake(6), w=fake(7), y=fake(2)), b"y must not overlap v"),
    (dict(gate=fake(6), w=fake(7), y=fake(5) + 1024), b"o must not overlap y"),
    (dict(s0=fake(8), sT=fake(8) + 64), b"partly overlap"),         # states offset, not equal
    (dict(sT=fake(1) + 256), b"final state must not overlap k"),
    (dict(s0=fake(8), o=fake(8)), b"o must not overlap the state"),
])
def test_chunk_fwd_rejects_overlapping_buffers(lib, over, what):
    """The prefill kernels read their inputs chunk by chunk while writing outputs, so an
    output sharing bytes with an input (or with another output) is refused before any
    launch; only final_state == initial_state (the same pointer) is allowed."""
    assert chunk_call(lib, **over) == INVALID
    assert what in lib.kda_last_error()


def test_workspace_size(lib):
    """32 KiB per (chunk slot, head) for ceil(rows / 64) + N slots (N = n_seqs in varlen mode),
    then a 4-byte flag per (slot, head) and a 4-byte progress word per (sequence, head), each
    array rounded up to 256 bytes."""
    lib.kda_chunk_workspace_size.restype = ctypes.c_size_t
    r256 = lambda x: (x + 255) // 256 * 256
    size = lambda slots, H, N: slots * H * 32768 + r256(slots * H * 4) + r256(N * H * 4)
    assert lib.kda_chunk_workspace_size(1, 8192, 96, 0) == size(128 + 1, 96, 1)
    assert lib.kda_chunk_workspace_size(2, 65536, 96, 0) == size(2048 + 2, 96, 2)
    assert lib.kda_chunk_workspace_size(1, 100, 3, 4) == size(2 + 4, 3, 4)
    assert lib.kda_chunk_workspace_size(0, 64, 2, 0) == 0


@pytest.mark.parametrize("over,what", [
    (dict(ws=fake(8), ws_bytes=1024), b"workspace holds"),            # too small
    (dict(ws=fake(8) + 4, ws_bytes=1 << 22), b"16-byte aligned"),
    (dict(ws=fake(5), ws_bytes=1 << 22), b"workspace must not overlap o"),
])
def test_chunk_fwd_rejects_bad_workspace(lib, over, what):
    assert chunk_call(lib, **over) == INVALID
    assert what in lib.kda_last_error()


def test_set_wait_limit_range(lib):
    lib.kda_set_wait_limit.argtypes = [ctypes.c_int64]
    assert lib.kda_set_wait_limit(ctypes.c_int64(1 << 33)) == INVALID
    assert lib.kda_set_wait_limit(ctypes.c_int64(0)) == OK
    assert lib.kda_set_wait_limit(ctypes.c_int64(-1)) == OK  # back to the default


@pytest.mark.parametrize("values,T", [([0, 5, 3, 8], 8), ([1, 4, 8], 8), ([0, 4, 7], 8), ([0, -1, 8], 8)])
def test_chunk_fwd_rejects_bad_cu_seqlens(lib, values, T):
    arr, ptr = cu_host(values)
    assert chunk_call(lib, cu=FAKE, cu_host=ptr, n_seqs=len(values) - 1, T=T) == INVALID
    assert b"cu_seqlens" in lib.kda_last_error()


def test_recurrent_step_rejects(lib):
    f = lib.kda_recurrent_step
    base = [FAKE, FAKE, FAKE, BF16, FAKE, FAKE, FAKE, FAKE, FAKE, F32, 4, 2, 128, 128, 0.088, 1, None, BF16,
            None, 1e-5, None, None]
    bad_state = list(base)
    bad_state[7] = None  # state_out
    assert f(*bad_state) == INVALID
    bad_dim = list(base)
    bad_dim[12] = 96
    assert f(*bad_dim) == UNSUPPORTED
    misaligned = list(base)
    misaligned[6] = FAKE + 4
    assert f(*misaligned) == INVALID


def conv_step_call(lib, *, W=4, K=128, s_in=None, s_out=None, w=None, gates="plain", q=None):
    """kda_recurrent_step_conv on fake device pointers (B=4, H=2); returns the status."""
    P3 = ctypes.c_void_p * 3
    w = w or [fake(20), fake(21), fake(22)]
    s_in = [fake(23), fake(24), fake(25)] if s_in is None else s_in
    s_out = [fake(26), fake(27), fake(28)] if s_out is None else s_out
    g = (fake(4), fake(5), None, BF16, None, None, -5.0, None, BF16)
    lg = (None, None, fake(10), BF16, fake(11), fake(12), -5.0, fake(13), BF16)
    both = (fake(4), fake(5), fake(10), BF16, fake(11), fake(12), -5.0, fake(13), BF16)
    gate_args = {"plain": g, "logits": lg, "both": both}[gates]
    return lib.kda_recurrent_step_conv(
        q or fake(1), fake(2), fake(3), BF16, P3(*w), W, None if s_in == "none" else P3(*s_in),
        None if s_out == "none" else P3(*s_out), *gate_args, fake(6), fake(7), fake(8), F32, 4, 2, K, 128, 0.088,
        1, fake(14), BF16, fake(15), 1e-5, fake(16), None)


def test_recurrent_step_conv_rejects(lib):
    assert conv_step_call(lib, gates="both") == INVALID
    assert b"either g and beta" in lib.kda_last_error()
    assert conv_step_call(lib, W=5) == UNSUPPORTED
    assert conv_step_call(lib, W=1) == UNSUPPORTED
    assert conv_step_call(lib, K=64) == UNSUPPORTED
    assert conv_step_call(lib, s_out="none") == INVALID
    assert conv_step_call(lib, s_out=[fake(26), None, fake(28)]) == INVALID
    assert conv_step_call(lib, s_in=[fake(23), None, fake(25)]) == INVALID
    assert b"all three histories or none" in lib.kda_last_error()
    assert conv_step_call(lib, w=[fake(20), fake(21) + 4, fake(22)]) == INVALID  # misaligned
    # a new history over q, over another filter's history, or partly over its own
    assert conv_step_call(lib, s_out=[fake(26), fake(1), fake(28)]) == INVALID
    assert conv_step_call(lib, s_out=[fake(24), fake(27), fake(28)]) == INVALID
    assert conv_step_call(lib, s_out=[fake(23) + 16, fake(27), fake(28)]) == INVALID
    assert b"conv_state_in[0] itself" in lib.kda_last_error()
    assert conv_step_call(lib, s_out=[fake(26), fake(26) + 1024, fake(28)]) == INVALID
    # a weight under the step's output y
    assert conv_step_call(lib, w=[fake(20), fake(16), fake(22)]) == INVALID


def test_chunk_fwd_host_rejects(lib):
    f = lib.kda_chunk_fwd_host
    need = lib.kda_chunk_fwd_host_workspace_size(1, 2, 128, 128, 256)
    assert need > 2 * 256 * 2 * (3 * 128 * 4)  # two buffers of every segment tensor
    assert lib.kda_chunk_fwd_host_workspace_size(0, 2, 128, 128, 256) == 0

    def call(seg=256, ws=fake(30), ws_bytes=need, o=fake(8), chunk=64):
        return f(fake(1), fake(2), fake(3), BF16, fake(4), fake(5), None, fake(7), o, F32, 1, 1000, 2, 128, 128,
                 chunk, 0.088, 1, None, BF16, None, 1e-5, None, seg, ws, ws_bytes, 0, None)
    assert call(seg=100) == INVALID
    assert b"multiple of 64" in lib.kda_last_error()
    assert call(ws_bytes=4096) == INVALID
    assert b"kda_chunk_fwd_host_workspace_size" in lib.kda_last_error()
    assert call(ws=fake(30) + 16) == INVALID  # 256-byte alignment
    assert call(ws=None) == INVALID
    assert call(chunk=48) == UNSUPPORTED
    assert call(o=fake(2) + 64) == INVALID  # o over the host k
    assert b"must not overlap" in lib.kda_last_error()
    assert call(o=None) == INVALID


def test_recurrent_fwd_rejects(lib):
    f = lib.kda_recurrent_fwd
    base = [FAKE, FAKE, FAKE, BF16, FAKE, FAKE, None, None, FAKE, F32, None, None, None, 0, 1, 16, 2, 64, 64,
            0.125, 1, None, BF16, None, 1e-5, None, None]
    bad_states = list(base)
    bad_states[10] = FAKE + 4  # misaligned per-token states
    assert f(*bad_states) == INVALID
    no_v = list(base)
    no_v[2] = None
    assert f(*no_v) == INVALID


def test_gated_rmsnorm_rejects(lib):
    f = lib.kda_gated_rmsnorm
    assert f(FAKE, F32, FAKE, BF16, FAKE, ctypes.c_float(1e-5), FAKE, F32, ctypes.c_int64(4), 2, 100, None) == UNSUPPORTED
    assert f(FAKE, F32, FAKE, BF16, FAKE, ctypes.c_float(0.0), FAKE, F32, ctypes.c_int64(4), 2, 128, None) == INVALID
    assert f(None, F32, FAKE, BF16, FAKE, ctypes.c_float(1e-5), FAKE, F32, ctypes.c_int64(4), 2, 128, None) == INVALID
    # in place (o == y) with different element sizes would corrupt the buffer
    assert f(FAKE, BF16, FAKE, BF16, FAKE, ctypes.c_float(1e-5), FAKE, F32, ctypes.c_int64(4), 2, 128, None) == INVALID


def test_launch_count_starts_at_zero(lib):
    assert lib.kda_launch_count() == 0


def test_python_binding_fails_loudly_without_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    import kimi_delta_attention_gated_gb300 as kda
    q = torch.zeros(1, 4, 1, 32, dtype=torch.bfloat16)
    with pytest.raises(Exception):
        kda.chunk_fwd(q, q, q, torch.zeros(1, 4, 1, 32), torch.zeros(1, 4, 1), chunk=16)


def conv_call(lib, **over):
    a = dict(x=FAKE, xdt=BF16, w=FAKE, b=None, s0=None, sT=None, y=FAKE + (1 << 24), ydt=BF16, cu=None,
             cu_host=None, n_seqs=0, B=1, T=64, D=256, W=4, act=1)
    a.update(over)
    return lib.kda_short_conv_fwd(a["x"], a["xdt"], a["w"], a["b"], a["s0"], a["sT"], a["y"], a["ydt"], a["cu"],
                                  a["cu_host"], a["n_seqs"], a["B"], a["T"], a["D"], a["W"], a["act"], None)


@pytest.mark.parametrize("over,code", [
    (dict(x=None), INVALID),
    (dict(w=None), INVALID),
    (dict(W=5), UNSUPPORTED),
    (dict(W=1), UNSUPPORTED),
    (dict(D=100), UNSUPPORTED),                     # D must be a multiple of 8
    (dict(D=0), INVALID),
    (dict(xdt=5), UNSUPPORTED),
    (dict(act=2), INVALID),
    (dict(x=FAKE + 4), INVALID),                    # misaligned
    (dict(y=FAKE), INVALID),                        # y overlaps x
    (dict(s0=FAKE + (1 << 26), sT=FAKE + (1 << 26)), INVALID),   # in place only for a decode step
    (dict(cu=FAKE, n_seqs=0), INVALID),
    (dict(cu=FAKE, n_seqs=2, B=2), INVALID),
    (dict(cu_host=FAKE), INVALID),
    (dict(B=70000, T=40000), INVALID),              # B*T beyond int32
])
def test_short_conv_rejects(lib, over, code):
    assert conv_call(lib, **over) == code
    assert lib.kda_last_error()


def test_short_conv_rejects_bad_cu_seqlens(lib):
    arr, ptr = cu_host([0, 9, 4, 64])
    assert conv_call(lib, cu=FAKE, cu_host=ptr, n_seqs=3) == INVALID


def test_o_proj_rejects(lib):
    f = lib.kda_o_proj
    rows = ctypes.c_int64
    assert f(None, fake(1), fake(2), BF16, rows(4), 64, 128, None) == INVALID
    assert f(fake(0), fake(1), fake(2), BF16, rows(4), 96, 128, None) == UNSUPPORTED   # in_features % 64
    assert f(fake(0), fake(1), fake(2), BF16, rows(4), 64, 64, None) == UNSUPPORTED    # out_features % 128
    assert f(fake(0), fake(1), fake(2), 9, rows(4), 64, 128, None) == UNSUPPORTED
    assert f(fake(0) + 4, fake(1), fake(2), BF16, rows(4), 64, 128, None) == INVALID   # misaligned
    assert f(fake(0), fake(1), fake(0) + 256, BF16, rows(4), 64, 128, None) == INVALID  # out overlaps y
    assert f(None, None, None, BF16, rows(0), 64, 128, None) == OK                      # nothing to do
