"""Kimi Delta Attention core on GB300: Python binding of libkda.

Thin ctypes marshalling over the C ABI declared in include/kda.h: every step of
the computation runs in libkda's CUDA kernels; torch only allocates device memory
and supplies the current stream.  There is no CPU fallback: calling any function
without a built libkda (or without a GPU) raises.

Entry points (same names as the C ABI, minus the ``kda_`` prefix):
  chunk_fwd       chunked prefill  (q, k, v, g, beta, initial_state) -> (o, final_state[, y])
  recurrent_fwd   token-by-token form over T tokens, optional per-token states
  recurrent_step  one decode token per sequence with the fused gated norm
  gated_rmsnorm   y = RMSNorm_v(o) * w * sigmoid(gate) per (token, head)

Inputs may live on the host: they are copied to the current CUDA device, and the
results are copied back to the host, which makes the call end-to-end.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["chunk_fwd", "chunk_fwd_logits", "recurrent_fwd", "recurrent_step", "recurrent_step_logits",
           "gated_rmsnorm", "short_conv", "o_proj", "launch_count", "device_status", "set_wait_limit",
           "workspace_size", "release_workspaces", "prepass_hits",
           "library_path", "KDAError", "MODE_AUTO", "MODE_TENSOR", "MODE_FP32", "MODE_SPLIT"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libkda.so")
_lib = None
_lock = threading.Lock()

BF16, F32 = 0, 1
MODE_AUTO, MODE_TENSOR, MODE_FP32, MODE_SPLIT = 0, 1, 2, 3
_MODES = {"auto": MODE_AUTO, "tensor": MODE_TENSOR, "fp32": MODE_FP32, "split": MODE_SPLIT}
_STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
           4: "KDA_ERR_TIMEOUT"}


class KDAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libkda.so is not built ({_LIB_PATH}); run __graft_entry__.build() "
                               "or python kimi_delta_attention_gated_gb300/build.py")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        Z = ctypes.c_size_t
        lib.kda_chunk_fwd.argtypes = [P, P, P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I,
                                      P, I, P, F, P, P, Z, I, P]
        lib.kda_chunk_fwd_noalloc.argtypes = [P, P, P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I,
                                              P, I, P, F, P, I, P]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_workspace_size.argtypes = [I, I, I, I]
        lib.kda_chunk_workspace_size.restype = Z
        lib.kda_chunk_fwd_host_workspace_size.argtypes = [I, I, I, I, I]
        lib.kda_chunk_fwd_host_workspace_size.restype = Z
        lib.kda_chunk_fwd_host.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, I, P, F, P, I,
                                           P, Z, I, P]
        lib.kda_chunk_fwd_logits_host.argtypes = [P, P, P, I, P, I, P, P, F, P, I, P, P, P, I, I, I, I, I, I, I,
                                                  F, I, P, I, P, F, P, I, P, Z, I, P]
        lib.kda_recurrent_fwd.argtypes = [P, P, P, I, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, F, I,
                                          P, I, P, F, P, P]
        lib.kda_recurrent_step.argtypes = [P, P, P, I, P, P, P, P, P, I, I, I, I, I, F, I, P, I, P, F,
                                           P, P]
        lib.kda_gated_rmsnorm.argtypes = [P, I, P, I, P, F, P, I, ctypes.c_int64, I, I, P]
        lib.kda_short_conv_fwd.argtypes = [P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, I, P]
        lib.kda_chunk_fwd_logits.argtypes = [P, P, P, I, P, I, P, P, F, P, I, P, P, P, I, P, P, I, I, I, I, I, I,
                                             I, F, I, P, I, P, F, P, P, Z, I, P]
        lib.kda_recurrent_step_logits.argtypes = [P, P, P, I, P, I, P, P, F, P, I, P, P, P, I, I, I, I, I, F, I,
                                                  P, I, P, F, P, P]
        lib.kda_o_proj.argtypes = [P, P, P, I, ctypes.c_int64, I, I, P]
        P3 = ctypes.POINTER(ctypes.c_void_p)  # a host array of three device pointers, or NULL
        lib.kda_recurrent_step_conv.argtypes = [P, P, P, I, P3, I, P3, P3, P, P, P, I, P, P, F, P, I, P, P, P, I,
                                                I, I, I, I, F, I, P, I, P, F, P, P]
        for fn in ("kda_chunk_fwd", "kda_recurrent_fwd", "kda_recurrent_step", "kda_gated_rmsnorm",
                   "kda_short_conv_fwd", "kda_chunk_fwd_logits", "kda_recurrent_step_logits", "kda_o_proj",
                   "kda_recurrent_step_conv", "kda_chunk_fwd_host", "kda_chunk_fwd_logits_host"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.kda_device_status.argtypes = [P]
        lib.kda_device_status.restype = ctypes.c_int
        lib.kda_chunk_prepass_hits.argtypes = [P, ctypes.POINTER(ctypes.c_uint64)]
        lib.kda_chunk_prepass_hits.restype = ctypes.c_int
        lib.kda_set_wait_limit.argtypes = [ctypes.c_int64]
        lib.kda_set_wait_limit.restype = ctypes.c_int
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_launch_count.restype = ctypes.c_uint64
        lib.kda_version.restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        raise KDAError(status, _load().kda_last_error().decode())


def launch_count() -> int:
    """Kernels libkda has launched in this process."""
    return int(_load().kda_launch_count())


def device_status(stream=None):
    """Synchronise the stream (default: the current one) and raise KDAError with
    KDA_ERR_TIMEOUT if a bounded wait inside a kernel gave up since the last check
    (those outputs hold NaN).  Clears the device's counters."""
    st = ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
    _check(_load().kda_device_status(st))


def prepass_hits(stream=None) -> int:
    """Chunks of the concurrent prefill form that took their grams and UT transform from the
    pre-pass since the last call (synchronises the stream; clears the device's counter)."""
    st = ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
    n = ctypes.c_uint64(0)
    _check(_load().kda_chunk_prepass_hits(st, ctypes.byref(n)))
    return int(n.value)


def set_wait_limit(polls):
    """Bound on the streaming kernels' first-line waits (None or a negative value: the
    default; 0: every such wait gives up at once, for tests of the failure handling)."""
    _check(_load().kda_set_wait_limit(-1 if polls is None else int(polls)))


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _prep(t, device, dtype=None):
    """Contiguous device tensor (host tensors are copied; pinned ones asynchronously)."""
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        t = t.to(dtype)
    if t.device.type != "cuda":
        t = t.to(device, non_blocking=t.is_pinned())
    return t.contiguous()


def _device_of(*ts):
    for t in ts:
        if t is not None and t.device.type == "cuda":
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _cu(cu_seqlens, device):
    if cu_seqlens is None:
        return None, None, 0
    host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
    dev = cu_seqlens.to(device=device, dtype=torch.int32).contiguous()
    return dev, host, host.numel() - 1


def _to_host(ts, host, dests=None):
    """Copy results back to the host: into the caller's host tensors when given
    (asynchronously when they are pinned, then the stream is synchronised)."""
    if not host:
        return ts
    out = []
    for i, t in enumerate(ts):
        dst = dests[i] if dests is not None else None
        if t is None:
            out.append(None)
        elif dst is not None:
            dst.copy_(t, non_blocking=dst.is_pinned())
            out.append(dst)
        else:
            out.append(t.to("cpu"))
    torch.cuda.current_stream().synchronize()
    return tuple(out)


def _dev_out(t):
    """A caller-provided output on the host is computed on the device first."""
    return None if (t is None or t.device.type != "cuda") else t


def chunk_fwd(q, k, v, g, beta, initial_state=None, *, scale=None, chunk=64, use_qk_l2norm=True,
              cu_seqlens=None, output_final_state=True, gate=None, norm_w=None, eps=1e-5,
              out_dtype=torch.float32, mode="auto", return_o=True, o=None, y=None, final_state=None,
              workspace=None):
    """Chunked prefill.  q, k [B,T,H,K]; v [B,T,H,V]; g [B,T,H,K] fp32; beta [B,T,H] fp32;
    initial_state [N,H,K,V] fp32 or None.  With ``cu_seqlens`` (int, n_seqs + 1) B must be 1.
    Returns (o, final_state) or, with ``gate``/``norm_w``, (o, final_state, y) where
    y [B,T,H*V] is the sigmoid-gated RMSNorm of o (o is None when return_o=False).
    Preallocated outputs may be passed as o / y / final_state (final_state may be
    initial_state itself for an in-place update).  ``workspace``: None (the fused one-kernel
    tensor-core form), a uint8 device tensor of at least workspace_size(...) bytes, or
    "auto" (a per-device buffer this binding keeps).  With a workspace the fused kernel is
    joined by a pre-pass on the SMs it leaves idle (fewer (sequence, head) units than SMs),
    which forms chunks' grams and UT transform ahead of it (the concurrent form); with
    ``mode="split"`` the pre-pass instead forms every chunk's first and a per-head chain
    kernel follows (the split form).  Every form gives the same bits.  The kept buffer is
    shared by every "auto" call on a device: calls on streams that may run at the same time
    need workspaces of their own."""
    return _chunk(q, k, v, (g, beta), None, initial_state, scale, chunk, use_qk_l2norm, cu_seqlens,
                  output_final_state, gate, norm_w, eps, out_dtype, mode, return_o, o, y, final_state, workspace)


def chunk_fwd_logits(q, k, v, g_logits, beta_logits, A_log, initial_state=None, *, dt_bias=None,
                     g_lower_bound=-5.0, scale=None, chunk=64, use_qk_l2norm=True, cu_seqlens=None,
                     output_final_state=True, gate=None, norm_w=None, eps=1e-5, out_dtype=torch.float32,
                     mode="auto", return_o=True, o=None, y=None, final_state=None, workspace=None):
    """chunk_fwd with g = max(g_lower_bound, -exp(A_log[h]) * softplus(g_logits + dt_bias)) and
    beta = sigmoid(beta_logits) computed inside the kernels.  g_logits [B,T,H,K] and
    beta_logits [B,T,H] in bf16 or fp32; A_log [H]; dt_bias [H,K] (or [H*K]) or None;
    g_lower_bound None for no floor."""
    lb = float("-inf") if g_lower_bound is None else float(g_lower_bound)
    return _chunk(q, k, v, None, (g_logits, beta_logits, A_log, dt_bias, lb), initial_state, scale, chunk,
                  use_qk_l2norm, cu_seqlens, output_final_state, gate, norm_w, eps, out_dtype, mode, return_o, o, y,
                  final_state, workspace)


def workspace_size(B, T, H, n_seqs=0) -> int:
    """Bytes of workspace the split tensor-core prefill needs (kda_chunk_workspace_size)."""
    return int(_load().kda_chunk_workspace_size(int(B), int(T), int(H), int(n_seqs)))


_CHUNK_WS = {}


def _chunk_workspace(spec, dev, B, T, H, n_seqs):
    """(pointer, bytes) of the workspace for one call: None -> the fused form."""
    if spec is None:
        return None, 0
    need = workspace_size(B, T, H, n_seqs)
    if isinstance(spec, str):
        if spec != "auto":
            raise ValueError('workspace must be "auto", None or a device tensor')
        key = dev.index if dev.index is not None else torch.cuda.current_device()
        ws = _CHUNK_WS.get(key)
        if ws is None or ws.numel() < need:
            _CHUNK_WS.pop(key, None)
            ws = _CHUNK_WS[key] = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        return ctypes.c_void_p(ws.data_ptr()), ws.numel()
    return ctypes.c_void_p(spec.data_ptr()), spec.numel() * spec.element_size()


def release_workspaces():
    """Drop the workspaces this binding keeps (the next call allocates again)."""
    _CHUNK_WS.clear()


def _pinned(t):
    return t if t.is_pinned() else t.pin_memory()


def _chunk_host_streamed(q, k, v, gb, lg, initial_state, scale, chunk, use_qk_l2norm, output_final_state, gate,
                         norm_w, eps, out_dtype, mode, return_o, o, y, final_state):
    """A host-resident dense prompt through kda_chunk_fwd_host (_logits_host): the library
    streams it through the device in HOST_SEGMENT-token segments, copies in and out on two
    streams of its own while the kernels run on the current stream.  Inputs are made
    page-locked (copied once if they are not); outputs are page-locked host tensors (or the
    caller's).  The fused kernel runs each segment; the result equals one device call."""
    lib = _load()
    dev = torch.device("cuda", torch.cuda.current_device())
    B, T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    pin = lambda t: None if t is None else _pinned(t.detach().contiguous())
    host32 = lambda t: None if t is None else t.detach().to("cpu", torch.float32).contiguous()
    q, k, v = pin(q), pin(k), pin(v)
    want_o = return_o or gate is None or o is not None
    o_h = (o if o is not None else torch.empty((B, T, H, V), dtype=out_dtype).pin_memory()) if want_o else None
    y_h = norm_h = None
    if gate is not None:
        gate = pin(gate)
        norm_h = host32(norm_w)
        y_h = y if y is not None else torch.empty((B, T, H * V), dtype=out_dtype).pin_memory()
    fs_h = final_state if final_state is not None else (
        torch.empty((B, H, K, V), dtype=torch.float32).pin_memory() if output_final_state else None)
    s0 = host32(initial_state)
    need = int(lib.kda_chunk_fwd_host_workspace_size(B, H, K, V, HOST_SEGMENT))
    key = ("host", dev.index)
    ws = _CHUNK_WS.get(key)
    if ws is None or ws.numel() < need:
        _CHUNK_WS.pop(key, None)
        ws = _CHUNK_WS[key] = torch.empty(need, dtype=torch.uint8, device=dev)
    mode_i = _MODES[mode] if isinstance(mode, str) else int(mode)
    tail = (_ptr(s0), _ptr(fs_h), _ptr(o_h), _dt(o_h if o_h is not None else y_h), B, T, H, K, V, int(chunk),
            float(scale), int(bool(use_qk_l2norm)), _ptr(gate), _dt(gate) if gate is not None else BF16, _ptr(norm_h),
            float(eps), _ptr(y_h), HOST_SEGMENT, ctypes.c_void_p(ws.data_ptr()), ws.numel(), mode_i, _stream())
    if lg is None:
        g, beta = pin(gb[0].to(torch.float32)), pin(gb[1].to(torch.float32))
        _check(lib.kda_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), *tail))
    else:
        z, b, A_log, dt_bias, lb = lg
        z, b, A_log, dt_bias = pin(z), pin(b), host32(A_log), host32(dt_bias)
        _check(lib.kda_chunk_fwd_logits_host(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(z), _dt(z), _ptr(A_log),
                                             _ptr(dt_bias), lb, _ptr(b), _dt(b), *tail))
    torch.cuda.current_stream().synchronize()  # the outputs are in host memory once the stream is done
    o_ret = o_h if return_o or gate is None else None
    if gate is not None:
        return o_ret, fs_h, y_h
    return o_ret, fs_h


def _logit_args(lg, dev):
    z, b, A_log, dt_bias, lb = lg
    z, b = _prep(z, dev), _prep(b, dev)
    A_log = _prep(A_log, dev, torch.float32)
    dt_bias = _prep(dt_bias, dev, torch.float32)
    return z, b, A_log, dt_bias, lb


# Host-resident prompts at least this long are streamed through the device in segments
# of HOST_SEGMENT tokens (a multiple of the 64-token chunk).
HOST_SEGMENT = 1024


def _chunk(q, k, v, gb, lg, initial_state, scale, chunk, use_qk_l2norm, cu_seqlens, output_final_state, gate,
           norm_w, eps, out_dtype, mode, return_o, o, y, final_state, workspace=None):
    lib = _load()
    host = q.device.type != "cuda"
    on_host = lambda t: t is None or t.device.type == "cpu"
    if (host and cu_seqlens is None and q.shape[1] >= 2 * HOST_SEGMENT and workspace is None
            and on_host(o) and on_host(y) and on_host(final_state) and torch.cuda.is_available()):
        return _chunk_host_streamed(q, k, v, gb, lg, initial_state, scale, chunk, use_qk_l2norm,
                                    output_final_state, gate, norm_w, eps, out_dtype, mode, return_o, o, y,
                                    final_state)
    dev = _device_of(q, k, v)
    dests = (o, final_state, y) if host else None
    if host:
        o, final_state, y = _dev_out(o), _dev_out(final_state), _dev_out(y)
    q, k, v = _prep(q, dev), _prep(k, dev), _prep(v, dev)
    initial_state = _prep(initial_state, dev, torch.float32)
    B, T, H, K = q.shape
    V = v.shape[-1]
    cu_d, cu_h, n_seqs = _cu(cu_seqlens, dev)
    N = n_seqs if cu_d is not None else B
    if gate is not None:
        gate, norm_w = _prep(gate, dev), _prep(norm_w, dev, torch.float32)
        if y is None:
            y = torch.empty((B, T, H * V), device=dev, dtype=out_dtype)
    if o is None and (return_o or (dests is not None and dests[0] is not None) or gate is None):
        o = torch.empty((B, T, H, V), device=dev, dtype=out_dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, K, V), device=dev, dtype=torch.float32)
    if scale is None:
        scale = K ** -0.5
    mode_i = _MODES[mode] if isinstance(mode, str) else int(mode)
    ws_ptr, ws_bytes = _chunk_workspace(workspace if mode_i != MODE_FP32 else None, dev, B, T, H, n_seqs)
    tail = (_ptr(initial_state), _ptr(final_state), _ptr(o), _dt(o if o is not None else y), _ptr(cu_d), _ptr(cu_h),
            n_seqs, B, T, H, K, V, int(chunk), float(scale), int(bool(use_qk_l2norm)), _ptr(gate),
            _dt(gate) if gate is not None else BF16, _ptr(norm_w), float(eps), _ptr(y), ws_ptr, ws_bytes,
            mode_i, _stream())
    if lg is None:
        g, beta = _prep(gb[0], dev, torch.float32), _prep(gb[1], dev, torch.float32)
        _check(lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), *tail))
    else:
        z, b, A_log, dt_bias, lb = _logit_args(lg, dev)
        _check(lib.kda_chunk_fwd_logits(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(z), _dt(z), _ptr(A_log),
                                        _ptr(dt_bias), lb, _ptr(b), _dt(b), *tail))
    if gate is not None:
        return _to_host((o, final_state, y), host, dests)
    return _to_host((o, final_state), host, dests)


def recurrent_fwd(q, k, v, g, beta, initial_state=None, *, scale=None, use_qk_l2norm=True,
                  cu_seqlens=None, output_final_state=True, output_states=False, gate=None,
                  norm_w=None, eps=1e-5, out_dtype=torch.float32):
    """Token-by-token form over T tokens (fp32).  Returns (o, final_state[, states][, y])."""
    lib = _load()
    host = q.device.type != "cuda"
    dev = _device_of(q, k, v)
    q, k, v = _prep(q, dev), _prep(k, dev), _prep(v, dev)
    g, beta = _prep(g, dev, torch.float32), _prep(beta, dev, torch.float32)
    initial_state = _prep(initial_state, dev, torch.float32)
    B, T, H, K = q.shape
    V = v.shape[-1]
    cu_d, cu_h, n_seqs = _cu(cu_seqlens, dev)
    N = n_seqs if cu_d is not None else B
    o = torch.empty((B, T, H, V), device=dev, dtype=out_dtype)
    final_state = torch.empty((N, H, K, V), device=dev, dtype=torch.float32) if output_final_state else None
    states = torch.empty((B, T, H, K, V), device=dev, dtype=torch.float32) if output_states else None
    y = None
    if gate is not None:
        gate, norm_w = _prep(gate, dev), _prep(norm_w, dev, torch.float32)
        y = torch.empty((B, T, H * V), device=dev, dtype=out_dtype)
    if scale is None:
        scale = K ** -0.5
    _check(lib.kda_recurrent_fwd(
        _ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(final_state),
        _ptr(o), _dt(o), _ptr(states), _ptr(cu_d), _ptr(cu_h), n_seqs, B, T, H, K, V, float(scale),
        int(bool(use_qk_l2norm)), _ptr(gate), _dt(gate) if gate is not None else BF16, _ptr(norm_w),
        float(eps), _ptr(y), _stream()))
    out = [o, final_state]
    if output_states:
        out.append(states)
    if gate is not None:
        out.append(y)
    return _to_host(tuple(out), host)


def recurrent_step(q, k, v, g, beta, state, *, scale=None, use_qk_l2norm=True, gate=None, norm_w=None,
                   eps=1e-5, out_dtype=torch.float32, state_out=None, return_o=True, o=None, y=None, conv=None):
    """One decode token per sequence.  q, k [B,H,K]; v [B,H,V]; g [B,H,K]; beta [B,H];
    state [B,H,K,V] fp32 (or None).  ``state_out=state`` updates the state in place.

    ``conv=(weights, states_in[, states_out])`` fuses the q, k, v short convolutions
    (+ SiLU) ahead of the step (K = V = 128): q, k, v are then the raw projections,
    weights three [H*128, W] (or [H*128, 1, W]) filters, states_in three [B, W-1, H*128]
    fp32 histories (or None: zero history), states_out three buffers for the new ones
    (default: fresh; ``states_in`` itself updates them in place).
    Returns (o, state_out[, y][, conv_states_out])."""
    return _step(q, k, v, (g, beta), None, state, scale, use_qk_l2norm, gate, norm_w, eps, out_dtype, state_out,
                 return_o, o, y, conv)


def recurrent_step_logits(q, k, v, g_logits, beta_logits, A_log, state, *, dt_bias=None, g_lower_bound=-5.0,
                          scale=None, use_qk_l2norm=True, gate=None, norm_w=None, eps=1e-5, out_dtype=torch.float32,
                          state_out=None, return_o=True, o=None, y=None, conv=None):
    """recurrent_step with g and beta computed from their logits (see chunk_fwd_logits):
    g_logits [B,H,K], beta_logits [B,H]."""
    lb = float("-inf") if g_lower_bound is None else float(g_lower_bound)
    return _step(q, k, v, None, (g_logits, beta_logits, A_log, dt_bias, lb), state, scale, use_qk_l2norm, gate,
                 norm_w, eps, out_dtype, state_out, return_o, o, y, conv)


def _conv_args(conv, dev, B, H):
    """Marshal the fused convolutions' (weights, states_in[, states_out]) for the C call."""
    weights, s_in = conv[0], conv[1]
    s_out = conv[2] if len(conv) > 2 else None
    if len(weights) != 3 or (s_in is not None and len(s_in) != 3) or (s_out is not None and len(s_out) != 3):
        raise ValueError("conv takes three filters (q, k, v), three histories and three outputs")
    ws = [_prep(w[:, 0, :] if w.dim() == 3 else w, dev, torch.float32) for w in weights]
    W = ws[0].shape[1]
    sin = None if s_in is None else [_prep(x, dev, torch.float32) for x in s_in]
    if s_out is None:
        s_out = [torch.empty((B, W - 1, H * 128), device=dev, dtype=torch.float32) for _ in range(3)]
    P3 = ctypes.c_void_p * 3
    ptr3 = lambda ts: P3(*[t.data_ptr() for t in ts])
    keep = (ws, sin, s_out)  # the tensors stay alive through the call
    return ptr3(ws), W, (ptr3(sin) if sin is not None else None), ptr3(s_out), tuple(s_out), keep


def _step(q, k, v, gb, lg, state, scale, use_qk_l2norm, gate, norm_w, eps, out_dtype, state_out, return_o, o, y,
          conv=None):
    lib = _load()
    host = q.device.type != "cuda"
    dev = _device_of(q, k, v, state)
    q, k, v = _prep(q, dev), _prep(k, dev), _prep(v, dev)
    state = _prep(state, dev, torch.float32)
    B, H, K = q.shape
    V = v.shape[-1]
    if state_out is None:
        state_out = torch.empty((B, H, K, V), device=dev, dtype=torch.float32)
    if gate is not None:
        gate, norm_w = _prep(gate, dev), _prep(norm_w, dev, torch.float32)
        if y is None:
            y = torch.empty((B, H * V), device=dev, dtype=out_dtype)
    if o is None and (return_o or gate is None):
        o = torch.empty((B, H, V), device=dev, dtype=out_dtype)
    if scale is None:
        scale = K ** -0.5
    tail = (_ptr(state), _ptr(state_out), _ptr(o), _dt(o if o is not None else y), B, H, K, V, float(scale),
            int(bool(use_qk_l2norm)), _ptr(gate), _dt(gate) if gate is not None else BF16, _ptr(norm_w), float(eps),
            _ptr(y), _stream())
    if conv is not None:
        cw, W, cin, cout_p, cout, _keep = _conv_args(conv, dev, B, H)
        if lg is None:
            g, beta = _prep(gb[0], dev, torch.float32), _prep(gb[1], dev, torch.float32)
            gates = (_ptr(g), _ptr(beta), None, BF16, None, None, 0.0, None, BF16)
        else:
            z, b, A_log, dt_bias, lb = _logit_args(lg, dev)
            gates = (None, None, _ptr(z), _dt(z), _ptr(A_log), _ptr(dt_bias), lb, _ptr(b), _dt(b))
        _check(lib.kda_recurrent_step_conv(_ptr(q), _ptr(k), _ptr(v), _dt(q), cw, W, cin, cout_p, *gates, *tail))
        res = (o, state_out, y) if gate is not None else (o, state_out)
        if host:
            res = _to_host(res + cout, True)
            return res[:-3] + (res[-3:],)
        return res + (cout,)
    if lg is None:
        g, beta = _prep(gb[0], dev, torch.float32), _prep(gb[1], dev, torch.float32)
        _check(lib.kda_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), *tail))
    else:
        z, b, A_log, dt_bias, lb = _logit_args(lg, dev)
        _check(lib.kda_recurrent_step_logits(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(z), _dt(z), _ptr(A_log),
                                             _ptr(dt_bias), lb, _ptr(b), _dt(b), *tail))
    if gate is not None:
        return _to_host((o, state_out, y), host)
    return _to_host((o, state_out), host)


def gated_rmsnorm(o, gate, w, eps=1e-5, *, out_dtype=torch.float32, y=None):
    """y [.., H*V] = o / sqrt(mean_v(o^2) + eps) * w * sigmoid(gate) over each (token, head)."""
    lib = _load()
    host = o.device.type != "cuda"
    dev = _device_of(o, gate)
    o, gate, w = _prep(o, dev), _prep(gate, dev), _prep(w, dev, torch.float32)
    H, V = o.shape[-2], o.shape[-1]
    rows = o.numel() // (H * V)
    if y is None:
        y = torch.empty(o.shape[:-2] + (H * V,), device=dev, dtype=out_dtype)
    _check(lib.kda_gated_rmsnorm(_ptr(o), _dt(o), _ptr(gate), _dt(gate), _ptr(w), float(eps), _ptr(y), _dt(y),
                                 rows, H, V, _stream()))
    return _to_host((y,), host)[0]


def short_conv(x, weight, bias=None, conv_state=None, *, cu_seqlens=None, activation="silu",
               output_final_state=True, out_dtype=None, y=None, final_state=None):
    """Causal depthwise short convolution (+ SiLU) along the sequence.

    x [B,T,D] (bf16 or fp32); weight [D,W] (or the Conv1d weight [D,1,W]); bias [D] or
    None; conv_state [N,W-1,D] fp32 or None (the W-1 inputs before each sequence,
    oldest first).  With ``cu_seqlens`` B must be 1.  A decode step is T = 1;
    ``final_state=conv_state`` then updates the state in place.
    Returns (y [B,T,D], final_state [N,W-1,D] or None)."""
    lib = _load()
    host = x.device.type != "cuda"
    dev = _device_of(x, conv_state)
    dests = (y, final_state) if host else None
    if host:
        y, final_state = _dev_out(y), _dev_out(final_state)
    x = _prep(x, dev)
    if weight.dim() == 3:
        weight = weight[:, 0, :]
    weight = _prep(weight, dev, torch.float32)
    bias = _prep(bias, dev, torch.float32)
    conv_state = _prep(conv_state, dev, torch.float32)
    B, T, D = x.shape
    W = weight.shape[1]
    cu_d, cu_h, n_seqs = _cu(cu_seqlens, dev)
    N = n_seqs if cu_d is not None else B
    if y is None:
        y = torch.empty((B, T, D), device=dev, dtype=out_dtype or x.dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, W - 1, D), device=dev, dtype=torch.float32)
    act = {"silu": 1, "swish": 1, None: 0, "none": 0, "identity": 0}[activation]
    _check(lib.kda_short_conv_fwd(
        _ptr(x), _dt(x), _ptr(weight), _ptr(bias), _ptr(conv_state), _ptr(final_state), _ptr(y), _dt(y),
        _ptr(cu_d), _ptr(cu_h), n_seqs, B, T, D, W, act, _stream()))
    return _to_host((y, final_state), host, dests)


def o_proj(y, w_o, *, out_dtype=torch.bfloat16, out=None):
    """out [rows, out_features] = y [rows, in_features] @ w_o[out_features, in_features]^T
    (bf16 operands, fp32 accumulation, on the library's tcgen05 GEMM).  y may carry extra
    leading dimensions."""
    lib = _load()
    host = y.device.type != "cuda"
    dev = _device_of(y, w_o)
    y2 = _prep(y, dev, torch.bfloat16).reshape(-1, y.shape[-1])
    w = _prep(w_o, dev, torch.bfloat16)
    rows, K = y2.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("w_o must be [out_features, in_features]")
    dest = out if host else None
    if out is None or host:
        out = torch.empty((rows, N), device=dev, dtype=out_dtype)
    _check(lib.kda_o_proj(_ptr(y2), _ptr(w), _ptr(out), _dt(out), rows, K, N, _stream()))
    res = out.reshape(*y.shape[:-1], N)
    if host:
        return _to_host((res,), True, (dest,))[0]
    return res
