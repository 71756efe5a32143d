"""fp64 CPU oracle for the Kimi Delta Attention core -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and it never imports them: the
two share nothing but the seeded input arrays.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, one thread per group of
(sequence, head) units).  This module compiles it with gcc on first use and wraps
it with ctypes.  Page citations for every formula are in the C file's header:
the recurrence follows the nnterp encyclopedia page "Kimi-Linear" (sections 02,
03 and 04), the gated norm the Kimi-K3 atlas page "gate-project" (sections
"Parameters" and "Code").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

DEFAULT_L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into libkda_oracle.so (plain gcc, no GPU)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.kda_oracle_recurrent.argtypes = [
                P, P, P, P, P, P, P, P, P, P,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            ]
            lib.kda_oracle_recurrent.restype = ctypes.c_int
            lib.kda_oracle_gated_rmsnorm.argtypes = [
                P, P, P, ctypes.c_double, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            ]
            lib.kda_oracle_gated_rmsnorm.restype = ctypes.c_int
            lib.kda_oracle_gates.argtypes = [P, P, P, ctypes.c_double, P, P, P, ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_int]
            lib.kda_oracle_gates.restype = ctypes.c_int
            lib.kda_oracle_short_conv.argtypes = [
                P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int,
            ]
            lib.kda_oracle_short_conv.restype = ctypes.c_int
            lib.kda_oracle_version.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def recurrent(q, k, v, g, beta, initial_state=None, *, scale=None, use_qk_l2norm=True,
              l2_eps=DEFAULT_L2_EPS, cu_seqlens=None, return_states=False, n_threads=None):
    """Token-by-token fp64 recurrence.

    Dense form: q, k, g [B,T,H,K]; v [B,T,H,V]; beta [B,T,H]; initial_state
    [B,H,K,V] or None.  Varlen form (``cu_seqlens`` given, int, n_seqs+1 entries):
    the leading dimension is 1 (or absent) and initial_state is [n_seqs,H,K,V].
    Returns ``(o [.., T, H, V] float64, final_state [N,H,K,V] float64[, states])``.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    g, beta = _f64(g), _f64(beta)  # exact for fp32 inputs; fp64 gates from gates() pass unrounded
    if q.ndim == 3:  # [T,H,K] packed varlen without batch dim
        q, k, v, g, beta = q[None], k[None], v[None], g[None], beta[None]
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("shape mismatch between q, k, v, g, beta")
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if B != 1:
            raise ValueError("varlen needs batch 1")
        N = cu.shape[0] - 1
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must start at 0, end at T and not decrease")
    else:
        cu = None
        N = B
    s0 = None if initial_state is None else _f64(initial_state)
    if s0 is not None and s0.shape != (N, H, K, V):
        raise ValueError(f"initial_state must be {(N, H, K, V)}")
    o = np.zeros((B, T, H, V), dtype=np.float64)
    sf = np.zeros((N, H, K, V), dtype=np.float64)
    states = np.zeros((B, T, H, K, V), dtype=np.float64) if return_states else None
    lib = _load()
    rc = lib.kda_oracle_recurrent(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0), _ptr(o), _ptr(sf), _ptr(states),
        _ptr(cu), N if cu is not None else 0, B, T, H, K, V, float(scale), int(bool(use_qk_l2norm)),
        float(l2_eps), int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_recurrent failed with {rc}")
    if return_states:
        return o, sf, states
    return o, sf


def gated_rmsnorm(o, gate, w, eps=1e-5):
    """y [.., H*V] = o / sqrt(mean_v(o^2)+eps) * w * sigmoid(gate), per (token, head)."""
    o = _f64(o)
    gate = _f32(gate)
    w = _f32(w)
    H, V = o.shape[-2], o.shape[-1]
    if gate.shape != o.shape or w.shape != (V,):
        raise ValueError("gate must match o and w must be [V]")
    rows = int(np.prod(o.shape[:-2]))
    y = np.zeros(o.shape[:-2] + (H * V,), dtype=np.float64)
    rc = _load().kda_oracle_gated_rmsnorm(_ptr(o), _ptr(gate), _ptr(w), float(eps), _ptr(y), rows, H, V)
    if rc != 0:
        raise RuntimeError(f"kda_oracle_gated_rmsnorm failed with {rc}")
    return y


def gates(z, A_log, b, dt_bias=None, lower_bound=None):
    """g [.., H, K] and beta [.., H] (fp64) from the decay logits z [.., H, K], A_log [H],
    dt_bias [H, K] (or [H*K]) or None, the write-strength logits b [.., H] and an optional
    lower bound.  Formula and page citations: ``kda_oracle_gates`` in kda_oracle.c."""
    z = _f32(z)
    b = _f32(b)
    H, K = z.shape[-2], z.shape[-1]
    A_log = _f32(A_log).reshape(H)
    dtb = None if dt_bias is None else _f32(dt_bias).reshape(H, K)
    if b.shape != z.shape[:-1]:
        raise ValueError("b must be z without its last axis")
    rows = int(np.prod(z.shape[:-2]))
    g = np.zeros(z.shape, dtype=np.float64)
    beta = np.zeros(b.shape, dtype=np.float64)
    lb = -np.inf if lower_bound is None else float(lower_bound)
    rc = _load().kda_oracle_gates(_ptr(z), _ptr(A_log), _ptr(dtb), lb, _ptr(b), _ptr(g), _ptr(beta), rows, H, K)
    if rc != 0:
        raise RuntimeError(f"kda_oracle_gates failed with {rc}")
    return g, beta


def short_conv(x, weight, bias=None, conv_state=None, *, cu_seqlens=None, activation="silu"):
    """Causal depthwise convolution along the sequence (+ SiLU), fp64.

    x [B,T,D] (or [T,D] packed varlen), weight [D,W], bias [D] or None, conv_state
    [N,W-1,D] or None (the W-1 inputs before each sequence, oldest first).
    Returns ``(y [.., T, D] float64, final_state [N, W-1, D] float64)``.
    Formula and page citations: ``kda_oracle_short_conv`` in kda_oracle.c.
    """
    x = _f32(x)
    if x.ndim == 2:
        x = x[None]
    B, T, D = x.shape
    w = _f64(weight)
    if w.ndim != 2 or w.shape[0] != D:
        raise ValueError("weight must be [D, W]")
    W = w.shape[1]
    b = None if bias is None else _f64(bias)
    if b is not None and b.shape != (D,):
        raise ValueError("bias must be [D]")
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if B != 1 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("varlen needs batch 1 and cu_seqlens from 0 to T, non-decreasing")
        N = cu.shape[0] - 1
    else:
        cu, N = None, B
    s0 = None if conv_state is None else _f64(conv_state)
    if s0 is not None and s0.shape != (N, W - 1, D):
        raise ValueError(f"conv_state must be {(N, W - 1, D)}")
    y = np.zeros((B, T, D), dtype=np.float64)
    sf = np.zeros((N, W - 1, D), dtype=np.float64)
    act = {"silu": 1, "swish": 1, None: 0, "none": 0, "identity": 0}[activation]
    rc = _load().kda_oracle_short_conv(_ptr(x), _ptr(w), _ptr(b), _ptr(s0), _ptr(y), _ptr(sf), _ptr(cu),
                                       N if cu is not None else 0, B, T, D, W, act)
    if rc != 0:
        raise RuntimeError(f"kda_oracle_short_conv failed with {rc}")
    return y, sf


def o_proj(y, w_o):
    """The layer's output projection, out = y @ w_o^T in fp64 (nn.Linear without bias;
    Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters" and "Code").
    A library matmul serves as the one step."""
    return np.asarray(y, np.float64) @ np.asarray(w_o, np.float64).T


def version() -> int:
    return int(_load().kda_oracle_version())
