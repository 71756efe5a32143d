"""Pins for the fp64 oracle: it is checked against things other than itself.

Every check is written as a function of a *runner* (anything with the oracle's
call signature), so the same checks also run against deliberately wrong
recurrences (mutants built here in numpy): each mutant must fail at least one pin,
which shows the pins would catch that mistake in the oracle.

What the pins rest on:
  * the recurrence's definition (gated delta rule, per-key-channel decay applied
    before the write; nnterp encyclopedia "Kimi-Linear", sections 03 and 04);
  * closed forms that follow from it: frozen state (beta = 0, g = 0), pure decay
    (beta = 0), a single token from a zero state, the write-then-read identity
    (beta = 1, q = k), orthonormal keys (row-wise erase);
  * brute force: the explicit product of per-token transition matrices
    M_t = (I - beta_t k_t k_t^T) Diag(exp g_t), in fp64 and in exact rational
    arithmetic (fractions);
  * structure: split-halves with the state handed across, column (value)
    independence, varlen == separate runs;
  * the gated norm against torch's rms_norm library routine and its limits;
  * a hand-worked two-token example stored under tests/golden/.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
RTOL = 1e-11


# --------------------------------------------------------------------------
# runners


def oracle_runner(q, k, v, g, beta, s0=None, scale=1.0, l2=True):
    """q,k,g [T,H,K]; v [T,H,V]; beta [T,H]; s0 [H,K,V] -> (o [T,H,V], S [H,K,V])."""
    o, s = oracle.recurrent(q[None], k[None], v[None], g[None], beta[None],
                            None if s0 is None else s0[None], scale=scale, use_qk_l2norm=l2,
                            n_threads=2)
    return o[0], s[0]


def make_mutant(kind):
    """A deliberately wrong recurrence (numpy fp64 loop), for tiny inputs only."""

    def run(q, k, v, g, beta, s0=None, scale=1.0, l2=True):
        q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
        T, H, K = q.shape
        V = v.shape[-1]
        o = np.zeros((T, H, V))
        S_all = np.zeros((H, K, V))
        for h in range(H):
            S = np.zeros((K, V)) if s0 is None else np.array(s0[h], np.float64)
            for t in range(T):
                qt, kt = q[t, h], k[t, h]
                if l2 and kind != "no_l2norm":
                    qt = qt / math.sqrt(qt @ qt + oracle.DEFAULT_L2_EPS)
                    kt = kt / math.sqrt(kt @ kt + oracle.DEFAULT_L2_EPS)
                a = np.exp(g[t, h])
                if kind == "decay_after_write":
                    d = beta[t, h] * (v[t, h] - S.T @ kt)
                    S = (S + np.outer(kt, d)) * a[:, None]
                elif kind == "decay_values":  # decays value columns instead of key rows
                    S = S * np.resize(a, V)[None, :]
                    d = beta[t, h] * (v[t, h] - S.T @ kt)
                    S = S + np.outer(kt, d)
                elif kind == "beta_only_on_v":
                    S = S * a[:, None]
                    d = beta[t, h] * v[t, h] - S.T @ kt
                    S = S + np.outer(kt, d)
                else:
                    S = S * a[:, None]
                    d = beta[t, h] * (v[t, h] - S.T @ kt)
                    if kind == "readout_before_write":
                        o[t, h] = scale * (S.T @ qt)
                    S = S + np.outer(kt, d)
                if kind != "readout_before_write":
                    o[t, h] = scale * (S.T @ qt)
            S_all[h] = S
        return o, S_all

    return run


MUTANTS = ["decay_after_write", "decay_values", "beta_only_on_v", "readout_before_write", "no_l2norm"]


# --------------------------------------------------------------------------
# helpers


def rnd(rng, *shape):
    return rng.standard_normal(shape).astype(np.float32)


def decays(rng, *shape, lo=-1.5):
    return (rng.random(shape) * lo).astype(np.float32)


def l2n(x):
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + oracle.DEFAULT_L2_EPS)


def close(a, b, rtol=RTOL):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, f"shape {a.shape} != {b.shape}"
    if a.size == 0:
        return
    scale = max(1.0, float(np.abs(b).max()))
    err = float(np.abs(a - b).max()) / scale
    assert err <= rtol, f"max rel error {err:.3e} > {rtol:.1e}"


# --------------------------------------------------------------------------
# the pins, each a function of a runner


def check_frozen_state(run):
    """beta = 0 and g = 0: the state never changes, o_t = scale * S0^T q^_t."""
    rng = np.random.default_rng(1)
    T, H, K, V = 7, 2, 5, 3
    q, k, v = rnd(rng, T, H, K), rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = np.zeros((T, H, K), np.float32)
    beta = np.zeros((T, H), np.float32)
    s0 = rnd(rng, H, K, V)
    o, s = run(q, k, v, g, beta, s0, scale=0.37)
    close(s, s0)
    close(o, 0.37 * np.einsum("hkv,thk->thv", s0.astype(np.float64), l2n(q)))


def check_decay_closed_form(run):
    """beta = 0: S_t = Diag(exp sum_{s<=t} g_s) S0 and o_t = scale S0^T (exp(G_t) * q^_t)."""
    rng = np.random.default_rng(2)
    T, H, K, V = 9, 2, 4, 4
    q, k, v = rnd(rng, T, H, K), rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = np.zeros((T, H), np.float32)
    s0 = rnd(rng, H, K, V)
    o, s = run(q, k, v, g, beta, s0, scale=0.5)
    G = np.cumsum(g.astype(np.float64), axis=0)  # [T,H,K]
    close(s, np.exp(G[-1])[:, :, None] * s0)
    close(o, 0.5 * np.einsum("hkv,thk->thv", s0.astype(np.float64), np.exp(G) * l2n(q)))


def check_single_token(run):
    """One token from a zero state: S = beta k^ v^T, o = scale beta (k^.q^) v."""
    rng = np.random.default_rng(3)
    H, K, V = 3, 6, 5
    q, k, v = rnd(rng, 1, H, K), rnd(rng, 1, H, K), rnd(rng, 1, H, V)
    g = decays(rng, 1, H, K)
    beta = rng.random((1, H)).astype(np.float32)
    o, s = run(q, k, v, g, beta, None, scale=0.25)
    kh, qh = l2n(k[0]), l2n(q[0])
    b = beta[0].astype(np.float64)
    close(s, b[:, None, None] * np.einsum("hk,hv->hkv", kh, v[0].astype(np.float64)))
    close(o[0], 0.25 * (b * (kh * qh).sum(-1))[:, None] * v[0].astype(np.float64))


def check_split_halves(run):
    """Running T tokens equals running T1 then T - T1 with the state handed across."""
    rng = np.random.default_rng(4)
    T, H, K, V = 12, 2, 4, 3
    q, k, v = rnd(rng, T, H, K), rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = rng.random((T, H)).astype(np.float32)
    s0 = rnd(rng, H, K, V)
    o, s = run(q, k, v, g, beta, s0, scale=0.3)
    for T1 in (1, 5, 11):
        o1, s1 = run(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], s0, scale=0.3)
        o2, s2 = run(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], s1, scale=0.3)
        close(np.concatenate([o1, o2]), o)
        close(s2, s)


def brute_force(q, k, v, g, beta, s0, scale, l2=True):
    """Explicit transition products: S_t = M_t S_{t-1} + beta_t k_t v_t^T,
    M_t = (I - beta_t k_t k_t^T) Diag(exp g_t); o_t = scale S_t^T q_t."""
    T, H, K = q.shape
    V = v.shape[-1]
    qn = l2n(q) if l2 else np.asarray(q, np.float64)
    kn = l2n(k) if l2 else np.asarray(k, np.float64)
    o = np.zeros((T, H, V))
    S_out = np.zeros((H, K, V))
    for h in range(H):
        # S_T = (M_T...M_1) S0 + sum_t (M_T...M_{t+1}) beta_t k_t v_t^T, built from products
        Ms = [(np.eye(K) - beta[t, h] * np.outer(kn[t, h], kn[t, h])) @ np.diag(np.exp(g[t, h].astype(np.float64)))
              for t in range(T)]
        for t in range(T):
            P = np.eye(K)
            acc = np.zeros((K, V))
            for s in range(t, -1, -1):  # s = t, t-1, ..., 0 ; P = M_t ... M_{s+1}
                acc += P @ (beta[s, h] * np.outer(kn[s, h], v[s, h].astype(np.float64)))
                P = P @ Ms[s]
            St = P @ np.asarray(s0[h], np.float64) + acc
            o[t, h] = scale * St.T @ qn[t, h]
            if t == T - 1:
                S_out[h] = St
    return o, S_out


def check_brute_force(run):
    rng = np.random.default_rng(5)
    T, H, K, V = 8, 2, 4, 3
    q, k, v = rnd(rng, T, H, K), rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = rng.random((T, H)).astype(np.float32)
    s0 = rnd(rng, H, K, V)
    o, s = run(q, k, v, g, beta, s0, scale=0.4)
    ob, sb = brute_force(q, k, v, g, beta, s0, 0.4)
    close(o, ob, 1e-10)
    close(s, sb, 1e-10)


def check_write_read_identity(run):
    """beta = 1 and q = k (exact unit norm, kernel norm off): o_t = scale v_t for any g, S0."""
    rng = np.random.default_rng(6)
    T, H, K, V = 10, 2, 4, 5
    signs = rng.choice([-0.5, 0.5], size=(T, H, K)).astype(np.float32)  # |k| = 1 exactly
    v = rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = np.ones((T, H), np.float32)
    s0 = rnd(rng, H, K, V)
    o, _ = run(signs, signs, v, g, beta, s0, scale=0.7, l2=False)
    close(o, 0.7 * v.astype(np.float64))


def check_column_independence(run, rtol=1e-14):
    """Value columns evolve independently: V-slices run apart equal the full run."""
    rng = np.random.default_rng(7)
    T, H, K, V = 9, 2, 4, 6
    q, k, v = rnd(rng, T, H, K), rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = rng.random((T, H)).astype(np.float32)
    s0 = rnd(rng, H, K, V)
    o, s = run(q, k, v, g, beta, s0, scale=0.3)
    for a, b in ((0, 2), (2, 3), (3, 6)):
        oa, sa = run(q, k, np.ascontiguousarray(v[..., a:b]), g, beta, np.ascontiguousarray(s0[..., a:b]), scale=0.3)
        close(oa, o[..., a:b], rtol)
        close(sa, s[..., a:b], rtol)


def check_orthonormal_keys(run):
    """k_t = e_t (t < K): row i is decayed, erased by (1 - beta_i |k^|^2), written beta_i |k^| v_i."""
    rng = np.random.default_rng(8)
    K, V, H = 5, 3, 1
    T = K
    k = np.zeros((T, H, K), np.float32)
    for t in range(T):
        k[t, 0, t] = 1.0
    q, v = rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = rng.random((T, H)).astype(np.float32)
    s0 = rnd(rng, H, K, V)
    _, s = run(q, k, v, g, beta, s0, scale=1.0)
    c = 1.0 / math.sqrt(1.0 + oracle.DEFAULT_L2_EPS)  # |k^| after the kernel's L2 norm
    G = np.cumsum(g[:, 0, :].astype(np.float64), axis=0)  # [T,K]
    exp_s = np.zeros((K, V))
    for i in range(K):
        before = math.exp(G[i, i]) * s0[0, i].astype(np.float64)  # decayed through step i
        b = float(beta[i, 0])
        row = (1 - b * c * c) * before + b * c * v[i, 0].astype(np.float64)
        exp_s[i] = math.exp(G[-1, i] - G[i, i]) * row  # decayed after step i
    close(s[0], exp_s)


def check_exact_rational(run):
    """g = 0, kernel norm off, small rational inputs: brute force in exact fractions."""
    rng = np.random.default_rng(9)
    T, K, V = 5, 3, 2
    ints = lambda *s: rng.integers(-4, 5, size=s)
    qi, ki, vi = ints(T, K), ints(T, K), ints(T, V)
    q = (qi / 4).astype(np.float32)[:, None]
    k = (ki / 4).astype(np.float32)[:, None]
    v = (vi / 2).astype(np.float32)[:, None]
    b = rng.integers(0, 5, size=T) / 4
    beta = b.astype(np.float32)[:, None]
    g = np.zeros((T, 1, K), np.float32)
    o, s = run(q, k, v, g, beta, None, scale=1.0, l2=False)
    S = [[Fraction(0)] * V for _ in range(K)]
    for t in range(T):
        kt = [Fraction(int(x), 4) for x in ki[t]]
        qt = [Fraction(int(x), 4) for x in qi[t]]
        vt = [Fraction(int(x), 2) for x in vi[t]]
        bt = Fraction(int(b[t] * 4), 4)
        u = [sum(S[i][j] * kt[i] for i in range(K)) for j in range(V)]
        d = [bt * (vt[j] - u[j]) for j in range(V)]
        S = [[S[i][j] + kt[i] * d[j] for j in range(V)] for i in range(K)]
        ot = [sum(S[i][j] * qt[i] for i in range(K)) for j in range(V)]
        close(o[t, 0], [float(x) for x in ot], 1e-14)
    close(s[0], [[float(x) for x in row] for row in S], 1e-14)


PINS = [check_frozen_state, check_decay_closed_form, check_single_token, check_split_halves,
        check_brute_force, check_write_read_identity, check_column_independence,
        check_orthonormal_keys, check_exact_rational]


# --------------------------------------------------------------------------
# tests


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle_runner)


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_mutant(kind):
    mutant = make_mutant(kind)
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {kind} passed every pin"


def test_oracle_columns_bitwise_independent():
    """In the oracle the value columns do not even share rounding: slices are bitwise equal."""
    check_column_independence(oracle_runner, rtol=0.0)


def test_mutant_harness_is_faithful():
    """The numpy loop with no mutation agrees with the oracle (so mutants differ only by their bug)."""
    for pin in PINS:
        pin(make_mutant("none"))


def test_worked_example_golden():
    """A two-token example derived by hand (tests/golden/worked_example.json)."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    arr = lambda name: np.asarray(ex["inputs"][name], np.float32)
    o, s = oracle_runner(arr("q"), arr("k"), arr("v"), arr("g"), arr("beta"), None,
                         scale=ex["inputs"]["scale"], l2=ex["inputs"]["use_qk_l2norm"])
    close(o, np.asarray(ex["expected"]["o"]), 1e-7)
    close(s, np.asarray(ex["expected"]["final_state"]), 1e-7)


def test_regression_golden():
    """Oracle output on a fixed small case equals the committed values written by
    tests/golden/make_golden.py (which calls only oracle/)."""
    with open(os.path.join(GOLDEN, "tiny_recurrence.json")) as f:
        ex = json.load(f)
    inp = {k: np.asarray(v, np.float32) if isinstance(v, list) else v for k, v in ex["inputs"].items()}
    o, s = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                            np.asarray(ex["inputs"]["initial_state"], np.float64), scale=inp["scale"])
    close(o, np.asarray(ex["expected"]["o"]), 1e-12)
    close(s, np.asarray(ex["expected"]["final_state"]), 1e-12)


def test_varlen_equals_separate_runs():
    rng = np.random.default_rng(10)
    lens = [3, 0, 7, 1]
    Tt, H, K, V = sum(lens), 2, 4, 3
    q, k, v = rnd(rng, 1, Tt, H, K), rnd(rng, 1, Tt, H, K), rnd(rng, 1, Tt, H, V)
    g = decays(rng, 1, Tt, H, K)
    beta = rng.random((1, Tt, H)).astype(np.float32)
    s0 = rnd(rng, len(lens), H, K, V)
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, s = oracle.recurrent(q, k, v, g, beta, s0, scale=0.5, cu_seqlens=cu)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        on, sn = oracle.recurrent(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], s0[n:n + 1], scale=0.5)
        close(o[:, a:b], on, 0.0)
        close(s[n], sn[0], 0.0)


def test_per_token_states():
    """The per-token state readout: its last entry is the final state and each entry
    reproduces o_t = scale S_t^T q^_t."""
    rng = np.random.default_rng(11)
    T, H, K, V = 6, 2, 4, 3
    q, k, v = rnd(rng, 1, T, H, K), rnd(rng, 1, T, H, K), rnd(rng, 1, T, H, V)
    g = decays(rng, 1, T, H, K)
    beta = rng.random((1, T, H)).astype(np.float32)
    o, s, st = oracle.recurrent(q, k, v, g, beta, scale=0.5, return_states=True)
    close(st[0, -1], s[0], 0.0)
    close(o[0], 0.5 * np.einsum("thkv,thk->thv", st[0], l2n(q[0])))


def test_qk_norm_scale_invariance():
    """With the kernel L2 norm on, scaling q or k rows by a positive factor only moves
    the result through the epsilon inside the square root."""
    rng = np.random.default_rng(12)
    T, H, K, V = 6, 2, 8, 4
    q, k, v = rnd(rng, T, H, K), rnd(rng, T, H, K), rnd(rng, T, H, V)
    g = decays(rng, T, H, K)
    beta = rng.random((T, H)).astype(np.float32)
    o1, s1 = oracle_runner(q, k, v, g, beta, scale=0.3)
    o2, s2 = oracle_runner(q * 4, k * 8, v, g, beta, scale=0.3)
    close(o1, o2, 1e-6)
    close(s1, s2, 1e-6)


# --------------------------------------------------------------------------
# gated RMSNorm


def test_norm_matches_library_rmsnorm():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    rows, H, V = 5, 3, 16
    o = rng.standard_normal((rows, H, V))
    gate = rnd(rng, rows, H, V)
    w = (1 + 0.1 * rng.standard_normal(V)).astype(np.float32)
    y = oracle.gated_rmsnorm(o, gate, w, eps=1e-5)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), (V,), torch.from_numpy(w.astype(np.float64)), eps=1e-5)
    ref = ref * torch.sigmoid(torch.from_numpy(gate.astype(np.float64)))
    close(y, ref.reshape(rows, H * V).numpy(), 1e-12)


def test_norm_limits():
    """w = 1: a saturated gate leaves unit RMS per head (up to eps); gate = 0 halves it."""
    rng = np.random.default_rng(14)
    rows, H, V = 4, 2, 128
    o = rng.standard_normal((rows, H, V))
    w = np.ones(V, np.float32)
    y_open = oracle.gated_rmsnorm(o, np.full((rows, H, V), 60.0, np.float32), w, eps=1e-5).reshape(rows, H, V)
    ms = (o * o).mean(-1)
    close(np.sqrt((y_open ** 2).mean(-1)), np.sqrt(ms / (ms + 1e-5)), 1e-12)
    y_half = oracle.gated_rmsnorm(o, np.zeros((rows, H, V), np.float32), w, eps=1e-5).reshape(rows, H, V)
    close(y_half, 0.5 * y_open, 1e-15)


def test_norm_weight_is_one_vector_shared_by_heads():
    """The gated norm holds head_dim = 128 weights shared by every head: with 96 heads
    of 128 features the output projection holds 12288 * 7168 = 88,080,384 weights and
    gate-project 88,080,512 in all (Kimi-K3 atlas, gate-project, section "Parameters")."""
    H, V, hidden = 96, 128, 7168
    assert H * V * hidden == 88_080_384
    assert H * V * hidden + V == 88_080_512
    rng = np.random.default_rng(15)
    o = rng.standard_normal((2, 3, V))
    gate = rnd(rng, 2, 3, V)
    w = (1 + rng.standard_normal(V)).astype(np.float32)
    y = oracle.gated_rmsnorm(o, gate, w).reshape(2, 3, V)
    for h in range(3):
        yh = oracle.gated_rmsnorm(o[:, h:h + 1], gate[:, h:h + 1], w).reshape(2, V)
        close(y[:, h], yh, 0.0)
    with pytest.raises(ValueError):
        oracle.gated_rmsnorm(o, gate, np.ones(3 * V, np.float32))
