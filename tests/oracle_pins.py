"""Pins for the CPU oracle: checks against facts that the pages and the
mathematics fix, none of which re-types the oracle's own loop.

Each pin takes an oracle library handle (``lib``) so that the same checks can
be run on deliberately broken copies of the oracle (tests/test_oracle_mutants.py)
to show that a plausible mistake fails at least one of them.

Sources: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
NVIDIA CUDA Tile" (sections "The Mamba-2 Recurrence", "Step 1/2/3", "Kernel 1:
chunk_cumsum", "Kernel 2: fwd_pass_state") and its zhiding.cn rendering
(section "Mamba-2架构").
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def random_problem(seed, b=2, L=37, H=4, P=3, N=5, G=2, with_init=True, with_D=True,
                   A_zero=False, dt_zero=False):
    """Small seeded problem with the pages' sign conventions (dt > 0, A < 0)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((b, L, H, P))
    B = rng.standard_normal((b, L, G, N))
    C = rng.standard_normal((b, L, G, N))
    dt = np.log1p(np.exp(rng.normal(-1.0, 0.7, (b, L, H))))
    if dt_zero:
        dt = np.zeros_like(dt)
    A = -np.exp(rng.uniform(0.0, math.log(16.0), H))
    if A_zero:
        A = np.zeros_like(A)
    D = rng.standard_normal(H) if with_D else None
    init = rng.normal(0.0, 0.5, (b, H, P, N)) if with_init else None
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D, init_state=init)


def _rel(a, b):
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


# --- pins -----------------------------------------------------------------

def pin_hand_example(lib):
    """Two tokens worked by hand from the recurrence (tests/golden/two_token_hand.json)."""
    with open(os.path.join(GOLDEN, "two_token_hand.json")) as f:
        g = json.load(f)
    b, L, H, P, N, G = (g[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups"))
    y, fin = oracle.recurrence(
        np.array(g["x"]).reshape(b, L, H, P), np.array(g["dt"]).reshape(b, L, H),
        np.array(g["A"]), np.array(g["B"]).reshape(b, L, G, N),
        np.array(g["C"]).reshape(b, L, G, N), np.array(g["D"]),
        np.array(g["init_state"]).reshape(b, H, P, N), lib=lib)
    assert np.allclose(y.ravel(), g["y"], rtol=0, atol=1e-12), (y.ravel(), g["y"])
    assert np.allclose(fin.ravel(), g["final_state"], rtol=0, atol=1e-12)


def pin_chunked_closed_form(lib):
    """The chunked closed form (jump + chunk outputs, 'Step 3') equals the
    recurrence for several chunk lengths, including Q=1 and a ragged tail."""
    prob = random_problem(1, L=45)
    y_ref, f_ref = oracle.recurrence(**prob, lib=lib)
    for Q in (1, 4, 16, 64):
        y, f = oracle.chunked(**prob, chunk=Q, lib=lib)
        assert _rel(y, y_ref) < 1e-12, (Q, _rel(y, y_ref))
        assert _rel(f, f_ref) < 1e-12, (Q, _rel(f, f_ref))


def pin_linear_attention(lib):
    """With A = 0 there is no decay and the chunk output is causal linear
    attention, Y = C h0 + ((C B^T) o M) (dt X) + D X ('Step 2'), evaluated here
    by brute force over all token pairs (groups shared by H/G heads, P != N)."""
    prob = random_problem(2, b=2, L=29, H=4, P=3, N=5, G=2, A_zero=True)
    y, fin = oracle.recurrence(**prob, lib=lib)
    x, dt, B, C, D, h0 = (prob[k] for k in ("x", "dt", "B", "C", "D", "init_state"))
    b, L, H, P = x.shape
    G = B.shape[2]
    gi = np.arange(H) // (H // G)
    Bh, Ch = B[:, :, gi, :], C[:, :, gi, :]                       # [b, L, H, N]
    cb = np.einsum("bihn,bjhn->bhij", Ch, Bh)                      # C_i . B_j
    mask = np.tril(np.ones((L, L)))
    intra = np.einsum("bhij,bjh,bjhp->bihp", cb * mask, dt, x)
    inter = np.einsum("bihn,bhpn->bihp", Ch, h0)
    y_bf = inter + intra + D[None, None, :, None] * x
    assert _rel(y, y_bf) < 1e-12, _rel(y, y_bf)
    f_bf = h0 + np.einsum("bjh,bjhn,bjhp->bhpn", dt, Bh, x)
    assert _rel(fin, f_bf) < 1e-12


def pin_dt_zero(lib):
    """dt = 0 makes the decay exp(0) = 1 and writes nothing: the state passes
    through unchanged ('The Mamba-2 Recurrence'), and y_t = C_t h0 + D x_t."""
    prob = random_problem(3, dt_zero=True)
    y, fin = oracle.recurrence(**prob, lib=lib)
    assert np.array_equal(fin, prob["init_state"])
    H, G = prob["x"].shape[2], prob["B"].shape[2]
    Ch = prob["C"][:, :, np.arange(H) // (H // G), :]
    y_ref = np.einsum("bthn,bhpn->bthp", Ch, prob["init_state"]) + \
        prob["D"][None, None, :, None] * prob["x"]
    assert _rel(y, y_ref) < 1e-13


def pin_geometric(lib):
    """P = N = 1, B = C = x = 1, constant a = A*dt, h0 = 0: the recurrence is a
    geometric series, h_t = dt (1 - e^{a(t+1)}) / (1 - e^a), and y_t = h_t + D."""
    L, dtv, Av, Dv = 50, 0.3, -1.7, 0.25
    x = np.ones((1, L, 1, 1)); B = np.ones((1, L, 1, 1)); C = np.ones((1, L, 1, 1))
    dt = np.full((1, L, 1), dtv)
    y, fin = oracle.recurrence(x, dt, np.array([Av]), B, C, np.array([Dv]), None, lib=lib)
    a = Av * dtv
    t = np.arange(L)
    h = dtv * (1.0 - np.exp(a * (t + 1))) / (1.0 - np.exp(a))
    assert np.allclose(y.ravel(), h + Dv, rtol=1e-13, atol=0)
    assert abs(fin.ravel()[0] - h[-1]) < 1e-13


def pin_D_isolation(lib):
    """B = 0 and h0 = 0 leave the state at zero, so y = D x exactly."""
    prob = random_problem(4, with_init=False)
    prob["B"] = np.zeros_like(prob["B"])
    y, fin = oracle.recurrence(**prob, lib=lib)
    assert np.array_equal(y, prob["D"][None, None, :, None] * prob["x"])
    assert not np.any(fin)


def pin_split_composition(lib):
    """Feeding final_state back as init_state ('Kernel 2: fwd_pass_state', the
    streaming use) composes: run(0..L1) then run(L1..L) equals run(0..L)."""
    prob = random_problem(5, L=41)
    y_ref, f_ref = oracle.recurrence(**prob, lib=lib)
    for L1 in (1, 7, 20, 40):
        p1 = dict(prob); p2 = dict(prob)
        for k in ("x", "dt", "B", "C"):
            p1[k] = prob[k][:, :L1]
            p2[k] = prob[k][:, L1:]
        y1, f1 = oracle.recurrence(**p1, lib=lib)
        p2["init_state"] = f1
        y2, f2 = oracle.recurrence(**p2, lib=lib)
        assert _rel(np.concatenate([y1, y2], axis=1), y_ref) < 1e-13
        assert _rel(f2, f_ref) < 1e-13


def pin_linearity(lib):
    """For fixed dt, A, B, C, D the map (x, h0) -> (y, final_state) is linear."""
    p1 = random_problem(6); p2 = random_problem(7)
    for k in ("dt", "A", "B", "C", "D"):
        p2[k] = p1[k]
    al, be = 0.7, -1.3
    pm = dict(p1)
    pm["x"] = al * p1["x"] + be * p2["x"]
    pm["init_state"] = al * p1["init_state"] + be * p2["init_state"]
    y1, f1 = oracle.recurrence(**p1, lib=lib)
    y2, f2 = oracle.recurrence(**p2, lib=lib)
    ym, fm = oracle.recurrence(**pm, lib=lib)
    assert _rel(ym, al * y1 + be * y2) < 1e-12
    assert _rel(fm, al * f1 + be * f2) < 1e-12


def pin_checkpoints(lib):
    """The recorded chunk-start states are the final states of the prefixes
    [0, c*Q) -- the states the chunked method carries between chunks."""
    prob = random_problem(8, L=30)
    Q = 8
    _, _, ck = oracle.recurrence(**prob, ckpt_every=Q, lib=lib)
    assert ck.shape[2] == 4
    assert np.array_equal(ck[:, :, 0], prob["init_state"])
    for c in range(1, 4):
        p = dict(prob)
        for k in ("x", "dt", "B", "C"):
            p[k] = prob[k][:, :c * Q]
        _, f = oracle.recurrence(**p, lib=lib)
        assert _rel(ck[:, :, c], f) < 1e-13


def pin_chunk_cumsum(lib):
    """G = log2(e) * inclusive in-chunk sum of A*dt ('Kernel 1: chunk_cumsum'):
    with constant dt it is log2(e)*A*dt*(k+1) at position k of each chunk, and
    2^(G at a chunk's last token) is the product of that chunk's decays."""
    b, L, H, Q = 2, 50, 3, 16
    A = np.array([-1.0, -2.5, -7.0])
    dt = np.full((b, L, H), 0.125)
    G = oracle.chunk_cumsum(dt, A, Q, lib=lib)
    k = (np.arange(L) % Q) + 1
    expect = (A[None, :, None] * 0.125 * k[None, None, :]) / math.log(2.0)
    assert np.allclose(G, np.broadcast_to(expect, G.shape), rtol=1e-14, atol=1e-14)
    rng = np.random.default_rng(9)
    dt = rng.uniform(0.01, 0.5, (b, L, H))
    G = oracle.chunk_cumsum(dt, A, Q, lib=lib)
    for c0 in range(0, L, Q):
        last = min(c0 + Q, L) - 1
        prod = np.prod(np.exp(A[None, :, None] * np.moveaxis(dt, 1, 2)[:, :, c0:last + 1]), axis=2)
        assert np.allclose(np.exp2(G[:, :, last]), prod, rtol=1e-12)
    assert np.all(np.diff(G.reshape(b, H, L), axis=2)[:, :, np.arange(L - 1) % Q != Q - 1] < 0)


# --- causal conv1d (Helion hackathon gallery, "Causal Conv1d (causal_conv1d)":
# out[b, d, t] = bias[d] + sum_k weight[d, k] x[b, d, t - W + 1 + k], left zero padding)

def pin_conv1d_hand_example(lib):
    """x = [1, 2, 3, 4], taps [1, 0, -1], bias 0.25, worked by hand:
    out[t] = x[t-2] - x[t]  ->  [-1, -2, -2, -2] + 0.25."""
    out = oracle.causal_conv1d(np.array([[[1.0, 2.0, 3.0, 4.0]]]), np.array([[1.0, 0.0, -1.0]]),
                               np.array([0.25]), lib=lib)
    np.testing.assert_allclose(out[0, 0], [-0.75, -1.75, -1.75, -1.75], rtol=0, atol=1e-15)


def pin_conv1d_library(lib):
    """Each row is numpy's full convolution with the reversed taps, cut to the
    first L samples (the causal part), plus the bias."""
    rng = np.random.default_rng(11)
    b, d, L, W = 2, 5, 23, 4
    x = rng.standard_normal((b, d, L))
    w = rng.standard_normal((d, W))
    bias = rng.standard_normal(d)
    out = oracle.causal_conv1d(x, w, bias, lib=lib)
    for i in range(b):
        for c in range(d):
            ref = np.convolve(x[i, c], w[c, ::-1])[:L] + bias[c]
            np.testing.assert_allclose(out[i, c], ref, rtol=1e-12, atol=1e-12)


def pin_conv1d_impulse_and_causality(lib):
    """A unit impulse at t0 returns the taps in reverse from t0 on (nothing
    before t0: no output reads the future), and width 1 is a per-channel scale."""
    W, L, t0 = 4, 12, 5
    w = np.array([[0.5, -1.0, 2.0, 3.0]])
    x = np.zeros((1, 1, L)); x[0, 0, t0] = 1.0
    out = oracle.causal_conv1d(x, w, None, lib=lib)[0, 0]
    expect = np.zeros(L); expect[t0:t0 + W] = w[0, ::-1]
    np.testing.assert_array_equal(out, expect)
    rng = np.random.default_rng(12)
    x2 = rng.standard_normal((2, 3, 9)); w1 = rng.standard_normal((3, 1)); b1 = rng.standard_normal(3)
    out1 = oracle.causal_conv1d(x2, w1, b1, lib=lib)
    np.testing.assert_allclose(out1, x2 * w1[None, :, :] + b1[None, :, None], rtol=1e-15, atol=1e-15)


# --- Gated DeltaNet chunk kernels (Helion hackathon gallery, "GDN chunk_fwd_h" and
# "GDN chunk_fwd_o": per chunk store h, v_new = u - w h, gate exp(g_last - g_t),
# h *= exp(g_last), h += k^T v_gated; o = (q h) exp(g) + causal((q k^T) exp(g_i - g_j)) v_new)

def _gdn_problem(seed, B=2, T=11, H=2, K=3, V=4, chunk=4, w_zero=False, k_zero=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = np.zeros((B, T, H, K)) if k_zero else rng.standard_normal((B, T, H, K)) / 2
    w = np.zeros((B, T, H, K)) if w_zero else rng.standard_normal((B, T, H, K)) / 4
    u = rng.standard_normal((B, T, H, V))
    gamma = -np.abs(rng.normal(0.2, 0.1, (B, T, H)))        # per-token log gates (<= 0)
    g = np.zeros_like(gamma)                                 # in-chunk inclusive cumsum
    for t in range(T):
        g[:, t] = gamma[:, t] + (g[:, t - 1] if t % chunk else 0.0)
    h0 = rng.standard_normal((B, H, K, V))
    return q, k, w, u, gamma, g, h0


def pin_gdn_linear_attention(lib):
    """With w = 0 there is no delta correction (v_new = u) and the two kernels are
    gated linear attention: token by token, S_t = exp(gamma_t) S_{t-1} + k_t u_t^T
    and o_t = q_t^T S_t, whatever the chunk size (brute force on a tiny problem)."""
    for chunk in (1, 3, 4, 16):
        q, k, w, u, gamma, g, h0 = _gdn_problem(21, chunk=chunk, w_zero=True)
        h, v_new, fin = oracle.gdn_fwd_h(k, w, u, g, h0, chunk=chunk, lib=lib)
        o = oracle.gdn_fwd_o(q, k, v_new, h, g, chunk=chunk, lib=lib)
        np.testing.assert_array_equal(v_new, u)
        B, T, H, K = q.shape
        for b in range(B):
            for hh in range(H):
                S = h0[b, hh].copy()
                for t in range(T):
                    S = math.exp(gamma[b, t, hh]) * S + np.outer(k[b, t, hh], u[b, t, hh])
                    np.testing.assert_allclose(o[b, t, hh], q[b, t, hh] @ S, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(fin[b, hh], S, rtol=1e-12, atol=1e-12)


def pin_gdn_hand_example(lib):
    """K = V = 1, one chunk of two tokens, worked by hand: h0 = 2, k = (1, 1),
    w = (0.5, 0.25), u = (3, 1), g = (-0.1, -0.3), q = (1, 2):
    v_new = (2, 0.5); final = 2e^-0.3 + 2e^-0.2 + 0.5;
    o = (2e^-0.1 + 2, 4e^-0.3 + 4e^-0.2 + 1)."""
    sh = lambda a: np.array(a, float).reshape(1, 2, 1, 1)
    k, w, u, q = sh([1, 1]), sh([0.5, 0.25]), sh([3, 1]), sh([1, 2])
    g = np.array([-0.1, -0.3]).reshape(1, 2, 1)
    h0 = np.array(2.0).reshape(1, 1, 1, 1)
    h, v_new, fin = oracle.gdn_fwd_h(k, w, u, g, h0, chunk=2, lib=lib)
    o = oracle.gdn_fwd_o(q, k, v_new, h, g, chunk=2, lib=lib)
    e = math.exp
    np.testing.assert_allclose(h.ravel(), [2.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(v_new.ravel(), [2.0, 0.5], rtol=0, atol=1e-15)
    np.testing.assert_allclose(fin.ravel(), [2 * e(-0.3) + 2 * e(-0.2) + 0.5], rtol=1e-15)
    np.testing.assert_allclose(o.ravel(), [2 * e(-0.1) + 2, 4 * e(-0.3) + 4 * e(-0.2) + 1],
                               rtol=1e-15)


def pin_gdn_k_zero_and_linearity(lib):
    """With k = 0 the state only decays: h_c = h0 exp(sum of the earlier chunks'
    g_last) and v_new = u - w h_c.  For fixed k, w, g the map (u, h0) -> (h, v_new,
    final) is linear."""
    chunk = 4
    q, k, w, u, gamma, g, h0 = _gdn_problem(22, chunk=chunk, k_zero=True)
    h, v_new, fin = oracle.gdn_fwd_h(k, w, u, g, h0, chunk=chunk, lib=lib)
    B, T, H, K = k.shape
    for c in range(h.shape[2]):
        past = np.zeros((B, H))
        for cc in range(c):
            past = past + g[:, min(cc * chunk + chunk, T) - 1]
        hc = h0 * np.exp(past)[:, :, None, None]
        np.testing.assert_allclose(h[:, :, c], hc, rtol=1e-12, atol=1e-12)
        for t in range(c * chunk, min(c * chunk + chunk, T)):
            np.testing.assert_allclose(v_new[:, t], u[:, t] - np.einsum("bhk,bhkv->bhv", w[:, t], hc),
                                       rtol=1e-12, atol=1e-12)
    p1 = _gdn_problem(23, chunk=chunk); p2 = _gdn_problem(24, chunk=chunk)
    _, k, w, u1, _, g, h01 = p1
    u2, h02 = p2[3], p2[6]
    r1 = oracle.gdn_fwd_h(k, w, u1, g, h01, chunk=chunk, lib=lib)
    r2 = oracle.gdn_fwd_h(k, w, u2, g, h02, chunk=chunk, lib=lib)
    r3 = oracle.gdn_fwd_h(k, w, 2 * u1 - u2, g, 2 * h01 - h02, chunk=chunk, lib=lib)
    for a1, a2, a3 in zip(r1, r2, r3):
        np.testing.assert_allclose(a3, 2 * a1 - a2, rtol=1e-10, atol=1e-10)


ALL_PINS = [pin_hand_example, pin_chunked_closed_form, pin_linear_attention, pin_dt_zero,
            pin_geometric, pin_D_isolation, pin_split_composition, pin_linearity,
            pin_checkpoints, pin_chunk_cumsum, pin_conv1d_hand_example, pin_conv1d_library,
            pin_conv1d_impulse_and_causality, pin_gdn_linear_attention, pin_gdn_hand_example,
            pin_gdn_k_zero_and_linearity]
