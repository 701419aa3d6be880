"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one part of the oracle against a closed form worked by hand
(tests/golden/), a library routine the definition reduces to, an invariant
that characterises the result, or brute force by a different route.  A
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong head map or snapshot offset) fails at least one.
"""
import math
import os

import numpy as np
import pytest

from oracle import gdn_oracle as O
from speculative_decode_verify_gdn_gb300.synth import Dims, Dists, Gen, make_layer, make_round, bf16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_named(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *vals = line.split()
            out[name] = np.array([float(v) for v in vals])
    return out


def _tiny_problem(seed=5, B=2, K=5, Hk=2, Hv=4, dk=8, dv=6, W=4, dists=Dists()):
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv, W=W)
    g = Gen(seed)
    lay = make_layer(g, d, dists)
    rnd = make_round(g, d, dists)
    return d, lay, rnd


def _verify(d, lay, rnd, **kw):
    return O.verify_step(d, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                         lay.A_log, lay.dt_bias, lay.conv_w, lay.conv_state, lay.state, **kw)


# ---------------------------------------------------------------- a1 conv

def test_conv_hand_example():
    gd = _read_named(os.path.join(GOLDEN, "conv_step_hand.txt"))
    hist = gd["hist"].reshape(1, 3, 1)
    x = gd["x"].reshape(1, 2, 1)
    w = gd["w"].reshape(1, 4)
    y, inter, hist_out = O.conv_step(x, w, hist)
    pre = gd["pre"]
    expect = pre / (1.0 + np.exp(-pre))
    np.testing.assert_allclose(y[0, :, 0], expect, rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(inter[0, 0, :, 0], gd["hist_after_0"])
    np.testing.assert_array_equal(inter[0, 1, :, 0], gd["hist_after_1"])
    np.testing.assert_array_equal(hist_out[0, :, 0], gd["hist_after_1"])


def test_conv_equals_numpy_correlate():
    """Per channel the conv is numpy.correlate(window, taps, 'valid') followed by SiLU."""
    rng = np.random.default_rng(0)
    B, K, C, W = 2, 7, 5, 4
    x = rng.standard_normal((B, K, C))
    w = rng.standard_normal((C, W))
    hist = rng.standard_normal((B, W - 1, C))
    y, _, _ = O.conv_step(x, w, hist)
    for b in range(B):
        for c in range(C):
            win = np.concatenate([hist[b, :, c], x[b, :, c]])
            z = np.correlate(win, w[c], mode="valid")
            np.testing.assert_allclose(y[b, :, c], z * (0.5 * (1 + np.tanh(z / 2))), rtol=1e-13, atol=1e-14)


def test_conv_one_hot_taps():
    rng = np.random.default_rng(1)
    B, K, C, W = 1, 6, 3, 4
    x = rng.standard_normal((B, K, C))
    hist = rng.standard_normal((B, W - 1, C))
    w_new = np.zeros((C, W)); w_new[:, W - 1] = 1.0
    y, _, _ = O.conv_step(x, w_new, hist)
    np.testing.assert_allclose(y, x / (1 + np.exp(-x)), rtol=1e-15)
    w_old = np.zeros((C, W)); w_old[:, 0] = 1.0
    y, _, _ = O.conv_step(x, w_old, hist)
    lagged = np.concatenate([hist, x[:, :K - (W - 1)]], axis=1)   # y_t = SiLU(win[t]) = x_{t-3}
    np.testing.assert_allclose(y, lagged / (1 + np.exp(-lagged)), rtol=1e-15)


def test_conv_window_equals_token_steps_and_snapshots():
    """A K-token window equals K one-token steps; snapshot t is the history after token t."""
    rng = np.random.default_rng(2)
    B, K, C, W = 2, 5, 4, 4
    x = rng.standard_normal((B, K, C))
    w = rng.standard_normal((C, W))
    hist = rng.standard_normal((B, W - 1, C))
    y, inter, hist_out = O.conv_step(x, w, hist)
    h = hist
    for t in range(K):
        y1, inter1, h = O.conv_step(x[:, t:t + 1], w, h)
        np.testing.assert_array_equal(y1[:, 0], y[:, t])
        np.testing.assert_array_equal(h, inter[:, t])
    np.testing.assert_array_equal(hist_out, h)


# ---------------------------------------------------------------- a2 L2 norm

def test_l2_norm_unit_and_parallel():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((3, 4, 128)) * 3
    n0 = O.l2_normalize(z, 0.0)
    np.testing.assert_allclose(np.linalg.norm(n0, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(n0 * np.linalg.norm(z, axis=-1, keepdims=True), z, rtol=1e-13)
    eps = 1e-6
    n1 = O.l2_normalize(z, eps)
    s = np.sum(z * z, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(n1, axis=-1), np.sqrt(s / (s + eps)), rtol=1e-14)
    assert np.all(np.abs(np.linalg.norm(n1, axis=-1) - 1.0) < 1e-6)


# ---------------------------------------------------------------- a3 gates

def test_raw_gates_closed_form_points():
    rows = np.loadtxt(os.path.join(GOLDEN, "raw_gates_points.txt"), comments="#")
    a, dt, alog, b, beta_ref, g_ref = rows.T
    for i in range(rows.shape[0]):
        beta, g = O.raw_gates(np.array([[[a[i]]]]), np.array([[[b[i]]]]), np.array([alog[i]]), np.array([dt[i]]))
        assert beta.item() == pytest.approx(beta_ref[i], rel=1e-14)
        assert g.item() == pytest.approx(g_ref[i], rel=1e-13)


def test_raw_gates_against_libm_and_threshold():
    z = np.linspace(-30, 40, 1401)
    sp = O.softplus_clipped(z)
    ref = np.array([zz if zz > 20 else math.log1p(math.exp(zz)) for zz in z])
    np.testing.assert_allclose(sp, ref, rtol=1e-15)
    np.testing.assert_allclose(sp[z <= 20], np.logaddexp(0.0, z[z <= 20]), rtol=1e-14)
    # just above the threshold the identity is used (softplus(z) - z < e^-20 there)
    assert O.softplus_clipped(np.array(20.5)).item() == 20.5
    beta, _ = O.raw_gates(np.zeros((1, 1, 3)), np.array([[[-np.inf, 0.0, np.inf]]]), np.zeros(3), np.zeros(3))
    np.testing.assert_array_equal(beta[0, 0], [0.0, 0.5, 1.0])
    _, g = O.raw_gates(np.full((1, 1, 2), 0.3), np.zeros((1, 1, 2)), np.array([-np.inf, np.inf]), np.zeros(2))
    np.testing.assert_array_equal(g[0, 0], [1.0, 0.0])


# ---------------------------------------------------------------- a4 delta rule

def test_delta_rule_hand_example():
    gd = _read_named(os.path.join(GOLDEN, "delta_rule_2x2.txt"))
    S0 = gd["S0"].reshape(1, 1, 2, 2)
    kn = np.stack([gd["k1"], gd["k2"]]).reshape(1, 2, 1, 2)
    qn = np.stack([gd["q1"], gd["q2"]]).reshape(1, 2, 1, 2)
    v = np.stack([gd["v1"], gd["v2"]]).reshape(1, 2, 1, 2)
    beta = np.array([gd["beta1"][0], gd["beta2"][0]]).reshape(1, 2, 1)
    g = np.array([gd["g1"][0], gd["g2"][0]]).reshape(1, 2, 1)
    o, states = O.delta_rule(qn, kn, v, beta, g, S0)
    np.testing.assert_allclose(states[0, 0, 0].ravel(), gd["S1"], atol=1e-15)
    np.testing.assert_allclose(states[0, 1, 0].ravel(), gd["S2"], atol=1e-15)
    np.testing.assert_allclose(o[0, 0, 0], gd["o1"], atol=1e-15)
    np.testing.assert_allclose(o[0, 1, 0], gd["o2"], atol=1e-15)


def _rand_rule(seed, B=2, K=6, Hk=2, Hv=4, dk=7, dv=5):
    rng = np.random.default_rng(seed)
    kn = O.l2_normalize(rng.standard_normal((B, K, Hk, dk)), 0.0)
    qn = O.l2_normalize(rng.standard_normal((B, K, Hk, dk)), 0.0)
    v = rng.standard_normal((B, K, Hv, dv))
    beta = rng.uniform(0.05, 0.95, (B, K, Hv))
    g = rng.uniform(0.3, 1.0, (B, K, Hv))
    S0 = rng.standard_normal((B, Hv, dv, dk)) * 0.3
    return qn, kn, v, beta, g, S0


def test_delta_rule_identity_when_beta0_g1():
    qn, kn, v, beta, g, S0 = _rand_rule(10)
    o, states = O.delta_rule(qn, kn, v, np.zeros_like(beta), np.ones_like(g), S0, q_scale=0.7)
    for t in range(states.shape[1]):
        np.testing.assert_array_equal(states[:, t], S0)
    r = S0.shape[1] // qn.shape[2]
    q_rep = np.repeat(qn, r, axis=2)                               # [B,K,Hv,dk]
    ref = 0.7 * np.matmul(S0[:, None], q_rep[..., None])[..., 0]   # plain matvec S0 q
    np.testing.assert_allclose(o, ref, rtol=1e-13, atol=1e-14)


def test_delta_rule_full_forget_closed_form():
    qn, kn, v, beta, g, S0 = _rand_rule(11)
    o, states = O.delta_rule(qn, kn, v, beta, np.zeros_like(g), S0)
    r = S0.shape[1] // qn.shape[2]
    k_rep = np.repeat(kn, r, axis=2)
    q_rep = np.repeat(qn, r, axis=2)
    S_ref = beta[..., None, None] * v[..., :, None] * k_rep[..., None, :]
    np.testing.assert_allclose(states, S_ref, rtol=1e-14, atol=1e-15)
    o_ref = beta[..., None] * np.sum(k_rep * q_rep, axis=-1)[..., None] * v
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-15)


def test_delta_rule_characterising_invariants():
    """S_t k_t = (1-beta) g S_{t-1} k_t + beta v_t and S_t w = g S_{t-1} w for w orthogonal to k_t.

    These two relations determine S_t uniquely (k_t and its orthogonal
    complement span the key space), so they pin every term of the update.
    """
    qn, kn, v, beta, g, S0 = _rand_rule(12)
    o, states = O.delta_rule(qn, kn, v, beta, g, S0)
    B, K, Hk, dk = kn.shape
    Hv = S0.shape[1]
    rng = np.random.default_rng(99)
    prev = S0
    for t in range(K):
        S = states[:, t]
        for h in range(Hv):
            kh = h // (Hv // Hk)
            k = kn[:, t, kh]
            lhs = np.einsum("bij,bj->bi", S[:, h], k)
            rhs = (1 - beta[:, t, h, None]) * g[:, t, h, None] * np.einsum("bij,bj->bi", prev[:, h], k) \
                + beta[:, t, h, None] * v[:, t, h]
            np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-13)
            w = rng.standard_normal((B, dk))
            w -= np.sum(w * k, axis=-1, keepdims=True) * k          # orthogonal to k_t
            np.testing.assert_allclose(np.einsum("bij,bj->bi", S[:, h], w),
                                       g[:, t, h, None] * np.einsum("bij,bj->bi", prev[:, h], w), rtol=1e-11, atol=1e-12)
            # o_t is the state after token t applied to q_t
            np.testing.assert_allclose(o[:, t, h], np.einsum("bij,bj->bi", S[:, h], qn[:, t, kh]), rtol=1e-13, atol=1e-14)
        # contraction bound: ||S_t|| <= g ||S_{t-1}|| + beta ||v_t||
        nS = np.linalg.norm(S.reshape(B, Hv, -1), axis=-1)
        bound = g[:, t] * np.linalg.norm(prev.reshape(B, Hv, -1), axis=-1) + beta[:, t] * np.linalg.norm(v[:, t], axis=-1)
        assert np.all(nS <= bound * (1 + 1e-12))
        prev = S


def test_delta_rule_beta1_writes_v():
    qn, kn, v, beta, g, S0 = _rand_rule(13)
    _, states = O.delta_rule(qn, kn, v, np.ones_like(beta), g, S0)
    Hk = kn.shape[2]
    r = S0.shape[1] // Hk
    k_rep = np.repeat(kn, r, axis=2)
    np.testing.assert_allclose(np.einsum("btHij,btHj->btHi", states, k_rep), v, rtol=1e-12, atol=1e-13)


def test_delta_rule_equals_transition_matrix_form():
    """Brute force by another route: S_t = g_t S_{t-1} (I - beta_t k k^T) + beta_t v k^T, with explicit
    dk x dk transition matrices and matrix products (the textbook form of the gated delta rule)."""
    qn, kn, v, beta, g, S0 = _rand_rule(14, B=1, K=4, Hk=1, Hv=2, dk=3, dv=3)
    o, states = O.delta_rule(qn, kn, v, beta, g, S0)
    for h in range(2):
        S = S0[0, h].copy()
        for t in range(4):
            k = kn[0, t, 0][:, None]
            T = g[0, t, h] * (np.eye(3) - beta[0, t, h] * (k @ k.T))
            S = S @ T + beta[0, t, h] * (v[0, t, h][:, None] @ k.T)
            np.testing.assert_allclose(states[0, t, h], S, rtol=1e-13, atol=1e-14)


def test_delta_rule_equals_chunk_closed_form():
    """Brute force by the chunk (WY) route: solve the unit lower-triangular system for
    u_t = beta_t (v_t - g_t S_{t-1} k_t) with a library solver, then
    S_t = Gamma_t S0 + sum_j (Gamma_t / Gamma_j) u_j k_j^T."""
    qn, kn, v, beta, g, S0 = _rand_rule(15, B=1, K=6, Hk=1, Hv=1, dk=5, dv=4)
    o, states = O.delta_rule(qn, kn, v, beta, g, S0)
    K = 6
    k = kn[0, :, 0]; q = qn[0, :, 0]; V = v[0, :, 0]; be = beta[0, :, 0]; gg = g[0, :, 0]; S = S0[0, 0]
    Gam = np.cumprod(gg)
    D = np.array([[Gam[t] / Gam[j] if j <= t else 0.0 for j in range(K)] for t in range(K)])
    A = np.eye(K) + np.tril(be[:, None] * D * (k @ k.T), -1)
    rhs = be[:, None] * (V - Gam[:, None] * (k @ S.T))
    U = np.linalg.solve(A, rhs)                                   # rows u_t
    for t in range(K):
        St = Gam[t] * S + sum(D[t, j] * np.outer(U[j], k[j]) for j in range(t + 1))
        np.testing.assert_allclose(states[0, t, 0], St, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o[0, t, 0], St @ q[t], rtol=1e-12, atol=1e-13)


def test_head_broadcast_equals_explicit_repeat():
    """Grouped broadcast (v-head h reads q/k head h // r) equals repeating q/k heads explicitly."""
    qn, kn, v, beta, g, S0 = _rand_rule(16, Hk=2, Hv=6)
    o, states = O.delta_rule(qn, kn, v, beta, g, S0)
    o2, states2 = O.delta_rule(np.repeat(qn, 3, axis=2), np.repeat(kn, 3, axis=2), v, beta, g, S0)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(states, states2)
    # and differs from the interleaved map h % Hk, so the test can tell the two apart
    o3, _ = O.delta_rule(np.tile(qn, (1, 1, 3, 1)), np.tile(kn, (1, 1, 3, 1)), v, beta, g, S0)
    assert np.max(np.abs(o3 - o)) > 1e-3


# ---------------------------------------------------------------- composition, intermediates, rollback

def test_window_equals_one_token_steps():
    d, lay, rnd = _tiny_problem(20)
    full = _verify(d, lay, rnd, q_scale=0.9)
    st, cs = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    d1 = Dims(B=d.B, K=1, Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv, W=d.W)
    for t in range(d.K):
        one = O.verify_step(d1, bf16_bits_to_f32(rnd.x[:, t:t + 1]), bf16_bits_to_f32(rnd.a[:, t:t + 1]),
                            bf16_bits_to_f32(rnd.b[:, t:t + 1]), lay.A_log, lay.dt_bias, lay.conv_w, cs, st, q_scale=0.9)
        np.testing.assert_allclose(one["out"][:, 0], full["out"][:, t], rtol=1e-12, atol=1e-13)
        st, cs = one["state_out"], one["conv_state_out"]
        np.testing.assert_allclose(st, full["states"][:, t], rtol=1e-12, atol=1e-13)
        np.testing.assert_array_equal(cs, full["conv_inter"][:, t])
    np.testing.assert_allclose(st, full["state_out"], rtol=1e-12, atol=1e-13)


def test_intermediates_equal_shorter_runs():
    d, lay, rnd = _tiny_problem(21)
    full = _verify(d, lay, rnd)
    assert full["state_inter"].shape[1] == d.K - 1
    for i in range(d.K - 1):
        dd = Dims(B=d.B, K=i + 1, Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv, W=d.W)
        part = O.verify_step(dd, bf16_bits_to_f32(rnd.x[:, :i + 1]), bf16_bits_to_f32(rnd.a[:, :i + 1]),
                             bf16_bits_to_f32(rnd.b[:, :i + 1]), lay.A_log, lay.dt_bias, lay.conv_w,
                             lay.conv_state, lay.state)
        np.testing.assert_array_equal(part["state_out"], full["state_inter"][:, i])
        np.testing.assert_array_equal(part["conv_state_out"], full["conv_inter"][:, i])


def test_rollback_reproduces_accepted_prefix_run():
    d, lay, rnd = _tiny_problem(22, B=4, K=5)
    full = _verify(d, lay, rnd)
    acc = np.array([0, 2, 5, 1])
    st, cs = O.rollback(acc, lay.state, full["states"], lay.conv_state, full["conv_inter"])
    for bi, L in enumerate(acc):
        if L == 0:
            np.testing.assert_array_equal(st[bi], lay.state[bi])
            np.testing.assert_array_equal(cs[bi], lay.conv_state[bi])
            continue
        dd = Dims(B=d.B, K=int(L), Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv, W=d.W)
        part = O.verify_step(dd, bf16_bits_to_f32(rnd.x[:, :L]), bf16_bits_to_f32(rnd.a[:, :L]),
                             bf16_bits_to_f32(rnd.b[:, :L]), lay.A_log, lay.dt_bias, lay.conv_w,
                             lay.conv_state, lay.state)
        np.testing.assert_array_equal(st[bi], part["state_out"][bi])
        # the history after L tokens is the W-1 newest rows of [hist; x_0..x_{L-1}]
        win = np.concatenate([lay.conv_state[bi], bf16_bits_to_f32(rnd.x[bi, :L])], axis=0)
        np.testing.assert_array_equal(cs[bi], win[-(d.W - 1):])
    with pytest.raises(ValueError):
        O.rollback(np.array([6, 0, 0, 0]), lay.state, full["states"], lay.conv_state, full["conv_inter"])


def test_rollback_resume_equals_concatenated_run():
    """Verify, roll back to L, verify the next window: equals one run over the accepted tokens."""
    d, lay, rnd1 = _tiny_problem(23, B=1, K=4, Hk=1, Hv=2, dk=4, dv=3)
    g = Gen(123)
    rnd2 = make_round(g, d, Dists())
    L = 2
    r1 = _verify(d, lay, rnd1)
    st, cs = O.rollback(np.array([L]), lay.state, r1["states"], lay.conv_state, r1["conv_inter"])
    r2 = O.verify_step(d, bf16_bits_to_f32(rnd2.x), bf16_bits_to_f32(rnd2.a), bf16_bits_to_f32(rnd2.b),
                       lay.A_log, lay.dt_bias, lay.conv_w, cs, st)
    cat = lambda u, w: np.concatenate([u[:, :L], w], axis=1)
    dd = Dims(B=1, K=L + d.K, Hk=1, Hv=2, dk=4, dv=3, W=4)
    ref = O.verify_step(dd, bf16_bits_to_f32(cat(rnd1.x, rnd2.x)), bf16_bits_to_f32(cat(rnd1.a, rnd2.a)),
                        bf16_bits_to_f32(cat(rnd1.b, rnd2.b)), lay.A_log, lay.dt_bias, lay.conv_w,
                        lay.conv_state, lay.state)
    np.testing.assert_allclose(r2["out"], ref["out"][:, L:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r2["state_out"], ref["state_out"], rtol=1e-12, atol=1e-13)


def test_verify_step_splits_channels_q_k_v():
    """Zeroing the conv taps of one slab zeroes its role: with the k slab at zero every key is 0
    (only the eps keeps the norm finite), so the state only decays and o_t = Gamma_t S0 q_t."""
    d, lay, rnd = _tiny_problem(24, K=3)
    w = lay.conv_w.copy()
    w[d.Hk * d.dk:2 * d.Hk * d.dk] = 0.0                        # k slab
    res = O.verify_step(d, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                        lay.A_log, lay.dt_bias, w, lay.conv_state, lay.state)
    beta, g = O.raw_gates(bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b), lay.A_log, lay.dt_bias)
    gam = np.cumprod(g, axis=1)                                  # [B,K,Hv]
    for t in range(d.K):
        np.testing.assert_allclose(res["states"][:, t], gam[:, t, :, None, None] * lay.state, rtol=1e-12)


# ---------------------------------------------------------------- token trees

def _tree_problem(seed, parent, Hk=2, Hv=4, dk=6, dv=5):
    parent = np.asarray(parent)
    B, K = parent.shape
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(seed)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    return d, lay, rnd


def _tree(d, lay, rnd, parent, **kw):
    return O.tree_verify_step(d, parent, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                              lay.A_log, lay.dt_bias, lay.conv_w, lay.conv_state, lay.state, **kw)


def test_tree_of_a_chain_equals_the_window():
    parent = np.array([[-1, 0, 1, 2, 3, 4], [-1, 0, 1, 2, 3, 4]])
    d, lay, rnd = _tree_problem(40, parent)
    tr = _tree(d, lay, rnd, parent, q_scale=0.8)
    ch = _verify(d, lay, rnd, q_scale=0.8)
    for key in ("out", "states", "conv_inter", "y"):
        np.testing.assert_allclose(tr[key], ch[key], rtol=1e-13, atol=1e-14)


def test_tree_nodes_equal_their_root_paths():
    """Each node's output, state and history equal a plain window over its root-to-node path."""
    parent = np.array([[-1, 0, 0, 1, -1, 3, 2, 6, 1], [-1, -1, 1, 0, 3, 3, 5, 2, 7]])
    d, lay, rnd = _tree_problem(41, parent)
    tr = _tree(d, lay, rnd, parent)
    for bi in range(parent.shape[0]):
        for t in range(parent.shape[1]):
            path = O.tree_path(parent[bi], t)
            dd = Dims(B=1, K=len(path), Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv)
            sl = lambda z: z[bi:bi + 1][:, path]
            ch = O.verify_step(dd, bf16_bits_to_f32(sl(rnd.x)), bf16_bits_to_f32(sl(rnd.a)), bf16_bits_to_f32(sl(rnd.b)),
                               lay.A_log, lay.dt_bias, lay.conv_w, lay.conv_state[bi:bi + 1], lay.state[bi:bi + 1])
            np.testing.assert_allclose(tr["out"][bi, t], ch["out"][0, -1], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(tr["states"][bi, t], ch["state_out"][0], rtol=1e-12, atol=1e-13)
            np.testing.assert_array_equal(tr["conv_inter"][bi, t], ch["conv_state_out"][0])


def test_tree_star_is_independent_one_token_steps():
    """All nodes children of the committed state: each is a one-token step from S0 (no
    node sees another), so permuting the nodes permutes the results."""
    parent = np.full((1, 5), -1)
    d, lay, rnd = _tree_problem(42, parent)
    tr = _tree(d, lay, rnd, parent)
    perm = np.array([3, 0, 4, 1, 2])
    from speculative_decode_verify_gdn_gb300.synth import Round
    rp = Round(rnd.x[:, perm], rnd.a[:, perm], rnd.b[:, perm], rnd.accept_len)
    tp = _tree(d, lay, rp, parent)
    np.testing.assert_allclose(tp["out"], tr["out"][:, perm], rtol=1e-13)
    np.testing.assert_allclose(tp["states"], tr["states"][:, perm], rtol=1e-13)


def test_tree_rejects_bad_parents():
    parent = np.array([[-1, 0, 2]])
    d, lay, rnd = _tree_problem(43, parent)
    with pytest.raises(ValueError):
        _tree(d, lay, rnd, parent)


# ---------------------------------------------------------------- gated output norm

def test_gated_norm_hand_example():
    gd = _read_named(os.path.join(GOLDEN, "gated_norm_hand.txt"))
    out = O.gated_rms_norm(gd["o"], gd["z"], gd["w"], eps=gd["eps"][0])
    np.testing.assert_allclose(out, gd["out"], rtol=1e-15, atol=1e-15)


def test_gated_norm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(7)
    o = rng.standard_normal((3, 5, 128))
    z = rng.standard_normal((3, 5, 128))
    w = rng.uniform(0.5, 1.5, 128)
    a = O.gated_rms_norm(o, z, w, eps=0.0)
    np.testing.assert_allclose(O.gated_rms_norm(7.5 * o, z, w, eps=0.0), a, rtol=1e-13)
    # dividing out weight and gate leaves a vector of unit RMS
    core = a / (w * (z / (1 + np.exp(-z))))
    np.testing.assert_allclose(np.sqrt(np.mean(core ** 2, axis=-1)), 1.0, rtol=1e-12)
    # the gate enters through SiLU only: z -> large makes the gate the identity on z
    big = O.gated_rms_norm(o, np.full_like(z, 40.0), np.ones(128), eps=0.0)
    np.testing.assert_allclose(big, 40.0 * o / np.sqrt(np.mean(o ** 2, axis=-1, keepdims=True)), rtol=1e-13)


# ---------------------------------------------------------------- prefill (whole prompts, packed)
def _prefill_problem(seed, lens, Hk=2, Hv=4, dk=8, dv=6, dists=Dists()):
    """Ragged prompts packed token-major, with the per-prompt state and history."""
    B, N = len(lens), int(sum(lens))
    d = Dims(B=B, K=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(seed)
    lay = make_layer(g, d, dists)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = g.normal((N, d.C), 1.0)
    a = g.normal((N, Hv), 1.0)
    b = g.normal((N, Hv), 1.0)
    return d, lay, cu, x, a, b


def _prefill(d, lay, cu, x, a, b, state=None, conv=None, block=64):
    return O.prefill(d, cu, x, a, b, lay.A_log, lay.dt_bias, lay.conv_w,
                     lay.conv_state if conv is None else conv, lay.state if state is None else state,
                     q_scale=0.9, block=block)


def test_prefill_is_independent_of_the_token_block():
    """Feeding the prompt in blocks of 64, 5 or 1 tokens does the same per-token arithmetic,
    so the results agree bit for bit: the state and history are carried across blocks."""
    d, lay, cu, x, a, b = _prefill_problem(31, [23, 9])
    r64 = _prefill(d, lay, cu, x, a, b, block=64)
    for blk in (5, 1):
        r = _prefill(d, lay, cu, x, a, b, block=blk)
        for key in ("out", "state_out", "conv_state_out"):
            np.testing.assert_array_equal(r[key], r64[key])


def test_prefill_packing_equals_prompts_alone():
    lens = [7, 0, 13, 2, 1]
    d, lay, cu, x, a, b = _prefill_problem(32, lens)
    r = _prefill(d, lay, cu, x, a, b)
    for i in range(len(lens)):
        s, e = int(cu[i]), int(cu[i + 1])
        d1 = Dims(B=1, K=1, Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv)
        r1 = O.prefill(d1, [0, e - s], x[s:e], a[s:e], b[s:e], lay.A_log, lay.dt_bias, lay.conv_w,
                       lay.conv_state[i:i + 1], lay.state[i:i + 1], q_scale=0.9)
        np.testing.assert_array_equal(r["out"][s:e], r1["out"])
        np.testing.assert_array_equal(r["state_out"][i], r1["state_out"][0])
        np.testing.assert_array_equal(r["conv_state_out"][i], r1["conv_state_out"][0])


def test_prefill_empty_prompt_keeps_state_and_history():
    d, lay, cu, x, a, b = _prefill_problem(33, [0, 4])
    r = _prefill(d, lay, cu, x, a, b)
    np.testing.assert_array_equal(r["state_out"][0], lay.state[0])
    np.testing.assert_array_equal(r["conv_state_out"][0], lay.conv_state[0])


def test_prefill_split_prompt_equals_one_call():
    """A prompt prefilled in two calls, the second starting from the first's state and
    history, equals one call over the whole prompt."""
    d, lay, cu, x, a, b = _prefill_problem(34, [30])
    whole = _prefill(d, lay, cu, x, a, b)
    first = _prefill(d, lay, np.array([0, 12]), x[:12], a[:12], b[:12])
    second = _prefill(d, lay, np.array([0, 18]), x[12:], a[12:], b[12:], state=first["state_out"],
                      conv=first["conv_state_out"])
    np.testing.assert_allclose(np.concatenate([first["out"], second["out"]]), whole["out"], rtol=0, atol=0)
    np.testing.assert_array_equal(second["state_out"], whole["state_out"])
    np.testing.assert_array_equal(second["conv_state_out"], whole["conv_state_out"])


def test_prefill_zero_input_tail_is_pure_decay():
    """Once the W-1 history rows have left the conv window, an all-zero input has q = k = v = 0:
    the outputs vanish and the state only decays, S_T = (prod of g over those tokens) S."""
    lens = [70]
    d, lay, cu, x, a, b = _prefill_problem(35, lens)
    x[:] = 0.0
    r = _prefill(d, lay, cu, x, a, b)
    W = d.W
    head = _prefill(d, lay, np.array([0, W - 1]), x[:W - 1], a[:W - 1], b[:W - 1])
    _, g = O.raw_gates(a[W - 1:], b[W - 1:], lay.A_log, lay.dt_bias)
    decay = np.prod(g, axis=0)                                   # [Hv]
    np.testing.assert_allclose(r["state_out"][0], decay[:, None, None] * head["state_out"][0], rtol=1e-12, atol=0)
    assert np.all(r["out"][W - 1:] == 0.0)
    assert np.all(r["conv_state_out"][0] == 0.0)


def test_prefill_rejects_bad_seqlens():
    d, lay, cu, x, a, b = _prefill_problem(36, [4, 4])
    for bad in ([0, 5, 4], [1, 4, 8], [0, 4, 7]):
        with pytest.raises(ValueError):
            _prefill(d, lay, np.array(bad), x, a, b)
