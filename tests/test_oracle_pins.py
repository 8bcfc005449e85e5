"""Pins of the fp64 oracle to things other than itself.

Each test fixes one part of the oracle against brute force, a closed form, an
identity of the mathematics, or an independently written formulation, chosen
so that a plausible mistake (a dropped term, a flipped sign, a transposed
state, a wrong tap order or head mapping) fails at least one of them.
"""
import numpy as np
import pytest
from scipy.linalg import solve_triangular
from scipy.special import expit

import oracle
from gated_deltanet_state_gb300 import inputs

rng = np.random.default_rng(1234)


def _unit(n, T):
    k = rng.standard_normal((T, n))
    return k / np.linalg.norm(k, axis=1, keepdims=True)


def _case(T=6, dk=4, dv=3, S0_scale=0.5):
    q = _unit(dk, T)
    k = _unit(dk, T)
    v = rng.standard_normal((T, dv))
    a = np.exp(-rng.uniform(0.0, 0.5, T))
    b = rng.uniform(0.05, 0.95, T)
    S0 = S0_scale * rng.standard_normal((dv, dk))
    return q, k, v, a, b, S0


def product_form(q, k, v, a, b, S0):
    """Unrolled closed form of the gated delta rule, with dense matrices:
    S_T = S0 prod_t (a_t M_t) + sum_t b_t v_t k_t^T prod_{s>t} (a_s M_s),
    M_t = I - b_t k_t k_t^T (products left to right in t); o_t = S_t q_t."""
    T, dk = k.shape
    M = [a[t] * (np.eye(dk) - b[t] * np.outer(k[t], k[t])) for t in range(T)]
    outs, S_t = [], None
    for tt in range(1, T + 1):
        P = np.eye(dk)
        for t in range(tt):
            P = P @ M[t]
        S_t = S0 @ P
        for t in range(tt):
            R = np.eye(dk)
            for s in range(t + 1, tt):
                R = R @ M[s]
            S_t = S_t + b[t] * np.outer(v[t], k[t]) @ R
        outs.append(S_t @ q[tt - 1])
    return S_t, np.array(outs)


def chunk_form(q, k, v, g, b, S0, C):
    """Chunked (WY / UT-transform) formulation, written independently of the
    token loop.  Per chunk with start state S0 and in-chunk cumulative log
    decay G: A_ij = b_i e^{G_i-G_j} k_i.k_j (j < i), T = (I+A)^{-1},
    U = T (diag(b) V - diag(b e^G) K S0^T), O = diag(e^G) Q S0^T + P U with
    P_ij = e^{G_i-G_j} q_i.k_j (j <= i), S_C = e^{G_C} S0 + U^T diag(e^{G_C-G}) K."""
    Tn = k.shape[0]
    S = S0.copy()
    outs = []
    for c0 in range(0, Tn, C):
        Q, K, V = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C]
        gc, bc = g[c0:c0 + C], b[c0:c0 + C]
        n = K.shape[0]
        G = np.cumsum(gc)
        D = np.exp(G[:, None] - G[None, :])
        A = np.tril(bc[:, None] * D * (K @ K.T), -1)
        rhs = bc[:, None] * V - (bc * np.exp(G))[:, None] * (K @ S.T)
        U = solve_triangular(np.eye(n) + A, rhs, lower=True, unit_diagonal=True)
        P = np.tril(D * (Q @ K.T))
        outs.append(np.exp(G)[:, None] * (Q @ S.T) + P @ U)
        S = np.exp(G[-1]) * S + U.T @ (np.exp(G[-1] - G)[:, None] * K)
    return S, np.concatenate(outs)


# --------------------------------------------------------------- recurrence

def test_recurrence_matches_product_form():
    for trial in range(4):
        q, k, v, a, b, S0 = _case(T=5 + trial, dk=4, dv=3)
        S, o = oracle.recurrence(q, k, v, a, b, S0)
        S_ref, o_ref = product_form(q, k, v, a, b, S0)
        np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)


def test_recurrence_nonsquare_state_orientation():
    # dv != dk catches a transposed state (S is [dv][dk], o = S q has dv rows).
    q, k, v, a, b, S0 = _case(T=4, dk=5, dv=2)
    S, o = oracle.recurrence(q, k, v, a, b, S0)
    S_ref, o_ref = product_form(q, k, v, a, b, S0)
    assert S.shape == (2, 5) and o.shape == (4, 2)
    np.testing.assert_allclose(S, S_ref, atol=1e-12)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)


def test_identity_no_write_no_decay_is_exact():
    q, k, v, a, b, S0 = _case(T=7)
    S, o = oracle.recurrence(q, k, v, np.ones(7), np.zeros(7), S0)
    assert np.array_equal(S, S0)
    np.testing.assert_allclose(o, (S0 @ q.T).T, atol=1e-14)


def test_identity_no_write_pure_decay():
    q, k, v, a, b, S0 = _case(T=7)
    S, _ = oracle.recurrence(q, k, v, a, np.zeros(7), S0)
    np.testing.assert_allclose(S, np.prod(a) * S0, rtol=1e-13, atol=1e-15)


def test_identity_delta_rule_retrieval():
    # b = 1 and unit k: the state maps k_t exactly onto v_t after step t.
    q, k, v, a, b, S0 = _case(T=6)
    for t in range(1, 7):
        S, _ = oracle.recurrence(q[:t], k[:t], v[:t], a[:t], np.ones(t), S0)
        np.testing.assert_allclose(S @ k[t - 1], v[t - 1], atol=1e-12)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunk_form_equals_recurrence(C):
    T, dk, dv = 150, 16, 8
    q, k = _unit(dk, T), _unit(dk, T)
    v = rng.standard_normal((T, dv))
    g = -np.log1p(np.exp(rng.standard_normal(T))) * 0.1
    b = expit(rng.standard_normal(T))
    S0 = 0.3 * rng.standard_normal((dv, dk))
    S, o = oracle.recurrence(q, k, v, np.exp(g), b, S0)
    S_c, o_c = chunk_form(q, k, v, g, b, S0, C)
    np.testing.assert_allclose(S, S_c, rtol=0, atol=1e-10)
    np.testing.assert_allclose(o, o_c, rtol=0, atol=1e-10)


# --------------------------------------------------------------- conv, norm

def test_conv_impulse_gives_silu_of_taps_in_reverse():
    w = np.array([[0.7, -1.3, 0.4, 2.1]])
    x = np.zeros((7, 1))
    x[0, 0] = 1.0
    y = oracle.conv_silu(x, np.zeros((3, 1)), w)[:, 0]
    silu = lambda z: z * expit(z)
    # tap 3 multiplies the current row, tap 0 the row three steps back
    np.testing.assert_allclose(y[:4], silu(w[0, ::-1]), atol=1e-15)
    np.testing.assert_allclose(y[4:], 0.0, atol=0)


def test_conv_window_row0_is_oldest():
    w = np.array([[0.7, -1.3, 0.4, 2.1]])
    silu = lambda z: z * expit(z)
    for r in range(3):
        win = np.zeros((3, 1))
        win[r, 0] = 1.0
        y = oracle.conv_silu(np.zeros((4, 1)), win, w)[:, 0]
        # window row r sits at position r-3; it meets tap (r - t) at row t
        expect = [silu(w[0, r - t]) if r - t >= 0 else 0.0 for t in range(4)]
        np.testing.assert_allclose(y, expect, atol=1e-15)


def test_conv_window_carry_splits_exactly():
    cd = 5
    x = rng.standard_normal((12, cd))
    w = rng.standard_normal((cd, 4))
    win = rng.standard_normal((3, cd))
    full = oracle.conv_silu(x, win, w)
    first = oracle.conv_silu(x[:7], win, w)
    second = oracle.conv_silu(x[7:], x[4:7], w)
    assert np.array_equal(full, np.concatenate([first, second]))


def test_l2norm_closed_form():
    v = rng.standard_normal(33)
    out = oracle.l2norm(v, scale=0.5, eps=1e-6)
    np.testing.assert_allclose(out, 0.5 * v / np.sqrt(np.sum(v * v) + 1e-6), rtol=1e-15)
    np.testing.assert_allclose(np.linalg.norm(oracle.l2norm(v, 1.0, 0.0)), 1.0, rtol=1e-15)


# --------------------------------------------------------------- full layer

def _numpy_layer(d, x, g, beta, w, S0, win0):
    """The whole layer written out in numpy for a tiny case: conv with scipy's
    SiLU, explicit channel split, blocked head mapping, product-form state."""
    xh = np.concatenate([win0, x])
    T = x.shape[0]
    z = sum(w[:, i][None, :] * xh[i:i + T] for i in range(4))
    y = z * expit(z)
    o = np.zeros((T, d.Hv, d.dv))
    S_out = np.zeros((d.Hv, d.dv, d.dk))
    for h in range(d.Hv):
        j = h // (d.Hv // d.Hqk)
        q = y[:, j * d.dk:(j + 1) * d.dk]
        k = y[:, d.Hqk * d.dk + j * d.dk:d.Hqk * d.dk + (j + 1) * d.dk]
        v = y[:, 2 * d.Hqk * d.dk + h * d.dv:2 * d.Hqk * d.dk + (h + 1) * d.dv]
        q = d.q_scale * q / np.sqrt((q * q).sum(1, keepdims=True) + d.eps)
        k = k / np.sqrt((k * k).sum(1, keepdims=True) + d.eps)
        S_out[h], o[:, h] = product_form(q, k, v, np.exp(g[:, h]), beta[:, h], S0[h])
    return o, S_out


def test_layer_matches_numpy_brute_force():
    d = oracle.Dims(Hqk=2, Hv=4, dk=3, dv=2, q_scale=0.7)
    T = 6
    x = rng.standard_normal((T, d.conv_dim))
    g = -np.log1p(np.exp(rng.standard_normal((T, d.Hv)))) * 0.1
    beta = expit(rng.standard_normal((T, d.Hv)))
    w = 0.5 * rng.standard_normal((d.conv_dim, 4))
    S0 = 0.3 * rng.standard_normal((d.Hv, d.dv, d.dk))
    win0 = rng.standard_normal((3, d.conv_dim))
    r = oracle.prefill(d, [0, T], [0], 1 << 40, x, g, beta, w, S0[None], win0[None])
    o_ref, S_ref = _numpy_layer(d, x, g, beta, w, S0, win0)
    np.testing.assert_allclose(r["o"], o_ref, atol=1e-12)
    np.testing.assert_allclose(r["S"][0], S_ref, atol=1e-12)
    assert np.array_equal(r["win"][0], x[-3:])


def test_head_mapping_is_blocked():
    # Zero taps on the q/k channels of qk head 1: only v heads 2 and 3 (the
    # blocked mapping h -> h // (Hv/Hqk)) see k = 0 and keep a zero state.
    d = oracle.Dims(Hqk=2, Hv=4, dk=4, dv=4)
    T = 5
    x = rng.standard_normal((T, d.conv_dim))
    w = rng.standard_normal((d.conv_dim, 4))
    for base in (0, d.Hqk * d.dk):
        w[base + d.dk:base + 2 * d.dk] = 0.0
    g = np.full((T, d.Hv), -0.05)
    beta = np.full((T, d.Hv), 0.5)
    r = oracle.prefill(d, [0, T], [0], 1 << 40, x, g, beta, w)
    S = r["S"][0]
    assert np.all(S[2:] == 0.0) and np.all(r["o"][:, 2:] == 0.0)
    assert np.all(np.abs(S[:2]).sum(axis=(1, 2)) > 0)


# --------------------------------------------------------------- checkpoints

def _tiny_inputs(T, seed=0, shape=inputs.TINY):
    ti = inputs.token_inputs(shape, T, seed)
    return ti["x"], ti["g"], ti["beta"], inputs.conv_weights(shape, seed)


def _dims(shape):
    return oracle.Dims(shape.num_qk_heads, shape.num_v_heads, shape.head_dim_k, shape.head_dim_v,
                       shape.q_scale, shape.norm_eps)


def test_checkpoint_is_state_after_block():
    sh = inputs.TINY
    d = _dims(sh)
    x, g, beta, w = _tiny_inputs(256)
    full = oracle.prefill(d, [0, 256], [0], sh.block_size, x, g, beta, w)
    assert full["ck_S"].shape[0] == 4  # boundaries 64, 128, 192, 256
    for j, P in enumerate([64, 128, 192, 256]):
        part = oracle.prefill(d, [0, P], [0], 1 << 40, x[:P], g[:P], beta[:P], w)
        assert np.array_equal(full["ck_S"][j], part["S"][0])
        assert np.array_equal(full["ck_win"][j], part["win"][0])


def test_resume_from_checkpoint_equals_cold_bitwise():
    sh = inputs.TINY
    d = _dims(sh)
    x, g, beta, w = _tiny_inputs(256)
    cold = oracle.prefill(d, [0, 256], [0], sh.block_size, x, g, beta, w)
    P = 192  # hit at 3 blocks -> resume from block 2 (state after 192 tokens)
    res = oracle.prefill(d, [0, 256 - P], [P], sh.block_size, x[P:], g[P:], beta[P:], w,
                         cold["ck_S"][2][None], cold["ck_win"][2][None])
    assert np.array_equal(res["o"], cold["o"][P:])
    assert np.array_equal(res["S"], cold["S"])
    assert np.array_equal(res["ck_S"][0], cold["ck_S"][3])


def test_batch_of_sequences_is_independent():
    sh = inputs.TINY
    d = _dims(sh)
    xa, ga, ba, w = _tiny_inputs(100, seed=1)
    xb, gb, bb, _ = _tiny_inputs(70, seed=2)
    both = oracle.prefill(d, [0, 100, 170], [0, 0], sh.block_size,
                          np.concatenate([xa, xb]), np.concatenate([ga, gb]), np.concatenate([ba, bb]), w)
    a = oracle.prefill(d, [0, 100], [0], sh.block_size, xa, ga, ba, w)
    b = oracle.prefill(d, [0, 70], [0], sh.block_size, xb, gb, bb, w)
    assert np.array_equal(both["o"][:100], a["o"]) and np.array_equal(both["o"][100:], b["o"])
    assert np.array_equal(both["S"][1], b["S"][0])


def test_decode_equals_one_token_prefill_and_chains():
    sh = inputs.TINY
    d = _dims(sh)
    x, g, beta, w = _tiny_inputs(9)
    full = oracle.prefill(d, [0, 9], [0], 1 << 40, x, g, beta, w)
    part = oracle.prefill(d, [0, 8], [0], 1 << 40, x[:8], g[:8], beta[:8], w)
    o, S, win = oracle.decode(d, x[8:9], g[8:9], beta[8:9], w, part["S"], part["win"])
    assert np.array_equal(o[0], full["o"][8])
    assert np.array_equal(S, full["S"]) and np.array_equal(win, full["win"])


# --------------------------------------------------------------- replay

def test_replay_flush_after_rollback_equals_accepted_only():
    sh = inputs.TINY
    d = _dims(sh)
    N, m, L = 3, 5, oracle.CONV_K * 8
    x, g, beta, w = _tiny_inputs(40)
    st = inputs.random_state(sh, N, 3)
    S0, win0 = st["S"].double().numpy(), st["win"].double().numpy()
    log_x = np.zeros((N, 32, d.conv_dim)); log_g = np.zeros((N, 32, d.Hv)); log_b = np.zeros((N, 32, d.Hv))
    n0 = np.array([0, 2, 4])
    xs = x.double().numpy().reshape(-1)[:N * 12 * d.conv_dim].reshape(N, 12, d.conv_dim)
    gs = g.double().numpy()[:36].reshape(N, 12, d.Hv)
    bs = beta.double().numpy()[:36].reshape(N, 12, d.Hv)
    for r in range(N):
        log_x[r, :n0[r]] = xs[r, :n0[r]]; log_g[r, :n0[r]] = gs[r, :n0[r]]; log_b[r, :n0[r]] = bs[r, :n0[r]]
    new_x = np.stack([xs[r, n0[r]:n0[r] + m] for r in range(N)])
    new_g = np.stack([gs[r, n0[r]:n0[r] + m] for r in range(N)])
    new_b = np.stack([bs[r, n0[r]:n0[r] + m] for r in range(N)])
    o_new = oracle.replay_append(d, w, S0, win0, log_x, log_g, log_b, n0, new_x, new_g, new_b)
    accepted = np.array([0, 3, 5])
    for r in range(N):
        log_x[r, n0[r]:n0[r] + m] = new_x[r]; log_g[r, n0[r]:n0[r] + m] = new_g[r]; log_b[r, n0[r]:n0[r] + m] = new_b[r]
    lens = oracle.replay_rollback(n0 + m, accepted, m)
    assert list(lens) == list(n0 + accepted)
    S1, win1 = oracle.replay_flush(d, w, S0, win0, log_x, log_g, log_b, lens)
    for r in range(N):
        T = n0[r] + m
        seq = oracle.prefill(d, [0, T], [0], 1 << 40, xs[r, :T], gs[r, :T], bs[r, :T], w,
                             S0[r][None], win0[r][None])
        # append outputs = the sequential outputs of the new rows
        np.testing.assert_allclose(o_new[r], seq["o"][n0[r]:T], rtol=0, atol=1e-13)
        keep = n0[r] + accepted[r]
        ref = oracle.prefill(d, [0, keep], [0], 1 << 40, xs[r, :keep], gs[r, :keep], bs[r, :keep], w,
                             S0[r][None], win0[r][None])
        np.testing.assert_allclose(S1[r], ref["S"][0], rtol=0, atol=1e-13)
        assert np.array_equal(win1[r], ref["win"][0])


def test_replay_flush_of_empty_log_is_identity():
    sh = inputs.TINY
    d = _dims(sh)
    st = inputs.random_state(sh, 2, 5)
    S0, win0 = st["S"].double().numpy(), st["win"].double().numpy()
    z = np.zeros((2, 32, d.conv_dim)); zg = np.zeros((2, 32, d.Hv))
    S1, win1 = oracle.replay_flush(d, inputs.conv_weights(sh, 0), S0, win0, z, zg, zg, [0, 0])
    assert np.array_equal(S1, S0) and np.array_equal(win1, win0)


# ---------------------------------------------------------------- packed core
# "Hybrid linear attention (gated DeltaNet)", "Packed-core traces": gates from
# the packed b | a rows with dt_bias and A_log, gated RMS norm of the outputs.

def test_core_gates_closed_forms():
    import math
    Hv = 2
    # b | a order: b = ln 3 gives beta = 3/4; a = 0, dt_bias = 0, A_log = 0 gives g = -ln 2
    g, beta = oracle.core_gates([[math.log(3.0), 0.0, 0.0, 0.0]], [0.0, 0.0], [0.0, 0.0], Hv)
    assert beta[0, 0] == pytest.approx(0.75, abs=1e-15) and beta[0, 1] == pytest.approx(0.5, abs=1e-15)
    assert g[0, 0] == pytest.approx(-math.log(2.0), abs=1e-15)
    # A_log = ln 3 scales the decay by 3; dt_bias shifts a
    g, _ = oracle.core_gates([[0.0, 0.0, 1.0, -1.0]], [math.log(3.0), 0.0], [0.0, 1.0], Hv)
    assert g[0, 0] == pytest.approx(-3.0 * math.log1p(math.e), rel=1e-14)
    assert g[0, 1] == pytest.approx(-math.log(2.0), rel=1e-14)
    # tails: softplus(40) = 40 + log1p(e^-40); softplus(-40) = log1p(e^-40)
    g, _ = oracle.core_gates([[0.0, 0.0, 40.0, -40.0]], [0.0, 0.0], [0.0, 0.0], Hv)
    assert g[0, 0] == pytest.approx(-(40.0 + math.log1p(math.exp(-40.0))), rel=1e-15)
    assert g[0, 1] == pytest.approx(-math.log1p(math.exp(-40.0)), rel=1e-12)


def test_gated_rmsnorm_closed_forms():
    import math
    silu2 = 2.0 / (1.0 + math.exp(-2.0))
    # o = (3, 4), eps = 0: rms = sqrt(12.5)
    y = oracle.gated_rmsnorm([3.0, 4.0], [2.0, 2.0], [1.0, 0.5], 0.0)
    r = math.sqrt(12.5)
    assert y[0] == pytest.approx(3.0 / r * silu2, rel=1e-15)
    assert y[1] == pytest.approx(4.0 / r * 0.5 * silu2, rel=1e-15)
    # a constant vector normalises to its sign (eps = 0), with eps: 1 / sqrt(1 + eps / c^2)
    y = oracle.gated_rmsnorm(np.full(8, -0.25), np.full(8, 2.0), np.ones(8), 0.0)
    assert np.allclose(y, -silu2, rtol=1e-15, atol=0)
    y = oracle.gated_rmsnorm(np.full(8, 0.5), np.full(8, 2.0), np.ones(8), 0.25)
    assert np.allclose(y, silu2 / math.sqrt(2.0), rtol=1e-15, atol=0)
    # scale and sign invariance (eps = 0); a zero gate zeroes the row
    rng = np.random.default_rng(3)
    o, z, w = rng.normal(size=16), rng.normal(size=16), rng.normal(size=16)
    assert np.allclose(oracle.gated_rmsnorm(7.5 * o, z, w, 0.0), oracle.gated_rmsnorm(o, z, w, 0.0), rtol=1e-13)
    assert np.allclose(oracle.gated_rmsnorm(-o, z, w, 0.0), -oracle.gated_rmsnorm(o, z, w, 0.0), rtol=1e-13)
    assert np.all(oracle.gated_rmsnorm(o, np.zeros(16), w, 1e-6) == 0.0)


def test_core_prefill_is_the_recurrence_on_the_qkv_part():
    """The packed core splits each row into x = q | k | v and z and takes its
    gates from b | a: the states equal the plain prefill's on (x, g, beta),
    and y is the gated norm of its outputs."""
    d = oracle.Dims(1, 2, 4, 4)
    T = 9
    rng = np.random.default_rng(5)
    x = rng.normal(size=(T, d.conv_dim))
    z = rng.normal(size=(T, d.Hv * d.dv))
    ba = rng.normal(size=(T, 2 * d.Hv))
    A_log, dt_bias, nw = rng.normal(size=d.Hv) * 0.3, rng.normal(size=d.Hv) * 0.3, rng.normal(size=d.dv)
    w = rng.normal(size=(d.conv_dim, 4)) * 0.5
    r = oracle.core_prefill(d, [0, T], [0], 4, np.concatenate([x, z], 1), ba, w, A_log, dt_bias, nw, 1e-6)
    # gates written out by hand for token 3, head 1
    b, a = ba[3, 1], ba[3, d.Hv + 1]
    g31 = -np.exp(A_log[1]) * np.log1p(np.exp(a + dt_bias[1]))
    beta31 = 1.0 / (1.0 + np.exp(-b))
    g, beta = oracle.core_gates(ba, A_log, dt_bias, d.Hv)
    assert g[3, 1] == pytest.approx(g31, rel=1e-13) and beta[3, 1] == pytest.approx(beta31, rel=1e-14)
    ref = oracle.prefill(d, [0, T], [0], 4, x, g, beta, w)
    assert np.array_equal(r["S"], ref["S"]) and np.array_equal(r["o"], ref["o"])
    o = ref["o"][5, 0]
    y = o / np.sqrt(np.mean(o * o) + 1e-6) * nw * (z[5, :d.dv] / (1.0 + np.exp(-z[5, :d.dv])))
    assert np.allclose(r["y"][5, 0], y, rtol=1e-13, atol=1e-15)
