"""Pins of the dense per-token transition scan oracle (``oracle/frame_scan.py``).

The scan follows SANA's distributed_scan.py page (cp_frame_gdn_scan and its local scan):
KV state S[t] = S[t-1] @ W_kv[t] + U_kv[t] (right multiply), Z state
s[t] = W_z[t] @ s[t-1] + u_z[t] (left multiply), truncate_to_active, and the
context-parallel correction over segments. Each pin below is fixed by the mathematics, not
by the oracle's own formula: closed forms of scalar and diagonal transitions, the product
form with zero input, the transposition identity between the two conventions, and the
segment-split identity that the page's correction rests on (linearity of the recurrence).
"""
import numpy as np
import pytest

from oracle import frame_scan as F


def rand_case(rng, BH=2, T=9, D=4, contraction=0.6):
    W_kv = contraction * rng.standard_normal((BH, T, D, D)) / np.sqrt(D)
    W_z = contraction * rng.standard_normal((BH, T, D, D)) / np.sqrt(D)
    U_kv = rng.standard_normal((BH, T, D, D))
    u_z = rng.standard_normal((BH, T, D))
    S0 = rng.standard_normal((BH, D, D))
    s0 = rng.standard_normal((BH, D))
    return W_kv, U_kv, W_z, u_z, S0, s0


def test_identity_transitions_accumulate_inputs():
    # W = I: S[t] = S0 + sum_{s<=t} U[s]; with a constant input that is S0 + (t+1) U
    rng = np.random.default_rng(1)
    BH, T, D = 2, 7, 3
    eye = np.broadcast_to(np.eye(D), (BH, T, D, D))
    C = rng.standard_normal((BH, 1, D, D))
    c = rng.standard_normal((BH, 1, D))
    S0 = rng.standard_normal((BH, D, D))
    s0 = rng.standard_normal((BH, D))
    S, s, St, st = F.scan(eye, np.broadcast_to(C, (BH, T, D, D)), eye, np.broadcast_to(c, (BH, T, D)), S0, s0)
    for t in range(T):
        np.testing.assert_allclose(S[:, t], S0 + (t + 1) * C[:, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s[:, t], s0 + (t + 1) * c[:, 0], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(St, S[:, -1])
    np.testing.assert_array_equal(st, s[:, -1])


def test_scalar_transitions_closed_form():
    # W[t] = a_t I: S[t] = (prod_{r<=t} a_r) S0 + sum_{s<=t} (prod_{s<r<=t} a_r) U[s]
    rng = np.random.default_rng(2)
    BH, T, D = 1, 6, 3
    a = rng.uniform(0.3, 1.2, size=T)
    W = np.stack([a[t] * np.eye(D) for t in range(T)])[None]
    U = rng.standard_normal((BH, T, D, D))
    u = rng.standard_normal((BH, T, D))
    S0 = rng.standard_normal((BH, D, D))
    s0 = rng.standard_normal((BH, D))
    S, s, _, _ = F.scan(W, U, W, u, S0, s0)
    for t in range(T):
        ref = np.prod(a[: t + 1]) * S0[0] + sum(np.prod(a[r + 1: t + 1]) * U[0, r] for r in range(t + 1))
        refz = np.prod(a[: t + 1]) * s0[0] + sum(np.prod(a[r + 1: t + 1]) * u[0, r] for r in range(t + 1))
        np.testing.assert_allclose(S[0, t], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s[0, t], refz, rtol=1e-12, atol=1e-12)


def test_diagonal_z_transitions_are_independent_first_order_recurrences():
    rng = np.random.default_rng(3)
    BH, T, D = 1, 8, 5
    d = rng.uniform(-1.0, 1.0, size=(T, D))
    W_z = np.stack([np.diag(d[t]) for t in range(T)])[None]
    u = rng.standard_normal((BH, T, D))
    s0 = rng.standard_normal((BH, D))
    W_kv = np.broadcast_to(np.eye(D), (BH, T, D, D))
    _, s, _, _ = F.scan(W_kv, np.zeros((BH, T, D, D)), W_z, u, None, s0)
    for i in range(D):
        x = s0[0, i]
        for t in range(T):
            x = d[t, i] * x + u[0, t, i]  # scalar first-order recurrence of channel i
            assert abs(s[0, t, i] - x) <= 1e-12 * max(1.0, abs(x))


def test_zero_input_is_the_product_of_transitions():
    # U = 0: S[t] = S0 W[0] W[1] ... W[t] and s[t] = W[t] ... W[0] s0
    rng = np.random.default_rng(4)
    W_kv, _, W_z, _, S0, s0 = rand_case(rng, BH=1, T=5, D=4, contraction=1.0)
    S, s, _, _ = F.scan(W_kv, np.zeros_like(W_kv), W_z, np.zeros((1, 5, 4)), S0, s0)
    for t in range(5):
        ref = np.linalg.multi_dot([S0[0]] + [W_kv[0, r] for r in range(t + 1)])
        refz = np.linalg.multi_dot([W_z[0, r] for r in range(t, -1, -1)] + [s0[0][:, None]])[:, 0]
        np.testing.assert_allclose(S[0, t], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s[0, t], refz, rtol=1e-12, atol=1e-12)


def test_left_and_right_conventions_are_transposes():
    # s[t] = W_z[t] s[t-1] + u[t] is the row-vector scan r[t] = r[t-1] W_z[t]^T + u[t]^T: row 0 of a
    # KV scan whose state keeps only row 0
    rng = np.random.default_rng(5)
    BH, T, D = 2, 6, 4
    _, _, W_z, u, _, s0 = rand_case(rng, BH=BH, T=T, D=D)
    W_kv = np.swapaxes(W_z, -1, -2)
    U_kv = np.zeros((BH, T, D, D))
    U_kv[:, :, 0, :] = u
    S0 = np.zeros((BH, D, D))
    S0[:, 0, :] = s0
    S, s, _, _ = F.scan(W_kv, U_kv, W_z, u, S0, s0)
    np.testing.assert_allclose(S[:, :, 0, :], s, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(S[:, :, 1:, :], 0.0)


@pytest.mark.parametrize("active", [1, 4, 9])
def test_truncate_to_active_holds_the_state(active):
    rng = np.random.default_rng(6)
    W_kv, U_kv, W_z, u_z, S0, s0 = rand_case(rng)
    S, s, St, st = F.scan(W_kv, U_kv, W_z, u_z, S0, s0, active=active)
    Sf, sf, _, _ = F.scan(W_kv, U_kv, W_z, u_z, S0, s0)
    np.testing.assert_array_equal(S[:, :active], Sf[:, :active])
    np.testing.assert_array_equal(s[:, :active], sf[:, :active])
    for t in range(active, S.shape[1]):
        np.testing.assert_array_equal(S[:, t], S[:, active - 1])
        np.testing.assert_array_equal(s[:, t], s[:, active - 1])
    np.testing.assert_array_equal(St, Sf[:, active - 1])
    np.testing.assert_array_equal(st, sf[:, active - 1])
    with pytest.raises(ValueError):
        F.scan(W_kv, U_kv, W_z, u_z, active=0)


@pytest.mark.parametrize("seg,active", [(1, None), (3, None), (4, None), (9, None), (4, 6), (2, 3)])
def test_split_scan_equals_the_scan(seg, active):
    # the page's correction S[t] = S_local[t] + S_init W_cum[t] rests on linearity: it must give
    # the position-by-position scan for any segment length, ragged tail included
    rng = np.random.default_rng(7)
    W_kv, U_kv, W_z, u_z, S0, s0 = rand_case(rng)
    ref = F.scan(W_kv, U_kv, W_z, u_z, S0, s0, active=active)
    got = F.split_scan(W_kv, U_kv, W_z, u_z, seg, S0, s0, active=active)
    for x, y in zip(got, ref):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-10)


def test_composition_order_is_pinned():
    # a planted mistake in the composition (left instead of right multiply for KV) breaks the
    # split identity: the transitions do not commute
    rng = np.random.default_rng(8)
    W_kv, U_kv, W_z, u_z, S0, s0 = rand_case(rng, T=6)
    ref = F.scan(W_kv, U_kv, W_z, u_z, S0, s0)[0]
    h_kv, M_kv, h_z, M_z = [], [], [], []
    for a in range(0, 6, 3):
        S_loc, s_loc, _, _ = F.scan(W_kv[:, a:a + 3], U_kv[:, a:a + 3], W_z[:, a:a + 3], u_z[:, a:a + 3])
        ckv, cz = F.cumulative_products(W_kv[:, a:a + 3], W_z[:, a:a + 3])
        h_kv.append(S_loc[:, -1]), M_kv.append(ckv[:, -1]), h_z.append(s_loc[:, -1]), M_z.append(cz[:, -1])
    S_init, _, S_end, _ = F.exclusive_compose(np.stack(h_kv), np.stack(M_kv), np.stack(h_z), np.stack(M_z), S0, s0)
    np.testing.assert_allclose(S_end, ref[:, -1], rtol=1e-10, atol=1e-10)
    wrong = np.stack(M_kv)[1] @ (np.stack(M_kv)[0] @ S0 + h_kv[0]) + h_kv[1]  # planted: M S instead of S M
    assert np.abs(wrong - ref[:, -1]).max() > 1e-3
