"""Pins for the CPU oracle: it is checked against things other than itself.

* exact rational values of the unrolled-product form (live and stored in
  tests/golden/exact_tiny.json);
* closed forms the recurrence must satisfy (with g = 0, beta = 1
  and unit k, the updated state satisfies S_t^T k_t = v_t exactly; beta = 0
  leaves pure decay; a = 0 leaves one rank-one write);
* central finite differences for the reverse mode, and the adjoint identity
  dh0 = M^T dht when dO = 0;
* segment-summary invariants (composition over any split reproduces the
  unsplit state; linearity S(h0) = S(0) + M h0; identity padding);
* packed documents equal separate runs;
* planted mistakes (wrong base, swapped decay order) are caught.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import brute, recurrence as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "exact_tiny.json")


def _rand_case(rng, B, T, H, K, V, per_key=False, gscale=0.3, h0=True):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H, K) if per_key else (B, T, H)))) * gscale
    s = rng.standard_normal((B, H, K, V)) * 0.3 if h0 else None
    return q, k, v, g, beta, s


def _dec(x):
    if isinstance(x, list):
        return [_dec(y) for y in x]
    return Fraction(x)


def _as_float(x):
    return np.array(_dec(x), dtype=object).astype(np.float64)


@pytest.mark.parametrize("name", ["scalar_gate_exp2", "per_key_gate_exp2"])
def test_oracle_matches_stored_exact_values(name):
    c = json.load(open(GOLDEN))["cases"][name]
    q, k, v, h0 = (_as_float(c[x]) for x in ("q", "k", "v", "h0"))
    g = _as_float(c["g"])
    beta = _as_float(c["beta"])
    scale = float(Fraction(c["scale"]))
    o, ht = R.forward(q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
                      beta[None, :, None], h0[None, None], scale=scale, per_key=c["per_key"],
                      use_exp2=True)
    np.testing.assert_allclose(o[0, :, 0], _as_float(c["o"]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ht[0, 0], _as_float(c["ht"]), rtol=1e-13, atol=1e-13)
    S, M = R.segment_summary(k[None, :, None], v[None, :, None], g[None, :, None],
                             beta[None, :, None], seg_len=len(c["k"]), per_key=c["per_key"],
                             use_exp2=True)
    np.testing.assert_allclose(M[0, 0, 0], _as_float(c["M"]), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("per_key", [False, True])
def test_oracle_matches_live_brute_force(per_key):
    rng = np.random.default_rng(7)
    T, K, V = 6, 3, 2
    # dyadic rationals, integer base-2 gates: exact in Fraction and in fp64
    qi = rng.integers(-4, 5, (T, K)) / 4.0
    ki = rng.integers(-4, 5, (T, K)) / 4.0
    vi = rng.integers(-8, 9, (T, V)) / 4.0
    bi = rng.integers(1, 5, T) / 4.0
    gi = rng.integers(-2, 1, (T, K) if per_key else T).astype(np.float64)
    hi = rng.integers(-4, 5, (K, V)) / 4.0
    F = lambda a: [[Fraction(x) for x in r] for r in a] if np.ndim(a) == 2 else [Fraction(x) for x in a]  # noqa: E731
    o_ex, S_ex = brute.states(F(qi), F(ki), F(vi), [list(map(int, r)) for r in gi] if per_key
                              else [int(x) for x in gi], F(bi), F(hi), Fraction(1, 2), per_key)
    o, ht = R.forward(qi[None, :, None], ki[None, :, None], vi[None, :, None], gi[None, :, None],
                      bi[None, :, None], hi[None, None], scale=0.5, per_key=per_key, use_exp2=True)
    np.testing.assert_allclose(o[0, :, 0], np.array(o_ex, dtype=np.float64), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ht[0, 0], np.array(S_ex, dtype=np.float64), rtol=1e-12, atol=1e-12)


def test_planted_mistakes_are_caught():
    """A wrong gate base or a swapped decay order must break the exact pin."""
    c = json.load(open(GOLDEN))["cases"]["per_key_gate_exp2"]
    q, k, v, h0, g, beta = (_as_float(c[x]) for x in ("q", "k", "v", "h0", "g", "beta"))
    args = (q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
            beta[None, :, None], h0[None, None])
    o_wrong_base, _ = R.forward(*args, scale=0.5, per_key=True, use_exp2=False)
    assert np.abs(o_wrong_base[0, :, 0] - _as_float(c["o"])).max() > 1e-3
    # decay applied after the rank-one correction: Diag(a)(I - b k k^T)
    gd = _dec(c["g"])
    A_swapped = []
    for t in range(len(gd)):
        a = [Fraction(2) ** int(x) for x in gd[t]]
        base = brute.transition(_dec(c["k"])[t], _dec(c["beta"])[t], [Fraction(1)] * 3)
        A_swapped.append([[a[i] * base[i][j] for j in range(3)] for i in range(3)])
    M_swapped = brute._eye(3)
    for A in A_swapped:
        M_swapped = brute._matmul(A, M_swapped)
    assert np.abs(np.array(M_swapped, dtype=np.float64) - _as_float(c["M"])).max() > 1e-3


def test_closed_form_unit_key_full_write():
    """g = 0, beta = 1, |k| = 1  =>  S_t^T k_t = v_t exactly (the delta rule's full write)."""
    rng = np.random.default_rng(3)
    B, T, H, K, V = 1, 40, 2, 16, 8
    q, k, v, g, beta, h0 = _rand_case(rng, B, T, H, K, V)
    o, _ = R.forward(k, k, v, np.zeros_like(g), np.ones_like(beta), h0, scale=1.0)
    np.testing.assert_allclose(o, v, atol=1e-12)


def test_closed_form_zero_beta_is_pure_decay():
    rng = np.random.default_rng(4)
    q, k, v, g, beta, h0 = _rand_case(rng, 2, 30, 2, 8, 5)
    for use_exp2 in (False, True):
        o, ht = R.forward(q, k, v, g, np.zeros_like(beta), h0, scale=0.7, use_exp2=use_exp2)
        base = 2.0 if use_exp2 else math.e
        G = np.cumsum(g, axis=1)                                    # [B,T,H]
        St = base ** G[..., None, None] * h0[:, None]                # [B,T,H,K,V]
        np.testing.assert_allclose(o, 0.7 * np.einsum("bthkv,bthk->bthv", St, q), atol=1e-12)
        np.testing.assert_allclose(ht, St[:, -1], atol=1e-12)


def test_closed_form_full_forget_is_one_write():
    """a = 0 (base-2 gate of -2000 underflows to exactly 0): o_t = scale b_t (k_t.q_t) v_t."""
    rng = np.random.default_rng(5)
    q, k, v, g, beta, h0 = _rand_case(rng, 1, 20, 3, 8, 6, per_key=True)
    o, ht = R.forward(q, k, v, np.full_like(g, -2000.0), beta, h0, scale=0.9, per_key=True,
                      use_exp2=True)
    want = 0.9 * beta[..., None] * np.sum(k * q, axis=-1)[..., None] * v
    np.testing.assert_allclose(o, want, atol=1e-12)
    np.testing.assert_allclose(ht[0], beta[0, -1, :, None, None] * k[0, -1, :, :, None]
                               * v[0, -1, :, None, :], atol=1e-12)


@pytest.mark.parametrize("per_key,use_exp2", [(False, False), (True, True), (False, True)])
def test_reverse_mode_matches_central_differences(per_key, use_exp2):
    rng = np.random.default_rng(11)
    q, k, v, g, beta, h0 = _rand_case(rng, 2, 13, 2, 5, 4, per_key=per_key)
    dO = rng.standard_normal(v.shape)
    o, ht = R.forward(q, k, v, g, beta, h0, per_key=per_key, use_exp2=use_exp2)
    dht = rng.standard_normal(ht.shape)
    grads = R.backward(q, k, v, g, beta, h0, dO, dht, per_key=per_key, use_exp2=use_exp2)

    def loss(*a):
        o, ht = R.forward(*a, per_key=per_key, use_exp2=use_exp2)
        return float((o * dO).sum() + (ht * dht).sum())

    args = [q, k, v, g, beta, h0]
    for i, name in enumerate(["dq", "dk", "dv", "dg", "dbeta", "dh0"]):
        d = rng.standard_normal(args[i].shape)
        eps = 1e-6
        hi = [x.copy() for x in args]
        lo = [x.copy() for x in args]
        hi[i] += eps * d
        lo[i] -= eps * d
        fd = (loss(*hi) - loss(*lo)) / (2 * eps)
        an = float((grads[name] * d).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_adjoint_identity_and_linearity():
    """dO = 0 => dh0 = M^T dht; and S(h0) = S(0) + M h0 (SANA step-5 linearity)."""
    rng = np.random.default_rng(12)
    for per_key in (False, True):
        q, k, v, g, beta, h0 = _rand_case(rng, 1, 70, 2, 6, 5, per_key=per_key)
        _, M = R.segment_summary(k, v, g, beta, seg_len=70, per_key=per_key)
        M = M[:, :, 0]
        dht = rng.standard_normal(h0.shape)
        gr = R.backward(q, k, v, g, beta, h0, None, dht, per_key=per_key)
        np.testing.assert_allclose(gr["dh0"], np.einsum("bhij,bhiv->bhjv", M, dht), atol=1e-12)
        _, ht = R.forward(q, k, v, g, beta, h0, per_key=per_key)
        _, ht0 = R.forward(q, k, v, g, beta, None, per_key=per_key)
        np.testing.assert_allclose(ht, ht0 + np.einsum("bhij,bhjv->bhiv", M, h0), atol=1e-12)


@pytest.mark.parametrize("seg_len", [64, 50, 17])
def test_segment_composition_reproduces_unsplit_state(seg_len):
    rng = np.random.default_rng(13)
    q, k, v, g, beta, h0 = _rand_case(rng, 2, 150, 2, 6, 5, per_key=True)
    S, M = R.segment_summary(k, v, g, beta, seg_len, per_key=True, use_exp2=True)
    S_init, ht = R.segment_merge(S, M, h0)
    _, ht_ref = R.forward(q, k, v, g, beta, h0, per_key=True, use_exp2=True)
    np.testing.assert_allclose(ht, ht_ref, atol=1e-11)
    for s in range(S.shape[2]):
        t = s * seg_len
        if t == 0:
            want = h0
        else:
            _, want = R.forward(q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t], h0,
                                per_key=True, use_exp2=True)
        np.testing.assert_allclose(S_init[:, :, s], want, atol=1e-11)


def test_identity_padding_leaves_state_unchanged():
    """Tokens with a = 1 and beta = 0 are identity maps (truncate_to_active in SANA)."""
    rng = np.random.default_rng(14)
    q, k, v, g, beta, h0 = _rand_case(rng, 1, 40, 2, 6, 5)
    _, ht = R.forward(q, k, v, g, beta, h0)
    pad = lambda x, val: np.concatenate([x, np.full((1, 25) + x.shape[2:], val)], axis=1)  # noqa: E731
    qp, kp, vp = (np.concatenate([x, rng.standard_normal((1, 25) + x.shape[2:])], axis=1)
                  for x in (q, k, v))
    _, ht_pad = R.forward(qp, kp, vp, pad(g, 0.0), pad(beta, 0.0), h0)
    np.testing.assert_allclose(ht_pad, ht, atol=1e-12)


def test_packed_documents_equal_separate_runs():
    rng = np.random.default_rng(15)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 200, 2, 6, 5)
    cu = np.array([0, 37, 100, 164, 200])
    h0 = rng.standard_normal((4, 2, 6, 5))
    o, ht = R.forward(q[0], k[0], v[0], g[0], beta[0], h0, cu=cu)
    dO = rng.standard_normal(o.shape)
    gr = R.backward(q[0], k[0], v[0], g[0], beta[0], h0, dO, None, cu=cu)
    for n in range(4):
        s = slice(cu[n], cu[n + 1])
        on, hn = R.forward(q[:, s], k[:, s], v[:, s], g[:, s], beta[:, s], h0[n:n + 1])
        np.testing.assert_allclose(o[s], on[0], atol=1e-12)
        np.testing.assert_allclose(ht[n], hn[0], atol=1e-12)
        gn = R.backward(q[:, s], k[:, s], v[:, s], g[:, s], beta[:, s], h0[n:n + 1],
                        dO[None, s], None)
        np.testing.assert_allclose(gr["dk"][s], gn["dk"][0], atol=1e-12)
        np.testing.assert_allclose(gr["dh0"][n], gn["dh0"][0], atol=1e-12)


@pytest.mark.parametrize("per_key", [False, True])
def test_input_maps_reverse_mode_matches_central_differences(per_key):
    """The in-kernel q/k norm and beta sigmoid: the oracle's chain rule through both maps
    against central differences of its own forward on raw inputs."""
    rng = np.random.default_rng(13)
    q, k, v, g, beta, h0 = _rand_case(rng, 1, 11, 2, 6, 3, per_key=per_key)
    q, k = 3.0 * rng.standard_normal(q.shape), 0.2 * rng.standard_normal(k.shape)  # raw, unnormalised
    braw = rng.standard_normal(beta.shape)
    dO = rng.standard_normal(v.shape)
    kw = dict(per_key=per_key, use_exp2=per_key, use_qk_l2norm=True, beta_sigmoid=True)
    o, ht = R.forward(q, k, v, g, braw, h0, **kw)
    dht = rng.standard_normal(ht.shape)
    grads = R.backward(q, k, v, g, braw, h0, dO, dht, **kw)

    def loss(*a):
        o, ht = R.forward(*a, **kw)
        return float((o * dO).sum() + (ht * dht).sum())

    args = [q, k, v, g, braw, h0]
    for i, name in enumerate(["dq", "dk", "dv", "dg", "dbeta", "dh0"]):
        d = rng.standard_normal(args[i].shape)
        eps = 1e-6
        hi = [x.copy() for x in args]
        lo = [x.copy() for x in args]
        hi[i] += eps * d
        lo[i] -= eps * d
        fd = (loss(*hi) - loss(*lo)) / (2 * eps)
        an = float((grads[name] * d).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_input_maps_fixed_points():
    """sigmoid(0) = 1/2 exactly; the norm is invariant to scaling its input when
    sum x^2 >> eps; a row with sum x^2 = eps comes out with squared norm exactly 1/2."""
    rng = np.random.default_rng(14)
    q, k, v, g, beta, h0 = _rand_case(rng, 1, 9, 1, 4, 3)
    o_half, ht_half = R.forward(q, k, v, g, np.full_like(beta, 0.5), h0)
    o_sig, ht_sig = R.forward(q, k, v, g, np.zeros_like(beta), h0, beta_sigmoid=True)
    np.testing.assert_array_equal(o_sig, o_half)
    np.testing.assert_array_equal(ht_sig, ht_half)
    qr, kr = 5.0 * rng.standard_normal(q.shape), 7.0 * rng.standard_normal(k.shape)
    o1, _ = R.forward(qr, kr, v, g, beta, h0, use_qk_l2norm=True)
    o2, _ = R.forward(1e3 * qr, 1e3 * kr, v, g, beta, h0, use_qk_l2norm=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-6, atol=1e-9)
    x = np.full((1, 1, 1, 4), math.sqrt(R.L2_EPS / 4))  # sum x^2 = eps
    xn, _ = R.l2norm(x)
    assert abs(float((xn * xn).sum()) - 0.5) < 1e-15


@pytest.mark.parametrize("per_key,seg_len", [(False, 5), (True, 7)])
def test_split_backward_reproduces_unsplit_backward(per_key, seg_len):
    """Backward segment summaries + the adjoint merge, then every segment's reverse pass
    seeded with its exit gradient (and its forward with the merged entry state), give the
    unsplit gradients; the merge's dh0 is the unsplit dh0."""
    rng = np.random.default_rng(15)
    q, k, v, g, beta, h0 = _rand_case(rng, 2, 19, 2, 5, 4, per_key=per_key)
    dO = rng.standard_normal(v.shape)
    kw = dict(per_key=per_key, use_exp2=per_key)
    o, ht = R.forward(q, k, v, g, beta, h0, **kw)
    dht = rng.standard_normal(ht.shape)
    want = R.backward(q, k, v, g, beta, h0, dO, dht, **kw)
    S, M = R.segment_summary(k, v, g, beta, seg_len, **kw)
    S_init, _ = R.segment_merge(S, M, h0)
    dS_ext = R.segment_summary_bwd(q, k, v, g, beta, dO, seg_len, **kw)
    dS_exit, dh0 = R.segment_merge_bwd(dS_ext, M, dht)
    np.testing.assert_allclose(dh0, want["dh0"], rtol=1e-10, atol=1e-12)
    nseg = S.shape[2]
    for s in range(nseg):
        sl = lambda x: x[:, s * seg_len:(s + 1) * seg_len]  # noqa: E731
        got = R.backward(sl(q), sl(k), sl(v), sl(g), sl(beta), S_init[:, :, s], sl(dO), dS_exit[:, :, s], **kw)
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(got[name], sl(want[name]), rtol=1e-9, atol=1e-11)
        # the segment's entry gradient is the merge's: M_s^T dS_exit + dS_ext
        if s > 0:
            np.testing.assert_allclose(got["dh0"], dS_exit[:, :, s - 1], rtol=1e-9, atol=1e-11)


def test_backward_summary_with_no_output_gradient_is_pure_transport():
    """dO = 0: every backward summary vanishes and dh0 = M_0^T ... M_{n-1}^T dht."""
    rng = np.random.default_rng(16)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 12, 1, 4, 3, per_key=True)
    dO = np.zeros(v.shape)
    dS_ext = R.segment_summary_bwd(q, k, v, g, beta, dO, 4, per_key=True, use_exp2=True)
    assert np.abs(dS_ext).max() == 0.0
    _, M = R.segment_summary(k, v, g, beta, 4, per_key=True, use_exp2=True)
    dht = rng.standard_normal((1, 1, 4, 3))
    _, dh0 = R.segment_merge_bwd(dS_ext, M, dht)
    want = dht[0, 0]
    for s in range(M.shape[2] - 1, -1, -1):
        want = M[0, 0, s].T @ want
    np.testing.assert_allclose(dh0[0, 0], want, rtol=1e-12, atol=1e-14)
