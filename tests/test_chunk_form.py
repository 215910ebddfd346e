"""Pins for the chunk-form oracle: it must equal the token recurrence (a
different algorithm) and satisfy the UT-transform invariants."""
import numpy as np
import pytest

from oracle import chunk_form as CF, recurrence as R
from tests.test_oracle_pins import _rand_case


@pytest.mark.parametrize("per_key,use_exp2,T", [(False, False, 150), (True, True, 129),
                                                (False, True, 64), (True, False, 63)])
def test_chunk_forward_equals_token_recurrence(per_key, use_exp2, T):
    rng = np.random.default_rng(21)
    q, k, v, g, beta, h0 = _rand_case(rng, 2, T, 2, 8, 6, per_key=per_key)
    o, ht = R.forward(q, k, v, g, beta, h0, per_key=per_key, use_exp2=use_exp2, scale=0.3)
    c = CF.forward(q, k, v, g, beta, h0, per_key=per_key, use_exp2=use_exp2, scale=0.3)
    np.testing.assert_allclose(c["o"], o, atol=1e-12)
    np.testing.assert_allclose(c["ht"], ht, atol=1e-12)
    # entry state of every chunk equals the token state at the chunk start
    for ci in range(-(-T // 64)):
        t = ci * 64
        if t == 0:
            want = h0
        else:
            _, want = R.forward(q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t], h0,
                                per_key=per_key, use_exp2=use_exp2)
        np.testing.assert_allclose(c["h_chunks"][:, :, ci], want, atol=1e-12)


def test_ut_transform_invariants():
    rng = np.random.default_rng(22)
    q, k, v, g, beta, h0 = _rand_case(rng, 1, 100, 1, 8, 4)
    c = CF.forward(q, k, v, g, beta, h0)
    for c0, c1 in ((0, 64), (64, 100)):
        n = c1 - c0
        A = c["A"][0, c0:c1, 0, :n]
        R_ = CF.chunk_intermediates(q[0, c0:c1, 0], k[0, c0:c1, 0], v[0, c0:c1, 0],
                                    g[0, c0:c1, 0], beta[0, c0:c1, 0], np.zeros((8, 4)), 1.0,
                                    False, False)
        np.testing.assert_allclose((np.eye(n) + R_["L"]) @ A, np.eye(n), atol=1e-12)
        assert np.allclose(np.triu(A, 1), 0) and np.allclose(np.diag(A), 1)
        assert np.all(c["A"][0, c0:c1, 0, n:] == 0)
        # cumulative gate restarts at the chunk start
        np.testing.assert_allclose(c["g_cumsum"][0, c0:c1, 0], np.cumsum(g[0, c0:c1, 0]))


def test_chunk_forward_packed_and_chunk_order():
    rng = np.random.default_rng(23)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 300, 2, 6, 5)
    cu = np.array([0, 37, 101, 229, 300])
    h0 = rng.standard_normal((4, 2, 6, 5))
    o, ht = R.forward(q[0], k[0], v[0], g[0], beta[0], h0, cu=cu)
    c = CF.forward(q[0], k[0], v[0], g[0], beta[0], h0, cu=cu)
    np.testing.assert_allclose(c["o"], o, atol=1e-12)
    np.testing.assert_allclose(c["ht"], ht, atol=1e-12)
    nchunks = sum(-(-(cu[i + 1] - cu[i]) // 64) for i in range(4))
    assert c["h_chunks"].shape == (nchunks, 2, 6, 5)
    # chunk 0 of document 2 is its initial state
    idx = -(-37 // 64) + -(-64 // 64)
    np.testing.assert_allclose(c["h_chunks"][idx], h0[2])


@pytest.mark.parametrize("per_key,use_exp2", [(False, False), (True, True)])
def test_chunk_backward_equals_token_reverse_mode(per_key, use_exp2):
    rng = np.random.default_rng(24)
    q, k, v, g, beta, h0 = _rand_case(rng, 1, 140, 2, 6, 5, per_key=per_key)
    dO = rng.standard_normal(v.shape)
    dht = rng.standard_normal(h0.shape)
    a = R.backward(q, k, v, g, beta, h0, dO, dht, per_key=per_key, use_exp2=use_exp2)
    b = CF.backward(q, k, v, g, beta, h0, dO, dht, per_key=per_key, use_exp2=use_exp2)
    for name in a:
        np.testing.assert_allclose(b[name], a[name], atol=1e-11, err_msg=name)


def test_chunk_transfer_composes_to_segment_transfer():
    rng = np.random.default_rng(25)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 128, 1, 6, 5, per_key=True)
    _, M = R.segment_summary(k, v, g, beta, 128, per_key=True, use_exp2=True)
    M0 = CF.transfer_chunks(k[0, :64, 0], g[0, :64, 0], beta[0, :64, 0], per_key=True, use_exp2=True)
    M1 = CF.transfer_chunks(k[0, 64:, 0], g[0, 64:, 0], beta[0, 64:, 0], per_key=True, use_exp2=True)
    np.testing.assert_allclose(M1 @ M0, M[0, 0, 0], atol=1e-12)
