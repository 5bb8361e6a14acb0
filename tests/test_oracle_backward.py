"""Pins for the backward oracle: the gradients must be the derivatives of the
(pinned) forward oracle, checked by central finite differences in fp64, plus
closed forms that a wrong sign, a transposed operand or a missing delta term
would break."""
import numpy as np
import pytest

import oracle


def loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attention(q, k, v, scale, causal, threads=1)
    return float((o * dout.astype(np.float64)).sum())


def finite_difference(q, k, v, dout, scale, causal, which, idx, eps):
    args = [q.astype(np.float64), k.astype(np.float64), v.astype(np.float64)]
    hi = [a.copy() for a in args]
    lo = [a.copy() for a in args]
    hi[which][idx] += eps
    lo[which][idx] -= eps
    # the forward oracle reads float32: perturb by an exactly representable eps
    f = lambda a: loss(*(x.astype(np.float32) for x in a), dout, scale, causal)
    return (f(hi) - f(lo)) / (2 * eps)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_gradients_match_finite_differences(seed, causal):
    rng = np.random.default_rng(400 + seed)
    B, H, N, d = 1, 2, 7, 5
    # inputs on a 2^-6 grid so that x +- 2^-10 stays exact in float32
    q, k, v, dout = (np.round(rng.standard_normal((B, H, N, d)) * 64) / 64 for _ in range(4))
    q, k, v, dout = (x.astype(np.float32) for x in (q, k, v, dout))
    scale = 0.5
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, scale, causal)
    eps = 2.0 ** -10
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for idx in [(0, 0, 0, 0), (0, 1, 3, 2), (0, 1, 6, 4), (0, 0, 5, 1)]:
            fd = finite_difference(q, k, v, dout, scale, causal, which, idx, eps)
            assert abs(fd - grad[idx]) < 2e-5 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


def test_uniform_weights_give_mean_gradient_for_values():
    """Q = 0: every weight of a non-causal row is 1/N, so dV_j is the mean of
    the dO rows for every key j.  With all V rows equal, dP_ij = dO_i . v does
    not depend on j, so dS = 0 and dQ = dK = 0 exactly."""
    rng = np.random.default_rng(410)
    B, H, N, d = 1, 1, 9, 4
    q = np.zeros((B, H, N, d), np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    v = np.tile(rng.standard_normal((1, 1, 1, d)).astype(np.float32), (1, 1, N, 1))
    dout = rng.standard_normal((B, H, N, d)).astype(np.float32)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, 0.3, False)
    mean = dout[0, 0].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(dv[0, 0], np.tile(mean, (N, 1)), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)


def test_key_gradients_sum_to_zero_per_query_shift():
    """Adding one vector c to every key shifts each row's scores by a constant,
    which softmax ignores: L does not change, so sum_j dK_j . c = 0 for every
    c, i.e. sum_j dK_j = 0 (per head, without the causal mask)."""
    rng = np.random.default_rng(420)
    q, k, v, dout = (rng.standard_normal((2, 2, 11, 6)).astype(np.float32) for _ in range(4))
    _, dk, _ = oracle.attention_backward(q, k, v, dout, 0.4, False)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


def test_value_gradient_is_linear_in_upstream_gradient():
    rng = np.random.default_rng(430)
    q, k, v = (rng.standard_normal((1, 1, 8, 3)).astype(np.float32) for _ in range(3))
    g1 = (rng.integers(-8, 9, (1, 1, 8, 3)) / 4).astype(np.float32)
    g2 = (rng.integers(-8, 9, (1, 1, 8, 3)) / 4).astype(np.float32)
    a = oracle.attention_backward(q, k, v, g1, 0.5, True)
    b = oracle.attention_backward(q, k, v, g2, 0.5, True)
    c = oracle.attention_backward(q, k, v, g1 + 2 * g2, 0.5, True)
    for x, y, z in zip(a, b, c):
        np.testing.assert_allclose(z, x + 2 * y, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_gradients_equal_the_full_gradients(causal):
    """The subset form evaluates the same definition: on shapes the full
    oracle handles it must give the same dQ rows and dK, dV rows (a wrong
    mask direction, a row statistic of the wrong head or a missing delta
    term would break this)."""
    rng = np.random.default_rng(420 + causal)
    B, H, N, d = 2, 3, 37, 6
    q, k, v, dout = (rng.standard_normal((B, H, N, d)).astype(np.float32) for _ in range(4))
    scale = 0.4
    dq, dk, dv = (x.reshape(-1, d) for x in oracle.attention_backward(q, k, v, dout, scale, causal))
    rows = np.array([0, 5, N - 1, N, 2 * N + 17, B * H * N - 1])
    keys = np.array([0, 1, N - 1, 3 * N, 3 * N + 20, B * H * N - 2, B * H * N - 1])
    sq, sk, sv = oracle.attention_backward_sampled(q, k, v, dout, scale, causal, rows, keys)
    np.testing.assert_allclose(sq, dq[rows], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sk, dk[keys], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sv, dv[keys], rtol=1e-10, atol=1e-12)
