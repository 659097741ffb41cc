"""Pins of the confidence-head oracle: closed forms of the sigmoid and of temperature
scaling, one-hot inputs that select single weights, and the embedding of the right previous
token recovered from the output."""
import numpy as np

from oracle import confidence


def _rand(seed, B=3, N=4, H=6, V=9, r=5):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B * N, H)), rng.standard_normal((V, r)), rng.integers(0, V, B),
            rng.integers(0, V, (B, N)), rng.standard_normal(H), rng.standard_normal(r),
            float(rng.standard_normal()), rng.uniform(0.5, 2.0, N))


def test_zero_weights_give_sigmoid_of_scaled_bias():
    h, w1, a, x, wh, we, beta, tau = _rand(1)
    c = confidence(h, w1, a, x, 0 * wh, 0 * we, 0.7, tau)
    np.testing.assert_allclose(c, np.broadcast_to(1 / (1 + np.exp(-0.7 / tau)), c.shape), rtol=0, atol=1e-15)
    c0 = confidence(h, w1, a, x, 0 * wh, 0 * we, 0.0, tau)
    assert np.all(c0 == 0.5)


def test_one_hot_hidden_selects_one_weight_and_sign_symmetry():
    h, w1, a, x, wh, we, beta, tau = _rand(2)
    h = np.zeros_like(h)
    h[:, 3] = 1.0
    c = confidence(h, w1, 0 * a, 0 * x, wh, 0 * we, 0.0, np.ones(4))
    np.testing.assert_allclose(c, 1 / (1 + np.exp(-wh[3])), rtol=0, atol=1e-15)
    c_neg = confidence(h, w1, 0 * a, 0 * x, -wh, 0 * we, 0.0, np.ones(4))
    np.testing.assert_allclose(c + c_neg, 1.0, rtol=0, atol=1e-15)            # sigma(-z) = 1 - sigma(z)


def test_embedding_is_of_the_previous_token_anchor_first():
    h, w1, a, x, wh, we, beta, tau = _rand(3)
    w1 = np.zeros_like(w1)
    w1[:, 0] = np.arange(w1.shape[0])                # E[prev] . e_0 = prev
    we = np.zeros_like(we)
    we[0] = 1.0
    c = confidence(h, w1, a, x, 0 * wh, we, 0.0, np.ones(4))
    prev = np.log(c / (1 - c))                       # the logit recovers prev
    np.testing.assert_allclose(prev[:, 0], a, atol=1e-9)
    np.testing.assert_allclose(prev[:, 1:], x[:, :-1], atol=1e-9)


def test_temperature_scales_the_logit_and_large_temperature_flattens():
    h, w1, a, x, wh, we, beta, tau = _rand(4)
    c1 = confidence(h, w1, a, x, wh, we, beta, np.ones(4))
    c2 = confidence(h, w1, a, x, wh, we, beta, np.full(4, 2.0))
    z1, z2 = np.log(c1 / (1 - c1)), np.log(c2 / (1 - c2))
    np.testing.assert_allclose(z2, z1 / 2, rtol=1e-9, atol=1e-12)
    c_big = confidence(h, w1, a, x, wh, we, beta, np.full(4, 1e9))
    np.testing.assert_allclose(c_big, 0.5, atol=1e-8)
