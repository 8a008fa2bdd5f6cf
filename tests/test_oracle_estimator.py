"""Pins of the oracle's online acceptance estimator (jianc99/sglang PR #8,
DFLASH adaptive-verification commits: a logistic model p_k = sigmoid(slope *
x_k + bias_k) on x_k = logit(q_max) of the draft distribution, refit while
serving by damped Newton steps on IRLS statistics).

Closed-form features on hand-built rows, scipy's expit for the prediction, the
Newton step against finite-difference derivatives of the log-likelihood and a
dense solve, the observation set by hand, and the refit behaviour the page
reports: from a slope well above the optimum the slope reaches the generating
value, and on a feature without signal it falls to about zero.
"""
import numpy as np
import pytest
import scipy.special

import oracle


def _row(vals, V=8):
    r = np.full(V, -np.inf, np.float32)
    r[:len(vals)] = vals
    return r


def test_feature_closed_forms():
    rows = np.stack([
        _row([np.log(3.0), 0.0]),                   # q = (3/4, 1/4): x = ln 3
        _row([np.log(3.0), 0.0]),                   # at T = 2: q ~ (sqrt 3, 1): x = ln sqrt 3
        _row([np.log(3.0), 0.0]),                   # greedy request: T = 1
        _row([0.0] * 8),                            # uniform over 8: x = -ln 7
        _row([5.0, 1.0, 0.5]),                      # top-k 1: a single kept token -> +40
        _row([0.0, -100.0]),                        # q_max ~ 1 - e^-100 -> clamped to +40
        _row([2.0, 1.0, 1.0, 1.0]),                 # top-k 2 keeps {0, 1}: x = 1
    ])
    draft = rows[:, None, :]                        # n = 7 requests, K = 1
    T = np.array([1.0, 2.0, 0.0, 1.0, 1.0, 1.0, 1.0], np.float32)
    tk = np.array([0, 0, 0, 0, 1, 0, 2], np.int32)
    x = oracle.est_features(draft, T, tk)[:, 0]
    want = [np.log(3.0), 0.5 * np.log(3.0), np.log(3.0), -np.log(7.0), 40.0, 40.0, 1.0]
    assert np.allclose(x, want, rtol=1e-6, atol=1e-6), (x, want)
    # uniform over 2 tokens: q_max = 1/2, x = 0
    x0 = oracle.est_features(_row([0.0, 0.0])[None, None, :], np.ones(1, np.float32))
    assert abs(x0[0, 0]) < 1e-12


def test_prediction_is_the_logistic_function():
    est = oracle.Estimator(3)
    x = np.array([[0.0, 1.0, -2.0], [40.0, -40.0, 3.5]])
    p = est.predict(x)
    assert np.allclose(p, scipy.special.expit(0.5 * x - 0.2), rtol=1e-14)
    assert est.slope == 0.5 and np.all(est.bias == -0.2)


def _loglik(theta, obs, K):
    a, b = theta[0], theta[1:]
    s = 0.0
    for x, k, y in obs:
        z = a * x + b[k]
        s += y * z - np.logaddexp(0.0, z)
    return s


def _observations(x, acc, vl, K):
    obs = []
    for r in range(len(acc)):
        last = min(acc[r], vl[r] - 1)
        for k in range(last + 1):
            obs.append((x[r, k], k, 1.0 if k < acc[r] else 0.0))
    return obs


def test_refit_is_a_damped_ridge_newton_step():
    rng = np.random.default_rng(3)
    K, n = 4, 40
    x = rng.normal(0, 1.5, (n, K))
    vl = rng.integers(1, K + 1, n)
    acc = np.array([rng.integers(0, v + 1) for v in vl])
    est = oracle.Estimator(K)
    theta0 = est.state[:1 + K].copy()
    est.observe(x, acc, acc + 1, vl, refit_every=1)          # one call, one refit
    obs = _observations(x, acc, vl, K)
    # derivatives of the log-likelihood by central differences
    h = 1e-4
    m = K + 1
    g = np.zeros(m)
    H = np.zeros((m, m))
    for i in range(m):
        e = np.zeros(m); e[i] = h
        g[i] = (_loglik(theta0 + e, obs, K) - _loglik(theta0 - e, obs, K)) / (2 * h)
        for j in range(m):
            f = np.zeros(m); f[j] = h
            H[i, j] = (_loglik(theta0 + e + f, obs, K) - _loglik(theta0 + e - f, obs, K)
                       - _loglik(theta0 - e + f, obs, K) + _loglik(theta0 - e - f, obs, K)) / (4 * h * h)
    step = np.linalg.solve(-H + 1e-3 * np.eye(m), g)
    d = len(obs) / (len(obs) + 50.0)
    assert theta0[0] + d * step[0] >= 0                       # no halving in this case
    assert np.allclose(est.state[:1 + K], theta0 + d * step, rtol=1e-5, atol=1e-6)
    assert np.all(est.state[1 + K:4 * K + 4] == 0.0)          # statistics cleared


def test_observed_positions_stop_at_the_first_rejection():
    K = 3
    x = np.array([[1.0, 2.0, 3.0], [0.5, 0.5, 0.5], [1.0, 1.0, 1.0], [2.0, 2.0, 2.0]])
    acc = np.array([1, 3, 0, 0])
    emitted = np.array([2, 4, 1, 0])            # request 3 is an error: not observed
    vl = np.array([3, 3, 2, 3])
    est = oracle.Estimator(K)
    est.observe(x, acc, emitted, vl, refit_every=0)
    # r0: k = 0 accepted, k = 1 rejected; r1: all three accepted; r2: k = 0 rejected
    assert est.state[4 * K + 3] == 2 + 3 + 1
    g_b = est.state[K + 3:2 * K + 3]
    p = lambda xv, k: scipy.special.expit(0.5 * xv - 0.2)
    want0 = (1 - p(1.0, 0)) + (1 - p(0.5, 0)) + (0 - p(1.0, 0))
    want1 = (0 - p(2.0, 1)) + (1 - p(0.5, 1))
    want2 = (1 - p(0.5, 2))
    assert np.allclose(g_b, [want0, want1, want2], rtol=1e-12)


def _simulate(est, rng, slope, bias, n_calls, n=64, K=4, signal=True):
    for _ in range(n_calls):
        x = rng.normal(0.0, 2.0, (n, K))
        z = (slope * x if signal else 0.0) + bias
        alive = rng.uniform(size=(n, K)) < scipy.special.expit(z)
        acc = np.array([np.argmin(a) if not a.all() else K for a in alive])
        est.observe(x, acc, acc + 1, None, refit_every=100)


def test_refit_from_a_high_slope_reaches_the_generating_slope():
    rng = np.random.default_rng(4)
    est = oracle.Estimator(4)
    est.state[0] = 3.0
    bias = np.array([1.0, 0.5, 0.0, -0.5])
    _simulate(est, rng, 1.0, bias, 1000)                      # ten refits
    assert 0.85 < est.slope < 1.15, est.slope
    assert np.allclose(est.bias, bias, atol=0.25), est.bias


def test_refit_without_signal_drives_the_slope_to_zero():
    rng = np.random.default_rng(5)
    est = oracle.Estimator(4)
    _simulate(est, rng, 0.0, np.array([0.5, 0.2, 0.0, -0.3]), 1000, signal=False)
    assert 0.0 <= est.slope < 0.1, est.slope


def test_estimator_pins_catch_planted_mistakes(tmp_path):
    with oracle.planted(10, str(tmp_path)):           # whole window observed
        with pytest.raises(AssertionError):
            test_observed_positions_stop_at_the_first_rejection()
    with oracle.planted(11, str(tmp_path)):           # crossing step dropped, never halved
        with pytest.raises(AssertionError):
            test_refit_from_a_high_slope_reaches_the_generating_slope()
