"""Pins of the oracle's GAE, statistics and normalisation.

"Teaching Mario to speedrun", sec. 4 (discounted return), sec. 6 "Better
advantages" (delta_t and the GAE sum), sec. 7 (terminals = 1 where an episode
just ended).  Every check compares the oracle's backward recursion with
something other than itself: the sums as the page writes them, evaluated term
by term, their lambda = 1 and lambda = 0 special cases, and numpy's moments.
"""
import itertools

import numpy as np
import pytest

import oracle


def _rand(T, N, seed):
    rng = np.random.default_rng(seed)
    r = rng.normal(size=(T, N)).astype(np.float32)
    v = rng.normal(size=(T, N)).astype(np.float32)
    d = (rng.random((T, N)) < 0.2).astype(np.float32)
    b = rng.normal(size=N).astype(np.float32)
    return r, v, d, b


def _direct_gae(r, v, d, b, gamma, lam):
    """A_t = sum_l (gamma lambda)^l [prod_{j<l} (1 - d_{t+j})] delta_{t+l},
    delta_t = r_t + gamma (1 - d_t) V_{t+1} - V_t, V_T = boot: the page's sum,
    truncated where an episode ends, evaluated term by term."""
    T, N = r.shape
    r, v, d, b = (np.asarray(x, np.float64) for x in (r, v, d, b))
    vn = np.vstack([v[1:], b[None, :]])
    delta = r + gamma * (1 - d) * vn - v
    A = np.zeros((T, N))
    for n in range(N):
        for t in range(T):
            s, alive = 0.0, 1.0
            for l in range(T - t):
                s += (gamma * lam) ** l * alive * delta[t + l, n]
                alive *= 1 - d[t + l, n]
            A[t, n] = s
    return A


def _return_to_go(r, d, b, gamma):
    """G_t = r_t + gamma r_{t+1} + gamma^2 r_{t+2} + ... up to the end of the
    episode, bootstrapped with boot when the rollout ends first (sec. 4)."""
    T, N = r.shape
    G = np.zeros((T, N))
    for n in range(N):
        for t in range(T):
            s, k = 0.0, t
            while True:
                s += gamma ** (k - t) * float(r[k, n])
                if d[k, n] != 0:
                    break
                if k == T - 1:
                    s += gamma ** (T - t) * float(b[n])
                    break
                k += 1
            G[t, n] = s
    return G


@pytest.mark.parametrize("T,N", [(4, 2), (1, 3), (9, 5)])
def test_lambda_one_is_discounted_return(T, N):
    r, v, d, b = _rand(T, N, 1)
    adv, ret = oracle.gae(r, v, d, b, 0.97, 1.0)
    G = _return_to_go(r, d, b, 0.97)
    np.testing.assert_allclose(ret, G, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(adv + v, G, rtol=1e-12, atol=1e-12)


def test_lambda_zero_is_td_error():
    T, N = 7, 4
    r, v, d, b = _rand(T, N, 2)
    adv, _ = oracle.gae(r, v, d, b, 0.9, 0.0)
    vn = np.vstack([v[1:], b[None, :]]).astype(np.float64)
    td = r.astype(np.float64) + 0.9 * (1 - d.astype(np.float64)) * vn - v
    np.testing.assert_allclose(adv, td, rtol=1e-13, atol=1e-13)


def test_recursion_equals_sum_over_every_done_pattern():
    """Brute force: T = 4, N = 2, all 2^8 done patterns."""
    T, N = 4, 2
    rng = np.random.default_rng(3)
    r = rng.normal(size=(T, N)).astype(np.float32)
    v = rng.normal(size=(T, N)).astype(np.float32)
    b = rng.normal(size=N).astype(np.float32)
    for bits in itertools.product([0.0, 1.0], repeat=T * N):
        d = np.array(bits, np.float32).reshape(T, N)
        adv, ret = oracle.gae(r, v, d, b, 0.99, 0.95)
        ref = _direct_gae(r, v, d, b, 0.99, 0.95)
        np.testing.assert_allclose(adv, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(ret, ref + v, rtol=1e-12, atol=1e-12)


def test_all_done_and_zero_gamma():
    r, v, d, b = _rand(5, 3, 4)
    adv, ret = oracle.gae(r, v, np.ones_like(d), b, 0.99, 0.95)
    np.testing.assert_allclose(adv, r.astype(np.float64) - v, atol=1e-15)
    np.testing.assert_allclose(ret, r.astype(np.float64), atol=1e-6)
    adv0, _ = oracle.gae(r, v, d, b, 0.0, 0.95)
    np.testing.assert_allclose(adv0, r.astype(np.float64) - v, atol=1e-15)


def test_rollout_boundary_bootstraps_only_the_last_step():
    r = np.zeros((3, 1), np.float32)
    v = np.zeros((3, 1), np.float32)
    d = np.zeros((3, 1), np.float32)
    b = np.array([1.0], np.float32)
    adv, _ = oracle.gae(r, v, d, b, 0.5, 1.0)
    np.testing.assert_allclose(adv[:, 0], [0.125, 0.25, 0.5], atol=0)


def test_moments_match_numpy():
    x = np.random.default_rng(5).normal(3.0, 2.0, size=10007)
    m, s = oracle.moments(x)
    assert abs(m - np.mean(x)) <= 1e-13 * abs(np.mean(x))
    assert abs(s - np.std(x, ddof=1)) <= 1e-12 * np.std(x, ddof=1)
    out = oracle.normalize(x, m, s)
    np.testing.assert_allclose(out, (x - np.mean(x)) / (np.std(x, ddof=1) + 1e-8), rtol=1e-11,
                               atol=1e-13)


def test_constant_advantages_normalise_to_zero():
    x = np.full(100, 2.5)
    m, s = oracle.moments(x)
    assert m == 2.5 and s == 0.0
    assert np.all(oracle.normalize(x, m, s) == 0.0)
