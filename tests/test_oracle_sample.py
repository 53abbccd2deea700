"""Pins of the oracle's rollout-side policy step (action sampling).

"Teaching Mario to speedrun", sec. 6 "The whole algorithm" step 1 and sec. 7
(logits, value = policy(obs); actions = sample(logits); old_prob kept);
"PlayTrain", Appendix F.2 (mulberry32).  The sampling rule is the reading
stated in ppo_oracle.c (inverse CDF per head, Box-Muller per Gaussian
dimension, 24-bit uniforms from counter-indexed mulberry32 draws).  Pinned
against: the already pinned mulberry32 stream, hand-computed category
boundaries, numpy's searchsorted on scipy's softmax, closed Box-Muller
points, the empirical distribution of many draws (chi-square / moments), and
the pinned forward pass and log-probability.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle


def test_counter_jump_equals_stream():
    for seed in (0, 1, 0xDEADBEEF):
        s = oracle.mulberry32_stream(seed, 70)
        for k in (0, 1, 2, 37, 69):
            assert oracle.mulberry32_at(seed, k) == s[k]
    # far counters wrap modulo 2^32 like the state does
    st = oracle.mulberry32_stream(7, 1)[0]
    assert oracle.mulberry32_at(7, 2 ** 32) == st


def test_uniform24():
    assert oracle.uniform24(0) == 0.0
    assert oracle.uniform24(255) == 0.0
    assert oracle.uniform24(256) == 2.0 ** -24
    assert oracle.uniform24(0xFFFFFFFF) == 1.0 - 2.0 ** -24


def test_categorical_boundaries_by_hand():
    z = np.log([0.2, 0.3, 0.5])
    cases = [(0.0, 0), (0.19999, 0), (0.20001, 1), (0.49999, 1), (0.50001, 2), (0.99999, 2)]
    for u, k in cases:
        assert oracle.sample_categorical(z, u) == k, (u, k)
    # a category of (numerically) zero probability is never chosen
    z = np.array([0.0, -1e4, 0.0])
    assert oracle.sample_categorical(z, 0.4999) == 0
    assert oracle.sample_categorical(z, 0.5001) == 2
    # one category: always it
    assert oracle.sample_categorical(np.array([3.0]), 0.999) == 0


def test_categorical_equals_searchsorted():
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(1, 10))
        z = rng.normal(0, 2, n)
        p = scipy.special.softmax(z)
        for u in rng.random(20):
            # away from boundaries, where rounding order could matter
            cdf = np.cumsum(p)
            if np.min(np.abs(cdf - u)) < 1e-12:
                continue
            ref = min(int(np.searchsorted(cdf, u, side="right")), n - 1)
            assert oracle.sample_categorical(z, u) == ref


def test_box_muller_points_and_distribution():
    assert oracle.box_muller(0.0, 0.3) == 0.0
    assert abs(oracle.box_muller(1 - math.exp(-0.5), 0.0) - 1.0) < 1e-15
    assert abs(oracle.box_muller(1 - math.exp(-2.0), 0.5) + 2.0) < 1e-14
    raw = oracle.mulberry32_stream(3, 40000)
    u = np.array([oracle.uniform24(x) for x in raw])
    n = np.array([oracle.box_muller(a, b) for a, b in zip(u[0::2], u[1::2])])
    assert abs(n.mean()) < 0.03 and abs(n.std() - 1.0) < 0.03
    assert scipy.stats.kstest(n, "norm").pvalue > 1e-3


NET = oracle.Net(obs_dim=5, h1=6, h2=7, act=0, heads=(4, 3, 2), n_gauss=2)


def _setup(seed, n=40):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.7, NET.num_params)
    obs = rng.normal(size=(n, NET.obs_dim)).astype(np.float32)
    return p, obs


def test_policy_act_reproduced_from_its_definition():
    p, obs = _setup(1)
    seed, draw0 = 99, 12345
    act, actc, logp, val = oracle.policy_act(NET, p, obs, seed, draw0)
    z = oracle.forward(NET, p, obs)
    NH, G = len(NET.heads), NET.n_gauss
    K = NH + 2 * G
    C = NET.out_cols
    logstd = p[-G:]
    for i in range(obs.shape[0]):
        d = [oracle.mulberry32_at(seed, draw0 + i * K + k) for k in range(K)]
        u = [(x >> 8) / 2.0 ** 24 for x in d]
        off = 0
        for h, nh in enumerate(NET.heads):
            cdf = np.cumsum(scipy.special.softmax(z[i, off:off + nh]))
            ref = min(int(np.searchsorted(cdf, u[h], side="right")), nh - 1)
            assert act[i, h] == ref
            off += nh
        for g in range(G):
            u1, u2 = u[NH + 2 * g], u[NH + 2 * g + 1]
            nrm = math.sqrt(-2 * math.log(1 - u1)) * math.cos(2 * math.pi * u2)
            assert abs(actc[i, g] - (z[i, off + g] + math.exp(logstd[g]) * nrm)) < 1e-12
        assert abs(val[i] - z[i, C - 1]) < 1e-13
    # the kept log-probability is the pinned policy log-probability of the
    # stored (fp32) action
    lp, _ = oracle.policy_logp(NET, p, obs, act, actc.astype(np.float32))
    np.testing.assert_allclose(logp, lp, rtol=1e-13, atol=1e-13)


def test_policy_act_draws_follow_the_distribution():
    p, obs = _setup(2, n=1)
    reps = 20000
    obs_rep = np.repeat(obs, reps, axis=0)
    act, actc, _, _ = oracle.policy_act(NET, p, obs_rep, seed=5, draw0=0)
    z = oracle.forward(NET, p, obs)[0]
    off = 0
    for h, nh in enumerate(NET.heads):
        prob = scipy.special.softmax(z[off:off + nh])
        counts = np.bincount(act[:, h], minlength=nh)
        chi2 = scipy.stats.chisquare(counts, prob * reps)
        assert chi2.pvalue > 1e-4, (h, counts, prob * reps)
        off += nh
    logstd = p[-NET.n_gauss:]
    for g in range(NET.n_gauss):
        mu, sd = z[off + g], math.exp(logstd[g])
        assert abs(actc[:, g].mean() - mu) < 4 * sd / math.sqrt(reps)
        assert abs(actc[:, g].std() / sd - 1.0) < 0.03


def test_policy_act_is_a_function_of_seed_and_counter():
    p, obs = _setup(3)
    a1 = oracle.policy_act(NET, p, obs, 7, 0)
    a2 = oracle.policy_act(NET, p, obs, 7, 0)
    for x, y in zip(a1, a2):
        np.testing.assert_array_equal(x, y)
    # agent i at counter draw0 is agent 0 at counter draw0 + i K
    K = len(NET.heads) + 2 * NET.n_gauss
    b = oracle.policy_act(NET, p, obs[5:6], 7, 5 * K)
    np.testing.assert_array_equal(b[0][0], a1[0][5])
    np.testing.assert_array_equal(b[1][0], a1[1][5])
    c = oracle.policy_act(NET, p, obs, 8, 0)
    assert not np.array_equal(c[0], a1[0])
