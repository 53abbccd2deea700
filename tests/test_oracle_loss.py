"""Pins of the oracle's MLP actor-critic loss and gradient.

"Teaching Mario to speedrun", sec. 5 (gradient of the log-softmax),
sec. 6 (shared actor-critic, one head per action part, clipped ratio, value
and entropy terms); "boesch.dev DDNet RL", "What the agent sees and does"
(hybrid discrete + continuous actions).

The oracle is pinned against: central finite differences of its own loss
(backward vs forward), closed forms of special cases (uniform heads, r = 1,
r = 2 clipped / unclipped, V = R), brute-force enumeration of the joint
action space, scipy's Gaussian log-density and entropy, and an independent
float64 torch autograd implementation.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle


def _setup(net, B, seed, scale=0.5):
    rng = np.random.default_rng(seed)
    params = rng.normal(0, scale, net.num_params)
    obs = rng.normal(size=(B, net.obs_dim)).astype(np.float32)
    act = np.stack([rng.integers(0, n, B) for n in net.heads], 1).astype(np.int32)
    actc = rng.normal(size=(B, net.n_gauss)).astype(np.float32)
    logp_old = rng.normal(-2.0, 0.7, B).astype(np.float32)
    adv = rng.normal(size=B)
    ret = rng.normal(size=B)
    return params, obs, act, actc, logp_old, adv, ret


def _logp_ent(net, params, obs, act, actc, row):
    """Per-row log-probability and entropy read from the oracle's stats:
    with logp_old = 0, advantage -1 and an unbounded clip range the policy
    term of the loss is exactly the probability ratio exp(logp)."""
    B = obs.shape[0]
    _, _, st, _ = oracle.loss_grad(net, params, [row], obs, act, actc, np.zeros(B, np.float32),
                                   -np.ones(B), np.zeros(B), clip=1e9, vf_coef=0.0,
                                   ent_coef=0.0)
    return math.log(st[1]), st[3]


NETS = [
    oracle.Net(3, 4, 4, act=0, heads=(3, 2), n_gauss=1),
    oracle.Net(3, 4, 5, act=1, heads=(2, 3, 2), n_gauss=0),
    oracle.Net(2, 3, 3, act=0, heads=(4,), n_gauss=2),
]


@pytest.mark.parametrize("net", NETS)
@pytest.mark.parametrize("normalize", [False, True])
def test_gradient_matches_central_differences(net, normalize):
    B = 7
    params, obs, act, actc, logp_old, adv, ret = _setup(net, B, 11)
    idx = np.array([4, 0, 6, 2, 2], np.int32)
    kw = dict(clip=0.2, vf_coef=0.5, ent_coef=0.01, normalize=normalize, adv_mean=0.3,
              adv_std=1.7)
    _, g, _, _ = oracle.loss_grad(net, params, idx, obs, act, actc, logp_old, adv, ret, **kw)
    h = 1e-6
    fd = np.empty_like(g)
    for i in range(net.num_params):
        p1 = params.copy(); p1[i] += h
        p0 = params.copy(); p0[i] -= h
        l1 = oracle.loss_grad(net, p1, idx, obs, act, actc, logp_old, adv, ret, **kw)[0]
        l0 = oracle.loss_grad(net, p0, idx, obs, act, actc, logp_old, adv, ret, **kw)[0]
        fd[i] = (l1 - l0) / (2 * h)
    np.testing.assert_allclose(g, fd, rtol=1e-5, atol=1e-8)


def test_uniform_heads_closed_form():
    net = oracle.Net(3, 4, 4, act=0, heads=(3, 2, 2))
    params, obs, act, actc, logp_old, adv, ret = _setup(net, 5, 2)
    C, H2 = net.out_cols, net.h2
    off = net.num_params - (C * H2 + C + net.n_gauss)
    params[off:off + C * H2 + C] = 0.0           # W3 = 0, b3 = 0
    for r in range(5):
        lp, ent = _logp_ent(net, params, obs, act, actc, r)
        assert abs(lp + math.log(3) + 2 * math.log(2)) < 1e-12
        assert abs(ent - (math.log(3) + 2 * math.log(2))) < 1e-12


def test_joint_action_probabilities_sum_to_one_and_entropy_is_exact():
    net = oracle.Net(3, 4, 4, act=0, heads=(3, 2, 4))
    params, obs, _, actc, _, _, _ = _setup(net, 1, 3, scale=1.0)
    probs = []
    ent = None
    for a in itertools.product(*[range(n) for n in net.heads]):
        act = np.array([a], np.int32)
        lp, ent = _logp_ent(net, params, obs, act, actc, 0)
        probs.append(math.exp(lp))
    probs = np.array(probs)
    assert abs(probs.sum() - 1.0) < 1e-12
    assert abs(ent - float(-(probs * np.log(probs)).sum())) < 1e-12


def test_heads_are_log_softmax_of_forward_logits():
    net = oracle.Net(3, 4, 4, act=1, heads=(3, 2))
    params, obs, act, actc, _, _, _ = _setup(net, 4, 4, scale=1.0)
    z = oracle.forward(net, params, obs)
    for r in range(4):
        ref = (scipy.special.log_softmax(z[r, 0:3])[act[r, 0]]
               + scipy.special.log_softmax(z[r, 3:5])[act[r, 1]])
        lp, _ = _logp_ent(net, params, obs, act, actc, r)
        assert abs(lp - ref) < 1e-12


def test_forward_is_three_affine_maps():
    """Forward of a non-square net against numpy matrix products (catches a
    transposed weight or a swapped layer)."""
    for act in (0, 1):
        net = oracle.Net(5, 3, 4, act=act, heads=(2, 3), n_gauss=1)
        params, obs, *_ = _setup(net, 6, 5, scale=1.0)
        D, H1, H2, C = 5, 3, 4, net.out_cols
        o = 0
        W1 = params[o:o + H1 * D].reshape(H1, D); o += H1 * D
        b1 = params[o:o + H1]; o += H1
        W2 = params[o:o + H2 * H1].reshape(H2, H1); o += H2 * H1
        b2 = params[o:o + H2]; o += H2
        W3 = params[o:o + C * H2].reshape(C, H2); o += C * H2
        b3 = params[o:o + C]
        f = np.tanh if act == 0 else (lambda x: np.maximum(x, 0))
        ref = f(f(obs.astype(np.float64) @ W1.T + b1) @ W2.T + b2) @ W3.T + b3
        np.testing.assert_allclose(oracle.forward(net, params, obs), ref, rtol=1e-12, atol=1e-12)


def test_gaussian_head_matches_scipy():
    net = oracle.Net(3, 4, 4, act=0, heads=(2,), n_gauss=2)
    params, obs, act, actc, _, _, _ = _setup(net, 3, 6)
    C, H2 = net.out_cols, net.h2
    off = net.num_params - (C * H2 + C + 2)
    params[off:off + C * H2] = 0.0
    mu = np.array([0.3, -1.1])
    s = np.array([-0.4, 0.25])
    params[off + C * H2: off + C * H2 + C] = [0.0, 0.0, mu[0], mu[1], 0.7]
    params[-2:] = s
    for r in range(3):
        lp, ent = _logp_ent(net, params, obs, act, actc, r)
        ref = -math.log(2) + sum(scipy.stats.norm.logpdf(actc[r, g], mu[g], math.exp(s[g]))
                                 for g in range(2))
        ref_ent = math.log(2) + sum(scipy.stats.norm(mu[g], math.exp(s[g])).entropy()
                                    for g in range(2))
        assert abs(lp - ref) < 1e-10
        assert abs(ent - ref_ent) < 1e-12


def _logp_all(net, params, obs, act, actc, rows):
    return np.array([_logp_ent(net, params, obs, act, actc, r)[0] for r in rows])


def test_ratio_one_gives_the_vanilla_policy_gradient():
    """At ratio = 1 the clipped surrogate's gradient is -mean(A grad logp)."""
    net = oracle.Net(3, 4, 4, act=0, heads=(3, 2), n_gauss=1)
    B = 6
    params, obs, act, actc, _, adv, ret = _setup(net, B, 7)
    rows = np.arange(B, dtype=np.int32)
    logp = _logp_all(net, params, obs, act, actc, rows)
    _, g, st, _ = oracle.loss_grad(net, params, rows, obs, act, actc, logp.astype(np.float32),
                                   adv, ret, clip=0.2, vf_coef=0.0, ent_coef=0.0)
    assert abs(st[1] + adv.mean()) < 1e-6          # pg loss at r = 1 is -mean(A)
    h = 1e-6
    fd = np.empty_like(g)
    for i in range(net.num_params):
        p1 = params.copy(); p1[i] += h
        p0 = params.copy(); p0[i] -= h
        f1 = -np.mean(adv * _logp_all(net, p1, obs, act, actc, rows))
        f0 = -np.mean(adv * _logp_all(net, p0, obs, act, actc, rows))
        fd[i] = (f1 - f0) / (2 * h)
    np.testing.assert_allclose(g, fd, rtol=2e-5, atol=1e-7)


def test_clipped_samples_have_zero_policy_gradient():
    net = oracle.Net(3, 4, 4, act=0, heads=(3, 2))
    B = 5
    params, obs, act, actc, _, _, ret = _setup(net, B, 8)
    rows = np.arange(B, dtype=np.int32)
    logp = _logp_all(net, params, obs, act, actc, rows)
    logp_old = (logp - math.log(2.0)).astype(np.float32)          # ratio = 2
    pos = np.abs(np.random.default_rng(1).normal(size=B)) + 0.1
    _, g, st, _ = oracle.loss_grad(net, params, rows, obs, act, actc, logp_old, pos, ret,
                                   clip=0.2, vf_coef=0.0, ent_coef=0.0)
    assert np.all(g == 0.0)
    assert abs(st[1] + 1.2 * pos.mean()) < 1e-6                    # -clip(r) A
    assert st[4] == 1.0                                            # clipfrac
    assert abs(st[5] - (1.0 - math.log(2.0))) < 1e-6               # (r-1) - log r
    # negative advantages at r = 2: the unclipped term is the minimum
    _, gneg, stn, _ = oracle.loss_grad(net, params, rows, obs, act, actc, logp_old, -pos, ret,
                                       clip=0.2, vf_coef=0.0, ent_coef=0.0)
    assert abs(stn[1] - 2.0 * pos.mean()) < 1e-6
    _, g1, _, _ = oracle.loss_grad(net, params, rows, obs, act, actc, logp.astype(np.float32),
                                   -pos, ret, clip=0.2, vf_coef=0.0, ent_coef=0.0)
    # logp_old is float32, so both ratios carry ~|logp| * 6e-8 relative rounding
    np.testing.assert_allclose(gneg, 2.0 * g1, rtol=1e-5, atol=1e-12)


def test_value_term_closed_form():
    net = oracle.Net(3, 4, 4, act=0, heads=(3, 2))
    B = 6
    params, obs, act, actc, logp_old, _, _ = _setup(net, B, 9)
    rows = np.arange(B, dtype=np.int32)
    V = oracle.forward(net, params, obs)[:, -1]
    zero = np.zeros(B)
    _, g, st, _ = oracle.loss_grad(net, params, rows, obs, act, actc, logp_old, zero, V,
                                   vf_coef=0.5, ent_coef=0.0)
    assert np.max(np.abs(g)) < 1e-14 and abs(st[2]) < 1e-28        # V = R
    _, g, st, _ = oracle.loss_grad(net, params, rows, obs, act, actc, logp_old, zero, V - 1.0,
                                   vf_coef=0.5, ent_coef=0.0)
    assert abs(st[2] - 1.0) < 1e-12 and abs(st[0] - 0.5) < 1e-12
    assert abs(g[net.num_params - 1] - 2 * 0.5 * 1.0) < 1e-12      # d/d b_V of 0.5 mean (V-R)^2


def _torch_loss(net, params, obs, act, actc, logp_old, adv, ret, idx, clip, vf, ent_c):
    """Independent float64 restatement with torch autograd."""
    import torch
    p = torch.tensor(params, dtype=torch.float64, requires_grad=True)
    D, H1, H2, C, G = net.obs_dim, net.h1, net.h2, net.out_cols, net.n_gauss
    o = 0
    def take(n, shape):
        nonlocal o
        t = p[o:o + n].reshape(shape); o += n
        return t
    W1 = take(H1 * D, (H1, D)); b1 = take(H1, (H1,))
    W2 = take(H2 * H1, (H2, H1)); b2 = take(H2, (H2,))
    W3 = take(C * H2, (C, H2)); b3 = take(C, (C,)); ls = take(G, (G,))
    f = torch.tanh if net.act == 0 else torch.relu
    x = torch.tensor(obs[idx], dtype=torch.float64)
    z = f(f(x @ W1.T + b1) @ W2.T + b2) @ W3.T + b3
    a = torch.tensor(act[idx], dtype=torch.long)
    logp = torch.zeros(len(idx), dtype=torch.float64)
    ent = torch.zeros(len(idx), dtype=torch.float64)
    c0 = 0
    for h, n in enumerate(net.heads):
        dist = torch.distributions.Categorical(logits=z[:, c0:c0 + n])
        logp = logp + dist.log_prob(a[:, h]); ent = ent + dist.entropy(); c0 += n
    if G:
        nd = torch.distributions.Normal(z[:, c0:c0 + G], torch.exp(ls).expand(len(idx), G))
        ac = torch.tensor(actc[idx], dtype=torch.float64)
        logp = logp + nd.log_prob(ac).sum(1); ent = ent + nd.entropy().sum(1)
    V = z[:, -1]
    A = torch.tensor(adv[idx], dtype=torch.float64)
    R = torch.tensor(ret[idx], dtype=torch.float64)
    r = torch.exp(logp - torch.tensor(logp_old[idx], dtype=torch.float64))
    pg = -torch.minimum(r * A, torch.clamp(r, 1 - clip, 1 + clip) * A)
    loss = pg.mean() + vf * ((V - R) ** 2).mean() - ent_c * ent.mean()
    loss.backward()
    return loss.item(), p.grad.numpy()


@pytest.mark.parametrize("net", NETS + [oracle.Net(6, 8, 8, act=0, heads=(9, 2, 2, 2))])
def test_matches_torch_autograd(net):
    B = 16
    params, obs, act, actc, logp_old, adv, ret = _setup(net, B, 13)
    idx = np.random.default_rng(0).permutation(B)[:12].astype(np.int32)
    loss, g, _, _ = oracle.loss_grad(net, params, idx, obs, act, actc, logp_old, adv, ret,
                                     clip=0.2, vf_coef=0.5, ent_coef=0.01)
    tl, tg = _torch_loss(net, params, obs, act, actc, logp_old, adv, ret, idx, 0.2, 0.5, 0.01)
    assert abs(loss - tl) < 1e-12 * max(1.0, abs(tl))
    np.testing.assert_allclose(g, tg, rtol=1e-10, atol=1e-13)


def test_policy_logp_matches_scipy_and_the_loss():
    net = oracle.Net(3, 4, 4, act=1, heads=(3, 2), n_gauss=2)
    params, obs, act, actc, _, _, _ = _setup(net, 6, 12, scale=1.0)
    lp, ent = oracle.policy_logp(net, params, obs, act, actc)
    z = oracle.forward(net, params, obs)
    ls = params[-2:]
    for r in range(6):
        ref = (scipy.special.log_softmax(z[r, 0:3])[act[r, 0]]
               + scipy.special.log_softmax(z[r, 3:5])[act[r, 1]]
               + sum(scipy.stats.norm.logpdf(actc[r, g], z[r, 5 + g], math.exp(ls[g]))
                     for g in range(2)))
        assert abs(lp[r] - ref) < 1e-10
        lp2, ent2 = _logp_ent(net, params, obs, act, actc, r)
        assert abs(lp[r] - lp2) < 1e-12 and abs(ent[r] - ent2) < 1e-12


# ---- bf16-operand mode -------------------------------------------------------
def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.normal(size=2000) * 10.0 ** rng.integers(-30, 30, 2000),
                         [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 1.0078125, -2.5, 3e-39,
                          1e-45, 3.3895313892515355e38]])
    ref = torch.tensor(xs, dtype=torch.float64).float().bfloat16().double().numpy()
    got = np.array([oracle.round_bf16(x) for x in xs])
    np.testing.assert_array_equal(got, ref)


def test_bf16_mode_is_exact_on_representable_operands():
    """ReLU net whose weights, observations, activations and value signal are
    all bf16-exact dyadics: bf16-operand mode must equal the fp64 mode bit
    for bit (no rounding of anything that was not rounded, no lost term)."""
    net = oracle.Net(4, 4, 4, act=1, heads=(2,), n_gauss=0)
    rng = np.random.default_rng(4)
    params = rng.integers(-4, 5, net.num_params) / 8.0
    obs = rng.integers(-3, 4, (4, 4)).astype(np.float32)
    act = np.zeros((4, 1), np.int32)
    z = oracle.forward(net, params, obs)
    ret = z[:, -1] - rng.integers(-2, 3, 4) / 4.0          # V - R dyadic
    kw = dict(clip=0.2, vf_coef=0.5, ent_coef=0.0)
    args = (net, params, np.arange(4, dtype=np.int32), obs, act, None, np.zeros(4, np.float32),
            np.zeros(4), ret)
    l0, g0, s0, _ = oracle.loss_grad(*args, **kw)
    l1, g1, s1, _ = oracle.loss_grad(*args, bf16_operands=True, **kw)
    assert l0 == l1
    np.testing.assert_array_equal(g0, g1)


@pytest.mark.parametrize("seed", [0, 1])
def test_bf16_mode_is_close_to_fp64_on_tanh_nets(seed):
    net = oracle.Net(16, 32, 32, act=0, heads=(9, 2, 2, 2))
    params, obs, act, actc, logp_old, adv, ret = _setup(net, 64, seed, scale=0.2)
    idx = np.arange(64, dtype=np.int32)
    _, g0, s0, _ = oracle.loss_grad(net, params, idx, obs, act, actc, logp_old, adv, ret,
                                    clip=10.0)
    _, g1, s1, _ = oracle.loss_grad(net, params, idx, obs, act, actc, logp_old, adv, ret,
                                    clip=10.0, bf16_operands=True)
    assert np.linalg.norm(g1 - g0) / np.linalg.norm(g0) < 2e-2
    assert np.linalg.norm(g1 - g0) > 0          # the mode does round something
