"""Pins of the oracle's gradient-norm clip, Adam step and whole update.

"PlayTrain", Table 8 (PPO column): Adam, gradient-norm clip 0.5.
Checked against Adam's step-1 closed form and against torch's float64
Adam / clip_grad_norm_ as independent library references; the whole update is
checked to be exactly the composition of its (separately pinned) parts.
"""
import numpy as np
import pytest

import oracle


def test_adam_first_step_closed_form():
    rng = np.random.default_rng(0)
    p = rng.normal(size=100)
    g = rng.normal(size=100)
    g[:5] = 0.0
    p1, m1, v1 = oracle.adam(p, g, np.zeros(100), np.zeros(100), 1, 1e-3)
    np.testing.assert_allclose(p1, p - 1e-3 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=1e-15)
    assert np.all(p1[:5] == p[:5])
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-12)


def test_adam_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    p0 = rng.normal(size=257)
    w = torch.tensor(p0.copy(), dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([w], lr=2.5e-4, betas=(0.9, 0.999), eps=1e-8)
    p, m, v = p0.copy(), np.zeros(257), np.zeros(257)
    for step in range(1, 8):
        g = rng.normal(size=257) * (0.1 ** step)
        w.grad = torch.tensor(g)
        opt.step()
        p, m, v = oracle.adam(p, g, m, v, step, 2.5e-4)
    np.testing.assert_allclose(p, w.detach().numpy(), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("scale", [0.01, 10.0])
def test_clip_grad_norm_matches_torch(scale):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(2).normal(size=300) * scale
    n, gc = oracle.clip_grad_norm(g, 0.5)
    t = torch.tensor(g.copy(), dtype=torch.float64, requires_grad=True)
    t.grad = torch.tensor(g.copy())
    tn = torch.nn.utils.clip_grad_norm_([t], 0.5)
    assert abs(n - tn.item()) < 1e-12 * tn.item()
    np.testing.assert_allclose(gc, t.grad.numpy(), rtol=1e-13)
    n0, g0 = oracle.clip_grad_norm(g, 0.0)          # 0 disables clipping
    assert np.array_equal(g0, g)


def test_update_is_the_composition_of_its_parts():
    from policy_rl_gb300 import synth
    w = synth.WORKLOADS["tiny"].scaled(T=16, N=8, minibatches=4, epochs=2)
    ro = synth.rollout(w)
    p0 = synth.init_params(w).astype(np.float64)
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, seed=3)
    res = oracle.update(net, hp, w.T, w.N, w.epochs, w.minibatches, ro.obs, ro.act_disc,
                        ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    adv, ret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
    mean, sd = oracle.moments(adv)
    p, m, v, step = p0.copy(), np.zeros_like(p0), np.zeros_like(p0), 0
    mb = w.B // w.minibatches
    for e in range(w.epochs):
        perm = oracle.perm(3, e, w.B)
        for k in range(w.minibatches):
            _, g, st, _ = oracle.loss_grad(net, p, perm[k * mb:(k + 1) * mb], ro.obs, ro.act_disc,
                                           ro.act_cont, ro.logp_old, adv.ravel(), ret.ravel(),
                                           normalize=True, adv_mean=mean, adv_std=sd)
            _, g = oracle.clip_grad_norm(g, 0.5)
            step += 1
            p, m, v = oracle.adam(p, g, m, v, step, 2.5e-4)
            np.testing.assert_array_equal(res.stats[e * w.minibatches + k], st)
    assert res.step == step
    np.testing.assert_array_equal(res.params, p)
    np.testing.assert_array_equal(res.adv, adv)
