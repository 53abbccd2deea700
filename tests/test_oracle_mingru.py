"""Pins of the oracle's recurrent (MinGRU) policy.

"Teaching Mario to speedrun", sec. 8: bias-free encoder, four MinGRU layers
whose gates depend only on the input and whose state clears when an episode
ends, one decoder matrix to the heads and the value.  MinGRU per Feng et al.
2024: z = sigmoid(W_z u + b_z), h~ = W_h u + b_h, h = (1 - z) h_prev + z h~.
Pinned against:
- central finite differences of the oracle's own loss (backpropagation
  through time vs forward), with terminals inside the segments;
- an independent float64 torch autograd implementation of the same policy and
  PPO loss (gradients and statistics);
- z = 1 (saturated gates): the recurrence is the feed-forward stack
  W_dec (W_h (... (W_enc x) ...)), computed with numpy;
- a terminal at step t cuts every influence of earlier steps and of the
  carried state on later outputs (exactly).
"""
import numpy as np
import pytest

import oracle

RNN = oracle.Rnn(obs_dim=3, hidden=4, layers=2, heads=(3, 2), n_gauss=1)


def _data(rnn, T, N, seed, p_done=0.2):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.5, rnn.num_params)
    B = T * N
    obs = rng.normal(size=(B, rnn.obs_dim)).astype(np.float32)
    act = np.stack([rng.integers(0, n, B) for n in rnn.heads], 1).astype(np.int32)
    actc = rng.normal(size=(B, rnn.n_gauss)).astype(np.float32)
    lp = rng.normal(-2.0, 0.3, B).astype(np.float32)
    adv = rng.normal(size=B)
    ret = rng.normal(size=B)
    done = (rng.random((T, N)) < p_done).astype(np.float32)
    h0 = rng.normal(0, 0.5, size=(N, rnn.layers, rnn.hidden))
    return p, obs, act, actc, lp, adv, ret, done, h0


def test_bptt_gradient_matches_finite_differences():
    T, N = 6, 3
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(RNN, T, N, 1)
    done[2, 2] = 1.0                          # a terminal inside a used segment
    envs = np.array([2, 0], np.int32)
    kw = dict(clip=100.0)                     # smooth (unclipped) branch everywhere
    _, g, _, _ = oracle.rnn_loss_grad(RNN, p, envs, obs, act, actc, lp, adv, ret, done, h0, **kw)
    eps = 1e-6
    fd = np.empty_like(p)
    for i in range(p.size):
        q = p.copy()
        q[i] += eps
        lp_, *_ = oracle.rnn_loss_grad(RNN, q, envs, obs, act, actc, lp, adv, ret, done, h0, **kw)
        q[i] -= 2 * eps
        lm_, *_ = oracle.rnn_loss_grad(RNN, q, envs, obs, act, actc, lp, adv, ret, done, h0, **kw)
        fd[i] = (lp_ - lm_) / (2 * eps)
    np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-9)


def _torch_loss(rnn, p, envs, obs, act, actc, lp, adv, ret, done, h0, clip, vf, ent_c):
    torch = pytest.importorskip("torch")
    T, N = done.shape
    D, H, L, C = rnn.obs_dim, rnn.hidden, rnn.layers, rnn.out_cols
    P = torch.tensor(p, dtype=torch.float64, requires_grad=True)
    o = 0

    def take(*shape):
        nonlocal o
        n = int(np.prod(shape))
        t = P[o:o + n].reshape(*shape)
        o += n
        return t
    Wenc = take(H, D)
    layers = [(take(H, H), take(H), take(H, H), take(H)) for _ in range(L)]
    Wdec = take(C, H)
    logstd = take(rnn.n_gauss)
    rows, zs = [], []
    for n in envs:
        h = [torch.tensor(h0[n, l], dtype=torch.float64) for l in range(L)]
        for t in range(T):
            if t > 0 and done[t - 1, n] != 0:
                h = [torch.zeros(H, dtype=torch.float64) for _ in range(L)]
            u = Wenc @ torch.tensor(obs[t * N + n], dtype=torch.float64)
            for l, (Wz, bz, Wh, bh) in enumerate(layers):
                z = torch.sigmoid(Wz @ u + bz)
                h[l] = (1 - z) * h[l] + z * (Wh @ u + bh)
                u = h[l]
            zs.append(Wdec @ u)
            rows.append(t * N + n)
    Z = torch.stack(zs)
    rows = np.array(rows)
    logp = torch.zeros(len(rows), dtype=torch.float64)
    ent = torch.zeros(len(rows), dtype=torch.float64)
    off = 0
    for h, nh in enumerate(rnn.heads):
        ls = torch.log_softmax(Z[:, off:off + nh], dim=1)
        a = torch.tensor(act[rows, h], dtype=torch.long)
        logp = logp + ls[torch.arange(len(rows)), a]
        ent = ent - (ls.exp() * ls).sum(1)
        off += nh
    for g in range(rnn.n_gauss):
        mu = Z[:, off + g]
        a = torch.tensor(actc[rows, g], dtype=torch.float64)
        logp = logp - (a - mu) ** 2 / (2 * torch.exp(2 * logstd[g])) - logstd[g] \
            - 0.5 * np.log(2 * np.pi)
        ent = ent + 0.5 + 0.5 * np.log(2 * np.pi) + logstd[g]
    A = torch.tensor(adv[rows], dtype=torch.float64)
    R = torch.tensor(ret[rows], dtype=torch.float64)
    ratio = torch.exp(logp - torch.tensor(lp[rows], dtype=torch.float64))
    pg = -torch.minimum(ratio * A, torch.clamp(ratio, 1 - clip, 1 + clip) * A)
    V = Z[:, C - 1]
    loss = pg.mean() + vf * ((V - R) ** 2).mean() - ent_c * ent.mean()
    loss.backward()
    return loss.item(), P.grad.numpy(), pg.mean().item(), ((V - R) ** 2).mean().item(), \
        ent.mean().item()


@pytest.mark.parametrize("layers,hidden,G", [(2, 4, 1), (4, 8, 0), (4, 6, 2)])
def test_matches_torch_autograd(layers, hidden, G):
    rnn = oracle.Rnn(obs_dim=5, hidden=hidden, layers=layers, heads=(4, 2, 3), n_gauss=G)
    T, N = 9, 4
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, 2 + layers)
    envs = np.array([3, 1, 0], np.int32)
    loss, g, st, _ = oracle.rnn_loss_grad(rnn, p, envs, obs, act, actc, lp, adv, ret, done, h0)
    tl, tg, tpg, tvl, tent = _torch_loss(rnn, p, envs, obs, act, actc, lp, adv, ret, done, h0,
                                         0.2, 0.5, 0.01)
    assert abs(loss - tl) < 1e-12 * max(1, abs(tl))
    np.testing.assert_allclose(st[[1, 2, 3]], [tpg, tvl, tent], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g, tg, rtol=1e-10, atol=1e-13)


def test_saturated_gates_are_a_feed_forward_stack():
    rnn = oracle.Rnn(obs_dim=4, hidden=5, layers=3, heads=(2,), n_gauss=0)
    T, N = 4, 2
    p, obs, *_, done, h0 = _data(rnn, T, N, 7)
    D, H, L, C = rnn.obs_dim, rnn.hidden, rnn.layers, rnn.out_cols
    q = p.copy()
    o = H * D
    Ws = []
    for _ in range(L):
        q[o + H * H:o + H * H + H] = 60.0          # b_z: sigmoid(60) == 1 in fp64
        Ws.append((q[o + H * H + H:o + 2 * H * H + H].reshape(H, H),
                   q[o + 2 * H * H + H:o + 2 * H * H + 2 * H]))
        o += 2 * H * H + 2 * H
    Wenc = q[:H * D].reshape(H, D)
    Wdec = q[o:o + C * H].reshape(C, H)
    z = oracle.rnn_forward(rnn, q, obs, done, h0[1], n=1)
    for t in range(T):
        u = Wenc @ obs[t * N + 1].astype(np.float64)
        for Wh, bh in Ws:
            u = Wh @ u + bh
        np.testing.assert_allclose(z[t], Wdec @ u, rtol=1e-13, atol=1e-13)


def test_terminal_cuts_the_past():
    rnn = oracle.Rnn(obs_dim=3, hidden=4, layers=4, heads=(3,), n_gauss=0)
    T, N = 8, 1
    p, obs, *_, done, h0 = _data(rnn, T, N, 9, p_done=0.0)
    done[3, 0] = 1.0                                 # episode ends during step 3
    z = oracle.rnn_forward(rnn, p, obs, done, h0[0])
    obs2 = obs.copy()
    obs2[:4] += 1.0                                  # change steps 0..3 and the carried state
    z2 = oracle.rnn_forward(rnn, p, obs2, done, h0[0] + 1.0)
    np.testing.assert_array_equal(z[4:], z2[4:])
    assert not np.allclose(z[:4], z2[:4])


def test_rnn_update_is_the_composition():
    rnn = oracle.Rnn(obs_dim=3, hidden=4, layers=2, heads=(3, 2), n_gauss=1)
    T, N, E, M = 5, 8, 2, 2
    p, obs, act, actc, lp, _, _, done, h0 = _data(rnn, T, N, 11)
    rng = np.random.default_rng(12)
    val = rng.normal(size=(T, N)).astype(np.float32)
    rew = rng.normal(size=(T, N)).astype(np.float32)
    boot = rng.normal(size=N).astype(np.float32)
    hp = oracle.Hyper(lr=1e-3, seed=21)
    q, m, v, step, stats = oracle.rnn_update(rnn, hp, T, N, E, M, obs, act, actc, lp, val, rew,
                                             done, boot, h0, p)
    adv, ret = oracle.gae(rew, val, done, boot, hp.gamma, hp.lam)
    mean, sd = oracle.moments(adv)
    r, mr, vr = p.copy(), np.zeros(p.size), np.zeros(p.size)
    ns = N // M
    k = 0
    for e in range(E):
        perm = oracle.perm(hp.seed, e, N)
        for j in range(M):
            _, g, st, _ = oracle.rnn_loss_grad(rnn, r, perm[j * ns:(j + 1) * ns], obs, act, actc,
                                               lp, adv.ravel(), ret.ravel(), done, h0,
                                               normalize=True, adv_mean=mean, adv_std=sd)
            np.testing.assert_allclose(stats[k], st, rtol=1e-12, atol=1e-14)
            _, g = oracle.clip_grad_norm(g, hp.max_grad_norm)
            k += 1
            r, mr, vr = oracle.adam(r, g, mr, vr, k, hp.lr)
    assert step == E * M
    np.testing.assert_allclose(q, r, rtol=1e-12, atol=1e-14)


# ---- bf16-operand mode of the recurrent policy ----------------------------------
def test_rnn_bf16_mode_is_exact_on_representable_operands():
    """Saturated gates (b_z = 40: z = 1 exactly in fp64), dyadic weights and
    observations, no entropy term, zero advantages and a dyadic value error:
    every stored product and backpropagated value is bf16-exact, so the
    bf16-operand mode equals the fp64 mode bit for bit (it rounds nothing
    that was not rounded and drops no term)."""
    rnn = oracle.Rnn(obs_dim=3, hidden=4, layers=2, heads=(2,), n_gauss=0)
    rng = np.random.default_rng(7)
    T, N = 4, 2
    p = rng.integers(-2, 3, rnn.num_params) / 8.0
    D, H, L = rnn.obs_dim, rnn.hidden, rnn.layers
    per = 2 * H * H + 2 * H
    for l in range(L):
        p[H * D + l * per + H * H:H * D + l * per + H * H + H] = 40.0   # b_z
    obs = rng.integers(-2, 3, (T * N, D)).astype(np.float32)
    act = np.zeros((T * N, 1), np.int32)
    lp = np.zeros(T * N, np.float32)
    adv = np.zeros(T * N)
    done = np.zeros((T, N), np.float32)
    h0 = np.zeros((N, L, H))
    envs = np.arange(N, dtype=np.int32)
    # V from the fp64 forward, so that V - R is a small dyadic
    z = np.stack([oracle.rnn_forward(rnn, p, obs, done, h0[n], n) for n in range(N)],
                 axis=1)                                       # [T][N][C]
    ret = (z[..., -1].reshape(-1) - rng.integers(-2, 3, T * N) / 4.0)
    kw = dict(clip=0.2, vf_coef=0.5, ent_coef=0.0)
    l0, g0, _, _ = oracle.rnn_loss_grad(rnn, p, envs, obs, act, None, lp, adv, ret, done, h0, **kw)
    l1, g1, _, _ = oracle.rnn_loss_grad(rnn, p, envs, obs, act, None, lp, adv, ret, done, h0,
                                        bf16_operands=True, **kw)
    assert l0 == l1
    np.testing.assert_array_equal(g0, g1)
    assert np.abs(g0).sum() > 0


@pytest.mark.parametrize("seed", [0, 1])
def test_rnn_bf16_mode_is_close_to_fp64(seed):
    rnn = oracle.Rnn(obs_dim=16, hidden=32, layers=3, heads=(9, 2), n_gauss=1)
    T, N = 16, 4
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, seed, p_done=0.1)
    p *= 0.4
    envs = np.arange(N, dtype=np.int32)
    kw = dict(clip=10.0)
    _, g0, s0, _ = oracle.rnn_loss_grad(rnn, p, envs, obs, act, actc, lp, adv, ret, done, h0,
                                        **kw)
    _, g1, s1, _ = oracle.rnn_loss_grad(rnn, p, envs, obs, act, actc, lp, adv, ret, done, h0,
                                        bf16_operands=True, **kw)
    assert np.linalg.norm(g1 - g0) / np.linalg.norm(g0) < 2e-2
    assert np.linalg.norm(g1 - g0) > 0          # the mode does round something
    np.testing.assert_allclose(s1, s0, rtol=2e-2, atol=1e-6)
