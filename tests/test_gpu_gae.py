"""GAE kernel vs the oracle ("Teaching Mario to speedrun", sec. 6 "Better
advantages").  Tolerance: |x - y| <= 1e-5 (|y| + rms(y)) element by element
for advantages, returns and normalised advantages (fp32 scan against the fp64
oracle); mean/std within 1e-5 relative to rms(A)."""
import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import assert_elementwise, dev, host

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny", 128, 64),
    ("ragged", 37, 1000),        # T not a multiple of the 16-step chunk, N not of 128
    ("one_env", 300, 1),
    ("one_step", 1, 777),
    ("mario", 128, 2048),
    ("gae_stress", 1024, 65536),  # full-size bandwidth workload
]


def _run(T, N, w, seed=0):
    import torch
    import policy_rl_gb300 as P
    w = w.scaled(T=T, N=N)
    ro = synth.rollout(w, seed=seed)
    adv = torch.empty(T, N, device="cuda")
    ret = torch.empty(T, N, device="cuda")
    advn = torch.empty(T, N, device="cuda")
    stats = torch.empty(4, device="cuda")
    work = torch.empty(P.ppo_gae_workspace_bytes(T, N), dtype=torch.uint8, device="cuda")
    P.ppo_gae(dev(ro.rew), dev(ro.val), dev(ro.done), dev(ro.boot), w.gamma, w.lam, adv, ret,
              advn, stats, work)
    torch.cuda.synchronize()
    return ro, w, host(adv), host(ret), host(advn), host(stats)


@pytest.mark.parametrize("name,T,N", CASES)
def test_gae_matches_oracle(name, T, N):
    base = synth.WORKLOADS["gae_stress" if name == "gae_stress" else "tiny"]
    ro, w, adv, ret, advn, st = _run(T, N, base)
    oadv, oret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
    assert_elementwise(adv, oadv, 1e-5)
    assert_elementwise(ret, oret, 1e-5)
    m, s = oracle.moments(oadv)
    rms = float(np.sqrt(np.mean(oadv * oadv)))
    assert abs(st[0] - m) <= 1e-5 * rms
    if T * N > 1:
        assert abs(st[1] - s) <= 1e-5 * s
        assert_elementwise(advn, oracle.normalize(oadv, m, s), 1e-5)


def test_gae_all_done_and_no_done():
    import torch
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["tiny"].scaled(T=40, N=300)
    ro = synth.rollout(w)
    for done in (np.ones_like(ro.done), np.zeros_like(ro.done)):
        adv = torch.empty(40, 300, device="cuda")
        ret = torch.empty(40, 300, device="cuda")
        P.ppo_gae(dev(ro.rew), dev(ro.val), dev(done), dev(ro.boot), 0.99, 0.95, adv, ret)
        oadv, oret = oracle.gae(ro.rew, ro.val, done, ro.boot, 0.99, 0.95)
        assert_elementwise(host(adv), oadv, 1e-5)
        assert_elementwise(host(ret), oret, 1e-5)


def test_gae_is_deterministic():
    a = _run(256, 3000, synth.WORKLOADS["tiny"])
    b = _run(256, 3000, synth.WORKLOADS["tiny"])
    for x, y in zip(a[2:], b[2:]):
        assert np.array_equal(x, y)


def test_gae_rejects_bad_arguments():
    import torch
    import policy_rl_gb300 as P
    x = torch.zeros(8, 8, device="cuda")
    with pytest.raises(P.PpoError):       # stats requested without workspace
        P.ppo_gae(x, x, x, x[0], 0.99, 0.95, x, x, stats=torch.zeros(4, device="cuda"))
    big = torch.zeros(64, device="cuda")
    with pytest.raises(P.PpoError):       # misaligned view
        P.ppo_gae(big[1:].view(1, 63), big[1:].view(1, 63), big[1:].view(1, 63), big[1:],
                  0.99, 0.95, big[1:].view(1, 63), big[1:].view(1, 63))
