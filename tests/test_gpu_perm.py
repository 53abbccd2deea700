"""Minibatch permutation: bit-exact against the oracle ("Teaching Mario to
speedrun", sec. 6 shuffle; "PlayTrain", App. F.2 mulberry32)."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


def _perm(seed, epoch, B):
    import torch
    import policy_rl_gb300 as P
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    work = torch.empty(P.ppo_perm_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    P.ppo_minibatch_perm(seed, epoch, B, out, work)
    return out.cpu().numpy()


@pytest.mark.parametrize("B", [1, 2, 31, 4095, 4096, 4097, 8192, 100003, 262144])
@pytest.mark.parametrize("epoch", [0, 3])
def test_perm_bit_exact(B, epoch):
    assert np.array_equal(_perm(1234, epoch, B), oracle.perm(1234, epoch, B))


def test_perm_full_size_with_ties():
    """4,194,304 rows (64 steps x 65,536 envs): mulberry32 repeats keys at this
    length, so index order of ties is exercised."""
    B = 64 * 65536
    got = _perm(0, 2, B)
    ref = oracle.perm(0, 2, B)
    assert np.array_equal(got, ref)


def test_perm_seeds_wrap():
    for seed in (0xFFFFFFFF, 0x80000000):
        assert np.array_equal(_perm(seed, 1, 5000), oracle.perm(seed, 1, 5000))
