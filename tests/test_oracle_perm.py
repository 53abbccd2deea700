"""Pins of the oracle's mulberry32 and minibatch permutation.

"PlayTrain", Appendix F.2 listing "seeded RNG" defines mulberry32 in
JavaScript; "Teaching Mario to speedrun", sec. 6 shuffles the batch into
minibatches.  The permutation is the index order sorted by (key, index),
key i being draw number epoch*B + i.
"""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mulberry32_draws.txt")


def _js_mulberry32(seed, count):
    """The listing's JavaScript evaluated with JavaScript's number semantics:
    `t` is an unbounded double, `^ | >>>` convert through ToInt32/ToUint32,
    Math.imul keeps the low 32 bits of the product of two int32s, `+` adds
    doubles.  Independent of the oracle's uint32 C code."""
    def to_u32(x):
        return int(x) % 2**32

    def to_i32(x):
        x = to_u32(x)
        return x - 2**32 if x >= 2**31 else x

    def imul(a, b):
        return to_i32(to_i32(a) * to_i32(b))

    t = to_u32(seed)
    out = []
    for _ in range(count):
        t = t + 0x6D2B79F5                       # plain double addition
        n = imul(to_i32(t) ^ (to_u32(t) >> 15), to_i32(t) | 1)
        n = to_i32(n) ^ to_i32(n + imul(to_i32(n) ^ (to_u32(n) >> 7), to_i32(n) | 61))
        out.append(to_u32(to_i32(n) ^ (to_u32(n) >> 14)))
    return out


def test_mulberry32_matches_the_listing_semantics():
    for seed in (0, 1, 42, 0xDEADBEEF, 2**32 - 1):
        ref = _js_mulberry32(seed, 64)
        got = oracle.mulberry32_stream(seed, 64).tolist()
        assert got == ref, seed


def test_mulberry32_golden_draws():
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    for seed, k, val in rows:
        draws = oracle.mulberry32_stream(int(seed), int(k) + 1)
        assert int(draws[int(k)]) == int(val)


def test_mulberry32_is_uniform():
    x = oracle.mulberry32_stream(7, 20000).astype(np.float64) / 2**32
    assert abs(x.mean() - 0.5) < 0.01
    hist, _ = np.histogram(x, bins=16, range=(0, 1))
    chi2 = ((hist - 1250.0) ** 2 / 1250.0).sum()
    assert chi2 < 40.0     # 15 dof, p ~ 5e-4


def test_perm_is_sorted_by_key_then_index():
    B = 5000
    for epoch in (0, 1, 3):
        p = oracle.perm(123, epoch, B)
        assert sorted(p.tolist()) == list(range(B))
        keys = oracle.mulberry32_stream(123, (epoch + 1) * B)[epoch * B:]
        ref = np.argsort(keys, kind="stable")           # library sort, ties by index
        assert np.array_equal(p, ref.astype(np.int32))


def test_perm_ties_keep_index_order():
    """mulberry32 is not injective, so equal keys occur in long streams; the
    definition orders them by index."""
    B = 200000
    keys = oracle.mulberry32_stream(0, B)
    u, counts = np.unique(keys, return_counts=True)
    assert (counts > 1).any()
    p = oracle.perm(0, 0, B)
    assert np.array_equal(p, np.argsort(keys, kind="stable").astype(np.int32))
    for key in u[counts > 1][:5]:
        pos = np.nonzero(keys[p] == key)[0]
        assert np.all(np.diff(p[pos]) > 0)


def test_different_epochs_differ():
    a = oracle.perm(0, 0, 1000)
    b = oracle.perm(0, 1, 1000)
    assert not np.array_equal(a, b)
