"""ppo_gae_noalloc: the GAE entry point for callers that cannot allocate
device memory (for example while a stream is being captured into a CUDA
graph, or in loops that must never enter the allocator).  Its scratch is a
fixed array inside the library, so it is checked here against ppo_gae, which
takes a caller-allocated workspace: two calls in a row, different inputs, same
tolerance as the GAE parity tests (|x - y| <= 1e-5 (|y| + rms(y))).  This file
is collected last so that a run stopping at its first failure has already run
every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

from policy_rl_gb300 import synth
from tests._gpu import assert_elementwise

pytestmark = pytest.mark.gpu


def _call(fn_name, lib, tensors, T, N, gamma, lam, work=None):
    import torch
    rew, val, done, boot, adv, ret, advn, st = tensors
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if fn_name == "ppo_gae_noalloc":
        return lib.ppo_gae_noalloc(p(rew), p(val), p(done), p(boot), T, N, gamma, lam, p(adv),
                                   p(ret), p(advn), p(st), stream)
    return lib.ppo_gae(p(rew), p(val), p(done), p(boot), T, N, gamma, lam, p(adv), p(ret),
                       p(advn), p(st), p(work), work.numel(), stream)


# (T, N, seed, with a stats buffer): two calls in a row with a caller stats
# buffer; then one without it, where the normalisation reads {mean, std} from
# the library's own array, at N >= 32768 (512-thread scan blocks, fewer
# partials than at small N)
CALLS = [(96, 3000, 1, True), (40, 777, 2, True), (4, 40000, 3, False)]


def test_noalloc_gae_matches_workspace_gae_on_consecutive_calls():
    import torch
    from policy_rl_gb300 import _abi
    import policy_rl_gb300 as P
    lib = _abi.load()
    for T, N, seed, with_stats in CALLS:
        w = synth.WORKLOADS["tiny"].scaled(T=T, N=N)
        ro = synth.rollout(w, seed=seed)
        ins = [torch.from_numpy(np.ascontiguousarray(x)).cuda()
               for x in (ro.rew, ro.val, ro.done, ro.boot)]
        outs = {}
        for name in ("ppo_gae_noalloc", "ppo_gae"):
            o = [torch.empty(T, N, device="cuda") for _ in range(3)] + \
                [torch.empty(4, device="cuda") if with_stats else None]
            work = torch.empty(P.ppo_gae_workspace_bytes(T, N), dtype=torch.uint8,
                               device="cuda")
            assert _call(name, lib, ins + o, T, N, w.gamma, w.lam, work) == 0, name
            torch.cuda.synchronize()
            # the stats buffer holds {mean, std}; its last two floats are padding
            outs[name] = [t.cpu().numpy() for t in o[:3]]
            if with_stats:
                outs[name].append(o[3][:2].cpu().numpy())
        for got, ref in zip(outs["ppo_gae_noalloc"], outs["ppo_gae"]):
            assert_elementwise(got, ref, 1e-5)


def test_noalloc_gae_rejects_n_beyond_its_scratch():
    import torch
    from policy_rl_gb300 import _abi
    lib = _abi.load()
    x = torch.zeros(16, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ppo_gae_noalloc(p, p, p, p, 1, (1 << 20) + 1, 0.99, 0.95, p, p, p, p, s) == 4
